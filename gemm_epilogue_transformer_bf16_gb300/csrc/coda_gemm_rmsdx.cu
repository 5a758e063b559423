// Instantiations of the persistent GEMM with the EpiRmsDx epilogue (BN = 256),
// single-CTA, CTA-pair and two-pair (shared B) variants.
#include "coda_launch.cuh"

namespace coda {
cudaError_t launch_gemm_rmsdx(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                              const GemmArgs& a) {
  return launch_gemm_impl<256, EpiRmsDx<256>>(num_units, sms, cg, s, m, a);
}
}  // namespace coda
