// Instantiations of the persistent GEMM with the EpiQkRope epilogue in its
// half-split RoPE pairing (pairs (j, j + 64) of each head), BN = 256,
// single-CTA, CTA-pair and two-pair (shared B) variants.
#include "coda_launch.cuh"

namespace coda {
cudaError_t launch_gemm_qkrope_half(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                     const GemmArgs& a) {
  return launch_gemm_impl<256, EpiQkRope<256, true>>(num_units, sms, cg, s, m, a);
}
}  // namespace coda
