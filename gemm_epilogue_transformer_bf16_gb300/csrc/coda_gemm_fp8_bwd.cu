// Instantiations of the persistent GEMM on e4m3 operands (kind::f8f6f4) with
// the backward epilogues: dSwiGLU on the dH GEMM and the RMSNorm-backward
// input gradient (BN = 256; single-CTA, CTA-pair and two-pair variants).
#include "coda_launch.cuh"

namespace coda {
cudaError_t launch_gemm_dswiglu_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                    const GemmArgs& a) {
  return launch_gemm_impl<256, EpiDSwiglu<256>, true>(num_units, sms, cg, s, m, a);
}
cudaError_t launch_gemm_rmsdx_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                  const GemmArgs& a) {
  return launch_gemm_impl<256, EpiRmsDx<256>, true>(num_units, sms, cg, s, m, a);
}
}  // namespace coda
