// Instantiations of the persistent GEMM on e4m3 operands (kind::f8f6f4) with
// the EpiQkRope epilogue in both RoPE pairings (BN = 256; single-CTA,
// CTA-pair and two-pair variants).  The operand scales reach the epilogue as
// acc_rs / acc_cs.
#include "coda_launch.cuh"

namespace coda {
cudaError_t launch_gemm_qkrope_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                   const GemmArgs& a) {
  return launch_gemm_impl<256, EpiQkRope<256>, true>(num_units, sms, cg, s, m, a);
}
cudaError_t launch_gemm_qkrope_half_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                        const GemmArgs& a) {
  return launch_gemm_impl<256, EpiQkRope<256, true>, true>(num_units, sms, cg, s, m, a);
}
}  // namespace coda
