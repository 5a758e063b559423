// Instantiations of the persistent GEMM on e4m3 operands (kind::f8f6f4) with
// the cross-entropy epilogues: the online log-sum-exp state of the forward
// and the softmax gradient of the backward's recomputed logits (BN = 256;
// single-CTA, CTA-pair and two-pair variants).
#include "coda_launch.cuh"

namespace coda {
cudaError_t launch_gemm_celse_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                  const GemmArgs& a) {
  return launch_gemm_impl<256, EpiCeLse<256>, true>(num_units, sms, cg, s, m, a);
}
cudaError_t launch_gemm_cedlogits_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                      const GemmArgs& a) {
  return launch_gemm_impl<256, EpiCeDlogits<256>, true>(num_units, sms, cg, s, m, a);
}
}  // namespace coda
