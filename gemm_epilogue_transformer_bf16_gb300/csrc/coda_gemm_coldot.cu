// Instantiation of the persistent GEMM with the EpiColDot epilogue (BN = 256).
#include "coda_launch.cuh"

namespace coda {
cudaError_t launch_gemm_coldot(dim3 grid, cudaStream_t s, const CUtensorMap* m, const GemmArgs& a) {
  return launch_gemm_impl<256, EpiColDot<256>>(grid, s, m, a);
}
}  // namespace coda
