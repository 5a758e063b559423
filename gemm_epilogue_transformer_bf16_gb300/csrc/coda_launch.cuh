// Launch helper for one (tile width, epilogue) instantiation of
// coda_gemm_kernel: raises the dynamic shared-memory limit once per device and
// launches one 192-thread CTA per SM-slot of the persistent grid.
#pragma once
#include "coda_epilogues.cuh"
#include "coda_internal.h"

namespace coda {

template <int BN, class Epi>
cudaError_t launch_gemm_impl(dim3 grid, cudaStream_t s, const CUtensorMap* m, const GemmArgs& a) {
  constexpr uint32_t smem = GemmCfg<BN>::SMEM_BYTES;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(coda_gemm_kernel<BN, Epi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  coda_gemm_kernel<BN, Epi><<<grid, NUM_THREADS, smem, s>>>(m[0], m[1], m[2], m[3], a);
  return cudaGetLastError();
}

}  // namespace coda
