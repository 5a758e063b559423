// Launch helper for one (tile width, epilogue) instantiation of
// coda_gemm_kernel (m: six tensor maps -- A0, B0, A1, B1 and the two
// epilogue-ring tensors): raises the dynamic shared-memory limit once per device and
// launches the persistent grid -- one 192-thread CTA per SM, or, for the
// clustered variants (CTA pairs, two pairs sharing B), as many 2- or 4-CTA
// clusters as can be resident at once (cudaOccupancyMaxActiveClusters).
#pragma once
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include "coda_epilogues.cuh"
#include "coda_internal.h"

namespace coda {

// GEMM launches use programmatic dependent launch (CODA_PDL=0 in the
// environment turns it off, for comparisons).
inline bool programmatic_launch() {
  static const bool v = [] {
    const char* e = std::getenv("CODA_PDL");
    return e ? e[0] != '0' : true;
  }();
  return v;
}

template <int BN, class Epi, int CG, bool FP8>
cudaError_t launch_gemm_variant(int num_units, int sms, cudaStream_t s, const CUtensorMap* m, const GemmArgs& a) {
  constexpr uint32_t smem = GemmCfg<BN, (CG >= 2), EpiRing<Epi>::value>::SMEM_BYTES;
  // per device, set up once (first calls from several host threads are
  // serialised on `init`): the shared-memory limit and the resident-cluster
  // count; afterwards read without the lock
  static std::mutex init;
  static std::atomic<bool> attr_done[64];
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kern = coda_gemm_kernel<BN, Epi, CG, FP8>;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(init);
    if (!attr_done[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      attr_done[dev].store(true, std::memory_order_release);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  if constexpr (CG >= 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (max_clusters[dev].load(std::memory_order_acquire) == 0) {
      std::lock_guard<std::mutex> lock(init);
      if (max_clusters[dev].load(std::memory_order_relaxed) == 0) {
        cfg.gridDim = dim3(static_cast<unsigned>(sms - sms % CG));
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (n <= 0) return cudaErrorInvalidConfiguration;
        max_clusters[dev].store(n, std::memory_order_release);
#ifdef CODA_DEBUG_LAUNCH
        fprintf(stderr, "coda: cluster size %d, %d resident clusters\n", CG, n);
#endif
      }
    }
    const int resident = max_clusters[dev].load(std::memory_order_acquire);
    if (a.query_clusters) {
      *a.query_clusters = resident;
      return cudaSuccess;
    }
    const int cap = a.max_clusters > 0 ? std::min(a.max_clusters, resident) : resident;
    cfg.gridDim = dim3(static_cast<unsigned>(CG * std::min(num_units, cap)));
  } else {
    if (a.query_clusters) {
      *a.query_clusters = sms;
      return cudaSuccess;
    }
    const int cap = a.max_clusters > 0 ? std::min(a.max_clusters, sms) : sms;
    cfg.gridDim = dim3(static_cast<unsigned>(std::min(num_units, cap)));
  }
  if (programmatic_launch()) {
    // may start before the previous kernel in the stream has finished: the
    // kernel runs its prologue, then waits for it (griddep_wait)
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    ++cfg.numAttrs;
  }
  note_launch();
  e = cudaLaunchKernelEx(&cfg, kern, m[0], m[1], m[2], m[3], m[4], m[5], a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BN, class Epi, bool FP8 = false>
cudaError_t launch_gemm_impl(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                             const GemmArgs& a) {
  switch (cg) {
    case 1: return launch_gemm_variant<BN, Epi, 1, FP8>(num_units, sms, s, m, a);
    case 2: return launch_gemm_variant<BN, Epi, 2, FP8>(num_units, sms, s, m, a);
    case 4: return launch_gemm_variant<BN, Epi, 4, FP8>(num_units, sms, s, m, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace coda
