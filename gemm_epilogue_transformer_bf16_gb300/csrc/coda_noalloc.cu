// Linear + cross-entropy forward for callers that cannot allocate device
// memory.
//
// Some callers have no way to obtain scratch memory: a plugin or callback
// inside a host application that owns every byte of device memory and hands
// the plugin only its input and output buffers (no allocator, no workspace
// argument), or a latency-critical loop that must not call cudaMalloc
// because it may synchronise the device.  coda_linear_cross_entropy_noalloc
// serves them: it runs the same kernels as coda_linear_cross_entropy, but its
// scratch (the device status word, the per-row target logits and the
// (max, sum-exp) partials of every vocabulary chunk) lives in the file-scope
// device array below instead of a caller workspace.  The array is part of the
// library image: every GPU that loads libcoda.so holds these bytes until the
// process exits.
#include <mutex>

#include "coda.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;  // 8 MiB

static __device__ __align__(256) unsigned char g_ce_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_ce_scratch on the current device.  In host code the
// name g_ce_scratch is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.  It is
// kept for the life of the process; a cudaDeviceReset reloads the module at
// another address, which is why the header rules out calls after a reset.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ce_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" size_t coda_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int coda_linear_cross_entropy_noalloc(const coda_bf16* X, const coda_bf16* W, const int32_t* labels,
                                                 int32_t ignore_index, float* loss_mean, float* lse,
                                                 int32_t* n_valid, int32_t* status_out, int64_t M, int64_t V,
                                                 int64_t K, coda_stream stream) {
  if (M < 0 || V < 0 || K < 0) return CODA_ERR_INVALID_ARG;
  if (coda_linear_cross_entropy_workspace_size(M, V, K) > kNoAllocScratchBytes) return CODA_ERR_WORKSPACE;
  void* ws = scratch_on_current_device();
  if (!ws) return CODA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents.  Only the status word must
  // start at zero; every other byte the call reads, it writes first.
  if (cudaMemsetAsync(ws, 0, 256, s) != cudaSuccess) return CODA_ERR_CUDA;
  const int r = coda_linear_cross_entropy(X, W, labels, ignore_index, loss_mean, lse, n_valid, M, V, K, ws,
                                          kNoAllocScratchBytes, stream);
  if (r != CODA_OK) return r;
  if (status_out &&
      cudaMemcpyAsync(status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return CODA_ERR_CUDA;
  return CODA_OK;
}
