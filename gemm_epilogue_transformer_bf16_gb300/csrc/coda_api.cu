// Host side of libcoda.so: argument validation, TMA tensor-map encoding,
// tile-grid planning and the launch sequences of the named operators declared
// in include/coda.h.  Nothing here allocates device memory: scratch lives in
// the caller's workspace, whose first 256 bytes are the device status word.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <utility>
#include <mutex>

#include "coda.h"
#include "coda_internal.h"
#include "coda_status.h"

namespace coda {
namespace {
std::atomic<unsigned long long> g_launches{0};
}  // namespace
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace coda

using coda::EpiArgs;
using coda::GemmArgs;

namespace {

constexpr size_t WS_HEADER = 256;
constexpr int BN = 256;
constexpr uint64_t TIMEOUT_NS = 2000000000ull;  // 2 s per pipeline wait
constexpr int CE_TILES_PER_UNIT = 16;

// ------------------------------------------------------------------ helpers
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsCursor {
  uint8_t* base;
  size_t off;
  explicit WsCursor(void* ws) : base(static_cast<uint8_t*>(ws)), off(WS_HEADER) {}
  template <class T>
  T* take(size_t count) {
    T* p = reinterpret_cast<T*>(base + off);
    off = up256(off + count * sizeof(T));
    return p;
  }
};

struct SizeCursor {
  size_t off = WS_HEADER;
  template <class T>
  void take(size_t count) { off = up256(off + count * sizeof(T)); }
};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

std::atomic<int> g_num_sms[64];  // per device, cached on first use

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = g_num_sms[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_num_sms[dev].store(n, std::memory_order_relaxed);  // every thread stores the same value
  }
  return n;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix with row stride
// `ld` elements; box = box_cols x box_rows, 128-byte swizzle (or `swz`),
// zero fill.
bool encode_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld, uint32_t box_cols,
                uint32_t box_rows, int elem_bytes = 2, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A 2-D byte tensor map without swizzling (rows of `cols` bytes), for data
// that is not a matrix operand (the NVFP4 block scales).
bool encode_map_plain(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, uint32_t box_cols,
                      uint32_t box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// One GEMM + epilogue launch.
struct Plan {
  coda::EpiKind kind = coda::EpiKind::Plain;
  const void* A = nullptr;
  int64_t lda = 0;
  int a_mn = 0;
  const void* B = nullptr;
  int64_t ldb = 0;
  int b_mn = 0;
  const void* A2 = nullptr;  // concatenated-K second pair
  int64_t lda2 = 0;
  const void* B2 = nullptr;  // second pair's B, or SwiGLU up weight (b_dual)
  int64_t ldb2 = 0;
  int64_t K2 = 0;
  int b_dual = 0;
  int fp8 = 0;  // e4m3 operands (K-major only)
  int64_t M = 0, N = 0, K = 0;
  int n_per_unit = 1;
  int rope_half = 0;  // QkRope: half-split RoPE pairs
  float cluster_share = 0.f;  // in (0, 1): run on this share of the resident clusters (two GEMMs side by side)
  EpiArgs e{};
};

// Cluster size of a GEMM launch.  CTA pairs (cta_group::2, 256-row tiles)
// halve each SM's B traffic; two pairs on adjacent 256-row blocks that share
// the B tile through TMA multicast cut each SM's operand traffic by another
// quarter.  A problem of one 128-row block keeps single CTAs.  In the
// environment, CODA_CTA_PAIR=0 selects single CTAs everywhere and
// CODA_CTA_QUAD=0 stops at pairs (for comparisons); CODA_CTA_QUAD=2 keeps
// two-pair clusters for GEMMs with an MN-major operand or K <= 4096 only.
int cluster_ctas(int64_t M, int a_mn, int b_mn, int64_t K) {
  static const bool pairs = [] {
    const char* v = std::getenv("CODA_CTA_PAIR");
    return !(v && v[0] == '0');
  }();
  static const int quads = [] {
    const char* v = std::getenv("CODA_CTA_QUAD");
    return v ? std::atoi(v) : 1;
  }();
  if (!pairs || M <= coda::BM) return 1;
  if (M <= 2 * coda::BM || quads == 0) return 2;
  if (quads == 2 && !a_mn && !b_mn && K > 4096) return 2;
  return 4;
}

// Units of the M tile per raster group (2048 rows by default): concurrent
// tiles share these rows' A panel in L2 while B streams.  CODA_GROUP_M
// overrides it.
int group_m(int cg) {
  static const int env = [] {
    const char* v = std::getenv("CODA_GROUP_M");
    return v ? std::atoi(v) : 0;
  }();
  if (env > 0) return env;
  return 16 / cg;
}

// L2 cache-hint selection for the GEMM launches: bit 0 = A loads evict_last,
// bit 1 = B loads evict_first, bit 2 = streaming (evict-first) epilogue
// stores.  Default (-1): streaming stores for a launch whose outputs exceed
// STREAM_STORE_BYTES (they cannot stay in the 126 MB L2 anyway, and written
// normally they evict the operand panels that concurrent tiles re-read: on
// the gate/up GEMM of the block, 6.59 -> 5.82 GB of DRAM reads per launch at
// the same speed); smaller outputs stay in L2 for the kernel that reads them
// next.  CODA_L2_HINTS overrides with a fixed bit set.
constexpr int64_t STREAM_STORE_BYTES = 64ll << 20;

// The dSwiGLU epilogue requests its tile's rows of g and u into L2 before its
// chunk loop (on by default; CODA_AUX_PREFETCH=0 turns it off, for
// comparisons).
int aux_prefetch() {
  static const int v = [] {
    const char* e = std::getenv("CODA_AUX_PREFETCH");
    return (e && e[0] == '0') ? 0 : 1;
  }();
  return v;
}

// The plain epilogue runs a chunk loop compiled for its launch's features
// (row scale, residual, partial sums, second output) unless the launch
// needs others; CODA_EPI_LEAN=0 makes every launch take the general loop
// (for comparisons).
int epi_no_lean() {
  static const int v = [] {
    const char* e = std::getenv("CODA_EPI_LEAN");
    return (e && e[0] == '0') ? 1 : 0;
  }();
  return v;
}

// The plain epilogue's residual comes through the TMA ring (copies of 32 x
// 32 tiles into shared memory issued ahead of the chunk loop) instead of
// per-thread loads.  CODA_EPI_RING=0 turns it off (for comparisons).
bool epi_ring_enabled() {
  static const bool v = [] {
    const char* e = std::getenv("CODA_EPI_RING");
    return !(e && e[0] == '0');
  }();
  return v;
}

// A two-pair GEMM whose units fill the grid's last wave poorly runs as CTA
// pairs when that takes at least 7 % fewer waves (a pair and a two-pair unit
// take the same time per CTA; pairs lose the B multicast between pairs,
// worth about 3 %).  On by default; CODA_PAIR_WAVES=0 turns it off.
bool pair_waves_enabled() {
  static const bool v = [] {
    const char* e = std::getenv("CODA_PAIR_WAVES");
    return !(e && e[0] == '0');
  }();
  return v;
}
int l2_hints() {
  static const int v = [] {
    const char* e = std::getenv("CODA_L2_HINTS");
    return e ? std::atoi(e) : -1;
  }();
  return v;
}
int stream_stores(int64_t out_bytes) {
  const int h = l2_hints();
  if (h >= 0) return (h & 4) ? 1 : 0;
  return out_bytes > STREAM_STORE_BYTES ? 1 : 0;
}
int load_hints() {
  const int h = l2_hints();
  return h >= 0 ? (h & 3) : 0;
}

// Back-off (ns) of the GEMM's waiting warps: the producer between stages
// (0: it must refill a stage as soon as the MMAs release it) and the epilogue
// while the accumulator fills (its polling otherwise spends power the tensor
// cores could use under the power cap).  CODA_WAIT_SLEEP="producer,epilogue"
// overrides the defaults.
void wait_sleep(uint32_t& producer, uint32_t& epilogue) {
  static const std::pair<uint32_t, uint32_t> v = [] {
    uint32_t a = 0, b = 512;
    if (const char* e = std::getenv("CODA_WAIT_SLEEP")) {
      unsigned x = 0, y = 0;
      if (std::sscanf(e, "%u,%u", &x, &y) == 2) {
        a = x;
        b = y;
      }
    }
    return std::make_pair(a, b);
  }();
  producer = v.first;
  epilogue = v.second;
}

#define CK(x)                  \
  do {                         \
    int _r = (x);              \
    if (_r != CODA_OK) return _r; \
  } while (0)
#define CU(x) \
  do { if ((x) != cudaSuccess) return CODA_ERR_CUDA; } while (0)

// Events that order work across two streams within one call; destroyed when
// the call returns (destruction of a recorded event is deferred by the
// runtime until the work it tracks has completed).
class EventSet {
 public:
  explicit EventSet(int n) : n_(n < 12 ? n : 12) {
    for (int i = 0; i < n_; ++i)
      if (cudaEventCreateWithFlags(&e_[i], cudaEventDisableTiming) != cudaSuccess) ok_ = false;
  }
  ~EventSet() {
    for (int i = 0; i < n_; ++i)
      if (e_[i]) cudaEventDestroy(e_[i]);
  }
  EventSet(const EventSet&) = delete;
  EventSet& operator=(const EventSet&) = delete;
  bool ok() const { return ok_; }
  cudaEvent_t operator[](int i) const { return e_[i]; }

 private:
  int n_;
  bool ok_ = true;
  cudaEvent_t e_[12] = {};
};

// Kernel dispatch by epilogue kind and operand type.  With a.query_clusters
// set, reports the resident-cluster limit of that kernel instead of launching.
int dispatch(const Plan& p, int sms, int cg, cudaStream_t s, const CUtensorMap* maps, const GemmArgs& a) {
  const int nu = a.num_units;
  cudaError_t err;
  if (p.fp8) {
    switch (p.kind) {
      case coda::EpiKind::Plain: err = coda::launch_gemm_plain_fp8(nu, sms, cg, s, maps, a); break;
      case coda::EpiKind::Swiglu: err = coda::launch_gemm_swiglu_fp8(nu, sms, cg, s, maps, a); break;
      case coda::EpiKind::QkRope:
        err = p.rope_half ? coda::launch_gemm_qkrope_half_fp8(nu, sms, cg, s, maps, a)
                          : coda::launch_gemm_qkrope_fp8(nu, sms, cg, s, maps, a);
        break;
      case coda::EpiKind::CeLse: err = coda::launch_gemm_celse_fp8(nu, sms, cg, s, maps, a); break;
      case coda::EpiKind::CeDlogits: err = coda::launch_gemm_cedlogits_fp8(nu, sms, cg, s, maps, a); break;
      case coda::EpiKind::DSwiglu: err = coda::launch_gemm_dswiglu_fp8(nu, sms, cg, s, maps, a); break;
      case coda::EpiKind::RmsDx: err = coda::launch_gemm_rmsdx_fp8(nu, sms, cg, s, maps, a); break;
      default: return CODA_ERR_UNSUPPORTED;
    }
    return err == cudaSuccess ? CODA_OK : CODA_ERR_CUDA;
  }
  switch (p.kind) {
    case coda::EpiKind::Plain: err = coda::launch_gemm_plain(nu, sms, cg, s, maps, a); break;
    case coda::EpiKind::Swiglu: err = coda::launch_gemm_swiglu(nu, sms, cg, s, maps, a); break;
    case coda::EpiKind::DSwiglu: err = coda::launch_gemm_dswiglu(nu, sms, cg, s, maps, a); break;
    case coda::EpiKind::QkRope:
      err = p.rope_half ? coda::launch_gemm_qkrope_half(nu, sms, cg, s, maps, a)
                        : coda::launch_gemm_qkrope(nu, sms, cg, s, maps, a);
      break;
    case coda::EpiKind::CeLse: err = coda::launch_gemm_celse(nu, sms, cg, s, maps, a); break;
    case coda::EpiKind::CeDlogits: err = coda::launch_gemm_cedlogits(nu, sms, cg, s, maps, a); break;
    case coda::EpiKind::ColDot: err = coda::launch_gemm_coldot(nu, sms, cg, s, maps, a); break;
    case coda::EpiKind::Sigmoid: err = coda::launch_gemm_sigmoid(nu, sms, cg, s, maps, a); break;
    case coda::EpiKind::RmsDx: err = coda::launch_gemm_rmsdx(nu, sms, cg, s, maps, a); break;
    default: return CODA_ERR_INVALID_ARG;
  }
  return err == cudaSuccess ? CODA_OK : CODA_ERR_CUDA;
}

// Tensor maps and kernel arguments of one launch with cluster size `cg` over
// the N tiles [nb_base, nb_base + n_tiles).
int prepare(const Plan& p, int* status, int cg, int nb_base, int n_tiles, CUtensorMap* maps, GemmArgs& a) {
  const bool pair = cg >= 2;
  // K-major B rows one TMA copy stages: the tile's N, its half per pair CTA,
  // a quarter per CTA with two pairs (each copy multicast to both pairs)
  const uint32_t b_box_rows = static_cast<uint32_t>(BN / cg);
  std::memset(maps, 0, 6 * sizeof(CUtensorMap));
  // a k-slice is 128 bytes: 64 bf16 or 128 e4m3 elements
  const int esz = p.fp8 ? 1 : 2;
  const uint32_t kbox = p.fp8 ? 2 * coda::BK : coda::BK;
  if (p.fp8 && (p.a_mn || p.b_mn)) return CODA_ERR_UNSUPPORTED;
  auto enc_a = [&](CUtensorMap* m, const void* ptr, int64_t ld, int64_t Kc) {
    return p.a_mn ? encode_map(m, ptr, Kc, p.M, ld, 64, 64) : encode_map(m, ptr, p.M, Kc, ld, kbox, 128, esz);
  };
  auto enc_b = [&](CUtensorMap* m, const void* ptr, int64_t ld, int64_t Kc) {
    return p.b_mn ? encode_map(m, ptr, Kc, p.N, ld, 64, 64)
                  : encode_map(m, ptr, p.N, Kc, ld, kbox, b_box_rows, esz);
  };
  if (!enc_a(&maps[0], p.A, p.lda, p.K)) return CODA_ERR_CUDA;
  if (p.b_dual) {
    const uint32_t rows = cg == 4 ? BN / 4 : BN / 2;
    if (!encode_map(&maps[1], p.B, p.N, p.K, p.ldb, kbox, rows, esz)) return CODA_ERR_CUDA;
    if (!encode_map(&maps[3], p.B2, p.N, p.K, p.ldb2, kbox, rows, esz)) return CODA_ERR_CUDA;
    maps[2] = maps[0];
  } else {
    if (!enc_b(&maps[1], p.B, p.ldb, p.K)) return CODA_ERR_CUDA;
    if (p.K2 > 0) {
      if (!enc_a(&maps[2], p.A2, p.lda2, p.K2)) return CODA_ERR_CUDA;
      if (!enc_b(&maps[3], p.B2, p.ldb2, p.K2)) return CODA_ERR_CUDA;
    } else {
      maps[2] = maps[0];
      maps[3] = maps[1];
    }
  }
  a = GemmArgs{};
  a.M = static_cast<int>(p.M);
  a.N = static_cast<int>(p.N);
  a.num_m = static_cast<int>(cdiv(p.M, cg * coda::BM));
  a.num_n = n_tiles;
  a.nb_base = nb_base;
  a.kb0 = static_cast<int>(cdiv(p.K, kbox));
  a.kb1 = p.K2 > 0 ? static_cast<int>(cdiv(p.K2, kbox)) : 0;
  a.a_mn = p.a_mn;
  a.b_mn = p.b_mn;
  a.b_dual = p.b_dual;
  a.n_per_unit = p.n_per_unit;
  a.num_units = p.n_per_unit > 1 ? a.num_m * static_cast<int>(cdiv(a.num_n, p.n_per_unit)) : a.num_m * a.num_n;
  a.group_m = group_m(cg);
  a.idesc = p.fp8 ? coda::idesc_e4m3(pair ? 2 * coda::BM : coda::BM, BN)
                  : coda::idesc_bf16(pair ? 2 * coda::BM : coda::BM, BN, p.a_mn, p.b_mn);
  a.status = status;
  a.timeout_ns = TIMEOUT_NS;
  a.l2_hints = load_hints();
  wait_sleep(a.producer_sleep_ns, a.epilogue_sleep_ns);
  a.e = p.e;
  {
    // bytes the epilogue writes: D and the optional second, third and
    // fourth outputs, over the launch's share of the N tiles
    const int64_t cols = std::min<int64_t>(p.N, static_cast<int64_t>(n_tiles) * (p.b_dual ? BN / 2 : BN));
    const int n_out = 1 + (p.e.out1 != nullptr) + (p.e.out2 != nullptr) + (p.e.out3 != nullptr);
    const int64_t esz = p.e.d_f32 ? 4 : 2;
    a.e.st_stream = stream_stores(p.M * cols * esz * n_out);
  }
  a.e.aux_prefetch = aux_prefetch();
  a.e.no_lean = epi_no_lean();
  a.e.ring = 0;
  if (p.kind == coda::EpiKind::Plain && p.e.aux0 && epi_ring_enabled() && al16(p.e.aux0) && p.e.ld_aux0 % 8 == 0 &&
      p.e.ld_aux0 >= p.N) {
    // the residual as [M, N] with row stride ld_aux0, read in 32 x 32 boxes
    if (!encode_map(&maps[4], p.e.aux0, p.M, p.N, p.e.ld_aux0, 32, 32, 2, CU_TENSOR_MAP_SWIZZLE_64B))
      return CODA_ERR_CUDA;
    a.e.ring = 1;
  }
  return CODA_OK;
}

// Helper streams of a call issued on `s`: role 0 carries the CTA-pair slice
// of a split launch, roles 1 and 2 the dX and dW GEMMs of the sliced
// cross-entropy backward.  One non-blocking stream per (device, caller
// stream, role), created once and kept for the process, so that GEMMs the
// caller runs concurrently on different streams do not queue behind each
// other's helpers.
cudaStream_t side_stream(cudaStream_t s, int role = 0) {
  static std::mutex mu;
  constexpr int kSlots = 96;
  static int dev_of[kSlots];
  static int role_of[kSlots];
  static cudaStream_t key[kSlots];
  static cudaStream_t val[kSlots];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (dev_of[i] == dev && key[i] == s && role_of[i] == role) return val[i];
  if (used == kSlots) return nullptr;  // no more slots: the caller stays on s
  cudaStream_t t = nullptr;
  if (cudaStreamCreateWithFlags(&t, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
  dev_of[used] = dev;
  role_of[used] = role;
  key[used] = s;
  val[used] = t;
  ++used;
  return t;
}

// Split launches (CODA_SPLIT=1 in the environment; off by default): the
// two-pair kernel leaves the SMs its 4-CTA clusters cannot use (GPCs whose
// SM count is not a multiple of 4) idle.  A CTA-pair kernel sized to those
// SMs takes the last N tiles, on a second stream, and the split point
// balances the two kernels' waves (a two-pair unit and a pair unit take the
// same time).  Both kernels become runnable at the same moment, and where
// the pair kernel's CTAs are placed first they take SMs that the two-pair
// clusters needed, whose units then run late: in a loop of block steps the
// split made each step 5 % slower, and it came out ahead only with a timing
// event recorded between the step's stages.
bool split_enabled() {
  static const bool v = [] {
    const char* e = std::getenv("CODA_SPLIT");
    return e && e[0] == '1';
  }();
  return v;
}

int run(const Plan& p, int* status, cudaStream_t s) {
  if (p.M == 0 || p.N == 0) return CODA_OK;
  if (!get_encoder()) return CODA_ERR_CUDA;
  const int sms = num_sms();
  if (sms <= 0) return CODA_ERR_CUDA;
  const int cg = cluster_ctas(p.M, p.a_mn, p.b_mn, p.K + p.K2);
  const int num_n = static_cast<int>(cdiv(p.N, p.b_dual ? BN / 2 : BN));
  CUtensorMap maps[6];
  GemmArgs a;
  int cg_run = cg;
  if (p.cluster_share > 0.f && p.cluster_share < 1.f) {
    // a fixed share of the resident clusters, no split launch: the caller
    // runs another GEMM beside this one on the rest
    int resident = 0;
    CK(prepare(p, status, cg, 0, num_n, maps, a));
    a.query_clusters = &resident;
    CK(dispatch(p, sms, cg, s, maps, a));
    a.query_clusters = nullptr;
    a.max_clusters = std::max(1, static_cast<int>(resident * p.cluster_share + 0.5f));
    return dispatch(p, sms, cg, s, maps, a);
  }
  if (cg == 4 && p.n_per_unit <= 1 && (split_enabled() || pair_waves_enabled())) {
    // resident clusters of the two-pair and the pair kernel
    int q_max = 0, p_max = 0;
    CK(prepare(p, status, 4, 0, num_n, maps, a));
    a.query_clusters = &q_max;
    CK(dispatch(p, sms, 4, s, maps, a));
    CK(prepare(p, status, 2, 0, num_n, maps, a));
    a.query_clusters = &p_max;
    CK(dispatch(p, sms, 2, s, maps, a));
    const int extra = p_max - 2 * q_max;  // pairs that fit beside a full two-pair grid
    const int64_t mq = cdiv(p.M, 4 * coda::BM), mp = cdiv(p.M, 2 * coda::BM);
    int best = 0;
    int64_t tbest = q_max > 0 ? cdiv(mq * num_n, q_max) : 0;
    if (q_max > 0 && extra > 0 && num_n >= 4 && split_enabled()) {
      for (int np = 1; np <= num_n / 4; ++np) {
        const int64_t t = std::max(cdiv(mq * (num_n - np), q_max), cdiv(mp * np, extra));
        if (t < tbest) {
          tbest = t;
          best = np;
        }
      }
    }
    if (q_max > 0 && p_max > 0 && pair_waves_enabled() && cdiv(mp * num_n, p_max) * 100 <= tbest * 93) {
      cg_run = 2;
      best = 0;
    }
    if (best > 0) {
      cudaStream_t s2 = side_stream(s);
      if (s2) {
        EventSet ev(2);
        if (!ev.ok()) return CODA_ERR_CUDA;
        CU(cudaEventRecord(ev[0], s));
        CU(cudaStreamWaitEvent(s2, ev[0], 0));
        CK(prepare(p, status, 4, 0, num_n - best, maps, a));
        CK(dispatch(p, sms, 4, s, maps, a));
        CUtensorMap maps2[6];
        GemmArgs a2;
        CK(prepare(p, status, 2, num_n - best, best, maps2, a2));
        a2.max_clusters = extra;
        CK(dispatch(p, sms, 2, s2, maps2, a2));
        CU(cudaEventRecord(ev[1], s2));
        CU(cudaStreamWaitEvent(s, ev[1], 0));
        return CODA_OK;
      }
    }
  }
  CK(prepare(p, status, cg_run, 0, num_n, maps, a));
  return dispatch(p, sms, cg_run, s, maps, a);
}


// Argument checks.  `need` pointers must be non-null; every non-null pointer
// must be 16-byte aligned.
int req(const void* p) { return p ? CODA_OK : CODA_ERR_INVALID_ARG; }
int al(const void* p) { return (p == nullptr || al16(p)) ? CODA_OK : CODA_ERR_ALIGNMENT; }
int ldok(int64_t ld, int64_t cols) {
  if (ld < cols) return CODA_ERR_INVALID_ARG;
  return (ld % 8) ? CODA_ERR_ALIGNMENT : CODA_OK;
}
int dims_ok(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return CODA_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return CODA_ERR_UNSUPPORTED;
  if (N % 8 || K % 8) return CODA_ERR_UNSUPPORTED;
  if (K == 0 && M > 0 && N > 0) return CODA_ERR_UNSUPPORTED;
  return CODA_OK;
}
int ws_ok(const void* ws, size_t have, size_t need) {
  if (!ws || have < need) return CODA_ERR_WORKSPACE;
  return al16(ws) ? CODA_OK : CODA_ERR_ALIGNMENT;
}

cudaStream_t S(coda_stream s) { return static_cast<cudaStream_t>(s); }
const __nv_bfloat16* BF(const coda_bf16* p) { return reinterpret_cast<const __nv_bfloat16*>(p); }
__nv_bfloat16* BF(coda_bf16* p) { return reinterpret_cast<__nv_bfloat16*>(p); }

}  // namespace

extern "C" {

const char* coda_version(void) { return "coda-gb300 0.1.0 (sm_103a)"; }

uint64_t coda_launch_count(void) { return coda::g_launches.load(std::memory_order_relaxed); }

const char* coda_status_string(int st) {
  switch (st) {
    case CODA_OK: return "CODA_OK";
    case CODA_ERR_INVALID_ARG: return "CODA_ERR_INVALID_ARG";
    case CODA_ERR_ALIGNMENT: return "CODA_ERR_ALIGNMENT";
    case CODA_ERR_UNSUPPORTED: return "CODA_ERR_UNSUPPORTED";
    case CODA_ERR_WORKSPACE: return "CODA_ERR_WORKSPACE";
    case CODA_ERR_CUDA: return "CODA_ERR_CUDA";
    case CODA_ERR_TIMEOUT: return "CODA_ERR_TIMEOUT";
    case CODA_ERR_LABEL_RANGE: return "CODA_ERR_LABEL_RANGE";
    case CODA_ERR_POSITION_RANGE: return "CODA_ERR_POSITION_RANGE";
    default: return "CODA_ERR_UNKNOWN";
  }
}

int coda_get_status(const void* ws, coda_stream stream) {
  if (!ws) return CODA_ERR_INVALID_ARG;
  int word = 0;
  CU(cudaStreamSynchronize(S(stream)));
  CU(cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost));
  if (word & CODA_DEV_TIMEOUT) return CODA_ERR_TIMEOUT;
  if (word & CODA_DEV_LABEL_RANGE) return CODA_ERR_LABEL_RANGE;
  if (word & CODA_DEV_POSITION_RANGE) return CODA_ERR_POSITION_RANGE;
  return CODA_OK;
}

int coda_reset_status(void* ws, coda_stream stream) {
  if (!ws) return CODA_ERR_INVALID_ARG;
  CU(cudaMemsetAsync(ws, 0, sizeof(int), S(stream)));
  return CODA_OK;
}

int coda_selftest_wait_timeout(uint32_t limit_us, void* ws, coda_stream stream) {
  if (limit_us == 0 || limit_us > 1000000u) return CODA_ERR_INVALID_ARG;
  CK(ws_ok(ws, WS_HEADER, WS_HEADER));
  CU(coda::launch_selftest_wait_timeout(static_cast<uint64_t>(limit_us) * 1000ull, static_cast<int*>(ws),
                                        S(stream)));
  return CODA_OK;
}

// ------------------------------------------------------------------ generic
size_t coda_gemm_epilogue_workspace_size(void) { return WS_HEADER; }

int coda_gemm_epilogue(const coda_epilogue_desc* d, const coda_bf16* A, int64_t lda, int a_major,
                       const coda_bf16* B, int64_t ldb, int b_major, void* D, int64_t ldd, int d_dtype, int64_t M,
                       int64_t N, int64_t K, void* ws, size_t ws_bytes, coda_stream stream) {
  CK(req(d));
  CK(dims_ok(M, N, K));
  CK(ws_ok(ws, ws_bytes, WS_HEADER));
  if (a_major != CODA_K_MAJOR && a_major != CODA_MN_MAJOR) return CODA_ERR_INVALID_ARG;
  if (b_major != CODA_K_MAJOR && b_major != CODA_MN_MAJOR) return CODA_ERR_INVALID_ARG;
  if (d_dtype != CODA_BF16 && d_dtype != CODA_F32) return CODA_ERR_INVALID_ARG;
  if (d->map < CODA_MAP_NONE || d->map > CODA_MAP_DSIGMOID) return CODA_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return CODA_OK;
  CK(req(A));
  CK(req(B));
  CK(al(A));
  CK(al(B));
  CK(al(D));
  CK(ldok(lda, a_major == CODA_K_MAJOR ? K : M));
  if (d->map == CODA_MAP_SWIGLU) {
    CK(ldok(ldb, K));
  } else {
    CK(ldok(ldb, b_major == CODA_K_MAJOR ? K : N));
  }
  if (d_dtype == CODA_F32 && d->map != CODA_MAP_NONE) return CODA_ERR_UNSUPPORTED;
  if (d->map != CODA_MAP_CE_LSE && d->map != CODA_MAP_QKNORM_ROPE && d->map != CODA_MAP_DSIGMOID) {
    CK(req(D));
    CK(ldok(ldd, N));
  }
  for (int i = 0; i < 2; ++i) {
    CK(al(d->aux_in[i]));
    if (d->aux_in[i]) CK(ldok(d->ld_aux_in[i], N));
  }
  for (int i = 0; i < 3; ++i) {
    CK(al(d->aux_out[i]));
    if (!d->aux_out[i]) continue;
    if (d->map == CODA_MAP_QKNORM_ROPE && i == 0) {
      // the pre-norm save holds only the q and k heads
      CK(ldok(d->ld_aux_out[0], static_cast<int64_t>(d->n_q_heads + d->n_kv_heads) * 128));
    } else {
      CK(ldok(d->ld_aux_out[i], N));
    }
  }
  CK(al(d->row_scale));
  CK(al(d->col_scale));
  CK(al(d->partials));
  Plan p;
  p.A = A;
  p.lda = lda;
  p.a_mn = a_major;
  p.B = B;
  p.ldb = ldb;
  p.b_mn = b_major;
  p.M = M;
  p.N = N;
  p.K = K;
  if (d->operand_type != CODA_OPERAND_BF16 && d->operand_type != CODA_OPERAND_E4M3) return CODA_ERR_INVALID_ARG;
  if (d->operand_type == CODA_OPERAND_E4M3) {
    // e4m3 operands: K-major, 16-byte rows
    if (a_major != CODA_K_MAJOR || b_major != CODA_K_MAJOR) return CODA_ERR_UNSUPPORTED;
    if (K % 16 || (d->K2 && d->K2 % 16) || lda % 16 || ldb % 16) return CODA_ERR_UNSUPPORTED;
    if (d->map == CODA_MAP_COLDOT || d->map == CODA_MAP_SIGMOID || d->map == CODA_MAP_DSIGMOID)
      return CODA_ERR_UNSUPPORTED;
    CK(al(d->acc_row_scale));
    CK(al(d->acc_col_scale));
    p.fp8 = 1;
  } else if (d->acc_row_scale || d->acc_col_scale) {
    return CODA_ERR_INVALID_ARG;
  }
  EpiArgs& e = p.e;
  e.acc_rs = d->acc_row_scale;
  e.acc_cs = d->acc_col_scale;
  e.D = D;
  e.ldd = ldd;
  e.d_f32 = d_dtype == CODA_F32;
  e.beta = d->beta;
  e.row_scale = d->row_scale;
  e.col_scale = d->col_scale;
  e.aux0 = reinterpret_cast<const __nv_bfloat16*>(d->aux_in[0]);
  e.ld_aux0 = d->ld_aux_in[0];
  e.aux1 = reinterpret_cast<const __nv_bfloat16*>(d->aux_in[1]);
  e.ld_aux1 = d->ld_aux_in[1];
  e.row_coef = d->row_coef;
  e.out1 = reinterpret_cast<__nv_bfloat16*>(d->aux_out[0]);
  e.ld_out1 = d->ld_aux_out[0];
  e.out2 = reinterpret_cast<__nv_bfloat16*>(d->aux_out[1]);
  e.ld_out2 = d->ld_aux_out[1];
  e.out3 = reinterpret_cast<__nv_bfloat16*>(d->aux_out[2]);
  e.ld_out3 = d->ld_aux_out[2];
  e.partials = d->partials;
  e.ld_part = d->ld_partials;
  if (d->row_coef && !d->aux_in[1]) return CODA_ERR_INVALID_ARG;
  if (d->K2 > 0) {
    if (d->map == CODA_MAP_SWIGLU) return CODA_ERR_UNSUPPORTED;
    CK(req(d->A2));
    CK(req(d->B2));
    CK(al(d->A2));
    CK(al(d->B2));
    if (d->K2 % 8) return CODA_ERR_UNSUPPORTED;
    CK(ldok(d->lda2, a_major == CODA_K_MAJOR ? d->K2 : M));
    CK(ldok(d->ldb2, b_major == CODA_K_MAJOR ? d->K2 : N));
    p.A2 = d->A2;
    p.lda2 = d->lda2;
    p.B2 = d->B2;
    p.ldb2 = d->ldb2;
    p.K2 = d->K2;
  }
  switch (d->map) {
    case CODA_MAP_NONE:
      p.kind = coda::EpiKind::Plain;
      if (e.partials && e.ld_part < M) return CODA_ERR_INVALID_ARG;
      break;
    case CODA_MAP_SWIGLU:
      p.kind = coda::EpiKind::Swiglu;
      if (b_major != CODA_K_MAJOR || !d->B2) return CODA_ERR_UNSUPPORTED;
      CK(al(d->B2));
      CK(ldok(d->ldb2, K));
      p.b_dual = 1;
      p.B2 = d->B2;
      p.ldb2 = d->ldb2;
      break;
    case CODA_MAP_DSWIGLU:
      p.kind = coda::EpiKind::DSwiglu;
      if (!d->aux_in[0] || !d->aux_in[1] || !d->aux_out[0] || !d->aux_out[1]) return CODA_ERR_INVALID_ARG;
      if (e.partials && e.ld_part < M) return CODA_ERR_INVALID_ARG;
      break;
    case CODA_MAP_QKNORM_ROPE:
      p.kind = coda::EpiKind::QkRope;
      if (d->head_dim != 128) return CODA_ERR_UNSUPPORTED;
      if (d->rope_pairing != CODA_ROPE_INTERLEAVED && d->rope_pairing != CODA_ROPE_HALF) return CODA_ERR_INVALID_ARG;
      p.rope_half = d->rope_pairing == CODA_ROPE_HALF;
      if (d->n_q_heads <= 0 || d->n_kv_heads < 0) return CODA_ERR_INVALID_ARG;
      if (N != static_cast<int64_t>(d->n_q_heads + 2 * d->n_kv_heads) * 128) return CODA_ERR_INVALID_ARG;
      if (!d->positions || !d->cos_sin || d->max_pos <= 0 || !d->gamma_q || !d->Q) return CODA_ERR_INVALID_ARG;
      if (d->n_kv_heads > 0 && (!d->gamma_k || !d->K || !d->V)) return CODA_ERR_INVALID_ARG;
      CK(al(d->Q));
      CK(al(d->K));
      CK(al(d->V));
      CK(al(d->gamma_q));
      CK(al(d->gamma_k));
      CK(al(d->cos_sin));
      e.pos = d->positions;
      e.cos_sin = reinterpret_cast<const float2*>(d->cos_sin);
      e.max_pos = d->max_pos;
      e.n_q = d->n_q_heads;
      e.n_kv = d->n_kv_heads;
      e.eps = d->eps;
      e.gamma_q = d->gamma_q;
      e.gamma_k = d->gamma_k;
      e.Q = reinterpret_cast<__nv_bfloat16*>(d->Q);
      e.Kh = reinterpret_cast<__nv_bfloat16*>(d->K);
      e.V = reinterpret_cast<__nv_bfloat16*>(d->V);
      e.ldq = static_cast<int64_t>(d->n_q_heads) * 128;
      e.ldk = e.ldv = static_cast<int64_t>(d->n_kv_heads) * 128;
      break;
    case CODA_MAP_CE_LSE:
      p.kind = coda::EpiKind::CeLse;
      if (!d->labels || !d->target_logit || !d->partials) return CODA_ERR_INVALID_ARG;
      if (d->ld_partials < M) return CODA_ERR_INVALID_ARG;
      p.n_per_unit = d->vocab_tiles_per_unit > 0 ? d->vocab_tiles_per_unit : CE_TILES_PER_UNIT;
      e.labels = d->labels;
      e.target_logit = d->target_logit;
      break;
    case CODA_MAP_CE_DLOGITS:
      p.kind = coda::EpiKind::CeDlogits;
      if (!d->labels || !d->lse || !d->n_valid) return CODA_ERR_INVALID_ARG;
      e.labels = d->labels;
      e.ignore_index = d->ignore_index;
      e.lse = d->lse;
      e.n_valid = d->n_valid;
      e.dloss = d->dloss;
      e.onehot = 1;
      break;
    case CODA_MAP_COLDOT:
      p.kind = coda::EpiKind::ColDot;
      if (!d->aux_in[0]) return CODA_ERR_INVALID_ARG;
      if (e.partials && e.ld_part < N) return CODA_ERR_INVALID_ARG;
      break;
    case CODA_MAP_SIGMOID:
      p.kind = coda::EpiKind::Sigmoid;
      e.mode = 0;
      break;
    case CODA_MAP_DSIGMOID:
      p.kind = coda::EpiKind::Sigmoid;
      if (!d->aux_in[1] || !d->aux_out[0]) return CODA_ERR_INVALID_ARG;
      if (d->aux_out[1] && !d->aux_in[0]) return CODA_ERR_INVALID_ARG;
      e.mode = 1;
      break;
  }
  return run(p, static_cast<int*>(ws), S(stream));
}

// ------------------------------------------------------------------ RMSNorm pieces
int coda_fold_gamma(const coda_bf16* W, const float* gamma, coda_bf16* Wf, int64_t N, int64_t K,
                    coda_stream stream) {
  CK(dims_ok(N, 8, K));
  if (N == 0) return CODA_OK;
  CK(req(W));
  CK(req(gamma));
  CK(req(Wf));
  CK(al(W));
  CK(al(gamma));
  CK(al(Wf));
  const int sms = num_sms();
  if (sms <= 0) return CODA_ERR_CUDA;
  CU(coda::launch_fold_gamma(BF(W), gamma, BF(Wf), N, K, sms, S(stream)));
  return CODA_OK;
}

int coda_rms_rstd(const coda_bf16* X, int64_t ldx, int64_t M, int64_t K, float eps, float* rstd,
                  coda_stream stream) {
  CK(dims_ok(M, 8, K));
  if (M == 0) return CODA_OK;
  CK(req(X));
  CK(req(rstd));
  CK(al(X));
  CK(ldok(ldx, K));
  const int sms = num_sms();
  if (sms <= 0) return CODA_ERR_CUDA;
  CU(coda::launch_row_rstd(BF(X), ldx, M, K, eps, rstd, sms, S(stream)));
  return CODA_OK;
}

int coda_rmsnorm_scale(const coda_bf16* X, int64_t ldx, int64_t M, int64_t K, float eps, const float* gamma,
                       float* rstd, coda_bf16* U, int64_t ldu, coda_stream stream) {
  CK(dims_ok(M, 8, K));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)X, (const void*)gamma, (const void*)rstd, (const void*)U}) {
    CK(req(q));
    CK(al(q));
  }
  CK(ldok(ldx, K));
  CK(ldok(ldu, K));
  const int sms = num_sms();
  if (sms <= 0) return CODA_ERR_CUDA;
  CU(coda::launch_row_rstd(BF(X), ldx, M, K, eps, rstd, sms, S(stream), gamma, BF(U), ldu));
  return CODA_OK;
}

int coda_rope_table(float theta, int32_t head_dim, int32_t max_pos, float* cos_sin, coda_stream stream) {
  if (head_dim <= 0 || head_dim % 2 || max_pos <= 0 || !(theta > 0.f)) return CODA_ERR_INVALID_ARG;
  CK(req(cos_sin));
  CK(al(cos_sin));
  CU(coda::launch_rope_table(static_cast<double>(theta), head_dim, max_pos, reinterpret_cast<float2*>(cos_sin),
                             S(stream)));
  return CODA_OK;
}

// ------------------------------------------------------------------ rmsnorm_linear
size_t coda_rmsnorm_linear_workspace_size(int64_t, int64_t, int64_t) { return WS_HEADER; }

int coda_rmsnorm_linear(const coda_bf16* X, const float* rstd_in, const coda_bf16* Wf, const coda_bf16* R,
                        float eps, float* rstd_out, coda_bf16* Y, int64_t M, int64_t N, int64_t K, void* ws,
                        size_t ws_bytes, coda_stream stream) {
  CK(dims_ok(M, N, K));
  CK(ws_ok(ws, ws_bytes, coda_rmsnorm_linear_workspace_size(M, N, K)));
  if (M == 0) return CODA_OK;
  CK(req(X));
  CK(req(Wf));
  CK(req(Y));
  if (!rstd_in && !rstd_out) return CODA_ERR_INVALID_ARG;
  for (const void* q : {(const void*)X, (const void*)Wf, (const void*)R, (const void*)Y, (const void*)rstd_in,
                        (const void*)rstd_out})
    CK(al(q));
  const float* rs = rstd_in;
  if (!rs) {
    CK(coda_rms_rstd(X, K, M, K, eps, rstd_out, stream));
    rs = rstd_out;
  }
  Plan p;
  p.A = X;
  p.lda = K;
  p.B = Wf;
  p.ldb = K;
  p.M = M;
  p.N = N;
  p.K = K;
  p.e.D = Y;
  p.e.ldd = N;
  p.e.row_scale = rs;
  p.e.aux0 = BF(R);
  p.e.ld_aux0 = N;
  return run(p, static_cast<int*>(ws), S(stream));
}

size_t coda_rmsnorm_linear_bwd_workspace_size(int64_t M, int64_t N, int64_t K) {
  SizeCursor c;
  c.take<__nv_bfloat16>(static_cast<size_t>(M) * N);  // G'
  c.take<float>(M);                                    // coef
  c.take<float>(static_cast<size_t>(4 * cdiv(M, 128)) * K);  // dgamma partials per (token block, warp)
  return c.off;
}

int coda_rmsnorm_linear_bwd(const coda_bf16* dY, const coda_bf16* X, const coda_bf16* W, const float* gamma, const float* rstd, const coda_bf16* Y, const coda_bf16* R,
                            coda_bf16* dX, coda_bf16* dW, float* dgamma, int64_t M, int64_t N, int64_t K, void* ws,
                            size_t ws_bytes, coda_stream stream, coda_stream side_stream) {
  CK(dims_ok(M, N, K));
  CK(ws_ok(ws, ws_bytes, coda_rmsnorm_linear_bwd_workspace_size(M, N, K)));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)dY, (const void*)X, (const void*)W, (const void*)gamma, (const void*)rstd,
                        (const void*)Y, (const void*)dX, (const void*)dW, (const void*)dgamma})
    CK(req(q));
  for (const void* q : {(const void*)dY, (const void*)X, (const void*)W, (const void*)gamma, (const void*)rstd,
                        (const void*)Y, (const void*)R, (const void*)dX, (const void*)dW, (const void*)dgamma})
    CK(al(q));
  const int sms = num_sms();
  if (sms <= 0) return CODA_ERR_CUDA;
  WsCursor w(ws);
  __nv_bfloat16* Gp = w.take<__nv_bfloat16>(static_cast<size_t>(M) * N);
  float* coef = w.take<float>(M);
  const int64_t ntb = cdiv(M, 128);
  float* dgp = w.take<float>(static_cast<size_t>(4 * ntb) * K);
  int* status = static_cast<int*>(ws);
  cudaStream_t s = S(stream);
  CU(coda::launch_rms_bwd_prepass(BF(dY), BF(Y), BF(R), rstd, M, N, 1.f / static_cast<float>(K), Gp, coef, sms,
                                  s));
  // With a side stream, dW runs beside c -> dX (both read only G', X, W), so
  // each GEMM's partly filled last wave overlaps the other; they share only
  // the status word (atomic OR).
  cudaStream_t s2 = side_stream ? S(side_stream) : s;
  // With a side stream the two GEMMs (equal FLOPs) each take half of the
  // resident clusters and run side by side: their prologues and last
  // epilogues overlap instead of queueing (4096 x 2048 x 2048: 0.1352 ->
  // 0.1311 ms per step, 0.1344 -> 0.1255 ms as a graph).  CODA_RMS_SHARE=0
  // gives each the whole grid.
  static const bool share_on = [] {
    const char* v = std::getenv("CODA_RMS_SHARE");
    return !(v && v[0] == '0');
  }();
  const float share = (s2 != s && share_on) ? 0.5f : 0.f;
  EventSet ev(s2 != s ? 2 : 0);
  if (!ev.ok()) return CODA_ERR_CUDA;
  if (s2 != s) {
    CU(cudaEventRecord(ev[0], s));
    CU(cudaStreamWaitEvent(s2, ev[0], 0));
  }
  {  // D = G' W;  dX = gamma D - c X, dgamma column partials sum_i X_ik D_ik
    Plan p;
    p.kind = coda::EpiKind::RmsDx;
    p.A = Gp;
    p.lda = N;
    p.B = W;
    p.ldb = K;
    p.b_mn = 1;
    p.M = M;
    p.N = K;
    p.K = N;
    p.e.D = dX;
    p.e.ldd = K;
    p.e.row_coef = coef;
    p.e.aux1 = BF(X);
    p.e.ld_aux1 = K;
    p.e.col_scale = gamma;
    p.e.partials = dgp;
    p.e.ld_part = K;
    p.cluster_share = share;
    CK(run(p, status, s));
  }
  {  // dW = (G'^T X) diag(gamma)
    Plan p;
    p.A = Gp;
    p.lda = N;
    p.a_mn = 1;
    p.B = X;
    p.ldb = K;
    p.b_mn = 1;
    p.M = N;
    p.N = K;
    p.K = M;
    p.e.D = dW;
    p.e.ldd = K;
    p.e.col_scale = gamma;
    p.cluster_share = share;
    CK(run(p, status, s2));
  }
  CU(coda::launch_colsum(dgp, 4 * ntb, K, K, dgamma, s));
  if (s2 != s) {
    CU(cudaEventRecord(ev[1], s2));
    CU(cudaStreamWaitEvent(s, ev[1], 0));
  }
  return CODA_OK;
}

// ------------------------------------------------------------------ linear_residual
size_t coda_linear_residual_workspace_size(int64_t M, int64_t N, int64_t) {
  SizeCursor c;
  c.take<float>(static_cast<size_t>(cdiv(N, BN)) * M);
  return c.off;
}

int coda_linear_residual(const coda_bf16* X, const coda_bf16* W, const coda_bf16* R, coda_bf16* Y, float eps,
                         float* rstd_out, const float* gamma_next, coda_bf16* U_out, int64_t M, int64_t N, int64_t K,
                         void* ws, size_t ws_bytes, coda_stream stream) {
  CK(dims_ok(M, N, K));
  CK(ws_ok(ws, ws_bytes, coda_linear_residual_workspace_size(M, N, K)));
  if (M == 0) return CODA_OK;
  CK(req(X));
  CK(req(W));
  CK(req(Y));
  if ((gamma_next == nullptr) != (U_out == nullptr)) return CODA_ERR_INVALID_ARG;
  for (const void* q : {(const void*)X, (const void*)W, (const void*)R, (const void*)Y, (const void*)rstd_out,
                        (const void*)gamma_next, (const void*)U_out})
    CK(al(q));
  WsCursor w(ws);
  float* part = w.take<float>(static_cast<size_t>(cdiv(N, BN)) * M);
  Plan p;
  p.A = X;
  p.lda = K;
  p.B = W;
  p.ldb = K;
  p.M = M;
  p.N = N;
  p.K = K;
  p.e.D = Y;
  p.e.ldd = N;
  p.e.aux0 = BF(R);
  p.e.ld_aux0 = N;
  if (rstd_out) {
    p.e.partials = part;
    p.e.ld_part = M;
  }
  if (U_out) {  // U = Y ⊙ gamma_next: the next RMSNorm-reparameterised GEMM's input
    p.e.out1 = BF(U_out);
    p.e.ld_out1 = N;
    p.e.col_scale2 = gamma_next;
  }
  CK(run(p, static_cast<int*>(ws), S(stream)));
  if (rstd_out)
    CU(coda::launch_combine_rows(part, M, static_cast<int>(cdiv(N, BN)), M, 1.f / static_cast<float>(N), eps,
                                 nullptr, rstd_out, 0, S(stream)));
  return CODA_OK;
}

size_t coda_linear_residual_bwd_workspace_size(int64_t, int64_t, int64_t) { return WS_HEADER; }

int coda_linear_residual_bwd(const coda_bf16* dY, const coda_bf16* X, const coda_bf16* W, coda_bf16* dX,
                             coda_bf16* dW, int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes,
                             coda_stream stream) {
  CK(dims_ok(M, N, K));
  CK(ws_ok(ws, ws_bytes, WS_HEADER));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)dY, (const void*)X, (const void*)W, (const void*)dX, (const void*)dW}) {
    CK(req(q));
    CK(al(q));
  }
  int* status = static_cast<int*>(ws);
  {  // dX = dY W
    Plan p;
    p.A = dY;
    p.lda = N;
    p.B = W;
    p.ldb = K;
    p.b_mn = 1;
    p.M = M;
    p.N = K;
    p.K = N;
    p.e.D = dX;
    p.e.ldd = K;
    CK(run(p, status, S(stream)));
  }
  {  // dW = dY^T X
    Plan p;
    p.A = dY;
    p.lda = N;
    p.a_mn = 1;
    p.B = X;
    p.ldb = K;
    p.b_mn = 1;
    p.M = N;
    p.N = K;
    p.K = M;
    p.e.D = dW;
    p.e.ldd = K;
    CK(run(p, status, S(stream)));
  }
  return CODA_OK;
}

// ------------------------------------------------------------------ linear_swiglu
size_t coda_linear_swiglu_workspace_size(int64_t, int64_t, int64_t) { return WS_HEADER; }

int coda_linear_swiglu(const coda_bf16* X, const float* rstd, const coda_bf16* Wg, const coda_bf16* Wu,
                       coda_bf16* H, coda_bf16* g_save, coda_bf16* u_save, int64_t M, int64_t I, int64_t K,
                       void* ws, size_t ws_bytes, coda_stream stream) {
  CK(dims_ok(M, I, K));
  CK(ws_ok(ws, ws_bytes, WS_HEADER));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)X, (const void*)Wg, (const void*)Wu, (const void*)H}) CK(req(q));
  for (const void* q : {(const void*)X, (const void*)rstd, (const void*)Wg, (const void*)Wu, (const void*)H,
                        (const void*)g_save, (const void*)u_save})
    CK(al(q));
  Plan p;
  p.kind = coda::EpiKind::Swiglu;
  p.A = X;
  p.lda = K;
  p.B = Wg;
  p.ldb = K;
  p.B2 = Wu;
  p.ldb2 = K;
  p.b_dual = 1;
  p.M = M;
  p.N = I;
  p.K = K;
  p.e.D = H;
  p.e.ldd = I;
  p.e.row_scale = rstd;
  p.e.out1 = BF(g_save);
  p.e.ld_out1 = I;
  p.e.out2 = BF(u_save);
  p.e.ld_out2 = I;
  return run(p, static_cast<int*>(ws), S(stream));
}

size_t coda_linear_swiglu_bwd_workspace_size(int64_t M, int64_t I, int64_t K) {
  SizeCursor c;
  c.take<__nv_bfloat16>(static_cast<size_t>(M) * 2 * I);      // G' = [r dG | r dU]
  c.take<float>(static_cast<size_t>(cdiv(I, BN)) * M);        // row partials of sum(dG g + dU u)
  c.take<float>(M);                                            // coef
  c.take<float>(static_cast<size_t>(4 * cdiv(M, 128)) * K);   // dgamma partials per (token block, warp)
  return c.off;
}

int coda_linear_swiglu_bwd(const coda_bf16* dY, const coda_bf16* X, const float* rstd, const float* gamma,
                           const coda_bf16* Wg, const coda_bf16* Wu,
                           const coda_bf16* Wd, const coda_bf16* g, const coda_bf16* u, const coda_bf16* H,
                           const coda_bf16* dX_resid, coda_bf16* dX, coda_bf16* dWg, coda_bf16* dWu, coda_bf16* dWd,
                           float* dgamma, int64_t M, int64_t I, int64_t K, void* ws, size_t ws_bytes,
                           coda_stream stream, coda_stream side_stream) {
  CK(dims_ok(M, I, K));
  CK(ws_ok(ws, ws_bytes, coda_linear_swiglu_bwd_workspace_size(M, I, K)));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)dY, (const void*)X, (const void*)Wg, (const void*)Wu, (const void*)Wd,
                        (const void*)g, (const void*)u, (const void*)H, (const void*)dX, (const void*)dWg,
                        (const void*)dWu, (const void*)dWd})
    CK(req(q));
  for (const void* q : {(const void*)dY, (const void*)X, (const void*)rstd, (const void*)gamma, (const void*)Wg,
                        (const void*)Wu, (const void*)Wd, (const void*)g, (const void*)u, (const void*)H,
                        (const void*)dX_resid, (const void*)dX, (const void*)dWg, (const void*)dWu, (const void*)dWd,
                        (const void*)dgamma})
    CK(al(q));
  const bool norm = rstd != nullptr;
  if (norm && (!gamma || !dgamma)) return CODA_ERR_INVALID_ARG;
  WsCursor w(ws);
  __nv_bfloat16* Gp = w.take<__nv_bfloat16>(static_cast<size_t>(M) * 2 * I);
  float* spart = w.take<float>(static_cast<size_t>(cdiv(I, BN)) * M);
  float* coef = w.take<float>(M);
  const int64_t ntb = cdiv(M, 128);
  float* dgp = w.take<float>(static_cast<size_t>(4 * ntb) * K);
  int* status = static_cast<int*>(ws);
  cudaStream_t s = S(stream);
  // With a side stream the weight gradients run beside the dX chain:
  //   stream:  dH -> dSwiGLU (G') -> c -> dX
  //   side:    dWd,  then (after G') dWg, dWu
  // so each persistent GEMM's last, partly filled wave overlaps the other
  // chain's next GEMM.  They share only the status word (atomic OR).
  cudaStream_t s2 = side_stream ? S(side_stream) : s;
  EventSet ev(s2 != s ? 3 : 0);
  if (!ev.ok()) return CODA_ERR_CUDA;
  if (s2 != s) {
    CU(cudaEventRecord(ev[0], s));
    CU(cudaStreamWaitEvent(s2, ev[0], 0));
  }
  {  // dH = dY Wd  ->  dSwiGLU  ->  G' (+ row partials)
    Plan p;
    p.kind = coda::EpiKind::DSwiglu;
    p.A = dY;
    p.lda = K;
    p.B = Wd;
    p.ldb = I;
    p.b_mn = 1;
    p.M = M;
    p.N = I;
    p.K = K;
    p.e.aux0 = BF(g);
    p.e.ld_aux0 = I;
    p.e.aux1 = BF(u);
    p.e.ld_aux1 = I;
    p.e.out1 = Gp;
    p.e.ld_out1 = 2 * I;
    p.e.out2 = Gp + I;
    p.e.ld_out2 = 2 * I;
    p.e.row_scale = rstd;
    if (norm) {
      p.e.partials = spart;
      p.e.ld_part = M;
    }
    CK(run(p, status, s));
  }
  if (s2 != s) CU(cudaEventRecord(ev[1], s));
  {  // dWd = dY^T H (needs neither G' nor c)
    Plan p;
    p.A = dY;
    p.lda = K;
    p.a_mn = 1;
    p.B = H;
    p.ldb = I;
    p.b_mn = 1;
    p.M = K;
    p.N = I;
    p.K = M;
    p.e.D = dWd;
    p.e.ldd = I;
    CK(run(p, status, s2));
  }
  if (norm)
    CU(coda::launch_combine_rows(spart, M, static_cast<int>(cdiv(I, BN)), M, 1.f / static_cast<float>(K), 0.f,
                                 rstd, coef, 1, s));
  {  // D = G'_g Wg + G'_u Wu (one GEMM over K = 2I);  dX = gamma D - c X + dX_resid
     // with the dgamma column partials sum_i X_ik D_ik  (without RMSNorm: D + dX_resid)
    Plan p;
    p.kind = norm ? coda::EpiKind::RmsDx : coda::EpiKind::Plain;
    p.A = Gp;
    p.lda = 2 * I;
    p.B = Wg;
    p.ldb = K;
    p.b_mn = 1;
    p.A2 = Gp + I;
    p.lda2 = 2 * I;
    p.B2 = Wu;
    p.ldb2 = K;
    p.K2 = I;
    p.M = M;
    p.N = K;
    p.K = I;
    p.e.D = dX;
    p.e.ldd = K;
    p.e.aux0 = BF(dX_resid);
    p.e.ld_aux0 = K;
    if (norm) {
      p.e.row_coef = coef;
      p.e.aux1 = BF(X);
      p.e.ld_aux1 = K;
      p.e.col_scale = gamma;
      p.e.partials = dgp;
      p.e.ld_part = K;
    }
    CK(run(p, status, s));
  }
  if (s2 != s) CU(cudaStreamWaitEvent(s2, ev[1], 0));
  for (int which = 0; which < 2; ++which) {  // dWg, dWu = (G'^T X) diag(gamma)
    Plan p;
    p.A = Gp + which * I;
    p.lda = 2 * I;
    p.a_mn = 1;
    p.B = X;
    p.ldb = K;
    p.b_mn = 1;
    p.M = I;
    p.N = K;
    p.K = M;
    p.e.D = which ? dWu : dWg;
    p.e.ldd = K;
    p.e.col_scale = gamma;  // NULL without RMSNorm
    CK(run(p, status, s2));
  }
  if (s2 != s) {
    CU(cudaEventRecord(ev[2], s2));
    CU(cudaStreamWaitEvent(s, ev[2], 0));
  }
  if (norm) CU(coda::launch_colsum(dgp, 4 * ntb, K, K, dgamma, s));
  return CODA_OK;
}

// ------------------------------------------------------------------ linear_qknorm_rope
size_t coda_linear_qknorm_rope_workspace_size(int64_t, int64_t, int32_t, int32_t, int32_t) { return WS_HEADER; }

int coda_linear_qknorm_rope(const coda_bf16* X, const float* rstd, const coda_bf16* W, const float* gamma_q,
                            const float* gamma_k, const int32_t* pos, const float* cos_sin, int32_t max_pos,
                            float eps, int32_t n_q, int32_t n_kv, int32_t head_dim, int32_t rope_pairing,
                            coda_bf16* Q, coda_bf16* K,
                            coda_bf16* V, coda_bf16* qk_save, int64_t M, int64_t Kdim, void* ws, size_t ws_bytes,
                            coda_stream stream) {
  if (head_dim != 128) return CODA_ERR_UNSUPPORTED;
  if (n_q <= 0 || n_kv < 0) return CODA_ERR_INVALID_ARG;
  const int64_t N = static_cast<int64_t>(n_q + 2 * n_kv) * head_dim;
  CK(dims_ok(M, N, Kdim));
  CK(ws_ok(ws, ws_bytes, WS_HEADER));
  if (M == 0) return CODA_OK;
  coda_epilogue_desc d;
  std::memset(&d, 0, sizeof(d));
  d.map = CODA_MAP_QKNORM_ROPE;
  d.row_scale = rstd;
  d.aux_out[0] = qk_save;
  d.ld_aux_out[0] = static_cast<int64_t>(n_q + n_kv) * head_dim;
  d.positions = pos;
  d.cos_sin = cos_sin;
  d.max_pos = max_pos;
  d.n_q_heads = n_q;
  d.n_kv_heads = n_kv;
  d.head_dim = head_dim;
  d.rope_pairing = rope_pairing;
  d.eps = eps;
  d.gamma_q = gamma_q;
  d.gamma_k = gamma_k;
  d.Q = Q;
  d.K = K;
  d.V = V;
  CK(req(X));
  CK(req(W));
  CK(al(rstd));
  return coda_gemm_epilogue(&d, X, Kdim, CODA_K_MAJOR, W, Kdim, CODA_K_MAJOR, nullptr, N, CODA_BF16, M, N,
                            Kdim, ws, ws_bytes, stream);
}

// The QK backward map stages rows by bulk copies (default); CODA_QK_TMA=0
// in the environment selects the register-staged map (for comparisons).
static bool qk_tma_enabled() {
  static const bool v = [] {
    const char* e = std::getenv("CODA_QK_TMA");
    return !(e && e[0] == '0');
  }();
  return v;
}

static int qk_bwd_blocks(int64_t M) {
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cdiv(M, coda::QK_BWD_WARPS), 1184)));
}

// The per-head map of the QK-norm + RoPE backward into G' = r ⊙ [dq | dk | dv]
// (bf16 [M, N]); with coef it also writes the input RMSNorm's row coefficient
// c.  Token rows are staged by bulk copies (one block per SM) unless a row's
// tensors are too large for the shared-memory ring.  Then dgamma_q | dgamma_k
// from the blocks' partials (dgqk, nblk x 256).
static int qk_bwd_map(const coda_bf16* dQ, const coda_bf16* dK, const coda_bf16* dV, const coda_bf16* qk_save,
                      const coda_bf16* V, const float* gamma_q, const float* gamma_k, const int32_t* pos,
                      const float* cos_sin, int32_t max_pos, float eps, int32_t n_q, int32_t n_kv,
                      int32_t rope_pairing, const float* rstd, int64_t M, int64_t Kdim, __nv_bfloat16* Gp,
                      float* coef, float* dgqk, int nblk, float* dgamma_q, float* dgamma_k, int sms, int* status,
                      cudaStream_t s) {
  int nmap = nblk;
  if (qk_tma_enabled() && coda::qk_bwd_tma_stages(n_q, n_kv) > 0) {
    nmap = std::min(nblk, sms);
    CU(coda::launch_qk_bwd_tma(BF(dQ), BF(dK), BF(dV), BF(qk_save), BF(V), gamma_q, gamma_k, pos,
                               reinterpret_cast<const float2*>(cos_sin), max_pos, eps, n_q, n_kv, rstd, M,
                               1.f / static_cast<float>(Kdim), Gp, coef, dgqk, nmap, status, s,
                               rope_pairing == CODA_ROPE_HALF, TIMEOUT_NS));
  } else {
    CU(coda::launch_qk_bwd(BF(dQ), BF(dK), BF(dV), BF(qk_save), BF(V), gamma_q, gamma_k, pos,
                           reinterpret_cast<const float2*>(cos_sin), max_pos, eps, n_q, n_kv, rstd, M,
                           1.f / static_cast<float>(Kdim), Gp, coef, dgqk, nblk, status, s,
                           rope_pairing == CODA_ROPE_HALF));
  }
  CU(coda::launch_colsum(dgqk, nmap, 256, 256, dgamma_q, s, 128, dgamma_k));
  return CODA_OK;
}

size_t coda_linear_qknorm_rope_bwd_workspace_size(int64_t M, int64_t Kdim, int32_t n_q, int32_t n_kv,
                                                  int32_t head_dim) {
  const int64_t N = static_cast<int64_t>(n_q + 2 * n_kv) * head_dim;
  SizeCursor c;
  c.take<__nv_bfloat16>(static_cast<size_t>(M) * N);          // G'
  c.take<float>(M);                                           // coef
  c.take<float>(static_cast<size_t>(qk_bwd_blocks(M)) * 256);  // dgamma_q|k partials
  c.take<float>(static_cast<size_t>(4 * cdiv(M, 128)) * Kdim);  // dgamma_in partials per (token block, warp)
  return c.off;
}

int coda_linear_qknorm_rope_bwd(const coda_bf16* dQ, const coda_bf16* dK, const coda_bf16* dV,
                                const coda_bf16* qk_save, const coda_bf16* V, const float* gamma_q,
                                const float* gamma_k, const int32_t* pos, const float* cos_sin, int32_t max_pos,
                                float eps, int32_t n_q, int32_t n_kv, int32_t head_dim, int32_t rope_pairing,
                                const coda_bf16* X,
                                const float* rstd, const float* gamma_in, const coda_bf16* W_qkv,
                                const coda_bf16* dX_resid, coda_bf16* dX, coda_bf16* dW_qkv,
                                float* dgamma_in, float* dgamma_q, float* dgamma_k, int64_t M, int64_t Kdim, void* ws,
                                size_t ws_bytes, coda_stream stream) {
  if (head_dim != 128) return CODA_ERR_UNSUPPORTED;
  if (n_q <= 0 || n_kv <= 0 || max_pos <= 0) return CODA_ERR_INVALID_ARG;
  if (rope_pairing != CODA_ROPE_INTERLEAVED && rope_pairing != CODA_ROPE_HALF) return CODA_ERR_INVALID_ARG;
  const int64_t N = static_cast<int64_t>(n_q + 2 * n_kv) * head_dim;
  CK(dims_ok(M, N, Kdim));
  CK(ws_ok(ws, ws_bytes, coda_linear_qknorm_rope_bwd_workspace_size(M, Kdim, n_q, n_kv, head_dim)));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)dQ, (const void*)dK, (const void*)dV, (const void*)qk_save, (const void*)V,
                        (const void*)gamma_q, (const void*)gamma_k, (const void*)pos, (const void*)cos_sin,
                        (const void*)X, (const void*)W_qkv, (const void*)dX, (const void*)dW_qkv,
                        (const void*)dgamma_q, (const void*)dgamma_k})
    CK(req(q));
  for (const void* q : {(const void*)dQ, (const void*)dK, (const void*)dV, (const void*)qk_save, (const void*)V,
                        (const void*)gamma_q, (const void*)gamma_k, (const void*)cos_sin, (const void*)X,
                        (const void*)rstd, (const void*)gamma_in, (const void*)W_qkv, (const void*)dX_resid,
                        (const void*)dX, (const void*)dW_qkv, (const void*)dgamma_in, (const void*)dgamma_q,
                        (const void*)dgamma_k})
    CK(al(q));
  const bool norm = rstd != nullptr;
  if (norm && (!gamma_in || !dgamma_in)) return CODA_ERR_INVALID_ARG;
  const int sms = num_sms();
  if (sms <= 0) return CODA_ERR_CUDA;
  WsCursor w(ws);
  __nv_bfloat16* Gp = w.take<__nv_bfloat16>(static_cast<size_t>(M) * N);
  float* coef = w.take<float>(M);
  const int nblk = qk_bwd_blocks(M);
  float* dgqk = w.take<float>(static_cast<size_t>(nblk) * 256);
  const int64_t ntb = cdiv(M, 128);
  float* dgp = w.take<float>(static_cast<size_t>(4 * ntb) * Kdim);
  int* status = static_cast<int*>(ws);
  cudaStream_t s = S(stream);
  CK(qk_bwd_map(dQ, dK, dV, qk_save, V, gamma_q, gamma_k, pos, cos_sin, max_pos, eps, n_q, n_kv, rope_pairing, rstd,
                M, Kdim, Gp, norm ? coef : nullptr, dgqk, nblk, dgamma_q, dgamma_k, sms, status, s));
  {  // D = G' W_qkv;  dX = gamma_in D - c X + dX_resid with the dgamma_in column
     // partials sum_i X_ik D_ik  (without RMSNorm: D + dX_resid)
    Plan p;
    p.kind = norm ? coda::EpiKind::RmsDx : coda::EpiKind::Plain;
    p.A = Gp;
    p.lda = N;
    p.B = W_qkv;
    p.ldb = Kdim;
    p.b_mn = 1;
    p.M = M;
    p.N = Kdim;
    p.K = N;
    p.e.D = dX;
    p.e.ldd = Kdim;
    p.e.aux0 = BF(dX_resid);
    p.e.ld_aux0 = Kdim;
    if (norm) {
      p.e.row_coef = coef;
      p.e.aux1 = BF(X);
      p.e.ld_aux1 = Kdim;
      p.e.col_scale = gamma_in;
      p.e.partials = dgp;
      p.e.ld_part = Kdim;
    }
    CK(run(p, status, s));
  }
  {  // dW_qkv = (G'^T X) diag(gamma_in)
    Plan p;
    p.A = Gp;
    p.lda = N;
    p.a_mn = 1;
    p.B = X;
    p.ldb = Kdim;
    p.b_mn = 1;
    p.M = N;
    p.N = Kdim;
    p.K = M;
    p.e.D = dW_qkv;
    p.e.ldd = Kdim;
    p.e.col_scale = gamma_in;  // NULL without RMSNorm
    CK(run(p, status, s));
  }
  if (norm) CU(coda::launch_colsum(dgp, 4 * ntb, Kdim, Kdim, dgamma_in, s));
  return CODA_OK;
}

// ------------------------------------------------------------------ linear_cross_entropy
static int ce_chunks(int64_t V) { return static_cast<int>(cdiv(cdiv(V, BN), CE_TILES_PER_UNIT)); }
static int ce_blocks(int64_t M) {
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cdiv(M, coda::CE_COMBINE_THREADS), 256)));
}

size_t coda_linear_cross_entropy_workspace_size(int64_t M, int64_t V, int64_t) {
  SizeCursor c;
  c.take<float>(M);                                               // target logits
  c.take<float2>(static_cast<size_t>(ce_chunks(V)) * M);          // (max, sumexp) partials
  c.take<double>(ce_blocks(M));
  c.take<int>(ce_blocks(M));
  return c.off;
}

}  // extern "C"

// Linear + cross-entropy forward; `rstd` (optional) scales each row's logits
// (the final RMSNorm folded into the head).
// With fp8 set, X and W are e4m3 codes with per-row scales sx, sw.
static int ce_forward(const coda_bf16* X, const coda_bf16* W, const int32_t* labels, int32_t ignore_index,
                      const float* rstd, float* loss_mean, float* lse, int32_t* n_valid, int64_t M, int64_t V,
                      int64_t K, void* ws, size_t ws_bytes, coda_stream stream, int fp8 = 0,
                      const float* sx = nullptr, const float* sw = nullptr) {
  CK(dims_ok(M, V, K));
  CK(ws_ok(ws, ws_bytes, coda_linear_cross_entropy_workspace_size(M, V, K)));
  CK(req(loss_mean));
  CK(req(n_valid));
  if (M > 0)  // with no rows only the mean (NaN) and the count (0) are written
    for (const void* q : {(const void*)X, (const void*)W, (const void*)labels, (const void*)lse}) CK(req(q));
  CK(al(X));
  CK(al(W));
  if (V == 0) return CODA_ERR_INVALID_ARG;
  WsCursor w(ws);
  float* target = w.take<float>(M);
  const int nch = ce_chunks(V);
  float2* part = w.take<float2>(static_cast<size_t>(nch) * M);
  const int nblk = ce_blocks(M);
  double* bl = w.take<double>(nblk);
  int* bc = w.take<int>(nblk);
  int* status = static_cast<int*>(ws);
  cudaStream_t s = S(stream);
  if (M > 0) {
    Plan p;
    p.kind = coda::EpiKind::CeLse;
    p.A = X;
    p.lda = K;
    p.B = W;
    p.ldb = K;
    p.M = M;
    p.N = V;
    p.K = K;
    p.n_per_unit = CE_TILES_PER_UNIT;
    p.fp8 = fp8;
    p.e.acc_rs = sx;
    p.e.acc_cs = sw;
    p.e.row_scale = rstd;
    p.e.labels = labels;
    p.e.target_logit = target;
    p.e.partials = reinterpret_cast<float*>(part);
    p.e.ld_part = M;
    CK(run(p, status, s));
  }
  CU(coda::launch_ce_combine(part, M, nch, target, labels, ignore_index, M, V, lse, bl, bc, nblk, loss_mean, n_valid,
                             status, s));
  return CODA_OK;
}

// One NVFP4 GEMM launch: 128 x 256 tiles (b_dual: 128 gate + 128 up
// columns), k-slices of 256 elements; single CTAs, or clusters of cg CTAs
// on adjacent row blocks that each copy 256 / cg rows of the B tile.
int run_nvfp4(coda::EpiKind kind, const uint8_t* A, const uint8_t* B0, const uint8_t* B1, coda::Nvfp4Scales sc,
              int64_t M, int64_t N, int64_t K, int b_dual, const EpiArgs& e, int* status, cudaStream_t s) {
  if (M == 0 || N == 0) return CODA_OK;
  if (!get_encoder()) return CODA_ERR_CUDA;
  const int sms = num_sms();
  if (sms <= 0) return CODA_ERR_CUDA;
  if (coda::nvfp4_pairs(M)) {
    // CTA pairs: each CTA copies its own 128 rows of A and of B; the block
    // scales through byte maps of 256-byte rows (an 8-row box = one 2 KB group)
    CUtensorMap maps[6];
    std::memset(maps, 0, sizeof(maps));
    const int64_t kbytes = K / 2;
    auto sf_map = [&](CUtensorMap* m, const uint8_t* sf, int64_t rows) {
      const int64_t bytes = static_cast<int64_t>(coda_nvfp4_scale_bytes(rows, K));
      return encode_map_plain(m, sf, bytes / 256, 256, 256, 8);
    };
    if (!encode_map(&maps[0], A, M, kbytes, kbytes, 128, coda::BM, 1)) return CODA_ERR_CUDA;
    if (!encode_map(&maps[1], B0, N, kbytes, kbytes, 128, BN / 2, 1)) return CODA_ERR_CUDA;
    if (!encode_map(&maps[2], b_dual ? B1 : B0, N, kbytes, kbytes, 128, BN / 2, 1)) return CODA_ERR_CUDA;
    if (!sf_map(&maps[3], sc.a, M)) return CODA_ERR_CUDA;
    if (!sf_map(&maps[4], sc.b0, N)) return CODA_ERR_CUDA;
    if (!sf_map(&maps[5], b_dual ? sc.b1 : sc.b0, N)) return CODA_ERR_CUDA;
    GemmArgs a{};
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.num_m = static_cast<int>(cdiv(M, 2 * coda::BM));
    a.num_n = static_cast<int>(cdiv(N, b_dual ? BN / 2 : BN));
    a.kb0 = static_cast<int>(cdiv(K, 256));
    a.b_dual = b_dual;
    a.n_per_unit = 1;
    a.num_units = a.num_m * a.num_n;
    a.group_m = group_m(2);
    a.idesc = coda::nvfp4_idesc_pair();
    a.status = status;
    a.timeout_ns = TIMEOUT_NS;
    wait_sleep(a.producer_sleep_ns, a.epilogue_sleep_ns);
    a.e = e;
    a.e.st_stream = stream_stores(M * N * 2 * (1 + (e.out1 != nullptr) + (e.out2 != nullptr)));
    sc.kt = cdiv(K, 256);
    const cudaError_t err = coda::launch_gemm_nvfp4_pair(kind == coda::EpiKind::Swiglu ? 1 : 0, a.num_units, sms,
                                                         s, maps, a, sc);
    return err == cudaSuccess ? CODA_OK : CODA_ERR_CUDA;
  }
  const int cg = coda::nvfp4_cluster_size(M);
  // rows of one B copy: the whole tile (256, or 128 per weight when dual),
  // or a quarter of it when four CTAs share the tile
  const uint32_t b_rows = cg > 1 ? BN / cg : (b_dual ? BN / 2 : BN);
  CUtensorMap maps[3];
  std::memset(maps, 0, sizeof(maps));
  const int64_t kb = K / 2;  // bytes of codes per row
  if (!encode_map(&maps[0], A, M, kb, kb, 128, coda::BM, 1)) return CODA_ERR_CUDA;
  if (!encode_map(&maps[1], B0, N, kb, kb, 128, b_rows, 1)) return CODA_ERR_CUDA;
  if (b_dual) {
    if (!encode_map(&maps[2], B1, N, kb, kb, 128, b_rows, 1)) return CODA_ERR_CUDA;
  } else {
    maps[2] = maps[1];
  }
  GemmArgs a{};
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.num_m = static_cast<int>(cdiv(M, static_cast<int64_t>(cg) * coda::BM));
  a.num_n = static_cast<int>(cdiv(N, b_dual ? BN / 2 : BN));
  a.kb0 = static_cast<int>(cdiv(K, 256));
  a.b_dual = b_dual;
  a.n_per_unit = 1;
  a.num_units = a.num_m * a.num_n;
  a.group_m = group_m(cg);
  a.idesc = coda::nvfp4_idesc();
  a.status = status;
  a.timeout_ns = TIMEOUT_NS;
  wait_sleep(a.producer_sleep_ns, a.epilogue_sleep_ns);
  a.e = e;
  a.e.st_stream = stream_stores(M * N * 2 * (1 + (e.out1 != nullptr) + (e.out2 != nullptr)));
  sc.kt = cdiv(K, 256);
  cudaError_t err = kind == coda::EpiKind::Swiglu
                        ? coda::launch_gemm_swiglu_nvfp4(cg, a.num_units, sms, s, maps, a, sc)
                        : coda::launch_gemm_plain_nvfp4(cg, a.num_units, sms, s, maps, a, sc);
  return err == cudaSuccess ? CODA_OK : CODA_ERR_CUDA;
}

namespace {

// ------------------------------------------------------------------ cross-entropy backward, by vocabulary slice
// The backward never holds the gradient of the whole logit matrix: the
// vocabulary is cut into slices of CE_SLICE columns, and for each slice s
//   dZ_s = softmax part of (softmax - onehot) * w   (recomputed z; bf16)
//   dX  += dZ_s W_s                                  (fp32 running sum)
//   dW_s = dZ_s^T X                                  (its rows of dW)
// The one-hot terms (-w_i W[y_i] for dX, -sum_{i: y_i = v} w_i X[i] for dW)
// are applied exactly in fp32 in the epilogues; the last slice's dX GEMM adds
// the running sum and writes bf16.  dZ_s is double-buffered: slice s + 1's
// logits GEMM runs on the caller's stream while slice s's dX and dW GEMMs run
// on two helper streams, so the launches' partly filled last waves overlap.
// With the final RMSNorm folded into the head (rstd set) the stored dZ is
// row-scaled, each slice's epilogue also emits the row partials sum p z and
// the target logit for the RMSNorm-backward coefficient c_i, the last dX GEMM
// subtracts c_i X_i and adds the residual-stream gradient, and dW is scaled
// by gamma while its epilogue reduces W dW' over rows into dgamma partials.
constexpr int64_t CE_SLICE = 16384;  // vocabulary columns per slice (64 tiles)

int64_t ce_slice_cols(int64_t V) { return std::min<int64_t>(V, CE_SLICE); }

size_t ce_bwd_workspace(int64_t M, int64_t V, int64_t K, bool rms) {
  const int64_t sl = ce_slice_cols(V);
  const int64_t nsl = sl > 0 ? cdiv(V, sl) : 0;
  SizeCursor c;
  c.take<__nv_bfloat16>(static_cast<size_t>(M) * sl);      // dZ_s, buffer 0
  if (nsl > 1) {
    c.take<__nv_bfloat16>(static_cast<size_t>(M) * sl);    // dZ_s, buffer 1
    c.take<float>(static_cast<size_t>(M) * K);             // running dX (fp32)
  }
  c.take<float>(M);                                        // w_i (r_i w_i with rstd)
  c.take<int32_t>(M);                                      // label of valid rows
  c.take<int32_t>(V);                                      // counts per vocabulary row
  c.take<int32_t>(V);                                      // scatter cursors
  c.take<int32_t>(V + 1);                                  // CSR offsets
  c.take<int32_t>(M);                                      // CSR token indices
  if (rms) {
    c.take<float>(static_cast<size_t>(cdiv(V, BN)) * M);   // row partials sum p z
    c.take<float>(M);                                      // target logits
    c.take<float>(M);                                      // RMSNorm coefficient c
    c.take<float>(static_cast<size_t>(4 * cdiv(V, 128)) * K);  // dgamma partials
  }
  return c.off;
}

struct CeBwd {
  // e4m3 operands of the logits GEMM (Xq [M, K], Wq [V, K] codes with per-row
  // scales sx, sw), or null: the logits come from X, W
  const uint8_t* Xq = nullptr;
  const float* sx = nullptr;
  const uint8_t* Wq = nullptr;
  const float* sw = nullptr;
  const coda_bf16* X = nullptr;
  const coda_bf16* W = nullptr;      // the weight the logits GEMM reads (gamma-folded with rstd)
  const coda_bf16* W_raw = nullptr;  // rstd: the unfolded weight (dgamma partials)
  const float* rstd = nullptr;       // final RMSNorm folded into the head
  const float* gamma = nullptr;
  const int32_t* labels = nullptr;
  int32_t ignore_index = -100;
  const float* lse = nullptr;
  const int32_t* n_valid = nullptr;
  float dloss = 1.f;
  const coda_bf16* dX_resid = nullptr;
  coda_bf16* dX = nullptr;
  coda_bf16* dW = nullptr;
  float* dgamma = nullptr;
  int64_t M = 0, V = 0, K = 0;
};

int ce_backward(const CeBwd& a, void* ws, cudaStream_t s) {
  const int64_t M = a.M, V = a.V, K = a.K;
  const bool rms = a.rstd != nullptr;
  const int64_t sl = ce_slice_cols(V);
  const int nsl = static_cast<int>(cdiv(V, sl));
  WsCursor w(ws);
  __nv_bfloat16* dZ[2];
  dZ[0] = w.take<__nv_bfloat16>(static_cast<size_t>(M) * sl);
  dZ[1] = dZ[0];
  float* acc = nullptr;
  if (nsl > 1) {
    dZ[1] = w.take<__nv_bfloat16>(static_cast<size_t>(M) * sl);
    acc = w.take<float>(static_cast<size_t>(M) * K);
  }
  float* wrow = w.take<float>(M);
  int32_t* lrow = w.take<int32_t>(M);
  int32_t* counts = w.take<int32_t>(V);
  int32_t* cursor = w.take<int32_t>(V);
  int32_t* off = w.take<int32_t>(V + 1);
  int32_t* idx = w.take<int32_t>(M);
  float *pz = nullptr, *target = nullptr, *coef = nullptr, *dgp = nullptr;
  const int ntile = static_cast<int>(cdiv(V, BN));
  const int64_t nmb = cdiv(V, 128);
  if (rms) {
    pz = w.take<float>(static_cast<size_t>(ntile) * M);
    target = w.take<float>(M);
    coef = w.take<float>(M);
    dgp = w.take<float>(static_cast<size_t>(4 * nmb) * K);
  }
  int* status = static_cast<int*>(ws);
  CU(coda::launch_ce_onehot_prep(a.labels, a.ignore_index, M, V, a.n_valid, a.dloss, a.rstd, wrow, lrow, counts,
                                 cursor, off, idx, s));
  // helper streams for the dX and dW GEMMs; without them everything stays on s
  cudaStream_t sx = side_stream(s, 1), sw = side_stream(s, 2);
  if (!sx || !sw) sx = sw = s;
  const bool conc = sx != s;
  // events: 0 fork, 1-2 slice logits ready (per buffer), 3-4 dX done, 5-6 dW
  // done, 7 RMSNorm coefficient ready
  EventSet ev(8);
  if (!ev.ok()) return CODA_ERR_CUDA;
  if (conc) {
    CU(cudaEventRecord(ev[0], s));
    CU(cudaStreamWaitEvent(sx, ev[0], 0));
    CU(cudaStreamWaitEvent(sw, ev[0], 0));
  }
  for (int i = 0; i < nsl; ++i) {
    const int64_t v0 = static_cast<int64_t>(i) * sl;
    const int64_t vs = std::min<int64_t>(sl, V - v0);
    const int b = i & 1;
    const bool last = i == nsl - 1;
    const coda_bf16* Ws = a.W + v0 * K;
    if (conc && i >= 2) {  // buffer b is free once slice i - 2's dX and dW have read it
      CU(cudaStreamWaitEvent(s, ev[3 + b], 0));
      CU(cudaStreamWaitEvent(s, ev[5 + b], 0));
    }
    {  // dZ_s = softmax(z_s) * w (row-scaled with rstd); z_s recomputed
      Plan p;
      p.kind = coda::EpiKind::CeDlogits;
      p.A = a.X;
      p.lda = K;
      p.B = Ws;
      p.ldb = K;
      if (a.Xq) {  // the logits from the e4m3 operands
        p.fp8 = 1;
        p.A = a.Xq;
        p.B = a.Wq + v0 * K;
        p.e.acc_rs = a.sx;
        p.e.acc_cs = a.sw + v0;
      }
      p.M = M;
      p.N = vs;
      p.K = K;
      p.e.D = dZ[b];
      p.e.ldd = sl;
      p.e.labels = a.labels;
      p.e.ignore_index = a.ignore_index;
      p.e.lse = a.lse;
      p.e.n_valid = a.n_valid;
      p.e.dloss = a.dloss;
      p.e.col_base = v0;
      p.e.n_total = V;
      if (rms) {
        p.e.row_scale = a.rstd;
        p.e.partials = pz + (v0 / BN) * M;
        p.e.ld_part = M;
        p.e.target_logit = target;
      }
      CK(run(p, status, s));
    }
    if (conc) {
      CU(cudaEventRecord(ev[1 + b], s));
      CU(cudaStreamWaitEvent(sx, ev[1 + b], 0));
      CU(cudaStreamWaitEvent(sw, ev[1 + b], 0));
    }
    if (rms && last) {  // c_i from the row partials of every slice
      CU(coda::launch_ce_norm_coef(pz, M, ntile, target, a.rstd, wrow, M, 1.f / static_cast<float>(K), coef, s));
      if (conc) {
        CU(cudaEventRecord(ev[7], s));
        CU(cudaStreamWaitEvent(sx, ev[7], 0));
      }
    }
    {  // dX: running fp32 sum of dZ_s W_s; the last slice writes bf16 with the row terms
      Plan p;
      p.A = dZ[b];
      p.lda = sl;
      p.B = Ws;
      p.ldb = K;
      p.b_mn = 1;
      p.M = M;
      p.N = K;
      p.K = vs;
      p.e.ldd = K;
      if (!last) {
        p.e.D = acc;
        p.e.d_f32 = 1;
        p.e.beta = i > 0;
      } else {
        p.e.D = a.dX;
        p.e.acc_in = i > 0 ? acc : nullptr;
        p.e.ld_acc_in = K;
        p.e.row_coef = wrow;  // - w_i W[y_i] (r_i w_i Wf[y_i] with rstd)
        p.e.aux1 = BF(a.W);
        p.e.ld_aux1 = K;
        p.e.gather_rows = lrow;
        if (rms) {
          p.e.aux0 = BF(a.dX_resid);
          p.e.ld_aux0 = K;
          p.e.row_coef2 = coef;  // - c_i X_i
          p.e.aux3 = BF(a.X);
          p.e.ld_aux3 = K;
        }
      }
      CK(run(p, status, sx));
    }
    {  // dW rows of the slice: dZ_s^T X minus the one-hot rows (CSR of tokens per label)
      Plan p;
      p.A = dZ[b];
      p.lda = sl;
      p.a_mn = 1;
      p.B = a.X;
      p.ldb = K;
      p.b_mn = 1;
      p.M = vs;
      p.N = K;
      p.K = M;
      p.e.D = a.dW + v0 * K;
      p.e.ldd = K;
      p.e.aux2 = BF(a.X);
      p.e.ld_aux2 = K;
      p.e.csr_off = off + v0;
      p.e.csr_idx = idx;
      p.e.csr_w = wrow;
      if (rms) {  // dW = dW' diag(gamma); dgamma partials sum_rows W dW'
        p.kind = coda::EpiKind::ColDot;
        p.e.col_scale = a.gamma;
        p.e.aux0 = BF(a.W_raw + v0 * K);
        p.e.ld_aux0 = K;
        p.e.partials = dgp + (v0 / 128) * 4 * K;
        p.e.ld_part = K;
      }
      CK(run(p, status, sw));
    }
    if (conc) {
      CU(cudaEventRecord(ev[3 + b], sx));
      CU(cudaEventRecord(ev[5 + b], sw));
    }
  }
  if (conc) {  // join: the helper streams' last records cover all their work
    const int b = (nsl - 1) & 1;
    CU(cudaStreamWaitEvent(s, ev[3 + b], 0));
    CU(cudaStreamWaitEvent(s, ev[5 + b], 0));
  }
  if (rms) CU(coda::launch_colsum(dgp, 4 * nmb, K, K, a.dgamma, s));
  return CODA_OK;
}

}  // namespace

extern "C" {

int coda_linear_cross_entropy(const coda_bf16* X, const coda_bf16* W, const int32_t* labels, int32_t ignore_index,
                              float* loss_mean, float* lse, int32_t* n_valid, int64_t M, int64_t V, int64_t K,
                              void* ws, size_t ws_bytes, coda_stream stream) {
  return ce_forward(X, W, labels, ignore_index, nullptr, loss_mean, lse, n_valid, M, V, K, ws, ws_bytes, stream);
}

size_t coda_linear_cross_entropy_bwd_workspace_size(int64_t M, int64_t V, int64_t K) {
  return ce_bwd_workspace(M, V, K, false);
}

int coda_linear_cross_entropy_bwd(const coda_bf16* X, const coda_bf16* W, const int32_t* labels,
                                  int32_t ignore_index, const float* lse, const int32_t* n_valid, float dloss,
                                  coda_bf16* dX, coda_bf16* dW, int64_t M, int64_t V, int64_t K, void* ws,
                                  size_t ws_bytes, coda_stream stream) {
  CK(dims_ok(M, V, K));
  CK(ws_ok(ws, ws_bytes, coda_linear_cross_entropy_bwd_workspace_size(M, V, K)));
  CK(req(dW));
  if (M > 0)  // with no rows dW is zero and nothing else is touched
    for (const void* q : {(const void*)X, (const void*)W, (const void*)labels, (const void*)lse,
                          (const void*)n_valid, (const void*)dX})
      CK(req(q));
  for (const void* q : {(const void*)X, (const void*)W, (const void*)dX, (const void*)dW}) CK(al(q));
  if (V == 0) return CODA_ERR_INVALID_ARG;
  if (M == 0) {
    CU(cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * K * 2, S(stream)));
    return CODA_OK;
  }
  CeBwd a;
  a.X = X;
  a.W = W;
  a.labels = labels;
  a.ignore_index = ignore_index;
  a.lse = lse;
  a.n_valid = n_valid;
  a.dloss = dloss;
  a.dX = dX;
  a.dW = dW;
  a.M = M;
  a.V = V;
  a.K = K;
  return ce_backward(a, ws, S(stream));
}


// ------------------------------------------------------------------ final RMSNorm -> LM head -> CE
size_t coda_rmsnorm_linear_cross_entropy_workspace_size(int64_t M, int64_t V, int64_t K) {
  return coda_linear_cross_entropy_workspace_size(M, V, K);
}

int coda_rmsnorm_linear_cross_entropy(const coda_bf16* X, const float* rstd, const coda_bf16* Wf,
                                      const int32_t* labels, int32_t ignore_index, float* loss_mean, float* lse,
                                      int32_t* n_valid, int64_t M, int64_t V, int64_t K, void* ws, size_t ws_bytes,
                                      coda_stream stream) {
  if (M > 0) CK(req(rstd));
  return ce_forward(X, Wf, labels, ignore_index, rstd, loss_mean, lse, n_valid, M, V, K, ws, ws_bytes, stream);
}

size_t coda_rmsnorm_linear_cross_entropy_bwd_workspace_size(int64_t M, int64_t V, int64_t K) {
  return ce_bwd_workspace(M, V, K, true);
}

int coda_rmsnorm_linear_cross_entropy_bwd(const coda_bf16* X, const float* rstd, const float* gamma,
                                          const coda_bf16* W, const coda_bf16* Wf, const int32_t* labels,
                                          int32_t ignore_index, const float* lse, const int32_t* n_valid, float dloss,
                                          const coda_bf16* dX_resid, coda_bf16* dX, coda_bf16* dW, float* dgamma,
                                          int64_t M, int64_t V, int64_t K, void* ws, size_t ws_bytes,
                                          coda_stream stream) {
  CK(dims_ok(M, V, K));
  CK(ws_ok(ws, ws_bytes, coda_rmsnorm_linear_cross_entropy_bwd_workspace_size(M, V, K)));
  if (V == 0) return CODA_ERR_INVALID_ARG;
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)X, (const void*)rstd, (const void*)gamma, (const void*)W, (const void*)Wf,
                        (const void*)labels, (const void*)lse, (const void*)n_valid, (const void*)dX,
                        (const void*)dW, (const void*)dgamma})
    CK(req(q));
  for (const void* q : {(const void*)X, (const void*)gamma, (const void*)W, (const void*)Wf, (const void*)dX_resid,
                        (const void*)dX, (const void*)dW})
    CK(al(q));
  CeBwd a;
  a.X = X;
  a.W = Wf;
  a.W_raw = W;
  a.rstd = rstd;
  a.gamma = gamma;
  a.labels = labels;
  a.ignore_index = ignore_index;
  a.lse = lse;
  a.n_valid = n_valid;
  a.dloss = dloss;
  a.dX_resid = dX_resid;
  a.dX = dX;
  a.dW = dW;
  a.dgamma = dgamma;
  a.M = M;
  a.V = V;
  a.K = K;
  return ce_backward(a, ws, S(stream));
}


// ------------------------------------------------------------------ linear_sigmoid
size_t coda_linear_sigmoid_workspace_size(int64_t, int64_t, int64_t) { return WS_HEADER; }

int coda_linear_sigmoid(const coda_bf16* X, const coda_bf16* W, const coda_bf16* Z, coda_bf16* Y, int64_t M,
                        int64_t N, int64_t K, void* ws, size_t ws_bytes, coda_stream stream) {
  CK(dims_ok(M, N, K));
  CK(ws_ok(ws, ws_bytes, WS_HEADER));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)X, (const void*)W, (const void*)Y}) CK(req(q));
  for (const void* q : {(const void*)X, (const void*)W, (const void*)Z, (const void*)Y}) CK(al(q));
  Plan p;
  p.kind = coda::EpiKind::Sigmoid;
  p.A = X;
  p.lda = K;
  p.B = W;
  p.ldb = K;
  p.M = M;
  p.N = N;
  p.K = K;
  p.e.D = Y;
  p.e.ldd = N;
  p.e.aux0 = BF(Z);
  p.e.ld_aux0 = N;
  p.e.mode = 0;
  return run(p, static_cast<int*>(ws), S(stream));
}

size_t coda_linear_sigmoid_bwd_workspace_size(int64_t M, int64_t N, int64_t) {
  SizeCursor c;
  c.take<__nv_bfloat16>(static_cast<size_t>(M) * N);  // dz
  return c.off;
}

int coda_linear_sigmoid_bwd(const coda_bf16* dY, const coda_bf16* X, const coda_bf16* W, const coda_bf16* Z,
                            coda_bf16* dX, coda_bf16* dW, coda_bf16* dZ, int64_t M, int64_t N, int64_t K, void* ws,
                            size_t ws_bytes, coda_stream stream) {
  CK(dims_ok(M, N, K));
  CK(ws_ok(ws, ws_bytes, coda_linear_sigmoid_bwd_workspace_size(M, N, K)));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)dY, (const void*)X, (const void*)W, (const void*)dX, (const void*)dW})
    CK(req(q));
  if (Z && !dZ) return CODA_ERR_INVALID_ARG;
  for (const void* q : {(const void*)dY, (const void*)X, (const void*)W, (const void*)Z, (const void*)dX,
                        (const void*)dW, (const void*)dZ})
    CK(al(q));
  WsCursor w(ws);
  __nv_bfloat16* dz = w.take<__nv_bfloat16>(static_cast<size_t>(M) * N);
  int* status = static_cast<int*>(ws);
  cudaStream_t s = S(stream);
  {  // recompute z = X W^T; dz = dY (* Z) * s (1 - s); dZ = dY * s
    Plan p;
    p.kind = coda::EpiKind::Sigmoid;
    p.A = X;
    p.lda = K;
    p.B = W;
    p.ldb = K;
    p.M = M;
    p.N = N;
    p.K = K;
    p.e.aux0 = BF(Z);
    p.e.ld_aux0 = N;
    p.e.aux1 = BF(dY);
    p.e.ld_aux1 = N;
    p.e.out1 = dz;
    p.e.ld_out1 = N;
    p.e.out2 = Z ? BF(dZ) : nullptr;
    p.e.ld_out2 = N;
    p.e.mode = 1;
    CK(run(p, status, s));
  }
  {  // dX = dz W
    Plan p;
    p.A = dz;
    p.lda = N;
    p.B = W;
    p.ldb = K;
    p.b_mn = 1;
    p.M = M;
    p.N = K;
    p.K = N;
    p.e.D = dX;
    p.e.ldd = K;
    CK(run(p, status, s));
  }
  {  // dW = dz^T X
    Plan p;
    p.A = dz;
    p.lda = N;
    p.a_mn = 1;
    p.B = X;
    p.ldb = K;
    p.b_mn = 1;
    p.M = N;
    p.N = K;
    p.K = M;
    p.e.D = dW;
    p.e.ldd = K;
    CK(run(p, status, s));
  }
  return CODA_OK;
}


// ------------------------------------------------------------------ FP8 (e4m3) operands
int coda_quantize_fp8_rows(const coda_bf16* X, int64_t ldx, int64_t M, int64_t K, uint8_t* Xq, float* scale,
                           coda_stream stream) {
  if (M < 0 || K < 0) return CODA_ERR_INVALID_ARG;
  if (K % 16) return CODA_ERR_UNSUPPORTED;  // 16-byte rows for the e4m3 tensor maps
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)X, (const void*)Xq, (const void*)scale}) CK(req(q));
  CK(al(X));
  CK(al(Xq));
  CK(ldok(ldx, K));
  const int sms = num_sms();
  if (sms <= 0) return CODA_ERR_CUDA;
  CU(coda::launch_quantize_fp8_rows(BF(X), ldx, M, K, Xq, K, scale, sms, S(stream)));
  return CODA_OK;
}

size_t coda_linear_fp8_workspace_size(int64_t, int64_t, int64_t) { return WS_HEADER; }

int coda_linear_fp8(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw, const coda_bf16* R,
                    coda_bf16* Y, int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes, coda_stream stream) {
  CK(dims_ok(M, N, K));
  if (K % 16) return CODA_ERR_UNSUPPORTED;
  CK(ws_ok(ws, ws_bytes, WS_HEADER));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)Xq, (const void*)sx, (const void*)Wq, (const void*)sw, (const void*)Y})
    CK(req(q));
  for (const void* q : {(const void*)Xq, (const void*)Wq, (const void*)sw, (const void*)R, (const void*)Y})
    CK(al(q));
  Plan p;
  p.fp8 = 1;
  p.A = Xq;
  p.lda = K;
  p.B = Wq;
  p.ldb = K;
  p.M = M;
  p.N = N;
  p.K = K;
  p.e.D = Y;
  p.e.ldd = N;
  p.e.row_scale = sx;
  p.e.col_scale = sw;
  p.e.aux0 = BF(R);
  p.e.ld_aux0 = N;
  return run(p, static_cast<int*>(ws), S(stream));
}

size_t coda_linear_swiglu_fp8_workspace_size(int64_t, int64_t, int64_t) { return WS_HEADER; }

int coda_linear_swiglu_fp8(const uint8_t* Xq, const float* sx, const float* rstd, const uint8_t* Wgq,
                           const float* sg, const uint8_t* Wuq, const float* su, coda_bf16* H, coda_bf16* g_save,
                           coda_bf16* u_save, int64_t M, int64_t I, int64_t K, void* ws, size_t ws_bytes,
                           coda_stream stream) {
  CK(dims_ok(M, I, K));
  if (K % 16) return CODA_ERR_UNSUPPORTED;
  CK(ws_ok(ws, ws_bytes, WS_HEADER));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)Xq, (const void*)sx, (const void*)Wgq, (const void*)sg, (const void*)Wuq,
                        (const void*)su, (const void*)H})
    CK(req(q));
  for (const void* q : {(const void*)Xq, (const void*)Wgq, (const void*)Wuq, (const void*)sg, (const void*)su,
                        (const void*)H, (const void*)g_save, (const void*)u_save})
    CK(al(q));
  Plan p;
  p.kind = coda::EpiKind::Swiglu;
  p.fp8 = 1;
  p.A = Xq;
  p.lda = K;
  p.B = Wgq;
  p.ldb = K;
  p.B2 = Wuq;
  p.ldb2 = K;
  p.b_dual = 1;
  p.M = M;
  p.N = I;
  p.K = K;
  p.e.D = H;
  p.e.ldd = I;
  p.e.row_scale = sx;
  p.e.row_scale2 = rstd;
  p.e.col_scale = sg;
  p.e.col_scale2 = su;
  p.e.out1 = BF(g_save);
  p.e.ld_out1 = I;
  p.e.out2 = BF(u_save);
  p.e.ld_out2 = I;
  return run(p, static_cast<int*>(ws), S(stream));
}

int coda_quantize_fp8_cols(const coda_bf16* X, int64_t ldx, int64_t R, const coda_bf16* X2, int64_t ldx2,
                           int64_t R2, int64_t C, uint8_t* XTq, int64_t ldo, float* scale, coda_stream stream) {
  if (R < 0 || R2 < 0 || C < 0) return CODA_ERR_INVALID_ARG;
  if (!X2 && R2 > 0) return CODA_ERR_INVALID_ARG;
  const int64_t RT = R + R2;
  if (C % 8 || RT % 16) return CODA_ERR_UNSUPPORTED;  // 16-byte rows of bf16 input and e4m3 output
  if (C == 0 || RT == 0) return CODA_OK;
  for (const void* q : {(const void*)XTq, (const void*)scale}) CK(req(q));
  if (R > 0) {
    CK(req(X));
    CK(ldok(ldx, C));
  }
  if (R2 > 0) CK(ldok(ldx2, C));
  for (const void* q : {(const void*)X, (const void*)X2, (const void*)XTq}) CK(al(q));
  if (ldo < RT || ldo % 16) return ldo < RT ? CODA_ERR_INVALID_ARG : CODA_ERR_ALIGNMENT;
  const int sms = num_sms();
  if (sms <= 0) return CODA_ERR_CUDA;
  CU(coda::launch_quantize_fp8_cols(BF(X), ldx, R, BF(X2), ldx2, R2, C, XTq, ldo, scale, sms, S(stream)));
  return CODA_OK;
}

size_t coda_linear_qknorm_rope_fp8_workspace_size(int64_t, int64_t, int32_t, int32_t, int32_t) { return WS_HEADER; }

int coda_linear_qknorm_rope_fp8(const uint8_t* Xq, const float* sx, const float* rstd, const uint8_t* Wq,
                                const float* sw, const float* gamma_q, const float* gamma_k, const int32_t* pos,
                                const float* cos_sin, int32_t max_pos, float eps, int32_t n_q, int32_t n_kv,
                                int32_t head_dim, int32_t rope_pairing, coda_bf16* Q, coda_bf16* K, coda_bf16* V,
                                coda_bf16* qk_save, int64_t M, int64_t Kdim, void* ws, size_t ws_bytes,
                                coda_stream stream) {
  if (head_dim != 128) return CODA_ERR_UNSUPPORTED;
  if (n_q <= 0 || n_kv < 0) return CODA_ERR_INVALID_ARG;
  const int64_t N = static_cast<int64_t>(n_q + 2 * n_kv) * head_dim;
  CK(dims_ok(M, N, Kdim));
  if (Kdim % 16) return CODA_ERR_UNSUPPORTED;
  CK(ws_ok(ws, ws_bytes, WS_HEADER));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)Xq, (const void*)sx, (const void*)Wq, (const void*)sw}) CK(req(q));
  coda_epilogue_desc d;
  std::memset(&d, 0, sizeof(d));
  d.map = CODA_MAP_QKNORM_ROPE;
  d.operand_type = CODA_OPERAND_E4M3;
  d.acc_row_scale = sx;
  d.acc_col_scale = sw;
  d.row_scale = rstd;
  d.aux_out[0] = qk_save;
  d.ld_aux_out[0] = static_cast<int64_t>(n_q + n_kv) * head_dim;
  d.positions = pos;
  d.cos_sin = cos_sin;
  d.max_pos = max_pos;
  d.n_q_heads = n_q;
  d.n_kv_heads = n_kv;
  d.head_dim = head_dim;
  d.rope_pairing = rope_pairing;
  d.eps = eps;
  d.gamma_q = gamma_q;
  d.gamma_k = gamma_k;
  d.Q = Q;
  d.K = K;
  d.V = V;
  CK(al(rstd));
  return coda_gemm_epilogue(&d, reinterpret_cast<const coda_bf16*>(Xq), Kdim, CODA_K_MAJOR,
                            reinterpret_cast<const coda_bf16*>(Wq), Kdim, CODA_K_MAJOR, nullptr, N, CODA_BF16, M, N,
                            Kdim, ws, ws_bytes, stream);
}

size_t coda_linear_cross_entropy_fp8_workspace_size(int64_t M, int64_t V, int64_t K) {
  return coda_linear_cross_entropy_workspace_size(M, V, K);
}

int coda_linear_cross_entropy_fp8(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw,
                                  const int32_t* labels, int32_t ignore_index, float* loss_mean, float* lse,
                                  int32_t* n_valid, int64_t M, int64_t V, int64_t K, void* ws, size_t ws_bytes,
                                  coda_stream stream) {
  if (K % 16) return CODA_ERR_UNSUPPORTED;
  if (M > 0)
    for (const void* q : {(const void*)sx, (const void*)sw}) CK(req(q));
  CK(al(sw));
  return ce_forward(reinterpret_cast<const coda_bf16*>(Xq), reinterpret_cast<const coda_bf16*>(Wq), labels,
                    ignore_index, nullptr, loss_mean, lse, n_valid, M, V, K, ws, ws_bytes, stream, 1, sx, sw);
}

size_t coda_linear_cross_entropy_bwd_fp8_workspace_size(int64_t M, int64_t V, int64_t K) {
  return ce_bwd_workspace(M, V, K, false);
}

int coda_linear_cross_entropy_bwd_fp8(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw,
                                      const coda_bf16* X, const coda_bf16* W, const int32_t* labels,
                                      int32_t ignore_index, const float* lse, const int32_t* n_valid, float dloss,
                                      coda_bf16* dX, coda_bf16* dW, int64_t M, int64_t V, int64_t K, void* ws,
                                      size_t ws_bytes, coda_stream stream) {
  CK(dims_ok(M, V, K));
  if (K % 16) return CODA_ERR_UNSUPPORTED;
  CK(ws_ok(ws, ws_bytes, coda_linear_cross_entropy_bwd_fp8_workspace_size(M, V, K)));
  CK(req(dW));
  if (M > 0)
    for (const void* q : {(const void*)Xq, (const void*)sx, (const void*)Wq, (const void*)sw, (const void*)X,
                          (const void*)W, (const void*)labels, (const void*)lse, (const void*)n_valid,
                          (const void*)dX})
      CK(req(q));
  for (const void* q : {(const void*)Xq, (const void*)Wq, (const void*)sw, (const void*)X, (const void*)W,
                        (const void*)dX, (const void*)dW})
    CK(al(q));
  if (V == 0) return CODA_ERR_INVALID_ARG;
  if (M == 0) {
    CU(cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * K * 2, S(stream)));
    return CODA_OK;
  }
  CeBwd a;
  a.Xq = Xq;
  a.sx = sx;
  a.Wq = Wq;
  a.sw = sw;
  a.X = X;
  a.W = W;
  a.labels = labels;
  a.ignore_index = ignore_index;
  a.lse = lse;
  a.n_valid = n_valid;
  a.dloss = dloss;
  a.dX = dX;
  a.dW = dW;
  a.M = M;
  a.V = V;
  a.K = K;
  return ce_backward(a, ws, S(stream));
}

size_t coda_linear_dswiglu_fp8_workspace_size(int64_t M, int64_t I, int64_t) {
  SizeCursor c;
  c.take<float>(static_cast<size_t>(cdiv(I, BN)) * M);  // row partials of sum(dG g + dU u)
  return c.off;
}

int coda_linear_dswiglu_fp8(const uint8_t* dYq, const float* sdy, const uint8_t* WdTq, const float* swd,
                            const coda_bf16* g, const coda_bf16* u, const float* rstd, coda_bf16* Gp, float* row_out,
                            coda_bf16* H, int64_t M, int64_t I, int64_t K, void* ws, size_t ws_bytes,
                            coda_stream stream) {
  CK(dims_ok(M, I, K));
  if (K % 16) return CODA_ERR_UNSUPPORTED;
  CK(ws_ok(ws, ws_bytes, coda_linear_dswiglu_fp8_workspace_size(M, I, K)));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)dYq, (const void*)sdy, (const void*)WdTq, (const void*)swd, (const void*)g,
                        (const void*)u, (const void*)Gp})
    CK(req(q));
  for (const void* q : {(const void*)dYq, (const void*)WdTq, (const void*)swd, (const void*)g, (const void*)u,
                        (const void*)Gp, (const void*)H})
    CK(al(q));
  WsCursor w(ws);
  float* spart = w.take<float>(static_cast<size_t>(cdiv(I, BN)) * M);
  int* status = static_cast<int*>(ws);
  cudaStream_t s = S(stream);
  Plan p;
  p.kind = coda::EpiKind::DSwiglu;
  p.fp8 = 1;
  p.A = dYq;
  p.lda = K;
  p.B = WdTq;
  p.ldb = K;
  p.M = M;
  p.N = I;
  p.K = K;
  p.e.acc_rs = sdy;
  p.e.acc_cs = swd;
  p.e.aux0 = BF(g);
  p.e.ld_aux0 = I;
  p.e.aux1 = BF(u);
  p.e.ld_aux1 = I;
  p.e.out1 = BF(Gp);
  p.e.ld_out1 = 2 * I;
  p.e.out2 = BF(Gp) + I;
  p.e.ld_out2 = 2 * I;
  p.e.out3 = BF(H);
  p.e.ld_out3 = I;
  p.e.row_scale = rstd;
  if (row_out) {
    p.e.partials = spart;
    p.e.ld_part = M;
  }
  CK(run(p, status, s));
  // the N tiles' partials summed: with rstd the RMSNorm-backward coefficient
  // c_i = r_i^2 * sum / K, without it the sum itself
  if (row_out)
    CU(coda::launch_combine_rows(spart, M, static_cast<int>(cdiv(I, BN)), M,
                                 rstd ? 1.f / static_cast<float>(K) : 1.f, 0.f, rstd, row_out, 1, s));
  return CODA_OK;
}

size_t coda_rmsnorm_linear_dx_fp8_workspace_size(int64_t M, int64_t, int64_t K) {
  SizeCursor c;
  c.take<float>(static_cast<size_t>(4 * cdiv(M, 128)) * K);  // dgamma partials per (token block, warp)
  return c.off;
}

int coda_rmsnorm_linear_dx_fp8(const uint8_t* Gq, const float* sg, const uint8_t* WTq, const float* sw,
                               const coda_bf16* X, const float* gamma, const float* coef, const coda_bf16* dX_resid,
                               coda_bf16* dX, float* dgamma, int64_t M, int64_t N, int64_t K, void* ws,
                               size_t ws_bytes, coda_stream stream) {
  CK(dims_ok(M, K, N));
  if (N % 16) return CODA_ERR_UNSUPPORTED;
  CK(ws_ok(ws, ws_bytes, coda_rmsnorm_linear_dx_fp8_workspace_size(M, N, K)));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)Gq, (const void*)sg, (const void*)WTq, (const void*)sw, (const void*)X,
                        (const void*)gamma, (const void*)coef, (const void*)dX, (const void*)dgamma})
    CK(req(q));
  for (const void* q : {(const void*)Gq, (const void*)WTq, (const void*)sw, (const void*)X, (const void*)gamma,
                        (const void*)dX_resid, (const void*)dX})
    CK(al(q));
  WsCursor w(ws);
  const int64_t ntb = cdiv(M, 128);
  float* dgp = w.take<float>(static_cast<size_t>(4 * ntb) * K);
  int* status = static_cast<int*>(ws);
  cudaStream_t s = S(stream);
  Plan p;
  p.kind = coda::EpiKind::RmsDx;
  p.fp8 = 1;
  p.A = Gq;
  p.lda = N;
  p.B = WTq;
  p.ldb = N;
  p.M = M;
  p.N = K;
  p.K = N;
  p.e.acc_rs = sg;
  p.e.acc_cs = sw;
  p.e.D = dX;
  p.e.ldd = K;
  p.e.aux0 = BF(dX_resid);
  p.e.ld_aux0 = K;
  p.e.row_coef = coef;
  p.e.aux1 = BF(X);
  p.e.ld_aux1 = K;
  p.e.col_scale = gamma;
  p.e.partials = dgp;
  p.e.ld_part = K;
  CK(run(p, status, s));
  CU(coda::launch_colsum(dgp, 4 * ntb, K, K, dgamma, s));
  return CODA_OK;
}

size_t coda_linear_qknorm_rope_bwd_fp8_workspace_size(int64_t M, int64_t Kdim, int32_t n_q, int32_t n_kv,
                                                      int32_t head_dim) {
  const int64_t N = static_cast<int64_t>(n_q + 2 * n_kv) * head_dim;
  SizeCursor c;
  c.take<__nv_bfloat16>(static_cast<size_t>(M) * N);          // G'
  c.take<float>(M);                                           // coef
  c.take<float>(static_cast<size_t>(qk_bwd_blocks(M)) * 256);  // dgamma_q|k partials
  c.take<float>(static_cast<size_t>(4 * cdiv(M, 128)) * Kdim);  // dgamma_in partials per (token block, warp)
  c.take<uint8_t>(static_cast<size_t>(M) * N);                // Gq: G' per row
  c.take<float>(M);                                           // sg
  c.take<uint8_t>(static_cast<size_t>(N) * M);                // GTq: G'^T per column of G'
  c.take<float>(N);                                           // sgT
  return c.off;
}

int coda_linear_qknorm_rope_bwd_fp8(const coda_bf16* dQ, const coda_bf16* dK, const coda_bf16* dV,
                                    const coda_bf16* qk_save, const coda_bf16* V, const float* gamma_q,
                                    const float* gamma_k, const int32_t* pos, const float* cos_sin, int32_t max_pos,
                                    float eps, int32_t n_q, int32_t n_kv, int32_t head_dim, int32_t rope_pairing,
                                    const coda_bf16* X, const float* rstd, const float* gamma_in,
                                    const uint8_t* WTq, const float* sw, const uint8_t* UTq, const float* su,
                                    const coda_bf16* dX_resid, coda_bf16* dX, coda_bf16* dW_qkv, float* dgamma_in,
                                    float* dgamma_q, float* dgamma_k, int64_t M, int64_t Kdim, void* ws,
                                    size_t ws_bytes, coda_stream stream) {
  if (head_dim != 128) return CODA_ERR_UNSUPPORTED;
  if (n_q <= 0 || n_kv <= 0 || max_pos <= 0) return CODA_ERR_INVALID_ARG;
  if (rope_pairing != CODA_ROPE_INTERLEAVED && rope_pairing != CODA_ROPE_HALF) return CODA_ERR_INVALID_ARG;
  const int64_t N = static_cast<int64_t>(n_q + 2 * n_kv) * head_dim;
  CK(dims_ok(M, N, Kdim));
  if (M % 16) return CODA_ERR_UNSUPPORTED;  // 16-byte rows of the K-major token operands of the dW GEMM
  CK(ws_ok(ws, ws_bytes, coda_linear_qknorm_rope_bwd_fp8_workspace_size(M, Kdim, n_q, n_kv, head_dim)));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)dQ, (const void*)dK, (const void*)dV, (const void*)qk_save, (const void*)V,
                        (const void*)gamma_q, (const void*)gamma_k, (const void*)pos, (const void*)cos_sin,
                        (const void*)WTq, (const void*)sw, (const void*)UTq, (const void*)su, (const void*)dX,
                        (const void*)dW_qkv, (const void*)dgamma_q, (const void*)dgamma_k})
    CK(req(q));
  for (const void* q : {(const void*)dQ, (const void*)dK, (const void*)dV, (const void*)qk_save, (const void*)V,
                        (const void*)gamma_q, (const void*)gamma_k, (const void*)cos_sin, (const void*)X,
                        (const void*)rstd, (const void*)gamma_in, (const void*)WTq, (const void*)sw,
                        (const void*)UTq, (const void*)su, (const void*)dX_resid, (const void*)dX,
                        (const void*)dW_qkv, (const void*)dgamma_in, (const void*)dgamma_q, (const void*)dgamma_k})
    CK(al(q));
  const bool norm = rstd != nullptr;
  if (norm && (!gamma_in || !dgamma_in || !X)) return CODA_ERR_INVALID_ARG;
  const int sms = num_sms();
  if (sms <= 0) return CODA_ERR_CUDA;
  WsCursor w(ws);
  __nv_bfloat16* Gp = w.take<__nv_bfloat16>(static_cast<size_t>(M) * N);
  float* coef = w.take<float>(M);
  const int nblk = qk_bwd_blocks(M);
  float* dgqk = w.take<float>(static_cast<size_t>(nblk) * 256);
  const int64_t ntb = cdiv(M, 128);
  float* dgp = w.take<float>(static_cast<size_t>(4 * ntb) * Kdim);
  uint8_t* Gq = w.take<uint8_t>(static_cast<size_t>(M) * N);
  float* sg = w.take<float>(M);
  uint8_t* GTq = w.take<uint8_t>(static_cast<size_t>(N) * M);
  float* sgT = w.take<float>(N);
  int* status = static_cast<int*>(ws);
  cudaStream_t s = S(stream);
  CK(qk_bwd_map(dQ, dK, dV, qk_save, V, gamma_q, gamma_k, pos, cos_sin, max_pos, eps, n_q, n_kv, rope_pairing, rstd,
                M, Kdim, Gp, norm ? coef : nullptr, dgqk, nblk, dgamma_q, dgamma_k, sms, status, s));
  CU(coda::launch_quantize_fp8_rows(Gp, N, M, N, Gq, N, sg, sms, s));
  {  // D = G' W_qkv on the codes;  dX = gamma_in D - c X + dX_resid with the
     // dgamma_in column partials  (without RMSNorm: D + dX_resid)
    Plan p;
    p.kind = norm ? coda::EpiKind::RmsDx : coda::EpiKind::Plain;
    p.fp8 = 1;
    p.A = Gq;
    p.lda = N;
    p.B = WTq;
    p.ldb = N;
    p.M = M;
    p.N = Kdim;
    p.K = N;
    p.e.D = dX;
    p.e.ldd = Kdim;
    p.e.aux0 = BF(dX_resid);
    p.e.ld_aux0 = Kdim;
    if (norm) {
      p.e.acc_rs = sg;
      p.e.acc_cs = sw;
      p.e.row_coef = coef;
      p.e.aux1 = BF(X);
      p.e.ld_aux1 = Kdim;
      p.e.col_scale = gamma_in;
      p.e.partials = dgp;
      p.e.ld_part = Kdim;
    } else {
      p.e.row_scale = sg;
      p.e.col_scale = sw;
    }
    CK(run(p, status, s));
  }
  if (norm) CU(coda::launch_colsum(dgp, 4 * ntb, Kdim, Kdim, dgamma_in, s));
  CU(coda::launch_quantize_fp8_cols(Gp, N, M, nullptr, 0, 0, N, GTq, M, sgT, sms, s));
  {  // dW_qkv = G'^T U on the column codes of both
    Plan p;
    p.fp8 = 1;
    p.A = GTq;
    p.lda = M;
    p.B = UTq;
    p.ldb = M;
    p.M = N;
    p.N = Kdim;
    p.K = M;
    p.e.D = dW_qkv;
    p.e.ldd = Kdim;
    p.e.row_scale = sgT;
    p.e.col_scale = su;
    CK(run(p, status, s));
  }
  return CODA_OK;
}

// ------------------------------------------------------------------ NVFP4 operands
size_t coda_nvfp4_scale_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0) return 0;
  return static_cast<size_t>(cdiv(rows, 512) * 4 * cdiv(K, 256) * 2048);
}

int coda_quantize_nvfp4_rows(const coda_bf16* X, int64_t ldx, int64_t M, int64_t K, uint8_t* Xq, uint8_t* sf,
                             float* scale, coda_stream stream) {
  if (M < 0 || K < 0) return CODA_ERR_INVALID_ARG;
  if (K % 32) return CODA_ERR_UNSUPPORTED;  // 16-byte rows of packed codes for the tensor maps
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)X, (const void*)Xq, (const void*)sf, (const void*)scale}) CK(req(q));
  CK(al(X));
  CK(al(Xq));
  CK(al(sf));
  CK(ldok(ldx, K));
  const int sms = num_sms();
  if (sms <= 0) return CODA_ERR_CUDA;
  CU(coda::launch_quantize_nvfp4_rows(BF(X), ldx, M, K, Xq, sf, scale, sms, S(stream)));
  return CODA_OK;
}

int coda_rmsnorm_scale_nvfp4(const coda_bf16* X, int64_t ldx, int64_t M, int64_t K, float eps, const float* gamma,
                             float* rstd, uint8_t* Xq, uint8_t* sf, float* scale, coda_stream stream) {
  if (M < 0 || K < 0) return CODA_ERR_INVALID_ARG;
  if (K % 32) return CODA_ERR_UNSUPPORTED;
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)X, (const void*)gamma, (const void*)Xq, (const void*)sf, (const void*)scale})
    CK(req(q));
  for (const void* q : {(const void*)X, (const void*)gamma, (const void*)Xq, (const void*)sf}) CK(al(q));
  CK(ldok(ldx, K));
  const int sms = num_sms();
  if (sms <= 0) return CODA_ERR_CUDA;
  CU(coda::launch_quantize_nvfp4_rows(BF(X), ldx, M, K, Xq, sf, scale, sms, S(stream), gamma, rstd, eps));
  return CODA_OK;
}

size_t coda_linear_nvfp4_workspace_size(int64_t, int64_t, int64_t) { return WS_HEADER; }

int coda_linear_nvfp4(const uint8_t* Xq, const uint8_t* sfx, const float* sx, const uint8_t* Wq, const uint8_t* sfw,
                      const float* sw, const coda_bf16* R, coda_bf16* Y, int64_t M, int64_t N, int64_t K, void* ws,
                      size_t ws_bytes, coda_stream stream) {
  CK(dims_ok(M, N, K));
  if (K % 32) return CODA_ERR_UNSUPPORTED;
  CK(ws_ok(ws, ws_bytes, WS_HEADER));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)Xq, (const void*)sfx, (const void*)sx, (const void*)Wq, (const void*)sfw,
                        (const void*)sw, (const void*)Y})
    CK(req(q));
  for (const void* q : {(const void*)Xq, (const void*)sfx, (const void*)Wq, (const void*)sfw, (const void*)R,
                        (const void*)Y})
    CK(al(q));
  EpiArgs e{};
  e.D = Y;
  e.ldd = N;
  e.row_scale = sx;
  e.col_scale = sw;
  e.aux0 = BF(R);
  e.ld_aux0 = N;
  coda::Nvfp4Scales sc{sfx, sfw, sfw, 0};
  return run_nvfp4(coda::EpiKind::Plain, Xq, Wq, Wq, sc, M, N, K, 0, e, static_cast<int*>(ws), S(stream));
}

size_t coda_linear_swiglu_nvfp4_workspace_size(int64_t, int64_t, int64_t) { return WS_HEADER; }

int coda_linear_swiglu_nvfp4(const uint8_t* Xq, const uint8_t* sfx, const float* sx, const float* rstd,
                             const uint8_t* Wgq, const uint8_t* sfg, const float* sg, const uint8_t* Wuq,
                             const uint8_t* sfu, const float* su, coda_bf16* H, coda_bf16* g_save,
                             coda_bf16* u_save, int64_t M, int64_t I, int64_t K, void* ws, size_t ws_bytes,
                             coda_stream stream) {
  CK(dims_ok(M, I, K));
  if (K % 32) return CODA_ERR_UNSUPPORTED;
  CK(ws_ok(ws, ws_bytes, WS_HEADER));
  if (M == 0) return CODA_OK;
  for (const void* q : {(const void*)Xq, (const void*)sfx, (const void*)sx, (const void*)Wgq, (const void*)sfg,
                        (const void*)sg, (const void*)Wuq, (const void*)sfu, (const void*)su, (const void*)H})
    CK(req(q));
  for (const void* q : {(const void*)Xq, (const void*)sfx, (const void*)Wgq, (const void*)sfg, (const void*)Wuq,
                        (const void*)sfu, (const void*)sg, (const void*)su, (const void*)H, (const void*)g_save,
                        (const void*)u_save})
    CK(al(q));
  EpiArgs e{};
  e.D = H;
  e.ldd = I;
  e.row_scale = sx;
  e.row_scale2 = rstd;
  e.col_scale = sg;
  e.col_scale2 = su;
  e.out1 = BF(g_save);
  e.ld_out1 = I;
  e.out2 = BF(u_save);
  e.ld_out2 = I;
  coda::Nvfp4Scales sc{sfx, sfg, sfu, 0};
  return run_nvfp4(coda::EpiKind::Swiglu, Xq, Wgq, Wuq, sc, M, I, K, 1, e, static_cast<int*>(ws), S(stream));
}

}  // extern "C"
