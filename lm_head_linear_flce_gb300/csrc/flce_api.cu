// C ABI of the fused linear cross-entropy library: argument checks, the
// problem plan and workspace layout, tensor-map encoding and the launch
// sequences of flce_forward / flce_backward.  See include/flce.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/flce.h"
#include "flce_internal.h"

namespace flce {

namespace {

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1024;
constexpr int64_t kMaxH = 1 << 16;
constexpr int64_t kMaxShards = 1 << 16;
// Automatic backward blocking (no flce_set_backward_block caps): every token
// row in one block while that leaves at least 2048 vocab columns, so that dW
// is written once with no FP32 band; a dZ block of at most 32 Mi elements
// (64 MB) up to 8192 rows and 64 Mi (128 MB) above.
constexpr int64_t kSmallDzBlockElems = int64_t{32} << 20;
constexpr int64_t kLargeDzBlockElems = int64_t{64} << 20;
constexpr int64_t kSmallBlockRows = 8192;
constexpr int64_t kMinBlockCols = 2048;
// Above kSmallBlockRows rows the block may grow to this many elements (256 MB)
// so that a launch holds at least kMinWTiles dW tiles (one per CTA pair of a
// 152-SM GB300): fewer leave pairs idle while the launch's dW tiles finish.
constexpr int64_t kMaxAutoBlockElems = int64_t{128} << 20;
constexpr int64_t kMinWTiles = 76;
// The block's W rows (Vb x H bf16), which the recompute tiles sweep once per
// row tile, are kept within this many bytes, about half of L2, so that they
// are still there for the next row tile (binds only for H >= 4096).
constexpr int64_t kMaxWBlockBytes = int64_t{64} << 20;
constexpr size_t kAlign = 256;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;

std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitNs};
std::atomic<int64_t> g_block_rows{0};   // 0: automatic
std::atomic<int64_t> g_block_elems{0};  // 0: automatic

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Whether the byte ranges [a, a + na) and [b, b + nb) share a byte.
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na > 0 && nb > 0 && x < y + nb && y < x + na;
}
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct DeviceInfo {
  int sms = 0;
  bool ok = false;
};

// Per-device answer, cached: 0 until the first query on that device, then
// (SM count << 1) | (compute capability is 10.3).  Atomic, so concurrent
// first calls from several host threads are safe (they store the same value).
std::atomic<int> g_device_cache[64];

flce_status device_info(DeviceInfo* d) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLCE_ERR_CUDA;
  const bool cacheable = dev >= 0 && dev < 64;
  int v = cacheable ? g_device_cache[dev].load(std::memory_order_acquire) : 0;
  if (v == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FLCE_ERR_CUDA;
    v = (std::max(sms, 1) << 1) | ((major == 10 && minor == 3) ? 1 : 0);
    if (cacheable) g_device_cache[dev].store(v, std::memory_order_release);
  }
  d->sms = v >> 1;
  d->ok = (v & 1) != 0;
  return d->ok ? FLCE_OK : FLCE_ERR_UNSUPPORTED_DEVICE;
}

flce_status check_common(const void* X, const void* W, const int64_t* labels, int64_t N,
                         int64_t H, int64_t V, int64_t seq_len, int shift,
                         flce_reduction reduction, void* ws, size_t ws_bytes, Plan* plan) {
  if (N < 0 || H <= 0 || V <= 0) return FLCE_ERR_INVALID_ARG;
  if (reduction != FLCE_REDUCTION_MEAN && reduction != FLCE_REDUCTION_SUM)
    return FLCE_ERR_INVALID_ARG;
  if (H % 8 != 0 || H > kMaxH || N > kMaxDim || V > kMaxDim) return FLCE_ERR_UNSUPPORTED_SHAPE;
  if (!ws) return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (!X || !W || !labels)) return FLCE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W)) & 15)
    return FLCE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) return FLCE_ERR_INVALID_ARG;
  if (shift && N > 0) {
    const int64_t S = seq_len > 0 ? seq_len : N;
    if (N % S != 0) return FLCE_ERR_INVALID_ARG;
  }
  if (!make_plan(N, H, V, plan)) return FLCE_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < plan->total) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  return FLCE_OK;
}

// ------------------------------------------------------------ measurement
std::atomic<int64_t> g_launches{0};
std::atomic<bool> g_prof_on{false};
std::mutex g_prof_mu;
struct ProfRec {
  int kind;
  cudaEvent_t a, b;
  int launches = 1;
};
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Brackets one tensor-core launch with profiling events when enabled.
template <class F>
cudaError_t profiled(int kind, cudaStream_t s, F&& launch) {
  if (!g_prof_on.load()) return launch();
  std::lock_guard<std::mutex> lk(g_prof_mu);
  ProfRec r{kind, take_event(), take_event(), 1};
  if (r.a) cudaEventRecord(r.a, s);
  cudaError_t e = launch();
  if (r.b) cudaEventRecord(r.b, s);
  if (r.a && r.b) g_prof.push_back(r);
  return e;
}

// Brackets a run of consecutive launches (which may overlap each other) with
// one pair of profiling events; `launches` is how many the run holds.
ProfRec g_open{-1, nullptr, nullptr, 0};
void prof_begin(cudaStream_t s) {
  if (!g_prof_on.load()) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_open.a = take_event();
  if (g_open.a) cudaEventRecord(g_open.a, s);
}
void prof_end(int kind, int launches, cudaStream_t s) {
  if (!g_prof_on.load()) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_open.a) return;
  ProfRec r{kind, g_open.a, take_event(), launches};
  g_open.a = nullptr;
  if (!r.b) return;
  cudaEventRecord(r.b, s);
  r.launches = launches;
  g_prof.push_back(r);
}

// NVTX range over the host-side enqueue of one call (or one phase of it), so
// that a timeline tool groups the call's launches; costs a pointer check when
// no tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

#define FLCE_CUDA(x)                         \
  do {                                       \
    if ((x) != cudaSuccess) return FLCE_ERR_CUDA; \
  } while (0)

}  // namespace

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// 2-D tensor map over a row-major [outer][inner] matrix with 128-byte swizzle;
// out-of-bounds elements read as zero and are not written.
bool make_tmap(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapDataType dtype) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dtype, 2, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view (64 elements, rows, 64-element groups) of a row-major matrix with
// `inner` (a multiple of 64) elements per row: box 64 x 64 rows x 2 groups is
// one 128-column MN-major operand half in the 128-byte-swizzled layout.
bool make_tmap_mn3(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows,
                   uint64_t row_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || inner % 64 != 0) return false;
  cuuint64_t dims[3] = {64, rows, inner / 64};
  cuuint64_t strides[2] = {row_bytes, 128};
  cuuint32_t box[3] = {64, 64, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(); }

namespace {
std::atomic<unsigned long long> g_last_wait_limit{0};
}  // namespace

void note_wait_limit(unsigned long long limit_ns) { g_last_wait_limit.store(limit_ns); }

bool make_plan(int64_t N, int64_t H, int64_t V, Plan* p) {
  if (N < 0 || H <= 0 || V <= 0) return false;
  std::memset(p, 0, sizeof(*p));
  p->N = N;
  p->H = H;
  p->V = V;
  p->m_tiles = static_cast<int>(cdiv(N, kPairM));
  p->v_tiles = static_cast<int>(cdiv(V, kBN));
  p->fwd_group = forward_unit_tiles(p->v_tiles);
  p->v_units = static_cast<int>(cdiv(p->v_tiles, p->fwd_group));
  p->h_tiles = static_cast<int>(cdiv(H, kBN));
  // Backward blocking: a token block of Nb rows x a vocab block of Vb columns
  // of dZ is formed at a time (bf16, at most max_elems).  All rows in one
  // block when they fit, so dW needs no FP32 accumulator across blocks.
  const int64_t n_pad = std::max<int64_t>(int64_t{p->m_tiles} * kPairM, kPairM);
  int64_t max_elems = g_block_elems.load();
  if (max_elems <= 0)
    max_elems = n_pad <= kSmallBlockRows ? kSmallDzBlockElems : kLargeDzBlockElems;
  int64_t max_rows = g_block_rows.load();
  if (max_rows <= 0)
    max_rows = std::max<int64_t>(max_elems / kMinBlockCols / kPairM * kPairM, kPairM);
  if (n_pad <= max_rows) {
    p->Nb = n_pad;
  } else {
    const int64_t nblk = cdiv(n_pad, max_rows);
    p->Nb = cdiv(std::max(p->m_tiles, 1), nblk) * kPairM;
  }
  const int64_t v_pad = int64_t{p->v_tiles} * kBN;
  auto cols = [&](int64_t elems) {
    return std::min<int64_t>(v_pad, std::max<int64_t>(kBN, elems / p->Nb / kBN * kBN));
  };
  p->Vb = cols(max_elems);
  // large problems (every row in one block): grow the block while its dW tiles
  // would leave CTA pairs without one
  if (g_block_elems.load() <= 0 && n_pad > kSmallBlockRows && p->Nb == n_pad) {
    while ((p->Vb / kBN) * p->h_tiles < kMinWTiles && max_elems < kMaxAutoBlockElems &&
           p->Vb < v_pad) {
      max_elems *= 2;
      p->Vb = cols(max_elems);
    }
  }
  if (g_block_elems.load() <= 0)
    p->Vb = std::min<int64_t>(p->Vb, std::max<int64_t>(kBN, kMaxWBlockBytes / (2 * H) / kBN * kBN));
  p->n_blocks = N > 0 ? static_cast<int>(cdiv(N, p->Nb)) : 0;
  p->v_blocks = static_cast<int>(cdiv(V, p->Vb));
  p->multi_n = p->n_blocks > 1;

  size_t off = 0;
  p->off_err = off;
  off = align_up(off + 16);
  p->off_t = off;
  off = align_up(off + static_cast<size_t>(N) * 4);
  const size_t shared_start = off;
  // forward view
  p->off_zt = off;
  off = align_up(off + static_cast<size_t>(N) * 4);
  p->off_part = off;
  off = align_up(off + static_cast<size_t>(kFwdSplits) * N * 8);  // O(N * splits), not O(N * V)
  p->off_lossp = off;
  off = align_up(off + static_cast<size_t>(cdiv(N, kMergeRows) + 1) * 8);
  p->off_fcnt = off;  // forward unit ticket
  off = align_up(off + 4);
  const size_t fwd_end = off;
  // backward view (overlaps the forward view: the workspace need not persist)
  p->launches = p->n_blocks * p->v_blocks + 1;
  off = shared_start;
  p->off_cnt = off;
  off = align_up(off + static_cast<size_t>(p->launches) * 4);
  p->off_flags = off;  // per 256-row token tile: holds a valid target
  off = align_up(off + static_cast<size_t>(p->m_tiles) * 4);
  p->off_active = off;  // active tiles, ascending, then their count
  off = align_up(off + static_cast<size_t>(p->m_tiles + 1) * 4);
  // dense rows (rows with a valid target gathered to the front): per-tile
  // offsets, and per dense row its target and lse, per token row its dense index
  p->off_toff = off;
  off = align_up(off + static_cast<size_t>(p->m_tiles + 1) * 4);
  p->off_tc = off;
  off = align_up(off + static_cast<size_t>(N) * 4);
  p->off_lc = off;
  off = align_up(off + static_cast<size_t>(N) * 4);
  p->off_inv = off;
  off = align_up(off + static_cast<size_t>(N) * 4);
  p->off_done = off;  // per launch and local row tile: R-tile epilogue warps done
  off = align_up(off + static_cast<size_t>(p->n_blocks * p->v_blocks) * (p->Nb / kPairM) * 4);
  p->off_dxf = off;
  if (p->v_blocks > 1) off = align_up(off + static_cast<size_t>(N) * H * 4);
  p->off_dwf = off;
  if (p->multi_n) off = align_up(off + static_cast<size_t>(p->Vb) * H * 4);
  // two slots: block p is formed (and its dX part taken) while the dW part of
  // block p-1 is consumed.  Rows are padded by 64 elements so that the row
  // pitch is not a power of two.
  p->dz_ld = p->Vb + 64;
  p->off_dz = off;
  off = align_up(off + 2 * static_cast<size_t>(p->Nb) * p->dz_ld * 2);
  p->total = std::max(fwd_end, off);
  return true;
}

}  // namespace flce

using namespace flce;

extern "C" {

const char* flce_status_string(flce_status s) {
  switch (s) {
    case FLCE_OK: return "FLCE_OK";
    case FLCE_ERR_INVALID_ARG: return "FLCE_ERR_INVALID_ARG";
    case FLCE_ERR_UNSUPPORTED_SHAPE: return "FLCE_ERR_UNSUPPORTED_SHAPE";
    case FLCE_ERR_WORKSPACE_TOO_SMALL: return "FLCE_ERR_WORKSPACE_TOO_SMALL";
    case FLCE_ERR_LABEL_OUT_OF_RANGE: return "FLCE_ERR_LABEL_OUT_OF_RANGE";
    case FLCE_ERR_TIMEOUT: return "FLCE_ERR_TIMEOUT";
    case FLCE_ERR_CUDA: return "FLCE_ERR_CUDA";
    case FLCE_ERR_UNSUPPORTED_DEVICE: return "FLCE_ERR_UNSUPPORTED_DEVICE";
  }
  return "FLCE_ERR_UNKNOWN";
}

size_t flce_workspace_size(int64_t N, int64_t H, int64_t V) {
  if (N < 0 || H <= 0 || V <= 0 || H % 8 != 0 || H > kMaxH || N > kMaxDim || V > kMaxDim)
    return 0;
  Plan p;
  if (!make_plan(N, H, V, &p)) return 0;
  return p.total;
}

flce_status flce_backward_blocking(int64_t N, int64_t H, int64_t V, int64_t* Nb, int64_t* Vb) {
  if (!Nb || !Vb || N < 0 || H <= 0 || V <= 0 || H % 8 != 0 || H > kMaxH || N > kMaxDim ||
      V > kMaxDim)
    return FLCE_ERR_INVALID_ARG;
  Plan p;
  if (!make_plan(N, H, V, &p)) return FLCE_ERR_UNSUPPORTED_SHAPE;
  *Nb = p.Nb;
  *Vb = p.Vb;
  return FLCE_OK;
}

void flce_set_wait_limit_ns(int64_t limit_ns) {
  g_wait_limit_ns.store(limit_ns > 0 ? static_cast<unsigned long long>(limit_ns)
                                     : kDefaultWaitNs);
}

void flce_set_backward_block(int64_t max_rows, int64_t max_block_elems) {
  g_block_rows.store(max_rows > 0 ? std::max<int64_t>(max_rows / kPairM * kPairM, kPairM) : 0);
  g_block_elems.store(max_block_elems > 0 ? max_block_elems : 0);
}

}  // extern "C"

namespace {

// Shared body of flce_forward (loss and lse over the whole vocabulary) and
// flce_forward_vocab_shard (z_out non-null: this shard's lse and target logit).
flce_status forward_impl(const void* X, const void* W, const int64_t* labels, int64_t N,
                         int64_t H, int64_t V, const VocabSlice& vs, int64_t seq_len,
                         int64_t ignore_index, int shift, flce_reduction reduction, float* loss,
                         float* lse, float* z_out, int64_t* n_valid, void* workspace,
                         size_t workspace_bytes, flce_stream_t stream) {
  NvtxRange range(z_out ? "flce_forward_vocab_shard" : "flce_forward");
  Plan p;
  flce_status st = check_common(X, W, labels, N, H, V, seq_len, shift, reduction, workspace,
                                workspace_bytes, &p);
  if (st != FLCE_OK) return st;
  if ((!z_out && !loss) || !n_valid || (N > 0 && !lse)) return FLCE_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FLCE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* err = reinterpret_cast<int*>(ws + p.off_err);
  FLCE_CUDA(cudaMemsetAsync(err, 0, 16, s));
  FLCE_CUDA(cudaMemsetAsync(n_valid, 0, sizeof(int64_t), s));
  if (N == 0) {
    if (loss) FLCE_CUDA(cudaMemsetAsync(loss, 0, sizeof(float), s));
    return FLCE_OK;
  }
  FLCE_CUDA(cudaMemsetAsync(ws + p.off_fcnt, 0, 4, s));
  int* targets = reinterpret_cast<int*>(ws + p.off_t);
  float* zt = reinterpret_cast<float*>(ws + p.off_zt);
  float2* part = reinterpret_cast<float2*>(ws + p.off_part);
  double* lossp = reinterpret_cast<double*>(ws + p.off_lossp);
  const int S = static_cast<int>(seq_len > 0 ? seq_len : N);
  FLCE_CUDA(launch_prep_targets(labels, static_cast<int>(N), S, shift, ignore_index, vs,
                                targets, reinterpret_cast<long long*>(n_valid), err, s));

  CUtensorMap tx, tw;
  if (!make_tmap(&tx, X, H, N, H * 2, kBK, kBM) || !make_tmap(&tw, W, H, V, H * 2, kBK, kHalfN))
    return FLCE_ERR_CUDA;
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.tiles_m = p.m_tiles;
  a.tiles_n = p.v_tiles;
  a.group = p.fwd_group;
  a.units = p.m_tiles * p.v_units;
  a.band = forward_band_tiles(p.m_tiles, H);
  a.k_blocks = static_cast<int>(cdiv(H, kBK));
  a.N = static_cast<int>(N);
  a.H = static_cast<int>(H);
  a.V = static_cast<int>(V);
  a.targets = targets;
  a.partials = part;
  a.zt = zt;
  a.counter = reinterpret_cast<int*>(ws + p.off_fcnt);
  a.err = err;
  a.wait_limit_ns = g_wait_limit_ns.load();
  FLCE_CUDA(profiled(0, s, [&] { return launch_fwd_gemm(tx, tw, a, a.units, s); }));
  int nblocks = 0;
  FLCE_CUDA(launch_merge_lse(part, p.v_units, static_cast<int>(N), zt, targets, lse, lossp, s,
                             &nblocks, z_out));
  if (!z_out)
    FLCE_CUDA(launch_finalize_loss(lossp, nblocks, reinterpret_cast<const long long*>(n_valid),
                                   reduction == FLCE_REDUCTION_SUM ? 1 : 0, loss, s));
  return FLCE_OK;
}

// Shared body of flce_backward (dW written as bf16), flce_backward_accumulate
// (dW_acc += scale * dZ^T X in FP32) and flce_backward_vocab_shard (dX_acc +=
// scale * dZ W in FP32 over the shard's columns; dX is then null).
flce_status backward_impl(const void* X, const void* W, const int64_t* labels, int64_t N,
                          int64_t H, int64_t V, const VocabSlice& vs, int64_t seq_len,
                          int64_t ignore_index, int shift, flce_reduction reduction,
                          const float* lse, const int64_t* n_valid, const float* grad_loss,
                          void* dX, float* dX_acc, void* dW, float* dW_acc, void* workspace,
                          size_t workspace_bytes, flce_stream_t stream) {
  NvtxRange range(dX_acc ? "flce_backward_vocab_shard"
                         : (dW_acc ? "flce_backward_accumulate" : "flce_backward"));
  Plan p;
  flce_status st = check_common(X, W, labels, N, H, V, seq_len, shift, reduction, workspace,
                                workspace_bytes, &p);
  if (st != FLCE_OK) return st;
  if (!n_valid || !grad_loss || (N > 0 && !lse)) return FLCE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dX) | reinterpret_cast<uintptr_t>(dW) |
       reinterpret_cast<uintptr_t>(dW_acc) | reinterpret_cast<uintptr_t>(dX_acc)) & 15)
    return FLCE_ERR_INVALID_ARG;
  if (dX && dX_acc) return FLCE_ERR_INVALID_ARG;
  // The outputs are written while the inputs and the workspace are still read
  // (dX even holds the gathered rows of X during the call): no output may
  // overlap an input, the workspace or another output.
  {
    struct Range {
      const void* p;
      size_t n;
    };
    const size_t nh = static_cast<size_t>(N) * H, vh = static_cast<size_t>(V) * H;
    const Range outs[] = {{dX, nh * 2}, {dW, vh * 2}, {dW_acc, vh * 4}, {dX_acc, nh * 4}};
    const Range ins[] = {{X, nh * 2},       {W, vh * 2},        {labels, static_cast<size_t>(N) * 8},
                         {lse, static_cast<size_t>(N) * 4}, {n_valid, 8}, {grad_loss, 4},
                         {workspace, workspace_bytes}};
    for (int a = 0; a < 4; ++a) {
      if (!outs[a].p) continue;
      for (const Range& r : ins)
        if (r.p && overlaps(outs[a].p, outs[a].n, r.p, r.n)) return FLCE_ERR_INVALID_ARG;
      for (int b = a + 1; b < 4; ++b)
        if (outs[b].p && overlaps(outs[a].p, outs[a].n, outs[b].p, outs[b].n))
          return FLCE_ERR_INVALID_ARG;
    }
  }
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FLCE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* err = reinterpret_cast<int*>(ws + p.off_err);
  FLCE_CUDA(cudaMemsetAsync(err, 0, 16, s));
  if (N == 0) {
    if (dW) FLCE_CUDA(cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * H * 2, s));
    return FLCE_OK;  // nothing to add to dW_acc
  }
  const bool want_dw = dW || dW_acc;
  const bool want_dx = dX || dX_acc;
  if (!want_dx && !want_dw) return FLCE_OK;
  const int red = reduction == FLCE_REDUCTION_SUM ? 1 : 0;
  const long long* nv = reinterpret_cast<const long long*>(n_valid);
  int* targets = reinterpret_cast<int*>(ws + p.off_t);
  const int S = static_cast<int>(seq_len > 0 ? seq_len : N);
  // Rows without a valid target have dZ = 0: they add nothing to dW and their
  // dX rows are 0.  Dense rows: when bf16 dX goes through the FP32 accumulator
  // (V spans several vocab blocks), the rows with a target are gathered to the
  // front of the dX buffer (free until the final downcast, which puts the rows
  // back in token order) and the backward runs on ceil(rows / 256) dense
  // tiles.  Otherwise it runs on the 256-row token tiles that hold a target.
  const bool dense = dX && !dX_acc && p.v_blocks > 1;
  int* flags = reinterpret_cast<int*>(ws + p.off_flags);
  int* active = reinterpret_cast<int*>(ws + p.off_active);
  int* n_active = active + p.m_tiles;
  int* toff = reinterpret_cast<int*>(ws + p.off_toff);
  int* tc = reinterpret_cast<int*>(ws + p.off_tc);
  float* lc = reinterpret_cast<float*>(ws + p.off_lc);
  int* inv = reinterpret_cast<int*>(ws + p.off_inv);
  FLCE_CUDA(cudaMemsetAsync(flags, 0, static_cast<size_t>(p.m_tiles) * 4, s));
  FLCE_CUDA(launch_prep_targets(labels, static_cast<int>(N), S, shift, ignore_index, vs,
                                targets, nullptr, err, s, flags));
  const void* Xg = X;  // the X rows the backward reads
  const int* tg = targets;
  const float* lg = lse;
  if (dense) {
    FLCE_CUDA(launch_compact_rows(flags, p.m_tiles, toff, active, n_active, s));
    FLCE_CUDA(launch_gather_rows(X, targets, lse, toff, static_cast<int>(N), static_cast<int>(H),
                                 p.m_tiles, dX, tc, lc, inv, s));
    Xg = dX;
    tg = tc;
    lg = lc;
  } else {
    FLCE_CUDA(launch_compact_tiles(flags, p.m_tiles, active, n_active, s));
  }

  // the caller's FP32 buffer, or the workspace accumulator when V spans
  // several vocab blocks (a single block writes bf16 dX directly)
  float* dxf = dX_acc ? dX_acc : reinterpret_cast<float*>(ws + p.off_dxf);
  float* dwf = reinterpret_cast<float*>(ws + p.off_dwf);
  int* counters = reinterpret_cast<int*>(ws + p.off_cnt);
  __nv_bfloat16* dz0 = reinterpret_cast<__nv_bfloat16*>(ws + p.off_dz);
  __nv_bfloat16* dz1 = dz0 + static_cast<size_t>(p.Nb) * p.dz_ld;
  const bool dx_final = p.v_blocks == 1 && !dX_acc;
  const bool dw_final = !p.multi_n;
  const bool band = dW && !dw_final;  // bf16 dW over several token blocks: FP32 band
  FLCE_CUDA(cudaMemsetAsync(counters, 0, static_cast<size_t>(p.launches) * 4, s));
  int* row_done = reinterpret_cast<int*>(ws + p.off_done);
  const int tiles_per_block = static_cast<int>(p.Nb / kPairM);
  FLCE_CUDA(cudaMemsetAsync(row_done, 0,
                            static_cast<size_t>(p.n_blocks * p.v_blocks) * tiles_per_block * 4, s));
  if (dX && !dx_final) FLCE_CUDA(cudaMemsetAsync(dxf, 0, static_cast<size_t>(N) * H * 4, s));
  // rows of skipped tiles are never written by the dX tiles: start from zero
  if (dX && dx_final) FLCE_CUDA(cudaMemsetAsync(dX, 0, static_cast<size_t>(N) * H * 2, s));

  BwdMaps maps;
  if (!make_tmap(&maps.x_k, Xg, H, N, H * 2, kBK, kBM) ||
      !make_tmap(&maps.w_k, W, H, V, H * 2, kBK, kHalfN) ||
      !make_tmap(&maps.w_mn, W, H, V, H * 2, 64, 64) ||
      !make_tmap(&maps.x_mn, Xg, H, N, H * 2, 64, 64) ||
      !make_tmap(&maps.dz_k[0], dz0, p.Vb, p.Nb, p.dz_ld * 2, kBK, kBM) ||
      !make_tmap(&maps.dz_k[1], dz1, p.Vb, p.Nb, p.dz_ld * 2, kBK, kBM) ||
      !make_tmap(&maps.dz_st[0], dz0, p.Vb, p.Nb, p.dz_ld * 2, 64, 32) ||
      !make_tmap(&maps.dz_st[1], dz1, p.Vb, p.Nb, p.dz_ld * 2, 64, 32))
    return FLCE_ERR_CUDA;
  if (!make_tmap_mn3(&maps.dz_mn3[0], dz0, p.Vb, p.Nb, p.dz_ld * 2) ||
      !make_tmap_mn3(&maps.dz_mn3[1], dz1, p.Vb, p.Nb, p.dz_ld * 2))
    return FLCE_ERR_CUDA;
  const bool mn3d = H % 64 == 0 && make_tmap_mn3(&maps.w_mn3, W, H, V, H * 2) &&
                    make_tmap_mn3(&maps.x_mn3, Xg, H, N, H * 2);
  if (!mn3d) maps.w_mn3 = maps.x_mn3 = maps.dz_mn3[0];  // unused
  // epilogue targets: FP32 accumulators (reduce-add, 32 x 32 boxes) or the bf16
  // gradients written directly (64 x 32 boxes); an unused map repeats a valid one
  constexpr CUtensorMapDataType kF32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  bool ok = true;
  if (dX && dx_final)
    ok = make_tmap(&maps.dx_out, dX, H, N, H * 2, 64, 32);
  else if (want_dx)
    ok = make_tmap(&maps.dx_out, dxf, H, N, H * 4, 32, 32, kF32);
  else
    maps.dx_out = maps.dz_st[0];
  if (ok && dW_acc)
    ok = make_tmap(&maps.dw_out, dW_acc, H, V, H * 4, 32, 32, kF32);
  else if (ok && dW && dw_final)
    ok = make_tmap(&maps.dw_out, dW, H, V, H * 2, 64, 32);
  else if (ok && dW)
    ok = make_tmap(&maps.dw_out, dwf, H, p.Vb, H * 4, 32, 32, kF32);
  else
    maps.dw_out = maps.dz_st[0];
  if (!ok) return FLCE_ERR_CUDA;

  // dZ blocks in vocab-major order: b = vb * n_blocks + nb.  Token block nb
  // covers active tiles [nb * Nb/256, (nb + 1) * Nb/256); with tiles skipped the
  // last blocks hold fewer tiles or none (the kernels read the active count).
  const int nblk = p.n_blocks * p.v_blocks;
  auto block = [&](int b) {
    BlockDesc d;
    const int vb = b / p.n_blocks, nb = b % p.n_blocks;
    const int64_t col0 = int64_t{vb} * p.Vb;
    const int64_t vext = std::min<int64_t>(p.Vb, V - col0);
    d.tile0 = nb * tiles_per_block;
    d.col0 = static_cast<int>(col0);
    d.mt = std::min(tiles_per_block, p.m_tiles - d.tile0);
    d.vt = static_cast<int>(cdiv(vext, kBN));
    d.slot = b & 1;
    return d;
  };

  BwdArgs base;
  std::memset(&base, 0, sizeof(base));
  base.want_dx = want_dx ? 1 : 0;
  base.want_dw = want_dw ? 1 : 0;
  base.h_tiles = p.h_tiles;
  base.active = active;
  base.n_active = n_active;
  base.kb_h = static_cast<int>(cdiv(H, kBK));
  base.mn3d = mn3d ? 1 : 0;
  base.N = static_cast<int>(N);
  base.H = static_cast<int>(H);
  base.V = static_cast<int>(V);
  base.targets = tg;
  base.lse = lg;
  base.dz[0] = dz0;
  base.dz[1] = dz1;
  base.dz_ld = static_cast<int>(p.dz_ld);
  if (dX_acc) {
    base.dxf = dxf;
    base.dx_accumulate = 1;
  } else if (dX) {
    if (dx_final)
      base.dx_final = static_cast<__nv_bfloat16*>(dX);
    else
      base.dxf = dxf;
  }
  if (dW_acc) {
    base.dw_accumulate = 1;
  } else if (dW) {
    if (dw_final)
      base.dw_final = static_cast<__nv_bfloat16*>(dW);
    else
      base.dwf = dwf;
  }
  base.grad_loss = grad_loss;
  base.n_valid = nv;
  base.reduction = red;
  base.err = err;
  base.wait_limit_ns = g_wait_limit_ns.load();
  // X tiles of a row tile are handed out `x_lag` row tiles after its R tiles:
  // about two tiles per CTA pair are in flight (one in the MMA, the next
  // being loaded), so by then the R tiles of the row tile have finished.
  {
    const int vt = static_cast<int>(cdiv(std::min<int64_t>(p.Vb, V), kBN));
    const int per_row = vt + (want_dx ? p.h_tiles : 0);
    base.x_lag = static_cast<int>(cdiv(2 * (dev.sms / 2), per_row)) + 1;
  }

  // Launch p: recompute dZ block p (R tiles) and contract it into dX (X tiles)
  // as its row tiles complete, while block p-1 is contracted into dW (W tiles).
  NvtxRange gemm_range("backward GEMM launches");
  for (int lp = 0; lp <= nblk; ++lp) {
    BwdArgs a = base;
    a.counter = counters + lp;
    int tiles = 0;  // at most this many tiles (fewer when token tiles are skipped)
    if (lp < nblk) {
      a.r = block(lp);
      a.row_done = row_done + static_cast<size_t>(lp) * tiles_per_block;
      tiles += a.r.mt * a.r.vt;
      if (want_dx) tiles += a.r.mt * p.h_tiles;
    }
    int w_vb = -1, w_nb = -1;
    bool overlap = lp >= 1;  // directly after the previous backward launch
    if (lp >= 1) {
      const int b = lp - 1;
      a.w = block(b);
      w_vb = b / p.n_blocks;
      w_nb = b % p.n_blocks;
      if (want_dw) tiles += a.w.vt * p.h_tiles;
      if (band && w_nb == 0) {
        FLCE_CUDA(cudaMemsetAsync(dwf, 0, static_cast<size_t>(a.w.vt) * kBN * H * 4, s));
        overlap = false;
      }
    }
    if (band && lp >= 2 && (lp - 2) % p.n_blocks == p.n_blocks - 1)
      overlap = false;  // a band downcast sits between this launch and the previous one
    if (lp == 0) prof_begin(s);
    FLCE_CUDA(launch_bwd_gemm(maps, a, tiles, overlap, s));
    if (band && lp >= 1 && w_nb == p.n_blocks - 1) {
      const int64_t col0 = int64_t{w_vb} * p.Vb;
      const int64_t vext = std::min<int64_t>(p.Vb, V - col0);
      FLCE_CUDA(launch_downcast(dwf, static_cast<__nv_bfloat16*>(dW) + col0 * H,
                                static_cast<size_t>(vext) * H, grad_loss, nv, red, s));
    }
  }
  prof_end(1, nblk + 1, s);
  if (dense)
    FLCE_CUDA(launch_downcast_rows(dxf, static_cast<__nv_bfloat16*>(dX), inv, static_cast<int>(N),
                                   static_cast<int>(H), grad_loss, nv, red, s));
  else if (dX && !dx_final)
    FLCE_CUDA(launch_downcast(dxf, static_cast<__nv_bfloat16*>(dX), static_cast<size_t>(N) * H,
                              grad_loss, nv, red, s));
  return FLCE_OK;
}

// A vocabulary shard: columns [v_offset, v_offset + V) of a V_total-column
// vocabulary.
flce_status check_slice(int64_t V, int64_t v_offset, int64_t V_total, VocabSlice* vs) {
  if (V <= 0 || v_offset < 0 || V_total <= 0) return FLCE_ERR_INVALID_ARG;
  if (V_total > kMaxDim) return FLCE_ERR_UNSUPPORTED_SHAPE;
  if (v_offset > V_total - V) return FLCE_ERR_INVALID_ARG;
  *vs = VocabSlice{V_total, v_offset, V};
  return FLCE_OK;
}

}  // namespace

extern "C" {

flce_status flce_forward(const void* X, const void* W, const int64_t* labels, int64_t N,
                         int64_t H, int64_t V, int64_t seq_len, int64_t ignore_index, int shift,
                         flce_reduction reduction, float* loss, float* lse, int64_t* n_valid,
                         void* workspace, size_t workspace_bytes, flce_stream_t stream) {
  return forward_impl(X, W, labels, N, H, V, VocabSlice{V, 0, V}, seq_len, ignore_index, shift,
                      reduction, loss, lse, nullptr, n_valid, workspace, workspace_bytes, stream);
}

flce_status flce_forward_vocab_shard(const void* X, const void* W_shard, const int64_t* labels,
                                     int64_t N, int64_t H, int64_t V, int64_t v_offset,
                                     int64_t V_total, int64_t seq_len, int64_t ignore_index,
                                     int shift, float* lse_shard, float* z_shard,
                                     int64_t* n_valid, void* workspace, size_t workspace_bytes,
                                     flce_stream_t stream) {
  VocabSlice vs;
  flce_status st = check_slice(V, v_offset, V_total, &vs);
  if (st != FLCE_OK) return st;
  if (N > 0 && !z_shard) return FLCE_ERR_INVALID_ARG;
  // z_out must be non-null to select the shard outputs, even for N == 0
  float dummy = 0.f;
  return forward_impl(X, W_shard, labels, N, H, V, vs, seq_len, ignore_index, shift,
                      FLCE_REDUCTION_MEAN, nullptr, lse_shard, z_shard ? z_shard : &dummy,
                      n_valid, workspace, workspace_bytes, stream);
}

flce_status flce_merge_vocab_shards(const float* lse_parts, const float* z_parts, int64_t P,
                                    const int64_t* labels, int64_t N, int64_t V_total,
                                    int64_t seq_len, int64_t ignore_index, int shift,
                                    flce_reduction reduction, float* loss, float* lse,
                                    int64_t* n_valid, void* workspace, size_t workspace_bytes,
                                    flce_stream_t stream) {
  NvtxRange range("flce_merge_vocab_shards");
  if (N < 0 || P <= 0 || P > kMaxShards || V_total <= 0) return FLCE_ERR_INVALID_ARG;
  if (N > kMaxDim || V_total > kMaxDim || P * N > kMaxDim) return FLCE_ERR_UNSUPPORTED_SHAPE;
  if (reduction != FLCE_REDUCTION_MEAN && reduction != FLCE_REDUCTION_SUM)
    return FLCE_ERR_INVALID_ARG;
  if (!loss || !n_valid || !workspace) return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (!lse_parts || !z_parts || !labels || !lse)) return FLCE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) return FLCE_ERR_INVALID_ARG;
  if (shift && N > 0) {
    const int64_t S = seq_len > 0 ? seq_len : N;
    if (N % S != 0) return FLCE_ERR_INVALID_ARG;
  }
  // layout: the error word and the targets where a forward plan keeps them,
  // then the per-block loss partials
  const size_t off_t = align_up(16);
  const size_t off_lossp = off_t + align_up(static_cast<size_t>(N) * 4);
  const size_t need = off_lossp + align_up(static_cast<size_t>(cdiv(N, 256) + 1) * 8);
  if (workspace_bytes < need) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo dev;
  flce_status st = device_info(&dev);
  if (st != FLCE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* err = reinterpret_cast<int*>(ws);
  FLCE_CUDA(cudaMemsetAsync(err, 0, 16, s));
  FLCE_CUDA(cudaMemsetAsync(n_valid, 0, sizeof(int64_t), s));
  if (N == 0) {
    FLCE_CUDA(cudaMemsetAsync(loss, 0, sizeof(float), s));
    return FLCE_OK;
  }
  int* targets = reinterpret_cast<int*>(ws + off_t);
  double* lossp = reinterpret_cast<double*>(ws + off_lossp);
  const int S = static_cast<int>(seq_len > 0 ? seq_len : N);
  FLCE_CUDA(launch_prep_targets(labels, static_cast<int>(N), S, shift, ignore_index,
                                VocabSlice{V_total, 0, V_total}, targets,
                                reinterpret_cast<long long*>(n_valid), err, s));
  int nblocks = 0;
  FLCE_CUDA(launch_merge_shards(lse_parts, z_parts, static_cast<int>(P), static_cast<int>(N),
                                targets, lse, lossp, s, &nblocks));
  FLCE_CUDA(launch_finalize_loss(lossp, nblocks, reinterpret_cast<const long long*>(n_valid),
                                 reduction == FLCE_REDUCTION_SUM ? 1 : 0, loss, s));
  return FLCE_OK;
}

flce_status flce_backward_vocab_shard(const void* X, const void* W_shard, const int64_t* labels,
                                      int64_t N, int64_t H, int64_t V, int64_t v_offset,
                                      int64_t V_total, int64_t seq_len, int64_t ignore_index,
                                      int shift, flce_reduction reduction, const float* lse,
                                      const int64_t* n_valid, const float* grad_loss,
                                      float* dX_acc, void* dW_shard, void* workspace,
                                      size_t workspace_bytes, flce_stream_t stream) {
  VocabSlice vs;
  flce_status st = check_slice(V, v_offset, V_total, &vs);
  if (st != FLCE_OK) return st;
  return backward_impl(X, W_shard, labels, N, H, V, vs, seq_len, ignore_index, shift, reduction,
                       lse, n_valid, grad_loss, nullptr, dX_acc, dW_shard, nullptr, workspace,
                       workspace_bytes, stream);
}

flce_status flce_downcast_bf16(const float* src, void* dst, int64_t count,
                               flce_stream_t stream) {
  if (count < 0 || count % 8 != 0) return FLCE_ERR_INVALID_ARG;
  if (count == 0) return FLCE_OK;
  if (!src || !dst) return FLCE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15)
    return FLCE_ERR_INVALID_ARG;
  DeviceInfo dev;
  flce_status st = device_info(&dev);
  if (st != FLCE_OK) return st;
  FLCE_CUDA(launch_downcast(src, static_cast<__nv_bfloat16*>(dst), static_cast<size_t>(count),
                            nullptr, nullptr, 0, reinterpret_cast<cudaStream_t>(stream)));
  return FLCE_OK;
}

flce_status flce_backward(const void* X, const void* W, const int64_t* labels, int64_t N,
                          int64_t H, int64_t V, int64_t seq_len, int64_t ignore_index, int shift,
                          flce_reduction reduction, const float* lse, const int64_t* n_valid,
                          const float* grad_loss, void* dX, void* dW, void* workspace,
                          size_t workspace_bytes, flce_stream_t stream) {
  return backward_impl(X, W, labels, N, H, V, VocabSlice{V, 0, V}, seq_len, ignore_index, shift,
                       reduction, lse, n_valid, grad_loss, dX, nullptr, dW, nullptr, workspace,
                       workspace_bytes, stream);
}

flce_status flce_backward_accumulate(const void* X, const void* W, const int64_t* labels,
                                     int64_t N, int64_t H, int64_t V, int64_t seq_len,
                                     int64_t ignore_index, int shift, flce_reduction reduction,
                                     const float* lse, const int64_t* n_valid,
                                     const float* grad_loss, void* dX, float* dW_acc,
                                     void* workspace, size_t workspace_bytes,
                                     flce_stream_t stream) {
  if (!dW_acc) return FLCE_ERR_INVALID_ARG;
  return backward_impl(X, W, labels, N, H, V, VocabSlice{V, 0, V}, seq_len, ignore_index, shift,
                       reduction, lse, n_valid, grad_loss, dX, nullptr, nullptr, dW_acc,
                       workspace, workspace_bytes, stream);
}

flce_status flce_logits(const void* X, const void* W, int64_t N, int64_t H, int64_t V,
                        void* logits, int64_t ld_logits, flce_stream_t stream) {
  NvtxRange range("flce_logits");
  if (N < 0 || H <= 0 || V <= 0) return FLCE_ERR_INVALID_ARG;
  if (H % 8 != 0 || H > kMaxH || N > kMaxDim || V > kMaxDim) return FLCE_ERR_UNSUPPORTED_SHAPE;
  if (N == 0) return FLCE_OK;
  if (!X || !W || !logits || ld_logits < V || ld_logits % 8 != 0) return FLCE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W) |
       reinterpret_cast<uintptr_t>(logits)) & 15)
    return FLCE_ERR_INVALID_ARG;
  DeviceInfo dev;
  flce_status st = device_info(&dev);
  if (st != FLCE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CUtensorMap tx, tw, tout;
  if (!make_tmap(&tx, X, H, N, H * 2, kBK, kBM) || !make_tmap(&tw, W, H, V, H * 2, kBK, kHalfN) ||
      !make_tmap(&tout, logits, V, N, ld_logits * 2, 64, 32))
    return FLCE_ERR_CUDA;
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.tiles_m = static_cast<int>(cdiv(N, kPairM));
  a.tiles_n = static_cast<int>(cdiv(V, kBN));
  a.group = kFwdGroup;
  a.units = a.tiles_m * static_cast<int>(cdiv(a.tiles_n, kFwdGroup));
  a.band = forward_band_tiles(a.tiles_m, H);  // units dealt round robin, band by band
  a.k_blocks = static_cast<int>(cdiv(H, kBK));
  a.N = static_cast<int>(N);
  a.H = static_cast<int>(H);
  a.V = static_cast<int>(V);
  a.wait_limit_ns = g_wait_limit_ns.load();
  FLCE_CUDA(launch_logits_gemm(tx, tw, tout, a, a.units, s));
  return FLCE_OK;
}

flce_status flce_get_error(const void* workspace, flce_stream_t stream) {
  if (!workspace) return FLCE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FLCE_ERR_CUDA;
  int e = 0;
  if (cudaMemcpy(&e, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FLCE_ERR_CUDA;
  if (e & kErrTimeout) return FLCE_ERR_TIMEOUT;
  if (e & kErrLabel) return FLCE_ERR_LABEL_OUT_OF_RANGE;
  return FLCE_OK;
}

int64_t flce_kernel_launch_count(void) { return g_launches.load(); }

int64_t flce_last_launch_wait_limit_ns(void) {
  return static_cast<int64_t>(g_last_wait_limit.load());
}

void flce_profile_enable(int enable) { g_prof_on.store(enable != 0); }

flce_status flce_profile_collect(double* ms, int64_t* launches) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (int k = 0; k < 4; ++k) {
    if (ms) ms[k] = 0.0;
    if (launches) launches[k] = 0;
  }
  flce_status st = FLCE_OK;
  for (const ProfRec& r : g_prof) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess ||
        cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      st = FLCE_ERR_CUDA;
    if (r.kind >= 0 && r.kind < 4) {
      if (ms) ms[r.kind] += t;
      if (launches) launches[r.kind] += r.launches;
    }
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_prof.clear();
  return st;
}

flce_status flce_selftest_wait_timeout(int64_t limit_ns, void* workspace, size_t workspace_bytes,
                                       flce_stream_t stream) {
  if (!workspace || workspace_bytes < 256 || limit_ns <= 0) return FLCE_ERR_INVALID_ARG;
  DeviceInfo dev;
  flce_status st = device_info(&dev);
  if (st != FLCE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* err = static_cast<int*>(workspace);
  FLCE_CUDA(cudaMemsetAsync(err, 0, 16, s));
  FLCE_CUDA(launch_selftest_wait(static_cast<unsigned long long>(limit_ns), err, s));
  return FLCE_OK;
}

}  // extern "C"
