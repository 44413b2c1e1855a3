// flce_forward_noalloc: the forward pass with its scratch in a fixed,
// file-scope device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory at all: code that runs as a
// plugin inside a host framework which owns every device allocation and hands
// the plugin only its input and output buffers, or code on a latency-critical
// path where cudaMalloc / cudaFree (which synchronise the device) are not
// allowed.  For them this entry point needs nothing but the inputs and the
// outputs.  It launches the same kernels as flce_forward; only where the
// scratch lives differs.
//
// The scratch array (kNoallocScratchBytes) is part of the library's device
// image, so every GPU that loads the library holds it until the process exits.
// All calls share it and it keeps the last call's contents; the parts that must
// start at zero (the error word) are cleared by each call.  Calls whose work
// overlaps on the GPU (different streams, or different host threads without
// ordering) race on the shared scratch and must be serialised by the caller.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "../../include/flce.h"
#include "flce_internal.h"

namespace flce {
namespace {

constexpr size_t kNoallocScratchBytes = size_t{16} << 20;  // 16 MiB
constexpr size_t kNoallocAlign = 256;
constexpr int kMaxDevices = 64;

// Device-side scratch.  In host code this name is only a host-side stand-in
// for the symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

size_t up(size_t x) { return (x + kNoallocAlign - 1) / kNoallocAlign * kNoallocAlign; }

// Once per device, with that device current: device address of the scratch
// and the compute-capability check.
flce_status setup_device(int dev, void** scratch) {
  if (dev < 0 || dev >= kMaxDevices) return FLCE_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FLCE_ERR_CUDA;
    if (major != 10 || minor != 3) return FLCE_ERR_UNSUPPORTED_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return FLCE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *scratch = g_scratch_addr[dev];
  return FLCE_OK;
}

}  // namespace
}  // namespace flce

using namespace flce;

extern "C" flce_status flce_forward_noalloc(const void* X, const void* W, const int64_t* labels,
                                            int64_t N, int64_t H, int64_t V, int64_t seq_len,
                                            int64_t ignore_index, int shift,
                                            flce_reduction reduction, float* loss, float* lse,
                                            int64_t* n_valid, int* device_error,
                                            flce_stream_t stream) {
  if (N < 0 || H <= 0 || V <= 0) return FLCE_ERR_INVALID_ARG;
  if (reduction != FLCE_REDUCTION_MEAN && reduction != FLCE_REDUCTION_SUM)
    return FLCE_ERR_INVALID_ARG;
  if (H % 8 != 0 || H > (1 << 16) || N > (int64_t{1} << 30) || V > (int64_t{1} << 30))
    return FLCE_ERR_UNSUPPORTED_SHAPE;
  if (N > 0 && (!X || !W || !labels || !lse)) return FLCE_ERR_INVALID_ARG;
  if (!loss || !n_valid) return FLCE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W)) & 15)
    return FLCE_ERR_INVALID_ARG;
  if (shift && N > 0) {
    const int64_t S = seq_len > 0 ? seq_len : N;
    if (N % S != 0) return FLCE_ERR_INVALID_ARG;
  }
  // scratch layout (each piece starts on a 256-byte boundary): error word |
  // targets | target logits | lse partials | loss partials | unit counter
  const int64_t m_tiles = (N + kPairM - 1) / kPairM;
  const int64_t v_tiles = (V + kBN - 1) / kBN;
  const int group = forward_unit_tiles(v_tiles);
  const int64_t v_units = (v_tiles + group - 1) / group;
  const size_t off_t = up(16);
  const size_t off_zt = off_t + up(static_cast<size_t>(N) * 4);
  const size_t off_part = off_zt + up(static_cast<size_t>(N) * 4);
  const size_t off_lossp = off_part + up(static_cast<size_t>(v_units) * N * 8);
  const size_t off_cnt =
      off_lossp + up(static_cast<size_t>((N + kMergeRows - 1) / kMergeRows + 1) * 8);
  const size_t need = off_cnt + up(4);
  if (need > kNoallocScratchBytes) return FLCE_ERR_WORKSPACE_TOO_SMALL;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLCE_ERR_CUDA;
  void* scratch = nullptr;
  flce_status st = setup_device(dev, &scratch);
  if (st != FLCE_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(scratch);
  int* err = reinterpret_cast<int*>(base);
  if (cudaMemsetAsync(err, 0, 16, s) != cudaSuccess) return FLCE_ERR_CUDA;
  if (cudaMemsetAsync(n_valid, 0, sizeof(int64_t), s) != cudaSuccess) return FLCE_ERR_CUDA;
  if (N == 0) {
    if (cudaMemsetAsync(loss, 0, sizeof(float), s) != cudaSuccess) return FLCE_ERR_CUDA;
  } else {
    int* targets = reinterpret_cast<int*>(base + off_t);
    float* zt = reinterpret_cast<float*>(base + off_zt);
    float2* part = reinterpret_cast<float2*>(base + off_part);
    double* lossp = reinterpret_cast<double*>(base + off_lossp);
    int* counter = reinterpret_cast<int*>(base + off_cnt);
    if (cudaMemsetAsync(counter, 0, 4, s) != cudaSuccess) return FLCE_ERR_CUDA;
    const int S = static_cast<int>(seq_len > 0 ? seq_len : N);
    if (launch_prep_targets(labels, static_cast<int>(N), S, shift, ignore_index,
                            VocabSlice{V, 0, V}, targets, reinterpret_cast<long long*>(n_valid),
                            err, s) != cudaSuccess)
      return FLCE_ERR_CUDA;
    CUtensorMap tx, tw;
    if (!make_tmap(&tx, X, H, N, H * 2, kBK, kBM) ||
        !make_tmap(&tw, W, H, V, H * 2, kBK, kHalfN))
      return FLCE_ERR_CUDA;
    GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    a.tiles_m = static_cast<int>(m_tiles);
    a.tiles_n = static_cast<int>(v_tiles);
    a.group = group;
    a.units = static_cast<int>(m_tiles * v_units);
    a.band = forward_band_tiles(m_tiles, H);
    a.k_blocks = static_cast<int>((H + kBK - 1) / kBK);
    a.N = static_cast<int>(N);
    a.H = static_cast<int>(H);
    a.V = static_cast<int>(V);
    a.targets = targets;
    a.partials = part;
    a.zt = zt;
    a.counter = counter;
    a.err = err;
    a.wait_limit_ns = wait_limit_ns();  // flce_set_wait_limit_ns applies here too
    if (launch_fwd_gemm(tx, tw, a, a.units, s) != cudaSuccess)
      return FLCE_ERR_CUDA;
    int nblocks = 0;
    if (launch_merge_lse(part, static_cast<int>(v_units), static_cast<int>(N), zt, targets, lse,
                         lossp, s, &nblocks) != cudaSuccess ||
        launch_finalize_loss(lossp, nblocks, reinterpret_cast<const long long*>(n_valid),
                             reduction == FLCE_REDUCTION_SUM ? 1 : 0, loss, s) != cudaSuccess)
      return FLCE_ERR_CUDA;
  }
  if (device_error &&
      cudaMemcpyAsync(device_error, err, sizeof(int), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return FLCE_ERR_CUDA;
  return FLCE_OK;
}
