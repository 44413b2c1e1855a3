// Small SIMT kernels around the tensor-core GEMMs: target preparation, the
// per-row log-sum-exp merge with a deterministic loss reduction, the scaled
// FP32 -> bf16 downcast of the gradients, and the bounded-wait self-test.
#include "flce_device.cuh"
#include "flce_internal.h"

namespace flce {

namespace {

constexpr int kPrepThreads = 256;  // one 256-row token tile per block
static_assert(kPrepThreads == kPairM, "prep blocks are token tiles");
constexpr int kGatherSlice = 64;   // 16-byte columns of a row per gather block (1 KB)
constexpr int kMergeThreads = 256;  // rows per block of the shard merge
constexpr int kMergeGroups = 8;     // warps per block of the log-sum-exp merge
constexpr int kFinalThreads = 256;

// Effective target of every row after the optional per-sequence shift (the
// call `linear_cross_entropy(..., ignore_index=-100, shift=True, ...)` with
// labels = input_ids in the Qwen3.5-35B-A3B LoRA SFT blog post, listings
// `_patch_model_with_cce` and `prepare_dataset`): -1 when the row has no valid
// target.  Validity is judged against the whole vocabulary [0, V_total); the
// stored target is local to the columns [v_offset, v_offset + V_local) this
// call holds, or kTargetElsewhere when it lies in another vocabulary shard.
// Counts valid rows exactly.
__global__ void prep_targets_kernel(const int64_t* __restrict__ labels, int N, int seq_len,
                                    int shift, int64_t ignore_index, int64_t V_total,
                                    int64_t v_offset, int64_t V_local,
                                    int* __restrict__ targets, unsigned long long* n_valid,
                                    int* err, int* tile_flags) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  int ok = 0;
  if (i < N) {
    int64_t lab;
    if (shift) {
      const int pos = i % seq_len;
      lab = (pos + 1 < seq_len) ? labels[i + 1] : ignore_index;
    } else {
      lab = labels[i];
    }
    int t = -1;
    if (lab != ignore_index) {
      if (lab >= 0 && lab < V_total) {
        const int64_t loc = lab - v_offset;
        t = (loc >= 0 && loc < V_local) ? static_cast<int>(loc) : kTargetElsewhere;
        ok = 1;
      } else {
        atomicOr(err, kErrLabel);
      }
    }
    targets[i] = t;
  }
  const int cnt = __syncthreads_count(ok);
  if (n_valid && threadIdx.x == 0 && cnt) atomicAdd(n_valid, static_cast<unsigned long long>(cnt));
  // a block is one 256-row token tile: its count of rows with a valid target
  if (tile_flags && threadIdx.x == 0) tile_flags[blockIdx.x] = cnt;
}

// Block sum of the rows' losses in a fixed tree order (FP64), written by
// thread 0 to loss_partials[blockIdx.x].
__device__ __forceinline__ void block_loss_sum(double row_loss, double* red,
                                               double* __restrict__ loss_partials) {
  red[threadIdx.x] = row_loss;
  __syncthreads();
  for (int s = kMergeThreads / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) loss_partials[blockIdx.x] = red[0];
}

// lse_i = M + log sum_k s_k exp(m_k - M) over the forward's per-unit partials
// (m_k, s_k); row loss = lse_i - z_{i,t_i} for valid rows.  A block takes
// kMergeRows rows; each of its kMergeGroups warps merges every kMergeGroups-th
// partial of those rows in one pass (a running max and rescaled sum; the
// reads of a warp are 32 consecutive rows of one partial), then the first warp
// combines the groups and writes the FP64 sum of its rows' losses (fixed
// order).  With z_out (a vocabulary shard), lse is this shard's log-sum-exp,
// z_out its target logit (0 where the target lies in another shard) and no
// loss is formed.
__global__ void __launch_bounds__(kMergeRows * kMergeGroups)
    merge_lse_kernel(const float2* __restrict__ partials, int nchunks, int N,
                     const float* __restrict__ zt, const int* __restrict__ targets,
                     float* __restrict__ lse, double* __restrict__ loss_partials,
                     float* __restrict__ z_out) {
  __shared__ float2 grp[kMergeGroups][kMergeRows];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int i = blockIdx.x * kMergeRows + tx;
  float m = -INFINITY, sum = 0.f;
  if (i < N) {
    // every partial has a finite max (each unit holds at least one column)
    for (int k = ty; k < nchunks; k += kMergeGroups) {
      const float2 p = partials[static_cast<size_t>(k) * N + i];
      if (p.x > m) {
        sum = sum * expf(m - p.x) + p.y;
        m = p.x;
      } else {
        sum += p.y * expf(p.x - m);
      }
    }
  }
  grp[ty][tx] = make_float2(m, sum);
  __syncthreads();
  if (ty != 0) return;
  double row_loss = 0.0;
  if (i < N) {
    float M = grp[0][tx].x;
#pragma unroll
    for (int g = 1; g < kMergeGroups; ++g) M = fmaxf(M, grp[g][tx].x);
    float S = 0.f;
#pragma unroll
    for (int g = 0; g < kMergeGroups; ++g) {
      const float2 q = grp[g][tx];
      if (q.y != 0.f) S += q.y * expf(q.x - M);
    }
    const float l = M + logf(S);
    lse[i] = l;
    const int t = targets[i];
    const bool here = t >= 0 && t != kTargetElsewhere;
    if (z_out) z_out[i] = here ? zt[i] : 0.f;
    else if (here) row_loss = static_cast<double>(l) - static_cast<double>(zt[i]);
  }
  if (z_out) return;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) row_loss += __shfl_down_sync(0xffffffffu, row_loss, off);
  if (tx == 0) loss_partials[blockIdx.x] = row_loss;
}

// Merge of P vocabulary shards (Megatron-LM PR #2739, section 1: the vocabulary
// rows of the output layer are split across ranks): lse_i = log sum_r
// exp(lse_r,i) and z_i = sum_r z_r,i (one shard holds a valid target, the
// others give 0); row loss = lse_i - z_i for valid rows.
__global__ void merge_shards_kernel(const float* __restrict__ lse_parts,
                                    const float* __restrict__ z_parts, int P, int N,
                                    const int* __restrict__ targets, float* __restrict__ lse,
                                    double* __restrict__ loss_partials) {
  __shared__ double red[kMergeThreads];
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  double row_loss = 0.0;
  if (i < N) {
    float M = -INFINITY;
    for (int r = 0; r < P; ++r) M = fmaxf(M, lse_parts[static_cast<size_t>(r) * N + i]);
    float S = 0.f, z = 0.f;
    for (int r = 0; r < P; ++r) {
      S += expf(lse_parts[static_cast<size_t>(r) * N + i] - M);
      z += z_parts[static_cast<size_t>(r) * N + i];
    }
    const float l = M + logf(S);
    lse[i] = l;
    if (targets[i] >= 0) row_loss = static_cast<double>(l) - static_cast<double>(z);
  }
  block_loss_sum(row_loss, red, loss_partials);
}

// Sum of the block partials in a fixed order; mean divides by n_valid
// (0 when there is no valid target).
__global__ void finalize_loss_kernel(const double* __restrict__ loss_partials, int nblocks,
                                     const long long* __restrict__ n_valid, int reduction,
                                     float* __restrict__ loss) {
  __shared__ double red[kFinalThreads];
  double acc = 0.0;
  for (int b = threadIdx.x; b < nblocks; b += kFinalThreads) acc += loss_partials[b];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = kFinalThreads / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    double v = red[0];
    if (reduction == 0) {
      const long long n = *n_valid;
      v = n > 0 ? v / static_cast<double>(n) : 0.0;
    }
    *loss = static_cast<float>(v);
  }
}

// dst = bf16_rn(scale * src), scale = g / n_valid (mean) or g (sum), or 1
// without grad_loss: the FP32 buffer is rounded to bf16 once, after
// accumulation (Megatron-LM PR #2739, section 2).  Eight elements per thread;
// count is a multiple of 8.
__global__ void downcast_kernel(const float4* __restrict__ src, uint4* __restrict__ dst,
                                size_t count8, const float* __restrict__ grad_loss,
                                const long long* __restrict__ n_valid, int reduction) {
  float scale = grad_loss ? *grad_loss : 1.f;
  if (grad_loss && reduction == 0) {
    const long long n = *n_valid;
    scale = n > 0 ? scale / static_cast<float>(n) : 0.f;
  }
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < count8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 a = src[2 * i], b = src[2 * i + 1];
    __nv_bfloat162 p0 = __floats2bfloat162_rn(scale * a.x, scale * a.y);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(scale * a.z, scale * a.w);
    __nv_bfloat162 p2 = __floats2bfloat162_rn(scale * b.x, scale * b.y);
    __nv_bfloat162 p3 = __floats2bfloat162_rn(scale * b.z, scale * b.w);
    dst[i] = make_uint4(*reinterpret_cast<uint32_t*>(&p0), *reinterpret_cast<uint32_t*>(&p1),
                        *reinterpret_cast<uint32_t*>(&p2), *reinterpret_cast<uint32_t*>(&p3));
  }
}

// Lists the flagged tiles in ascending order (one block; a block-wide scan
// per 1024 tiles).
__global__ void compact_tiles_kernel(const int* __restrict__ flags, int m_tiles,
                                     int* __restrict__ active, int* __restrict__ n_active) {
  __shared__ int scan[1024];
  int base = 0;
  for (int t0 = 0; t0 < m_tiles; t0 += 1024) {
    const int t = t0 + threadIdx.x;
    const int f = (t < m_tiles && flags[t]) ? 1 : 0;
    scan[threadIdx.x] = f;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {  // inclusive Hillis-Steele scan
      const int v = threadIdx.x >= off ? scan[threadIdx.x - off] : 0;
      __syncthreads();
      scan[threadIdx.x] += v;
      __syncthreads();
    }
    if (f) active[base + scan[threadIdx.x] - 1] = t;
    base += scan[1023];
    __syncthreads();
  }
  if (threadIdx.x == 0) *n_active = base;
}

// Offsets of each tile's valid rows in the dense row order (an exclusive scan
// of the per-tile counts; toff[m_tiles] = all valid rows), and the dense
// row tiles as the backward's tile list: tiles 0 .. ceil(rows / 256) - 1.
// One block; a block-wide scan per 1024 tiles.
__global__ void compact_rows_kernel(const int* __restrict__ counts, int m_tiles,
                                    int* __restrict__ toff, int* __restrict__ active,
                                    int* __restrict__ n_active) {
  __shared__ int scan[1024];
  int base = 0;
  for (int t0 = 0; t0 < m_tiles; t0 += 1024) {
    const int t = t0 + threadIdx.x;
    const int c = t < m_tiles ? counts[t] : 0;
    scan[threadIdx.x] = c;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {  // inclusive Hillis-Steele scan
      const int v = threadIdx.x >= off ? scan[threadIdx.x - off] : 0;
      __syncthreads();
      scan[threadIdx.x] += v;
      __syncthreads();
    }
    if (t < m_tiles) toff[t] = base + scan[threadIdx.x] - c;
    base += scan[1023];
    __syncthreads();
  }
  const int tiles = (base + kPairM - 1) / kPairM;
  for (int t = threadIdx.x; t < tiles; t += blockDim.x) active[t] = t;
  if (threadIdx.x == 0) {
    toff[m_tiles] = base;
    *n_active = tiles;
  }
}

// The rows with a valid target, in order, copied to the front of a dense
// [N][H] bf16 buffer, with their targets and lse beside them; the rows after
// the last one, to the end of its 256-row tile (and not past N), are zeroed
// (target -1: dZ = 0, and X = 0 so that the dW contraction stays finite).
// inv maps every row to its dense index, or -1.  A row without a valid target
// has no term in the loss (the ignore_index call of the Qwen3.5-35B-A3B LoRA
// SFT blog post, listing `_patch_model_with_cce`), so its dZ row is 0 and it
// adds nothing to dX or dW: the backward runs on the dense rows only.
// Block (b, y): token tile b,
// 16-byte columns [64 y, 64 y + 64) of each row; block (b, 0) also writes the
// per-row arrays.
__global__ void __launch_bounds__(kPairM)
    gather_rows_kernel(const uint4* __restrict__ X, const int* __restrict__ targets,
                       const float* __restrict__ lse, const int* __restrict__ toff, int N,
                       int H8, int m_tiles, uint4* __restrict__ xc, int* __restrict__ tc,
                       float* __restrict__ lc, int* __restrict__ inv) {
  __shared__ int rows[kPairM];
  __shared__ int warp_cnt[kPairM / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = blockIdx.x * kPairM + tid;
  const int t = i < N ? targets[i] : -1;
  const bool valid = t != -1;
  const unsigned m = __ballot_sync(0xffffffffu, valid);
  if (lane == 0) warp_cnt[warp] = __popc(m);
  __syncthreads();
  int before = 0, cnt = 0;
  for (int w = 0; w < kPairM / 32; ++w) {
    before += w < warp ? warp_cnt[w] : 0;
    cnt += warp_cnt[w];
  }
  const int rank = before + __popc(m & ((1u << lane) - 1u));
  const int j0 = toff[blockIdx.x];
  if (valid) rows[rank] = i;
  if (blockIdx.y == 0) {
    if (i < N) inv[i] = valid ? j0 + rank : -1;
    if (valid) {
      tc[j0 + rank] = t;
      lc[j0 + rank] = lse[i];
    }
  }
  __syncthreads();
  const int c0 = blockIdx.y * kGatherSlice;
  const int width = min(H8, c0 + kGatherSlice) - c0;
  // (row, column) pairs of the slice, four loads in flight per thread
  const int total = cnt * width;
  for (int e0 = tid; e0 < total; e0 += 4 * kPairM) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u * kPairM;
      if (e < total)
        v[u] = X[static_cast<size_t>(rows[e / width]) * H8 + c0 + e % width];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u * kPairM;
      if (e < total) xc[static_cast<size_t>(j0 + e / width) * H8 + c0 + e % width] = v[u];
    }
  }
  const int rows_total = toff[m_tiles];
  const int pad_end = min(N, (rows_total + kPairM - 1) / kPairM * kPairM);
  for (int j = rows_total + blockIdx.x; j < pad_end; j += gridDim.x) {
    for (int c = c0 + tid; c < c0 + width; c += kPairM)
      xc[static_cast<size_t>(j) * H8 + c] = make_uint4(0, 0, 0, 0);
    if (blockIdx.y == 0 && tid == 0) {
      tc[j] = -1;
      lc[j] = 0.f;
    }
  }
}

// dX row i = bf16_rn(scale * src[inv[i]]) for the rows the backward ran on
// (scale as in downcast_kernel), 0 for the others: the dense rows' FP32
// accumulator put back in token order.  A block per row at a time.
__global__ void downcast_rows_kernel(const float4* __restrict__ src, uint4* __restrict__ dst,
                                     const int* __restrict__ inv, int N, int H8,
                                     const float* __restrict__ grad_loss,
                                     const long long* __restrict__ n_valid, int reduction) {
  float scale = grad_loss ? *grad_loss : 1.f;
  if (grad_loss && reduction == 0) {
    const long long n = *n_valid;
    scale = n > 0 ? scale / static_cast<float>(n) : 0.f;
  }
  for (int row = blockIdx.x; row < N; row += gridDim.x) {
    const int j = inv[row];
    uint4* d = dst + static_cast<size_t>(row) * H8;
    if (j < 0) {
      for (int c = threadIdx.x; c < H8; c += blockDim.x) d[c] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const float4* sr = src + static_cast<size_t>(j) * H8 * 2;
    for (int c = threadIdx.x; c < H8; c += blockDim.x) {
      const float4 a = sr[2 * c], b = sr[2 * c + 1];
      __nv_bfloat162 p0 = __floats2bfloat162_rn(scale * a.x, scale * a.y);
      __nv_bfloat162 p1 = __floats2bfloat162_rn(scale * a.z, scale * a.w);
      __nv_bfloat162 p2 = __floats2bfloat162_rn(scale * b.x, scale * b.y);
      __nv_bfloat162 p3 = __floats2bfloat162_rn(scale * b.z, scale * b.w);
      d[c] = make_uint4(*reinterpret_cast<uint32_t*>(&p0), *reinterpret_cast<uint32_t*>(&p1),
                        *reinterpret_cast<uint32_t*>(&p2), *reinterpret_cast<uint32_t*>(&p3));
    }
  }
}

// Waits on a barrier that nothing will ever complete; the bounded wait must
// give up, record the timeout and let the kernel return.
__global__ void selftest_wait_kernel(unsigned long long limit_ns, int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0u;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
    WaitCtx w{&abort_flag, err, limit_ns};
    wait_parity(smem_u32(&bar), 0u, w);
  }
}

}  // namespace

cudaError_t launch_prep_targets(const int64_t* labels, int N, int seq_len, int shift,
                                int64_t ignore_index, const VocabSlice& vs, int* targets,
                                long long* n_valid, int* err, cudaStream_t st, int* tile_flags) {
  if (N <= 0) return cudaSuccess;
  const int blocks = (N + kPrepThreads - 1) / kPrepThreads;
  prep_targets_kernel<<<blocks, kPrepThreads, 0, st>>>(
      labels, N, seq_len, shift, ignore_index, vs.V_total, vs.v_offset, vs.V_local, targets,
      reinterpret_cast<unsigned long long*>(n_valid), err, tile_flags);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_merge_lse(const float2* partials, int nchunks, int N, const float* zt,
                             const int* targets, float* lse, double* loss_partials,
                             cudaStream_t st, int* nblocks_out, float* z_out) {
  const int blocks = (N + kMergeRows - 1) / kMergeRows;
  *nblocks_out = blocks;
  if (blocks == 0) return cudaSuccess;
  merge_lse_kernel<<<blocks, dim3(kMergeRows, kMergeGroups), 0, st>>>(
      partials, nchunks, N, zt, targets, lse, loss_partials, z_out);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_merge_shards(const float* lse_parts, const float* z_parts, int P, int N,
                                const int* targets, float* lse, double* loss_partials,
                                cudaStream_t st, int* nblocks_out) {
  const int blocks = (N + kMergeThreads - 1) / kMergeThreads;
  *nblocks_out = blocks;
  if (blocks == 0) return cudaSuccess;
  merge_shards_kernel<<<blocks, kMergeThreads, 0, st>>>(lse_parts, z_parts, P, N, targets, lse,
                                                        loss_partials);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_finalize_loss(const double* loss_partials, int nblocks,
                                 const long long* n_valid, int reduction, float* loss,
                                 cudaStream_t st) {
  finalize_loss_kernel<<<1, kFinalThreads, 0, st>>>(loss_partials, nblocks, n_valid, reduction,
                                                    loss);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_downcast(const float* src, __nv_bfloat16* dst, size_t count,
                            const float* grad_loss, const long long* n_valid, int reduction,
                            cudaStream_t st) {
  const size_t count8 = count / 8;
  if (count8 == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t want = (count8 + 255) / 256;
  const int blocks = static_cast<int>(want < static_cast<size_t>(sms) * 8 ? want : sms * 8);
  downcast_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(src),
                                          reinterpret_cast<uint4*>(dst), count8, grad_loss,
                                          n_valid, reduction);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_compact_tiles(const int* tile_flags, int m_tiles, int* active, int* n_active,
                                 cudaStream_t st) {
  compact_tiles_kernel<<<1, 1024, 0, st>>>(tile_flags, m_tiles, active, n_active);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_compact_rows(const int* counts, int m_tiles, int* toff, int* active,
                                int* n_active, cudaStream_t st) {
  compact_rows_kernel<<<1, 1024, 0, st>>>(counts, m_tiles, toff, active, n_active);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* X, const int* targets, const float* lse,
                               const int* toff, int N, int H, int m_tiles, void* xc, int* tc,
                               float* lc, int* inv, cudaStream_t st) {
  if (N <= 0 || m_tiles <= 0) return cudaSuccess;
  const int H8 = H / 8;
  const dim3 grid(m_tiles, (H8 + kGatherSlice - 1) / kGatherSlice);
  gather_rows_kernel<<<grid, kPairM, 0, st>>>(static_cast<const uint4*>(X), targets, lse, toff,
                                              N, H8, m_tiles, static_cast<uint4*>(xc), tc, lc,
                                              inv);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_downcast_rows(const float* src, __nv_bfloat16* dst, const int* inv, int N,
                                 int H, const float* grad_loss, const long long* n_valid,
                                 int reduction, cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int blocks = N < sms * 16 ? N : sms * 16;
  downcast_rows_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(src),
                                               reinterpret_cast<uint4*>(dst), inv, N, H / 8,
                                               grad_loss, n_valid, reduction);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(unsigned long long limit_ns, int* err, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(limit_ns, err);
  note_launch();
  return cudaGetLastError();
}

}  // namespace flce
