// Persistent tcgen05 GEMM kernels for the fused linear cross-entropy.
//
// Tile kinds (see GemmKind):
//   FWD  Z = X W^T, epilogue: online log-sum-exp over the tile's vocab columns
//        and the target-logit gather (the vocabulary split of Megatron-LM PR
//        #2739 "[Dev] Fix Linear-Cross-Entropy Convergence Issue", section 2,
//        done per tile in FP32 instead of per slice in bf16).
//   R    Z = X W^T recomputed, epilogue: dZ = exp(Z - lse) - onehot(t) in FP32,
//        rounded to bf16 into a bounded dZ block (never N x V).
//   X    dX += dZ_block W_block   (dX = dZ W, ms-swift PR #9784, section
//        Mathematical Equivalence), FP32 accumulate.
//   W    dW += dZ_block^T X_block (dW = dZ^T X, same section), FP32 accumulate.
//
// Two kernels share the building blocks below:
//   flce_fwd_kernel  forward; static round-robin over work units of 4 vocab
//                    tiles of one row tile, so the epilogue can merge the
//                    log-sum-exp of 1024 columns before writing a partial.
//   flce_bwd_kernel  backward; one launch holds the R tiles of dZ block p and
//                    the W and X tiles of block p-1 (two dZ slots, so the
//                    tiles of one launch never depend on each other).  Tiles
//                    are handed out by a global atomic ticket, longest first
//                    (W, then R, then X).
//
// CTA layout (192 threads, one CTA per SM, persistent):
//   warp 0      TMA producer: 4-stage ring of (A 128x64, B 256x64) bf16 tiles,
//               128-byte swizzled, completion counted on mbarriers.  In the
//               backward it also takes the tickets and passes them to the other
//               warps through a small shared-memory ring.
//   warp 1      allocates 512 TMEM columns; one lane issues tcgen05.mma
//               (M=128, N=256, K=16) into one of two FP32 accumulators.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (warp w owns TMEM lanes
//               32*(w%4) .. +31, i.e. tile rows), then the kind's epilogue.
// The accumulator is double-buffered so the epilogue of tile i overlaps the
// MMAs of tile i+1.
#include "flce_device.cuh"
#include "flce_internal.h"

namespace flce {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTicketRing = 4;

struct Smem {
  uint32_t a_base, b_base;  // shared addresses of stage 0 (1024-aligned)
  uint32_t full, empty;     // barrier arrays (stage-indexed, 8 bytes apart)
  uint32_t tfull, tempty;   // accumulator barriers (2 each)
  uint32_t drain;           // MMA drain barrier
  uint32_t qfull, qempty;   // ticket ring barriers
  volatile int* tickets;    // ticket ring
  uint32_t* tmem_slot;
  volatile uint32_t* abort_flag;
};

// Carves the dynamic shared memory: stages, then barriers, then small slots.
__device__ Smem carve_smem(uint8_t* smem_raw) {
  Smem s;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  s.a_base = base;
  s.b_base = base + kStages * kAStageBytes;
  const uint32_t bar0 = s.b_base + kStages * kBStageBytes;
  s.full = bar0;
  s.empty = s.full + 8 * kStages;
  s.tfull = s.empty + 8 * kStages;
  s.tempty = s.tfull + 8 * kNumAcc;
  s.drain = s.tempty + 8 * kNumAcc;
  s.qfull = s.drain + 8;
  s.qempty = s.qfull + 8 * kTicketRing;
  const uint32_t tail = s.qempty + 8 * kTicketRing;
  uint8_t* g = smem_raw + (tail - raw);
  s.tickets = reinterpret_cast<volatile int*>(g);
  s.tmem_slot = reinterpret_cast<uint32_t*>(g + 4 * kTicketRing);
  s.abort_flag = reinterpret_cast<volatile uint32_t*>(g + 4 * kTicketRing + 4);
  return s;
}

__device__ void init_barriers(const Smem& s) {
  for (int i = 0; i < kStages; ++i) {
    mbar_init(s.full + 8 * i, 1);
    mbar_init(s.empty + 8 * i, 1);
  }
  for (int i = 0; i < kNumAcc; ++i) {
    mbar_init(s.tfull + 8 * i, 1);
    mbar_init(s.tempty + 8 * i, 4);
  }
  mbar_init(s.drain, 1);
  for (int i = 0; i < kTicketRing; ++i) {
    mbar_init(s.qfull + 8 * i, 1);
    mbar_init(s.qempty + 8 * i, 1 + 4);  // the MMA lane and the 4 epilogue warps
  }
  *s.abort_flag = 0u;
  fence_barrier_init();
  fence_proxy_async_smem();
}

struct Ring {
  uint32_t idx = 0, phase = 0;
  template <int N>
  __device__ void advance() {
    if (++idx == N) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float grad_scale(const float* grad_loss, const long long* n_valid,
                                            int reduction) {
  const float g = *grad_loss;
  if (reduction == 1) return g;
  const long long n = *n_valid;
  return n > 0 ? g / static_cast<float>(n) : 0.f;
}

// ------------------------------------------------------- k-block operand loads
// A 128x64 and B 256x64 for Z = X W^T (FWD and R): both K-major.
__device__ __forceinline__ void load_xw(const CUtensorMap* tx, const CUtensorMap* tw, uint32_t sa,
                                        uint32_t sb, int k, int arow, int brow, uint32_t full) {
  tma_load_2d(sa, tx, k, arow, full);
  tma_load_2d(sb, tw, k, brow, full);
}
// dX tile: A = dZ rows (K-major over vocab), B = W rows of the block (MN-major over H).
__device__ __forceinline__ void load_dx(const CUtensorMap* tdz, const CUtensorMap* twmn,
                                        uint32_t sa, uint32_t sb, int k, int m0, int h0,
                                        int vrow0, uint32_t full) {
  tma_load_2d(sa, tdz, k, m0, full);
#pragma unroll
  for (int q = 0; q < 4; ++q) tma_load_2d(sb + q * 8192, twmn, h0 + 64 * q, vrow0 + k, full);
}
// dW tile: A = dZ^T (MN-major over vocab), B = X rows of the block (MN-major over H).
__device__ __forceinline__ void load_dw(const CUtensorMap* tdzmn, const CUtensorMap* txmn,
                                        uint32_t sa, uint32_t sb, int k, int v0, int h0,
                                        int trow0, uint32_t full) {
#pragma unroll
  for (int q = 0; q < 2; ++q) tma_load_2d(sa + q * 8192, tdzmn, v0 + 64 * q, k, full);
#pragma unroll
  for (int q = 0; q < 4; ++q) tma_load_2d(sb + q * 8192, txmn, h0 + 64 * q, trow0 + k, full);
}

// ------------------------------------------------------- MMA of one k-block
// K-major: the 16-element K step is 32 bytes inside the swizzled row.
// MN-major: it is two 8-row core-matrix groups, 2048 bytes; 64-element groups
// along M/N are 8192 bytes apart (one 64x64 TMA box each).
template <bool A_MN, bool B_MN>
__device__ __forceinline__ void mma_kblock(uint32_t d, uint32_t sa, uint32_t sb, bool first) {
  constexpr uint32_t idesc = instr_desc_bf16(kBM, kBN, A_MN, B_MN);
#pragma unroll
  for (int k = 0; k < kBK / kUmmaK; ++k) {
    const uint64_t ad = A_MN ? smem_desc_sw128(sa + k * 2048, 8192, 1024)
                             : smem_desc_sw128(sa + k * 32, 0, 1024);
    const uint64_t bd = B_MN ? smem_desc_sw128(sb + k * 2048, 8192, 1024)
                             : smem_desc_sw128(sb + k * 32, 0, 1024);
    mma_bf16(d, ad, bd, idesc, (first && k == 0) ? 0u : 1u);
  }
}

// Runs the MMAs of one tile into accumulator d; false if aborted.
template <bool A_MN, bool B_MN>
__device__ bool mma_tile(uint32_t d, int k_blocks, const Smem& s, Ring& pipe, const WaitCtx& w) {
  for (int kb = 0; kb < k_blocks; ++kb) {
    if (!wait_parity(s.full + 8 * pipe.idx, pipe.phase, w)) return false;
    tc_fence_after();
    mma_kblock<A_MN, B_MN>(d, s.a_base + pipe.idx * kAStageBytes,
                           s.b_base + pipe.idx * kBStageBytes, kb == 0);
    mma_commit(s.empty + 8 * pipe.idx);  // frees the stage once these MMAs have read it
    pipe.advance<kStages>();
  }
  return true;
}

// ------------------------------------------------------- epilogues (one tile)
// Online log-sum-exp over this tile's columns, carried in (run_m, run_s).
__device__ __forceinline__ void epi_lse(uint32_t tbase, int n0, int V, int t, float* zt_row,
                                        float& run_m, float& run_s) {
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    const int j0 = n0 + 32 * c;
    if (j0 >= V) break;  // warp-uniform
    float v[32];
    tmem_ld32(tbase + 32 * c, v);
    if (j0 + 32 > V) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (j0 + i >= V) v[i] = -INFINITY;
    }
    float cm = v[0];
#pragma unroll
    for (int i = 1; i < 32; ++i) cm = fmaxf(cm, v[i]);
    const float nm = fmaxf(run_m, cm);
    const float nm2 = nm * kLog2e;
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) sum += exp2f(fmaf(v[i], kLog2e, -nm2));
    run_s = fmaf(run_s, exp2f(fmaf(run_m, kLog2e, -nm2)), sum);
    run_m = nm;
    if (static_cast<unsigned>(t - j0) < 32u) {
      float z = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (t - j0 == i) z = v[i];
      *zt_row = z;
    }
  }
}

// dZ = exp(Z - lse) - [j == t] (0 for ignored rows and columns >= V), bf16.
__device__ __forceinline__ void epi_dz(uint32_t tbase, int gcol0, int V, int t, float lse2,
                                       __nv_bfloat16* out) {
  const bool valid_row = t >= 0;
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    float v[32];
    tmem_ld32(tbase + 32 * c, v);
    const int j0 = gcol0 + 32 * c;
    uint32_t p[16];
    if (valid_row) {
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float d0 = exp2f(fmaf(v[i], kLog2e, -lse2));
        float d1 = exp2f(fmaf(v[i + 1], kLog2e, -lse2));
        if (j0 + i == t) d0 -= 1.f;
        if (j0 + i + 1 == t) d1 -= 1.f;
        if (j0 + i >= V) d0 = 0.f;
        if (j0 + i + 1 >= V) d1 = 0.f;
        p[i / 2] = pack_bf16x2(d0, d1);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) p[i] = 0u;
    }
    uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
  }
}

// FP32 reduce-add of one accumulator row into acc_row[h0 ...], or, when
// final_row is set, bf16(scale * value) stored there.
__device__ __forceinline__ void epi_acc(uint32_t tbase, int h0, int H, bool row_ok,
                                        float* acc_row, __nv_bfloat16* final_row, float scale) {
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    const int h = h0 + 32 * c;
    if (h >= H) break;  // warp-uniform
    float v[32];
    tmem_ld32(tbase + 32 * c, v);
    if (!row_ok) continue;
    if (final_row) {
      __nv_bfloat16* o = final_row + h;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (h + 8 * i < H) {
          uint4 pk = make_uint4(pack_bf16x2(scale * v[8 * i], scale * v[8 * i + 1]),
                                pack_bf16x2(scale * v[8 * i + 2], scale * v[8 * i + 3]),
                                pack_bf16x2(scale * v[8 * i + 4], scale * v[8 * i + 5]),
                                pack_bf16x2(scale * v[8 * i + 6], scale * v[8 * i + 7]));
          *reinterpret_cast<uint4*>(o + 8 * i) = pk;
        }
      }
    } else {
      float* o = acc_row + h;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (h + 4 * i < H)
          atomicAdd(reinterpret_cast<float4*>(o + 4 * i),
                    make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
      }
    }
  }
}

// Producer teardown: every stage's most recent load must have landed before
// the CTA may exit (its shared memory is the copy's destination).
__device__ void drain_loads(const Smem& s, uint32_t issued, const Ring& pipe, const WaitCtx& w0) {
  WaitCtx wd = w0;
  volatile uint32_t never = 0u;
  wd.abort = &never;  // keep waiting (bounded) even if the CTA aborted
  for (int i = 0; i < kStages; ++i) {
    if (!(issued & (1u << i))) continue;
    // stages before the ring position were last issued in the current lap
    const uint32_t ph = (static_cast<uint32_t>(i) < pipe.idx) ? pipe.phase : (pipe.phase ^ 1u);
    wait_parity(s.full + 8 * i, ph, wd);
  }
}

__device__ void drain_mma(const Smem& s, const WaitCtx& w0) {
  mma_commit(s.drain);
  WaitCtx wd = w0;
  volatile uint32_t never = 0u;
  wd.abort = &never;
  wait_parity(s.drain, 0u, wd);
}

// ======================================================================= FWD
// Units are dealt round robin; a unit is `group` consecutive vocab tiles of one
// row tile.  Units with the same vocab group are adjacent so CTAs running at
// the same time share the W rows in L2.
struct FwdSeq {
  int unit, g;
  __device__ void begin() {
    unit = blockIdx.x;
    g = 0;
  }
  __device__ bool valid(const GemmArgs& a) const { return unit < a.units; }
  __device__ int mt(const GemmArgs& a) const { return unit % a.tiles_m; }
  __device__ int nt(const GemmArgs& a) const { return (unit / a.tiles_m) * a.group + g; }
  __device__ bool last_in_unit(const GemmArgs& a) const {
    return g + 1 == a.group || nt(a) + 1 >= a.tiles_n;
  }
  __device__ void next(const GemmArgs& a) {
    if (last_in_unit(a)) {
      unit += gridDim.x;
      g = 0;
    } else {
      ++g;
    }
  }
};

}  // namespace

__global__ void __launch_bounds__(kGemmThreads, 1)
    flce_fwd_kernel(const __grid_constant__ CUtensorMap tma_x,
                    const __grid_constant__ CUtensorMap tma_w, const GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const Smem s = carve_smem(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    init_barriers(s);
    tma_prefetch_desc(&tma_x);
    tma_prefetch_desc(&tma_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(s.tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;
  const WaitCtx w{s.abort_flag, a.err, a.wait_limit_ns};

  if (warp == 0) {
    if (lane == 0) {
      Ring pipe;
      uint32_t issued = 0;
      FwdSeq seq;
      for (seq.begin(); seq.valid(a); seq.next(a)) {
        const int m0 = seq.mt(a) * kBM, n0 = seq.nt(a) * kBN;
        bool ok = true;
        for (int kb = 0; kb < a.k_blocks && ok; ++kb) {
          ok = wait_parity(s.empty + 8 * pipe.idx, pipe.phase ^ 1u, w);
          if (!ok) break;
          const uint32_t full = s.full + 8 * pipe.idx;
          mbar_arrive_expect_tx(full, kAStageBytes + kBStageBytes);
          load_xw(&tma_x, &tma_w, s.a_base + pipe.idx * kAStageBytes,
                  s.b_base + pipe.idx * kBStageBytes, kb * kBK, m0, n0, full);
          issued |= 1u << pipe.idx;
          pipe.advance<kStages>();
        }
        if (!ok) break;
      }
      drain_loads(s, issued, pipe, w);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      Ring pipe, accr;
      FwdSeq seq;
      for (seq.begin(); seq.valid(a); seq.next(a)) {
        if (!wait_parity(s.tempty + 8 * accr.idx, accr.phase ^ 1u, w)) break;
        tc_fence_after();
        if (!mma_tile<false, false>(tmem + accr.idx * kAccCols, a.k_blocks, s, pipe, w)) break;
        mma_commit(s.tfull + 8 * accr.idx);
        accr.advance<kNumAcc>();
      }
      drain_mma(s, w);
    }
  } else {
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    Ring accr;
    float run_m = -INFINITY, run_s = 0.f;
    FwdSeq seq;
    for (seq.begin(); seq.valid(a); seq.next(a)) {
      const int row = seq.mt(a) * kBM + r;
      const int n0 = seq.nt(a) * kBN;
      const int t = row < a.N ? a.targets[row] : -1;
      if (seq.g == 0) {
        run_m = -INFINITY;
        run_s = 0.f;
      }
      if (!wait_parity(s.tfull + 8 * accr.idx, accr.phase, w)) break;
      tc_fence_after();
      const uint32_t tbase =
          tmem + (static_cast<uint32_t>(q * 32) << 16) + accr.idx * kAccCols;
      epi_lse(tbase, n0, a.V, t, a.zt + (row < a.N ? row : 0), run_m, run_s);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s.tempty + 8 * accr.idx);
      accr.advance<kNumAcc>();
      if (seq.last_in_unit(a) && row < a.N) {
        const int chunk = seq.nt(a) / a.group;
        a.partials[static_cast<size_t>(chunk) * a.N + row] = make_float2(run_m, run_s);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ======================================================================= BWD
namespace {

struct Tile {
  int kind, m0, n0, k_blocks;
};

// Ticket order: W tiles of the XW block, then R tiles of the R block, then X
// tiles of the XW block (longest K first).  Within a kind, consecutive tickets
// share the operand that is reused most (the H columns or the vocab rows).
__device__ __forceinline__ Tile decode_ticket(const BwdArgs& a, int t) {
  if (t < a.w_tiles) {
    const int v = t % a.xw.vt128, h = t / a.xw.vt128;
    return {kKindW, v * kBM, h * kBN, a.xw.mt * (kBM / kBK)};
  }
  t -= a.w_tiles;
  if (t < a.r_tiles) {
    const int m = t % a.r.mt, v = t / a.r.mt;
    return {kKindR, m * kBM, v * kBN, a.kb_h};
  }
  t -= a.r_tiles;
  const int m = t % a.xw.mt, h = t / a.xw.mt;
  return {kKindX, m * kBM, h * kBN, a.xw.vt * (kBN / kBK)};
}

}  // namespace

__global__ void __launch_bounds__(kGemmThreads, 1)
    flce_bwd_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const Smem s = carve_smem(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int total = a.w_tiles + a.r_tiles + a.x_tiles;
  if (threadIdx.x == 0) init_barriers(s);
  if (warp == 1) {
    tmem_alloc(smem_u32(s.tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;
  const WaitCtx w{s.abort_flag, a.err, a.wait_limit_ns};

  if (warp == 0) {
    if (lane == 0) {
      Ring pipe, ring;
      uint32_t issued = 0;
      const CUtensorMap* dz_k = &maps.dz_k[a.xw.slot & 1];
      const CUtensorMap* dz_mn = &maps.dz_mn[a.xw.slot & 1];
      for (;;) {
        const int t = atomicAdd(a.counter, 1);
        if (!wait_parity(s.qempty + 8 * ring.idx, ring.phase ^ 1u, w)) break;
        s.tickets[ring.idx] = t;
        mbar_arrive(s.qfull + 8 * ring.idx);
        ring.advance<kTicketRing>();
        if (t >= total) break;
        const Tile tile = decode_ticket(a, t);
        bool ok = true;
        for (int kb = 0; kb < tile.k_blocks; ++kb) {
          ok = wait_parity(s.empty + 8 * pipe.idx, pipe.phase ^ 1u, w);
          if (!ok) break;
          const uint32_t full = s.full + 8 * pipe.idx;
          const uint32_t sa = s.a_base + pipe.idx * kAStageBytes;
          const uint32_t sb = s.b_base + pipe.idx * kBStageBytes;
          const int k = kb * kBK;
          mbar_arrive_expect_tx(full, kAStageBytes + kBStageBytes);
          if (tile.kind == kKindR)
            load_xw(&maps.x_k, &maps.w_k, sa, sb, k, a.r.row0 + tile.m0, a.r.col0 + tile.n0, full);
          else if (tile.kind == kKindX)
            load_dx(dz_k, &maps.w_mn, sa, sb, k, tile.m0, tile.n0, a.xw.col0, full);
          else
            load_dw(dz_mn, &maps.x_mn, sa, sb, k, tile.m0, tile.n0, a.xw.row0, full);
          issued |= 1u << pipe.idx;
          pipe.advance<kStages>();
        }
        if (!ok) break;
      }
      drain_loads(s, issued, pipe, w);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      Ring pipe, accr, ring;
      for (;;) {
        if (!wait_parity(s.qfull + 8 * ring.idx, ring.phase, w)) break;
        const int t = s.tickets[ring.idx];
        mbar_arrive(s.qempty + 8 * ring.idx);
        ring.advance<kTicketRing>();
        if (t >= total) break;
        const Tile tile = decode_ticket(a, t);
        if (!wait_parity(s.tempty + 8 * accr.idx, accr.phase ^ 1u, w)) break;
        tc_fence_after();
        const uint32_t d = tmem + accr.idx * kAccCols;
        bool ok;
        if (tile.kind == kKindR)
          ok = mma_tile<false, false>(d, tile.k_blocks, s, pipe, w);
        else if (tile.kind == kKindX)
          ok = mma_tile<false, true>(d, tile.k_blocks, s, pipe, w);
        else
          ok = mma_tile<true, true>(d, tile.k_blocks, s, pipe, w);
        if (!ok) break;
        mma_commit(s.tfull + 8 * accr.idx);
        accr.advance<kNumAcc>();
      }
      drain_mma(s, w);
    }
  } else {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    // scale g / n_valid (mean) or g (sum), applied when a tile writes bf16 directly
    const float scale =
        (a.dx_final || a.dw_final) ? grad_scale(a.grad_loss, a.n_valid, a.reduction) : 1.f;
    Ring accr, ring;
    for (;;) {
      if (!wait_parity(s.qfull + 8 * ring.idx, ring.phase, w)) break;
      const int t = s.tickets[ring.idx];
      __syncwarp();
      if (lane == 0) mbar_arrive(s.qempty + 8 * ring.idx);
      ring.advance<kTicketRing>();
      if (t >= total) break;
      const Tile tile = decode_ticket(a, t);
      // per-row context, read before waiting for the accumulator
      int grow = 0, tgt = -1;
      float lse2 = 0.f;
      if (tile.kind == kKindR) {
        grow = a.r.row0 + tile.m0 + r;
        if (grow < a.N) {
          tgt = a.targets[grow];
          lse2 = a.lse[grow] * kLog2e;
        }
      }
      if (!wait_parity(s.tfull + 8 * accr.idx, accr.phase, w)) break;
      tc_fence_after();
      const uint32_t tbase =
          tmem + (static_cast<uint32_t>(q * 32) << 16) + accr.idx * kAccCols;
      if (tile.kind == kKindR) {
        __nv_bfloat16* out = a.dz[a.r.slot & 1] +
                             static_cast<size_t>(tile.m0 + r) * a.dz_ld + tile.n0;
        epi_dz(tbase, a.r.col0 + tile.n0, a.V, tgt, lse2, out);
      } else if (tile.kind == kKindX) {
        const int row = a.xw.row0 + tile.m0 + r;
        const bool ok = row < a.N;
        epi_acc(tbase, tile.n0, a.H, ok,
                a.dxf ? a.dxf + static_cast<size_t>(row) * a.H : nullptr,
                a.dx_final ? a.dx_final + static_cast<size_t>(row) * a.H : nullptr, scale);
      } else {
        const int lv = tile.m0 + r;
        const int v = a.xw.col0 + lv;
        const bool ok = v < a.V;
        epi_acc(tbase, tile.n0, a.H, ok,
                a.dwf ? a.dwf + static_cast<size_t>(lv) * a.H : nullptr,
                a.dw_final ? a.dw_final + static_cast<size_t>(v) * a.H : nullptr, scale);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s.tempty + 8 * accr.idx);
      accr.advance<kNumAcc>();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ================================================================= launchers
cudaError_t launch_fwd_gemm(const CUtensorMap& tx, const CUtensorMap& tw, const GemmArgs& a,
                            int grid, cudaStream_t st) {
  if (grid <= 0) return cudaSuccess;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(flce_fwd_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kGemmSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  flce_fwd_kernel<<<grid, kGemmThreads, kGemmSmemBytes, st>>>(tx, tw, a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_bwd_gemm(const BwdMaps& maps, const BwdArgs& a, int grid, cudaStream_t st) {
  if (grid <= 0) return cudaSuccess;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(flce_bwd_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kGemmSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  flce_bwd_kernel<<<grid, kGemmThreads, kGemmSmemBytes, st>>>(maps, a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace flce
