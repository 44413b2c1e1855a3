// Persistent tcgen05 GEMM kernels for the fused linear cross-entropy.
//
// Tile kinds (the backward's three are GemmKind):
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
// Every tile is 256 x 256 and computed by a pair of CTAs on two SMs (a 2-CTA
// cluster) with tcgen05 cta_group::2: each CTA stages 128 rows of A and 128 of
// the 256 columns of B, the even CTA ("leader") issues the MMAs, and each CTA
// receives its 128 rows of the FP32 result in its own tensor memory.  Per SM
// this halves the B operand traffic of a 128 x 256 single-CTA tile.
//
// Two kernels share the building blocks below:
//   flce_fwd_kernel  forward; work units of 4 vocab tiles of one row tile
//                    (so the epilogue merges the log-sum-exp of 1024 columns
//                    before writing a partial), handed out by a global ticket
//                    that the leader's producer writes into both CTAs' rings;
//                    the logits-only variant deals units round robin.
//   flce_bwd_kernel  backward; one launch holds the R and X tiles of dZ block
//                    p and the W tiles of block p-1 (two dZ slots).  Tiles
//                    are handed out by a global atomic ticket row tile by row
//                    tile (see decode_ticket): the X tiles of a 256-row tile
//                    follow its R tiles and wait for their dZ stores through
//                    a per-row-tile counter; the W tiles come last.  The
//                    leader's producer takes each ticket and writes it into
//                    both CTAs' ticket rings.
//
// CTA layout (192 threads, one CTA per SM, persistent):
//   warp 0      TMA producer: 6-stage ring of (A 128x64, B 128x64) bf16 halves,
//               128-byte swizzled; both CTAs' copies complete on the leader's
//               barrier.
//   warp 1      allocates the 512 TMEM columns of both CTAs; in the leader one
//               lane issues tcgen05.mma (M=256, N=256, K=16) into one of two
//               FP32 accumulators and multicasts the commits to both CTAs.
//   warps 2..5  epilogue: tcgen05.ld of this CTA's accumulator rows (warp w owns
//               TMEM lanes 32*(w%4) .. +31), then the kind's epilogue.
#include <algorithm>
#include <atomic>

#include "flce_device.cuh"
#include "flce_internal.h"

namespace flce {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTicketRing = 4;
constexpr uint32_t kStageTx = 2 * (kAStageBytes + kBStageBytes);  // both CTAs of the pair
constexpr uint16_t kPairMask = 0x3;

struct Smem {
  uint32_t a_base, b_base;  // shared addresses of stage 0 (1024-aligned)
  uint32_t staging;         // epilogue staging buffers (backward only)
  uint32_t full, empty;     // barrier arrays (stage-indexed, 8 bytes apart)
  uint32_t tfull, tempty;   // accumulator barriers (2 each)
  uint32_t drain;           // MMA drain barrier
  uint32_t qfull, qempty;   // ticket ring barriers
  uint32_t tickets;         // ticket ring (shared address)
  volatile int* tickets_p;  // the same ring, generic pointer
  uint32_t* tmem_slot;
  volatile uint32_t* abort_flag;
};

// Carves the dynamic shared memory: stages, epilogue staging buffers (if
// any), then barriers, then small slots.  Identical in both CTAs of a pair, so
// an offset names the same object in either.
__device__ Smem carve_smem(uint8_t* smem_raw, uint32_t staging_bytes) {
  Smem s;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  s.a_base = base;
  s.b_base = base + kStages * kAStageBytes;
  s.staging = s.b_base + kStages * kBStageBytes;  // 1024-aligned
  const uint32_t bar0 = s.staging + staging_bytes;
  s.full = bar0;
  s.empty = s.full + 8 * kStages;
  s.tfull = s.empty + 8 * kStages;
  s.tempty = s.tfull + 8 * kNumAcc;
  s.drain = s.tempty + 8 * kNumAcc;
  s.qfull = s.drain + 8;
  s.qempty = s.qfull + 8 * kTicketRing;
  s.tickets = s.qempty + 8 * kTicketRing;
  s.tickets_p = reinterpret_cast<volatile int*>(smem_raw + (s.tickets - raw));
  uint8_t* g = smem_raw + (s.tickets + 4 * kTicketRing - raw);
  s.tmem_slot = reinterpret_cast<uint32_t*>(g);
  s.abort_flag = reinterpret_cast<volatile uint32_t*>(g + 4);
  return s;
}

__device__ void init_barriers(const Smem& s) {
  for (int i = 0; i < kStages; ++i) {
    mbar_init(s.full + 8 * i, 1);   // leader's producer (expect_tx for both CTAs)
    mbar_init(s.empty + 8 * i, 1);  // the leader's multicast MMA commit
  }
  for (int i = 0; i < kNumAcc; ++i) {
    mbar_init(s.tfull + 8 * i, 1);   // multicast MMA commit
    mbar_init(s.tempty + 8 * i, 8);  // 4 epilogue warps in each of the 2 CTAs
  }
  mbar_init(s.drain, 1);
  for (int i = 0; i < kTicketRing; ++i) {
    mbar_init(s.qfull + 8 * i, 1);
    // leader: its MMA lane and 4 epilogue warps; peer: its producer and 4 epilogue warps
    mbar_init(s.qempty + 8 * i, 10);
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

// Set-up shared by both kernels: barriers, the pair's TMEM, and a cluster
// barrier so that no CTA signals a barrier of its peer before the peer has
// initialised it.
__device__ uint32_t pair_setup(const Smem& s, int warp) {
  if (threadIdx.x == 0) init_barriers(s);
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(s.tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  return *s.tmem_slot;
}

// Teardown shared by both kernels: every role has drained; wait for the peer,
// then release the pair's TMEM.
__device__ void pair_teardown(uint32_t tmem, int warp) {
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

// ------------------------------------------------------- k-block operand loads
// Each CTA loads its own 128 A rows and 128 B columns; completion is counted
// on the leader's barrier `full` (a shared::cluster address).
// Z = X W^T (FWD and R): both K-major.  X, re-read for every vocab tile, is
// kept in L2 with an evict-last hint.
__device__ __forceinline__ void load_xw(const CUtensorMap* tx, const CUtensorMap* tw, uint32_t sa,
                                        uint32_t sb, int k, int arow, int brow, uint32_t full,
                                        uint64_t keep) {
  tma_load_2d_pair_hint(sa, tx, k, arow, full, keep);
  tma_load_2d_pair(sb, tw, k, brow, full);
}
// dX tile: A = dZ rows (K-major over vocab), B = W rows of the block (MN-major over H).
__device__ __forceinline__ void load_dx(const CUtensorMap* tdz, const CUtensorMap* twmn,
                                        const CUtensorMap* twmn3, bool mn3d, uint32_t sa,
                                        uint32_t sb, int k, int arow, int h0, int vrow0,
                                        uint32_t full) {
  tma_load_2d_pair(sa, tdz, k, arow, full);
  if (mn3d) {
    tma_load_3d_pair(sb, twmn3, 0, vrow0 + k, h0 / 64, full);
  } else {
#pragma unroll
    for (int q = 0; q < 2; ++q)
      tma_load_2d_pair(sb + q * 8192, twmn, h0 + 64 * q, vrow0 + k, full);
  }
}
// dW tile: A = dZ^T (MN-major over vocab), B = X rows of the block (MN-major over H).
// k: local dZ row of this k-block; xrow: the token row of X it corresponds to.
__device__ __forceinline__ void load_dw(const CUtensorMap* txmn, const CUtensorMap* tdzmn3,
                                        const CUtensorMap* txmn3, bool mn3d, uint32_t sa,
                                        uint32_t sb, int k, int v0, int h0, int xrow,
                                        uint32_t full, uint64_t keep) {
  tma_load_3d_pair(sa, tdzmn3, 0, k, v0 / 64, full);  // the dZ slot is always 64-aligned
  if (mn3d) {
    tma_load_3d_pair_hint(sb, txmn3, 0, xrow, h0 / 64, full, keep);
  } else {
#pragma unroll
    for (int q = 0; q < 2; ++q)
      tma_load_2d_pair_hint(sb + q * 8192, txmn, h0 + 64 * q, xrow, full, keep);
  }
}

// ------------------------------------------------------- MMA of one k-block
// K-major: the 16-element K step is 32 bytes inside the swizzled row; 8-row
// groups are 1024 bytes apart.  MN-major: the K step is two 8-row core-matrix
// groups, 2048 bytes; 64-element groups along M/N are 8192 bytes apart (one
// 64x64 TMA box each).
template <bool A_MN, bool B_MN>
__device__ __forceinline__ void mma_kblock(uint32_t d, uint32_t sa, uint32_t sb, bool first) {
  constexpr uint32_t idesc = instr_desc_bf16(kPairM, kBN, A_MN, B_MN);
#pragma unroll
  for (int k = 0; k < kBK / kUmmaK; ++k) {
    const uint64_t ad = A_MN ? smem_desc_sw128(sa + k * 2048, 8192, 1024)
                             : smem_desc_sw128(sa + k * 32, 0, 1024);
    const uint64_t bd = B_MN ? smem_desc_sw128(sb + k * 2048, 8192, 1024)
                             : smem_desc_sw128(sb + k * 32, 0, 1024);
    mma_bf16_pair(d, ad, bd, idesc, (first && k == 0) ? 0u : 1u);
  }
}

// Leader only: the MMAs of one tile into accumulator d; false if aborted.
template <bool A_MN, bool B_MN>
__device__ bool mma_tile(uint32_t d, int k_blocks, const Smem& s, Ring& pipe, const WaitCtx& w) {
  for (int kb = 0; kb < k_blocks; ++kb) {
    if (!wait_parity(s.full + 8 * pipe.idx, pipe.phase, w)) return false;
    tc_fence_after();
    mma_kblock<A_MN, B_MN>(d, s.a_base + pipe.idx * kAStageBytes,
                           s.b_base + pipe.idx * kBStageBytes, kb == 0);
    // frees the stage in both CTAs once these MMAs have read it
    mma_commit_pair_multicast(s.empty + 8 * pipe.idx, kPairMask);
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

// ------------------------------------------- staged epilogue (backward)
// Each epilogue warp owns two 4 KB staging buffers.  A chunk is 32 rows (one
// per lane) x 128 bytes, written in the 128-byte-swizzled layout of a TMA box
// (16-byte piece j of row r at (j ^ (r % 8)) * 16), then written to global
// memory by one TMA store or reduce-add issued by lane 0.  Rows or columns
// outside the tensor are clipped by the TMA unit.
struct Stager {
  uint32_t buf0;
  uint32_t cur = 0;
  __device__ uint32_t buf() const { return buf0 + cur * kStageBufBytes; }
  // the buffer about to be filled was last used two chunks ago
  __device__ void acquire(int lane) {
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
  }
  __device__ void write_row(int lane, const uint32_t (&w)[32]) const {
    const uint32_t row = buf() + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      st_shared_v4(row + ((j ^ (lane & 7)) << 4),
                   make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]));
  }
  // make the generic-proxy writes visible to the TMA unit, then hand over
  __device__ void publish() {
    fence_proxy_async_smem();
    __syncwarp();
  }
  __device__ void store(int lane, const CUtensorMap* m, int x, int y) {
    publish();
    if (lane == 0) {
      tma_store_2d(m, buf(), x, y);
      bulk_commit();
    }
    cur ^= 1u;
  }
  // the FP32 accumulators are streamed through L2 once per block: evict first
  __device__ void reduce_add(int lane, const CUtensorMap* m, int x, int y) {
    publish();
    if (lane == 0) {
      tma_reduce_add_2d_hint(m, buf(), x, y, l2_policy_evict_first());
      bulk_commit();
    }
    cur ^= 1u;
  }
};

// dZ tile rows of this warp: 64 columns per chunk, bf16 store into the slot.
__device__ __forceinline__ void epi_dz_staged(uint32_t tbase, int gcol0, int V, int t, float lse2,
                                              Stager& st, int lane, const CUtensorMap* m, int x0,
                                              int y) {
  const bool valid_row = t >= 0;
#pragma unroll 1
  for (int c = 0; c < kBN / 64; ++c) {
    float v[64];
    tmem_ld32(tbase + 64 * c, *reinterpret_cast<float(*)[32]>(&v[0]));
    tmem_ld32(tbase + 64 * c + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
    const int j0 = gcol0 + 64 * c;
    uint32_t p[32];
    if (valid_row) {
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
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
      for (int i = 0; i < 32; ++i) p[i] = 0u;
    }
    st.acquire(lane);
    st.write_row(lane, p);
    st.store(lane, m, x0 + 64 * c, y);
  }
}

// FP32 accumulator rows: reduce-add scale * value, 32 columns per chunk, into
// an FP32 buffer.
__device__ __forceinline__ void epi_reduce_staged(uint32_t tbase, int h0, int H, float scale,
                                                  Stager& st, int lane, const CUtensorMap* m,
                                                  int y) {
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    const int h = h0 + 32 * c;
    if (h >= H) break;  // warp-uniform
    float v[32];
    tmem_ld32(tbase + 32 * c, v);
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(scale * v[i]);
    st.acquire(lane);
    st.write_row(lane, w);
    st.reduce_add(lane, m, h, y);
  }
}

// Final gradient rows: bf16(scale * acc), 64 columns per chunk (zeros when the
// tile had no K, i.e. no accumulator was written).
__device__ __forceinline__ void epi_final_staged(uint32_t tbase, int h0, int H, float scale,
                                                 Stager& st, int lane, const CUtensorMap* m,
                                                 int y, bool zero = false) {
#pragma unroll 1
  for (int c = 0; c < kBN / 64; ++c) {
    const int h = h0 + 64 * c;
    if (h >= H) break;  // warp-uniform
    float v[64];
    if (zero) {
#pragma unroll
      for (int i = 0; i < 64; ++i) v[i] = 0.f;
    } else {
      tmem_ld32(tbase + 64 * c, *reinterpret_cast<float(*)[32]>(&v[0]));
      tmem_ld32(tbase + 64 * c + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
    }
    uint32_t p[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) p[i] = pack_bf16x2(scale * v[2 * i], scale * v[2 * i + 1]);
    st.acquire(lane);
    st.write_row(lane, p);
    st.store(lane, m, h, y);
  }
}

// Leader's producer teardown: every stage's most recent loads (from both CTAs)
// must have landed before either CTA may exit.
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

// Leader's MMA teardown: all issued MMAs complete before TMEM is released.
__device__ void drain_mma(const Smem& s, const WaitCtx& w0) {
  mma_commit_pair(s.drain);
  WaitCtx wd = w0;
  volatile uint32_t never = 0u;
  wd.abort = &never;
  wait_parity(s.drain, 0u, wd);
}

// ======================================================================= FWD
// A work unit is `group` consecutive vocab tiles of one 256-row tile; units of
// the same vocab group are numbered consecutively.  The loss forward hands
// units out by a global atomic ticket (the leader's producer takes it and
// publishes it to both CTAs' ticket rings), so pairs running at the same time
// always work on neighbouring units and share the W rows in L2, however far
// their progress drifts apart.  The logits path, which has no workspace for a
// ticket counter, deals units round robin instead.

// Row tile and vocab group of unit u: bands of a.band row tiles (the last one
// may be shorter), vocab group by vocab group within a band, row tile fastest.
struct Unit {
  int m, vg;
};
__device__ __forceinline__ Unit unit_of(const GemmArgs& a, int u) {
  const int vgroups = (a.tiles_n + a.group - 1) / a.group;
  const int full = a.tiles_m / a.band;              // bands of a.band row tiles
  const int in_full = full * a.band * vgroups;
  if (u < in_full) {
    const int b = u / (a.band * vgroups), r = u % (a.band * vgroups);
    return {b * a.band + r % a.band, r / a.band};
  }
  const int last = a.tiles_m - full * a.band;       // > 0 here
  const int r = u - in_full;
  return {full * a.band + r % last, r / last};
}

// Next unit for a role.  `leader_producer` takes tickets; the other roles read
// them from this CTA's ring.  Returns false if aborted.
template <bool DYN>
__device__ __forceinline__ bool next_unit(const GemmArgs& a, const Smem& s, Ring& ring,
                                          int& unit, bool leader_producer, bool peer_producer,
                                          bool cluster_scope, int lane, bool whole_warp,
                                          const WaitCtx& w) {
  if constexpr (!DYN) {
    unit = unit < 0 ? static_cast<int>(blockIdx.x >> 1) : unit + static_cast<int>(gridDim.x >> 1);
    return true;
  } else {
    if (leader_producer) {
      unit = atomicAdd(a.counter, 1);
      if (!wait_parity_cluster(s.qempty + 8 * ring.idx, ring.phase ^ 1u, w)) return false;
      s.tickets_p[ring.idx] = unit;
      st_shared_cluster_u32(mapa_shared(s.tickets + 4 * ring.idx, 1), static_cast<uint32_t>(unit));
      mbar_arrive(s.qfull + 8 * ring.idx);
      mbar_arrive_cluster(mapa_shared(s.qfull + 8 * ring.idx, 1));
    } else {
      const bool ok = cluster_scope ? wait_parity_cluster(s.qfull + 8 * ring.idx, ring.phase, w)
                                    : wait_parity(s.qfull + 8 * ring.idx, ring.phase, w);
      if (!ok) return false;
      unit = s.tickets_p[ring.idx];
      if (whole_warp) __syncwarp();
      if (!whole_warp || lane == 0) {
        if (peer_producer || cluster_scope)
          mbar_arrive_cluster(mapa_shared(s.qempty + 8 * ring.idx, 0));
        else
          mbar_arrive(s.qempty + 8 * ring.idx);
      }
    }
    ring.advance<kTicketRing>();
    return true;
  }
}

}  // namespace

// MODE kFwdLse: the forward of the loss (log-sum-exp epilogue), dynamic units.
// MODE kFwdLogits: plain logits Z = X W^T rounded to bf16 and stored through
// shared-memory staging (the inference path with no labels), static units.
constexpr int kFwdLse = 0;
constexpr int kFwdLogits = 1;

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    flce_fwd_kernel(const __grid_constant__ CUtensorMap tma_x,
                    const __grid_constant__ CUtensorMap tma_w,
                    const __grid_constant__ CUtensorMap tma_out, const GemmArgs a) {
  constexpr bool kDyn = MODE == kFwdLse;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const Smem s = carve_smem(smem_raw, MODE == kFwdLogits ? 4 * 2 * kStageBufBytes : 0);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tma_x);
    tma_prefetch_desc(&tma_w);
  }
  const uint32_t tmem = pair_setup(s, warp);
  const WaitCtx w{s.abort_flag, a.err, a.wait_limit_ns};

  if (warp == 0) {
    if (lane == 0) {
      Ring pipe, ring;
      uint32_t issued = 0;
      const uint64_t keep = l2_policy_evict_last();
      int u = -1;
      bool ok = true;
      while (ok && next_unit<kDyn>(a, s, ring, u, leader, !leader, true, lane, false, w) &&
             u < a.units) {
        const Unit un = unit_of(a, u);
        const int arow = un.m * kPairM + kBM * rank;
        for (int g = 0; g < a.group && ok; ++g) {
          const int nt = un.vg * a.group + g;
          if (nt >= a.tiles_n) break;
          const int brow = nt * kBN + kHalfN * rank;
          for (int kb = 0; kb < a.k_blocks; ++kb) {
            ok = wait_parity(s.empty + 8 * pipe.idx, pipe.phase ^ 1u, w);
            if (!ok) break;
            const uint32_t full = s.full + 8 * pipe.idx;
            if (leader) mbar_arrive_expect_tx(full, kStageTx);
            load_xw(&tma_x, &tma_w, s.a_base + pipe.idx * kAStageBytes,
                    s.b_base + pipe.idx * kBStageBytes, kb * kBK, arow, brow,
                    mapa_shared(full, 0), keep);
            issued |= 1u << pipe.idx;
            pipe.advance<kStages>();
          }
        }
      }
      if (leader) drain_loads(s, issued, pipe, w);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      Ring pipe, accr, ring;
      int u = -1;
      bool ok = true;
      while (ok && next_unit<kDyn>(a, s, ring, u, false, false, false, lane, false, w) &&
             u < a.units) {
        const Unit un = unit_of(a, u);
        for (int g = 0; g < a.group; ++g) {
          const int nt = un.vg * a.group + g;
          if (nt >= a.tiles_n) break;
          ok = wait_parity_cluster(s.tempty + 8 * accr.idx, accr.phase ^ 1u, w);
          if (!ok) break;
          tc_fence_after();
          ok = mma_tile<false, false>(tmem + accr.idx * kAccCols, a.k_blocks, s, pipe, w);
          if (!ok) break;
          mma_commit_pair_multicast(s.tfull + 8 * accr.idx, kPairMask);
          accr.advance<kNumAcc>();
        }
      }
      drain_mma(s, w);
    }
  } else {
    const int q = warp & 3;                    // TMEM lane quarter this warp may access
    const int r = kBM * rank + q * 32 + lane;  // row of the 256-row tile
    Stager st;
    st.buf0 = s.staging + static_cast<uint32_t>(q) * 2 * kStageBufBytes;
    Ring accr, ring;
    int u = -1;
    bool ok = true;
    while (ok && next_unit<kDyn>(a, s, ring, u, false, false, true, lane, true, w) &&
           u < a.units) {
      const Unit un = unit_of(a, u);
      const int row = un.m * kPairM + r;
      const int t = (MODE == kFwdLse && row < a.N) ? a.targets[row] : -1;
      float run_m = -INFINITY, run_s = 0.f;
      for (int g = 0; g < a.group; ++g) {
        const int nt = un.vg * a.group + g;
        if (nt >= a.tiles_n) break;
        ok = wait_parity(s.tfull + 8 * accr.idx, accr.phase, w);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tbase =
            tmem + (static_cast<uint32_t>(q * 32) << 16) + accr.idx * kAccCols;
        if (MODE == kFwdLogits)
          epi_final_staged(tbase, nt * kBN, a.V, 1.f, st, lane, &tma_out, row - lane);
        else
          epi_lse(tbase, nt * kBN, a.V, t, a.zt + (row < a.N ? row : 0), run_m, run_s);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(s.tempty + 8 * accr.idx, 0));
        accr.advance<kNumAcc>();
      }
      if (MODE == kFwdLse && ok && row < a.N)
        a.partials[static_cast<size_t>(un.vg) * a.N + row] = make_float2(run_m, run_s);
    }
    if (MODE == kFwdLogits) {
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }
  pair_teardown(tmem, warp);
}

// ======================================================================= BWD
namespace {

struct Tile {
  int kind, m0, n0, k_blocks;
};

// Tiles of this launch, from the number of 256-row tiles the backward runs on
// (written on the device before the first backward launch).
struct Counts {
  int mt_r, mt_w;  // 256-row tiles of the R block and of the W block
  int r_tiles, x_tiles, w_tiles, total;
  int lag;         // X tiles of row tile m follow the R tiles of row tile m + lag
  int first;       // R tiles handed out before the W tiles when w_early
  bool w_early;    // W tiles (K = the block's active rows) at least 3x as long as
                   // R tiles (K = H): hand them out after one wave of R tiles
};

__device__ __forceinline__ Counts tile_counts(const BwdArgs& a) {
  const int n = *a.n_active;
  Counts c;
  c.mt_r = max(0, min(a.r.mt, n - a.r.tile0));
  c.mt_w = max(0, min(a.w.mt, n - a.w.tile0));
  c.r_tiles = c.mt_r * a.r.vt;
  c.x_tiles = a.want_dx ? c.mt_r * a.h_tiles : 0;
  // with no active token tile a bf16 dW written directly still needs its zeros:
  // those W tiles run with K = 0 and store 0
  c.w_tiles = (a.want_dw && (c.mt_w > 0 || a.dw_final)) ? a.w.vt * a.h_tiles : 0;
  c.total = c.r_tiles + c.x_tiles + c.w_tiles;
  c.lag = min(a.x_lag, c.mt_r);
  c.w_early = c.mt_w * kPairM >= 3 * a.H;
  c.first = min(c.r_tiles, static_cast<int>(gridDim.x >> 1));
  return c;
}

// Row of the X the backward reads (a token row, or a dense row of the gathered
// copy) of local dZ row `l` of a block starting at tile-list entry tile0.
__device__ __forceinline__ int token_row(const BwdArgs& a, int tile0, int l) {
  return a.active[tile0 + (l >> 8)] * kPairM + (l & (kPairM - 1));
}

// Ticket order.  The R tiles of the block go row tile by row tile (vocab
// fastest: the pairs running at once share X rows and sweep the W block), and
// the X tiles of row tile m are handed out right after the R tiles of row tile
// m + lag (H-fastest: they share those dZ rows), so they read dZ rows and W
// block rows that were written or read moments before and are still in L2;
// an X tile waits (row_done) until every R tile of its row tile has stored.
// The launch ends on the W tiles of the previous block, complete before the
// launch began.  R tiles come first because only their mainloops may run
// while the previous launch drains (their dZ stores wait for it: the slot they
// write was last read there).
// m0: local row of the tile (dZ row for R/X tiles, vocab row for W tiles).
__device__ __forceinline__ Tile tile_r(const BwdArgs& a, int m, int v) {
  return {kKindR, m * kPairM, v * kBN, a.kb_h};
}
__device__ __forceinline__ Tile tile_x(const BwdArgs& a, int m, int h) {
  return {kKindX, m * kPairM, h * kBN, a.r.vt * (kBN / kBK)};
}

__device__ __forceinline__ Tile decode_rx(const BwdArgs& a, const Counts& c, int t);

// When the W tiles are long (w_early), they are handed out right after the
// first wave of R tiles (one per CTA pair) instead of last, so that the launch
// ends on the shorter kinds and the next launch, which waits for this one to
// end before its first store, is not held up by a tail of long W tiles.
__device__ __forceinline__ Tile decode_ticket(const BwdArgs& a, const Counts& c, int t) {
  if (!c.w_early) return decode_rx(a, c, t);
  if (t < c.first) return decode_rx(a, c, t);
  if (t < c.first + c.w_tiles) {
    const int u = t - c.first, ht = a.h_tiles;
    return {kKindW, (u / ht) * kPairM, (u % ht) * kBN, c.mt_w * (kPairM / kBK)};
  }
  return decode_rx(a, c, t - c.w_tiles);
}

// R and X tiles in their per-row-tile order, then (unless w_early) W tiles.
__device__ __forceinline__ Tile decode_rx(const BwdArgs& a, const Counts& c, int t) {
  const int vt = a.r.vt, ht = a.h_tiles;
  const int xt = a.want_dx ? ht : 0;  // X tiles per row tile
  // row tiles 0 .. lag-1: R tiles only
  const int n_head = c.lag * vt;
  if (t < n_head) return tile_r(a, t / vt, t % vt);
  t -= n_head;
  // row tiles lag .. mt_r-1: R tiles of row tile g + lag, then X tiles of g
  const int n_mid = (c.mt_r - c.lag) * (vt + xt);
  if (t < n_mid) {
    const int g = t / (vt + xt), j = t % (vt + xt);
    return j < vt ? tile_r(a, g + c.lag, j) : tile_x(a, g, j - vt);
  }
  t -= n_mid;
  // the X tiles of the last `lag` row tiles
  const int n_tail = c.lag * xt;
  if (t < n_tail) return tile_x(a, c.mt_r - c.lag + t / xt, t % xt);
  t -= n_tail;
  // W tiles of the previous block, H-fastest (they share dZ columns)
  const int h = t % ht, v = t / ht;
  return {kKindW, v * kPairM, h * kBN, c.mt_w * (kPairM / kBK)};
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    flce_bwd_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const Smem s = carve_smem(smem_raw, 4 * 2 * kStageBufBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  const Counts cnt = tile_counts(a);
  const int total = cnt.total;
  const uint32_t tmem = pair_setup(s, warp);
  const WaitCtx w{s.abort_flag, a.err, a.wait_limit_ns};
  // The next backward launch may start on SMs this grid frees.  It runs its
  // recompute mainloops at once and waits for this grid before it touches the
  // dZ slots (griddep_wait below).
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      Ring pipe, ring;
      uint32_t issued = 0;
      bool prior_done = false;  // the preceding grid (which wrote this dZ slot) has completed
      const uint64_t keep = l2_policy_evict_last();
      const CUtensorMap* dz_k = &maps.dz_k[a.r.slot & 1];    // X tiles: this launch's block
      const CUtensorMap* dz_mn3 = &maps.dz_mn3[a.w.slot & 1];  // W tiles: the previous block
      const bool mn3d = a.mn3d != 0;
      for (;;) {
        int t;
        if (leader) {
          // take a ticket and publish it in both CTAs' rings
          t = atomicAdd(a.counter, 1);
          if (!wait_parity_cluster(s.qempty + 8 * ring.idx, ring.phase ^ 1u, w)) break;
          s.tickets_p[ring.idx] = t;
          st_shared_cluster_u32(mapa_shared(s.tickets + 4 * ring.idx, 1),
                                static_cast<uint32_t>(t));
          mbar_arrive(s.qfull + 8 * ring.idx);
          mbar_arrive_cluster(mapa_shared(s.qfull + 8 * ring.idx, 1));
        } else {
          if (!wait_parity_cluster(s.qfull + 8 * ring.idx, ring.phase, w)) break;
          t = s.tickets_p[ring.idx];
          mbar_arrive_cluster(mapa_shared(s.qempty + 8 * ring.idx, 0));
        }
        ring.advance<kTicketRing>();
        if (t >= total) break;
        const Tile tile = decode_ticket(a, cnt, t);
        if (tile.kind == kKindW && !prior_done) {
          griddep_wait();  // the W tiles read the dZ slot the previous launch wrote
          prior_done = true;
        }
        // an X tile reads the dZ rows of its row tile, stored by this launch's
        // R tiles: wait until all 8 * vt epilogue warps of them have finished
        if (tile.kind == kKindX &&
            !wait_counter_geq(a.row_done + (tile.m0 >> 8), 8 * a.r.vt, w))
          break;
        const int arow = tile.m0 + kBM * rank;     // this CTA's A rows (M)
        const int bcol = tile.n0 + kHalfN * rank;  // this CTA's B columns (N)
        bool ok = true;
        for (int kb = 0; kb < tile.k_blocks; ++kb) {
          ok = wait_parity(s.empty + 8 * pipe.idx, pipe.phase ^ 1u, w);
          if (!ok) break;
          const uint32_t full = s.full + 8 * pipe.idx;
          const uint32_t full_c = mapa_shared(full, 0);
          const uint32_t sa = s.a_base + pipe.idx * kAStageBytes;
          const uint32_t sb = s.b_base + pipe.idx * kBStageBytes;
          const int k = kb * kBK;
          if (leader) mbar_arrive_expect_tx(full, kStageTx);
          if (tile.kind == kKindR)
            load_xw(&maps.x_k, &maps.w_k, sa, sb, k, token_row(a, a.r.tile0, arow),
                    a.r.col0 + bcol, full_c, keep);
          else if (tile.kind == kKindX)
            load_dx(dz_k, &maps.w_mn, &maps.w_mn3, mn3d, sa, sb, k, arow, bcol, a.r.col0,
                    full_c);
          else
            load_dw(&maps.x_mn, dz_mn3, &maps.x_mn3, mn3d, sa, sb, k, arow, bcol,
                    token_row(a, a.w.tile0, k), full_c, keep);
          issued |= 1u << pipe.idx;
          pipe.advance<kStages>();
        }
        if (!ok) break;
      }
      if (leader) drain_loads(s, issued, pipe, w);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      Ring pipe, accr, ring;
      for (;;) {
        if (!wait_parity(s.qfull + 8 * ring.idx, ring.phase, w)) break;
        const int t = s.tickets_p[ring.idx];
        mbar_arrive(s.qempty + 8 * ring.idx);
        ring.advance<kTicketRing>();
        if (t >= total) break;
        const Tile tile = decode_ticket(a, cnt, t);
        if (!wait_parity_cluster(s.tempty + 8 * accr.idx, accr.phase ^ 1u, w)) break;
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
        mma_commit_pair_multicast(s.tfull + 8 * accr.idx, kPairMask);
        accr.advance<kNumAcc>();
      }
      drain_mma(s, w);
    }
  } else {
    const int q = warp & 3;
    const int r = kBM * rank + q * 32 + lane;  // row of the 256-row tile
    // scale g / n_valid (mean) or g (sum), applied when a tile writes bf16 directly
    const float scale = (a.dx_final || a.dw_final || a.dw_accumulate || a.dx_accumulate)
                            ? grad_scale(a.grad_loss, a.n_valid, a.reduction)
                            : 1.f;
    Stager st;
    st.buf0 = s.staging + static_cast<uint32_t>(q) * 2 * kStageBufBytes;
    Ring accr, ring;
    bool prior_done = false;  // no dZ store before the preceding grid has completed
    for (;;) {
      if (!wait_parity_cluster(s.qfull + 8 * ring.idx, ring.phase, w)) break;
      const int t = s.tickets_p[ring.idx];
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(s.qempty + 8 * ring.idx, 0));
      ring.advance<kTicketRing>();
      if (t >= total) break;
      const Tile tile = decode_ticket(a, cnt, t);
      // per-row context, read before waiting for the accumulator
      int tgt = -1;
      float lse2 = 0.f;
      if (tile.kind == kKindR) {
        const int grow = token_row(a, a.r.tile0, tile.m0 + r);
        if (grow < a.N) {
          tgt = a.targets[grow];
          lse2 = a.lse[grow] * kLog2e;
        }
      }
      if (!wait_parity(s.tfull + 8 * accr.idx, accr.phase, w)) break;
      // before the first store or reduce-add: the previous launch has finished
      // reading the dZ slot the R tiles write, and its dX / dW additions come
      // first (a fixed order of FP32 additions)
      if (!prior_done) {
        griddep_wait();
        prior_done = true;
      }
      tc_fence_after();
      const uint32_t tbase =
          tmem + (static_cast<uint32_t>(q * 32) << 16) + accr.idx * kAccCols;
      const int y0 = tile.m0 + r - lane;  // first tile row of this warp
      if (tile.kind == kKindR) {
        epi_dz_staged(tbase, a.r.col0 + tile.n0, a.V, tgt, lse2, st, lane,
                      &maps.dz_st[a.r.slot & 1], tile.n0, y0);
        // publish: this warp's dZ rows of the tile are in global memory
        if (lane == 0) {
          bulk_wait_all();
          fence_proxy_async_global();
          red_release_gpu_add(a.row_done + (tile.m0 >> 8), 1);
        }
        __syncwarp();
      } else if (tile.kind == kKindX) {
        const int row = token_row(a, a.r.tile0, y0);
        if (a.dx_final)
          epi_final_staged(tbase, tile.n0, a.H, scale, st, lane, &maps.dx_out, row);
        else
          // the FP32 accumulator (scaled at the downcast), or the caller's FP32
          // buffer (scaled here)
          epi_reduce_staged(tbase, tile.n0, a.H, a.dx_accumulate ? scale : 1.f, st, lane,
                            &maps.dx_out, row);
      } else {
        if (a.dw_final)
          epi_final_staged(tbase, tile.n0, a.H, scale, st, lane, &maps.dw_out, a.w.col0 + y0,
                           tile.k_blocks == 0);
        else
          // an FP32 band (scaled later), or the caller's FP32 gradient (scaled here)
          epi_reduce_staged(tbase, tile.n0, a.H, a.dw_accumulate ? scale : 1.f, st, lane,
                            &maps.dw_out, a.dw_accumulate ? a.w.col0 + y0 : y0);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(s.tempty + 8 * accr.idx, 0));
      accr.advance<kNumAcc>();
    }
    // all staged stores and reductions complete before the CTA exits
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  // No CTA exits before the previous launch has completed, so that the
  // completion of this launch implies the completion of every earlier one.
  if (threadIdx.x == 0) griddep_wait();
  pair_teardown(tmem, warp);
}

// ================================================================= launchers
namespace {

constexpr int kMaxDevices = 64;

// Per-kernel launch set-up, per device: the CTA pairs that fit at once (0
// until the device's first launch).  Atomic: host threads may launch at once;
// racing first launches each set the same attribute and store the same count.
struct LaunchCache {
  std::atomic<int> pairs[kMaxDevices] = {};
};

// On the current device's first launch of `kernel`: raises its dynamic
// shared-memory limit to `smem` and counts the CTA pairs that fit at once.
// Later launches on that device read the count from `cache`.
cudaError_t prepare_launch(const void* kernel, int smem, LaunchCache* cache, int* pairs) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached) {
    const int n = cache->pairs[dev].load(std::memory_order_acquire);
    if (n > 0) {
      *pairs = n;
      return cudaSuccess;
    }
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sms / 2;
  }
  if (cached) cache->pairs[dev].store(n, std::memory_order_release);
  *pairs = n;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_fwd_gemm(const CUtensorMap& tx, const CUtensorMap& tw, const GemmArgs& a,
                            int units, cudaStream_t st) {
  if (units <= 0) return cudaSuccess;
  static LaunchCache cache;
  auto* k = flce_fwd_kernel<kFwdLse>;
  int pairs = 0;
  cudaError_t e = prepare_launch(reinterpret_cast<const void*>(k), kGemmSmemBytes, &cache, &pairs);
  if (e != cudaSuccess) return e;
  k<<<2 * std::min(units, pairs), kGemmThreads, kGemmSmemBytes, st>>>(tx, tw, tx, a);
  note_launch();
  note_wait_limit(a.wait_limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_logits_gemm(const CUtensorMap& tx, const CUtensorMap& tw,
                               const CUtensorMap& tout, const GemmArgs& a, int units,
                               cudaStream_t st) {
  if (units <= 0) return cudaSuccess;
  static LaunchCache cache;
  auto* k = flce_fwd_kernel<kFwdLogits>;
  int pairs = 0;
  cudaError_t e = prepare_launch(reinterpret_cast<const void*>(k), kBwdSmemBytes, &cache, &pairs);
  if (e != cudaSuccess) return e;
  k<<<2 * std::min(units, pairs), kGemmThreads, kBwdSmemBytes, st>>>(tx, tw, tout, a);
  note_launch();
  note_wait_limit(a.wait_limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_bwd_gemm(const BwdMaps& maps, const BwdArgs& a, int units, bool overlap_prior,
                            cudaStream_t st) {
  if (units <= 0) return cudaSuccess;
  static LaunchCache cache;
  int pairs = 0;
  cudaError_t e0 = prepare_launch(reinterpret_cast<const void*>(flce_bwd_kernel), kBwdSmemBytes,
                                  &cache, &pairs);
  if (e0 != cudaSuccess) return e0;
  const int n = std::min(units, pairs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * n, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = kBwdSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl;
  cfg.numAttrs = overlap_prior ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, flce_bwd_kernel, maps, a);
  note_launch();
  note_wait_limit(a.wait_limit_ns);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace flce
