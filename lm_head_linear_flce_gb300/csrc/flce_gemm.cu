// Persistent tcgen05 GEMM kernels for the fused linear cross-entropy.
//
// One kernel template, four tile kinds (see GemmKind):
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
// CTA layout (192 threads, one CTA per SM, persistent over work units):
//   warp 0      TMA producer: 4-stage ring of (A 128x64, B 256x64) bf16 tiles,
//               128-byte swizzled, completion counted on mbarriers.
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

struct Smem {
  uint32_t a_base, b_base;  // shared addresses of stage 0 (1024-aligned)
  uint32_t full, empty;     // barrier arrays (stage-indexed, 8 bytes apart)
  uint32_t tfull, tempty;   // accumulator barriers (2 each)
  uint32_t drain;           // MMA drain barrier
};

template <int KIND>
struct KindTraits;
template <>
struct KindTraits<kKindFwd> {
  static constexpr bool a_mn = false, b_mn = false;
};
template <>
struct KindTraits<kKindR> {
  static constexpr bool a_mn = false, b_mn = false;
};
template <>
struct KindTraits<kKindX> {
  static constexpr bool a_mn = false, b_mn = true;
};
template <>
struct KindTraits<kKindW> {
  static constexpr bool a_mn = true, b_mn = true;
};

// Iterates the (m-tile, n-tile) sequence of this CTA: units are dealt round
// robin; a unit is `group` consecutive n-tiles of one m-tile.  Units with the
// same n-group are adjacent so concurrently running CTAs share the large
// operand in L2.
struct TileSeq {
  int unit, g;
  __device__ void begin(const GemmArgs& a) {
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

__device__ __forceinline__ float grad_scale(const GemmArgs& a) {
  const float g = *a.grad_loss;
  if (a.reduction == 1) return g;
  const long long n = *a.n_valid;
  return n > 0 ? g / static_cast<float>(n) : 0.f;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------------ roles
template <int KIND>
__device__ void producer_loop(const CUtensorMap* ta, const CUtensorMap* tb, const GemmArgs& a,
                              const Smem& s, const WaitCtx& w, uint32_t& stage_out,
                              uint32_t& phase_out, uint32_t& issued_mask) {
  uint32_t stage = 0, phase = 0;
  constexpr uint32_t kTx = kAStageBytes + kBStageBytes;
  TileSeq seq;
  for (seq.begin(a); seq.valid(a); seq.next(a)) {
    const int m0 = seq.mt(a) * kBM;
    const int n0 = seq.nt(a) * kBN;
    for (int kb = 0; kb < a.k_blocks; ++kb) {
      if (!wait_parity(s.empty + 8 * stage, phase ^ 1u, w)) goto done;
      const uint32_t full = s.full + 8 * stage;
      const uint32_t sa = s.a_base + stage * kAStageBytes;
      const uint32_t sb = s.b_base + stage * kBStageBytes;
      const int k = kb * kBK;
      mbar_arrive_expect_tx(full, kTx);
      if (KIND == kKindFwd || KIND == kKindR) {
        tma_load_2d(sa, ta, k, a.row0 + m0, full);
        tma_load_2d(sb, tb, k, a.col0 + n0, full);
      } else if (KIND == kKindX) {
        tma_load_2d(sa, ta, k, m0, full);
#pragma unroll
        for (int q = 0; q < 4; ++q) tma_load_2d(sb + q * 8192, tb, n0 + 64 * q, a.col0 + k, full);
      } else {
#pragma unroll
        for (int q = 0; q < 2; ++q) tma_load_2d(sa + q * 8192, ta, m0 + 64 * q, k, full);
#pragma unroll
        for (int q = 0; q < 4; ++q) tma_load_2d(sb + q * 8192, tb, n0 + 64 * q, a.row0 + k, full);
      }
      issued_mask |= 1u << stage;
      stage_out = stage;
      phase_out = phase;
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
done:
  return;
}

template <int KIND>
__device__ void mma_loop(uint32_t tmem, const GemmArgs& a, const Smem& s, const WaitCtx& w) {
  using T = KindTraits<KIND>;
  constexpr uint32_t idesc = instr_desc_bf16(kBM, kBN, T::a_mn, T::b_mn);
  uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
  TileSeq seq;
  for (seq.begin(a); seq.valid(a); seq.next(a)) {
    if (!wait_parity(s.tempty + 8 * acc, acc_phase ^ 1u, w)) return;
    tc_fence_after();
    const uint32_t d = tmem + acc * kAccCols;
    for (int kb = 0; kb < a.k_blocks; ++kb) {
      if (!wait_parity(s.full + 8 * stage, phase, w)) return;
      tc_fence_after();
      const uint32_t sa = s.a_base + stage * kAStageBytes;
      const uint32_t sb = s.b_base + stage * kBStageBytes;
#pragma unroll
      for (int k = 0; k < kBK / kUmmaK; ++k) {
        // K-major: the 16-element K step is 32 bytes inside the swizzled row.
        // MN-major: it is two 8-row core-matrix groups, 2048 bytes.
        const uint64_t ad = T::a_mn ? smem_desc_sw128(sa + k * 2048, 8192, 1024)
                                    : smem_desc_sw128(sa + k * 32, 0, 1024);
        const uint64_t bd = T::b_mn ? smem_desc_sw128(sb + k * 2048, 8192, 1024)
                                    : smem_desc_sw128(sb + k * 32, 0, 1024);
        mma_bf16(d, ad, bd, idesc, (kb | k) != 0);
      }
      mma_commit(s.empty + 8 * stage);  // frees the stage once these MMAs have read it
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    mma_commit(s.tfull + 8 * acc);  // accumulator ready for the epilogue
    if (++acc == kNumAcc) {
      acc = 0;
      acc_phase ^= 1u;
    }
  }
}

// Forward epilogue: per row, running (max, sum of exp) over the unit's columns.
__device__ void epilogue_fwd(uint32_t tmem, const GemmArgs& a, const Smem& s, const WaitCtx& w,
                             int q, int lane) {
  uint32_t acc = 0, acc_phase = 0;
  const int r = q * 32 + lane;
  float run_m = -INFINITY, run_s = 0.f;
  TileSeq seq;
  for (seq.begin(a); seq.valid(a); seq.next(a)) {
    const int row = seq.mt(a) * kBM + r;
    const int n0 = seq.nt(a) * kBN;
    const int t = row < a.N ? a.targets[row] : -1;
    if (seq.g == 0) {
      run_m = -INFINITY;
      run_s = 0.f;
    }
    if (!wait_parity(s.tfull + 8 * acc, acc_phase, w)) return;
    tc_fence_after();
    const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      const int j0 = n0 + 32 * c;
      if (j0 >= a.V) break;  // warp-uniform
      float v[32];
      tmem_ld32(tbase + 32 * c, v);
      if (j0 + 32 > a.V) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (j0 + i >= a.V) v[i] = -INFINITY;
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
        a.zt[row] = z;
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(s.tempty + 8 * acc);
    if (++acc == kNumAcc) {
      acc = 0;
      acc_phase ^= 1u;
    }
    if (seq.last_in_unit(a) && row < a.N) {
      const int chunk = seq.nt(a) / a.group;
      a.partials[static_cast<size_t>(chunk) * a.N + row] = make_float2(run_m, run_s);
    }
  }
}

// Recompute epilogue: dZ tile (unscaled softmax - onehot) -> bf16 block buffer.
__device__ void epilogue_r(uint32_t tmem, const GemmArgs& a, const Smem& s, const WaitCtx& w,
                           int q, int lane) {
  uint32_t acc = 0, acc_phase = 0;
  const int r = q * 32 + lane;
  TileSeq seq;
  for (seq.begin(a); seq.valid(a); seq.next(a)) {
    const int lr = seq.mt(a) * kBM + r;   // row inside the block
    const int lc0 = seq.nt(a) * kBN;      // column inside the block
    const int grow = a.row0 + lr;
    int t = -1;
    float l2 = 0.f;
    if (grow < a.N) {
      t = a.targets[grow];
      l2 = a.lse[grow] * kLog2e;
    }
    const bool valid_row = t >= 0;
    if (!wait_parity(s.tfull + 8 * acc, acc_phase, w)) return;
    tc_fence_after();
    const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
    __nv_bfloat16* out = a.dz + static_cast<size_t>(lr) * a.dz_ld + lc0;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      float v[32];
      tmem_ld32(tbase + 32 * c, v);
      const int j0 = a.col0 + lc0 + 32 * c;
      uint32_t p[16];
      if (valid_row) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float d0 = exp2f(fmaf(v[i], kLog2e, -l2));
          float d1 = exp2f(fmaf(v[i + 1], kLog2e, -l2));
          if (j0 + i == t) d0 -= 1.f;
          if (j0 + i + 1 == t) d1 -= 1.f;
          if (j0 + i >= a.V) d0 = 0.f;
          if (j0 + i + 1 >= a.V) d1 = 0.f;
          p[i / 2] = pack_bf16x2(d0, d1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) p[i] = 0u;
      }
      uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(s.tempty + 8 * acc);
    if (++acc == kNumAcc) {
      acc = 0;
      acc_phase ^= 1u;
    }
  }
}

// Contraction epilogue (dX or dW): FP32 reduce-add into the accumulation
// buffer, or, when this launch produces the whole result, bf16(scale * acc).
template <int KIND>
__device__ void epilogue_acc(uint32_t tmem, const GemmArgs& a, const Smem& s, const WaitCtx& w,
                             int q, int lane) {
  uint32_t acc = 0, acc_phase = 0;
  const int r = q * 32 + lane;
  const float scale = a.final_out ? grad_scale(a) : 1.f;
  TileSeq seq;
  for (seq.begin(a); seq.valid(a); seq.next(a)) {
    const int lrow = seq.mt(a) * kBM + r;
    const int h0 = seq.nt(a) * kBN;
    // X: output row = token row; W: output row = vocab row
    int grow, limit;
    float* acc_row = nullptr;
    if (KIND == kKindX) {
      grow = a.row0 + lrow;
      limit = a.N;
      acc_row = a.acc ? a.acc + static_cast<size_t>(grow) * a.H : nullptr;
    } else {
      grow = a.col0 + lrow;
      limit = a.V;
      acc_row = a.acc ? a.acc + static_cast<size_t>(lrow) * a.H : nullptr;
    }
    const bool row_ok = grow < limit;
    if (!wait_parity(s.tfull + 8 * acc, acc_phase, w)) return;
    tc_fence_after();
    const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      const int h = h0 + 32 * c;
      if (h >= a.H) break;  // warp-uniform
      float v[32];
      tmem_ld32(tbase + 32 * c, v);
      if (!row_ok) continue;
      if (a.final_out) {
        __nv_bfloat16* o = a.final_out + static_cast<size_t>(grow) * a.H + h;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (h + 8 * i < a.H) {
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
          if (h + 4 * i < a.H)
            atomicAdd(reinterpret_cast<float4*>(o + 4 * i),
                      make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(s.tempty + 8 * acc);
    if (++acc == kNumAcc) {
      acc = 0;
      acc_phase ^= 1u;
    }
  }
}

}  // namespace

template <int KIND>
__global__ void __launch_bounds__(kGemmThreads, 1)
    flce_gemm_kernel(const __grid_constant__ CUtensorMap tma_a,
                     const __grid_constant__ CUtensorMap tma_b, const GemmArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  Smem s;
  s.a_base = base;
  s.b_base = base + kStages * kAStageBytes;
  const uint32_t bar0 = s.b_base + kStages * kBStageBytes;
  s.full = bar0;
  s.empty = bar0 + 8 * kStages;
  s.tfull = bar0 + 16 * kStages;
  s.tempty = s.tfull + 8 * kNumAcc;
  s.drain = s.tempty + 8 * kNumAcc;
  uint8_t* gbar_end = gbase + (s.drain + 8 - base);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbar_end);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(s.full + 8 * i, 1);
      mbar_init(s.empty + 8 * i, 1);
    }
    for (int i = 0; i < kNumAcc; ++i) {
      mbar_init(s.tfull + 8 * i, 1);
      mbar_init(s.tempty + 8 * i, 4);
    }
    mbar_init(s.drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  WaitCtx w{abort_flag, args.err, args.wait_limit_ns};

  if (warp == 0) {
    if (lane == 0) {
      uint32_t st = 0, ph = 0, issued = 0;
      producer_loop<KIND>(&tma_a, &tma_b, args, s, w, st, ph, issued);
      // Drain: every stage's most recent load must have landed before the CTA
      // may exit (its shared memory is the copy's destination).
      for (int i = 0; i < kStages; ++i) {
        if (!(issued & (1u << i))) continue;
        // most recent phase issued on stage i
        const uint32_t ph_i = (static_cast<uint32_t>(i) <= st) ? ph : (ph ^ 1u);
        WaitCtx wd{abort_flag, args.err, args.wait_limit_ns};
        volatile uint32_t never = 0u;
        wd.abort = &never;  // keep waiting even if the CTA aborted
        wait_parity(s.full + 8 * i, ph_i, wd);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      mma_loop<KIND>(tmem, args, s, w);
      // Drain: all issued MMAs complete before TMEM is released.
      mma_commit(s.drain);
      WaitCtx wd{abort_flag, args.err, args.wait_limit_ns};
      volatile uint32_t never = 0u;
      wd.abort = &never;
      wait_parity(s.drain, 0u, wd);
    }
  } else {
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    if (KIND == kKindFwd)
      epilogue_fwd(tmem, args, s, w, q, lane);
    else if (KIND == kKindR)
      epilogue_r(tmem, args, s, w, q, lane);
    else
      epilogue_acc<KIND>(tmem, args, s, w, q, lane);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_gemm(GemmKind kind, const CUtensorMap& ta, const CUtensorMap& tb,
                        const GemmArgs& a, int grid, cudaStream_t st) {
  if (grid <= 0) return cudaSuccess;
  static bool attr_done[4] = {false, false, false, false};
  cudaError_t e = cudaSuccess;
#define FLCE_LAUNCH(K)                                                                        \
  do {                                                                                        \
    if (!attr_done[K]) {                                                                      \
      e = cudaFuncSetAttribute(flce_gemm_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                               kGemmSmemBytes);                                               \
      if (e != cudaSuccess) return e;                                                         \
      attr_done[K] = true;                                                                    \
    }                                                                                         \
    flce_gemm_kernel<K><<<grid, kGemmThreads, kGemmSmemBytes, st>>>(ta, tb, a);               \
  } while (0)
  switch (kind) {
    case kKindFwd: FLCE_LAUNCH(kKindFwd); break;
    case kKindR: FLCE_LAUNCH(kKindR); break;
    case kKindX: FLCE_LAUNCH(kKindX); break;
    case kKindW: FLCE_LAUNCH(kKindW); break;
  }
#undef FLCE_LAUNCH
  note_launch();
  return cudaGetLastError();
}

}  // namespace flce
