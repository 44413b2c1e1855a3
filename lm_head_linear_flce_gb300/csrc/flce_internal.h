// Internal declarations shared by the host API and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace flce {

// Bits of the device error word (first int of the workspace).
constexpr int kErrLabel = 1;    // a target outside the vocabulary that is not ignore_index
constexpr int kErrTimeout = 2;  // a bounded wait ran out
// Rows per block of the forward's log-sum-exp merge: the loss partials hold
// one FP64 value per kMergeRows rows.
constexpr int kMergeRows = 32;
// Stored target of a valid row whose label lies in another vocabulary shard:
// no column of this call matches it, so the row has softmax terms only.
constexpr int kTargetElsewhere = 0x7fffffff;

// GEMM tile geometry (all tensor-core kernels).  Tiles are computed by a pair
// of CTAs (a 2-CTA cluster on two SMs) with tcgen05 cta_group::2: a tile is
// 256 rows x 256 columns; each CTA holds 128 rows of A and 128 of the 256 B
// columns in shared memory and 128 rows x 256 columns of the FP32 result in
// its tensor memory.
constexpr int kPairM = 256;     // tile rows over the pair (MMA M)
constexpr int kBM = 128;        // tile rows per CTA
constexpr int kBN = 256;        // tile columns (MMA N)
constexpr int kHalfN = 128;     // B columns per CTA
constexpr int kBK = 64;         // K per pipeline stage: one 128-byte swizzle row of bf16
constexpr int kUmmaK = 16;      // K per tcgen05.mma (bf16)
constexpr int kStages = 6;      // shared-memory pipeline depth
constexpr int kAStageBytes = kBM * kBK * 2;     // 16 KB
constexpr int kBStageBytes = kHalfN * kBK * 2;  // 16 KB
constexpr int kAccCols = kBN;   // FP32 accumulator columns per tile
constexpr int kNumAcc = 2;      // double-buffered accumulators
constexpr int kTmemCols = kAccCols * kNumAcc;  // 512: the whole tensor memory
constexpr int kGemmThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kFwdGroup = 4;    // fewest vocab tiles merged per forward work unit
// Most forward work units per 256-row tile: each unit covers a contiguous run
// of at least kFwdGroup vocab tiles and leaves one (max, sum-exp) partial per
// row, so the partials are O(N * kFwdSplits) whatever V is.  128 keeps units
// short enough (5 tiles at V = 152K) that the dynamic hand-out ends evenly.
constexpr int kFwdSplits = 128;
constexpr int kGemmSmemBytes = kStages * (kAStageBytes + kBStageBytes) + 1024 /*align*/ + 256;
// backward epilogue staging: per epilogue warp two 4 KB buffers (32 rows x 128 B)
constexpr int kStageBufBytes = 4096;
constexpr int kBwdSmemBytes = kGemmSmemBytes + 4 * 2 * kStageBufBytes;

// Kinds of GEMM tile.
enum GemmKind : int {
  kKindR = 1,    // Z = X W^T tile recomputed; epilogue: dZ = softmax - onehot -> bf16 block
  kKindX = 2,    // dX tile += dZ_block . W_block; A K-major, B MN-major
  kKindW = 3,    // dW tile += dZ_block^T . X_block; A MN-major, B MN-major
};

// Forward GEMM launch.
struct GemmArgs {
  int tiles_m, tiles_n, group, units, k_blocks;
  int band;  // row tiles per band: units go band by band, vocab group by vocab
             // group within a band, row tile fastest (a band's X rows stay in L2)
  int N, H, V;
  const int* targets;  // [N]: local column, -1 (no valid target) or kTargetElsewhere
  float2* partials;    // [units_n][N]: per-row (max, sum exp(z - max)) over a work unit
  float* zt;           // [N]: target logit
  int* counter;        // unit ticket counter (starts at 0); loss forward only
  int* err;
  unsigned long long wait_limit_ns;
};

// One dZ block of the backward: the 256-row tiles active[tile0 .. tile0 + mt)
// (at most `mt`; fewer when rows without a target were left out) x vocab
// columns [col0, col0 + vt*256), stored in dZ slot `slot`.  Local dZ row l of
// the block is row active[tile0 + l / 256] * 256 + l % 256 of the X the
// backward reads (a token row, or a dense row of the gathered copy).
struct BlockDesc {
  int tile0, col0;
  int mt;     // at most this many 256-row token tiles
  int vt;     // 256-column vocab tiles (R tiles per row tile; W tiles; X tiles' K / 256)
  int slot;
};

// Tensor maps of the backward (passed as one __grid_constant__ parameter).
struct BwdMaps {
  CUtensorMap x_k;       // X [N][H], box 64 x 128 (R: A operand)
  CUtensorMap w_k;       // W [V][H], box 64 x 128 (R: B operand, one CTA's half)
  CUtensorMap w_mn;      // W [V][H], box 64 x 64  (X: B operand, MN-major)
  CUtensorMap x_mn;      // X [N][H], box 64 x 64  (W: B operand, MN-major)
  CUtensorMap dz_k[2];   // dZ slot [Nb][Vb], box 64 x 128 (X: A operand)
  // MN-major operand halves as one box each: a 3-D view (64 elements, rows,
  // 64-element groups) with box 64 x 64 rows x 2 groups lands in shared memory
  // exactly as two 64 x 64 boxes 8 KB apart.  W and X use it when H % 64 == 0
  // (otherwise w_mn / x_mn, two boxes); the dZ slot always does (W: A operand).
  CUtensorMap w_mn3;     // W  (64, V, H/64)
  CUtensorMap x_mn3;     // X  (64, N, H/64)
  CUtensorMap dz_mn3[2]; // dZ slot (64, Nb, Vb/64)
  // epilogue stores, box = one warp's 32 rows x 128 bytes
  CUtensorMap dz_st[2];  // dZ slot [Nb][Vb] bf16, box 64 x 32 (R: dZ store)
  CUtensorMap dx_out;    // dX accumulator [N][H] f32 box 32 x 32 (reduce-add), or
                         // dX [N][H] bf16 box 64 x 32 (store) when written directly
  CUtensorMap dw_out;    // dW band [Vb][H] f32 box 32 x 32 (reduce-add), or
                         // dW [V][H] bf16 box 64 x 32 (store) when written directly
};

// One backward launch: the R tiles of block `r`, the X tiles of the same block
// (each X tile starts once the R tiles of its 256-row token tile have stored
// their dZ, counted in `row_done`), and the W tiles of block `w` (the previous
// block, complete when the launch starts).
struct BwdArgs {
  BlockDesc r, w;
  int* row_done;   // per local 256-row tile of block r: dZ stores finished, one
                   // count per epilogue warp (8 per R tile; 8 * r.vt when complete)
  int x_lag;       // X tiles of a row tile are handed out this many row tiles
                   // after its R tiles
  int want_dx, want_dw;  // which contractions run (dX tiles, dW tiles)
  int h_tiles;           // 256-column tiles of H
  const int* active;     // 256-row tiles of the rows the backward reads, ascending:
                         // the token tiles holding a target, or 0, 1, ... over
                         // the dense rows gathered to the front of X's copy
  const int* n_active;   // number of entries of `active`
  int kb_h;  // K blocks of the recompute (ceil(H / 64))
  int mn3d;  // 1: MN-major halves load as one 3-D box (w_mn3 / x_mn3 / dz_mn3)
  int N, H, V;
  const int* targets;  // per row of that X (token rows, or the dense rows)
  const float* lse;     // likewise
  __nv_bfloat16* dz[2];
  int dz_ld;
  float* dxf;                  // FP32 dX accumulator [N][H], or null
  __nv_bfloat16* dx_final;     // bf16 dX written directly (single vocab block), or null
  float* dwf;                  // FP32 dW band [Vb][H], or null
  __nv_bfloat16* dw_final;     // bf16 dW written directly (single token block), or null
  int dw_accumulate;           // 1: W tiles add scale * dW into the caller's FP32 gradient
  int dx_accumulate;           // 1: X tiles add scale * dX into the caller's FP32 buffer (dxf)
  const float* grad_loss;
  const long long* n_valid;
  int reduction;               // 0 mean, 1 sum
  int* counter;                // ticket counter of this launch (starts at 0)
  int* err;
  unsigned long long wait_limit_ns;
};

// Host-side plan of one problem: tile counts, backward blocking and the
// workspace layout.  Pure function of (N, H, V).
struct Plan {
  int64_t N, H, V;
  int m_tiles, v_tiles, h_tiles;
  int fwd_group;          // vocab tiles per forward work unit
  int v_units;            // forward work units per 256-row tile (<= kFwdSplits)
  int64_t Nb, Vb;         // backward block: token rows x vocab columns
  int64_t dz_ld;          // elements per dZ row in a slot (Vb plus padding)
  int n_blocks, v_blocks;
  bool multi_n;           // more than one token block: dW needs an FP32 band
  int launches;           // backward GEMM launches (one per dZ block, plus one)
  size_t off_err, off_t, off_zt, off_part, off_lossp, off_fcnt, off_cnt, off_flags, off_active,
      off_toff, off_tc, off_lc, off_inv, off_done, off_dxf, off_dwf, off_dz;
  size_t total;
};

bool make_plan(int64_t N, int64_t H, int64_t V, Plan* p);

// Row tiles per band of the forward's unit order: as many as keep the band's
// X rows (256 * H * 2 bytes per row tile) within kFwdBandBytes, balanced over
// the bands.  With one band the order is plain vocab group by vocab group.
constexpr int64_t kFwdBandBytes = int64_t{40} << 20;
inline int forward_band_tiles(int64_t m_tiles, int64_t H) {
  const int64_t per_tile = int64_t{256} * H * 2;
  int64_t cap = kFwdBandBytes / per_tile;
  if (cap < 1) cap = 1;
  const int64_t bands = (m_tiles + cap - 1) / cap;
  return static_cast<int>(bands > 0 ? (m_tiles + bands - 1) / bands : 1);
}

// Vocab tiles per forward work unit for a vocabulary of v_tiles 256-column
// tiles: at least kFwdGroup, and few enough units (<= kFwdSplits) per row tile.
inline int forward_unit_tiles(int64_t v_tiles) {
  const int64_t by_splits = (v_tiles + kFwdSplits - 1) / kFwdSplits;
  return static_cast<int>(by_splits > kFwdGroup ? by_splits : kFwdGroup);
}

// The limit every bounded wait of the next launches uses (flce_set_wait_limit_ns).
unsigned long long wait_limit_ns();

// Counts one kernel launch (see flce_kernel_launch_count).
void note_launch();
// Records the wait limit a tensor-core launch was given (see
// flce_last_launch_wait_limit_ns).
void note_wait_limit(unsigned long long limit_ns);

// 2-D tensor map over a row-major [outer][inner] matrix (rows `row_bytes`
// apart) with 128-byte swizzle and the given box; out-of-bounds elements read
// as zero and are not written.  False if the CUDA driver rejects it.
bool make_tmap(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);

// The vocabulary columns a call holds: [v_offset, v_offset + V_local) of a
// V_total-column vocabulary (the whole of it outside the vocabulary-parallel
// entry points).
struct VocabSlice {
  int64_t V_total, v_offset, V_local;
};

// Launchers (return cudaGetLastError()).
// targets[i]: -1 (no valid target), the local column, or kTargetElsewhere.
// tile_flags (or null): for every 256-row tile, its number of rows with a valid
// target.
cudaError_t launch_prep_targets(const int64_t* labels, int N, int seq_len, int shift,
                                int64_t ignore_index, const VocabSlice& vs, int* targets,
                                long long* n_valid, int* err, cudaStream_t st,
                                int* tile_flags = nullptr);
// active[0 .. *n_active) = indices of the flagged tiles, ascending.
cudaError_t launch_compact_tiles(const int* tile_flags, int m_tiles, int* active, int* n_active,
                                 cudaStream_t st);
// Dense rows: toff[0 .. m_tiles] = exclusive scan of the per-tile counts (the
// last entry: all valid rows), active[t] = t for the ceil(rows / 256) dense
// tiles, *n_active = their number.
cudaError_t launch_compact_rows(const int* counts, int m_tiles, int* toff, int* active,
                                int* n_active, cudaStream_t st);
// Copies the rows with a valid target of X [N][H] bf16 to the front of xc
// [N][H] (zeroing the rest of the last dense tile), their targets to tc and
// lse to lc, and writes inv[i] = the dense index of row i, or -1.  xc must not
// overlap X.
cudaError_t launch_gather_rows(const void* X, const int* targets, const float* lse,
                               const int* toff, int N, int H, int m_tiles, void* xc, int* tc,
                               float* lc, int* inv, cudaStream_t st);
// dst row i = bf16_rn(scale * src row inv[i]), or 0 where inv[i] < 0.
cudaError_t launch_downcast_rows(const float* src, __nv_bfloat16* dst, const int* inv, int N,
                                 int H, const float* grad_loss, const long long* n_valid,
                                 int reduction, cudaStream_t st);
// z_out non-null: a vocabulary shard's (lse, target logit) instead of a loss.
cudaError_t launch_merge_lse(const float2* partials, int nchunks, int N, const float* zt,
                             const int* targets, float* lse, double* loss_partials,
                             cudaStream_t st, int* nblocks_out, float* z_out = nullptr);
cudaError_t launch_merge_shards(const float* lse_parts, const float* z_parts, int P, int N,
                                const int* targets, float* lse, double* loss_partials,
                                cudaStream_t st, int* nblocks_out);
cudaError_t launch_finalize_loss(const double* loss_partials, int nblocks,
                                 const long long* n_valid, int reduction, float* loss,
                                 cudaStream_t st);
cudaError_t launch_downcast(const float* src, __nv_bfloat16* dst, size_t count,
                            const float* grad_loss, const long long* n_valid, int reduction,
                            cudaStream_t st);
cudaError_t launch_selftest_wait(unsigned long long limit_ns, int* err, cudaStream_t st);
// Tensor-core launches: `units` work items over at most as many CTA pairs as
// fit on the device at once.
cudaError_t launch_fwd_gemm(const CUtensorMap& tx, const CUtensorMap& tw, const GemmArgs& a,
                            int units, cudaStream_t st);
cudaError_t launch_logits_gemm(const CUtensorMap& tx, const CUtensorMap& tw,
                               const CUtensorMap& tout, const GemmArgs& a, int units,
                               cudaStream_t st);
// overlap_prior: the preceding operation of the stream is the previous backward
// launch, which this one may overlap (programmatic dependent launch).
cudaError_t launch_bwd_gemm(const BwdMaps& maps, const BwdArgs& a, int units, bool overlap_prior,
                            cudaStream_t st);

}  // namespace flce
