// Internal declarations shared by the host API and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace flce {

// Bits of the device error word (first int of the workspace).
constexpr int kErrLabel = 1;    // a target outside [0, V) that is not ignore_index
constexpr int kErrTimeout = 2;  // a bounded wait ran out

// GEMM tile geometry (all tensor-core kernels).
constexpr int kBM = 128;        // rows of a tile (MMA M)
constexpr int kBN = 256;        // columns of a tile (MMA N)
constexpr int kBK = 64;         // K per pipeline stage: one 128-byte swizzle row of bf16
constexpr int kUmmaK = 16;      // K per tcgen05.mma (bf16)
constexpr int kStages = 4;      // shared-memory pipeline depth
constexpr int kAStageBytes = kBM * kBK * 2;  // 16 KB
constexpr int kBStageBytes = kBN * kBK * 2;  // 32 KB
constexpr int kAccCols = kBN;   // FP32 accumulator columns per tile
constexpr int kNumAcc = 2;      // double-buffered accumulators
constexpr int kTmemCols = kAccCols * kNumAcc;  // 512: the whole tensor memory
constexpr int kGemmThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kFwdGroup = 4;    // vocab tiles merged per forward work unit
constexpr int kGemmSmemBytes = kStages * (kAStageBytes + kBStageBytes) + 1024 /*align*/ + 256;

// Kinds of GEMM tile.
enum GemmKind : int {
  kKindFwd = 0,  // Z = X W^T tile; epilogue: online log-sum-exp + target logit
  kKindR = 1,    // Z = X W^T tile recomputed; epilogue: dZ = softmax - onehot -> bf16 block
  kKindX = 2,    // dX tile += dZ_block . W_block; A K-major, B MN-major
  kKindW = 3,    // dW tile += dZ_block^T . X_block; A MN-major, B MN-major
};

struct GemmArgs {
  // tile grid of this launch
  int tiles_m, tiles_n, group, units, k_blocks;
  // coordinate offsets
  int row0;   // global token row of local row 0 (FWD/R/X: M rows; W: K rows)
  int col0;   // global vocab index of local column 0 (FWD/R: N cols; X: K rows; W: M rows)
  // problem sizes
  int N, H, V;
  // forward
  const int* targets;  // [N], -1 = no valid target
  float2* partials;    // [units_n][N]: per-row (max, sum exp(z - max)) over a work unit
  float* zt;           // [N]: target logit
  // backward recompute
  const float* lse;
  __nv_bfloat16* dz;   // dZ block buffer, row-major, dz_ld columns
  int dz_ld;
  // backward contractions
  float* acc;                 // FP32 accumulation target (dX: [N][H], dW band: [Vb][H])
  __nv_bfloat16* final_out;   // if non-null: write bf16(scale * result) here instead
  const float* grad_loss;
  const long long* n_valid;
  int reduction;              // 0 mean, 1 sum
  // errors / waits
  int* err;
  unsigned long long wait_limit_ns;
};

// Host-side plan of one problem: tile counts, backward blocking and the
// workspace layout.  Pure function of (N, H, V).
struct Plan {
  int64_t N, H, V;
  int m_tiles, v_tiles, v_units, h_tiles;
  int64_t Nb, Vb;         // backward block: token rows x vocab columns
  int n_blocks, v_blocks;
  bool multi_n;           // more than one token block: dW needs an FP32 band
  size_t off_err, off_t, off_zt, off_part, off_lossp, off_nvalid, off_dxf, off_dwf, off_dz;
  size_t total;
};

bool make_plan(int64_t N, int64_t H, int64_t V, Plan* p);

// Counts one kernel launch (see flce_kernel_launch_count).
void note_launch();

// Launchers (return cudaGetLastError()).
cudaError_t launch_prep_targets(const int64_t* labels, int N, int seq_len, int shift,
                                int64_t ignore_index, int V, int* targets,
                                long long* n_valid, int* err, cudaStream_t st);
cudaError_t launch_merge_lse(const float2* partials, int nchunks, int N, const float* zt,
                             const int* targets, float* lse, double* loss_partials,
                             cudaStream_t st, int* nblocks_out);
cudaError_t launch_finalize_loss(const double* loss_partials, int nblocks,
                                 const long long* n_valid, int reduction, float* loss,
                                 cudaStream_t st);
cudaError_t launch_downcast(const float* src, __nv_bfloat16* dst, size_t count,
                            const float* grad_loss, const long long* n_valid, int reduction,
                            cudaStream_t st);
cudaError_t launch_selftest_wait(unsigned long long limit_ns, int* err, cudaStream_t st);
cudaError_t launch_gemm(GemmKind kind, const CUtensorMap& ta, const CUtensorMap& tb,
                        const GemmArgs& a, int grid, cudaStream_t st);

}  // namespace flce
