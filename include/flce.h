/*
 * flce.h — fused linear cross-entropy on one GB300 GPU (sm_103a), C ABI.
 *
 * The operation (ms-swift PR #9784 "feat(sft): Add optional fused linear ce for
 * qwen2/qwen3 on npu", sections Background, What this PR does and Mathematical
 * Equivalence):
 *
 *     Z = X W^T                     X: N x H token hidden states, W: V x H
 *     loss = reduce_i CE(Z_i, t_i)  per-row cross-entropy against target t_i
 *     dX = dZ W,  dW = dZ^T X       dZ = (softmax(Z) - onehot(t)) * g / n_valid
 *
 * computed without ever holding the N x V logits.  The call surface mirrors
 * `linear_cross_entropy(hidden, weight, labels, ignore_index=-100, shift=True,
 * reduction="mean")` with W stored (vocab, hidden) (Qwen3.5-35B-A3B LoRA SFT
 * blog post, listing `_patch_model_with_cce`), and gradients are accumulated in
 * FP32 and rounded to bf16 only at the end (Megatron-LM PR #2739 "[Dev] Fix
 * Linear-Cross-Entropy Convergence Issue", section 2).
 *
 * Conventions shared by every entry point
 *   - Pointers marked "device" are CUDA device pointers on the current device;
 *     the caller allocates and owns every buffer.  The library allocates no
 *     device memory and keeps no state between calls.
 *   - Everything is enqueued on `stream` and runs asynchronously; no entry point
 *     synchronises except flce_get_error.
 *   - X and W are bf16, row-major, rows contiguous: X[i*H + h], W[v*H + h].
 *     H must be a multiple of 8 (16-byte rows for the TMA tensor copies) and
 *     both base pointers 16-byte aligned.
 *   - labels are int64.  With shift != 0, row s of each length-seq_len sequence
 *     is scored against labels[s+1] of the same sequence and the last row of
 *     every sequence is ignored; N must be a multiple of seq_len (seq_len <= 0
 *     means one sequence of N rows).  With shift == 0, row i uses labels[i].
 *   - A target equal to ignore_index is ignored, even if it lies in [0, V).  A
 *     target outside [0, V) that is not ignore_index sets
 *     FLCE_ERR_LABEL_OUT_OF_RANGE in the workspace error word (see
 *     flce_get_error) and its row is treated as ignored; the call still
 *     completes.
 *   - reduction MEAN divides by n_valid, the number of valid targets in the
 *     whole call; with n_valid == 0 the loss and gradients are 0.
 *   - Host-detectable errors (null pointers, bad sizes, short workspace,
 *     overlapping outputs of a backward call, a device older than sm_103) are
 *     returned at once and nothing is enqueued.  No exception crosses the ABI
 *     and no kernel traps.
 */
#ifndef FLCE_H
#define FLCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default stream. */
typedef struct CUstream_st* flce_stream_t;

typedef enum {
  FLCE_OK = 0,
  FLCE_ERR_INVALID_ARG = 1,        /* null pointer, bad enum, N % seq_len != 0 ... */
  FLCE_ERR_UNSUPPORTED_SHAPE = 2,  /* H % 8 != 0, H/V/N outside the supported range */
  FLCE_ERR_WORKSPACE_TOO_SMALL = 3,
  FLCE_ERR_LABEL_OUT_OF_RANGE = 4, /* device-detected: reported by flce_get_error */
  FLCE_ERR_TIMEOUT = 5,            /* device-detected: a bounded wait ran out */
  FLCE_ERR_CUDA = 6,               /* a CUDA runtime call failed */
  FLCE_ERR_UNSUPPORTED_DEVICE = 7  /* not an sm_103 (GB300-class) device */
} flce_status;

typedef enum { FLCE_REDUCTION_MEAN = 0, FLCE_REDUCTION_SUM = 1 } flce_reduction;

/*
 * Bytes of device workspace flce_forward and flce_backward need for these
 * sizes (one buffer serves both; it need not survive from forward to
 * backward).  It is O(N*H + Vb*H + Nb*Vb + 128*N + tiles), never O(N*V):
 * FP32 accumulators for dX and for one vocab band of dW, two bounded bf16
 * blocks of dZ (Nb x Vb each, at most 2^27 elements; see
 * flce_set_backward_block), per-row partial log-sum-exps (at most 128 per
 * row, whatever V is), and 16 bytes per row of targets and of the dense-row
 * maps of the backward.
 * Returns 0 for invalid sizes.
 */
size_t flce_workspace_size(int64_t N, int64_t H, int64_t V);

/*
 * Forward: loss, per-row log-sum-exp and the valid-target count.
 *
 *   X, W            device, bf16, see conventions.
 *   labels          device, int64 [N].
 *   loss            device float, 1 element: mean or sum of the per-row
 *                   losses lse_i - z_{i,t_i} over valid rows (deterministic).
 *   lse             device float [N]: log sum_j exp(Z_ij) for every row, valid
 *                   or not (it does not depend on labels).
 *   n_valid         device int64, 1 element (exact).
 *   workspace       device, >= flce_workspace_size(N, H, V) bytes, 256-byte
 *                   aligned; its error word is reset at the start of the call.
 * N == 0 is allowed: loss = 0 and n_valid = 0.
 */
flce_status flce_forward(const void* X, const void* W, const int64_t* labels,
                         int64_t N, int64_t H, int64_t V, int64_t seq_len,
                         int64_t ignore_index, int shift, flce_reduction reduction,
                         float* loss, float* lse, int64_t* n_valid,
                         void* workspace, size_t workspace_bytes, flce_stream_t stream);

/*
 * Backward: dX and/or dW for upstream gradient g of the loss.
 *
 *   lse, n_valid    device, as written by flce_forward for the same inputs.
 *   grad_loss       device float, 1 element: g = d(outer loss)/d(loss).
 *   dX              device bf16 [N, H] or NULL to skip it (e.g. when only W is
 *                   trained); written, not accumulated.  While the call runs
 *                   it may hold a dense copy of the rows of X that have a
 *                   valid target.
 *   dW              device bf16 [V, H] or NULL to skip it (a frozen LM head,
 *                   as in LoRA fine-tuning); written, not accumulated.
 * No output may overlap an input (X, W, labels, lse, n_valid, grad_loss), the
 * workspace or the other output: FLCE_ERR_INVALID_ARG (so for every backward
 * entry point, with dW_acc and dX_acc as outputs).
 * Gradients are accumulated in FP32 and rounded to bf16 (round to nearest even)
 * once, after the scale g / n_valid (mean) or g (sum) is applied in FP32.
 * Rows without a valid target contribute nothing: with dX requested and V
 * spanning several dZ blocks, the rows that have one are gathered into dX's
 * buffer and the contractions run on ceil(rows / 256) dense 256-row tiles (dX
 * is put back in token order, 0 on the other rows, by the final downcast);
 * otherwise they run on the 256-row token tiles that hold a valid target.
 * The other arguments have the same meaning as in flce_forward.
 */
flce_status flce_backward(const void* X, const void* W, const int64_t* labels,
                          int64_t N, int64_t H, int64_t V, int64_t seq_len,
                          int64_t ignore_index, int shift, flce_reduction reduction,
                          const float* lse, const int64_t* n_valid, const float* grad_loss,
                          void* dX, void* dW,
                          void* workspace, size_t workspace_bytes, flce_stream_t stream);

/*
 * Backward with dW accumulated into an existing FP32 gradient:
 *
 *   dW_acc[V][H] += s * dZ^T X        (s = g / n_valid for mean, g for sum)
 *
 * for a weight whose gradient has other contributions too, e.g. an LM head
 * tied to the input embedding, or gradient accumulation over micro-batches
 * (Megatron-LM PR #2739, section 1: the fused loss must feed the output
 * layer's own weight gradient).  dW_acc: device float [V][H], 16-byte
 * aligned, read and written (not overwritten).  dX (bf16 or NULL) and the
 * other arguments are as in flce_backward.  The FP32 additions into dW_acc and
 * into the internal dX accumulator happen in a fixed order (one per vocab /
 * token block, in launch order), so repeated calls give bitwise-identical
 * results.
 */
flce_status flce_backward_accumulate(const void* X, const void* W, const int64_t* labels,
                                     int64_t N, int64_t H, int64_t V, int64_t seq_len,
                                     int64_t ignore_index, int shift, flce_reduction reduction,
                                     const float* lse, const int64_t* n_valid,
                                     const float* grad_loss, void* dX, float* dW_acc,
                                     void* workspace, size_t workspace_bytes,
                                     flce_stream_t stream);

/*
 * Plain logits, for calls without labels (inference / generation): the
 * fused path falls back to the LM head itself, Z = X W^T (ms-swift PR #9784,
 * section Safety & Compatibility: "labels=None" falls back to lm_head).
 *
 *   logits     device bf16 [N][ld_logits], row-major; columns [V, ld_logits)
 *              are left untouched.  ld_logits >= V and a multiple of 8;
 *              16-byte aligned.  Each value is the FP32 accumulation rounded
 *              to bf16 (round to nearest even).
 * Needs no workspace and holds N x V memory by definition (the caller asked
 * for the logits).  Errors as for flce_forward.
 */
flce_status flce_logits(const void* X, const void* W, int64_t N, int64_t H, int64_t V,
                        void* logits, int64_t ld_logits, flce_stream_t stream);

/*
 * Vocabulary-parallel split (Megatron-LM PR #2739 "[Dev] Fix
 * Linear-Cross-Entropy Convergence Issue": section 1, the output layer is a
 * ColumnParallelLinear, so its vocabulary rows are split across P ranks;
 * section 2, the d_hidden contributions of the vocabulary slices are summed in
 * an FP32 buffer and downcast to bf16 once).  Every rank holds the same X and
 * labels and the W rows [v_offset, v_offset + V) of a V_total-row vocabulary.
 * Per rank, in order:
 *
 *   flce_forward_vocab_shard   this shard's per-row lse_r and target logit z_r
 *   (the caller gathers every rank's lse_r and z_r, e.g. one all-gather)
 *   flce_merge_vocab_shards    loss, the whole-vocabulary lse and n_valid
 *   flce_backward_vocab_shard  dW of the shard; dX_acc += this shard's dX part
 *   (the caller sums dX_acc over the ranks in FP32, e.g. one all-reduce)
 *   flce_downcast_bf16         dX in bf16
 *
 * Validity is judged against the whole vocabulary: a target in [0, V_total)
 * that lies in another rank's shard is valid here, with no one-hot term on
 * this rank.  Labels outside [0, V_total) are reported as in flce_forward.
 * Requires 0 <= v_offset and v_offset + V <= V_total.  The workspace is sized
 * with flce_workspace_size(N, H, V) of the shard.
 *
 * flce_forward_vocab_shard
 *   W_shard     device bf16 [V][H]: vocabulary rows v_offset .. v_offset+V-1.
 *   lse_shard   device float [N]: log sum over this shard's columns of exp(Z_ij).
 *   z_shard     device float [N]: Z_{i,t_i} if t_i is valid and in this shard,
 *               else 0.
 *   n_valid     device int64, 1 element: valid targets over the whole vocabulary.
 */
flce_status flce_forward_vocab_shard(const void* X, const void* W_shard, const int64_t* labels,
                                     int64_t N, int64_t H, int64_t V, int64_t v_offset,
                                     int64_t V_total, int64_t seq_len, int64_t ignore_index,
                                     int shift, float* lse_shard, float* z_shard,
                                     int64_t* n_valid, void* workspace, size_t workspace_bytes,
                                     flce_stream_t stream);

/*
 * flce_merge_vocab_shards
 *   lse_parts, z_parts  device float [P][N]: every rank's lse_shard and z_shard,
 *                       in any rank order (the same order in both).
 *   labels, seq_len, ignore_index, shift   as in the shard calls; V_total the
 *                       whole vocabulary.
 *   loss                device float: mean or sum over valid rows of
 *                       lse_i - z_i, with lse_i = log sum_r exp(lse_parts[r][i])
 *                       and z_i = sum_r z_parts[r][i] (deterministic).
 *   lse                 device float [N]: the whole-vocabulary log-sum-exp.
 *   n_valid             device int64, 1 element.
 *   workspace           any workspace valid for the shard calls with this N
 *                       (it needs 256 + 4N + 8(N/256 + 2) bytes, each term
 *                       rounded up to 256).
 * 1 <= P <= 65536.
 */
flce_status flce_merge_vocab_shards(const float* lse_parts, const float* z_parts, int64_t P,
                                    const int64_t* labels, int64_t N, int64_t V_total,
                                    int64_t seq_len, int64_t ignore_index, int shift,
                                    flce_reduction reduction, float* loss, float* lse,
                                    int64_t* n_valid, void* workspace, size_t workspace_bytes,
                                    flce_stream_t stream);

/*
 * flce_backward_vocab_shard
 *   lse, n_valid   device, as written by flce_merge_vocab_shards.
 *   grad_loss      device float, 1 element: g.
 *   dX_acc         device float [N][H], 16-byte aligned, or NULL:
 *                  dX_acc += s * dZ_r W_shard, s = g / n_valid (mean) or g
 *                  (sum), dZ_r the shard's columns of dZ; read and written (the
 *                  caller zeroes it first, or adds to another contribution).
 *   dW_shard       device bf16 [V][H] or NULL: this shard's rows of dW, written.
 * The other arguments are as in flce_forward_vocab_shard.
 */
flce_status flce_backward_vocab_shard(const void* X, const void* W_shard, const int64_t* labels,
                                      int64_t N, int64_t H, int64_t V, int64_t v_offset,
                                      int64_t V_total, int64_t seq_len, int64_t ignore_index,
                                      int shift, flce_reduction reduction, const float* lse,
                                      const int64_t* n_valid, const float* grad_loss,
                                      float* dX_acc, void* dW_shard, void* workspace,
                                      size_t workspace_bytes, flce_stream_t stream);

/*
 * dst[k] = bf16(src[k]) (round to nearest even) for k < count: the one
 * downcast of a summed FP32 gradient.  count a multiple of 8; both pointers
 * device, 16-byte aligned.
 */
flce_status flce_downcast_bf16(const float* src, void* dst, int64_t count,
                               flce_stream_t stream);

/*
 * Synchronises `stream`, then reads and returns the device error word written
 * by the last call that used this workspace (each call taking a workspace
 * resets the word when it starts): FLCE_OK, FLCE_ERR_LABEL_OUT_OF_RANGE or
 * FLCE_ERR_TIMEOUT (a timeout outranks a label error).  FLCE_ERR_CUDA if the
 * synchronisation itself fails.
 */
flce_status flce_get_error(const void* workspace, flce_stream_t stream);

/* A static, human-readable name for a status code. */
const char* flce_status_string(flce_status status);

/*
 * Limit, in nanoseconds, on every wait inside the library's kernels (default
 * 2e9), flce_forward_noalloc's included; it applies to calls made after it is
 * set.  A wait that runs out records FLCE_ERR_TIMEOUT and its kernel returns
 * early.  Values <= 0 restore the default.  Process-wide.
 */
void flce_set_wait_limit_ns(int64_t limit_ns);

/*
 * Tuning: caps the backward's dZ block at `max_rows` token rows (rounded down
 * to a multiple of 256, at least 256) and `max_block_elems` bf16 elements.
 * A value <= 0 leaves that cap automatic: at most 32 Mi elements (a 64 MB
 * block) when N <= 8192 and 64 Mi (128 MB) above, and every token row in one
 * block while that leaves at least 2048 vocab columns per block (so dW is
 * written once, with no FP32 accumulator across token blocks); above 8192
 * rows, with every row in one block, the cap doubles (up to 128 Mi elements,
 * 256 MB) while a block would hold fewer than 76 dW tiles of 256 x 256; and
 * the block's vocab width Vb is then capped so that its W rows (Vb x H bf16)
 * take at most 64 MiB (a multiple of 256 columns, at least 256).  Smaller
 * blocks mean less workspace and more FP32 accumulation traffic.
 * Process-wide; flce_workspace_size and the calls that use the workspace must
 * see the same setting.
 */
void flce_set_backward_block(int64_t max_rows, int64_t max_block_elems);

/*
 * The backward's dZ block for these sizes under the current setting: *Nb
 * token rows (a multiple of 256) by *Vb vocab columns (a multiple of 256).
 * V > *Vb means several vocab blocks, and then a backward with dX gathers
 * the rows that have a valid target (see flce_backward).  Host only.
 */
flce_status flce_backward_blocking(int64_t N, int64_t H, int64_t V, int64_t* Nb, int64_t* Vb);

/*
 * Measurement hooks.
 *
 * flce_kernel_launch_count: kernels this library has launched in this process
 * (tensor-core GEMMs and the small SIMT kernels; memsets not included).
 *
 * flce_last_launch_wait_limit_ns: the wait limit (ns) the most recent
 * tensor-core launch of any entry point was given (0 before the first), so a
 * caller can check that flce_set_wait_limit_ns reached the kernels.
 *
 * flce_profile_enable(1) makes later calls record CUDA events on the call's
 * stream around their tensor-core launches (events come from a pool the
 * library owns; no device memory is allocated): around the forward GEMM
 * launch, and around the whole run of backward GEMM launches of a call (those
 * launches overlap one another, so they are timed as one interval).
 * flce_profile_collect waits for those events, writes per-kind totals into
 * ms[4] and launches[4] (index 0: forward GEMM with its log-sum-exp epilogue,
 * 1: backward GEMM launches, each holding dZ-recompute, dX and dW tiles;
 * 2 and 3 are reserved and stay 0), clears the records and returns FLCE_OK,
 * or FLCE_ERR_CUDA.  flce_profile_enable(0) stops recording.
 */
int64_t flce_kernel_launch_count(void);
int64_t flce_last_launch_wait_limit_ns(void);
void flce_profile_enable(int enable);
flce_status flce_profile_collect(double* ms, int64_t* launches);

/*
 * Self-test of the bounded-wait path: enqueues one small kernel that waits on
 * a barrier nothing will ever complete, with a limit of `limit_ns`, then
 * records FLCE_ERR_TIMEOUT in the workspace error word and returns cleanly.
 * flce_get_error(workspace, stream) then reports FLCE_ERR_TIMEOUT.  Needs
 * workspace_bytes >= 256.
 */
flce_status flce_selftest_wait_timeout(int64_t limit_ns, void* workspace,
                                       size_t workspace_bytes, flce_stream_t stream);

/*
 * flce_forward with no workspace: for callers that cannot allocate device
 * memory (code running inside a host framework that owns every device
 * allocation and passes in only input and output buffers, or a path where the
 * device-synchronising cudaMalloc / cudaFree are not allowed).  The pages have
 * no counterpart: this is a deployment variant of flce_forward, same kernels,
 * same results.
 *
 *   Arguments as in flce_forward, minus the workspace.
 *   device_error    device int, 1 element, or NULL: receives this call's
 *                   device error bits (0 none, 1 label out of range, 2 wait
 *                   timeout).
 * The scratch is a fixed 16 MiB (16777216-byte) array in the library's device
 * image (held by every GPU that loads the library until the process exits).
 * A call needs, with up(x) = x rounded up to a multiple of 256,
 *     256                        error word
 *   + 2 * up(4 * N)              targets, target logits
 *   + up(8 * N * U)              per-row (max, sum-exp) of each work unit
 *   + up(8 * (ceil(N / 32) + 1)) per-block loss sums
 *   + 256                        work-unit counter
 * bytes, where T = ceil(V / 256) and U = ceil(T / max(4, ceil(T / 128))) <= 128
 * (U = 119 at V = 151936 or 152064): e.g. N = 16384 at V = 151936 fits.
 * Larger problems are rejected with FLCE_ERR_WORKSPACE_TOO_SMALL before
 * anything is enqueued.  Allocates nothing: no cudaMalloc, cudaFree or
 * allocating library call.  The first call on a device looks up the scratch
 * address there (cudaGetSymbolAddress); make that first call before any stream
 * capture on that device.  All calls share the scratch and it keeps the last
 * call's contents (each call clears what must start at zero); calls whose work
 * overlaps on the GPU race on it, so serialise them (one stream, or events).
 */
flce_status flce_forward_noalloc(const void* X, const void* W, const int64_t* labels,
                                 int64_t N, int64_t H, int64_t V, int64_t seq_len,
                                 int64_t ignore_index, int shift, flce_reduction reduction,
                                 float* loss, float* lse, int64_t* n_valid, int* device_error,
                                 flce_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FLCE_H */
