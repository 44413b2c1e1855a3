"""CPU float64 oracle for the vocabulary-parallel split of fused linear
cross-entropy.

TEST INFRASTRUCTURE ONLY, like the rest of this package: nothing on the product
path imports it, and it shares no code with the CUDA path.

Setting (Megatron-LM PR #2739, "Fix Linear-Cross-Entropy Convergence Issue",
section 1: the output layer is a ColumnParallelLinear, so each of the P ranks
holds a contiguous slice W[v0 : v0 + V_r] of the vocabulary rows; section 2:
the computation is split along the vocabulary and d_hidden is accumulated in
an FP32 buffer before one downcast to bf16).  Every rank sees the same X and
labels.

Per rank r, over its own columns only:
  lse_r[i] = log sum_{j in shard r} exp(Z_ij)
  z_r[i]   = Z_{i, t_i} if t_i falls in shard r, else 0
Merge (after gathering the P pairs of every row):
  lse[i] = log sum_r exp(lse_r[i])  (the log-sum-exp of all V logits)
  z[i]   = sum_r z_r[i]              (exactly one shard holds a valid target)
  loss   = sum over valid rows of (lse - z), divided by n_valid for "mean"
Backward, rank r, with the merged lse:
  dZ_r = s * valid_i * (exp(Z_ij - lse_i) - [j = t_i])   for j in shard r
  dX partial_r = dZ_r W_r  (summed over ranks: dX),  dW_r = dZ_r^T X

Validity is judged against the whole vocabulary [0, V_total): a row whose
target lies in another rank's shard is still valid here (it contributes its
softmax terms), it only has no one-hot term on this rank.
"""
from __future__ import annotations

import numpy as np

from .flce_oracle import IGNORE_INDEX, as_f64, effective_targets, grad_scale


def shard_forward(X, W_shard, labels, v_offset: int, V_total: int, *, seq_len=None,
                  shift=False, ignore_index=IGNORE_INDEX, row_block=256):
    """(lse_r float64 [N], z_r float64 [N], n_valid int, valid bool [N]) of one shard."""
    Xd, Wd = as_f64(X), as_f64(W_shard)
    N, Vr = Xd.shape[0], Wd.shape[0]
    t, valid, n_valid, _ = effective_targets(labels, V_total, seq_len=seq_len, shift=shift,
                                             ignore_index=ignore_index)
    local = valid & (t >= v_offset) & (t < v_offset + Vr)
    lse_r = np.empty(N)
    z_r = np.zeros(N)
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        Z = Xd[r0:r1] @ Wd.T
        m = Z.max(axis=1)
        lse_r[r0:r1] = m + np.log(np.exp(Z - m[:, None]).sum(axis=1))
        rows = np.nonzero(local[r0:r1])[0]
        z_r[r0 + rows] = Z[rows, t[r0 + rows] - v_offset]
    return lse_r, z_r, n_valid, valid


def merge_shards(lse_parts, z_parts, valid, n_valid: int, reduction="mean"):
    """(loss, lse [N]) from the gathered per-shard pairs, lse_parts/z_parts [P, N]."""
    L = np.asarray(lse_parts, np.float64)
    M = L.max(axis=0)
    lse = M + np.log(np.exp(L - M[None, :]).sum(axis=0))
    z = np.asarray(z_parts, np.float64).sum(axis=0)
    row_loss = np.where(valid, lse - z, 0.0)
    total = float(row_loss.sum())
    if reduction == "mean":
        return (total / n_valid if n_valid > 0 else 0.0), lse
    if reduction == "sum":
        return total, lse
    raise ValueError(reduction)


def shard_backward(X, W_shard, labels, v_offset: int, V_total: int, lse, *, seq_len=None,
                   shift=False, ignore_index=IGNORE_INDEX, reduction="mean", grad_loss=1.0,
                   row_block=256):
    """(dX partial float64 [N, H], dW_r float64 [V_r, H]) of one shard, with the
    merged lse of every row."""
    Xd, Wd = as_f64(X), as_f64(W_shard)
    N, Vr = Xd.shape[0], Wd.shape[0]
    t, valid, n_valid, _ = effective_targets(labels, V_total, seq_len=seq_len, shift=shift,
                                             ignore_index=ignore_index)
    s = grad_scale(reduction, n_valid, grad_loss)
    dX = np.zeros_like(Xd)
    dW = np.zeros_like(Wd)
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        Z = Xd[r0:r1] @ Wd.T
        P = np.exp(Z - np.asarray(lse[r0:r1], np.float64)[:, None])
        tt, vv = t[r0:r1], valid[r0:r1]
        here = np.nonzero(vv & (tt >= v_offset) & (tt < v_offset + Vr))[0]
        P[here, tt[here] - v_offset] -= 1.0
        P[~vv] = 0.0
        dZ = s * P
        dX[r0:r1] = dZ @ Wd
        dW += dZ.T @ Xd[r0:r1]
    return dX, dW


def split_bounds(V_total: int, sizes) -> list[tuple[int, int]]:
    """[(v0, V_r)] of consecutive shards with the given sizes (summing to V_total)."""
    out, v0 = [], 0
    for n in sizes:
        out.append((v0, int(n)))
        v0 += int(n)
    if v0 != V_total:
        raise ValueError("shard sizes must add up to the vocabulary size")
    return out
