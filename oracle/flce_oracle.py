"""CPU float64 oracle for fused linear cross-entropy.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or run
this module: only the tests, the smoke check in ``__graft_entry__`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA path.

What it computes is the plain, unfused definition, written out step by step:

* the unfused flow hidden -> LM-head Linear -> full logits -> CrossEntropy
  (ms-swift PR #9784, "feat(sft): Add optional fused linear ce for qwen2/qwen3 on
  npu", section Background; the Qwen3.5-35B-A3B LoRA SFT blog post, the
  "standard flow" diagram after `_patch_model_with_cce`);
* Z = X W^T, L = CE(Z, Y), dX = dZ W, dW = dZ^T X (PR #9784, section
  Mathematical Equivalence);
* the call ``linear_cross_entropy(hidden, weight, labels, ignore_index=-100,
  shift=True, reduction="mean")`` with W laid out (vocab, hidden) (blog post,
  listing `_patch_model_with_cce`).

Every row's full vocabulary of logits is held in float64 (rows are taken in
blocks only to bound host memory; no reordering of any sum beyond what BLAS
does inside one matrix product).  Inputs are upcast exactly to float64: bf16
tensors go bf16 -> float32 -> float64 with no rounding.

Readings of points the pages leave open (each is repeated in the design notes):

* shift: with shift on, position s of a sequence of length seq_len predicts the
  label at s+1; the last position of every sequence has no target and is
  ignored, so no label crosses a sequence boundary (blog post listing
  `_patch_model_with_cce` passes shift=True with labels = input_ids, listing
  `prepare_dataset`).
* mean: divides by the number of valid (non-ignored, post-shift) targets over
  the whole call.  With no valid target, the loss and both gradients are 0.
* a target outside [0, V) that is not ignore_index is reported and its row is
  treated as ignored.
* ignore_index wins even when it lies inside [0, V).
* lse is reported for every row, ignored or not: it does not depend on labels.
"""
from __future__ import annotations

import numpy as np

IGNORE_INDEX = -100


def as_f64(a) -> np.ndarray:
    """Exact upcast of a torch tensor (any float dtype, incl. bf16) or array."""
    if hasattr(a, "detach"):  # torch tensor, imported lazily by the caller
        a = a.detach().cpu()
        if str(a.dtype) in ("torch.bfloat16", "torch.float16"):
            a = a.float()
        a = a.numpy()
    return np.asarray(a, dtype=np.float64)


def as_i64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.asarray(a, dtype=np.int64)


def effective_targets(labels, V: int, *, seq_len: int | None = None, shift: bool = False,
                      ignore_index: int = IGNORE_INDEX):
    """Targets after the optional one-position shift, and the valid mask.

    Returns (t, valid, n_valid, out_of_range):
      t[i]          the label row i is scored against (ignore_index if none);
      valid[i]      t[i] != ignore_index and 0 <= t[i] < V;
      n_valid       number of valid rows (exact integer);
      out_of_range  rows whose target is neither ignore_index nor in [0, V).
    """
    labels = as_i64(labels)
    N = labels.shape[0]
    if shift:
        S = N if not seq_len else int(seq_len)
        if S <= 0 or N % S:
            raise ValueError("N must be a multiple of seq_len")
        lab = labels.reshape(-1, S) if N else labels.reshape(0, max(S, 1))
        t = np.full_like(lab, ignore_index)
        t[:, :-1] = lab[:, 1:]
        t = t.reshape(N)
    else:
        t = labels.copy()
    not_ignored = t != ignore_index
    out_of_range = not_ignored & ((t < 0) | (t >= V))
    valid = not_ignored & ~out_of_range
    return t, valid, int(valid.sum()), out_of_range


def grad_scale(reduction: str, n_valid: int, grad_loss: float = 1.0) -> float:
    """d loss / d (per-row loss): g / n_valid for mean (0 if n_valid == 0), g for sum."""
    if reduction == "mean":
        return float(grad_loss) / n_valid if n_valid > 0 else 0.0
    if reduction == "sum":
        return float(grad_loss)
    raise ValueError(reduction)


def _row_logsumexp(Z: np.ndarray) -> np.ndarray:
    m = Z.max(axis=1)
    return m + np.log(np.exp(Z - m[:, None]).sum(axis=1))


def logits_rows(X, W, rows) -> np.ndarray:
    """Full float64 logits Z[rows, :] = X[rows] W^T."""
    return as_f64(X)[rows] @ as_f64(W).T


def forward(X, W, labels, *, seq_len=None, shift=False, ignore_index=IGNORE_INDEX,
            reduction="mean", row_block=256):
    """Loss, per-row lse and n_valid of the unfused computation.

    Returns a dict with loss (float), lse (float64 [N]), row_loss (float64 [N],
    0 for ignored rows), z_target (float64 [N], nan for ignored rows), n_valid
    (int) and out_of_range (bool [N]).
    """
    Xd, Wd = as_f64(X), as_f64(W)
    N, V = Xd.shape[0], Wd.shape[0]
    t, valid, n_valid, oor = effective_targets(labels, V, seq_len=seq_len, shift=shift,
                                               ignore_index=ignore_index)
    lse = np.empty(N)
    zt = np.full(N, np.nan)
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        Z = Xd[r0:r1] @ Wd.T
        lse[r0:r1] = _row_logsumexp(Z)
        v = valid[r0:r1]
        zt[r0:r1][v] = Z[np.nonzero(v)[0], t[r0:r1][v]]
    row_loss = np.where(valid, lse - np.where(valid, zt, 0.0), 0.0)
    total = float(row_loss.sum())
    if reduction == "mean":
        loss = total / n_valid if n_valid > 0 else 0.0
    elif reduction == "sum":
        loss = total
    else:
        raise ValueError(reduction)
    return dict(loss=loss, lse=lse, row_loss=row_loss, z_target=zt, n_valid=n_valid,
                out_of_range=oor, targets=t, valid=valid)


def grad_logits(Z_rows: np.ndarray, lse_rows: np.ndarray, t_rows: np.ndarray,
                valid_rows: np.ndarray, scale: float) -> np.ndarray:
    """dL/dZ for a block of rows: scale * valid_i * (softmax(Z_i) - onehot(t_i))."""
    P = np.exp(Z_rows - lse_rows[:, None])
    idx = np.nonzero(valid_rows)[0]
    P[idx, t_rows[idx]] -= 1.0
    P[~valid_rows] = 0.0
    return scale * P


def backward(X, W, labels, *, seq_len=None, shift=False, ignore_index=IGNORE_INDEX,
             reduction="mean", grad_loss=1.0, lse=None, row_block=256):
    """float64 (dX [N,H], dW [V,H]) of the unfused computation.

    lse, if given, must be this oracle's own forward()["lse"]; otherwise it is
    recomputed here.
    """
    Xd, Wd = as_f64(X), as_f64(W)
    N, V = Xd.shape[0], Wd.shape[0]
    t, valid, n_valid, _ = effective_targets(labels, V, seq_len=seq_len, shift=shift,
                                             ignore_index=ignore_index)
    s = grad_scale(reduction, n_valid, grad_loss)
    dX = np.zeros_like(Xd)
    dW = np.zeros_like(Wd)
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        Z = Xd[r0:r1] @ Wd.T
        l = _row_logsumexp(Z) if lse is None else np.asarray(lse[r0:r1], np.float64)
        dZ = grad_logits(Z, l, t[r0:r1], valid[r0:r1], s)
        dX[r0:r1] = dZ @ Wd
        dW += dZ.T @ Xd[r0:r1]
    return dX, dW


def forward_backward(X, W, labels, *, seq_len=None, shift=False, ignore_index=IGNORE_INDEX,
                     reduction="mean", grad_loss=1.0, row_block=2048):
    """forward() and backward() in one pass over the row blocks: each block's
    logits Z = X_blk W^T are formed once and give that block's lse, target
    logits, dZ, dX rows and its term dZ_blk^T X_blk of dW (the chunk sum of
    PR #9784, section Mathematical Equivalence).  Same definition, same
    arithmetic per block as the two functions; it only avoids forming Z twice,
    which matters at the full workload sizes.

    Returns a dict with the keys of forward() plus dX [N,H] and dW [V,H]
    (float64).
    """
    Xd, Wd = as_f64(X), as_f64(W)
    N, V = Xd.shape[0], Wd.shape[0]
    t, valid, n_valid, oor = effective_targets(labels, V, seq_len=seq_len, shift=shift,
                                               ignore_index=ignore_index)
    s = grad_scale(reduction, n_valid, grad_loss)
    lse = np.empty(N)
    zt = np.full(N, np.nan)
    dX = np.zeros_like(Xd)
    dW = np.zeros_like(Wd)
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        Z = Xd[r0:r1] @ Wd.T
        l = _row_logsumexp(Z)
        lse[r0:r1] = l
        v = valid[r0:r1]
        zt[r0:r1][v] = Z[np.nonzero(v)[0], t[r0:r1][v]]
        dZ = grad_logits(Z, l, t[r0:r1], v, s)
        del Z
        dX[r0:r1] = dZ @ Wd
        dW += dZ.T @ Xd[r0:r1]
    row_loss = np.where(valid, lse - np.where(valid, zt, 0.0), 0.0)
    total = float(row_loss.sum())
    if reduction == "mean":
        loss = total / n_valid if n_valid > 0 else 0.0
    elif reduction == "sum":
        loss = total
    else:
        raise ValueError(reduction)
    return dict(loss=loss, lse=lse, row_loss=row_loss, z_target=zt, n_valid=n_valid,
                out_of_range=oor, targets=t, valid=valid, dX=dX, dW=dW)


# ---------------------------------------------------------------------------
# Sampled outputs for full-size checks: each is the same definition restricted
# to a few rows (of dX / lse) or a few vocab rows (of dW).
# ---------------------------------------------------------------------------

def rows_forward_backward(X, W, labels, rows, *, seq_len=None, shift=False,
                          ignore_index=IGNORE_INDEX, reduction="mean", grad_loss=1.0):
    """lse, row loss and dX for the given token rows only (each needs its full
    row of logits); the gradient scale uses the call-wide n_valid."""
    Wd = as_f64(W)
    V = Wd.shape[0]
    t, valid, n_valid, _ = effective_targets(labels, V, seq_len=seq_len, shift=shift,
                                             ignore_index=ignore_index)
    rows = np.asarray(rows, dtype=np.int64)
    if hasattr(X, "index_select"):  # torch tensor: upcast only the sampled rows
        import torch
        Xr = as_f64(X.index_select(0, torch.as_tensor(rows)))
    else:
        Xr = as_f64(X)[rows]
    Z = Xr @ Wd.T
    lse = _row_logsumexp(Z)
    tv, vv = t[rows], valid[rows]
    zt = np.where(vv, Z[np.arange(len(rows)), np.where(vv, tv, 0)], np.nan)
    s = grad_scale(reduction, n_valid, grad_loss)
    dZ = grad_logits(Z, lse, tv, vv, s)
    return dict(lse=lse, row_loss=np.where(vv, lse - np.nan_to_num(zt), 0.0),
                dX=dZ @ Wd, n_valid=n_valid)


def vocab_rows_dW(X, W, labels, lse, vocab_rows, *, seq_len=None, shift=False,
                  ignore_index=IGNORE_INDEX, reduction="mean", grad_loss=1.0,
                  row_block=4096):
    """dW[j, :] for the given vocab rows j.  Needs this oracle's lse for every
    token row: dW_j = sum_i dZ_ij x_i runs over all tokens."""
    Xd, Wd = as_f64(X), as_f64(W)
    V = Wd.shape[0]
    t, valid, n_valid, _ = effective_targets(labels, V, seq_len=seq_len, shift=shift,
                                             ignore_index=ignore_index)
    s = grad_scale(reduction, n_valid, grad_loss)
    js = np.asarray(vocab_rows, dtype=np.int64)
    Wj = Wd[js]
    out = np.zeros((len(js), Xd.shape[1]))
    for r0 in range(0, Xd.shape[0], row_block):
        r1 = min(Xd.shape[0], r0 + row_block)
        Zc = Xd[r0:r1] @ Wj.T                           # [rows, len(js)]
        P = np.exp(Zc - np.asarray(lse[r0:r1])[:, None])
        P -= (t[r0:r1, None] == js[None, :])
        P[~valid[r0:r1]] = 0.0
        out += (s * P).T @ Xd[r0:r1]
    return out
