"""Vocabulary-parallel fused linear cross-entropy over a torch.distributed group.

The setting of Megatron-LM PR #2739 ("[Dev] Fix Linear-Cross-Entropy
Convergence Issue"): the LM head is a ColumnParallelLinear (section 1), so rank
r of P holds the vocabulary rows W[v0_r : v0_r + V_r] and every rank holds the
same hidden states X and labels; the d_hidden contributions of the vocabulary
slices are summed in FP32 and downcast to bf16 once (section 2).

Per call, on every rank:

  forward   flce_forward_vocab_shard   -> this shard's lse_r, z_r     (kernels)
            all-gather of lse_r and z_r (2 x N floats per rank)        (collective)
            flce_merge_vocab_shards    -> loss, lse, n_valid          (kernels)
  backward  flce_backward_vocab_shard  -> dW_r; dX_acc += dX part     (kernels)
            all-reduce (sum) of dX_acc in FP32 (N x H floats)         (collective)
            flce_downcast_bf16         -> dX                          (kernel)

dW needs no exchange: each rank's rows of dW depend only on its rows of W.
The collectives are the only exchange; all arithmetic runs in the library's
kernels.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import (flce_backward_vocab_shard, flce_downcast_bf16, flce_forward_vocab_shard,
               flce_merge_vocab_shards)

__all__ = ["vocab_shard_bounds", "vocab_parallel_cross_entropy", "CUDA_OPS"]


def vocab_shard_bounds(V_total: int, world_size: int) -> list[tuple[int, int]]:
    """[(v_offset, V_r)] for each rank: contiguous, as equal as possible (the
    first V_total % world_size shards hold one row more)."""
    if world_size <= 0 or V_total < world_size:
        raise ValueError("need 1 <= world_size <= V_total")
    base, extra = divmod(V_total, world_size)
    out, v0 = [], 0
    for r in range(world_size):
        n = base + (1 if r < extra else 0)
        out.append((v0, n))
        v0 += n
    return out


class _CudaOps:
    """The shard kernels of this library (the default and only product path)."""
    forward_shard = staticmethod(flce_forward_vocab_shard)
    merge = staticmethod(flce_merge_vocab_shards)
    backward_shard = staticmethod(flce_backward_vocab_shard)
    downcast = staticmethod(flce_downcast_bf16)


CUDA_OPS = _CudaOps()


def _gather_rows(t: torch.Tensor, group, world: int) -> torch.Tensor:
    """[world, N] tensor of every rank's 1-D t, in rank order."""
    out = torch.empty((world, t.shape[0]), dtype=t.dtype, device=t.device)
    dist.all_gather(list(out.unbind(0)), t.contiguous(), group=group)
    return out


class _VocabParallelCE(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, W_shard, labels, v_offset, V_total, group, seq_len, ignore_index, shift,
                reduction, ops):
        world = dist.get_world_size(group)
        kw = dict(seq_len=seq_len, ignore_index=ignore_index, shift=shift)
        lse_r, z_r, _, ws = ops.forward_shard(X, W_shard, labels, v_offset, V_total, **kw)
        lse_parts = _gather_rows(lse_r, group, world)
        z_parts = _gather_rows(z_r, group, world)
        loss, lse, n_valid = ops.merge(lse_parts, z_parts, labels, V_total, reduction=reduction,
                                       workspace=ws, **kw)
        ctx.save_for_backward(X, W_shard, labels, lse, n_valid)
        ctx.cfg = (v_offset, V_total, group, seq_len, ignore_index, shift, reduction, ops)
        return loss.reshape(())

    @staticmethod
    def backward(ctx, grad):
        X, W_shard, labels, lse, n_valid = ctx.saved_tensors
        v_offset, V_total, group, seq_len, ignore_index, shift, reduction, ops = ctx.cfg
        need_dX, need_dW = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        dX_acc = torch.zeros(X.shape, dtype=torch.float32, device=X.device) if need_dX else None
        dW, _ = ops.backward_shard(X, W_shard, labels, v_offset, V_total, lse, n_valid,
                                   grad.detach(), dX_acc, seq_len=seq_len,
                                   ignore_index=ignore_index, shift=shift, reduction=reduction,
                                   need_dW=need_dW)
        dX = None
        if need_dX:
            dist.all_reduce(dX_acc, op=dist.ReduceOp.SUM, group=group)
            dX = ops.downcast(dX_acc)
        return dX, dW, None, None, None, None, None, None, None, None, None


def vocab_parallel_cross_entropy(hidden, weight_shard, labels, v_offset: int, V_total: int, *,
                                 group=None, ignore_index=-100, shift=False, reduction="mean",
                                 seq_len=None, ops=None):
    """Cross-entropy of hidden @ W.T against labels where this rank holds the
    vocabulary rows weight_shard = W[v_offset : v_offset + V_r].

    hidden: bf16 [B, S, H] or [N, H] (the same on every rank of `group`);
    labels: int64 [B, S] or [N] over the whole vocabulary [0, V_total).
    Returns the 0-dim float32 loss (identical on every rank); backward gives
    every rank the full dX (summed over the group in FP32) and its own rows of
    dW.  `ops` is the set of shard kernels (this library's by default).
    """
    if reduction not in ("mean", "sum"):
        raise ValueError(f"reduction must be 'mean' or 'sum', got {reduction!r}")
    if hidden.dim() == 3:
        B, S, H = hidden.shape
        seq_len = S
        hidden = hidden.reshape(B * S, H)
        labels = labels.reshape(B * S)
    return _VocabParallelCE.apply(hidden.contiguous(), weight_shard.contiguous(),
                                  labels.contiguous(), int(v_offset), int(V_total), group,
                                  seq_len, ignore_index, shift, reduction, ops or CUDA_OPS)
