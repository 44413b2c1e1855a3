"""The vocabulary-parallel exchange on CPU: gloo ranks, each holding a slice of
W's vocabulary rows, run vocab_parallel_cross_entropy with the shard kernels
replaced by a float64 model of them built from the oracle.  What is checked is
the host logic around the kernels: the shard bounds, the all-gather of
(lse_r, z_r) in rank order, the merge inputs, the FP32 all-reduce of dX, the
gradient scale and which gradients each rank gets.  Together the ranks must
reproduce the unsharded oracle."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from oracle import vocab_parallel as ovp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _OracleOps:
    """float64 stand-ins for the four shard kernels, same call signatures."""

    @staticmethod
    def forward_shard(X, W, labels, v_offset, V_total, *, seq_len=None, ignore_index=-100,
                      shift=False):
        l, z, nv, _ = ovp.shard_forward(X, W, labels, v_offset, V_total, seq_len=seq_len,
                                        shift=shift, ignore_index=ignore_index)
        return torch.from_numpy(l), torch.from_numpy(z), torch.tensor([nv]), None

    @staticmethod
    def merge(lse_parts, z_parts, labels, V_total, *, seq_len=None, ignore_index=-100,
              shift=False, reduction="mean", workspace=None):
        _, valid, nv, _ = oracle.effective_targets(labels, V_total, seq_len=seq_len,
                                                   shift=shift, ignore_index=ignore_index)
        loss, lse = ovp.merge_shards(lse_parts.numpy(), z_parts.numpy(), valid, nv, reduction)
        return torch.tensor([loss]), torch.from_numpy(lse), torch.tensor([nv])

    @staticmethod
    def backward_shard(X, W, labels, v_offset, V_total, lse, n_valid, grad, dX_acc, *,
                       seq_len=None, ignore_index=-100, shift=False, reduction="mean",
                       need_dW=True):
        dx, dw = ovp.shard_backward(X.detach(), W.detach(), labels, v_offset, V_total,
                                    lse.numpy(), seq_len=seq_len, shift=shift,
                                    ignore_index=ignore_index, reduction=reduction,
                                    grad_loss=float(grad))
        if dX_acc is not None:
            dX_acc += torch.from_numpy(dx).to(dX_acc.dtype)
        return (torch.from_numpy(dw).to(W.dtype) if need_dW else None), None

    @staticmethod
    def downcast(src):
        return src.clone()


def _case(seed, N=36, H=10, V=53):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((N, H)).astype(np.float32)
    W = (rng.standard_normal((V, H)) * 0.7).astype(np.float32)
    labels = rng.integers(0, V, N)
    labels[rng.random(N) < 0.2] = -100
    return X, W, labels


def _worker(rank, world, port, seed, kw, grad, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from lm_head_linear_flce_gb300.vocab_parallel import (vocab_parallel_cross_entropy,
                                                              vocab_shard_bounds)
        X, W, labels = _case(seed)
        v0, n = vocab_shard_bounds(W.shape[0], world)[rank]
        Xt = torch.from_numpy(X).requires_grad_(True)
        Wt = torch.from_numpy(W[v0:v0 + n].copy()).requires_grad_(True)
        loss = vocab_parallel_cross_entropy(Xt, Wt, torch.from_numpy(labels), v0, W.shape[0],
                                            ops=_OracleOps(), **kw)
        (grad * loss).backward()
        out[rank] = (float(loss), Xt.grad.numpy().copy(), Wt.grad.numpy().copy(), v0, n)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,kw,grad", [
    (2, dict(reduction="mean"), 1.0),
    (3, dict(reduction="sum", shift=True, seq_len=12), 0.5),
])
def test_ranks_reproduce_the_unsharded_oracle(world, kw, grad):
    seed = 40 + world
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), seed, kw, grad, out), nprocs=world, join=True)
    X, W, labels = _case(seed)
    ref = oracle.forward(X, W, labels, **kw)
    rdX, rdW = oracle.backward(X, W, labels, grad_loss=grad, **kw)
    got_dW = np.zeros_like(rdW)
    for r in range(world):
        loss, dX, dW, v0, n = out[r]
        assert loss == pytest.approx(ref["loss"], rel=1e-6)       # same loss on every rank
        np.testing.assert_allclose(dX, rdX, rtol=1e-5, atol=1e-7)  # full dX on every rank
        got_dW[v0:v0 + n] = dW
    np.testing.assert_allclose(got_dW, rdW, rtol=1e-5, atol=1e-7)


def test_shard_bounds():
    from lm_head_linear_flce_gb300.vocab_parallel import vocab_shard_bounds
    assert vocab_shard_bounds(10, 3) == [(0, 4), (4, 3), (7, 3)]
    assert vocab_shard_bounds(151936, 8)[-1] == (7 * 18992, 18992)
    with pytest.raises(ValueError):
        vocab_shard_bounds(2, 3)
