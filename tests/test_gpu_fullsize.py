"""Parity at the full workload sizes, in the launch configuration bench.py times
(default backward blocking).

For every workload the CPU oracle computes, in float64: the full forward (lse
of every row, the loss, n_valid), dX for a sample of token rows (each needs
its own full row of logits) and dW for a sample of vocab rows (each needs the
oracle's lse of every token).  The rest of dW is checked through an identity
that holds at any size: every row of dZ sums to zero, so the vocab rows of dW
sum to the zero vector.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import assert_grad, assert_loss, assert_lse, to_np

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

flce = pytest.importorskip("lm_head_linear_flce_gb300")


def pick_rows(valid, seq_len, N, rng, k=24):
    rows = {0, N - 1, seq_len - 1, min(N - 1, seq_len)}
    ign = np.nonzero(~valid)[0]
    val = np.nonzero(valid)[0]
    rows.update(rng.choice(ign, min(4, len(ign)), replace=False).tolist() if len(ign) else [])
    rows.update(rng.choice(val, min(k, len(val)), replace=False).tolist() if len(val) else [])
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", [w.name for w in workloads.WORKLOADS])
def test_full_size_parity(name):
    wl = workloads.get(name)
    X, W, labels = workloads.make_inputs(wl)
    dev = torch.device("cuda")
    Xd, Wd, Ld = X.to(dev), W.to(dev), labels.to(dev)
    kw = dict(seq_len=wl.S, shift=wl.shift, reduction=wl.reduction)
    g = 1.0
    loss, lse, nv, ws = flce.flce_forward(Xd, Wd, Ld, **kw)
    dX, dW, ws = flce.flce_backward(Xd, Wd, Ld, lse, nv, torch.full((1,), g, device=dev),
                                    workspace=ws, **kw)
    assert flce.flce_get_error(ws) == 0
    got_loss, got_lse, got_nv = loss.item(), lse.cpu().numpy(), int(nv.item())
    del Xd, Wd, Ld
    dXh = dX.cpu()
    dWh = dW.cpu()
    del dX, dW, ws
    torch.cuda.empty_cache()

    ref = oracle.forward(X, W, labels, **kw)
    assert got_nv == ref["n_valid"]
    assert_loss(got_loss, ref["loss"])
    assert_lse(got_lse, ref["lse"])

    rng = np.random.default_rng(7)
    rows = pick_rows(ref["valid"], wl.S, wl.N, rng)
    r = oracle.rows_forward_backward(X, W, labels, rows, grad_loss=g, **kw)
    got_dx = to_np(dXh[torch.as_tensor(rows)])
    assert_grad("dX rows", got_dx, r["dX"])
    ign = ~ref["valid"][rows]
    assert not got_dx[ign].any(), "ignored rows must have dX exactly 0"

    tv = ref["targets"][ref["valid"]]
    js = {0, wl.V - 1}
    js.update(rng.choice(tv, 6, replace=False).tolist())
    js.update(rng.integers(0, wl.V, 6).tolist())
    js = np.array(sorted(js))
    ref_dw = oracle.vocab_rows_dW(X, W, labels, ref["lse"], js, grad_loss=g, **kw)
    assert_grad("dW rows", to_np(dWh[torch.as_tensor(js)]), ref_dw)

    # sum over the vocabulary of dW is the zero vector (per-row sums of dZ vanish)
    dW64 = dWh.double()
    col = dW64.sum(0).norm().item()
    assert col <= 1e-2 * dW64.norm().item(), col
