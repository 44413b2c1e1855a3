"""Parity at the full workload sizes, in the launch configuration bench.py times
(default backward blocking), over whole matrices.

For every workload the CPU oracle runs the unfused computation in float64 on
the same bf16 inputs (one pass over row blocks: each block's full logits give
its lse, its dX rows and its term of dW) and the CUDA path is compared with it
on everything it returns: n_valid exactly, the loss, the lse of every row, all
of dX (N x H) and all of dW (V x H) by relative Frobenius error and cosine.
The pages' own equivalence check is a whole-gradient cosine (ms-swift PR
#9784, section Mathematical Equivalence), and the stress workload exists to
check FP32 accumulation of dX and dW across vocabulary slices (Megatron-LM PR
#2739, section 2).

A few sampled rows of dX and vocab rows of dW are checked first (cheap, and a
gross error shows up before the minutes of host work the whole oracle takes).
The measured errors are printed (run pytest with -s or -rA to see them).
"""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import (assert_grad, assert_loss, assert_lse, grad_metrics,
                           remember_oracle_forward, to_np)

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

    # fast pre-check on sampled rows (each needs only its own row of logits)
    t, valid, n_valid, _ = oracle.effective_targets(labels, wl.V, seq_len=wl.S, shift=wl.shift)
    assert got_nv == n_valid
    rng = np.random.default_rng(7)
    rows = pick_rows(valid, wl.S, wl.N, rng)
    r = oracle.rows_forward_backward(X, W, labels, rows, grad_loss=g, **kw)
    assert_lse(got_lse[rows], r["lse"])
    assert_grad("dX sampled rows", to_np(dXh[torch.as_tensor(rows)]), r["dX"])

    # the whole computation
    t0 = time.perf_counter()
    ref = oracle.forward_backward(X, W, labels, grad_loss=g, **kw)
    host_s = time.perf_counter() - t0
    remember_oracle_forward(name, ref)
    assert got_nv == ref["n_valid"]
    assert_loss(got_loss, ref["loss"])
    assert_lse(got_lse, ref["lse"])
    got_dx = to_np(dXh)
    ign = ~ref["valid"]
    assert not got_dx[ign].any(), "ignored rows must have dX exactly 0"
    dx_rel, dx_cos = grad_metrics(got_dx, ref["dX"])
    del got_dx
    ref.pop("dX")
    dw_rel, dw_cos = grad_metrics(to_np(dWh), ref["dW"])
    lse_err = float(np.abs(got_lse - ref["lse"]).max())
    loss_rel = abs(got_loss - ref["loss"]) / abs(ref["loss"]) if ref["loss"] else 0.0
    print(f"\nfull-size parity {name}: loss rel {loss_rel:.2e}, lse max abs {lse_err:.2e}, "
          f"dX rel {dx_rel:.3e} cos {dx_cos:.8f}, dW rel {dw_rel:.3e} cos {dw_cos:.8f} "
          f"(oracle {host_s:.0f} s on the host)")
    assert dx_rel <= 1e-2 and dx_cos >= 0.9999, ("dX", dx_rel, dx_cos)
    assert dw_rel <= 1e-2 and dw_cos >= 0.9999, ("dW", dw_rel, dw_cos)
