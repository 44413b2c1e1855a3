"""flce_forward_noalloc: the forward for callers that cannot allocate device
memory (a plugin inside a framework that owns all device allocations, or a
path where the device-synchronising cudaMalloc/cudaFree are not allowed).

It keeps its scratch in a fixed array inside the library, so these tests check
that two calls in a row (different shapes, the second over the first call's
leftovers) give the same results as flce_forward with a workspace, and that
problems too large for the array are refused before anything runs.  This file
sorts last so a stop-at-first-failure run has already run every other test.
"""
import pytest
import torch

import workloads
from tests._parity import assert_loss, assert_lse

pytestmark = pytest.mark.gpu

flce = pytest.importorskip("lm_head_linear_flce_gb300")


def _both(X, W, labels, **kw):
    dev = torch.device("cuda")
    Xd, Wd, Ld = X.to(dev), W.to(dev), labels.to(dev)
    ref_loss, ref_lse, ref_nv, _ = flce.flce_forward(Xd, Wd, Ld, **kw)
    loss, lse, nv, derr = flce.flce_forward_noalloc(Xd, Wd, Ld, **kw)
    torch.cuda.synchronize()
    return (loss.item(), lse.cpu().numpy(), int(nv.item()), int(derr.item()),
            ref_loss.item(), ref_lse.cpu().numpy(), int(ref_nv.item()))


def test_two_calls_match_the_workspace_forward():
    X1, W1, L1 = workloads.random_case(1000, 200, 3000, seed=21)
    X2, W2, L2 = workloads.random_case(384, 136, 1500, seed=22, ignore_frac=0.5)
    for (X, W, L), kw in (((X1, W1, L1), dict(seq_len=250, shift=True)),
                          ((X2, W2, L2), dict(reduction="sum"))):
        loss, lse, nv, derr, rloss, rlse, rnv = _both(X, W, L, **kw)
        assert derr == 0
        assert nv == rnv
        assert_loss(loss, rloss)
        assert_lse(lse, rlse)


def test_full_qwen2_7b_forward_fits_and_matches():
    wl = workloads.get("qwen2_7b")
    X, W, L = workloads.make_inputs(wl)
    for _ in range(2):
        loss, lse, nv, derr, rloss, rlse, rnv = _both(X, W, L, seq_len=wl.S, shift=wl.shift,
                                                      reduction=wl.reduction)
        assert derr == 0 and nv == rnv
        assert_loss(loss, rloss)
        assert_lse(lse, rlse)


def test_problem_larger_than_the_scratch_is_refused():
    dev = torch.device("cuda")
    X = torch.zeros(16384, 8, dtype=torch.bfloat16, device=dev)
    W = torch.zeros(151936, 8, dtype=torch.bfloat16, device=dev)
    L = torch.zeros(16384, dtype=torch.int64, device=dev)
    with pytest.raises(flce.FlceError) as e:
        flce.flce_forward_noalloc(X, W, L)
    assert e.value.status == 3  # FLCE_ERR_WORKSPACE_TOO_SMALL


def test_out_of_range_label_reported_through_device_error():
    X, W, L = workloads.random_case(256, 64, 500, seed=23)
    L[3] = 999
    dev = torch.device("cuda")
    loss, lse, nv, derr = flce.flce_forward_noalloc(X.to(dev), W.to(dev), L.to(dev))
    assert int(derr.item()) == 1
