"""flce_backward_accumulate (dW added in FP32 into an existing gradient) and
the bitwise repeatability of the backward's FP32 accumulations."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import assert_grad, to_np

pytestmark = pytest.mark.gpu

flce = pytest.importorskip("lm_head_linear_flce_gb300")


@pytest.fixture(autouse=True)
def _restore_defaults():
    yield
    flce.flce_set_backward_block(0, 0)


@pytest.mark.parametrize("N,H,V,blocks,red", [
    (600, 192, 2500, None, "mean"),
    (700, 136, 1500, (256, 256 * 512), "sum"),   # several token and vocab blocks
])
def test_accumulates_into_existing_fp32_gradient(N, H, V, blocks, red):
    if blocks:
        flce.flce_set_backward_block(*blocks)
    X, W, labels = workloads.random_case(N, H, V, seed=40 + N, w_std=0.08)
    dev = torch.device("cuda")
    Xd, Wd, Ld = X.to(dev), W.to(dev), labels.to(dev)
    loss, lse, nv, ws = flce.flce_forward(Xd, Wd, Ld, reduction=red)
    ref_dX, ref_dW = oracle.backward(X, W, labels, reduction=red, grad_loss=0.5)
    g = torch.Generator().manual_seed(1)
    base = torch.randn(V, H, generator=g) * float(np.abs(ref_dW).mean())
    acc = base.to(dev)
    dX, _ = flce.flce_backward_accumulate(Xd, Wd, Ld, lse, nv, torch.tensor([0.5], device=dev),
                                          acc, reduction=red, workspace=ws)
    assert flce.flce_get_error(ws) == 0
    added = acc.cpu().double().numpy() - base.double().numpy()
    assert_grad("dW added", added, ref_dW)
    assert_grad("dX", to_np(dX), ref_dX)


def test_backward_is_bitwise_repeatable():
    flce.flce_set_backward_block(256, 256 * 1024)
    X, W, labels = workloads.random_case(1000, 256, 5000, seed=50)
    dev = torch.device("cuda")
    Xd, Wd, Ld = X.to(dev), W.to(dev), labels.to(dev)
    loss, lse, nv, ws = flce.flce_forward(Xd, Wd, Ld)
    g = torch.ones(1, device=dev)
    outs = []
    for _ in range(2):
        dX, dW, _ = flce.flce_backward(Xd, Wd, Ld, lse, nv, g, workspace=ws)
        acc = torch.zeros(5000, 256, device=dev)
        flce.flce_backward_accumulate(Xd, Wd, Ld, lse, nv, g, acc, need_dX=False, workspace=ws)
        outs.append((dX.clone(), dW.clone(), acc.clone()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
