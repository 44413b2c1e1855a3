"""The forward and backward enqueue only kernels and memsets on the caller's
stream and allocate nothing, so a whole training step can be captured once in
a CUDA graph and replayed: replays must reproduce the eager results bit for
bit (every reduction in the path has a fixed order) and follow new input
values written into the captured buffers."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import assert_grad, assert_loss, to_np

pytestmark = pytest.mark.gpu

flce = pytest.importorskip("lm_head_linear_flce_gb300")


def _buffers(N, H, V, dev):
    return dict(loss=torch.empty(1, device=dev), lse=torch.empty(N, device=dev),
                nv=torch.empty(1, dtype=torch.int64, device=dev),
                dX=torch.empty(N, H, dtype=torch.bfloat16, device=dev),
                dW=torch.empty(V, H, dtype=torch.bfloat16, device=dev),
                ws=torch.empty(flce.workspace_size(N, H, V), dtype=torch.uint8, device=dev))


def _step(X, W, L, g, b, kw):
    lib = flce.library()
    N, H = X.shape
    V = W.shape[0]
    s = flce._stream(X.device)
    red = 0 if kw["reduction"] == "mean" else 1
    st = lib.flce_forward(flce._ptr(X), flce._ptr(W), flce._ptr(L), N, H, V, kw["seq_len"], -100,
                          int(kw["shift"]), red, flce._ptr(b["loss"]), flce._ptr(b["lse"]),
                          flce._ptr(b["nv"]), flce._ptr(b["ws"]), b["ws"].numel(), s)
    assert st == 0
    st = lib.flce_backward(flce._ptr(X), flce._ptr(W), flce._ptr(L), N, H, V, kw["seq_len"], -100,
                           int(kw["shift"]), red, flce._ptr(b["lse"]), flce._ptr(b["nv"]),
                           flce._ptr(g), flce._ptr(b["dX"]), flce._ptr(b["dW"]),
                           flce._ptr(b["ws"]), b["ws"].numel(), s)
    assert st == 0


@pytest.mark.parametrize("N,H,V,blocks", [(1000, 256, 5000, (256, 256 * 1024)),
                                          (512, 128, 3000, None)])
def test_captured_step_replays_bitwise_and_follows_new_inputs(N, H, V, blocks):
    if blocks:
        flce.flce_set_backward_block(*blocks)
    try:
        dev = torch.device("cuda")
        kw = dict(seq_len=N, shift=True, reduction="mean")
        X1, W1, L1 = workloads.random_case(N, H, V, seed=90, w_std=0.1)
        X2, W2, L2 = workloads.random_case(N, H, V, seed=91, w_std=0.1)
        X, W, L = X1.to(dev), W1.to(dev), L1.to(dev)
        g = torch.ones(1, device=dev)
        eager = _buffers(N, H, V, dev)
        _step(X, W, L, g, eager, kw)
        torch.cuda.synchronize()

        b = _buffers(N, H, V, dev)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            _step(X, W, L, g, b, kw)  # first call outside capture (lazy attribute setup)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            _step(X, W, L, g, b, kw)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        for k in ("loss", "lse", "nv", "dX", "dW"):
            assert torch.equal(b[k], eager[k]), k
        assert flce.flce_get_error(b["ws"]) == 0

        # new values in the captured input buffers: the replay follows them
        X.copy_(X2.to(dev))
        W.copy_(W2.to(dev))
        L.copy_(L2.to(dev))
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.forward(X2, W2, L2, **kw)
        rdX, rdW = oracle.backward(X2, W2, L2, lse=ref["lse"], **kw)
        assert int(b["nv"].item()) == ref["n_valid"]
        assert_loss(b["loss"].item(), ref["loss"])
        assert_grad("dX", to_np(b["dX"]), rdX)
        assert_grad("dW", to_np(b["dW"]), rdW)
    finally:
        flce.flce_set_backward_block(0, 0)
