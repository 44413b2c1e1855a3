"""Out-of-bounds writes, checked without a sanitizer: every buffer a call
writes (workspace, loss, lse, n_valid, dX, dW, the FP32 accumulators of the
accumulate and vocabulary-shard calls) is placed inside a larger allocation
whose surrounding bytes hold a known pattern; after the calls the pattern
must be intact, on ragged shapes and several backward blockings."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

flce = pytest.importorskip("lm_head_linear_flce_gb300")

GUARD = 4096       # bytes on each side (a multiple of 256 keeps the alignment)
PATTERN = 0xA5


class Guarded:
    """A typed view of `numel` elements with GUARD pattern bytes on each side."""

    def __init__(self, numel, dtype, dev):
        esize = torch.empty(0, dtype=dtype).element_size()
        nbytes = numel * esize
        self.raw = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device=dev)
        self.nbytes = nbytes
        self.t = self.raw[GUARD:GUARD + nbytes].view(dtype)

    def intact(self):
        return bool((self.raw[:GUARD] == PATTERN).all()) and \
            bool((self.raw[GUARD + self.nbytes:] == PATTERN).all())


@pytest.fixture(autouse=True)
def _restore_defaults():
    yield
    flce.flce_set_backward_block(0, 0)


@pytest.mark.parametrize("N,H,V,blocks", [
    (300, 200, 1000, None),
    (700, 136, 1500, (256, 256 * 512)),
    (130, 72, 257, (128, 128 * 256)),
    (96, 128, 70000, None),
])
def test_calls_write_only_inside_their_buffers(N, H, V, blocks):
    if blocks:
        flce.flce_set_backward_block(*blocks)
    dev = torch.device("cuda")
    X, W, L = workloads.random_case(N, H, V, seed=N + V, w_std=0.1)
    X, W, L = X.to(dev), W.to(dev), L.to(dev)
    ws = Guarded(flce.workspace_size(N, H, V), torch.uint8, dev)
    loss = Guarded(1, torch.float32, dev)
    lse = Guarded(N, torch.float32, dev)
    nv = Guarded(1, torch.int64, dev)
    dX = Guarded(N * H, torch.bfloat16, dev)
    dW = Guarded(V * H, torch.bfloat16, dev)
    dW_acc = Guarded(V * H, torch.float32, dev)
    dX_acc = Guarded(N * H, torch.float32, dev)
    dW_acc.t.zero_()
    dX_acc.t.zero_()
    lib = flce.library()
    s = flce._stream(dev)
    g = torch.ones(1, device=dev)
    P = flce._ptr
    assert lib.flce_forward(P(X), P(W), P(L), N, H, V, N, -100, 1, 0, P(loss.t), P(lse.t),
                            P(nv.t), P(ws.t), ws.nbytes, s) == 0
    assert lib.flce_backward(P(X), P(W), P(L), N, H, V, N, -100, 1, 0, P(lse.t), P(nv.t), P(g),
                             P(dX.t.view(N, H)), P(dW.t.view(V, H)), P(ws.t), ws.nbytes, s) == 0
    flce.flce_backward_accumulate(X, W, L, lse.t, nv.t, g, dW_acc.t.view(V, H), seq_len=N,
                                  shift=True, workspace=ws.t, dX=dX.t.view(N, H))
    half = V // 2
    flce.flce_backward_vocab_shard(X, W[half:].contiguous(), L, half, V, lse.t, nv.t, g,
                                   dX_acc.t.view(N, H), seq_len=N, shift=True, workspace=ws.t,
                                   dW=dW.t.view(V, H)[half:])
    assert flce.flce_get_error(ws.t) == 0
    for name, b in (("workspace", ws), ("loss", loss), ("lse", lse), ("n_valid", nv), ("dX", dX),
                    ("dW", dW), ("dW_acc", dW_acc), ("dX_acc", dX_acc)):
        assert b.intact(), f"{name}: bytes outside the buffer were written"
