"""GPU parity of the vocabulary-parallel entry points against the CPU float64
oracle.  The P ranks are emulated one after another on one GPU: each shard's
forward runs, the (lse_r, z_r) rows are stacked as an all-gather would, the
merge runs, and every shard's backward adds its dX part into one FP32 buffer
(what the all-reduce sums) before the one downcast.  The results must equal
the unsharded oracle within the same tolerances as the unsharded call."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import assert_grad, assert_loss, assert_lse, to_np

pytestmark = pytest.mark.gpu

flce = pytest.importorskip("lm_head_linear_flce_gb300")
from lm_head_linear_flce_gb300.vocab_parallel import vocab_shard_bounds  # noqa: E402


@pytest.fixture(autouse=True)
def _restore_defaults():
    yield
    flce.flce_set_backward_block(0, 0)


def emulate(X, W, labels, bounds, *, seq_len=None, shift=False, reduction="mean", grad=1.0,
            need_dX=True, need_dW=True):
    dev = torch.device("cuda")
    Xd, Wd, Ld = X.to(dev), W.to(dev), labels.to(dev)
    V = W.shape[0]
    kw = dict(seq_len=seq_len, shift=shift)
    lse_p, z_p, nvs, wss = [], [], [], []
    for v0, n in bounds:
        l, z, nv, ws = flce.flce_forward_vocab_shard(Xd, Wd[v0:v0 + n].contiguous(), Ld, v0, V,
                                                     **kw)
        lse_p.append(l)
        z_p.append(z)
        nvs.append(int(nv.item()))
        wss.append(ws)
    loss, lse, nv = flce.flce_merge_vocab_shards(torch.stack(lse_p), torch.stack(z_p), Ld, V,
                                                 reduction=reduction, workspace=wss[0], **kw)
    g = torch.tensor([grad], device=dev)
    dX_acc = torch.zeros(Xd.shape, dtype=torch.float32, device=dev) if need_dX else None
    dWs = []
    for (v0, n), ws in zip(bounds, wss):
        dW, _ = flce.flce_backward_vocab_shard(Xd, Wd[v0:v0 + n].contiguous(), Ld, v0, V, lse,
                                               nv, g, dX_acc, reduction=reduction,
                                               need_dW=need_dW, workspace=ws, **kw)
        dWs.append(dW)
    dX = flce.flce_downcast_bf16(dX_acc) if need_dX else None
    status = [flce.flce_get_error(ws) for ws in wss]
    return dict(loss=loss.item(), lse=lse.cpu().numpy(), n_valid=int(nv.item()), shard_nv=nvs,
                dX=None if dX is None else to_np(dX),
                dW=None if not need_dW else to_np(torch.cat(dWs)),
                lse_parts=[t.cpu().numpy() for t in lse_p], z_parts=[t.cpu().numpy() for t in z_p],
                status=status)


def check(X, W, labels, bounds, *, seq_len=None, shift=False, reduction="mean", grad=1.0,
          **kw):
    got = emulate(X, W, labels, bounds, seq_len=seq_len, shift=shift, reduction=reduction,
                  grad=grad, **kw)
    ref = oracle.forward(X, W, labels, seq_len=seq_len, shift=shift, reduction=reduction)
    dX, dW = oracle.backward(X, W, labels, seq_len=seq_len, shift=shift, reduction=reduction,
                             grad_loss=grad, lse=ref["lse"])
    assert got["n_valid"] == ref["n_valid"]
    assert all(nv == ref["n_valid"] for nv in got["shard_nv"])
    assert_loss(got["loss"], ref["loss"])
    assert_lse(got["lse"], ref["lse"])
    if got["dX"] is not None:
        assert_grad("dX", got["dX"], dX)
    if got["dW"] is not None:
        assert_grad("dW", got["dW"], dW)
    return got, ref


@pytest.mark.parametrize("N,H,V,P,shift,red", [
    (300, 200, 1000, 2, True, "mean"),    # ragged everything, shard edge inside a tile
    (512, 128, 2304, 3, False, "sum"),    # 768 columns per shard: exact tiles
    (700, 136, 1500, 4, True, "mean"),    # 375 columns per shard
])
def test_shards_match_oracle(N, H, V, P, shift, red):
    X, W, labels = workloads.random_case(N, H, V, seed=N + V + P, w_std=0.08)
    got, ref = check(X, W, labels, vocab_shard_bounds(V, P), seq_len=N // 2 if shift else None,
                     shift=shift, reduction=red, grad=0.75)
    assert got["status"] == [0] * P


def test_per_shard_outputs_match_the_shard_oracle():
    from oracle import vocab_parallel as ovp
    X, W, labels = workloads.random_case(400, 96, 900, seed=81, w_std=0.1)
    bounds = vocab_shard_bounds(900, 3)
    got = emulate(X, W, labels, bounds)
    for (v0, n), l, z in zip(bounds, got["lse_parts"], got["z_parts"]):
        rl, rz, _, _ = ovp.shard_forward(X, W[v0:v0 + n], labels, v0, 900)
        assert_lse(l, rl)
        here = rz != 0
        np.testing.assert_allclose(z[here], rz[here], rtol=2e-3, atol=2e-3)
        assert not z[~here].any()


def test_targets_on_shard_edges_and_a_shard_without_targets():
    N, H, V = 512, 64, 1200
    X, W, labels = workloads.random_case(N, H, V, seed=82, ignore_frac=0.0)
    bounds = [(0, 300), (300, 300), (600, 300), (900, 300)]
    labels[:] = 299           # last column of the first shard
    labels[1::4] = 300        # first column of the second
    labels[2::4] = 1199       # last column of the last
    labels[3::8] = 0          # the third shard, [600, 900), holds no target
    check(X, W, labels, bounds)


def test_shard_spanning_several_vocab_blocks():
    # small backward blocks: each shard's dX part accumulates over several vocab
    # blocks into the caller's FP32 buffer, and dW over several token blocks
    flce.flce_set_backward_block(256, 256 * 512)
    X, W, labels = workloads.random_case(700, 128, 3000, seed=83, w_std=0.1)
    check(X, W, labels, vocab_shard_bounds(3000, 2), grad=1.5)


def test_shards_with_skipped_token_tiles():
    N, H, V = 1300, 128, 2000
    X, W, labels = workloads.random_case(N, H, V, seed=84)
    labels[:600] = -100
    got, _ = check(X, W, labels, vocab_shard_bounds(V, 2), seq_len=N, shift=True)
    assert not got["dX"][:512].any()


@pytest.mark.parametrize("need_dX,need_dW", [(True, False), (False, True)])
def test_one_gradient_only(need_dX, need_dW):
    X, W, labels = workloads.random_case(384, 136, 1000, seed=85)
    got, _ = check(X, W, labels, vocab_shard_bounds(1000, 2), need_dX=need_dX, need_dW=need_dW)
    assert (got["dX"] is None) != need_dX and (got["dW"] is None) != need_dW


def test_label_outside_whole_vocabulary_is_flagged():
    X, W, labels = workloads.random_case(256, 64, 600, seed=86)
    labels[5] = 600
    got = emulate(X, W, labels, vocab_shard_bounds(600, 2))
    assert got["status"] == [4, 4]  # FLCE_ERR_LABEL_OUT_OF_RANGE on every shard
    lab2 = labels.clone()
    lab2[5] = -100
    ref = oracle.forward(X, W, lab2)
    assert got["n_valid"] == ref["n_valid"]
    assert_loss(got["loss"], ref["loss"])


@pytest.mark.slow
def test_full_qwen2_7b_split_across_four_ranks_sampled():
    wl = workloads.get("qwen2_7b")
    X, W, labels = workloads.make_inputs(wl)
    V = W.shape[0]
    bounds = vocab_shard_bounds(V, 4)
    kw = dict(seq_len=wl.S, shift=wl.shift, reduction=wl.reduction)
    got = emulate(X, W, labels, bounds, **kw)
    torch.cuda.empty_cache()
    ref = oracle.forward(X, W, labels, **kw)
    assert got["n_valid"] == ref["n_valid"]
    assert_loss(got["loss"], ref["loss"])
    assert_lse(got["lse"], ref["lse"])
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(X.shape[0], 24, replace=False))
    r = oracle.rows_forward_backward(X, W, labels, rows, **kw)
    assert_grad("dX rows", got["dX"][rows], r["dX"])
    # vocab rows on both sides of every shard edge, and a few inside
    js = {0, V - 1}
    for v0, _ in bounds[1:]:
        js.update((v0 - 1, v0))
    js.update(rng.integers(0, V, 6).tolist())
    js = np.array(sorted(js))
    ref_dw = oracle.vocab_rows_dW(X, W, labels, ref["lse"], js, **kw)
    assert_grad("dW rows", got["dW"][js], ref_dw)
    col = np.linalg.norm(got["dW"].sum(0))
    assert col <= 1e-2 * np.linalg.norm(got["dW"]), col


def test_autograd_module_over_one_rank_nccl_group():
    import datetime
    import socket
    import torch.distributed as dist
    from lm_head_linear_flce_gb300.vocab_parallel import vocab_parallel_cross_entropy
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    if dist.is_initialized():
        pytest.skip("a process group is already initialised")
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            timeout=datetime.timedelta(seconds=120))
    try:
        X, W, labels = workloads.random_case(512, 128, 1000, seed=87)
        dev = torch.device("cuda")
        Xd = X.to(dev).requires_grad_(True)
        Wd = W.to(dev).requires_grad_(True)
        loss = vocab_parallel_cross_entropy(Xd, Wd, labels.to(dev), 0, 1000)
        loss.backward()
        ref = oracle.forward(X, W, labels)
        dX, dW = oracle.backward(X, W, labels)
        assert_loss(loss.item(), ref["loss"])
        assert_grad("dX", to_np(Xd.grad), dX)
        assert_grad("dW", to_np(Wd.grad), dW)
    finally:
        dist.destroy_process_group()
