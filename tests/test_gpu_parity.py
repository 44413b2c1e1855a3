"""GPU parity of flce_forward / flce_backward against the CPU float64 oracle,
element by element, on small seeded cases that still span several tiles and a
ragged tail, and on the edge cases of the method."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import assert_grad, assert_loss, assert_lse, to_np

pytestmark = pytest.mark.gpu

flce = pytest.importorskip("lm_head_linear_flce_gb300")


@pytest.fixture(autouse=True)
def _restore_defaults():
    yield
    flce.flce_set_backward_block(0, 0)
    flce.flce_set_wait_limit_ns(0)


def run_case(X, W, labels, *, seq_len=None, shift=False, reduction="mean", ignore_index=-100,
             grad=1.0, need_dX=True, need_dW=True):
    dev = torch.device("cuda")
    Xd, Wd, Ld = X.to(dev), W.to(dev), labels.to(dev)
    loss, lse, nv, ws = flce.flce_forward(Xd, Wd, Ld, seq_len=seq_len, shift=shift,
                                          reduction=reduction, ignore_index=ignore_index)
    g = torch.tensor([grad], dtype=torch.float32, device=dev)
    dX, dW, ws = flce.flce_backward(Xd, Wd, Ld, lse, nv, g, seq_len=seq_len, shift=shift,
                                    reduction=reduction, ignore_index=ignore_index,
                                    need_dX=need_dX, need_dW=need_dW, workspace=ws)
    status = flce.flce_get_error(ws)
    return dict(loss=loss.item(), lse=lse.cpu().numpy(), n_valid=int(nv.item()),
                dX=None if dX is None else to_np(dX), dW=None if dW is None else to_np(dW),
                status=status)


def check_against_oracle(X, W, labels, *, seq_len=None, shift=False, reduction="mean",
                         ignore_index=-100, grad=1.0, **kw):
    got = run_case(X, W, labels, seq_len=seq_len, shift=shift, reduction=reduction,
                   ignore_index=ignore_index, grad=grad, **kw)
    ref = oracle.forward(X, W, labels, seq_len=seq_len, shift=shift, reduction=reduction,
                         ignore_index=ignore_index)
    dX, dW = oracle.backward(X, W, labels, seq_len=seq_len, shift=shift, reduction=reduction,
                             ignore_index=ignore_index, grad_loss=grad, lse=ref["lse"])
    assert got["n_valid"] == ref["n_valid"]
    assert_loss(got["loss"], ref["loss"])
    if X.shape[0]:
        assert_lse(got["lse"], ref["lse"])
    if got["dX"] is not None:
        assert_grad("dX", got["dX"], dX)
    if got["dW"] is not None:
        assert_grad("dW", got["dW"], dW)
    return got, ref


def test_tiny_workload():
    wl = workloads.get("tiny")
    X, W, labels = workloads.make_inputs(wl)
    got, _ = check_against_oracle(X, W, labels, shift=wl.shift, reduction=wl.reduction)
    assert got["status"] == 0


@pytest.mark.parametrize("N,H,V,S,shift,red,blocks", [
    (300, 200, 1000, 100, True, "mean", None),          # ragged N, H not a multiple of 64, ragged V
    (700, 136, 1500, 350, True, "sum", (256, 256 * 512)),  # several token and vocab blocks
    (512, 320, 2304, 256, False, "mean", (128, 128 * 256)),  # smallest blocks, exact tiles
    (1, 64, 7, None, False, "mean", None),               # one row, vocab smaller than a tile
    (130, 72, 257, None, False, "sum", (128, 128 * 256)),  # one column past a tile
    (2048, 192, 1500, 512, True, "mean", (2048, 2048 * 256)),  # every row, one vocab tile a block
])
def test_odd_shapes(N, H, V, S, shift, red, blocks):
    if blocks:
        flce.flce_set_backward_block(*blocks)
    X, W, labels = workloads.random_case(N, H, V, seed=N + H + V, w_std=0.08)
    check_against_oracle(X, W, labels, seq_len=S, shift=shift, reduction=red, grad=0.75)


def test_target_on_last_vocab_column_and_first():
    N, H, V = 256, 128, 1000
    X, W, labels = workloads.random_case(N, H, V, seed=5, ignore_frac=0.0)
    labels[::3] = V - 1
    labels[1::3] = 0
    check_against_oracle(X, W, labels)


def test_all_ignored_mean_is_zero():
    X, W, labels = workloads.random_case(200, 64, 600, seed=6)
    labels[:] = -100
    got, _ = check_against_oracle(X, W, labels)
    assert got["loss"] == 0.0 and got["n_valid"] == 0
    assert not got["dX"].any() and not got["dW"].any()


def test_single_valid_row():
    X, W, labels = workloads.random_case(300, 96, 777, seed=7)
    keep = labels[123].item() if labels[123] >= 0 else 5
    labels[:] = -100
    labels[123] = keep
    check_against_oracle(X, W, labels)


def test_ignore_index_inside_vocab():
    X, W, labels = workloads.random_case(256, 64, 512, seed=8, ignore_frac=0.0)
    labels[::4] = 3
    check_against_oracle(X, W, labels, ignore_index=3)


def test_batch_shift_has_no_cross_sequence_leak():
    B, S, H, V = 4, 96, 128, 900
    X, W, labels = workloads.random_case(B * S, H, V, seed=9)
    got, ref = check_against_oracle(X, W, labels, seq_len=S, shift=True)
    assert got["n_valid"] == ref["n_valid"]


def test_out_of_range_labels_flagged_rows_ignored():
    X, W, labels = workloads.random_case(256, 64, 500, seed=10)
    labels[7] = 500
    labels[8] = -5
    got = run_case(X, W, labels)
    assert got["status"] == 4  # FLCE_ERR_LABEL_OUT_OF_RANGE
    lab2 = labels.clone()
    lab2[7] = -100
    lab2[8] = -100
    ref = oracle.forward(X, W, lab2)
    dX, dW = oracle.backward(X, W, lab2)
    assert got["n_valid"] == ref["n_valid"]
    assert_loss(got["loss"], ref["loss"])
    assert_grad("dX", got["dX"], dX)
    assert_grad("dW", got["dW"], dW)


@pytest.mark.parametrize("need_dX,need_dW", [(True, False), (False, True)])
def test_one_gradient_only(need_dX, need_dW):
    flce.flce_set_backward_block(128, 128 * 512)
    X, W, labels = workloads.random_case(384, 136, 1200, seed=11)
    got, _ = check_against_oracle(X, W, labels, need_dX=need_dX, need_dW=need_dW)
    assert (got["dX"] is None) != need_dX and (got["dW"] is None) != need_dW


def test_empty_batch():
    dev = torch.device("cuda")
    X = torch.empty(0, 64, dtype=torch.bfloat16, device=dev)
    W = torch.randn(100, 64, device=dev).to(torch.bfloat16)
    labels = torch.empty(0, dtype=torch.int64, device=dev)
    loss, lse, nv, ws = flce.flce_forward(X, W, labels)
    dX, dW, _ = flce.flce_backward(X, W, labels, lse, nv, torch.ones(1, device=dev))
    assert loss.item() == 0.0 and nv.item() == 0
    assert dW.abs().sum().item() == 0.0


def test_autograd_entry_matches_raw_calls():
    wl = workloads.get("tiny")
    X, W, labels = workloads.make_inputs(wl, N=512, seed=3)
    dev = torch.device("cuda")
    Xd = X.to(dev).view(2, 256, -1).requires_grad_(True)
    Wd = W.to(dev).requires_grad_(True)
    loss = flce.linear_cross_entropy(Xd, Wd, labels.to(dev).view(2, 256), shift=True)
    (2.0 * loss).backward()
    ref = oracle.forward(X, W, labels, seq_len=256, shift=True)
    dX, dW = oracle.backward(X, W, labels, seq_len=256, shift=True, grad_loss=2.0)
    assert_loss(loss.item(), ref["loss"])
    assert_grad("dX", to_np(Xd.grad).reshape(512, -1), dX)
    assert_grad("dW", to_np(Wd.grad), dW)


def test_bounded_wait_selftest_times_out():
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    assert flce.flce_selftest_wait_timeout(20_000_000, ws) == 0
    assert flce.flce_get_error(ws) == 5  # FLCE_ERR_TIMEOUT
    # the context is still usable afterwards
    test_tiny_workload()


def test_repeat_calls_are_stable():
    X, W, labels = workloads.random_case(640, 256, 3000, seed=12)
    a = run_case(X, W, labels)
    b = run_case(X, W, labels)
    assert a["loss"] == b["loss"]  # deterministic loss reduction
    np.testing.assert_array_equal(a["lse"], b["lse"])


@pytest.mark.parametrize("H", [8, 16, 32, 40])
def test_small_hidden_sizes(H):
    X, W, labels = workloads.random_case(300, H, 700, seed=20 + H, w_std=0.3)
    check_against_oracle(X, W, labels, grad=1.5)


def test_single_class_vocabulary():
    # V = 1: softmax is 1 everywhere, so every valid row has loss 0 and no gradient
    X, W, labels = workloads.random_case(200, 64, 1, seed=30, ignore_frac=0.2)
    got, ref = check_against_oracle(X, W, labels)
    assert abs(got["loss"]) < 1e-6
    assert not got["dX"].any() and not got["dW"].any()


def test_shift_with_length_one_sequences_ignores_everything():
    X, W, labels = workloads.random_case(128, 64, 300, seed=31, ignore_frac=0.0)
    got, ref = check_against_oracle(X, W, labels, seq_len=1, shift=True)
    assert got["n_valid"] == 0 and got["loss"] == 0.0


@pytest.mark.parametrize("blocks", [None, (8192, 32 << 20)])
def test_more_than_8192_rows(blocks):
    # automatic blocking: all 8492 rows in one token block (64 Mi-element dZ
    # block); with 8192-row blocks: two token blocks, so dW accumulates in the
    # FP32 band; dX over several vocab blocks either way
    if blocks:
        flce.flce_set_backward_block(*blocks)
    X, W, labels = workloads.random_case(8192 + 300, 64, 9000, seed=32, w_std=0.2)
    check_against_oracle(X, W, labels, seq_len=8492, shift=True)


def test_many_vocab_blocks_few_rows():
    X, W, labels = workloads.random_case(96, 128, 70000, seed=33, w_std=0.1)
    check_against_oracle(X, W, labels, reduction="sum")


@pytest.mark.parametrize("blocks", [None, (256, 256 * 1024)])
def test_fully_ignored_token_tiles_are_skipped_correctly(blocks):
    # a long masked prompt (rows 0..1099) and a masked span (1400..1799): several
    # 256-row tiles hold no target and are dropped from the backward
    if blocks:
        flce.flce_set_backward_block(*blocks)
    N, H, V = 2300, 128, 3000
    X, W, labels = workloads.random_case(N, H, V, seed=70, ignore_frac=0.05)
    labels[:1100] = -100
    labels[1400:1800] = -100
    check_against_oracle(X, W, labels, grad=1.25)
    got, _ = check_against_oracle(X, W, labels, seq_len=N, shift=True, reduction="sum")
    assert not got["dX"][:1024].any()


def test_only_last_tile_active():
    X, W, labels = workloads.random_case(1024, 64, 900, seed=71, ignore_frac=0.0)
    labels[:1000] = -100
    check_against_oracle(X, W, labels)


@pytest.mark.parametrize("N,H,V", [
    (200, 16384, 600),     # long K for the recompute and for the dX / dW tiles' H sweep
    (64, 65536, 300),      # the largest supported H
    (40, 64, 300001),      # a vocabulary of 300K (many vocab blocks and forward units)
    (20000, 32, 700),      # three ragged token blocks of at most 8192 rows
])
def test_large_extents(N, H, V):
    if N > 8192:
        flce.flce_set_backward_block(8192, 32 << 20)
    X, W, labels = workloads.random_case(N, H, V, seed=N % 97 + H % 89 + V % 83,
                                         w_std=0.5 / np.sqrt(H) * 8)
    check_against_oracle(X, W, labels, reduction="sum", grad=0.5)


@pytest.mark.parametrize("name", ["qwen3_8b", "long_ctx", "stress"])
def test_reduced_workloads_keep_their_distributions(name):
    # each workload's own generator (Zipf labels with prompt spans, a masked
    # prefix, wide logits) at a size the oracle finishes quickly
    wl = workloads.get(name)
    X, W, labels = workloads.make_inputs(wl, N=1024 * wl.B, H=256, V=3000, seed=77)
    check_against_oracle(X, W, labels, seq_len=X.shape[0] // wl.B, shift=wl.shift,
                         reduction=wl.reduction, grad=0.5)


def test_every_target_the_same_class():
    X, W, labels = workloads.random_case(600, 96, 1300, seed=78, ignore_frac=0.0)
    labels[:] = 777
    check_against_oracle(X, W, labels, reduction="sum")


def test_two_token_sequences_with_shift():
    # seq_len 2: only the first row of every pair has a target
    X, W, labels = workloads.random_case(512, 64, 800, seed=79, ignore_frac=0.0)
    got, ref = check_against_oracle(X, W, labels, seq_len=2, shift=True)
    assert got["n_valid"] == 256


@pytest.mark.parametrize("need_dW", [True, False])
def test_dx_tiles_follow_their_row_tiles(need_dW):
    """The dX tiles of a 256-row tile start as soon as the recompute tiles of
    that row tile have stored their dZ, interleaved with later recompute tiles:
    16 row tiles per block (more than the hand-out lag of 11 at H = 2048 and
    2048-column vocab blocks), three vocab blocks with a ragged last one, and
    fully ignored row tiles between active ones."""
    N, H, V, S = 4096, 2048, 6000, 1024
    flce.flce_set_backward_block(N, N * 2048)
    X, W, labels = workloads.random_case(N, H, V, seed=31, w_std=0.03)
    labels[512:1024] = -100   # row tiles 2 and 3 (row 1023 ends a sequence)
    labels[2560:2817] = -100  # row tile 10: rows 2560-2815 score labels 2561-2816
    check_against_oracle(X, W, labels, seq_len=S, shift=True, reduction="mean", grad=1.3,
                         need_dW=need_dW)


def test_forward_row_bands_with_a_ragged_last_band():
    """The forward hands out its work units band by band (as many 256-row tiles
    as keep 40 MB of X): at H = 8192 a row tile holds 4 MB of X, so 11 row
    tiles (the last one ragged) go in bands of 6 and 5."""
    N, H, V = 2800, 8192, 3000
    X, W, labels = workloads.random_case(N, H, V, seed=41, x_std=0.5, w_std=0.01)
    check_against_oracle(X, W, labels, reduction="sum", grad=0.5)


@pytest.mark.parametrize("ignore_frac", [0.45, 0.0, 0.97])
def test_dense_rows_are_gathered_and_put_back(ignore_frac):
    # rows without a target scattered through every 256-row tile, several vocab
    # blocks (256 columns each), ragged N and a per-sequence shift: the
    # backward gathers the rows with a target into dense tiles inside dX's
    # buffer and runs on those; dX comes back in token order with the other
    # rows exactly 0.  Also: no row ignored (all gathered), nearly all ignored
    # (one dense tile, mostly padding).
    flce.flce_set_backward_block(1024, 1024 * 256)
    N, H, V, S = 1000, 136, 1300, 500
    X, W, labels = workloads.random_case(N, H, V, seed=91, ignore_frac=ignore_frac, w_std=0.1)
    assert flce.flce_backward_blocking(N, H, V) == (1024, 256)
    got, ref = check_against_oracle(X, W, labels, seq_len=S, shift=True, grad=0.5)
    t = torch.full((N,), -100, dtype=torch.int64)
    t.view(-1, S)[:, :-1] = labels.view(-1, S)[:, 1:]
    ignored = (t == -100).numpy()
    assert not got["dX"][ignored].any()
    assert got["dX"][~ignored].any(axis=1).all()


def test_outputs_overlapping_inputs_or_each_other_are_refused():
    # refused on the host before anything is enqueued (include/flce.h,
    # flce_backward): dX on X or on W's rows, dW on W, dX inside dW, an
    # output inside the workspace; separate buffers still work afterwards
    dev = torch.device("cuda")
    X, W, labels = workloads.random_case(300, 64, 700, seed=92)
    Xd, Wd, Ld = X.to(dev), W.to(dev), labels.to(dev)
    _, lse, nv, ws = flce.flce_forward(Xd, Wd, Ld)
    g = torch.ones(1, dtype=torch.float32, device=dev)
    dW_big = torch.empty_like(Wd)
    ws_view = ws[: 300 * 64 * 2].view(torch.bfloat16).view(300, 64)
    cases = [dict(dX=Xd, need_dW=False), dict(dX=Wd[:300], need_dW=False),
             dict(dW=Wd, need_dX=False), dict(dX=dW_big[:300], dW=dW_big),
             dict(dX=ws_view, need_dW=False)]
    for kw in cases:
        with pytest.raises(flce.FlceError, match="INVALID_ARG"):
            flce.flce_backward(Xd, Wd, Ld, lse, nv, g, workspace=ws, **kw)
    dX, dW, _ = flce.flce_backward(Xd, Wd, Ld, lse, nv, g, workspace=ws)
    assert torch.isfinite(dX.float()).all() and torch.isfinite(dW.float()).all()


def test_dense_rows_beyond_one_scan_chunk():
    # 1172 token tiles and about 1055 dense tiles: the one-block scan of the
    # per-tile counts and the dense tile list both span two 1024-tile chunks;
    # 37 token blocks (dW through the FP32 band) x 5 vocab blocks
    flce.flce_set_backward_block(8192, 8192 * 256)
    N, H, V = 300000, 32, 1200
    assert flce.flce_backward_blocking(N, H, V) == (8192, 256)
    X, W, labels = workloads.random_case(N, H, V, seed=93, w_std=0.5)
    check_against_oracle(X, W, labels, reduction="sum", grad=0.5)
