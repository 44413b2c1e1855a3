"""Pins of the CPU oracle to facts it does not compute itself.

Each test ties the oracle to something fixed by the pages or by mathematics:
hand-derived fixtures, closed forms (W = 0, V = 2), finite differences, exact
invariants, brute force on tiny inputs and a library routine.  Together they
are chosen so that a dropped term, a flipped sign, a wrong index, a transposed
operand or a wrong mean denominator anywhere in the oracle fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(N, H, V, seed, ignore_frac=0.25, w_std=0.5):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((N, H))
    W = rng.standard_normal((V, H)) * w_std
    labels = rng.integers(0, V, N)
    labels[rng.random(N) < ignore_frac] = -100
    return X, W, labels


# --------------------------------------------------------------------------
# hand-derived fixtures
# --------------------------------------------------------------------------

def test_shift_golden():
    g = json.load(open(os.path.join(GOLDEN, "shift_example.json")))
    t, valid, n_valid, oor = oracle.effective_targets(
        np.array(g["labels"]), g["V"], seq_len=g["seq_len"], shift=True,
        ignore_index=g["ignore_index"])
    assert t.tolist() == g["targets"]
    assert n_valid == g["n_valid"]
    assert valid.tolist() == [x != g["ignore_index"] for x in g["targets"]]
    assert not oor.any()


def test_two_class_golden():
    g = json.load(open(os.path.join(GOLDEN, "two_class_example.json")))
    X, W, lab = np.array(g["X"]), np.array(g["W"]), np.array(g["labels"])
    f = oracle.forward(X, W, lab)
    assert f["loss"] == pytest.approx(g["loss"], rel=1e-15)
    assert f["lse"][0] == pytest.approx(g["lse"], rel=1e-15)
    dX, dW = oracle.backward(X, W, lab)
    np.testing.assert_allclose(dX, g["dX"], rtol=1e-14)
    np.testing.assert_allclose(dW, g["dW"], rtol=1e-14)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_w_zero_closed_form(reduction):
    N, H, V = 40, 12, 33
    X, _, labels = _rand(N, H, V, 1)
    W = np.zeros((V, H))
    f = oracle.forward(X, W, labels, reduction=reduction)
    n = int((labels != -100).sum())
    assert f["n_valid"] == n
    np.testing.assert_allclose(f["lse"], math.log(V), rtol=1e-15)  # every row, ignored too
    expect = math.log(V) if reduction == "mean" else n * math.log(V)
    assert f["loss"] == pytest.approx(expect, rel=1e-14)
    dX, dW = oracle.backward(X, W, labels, reduction=reduction, grad_loss=0.7)
    assert np.all(dX == 0.0)
    s = 0.7 / n if reduction == "mean" else 0.7
    # dW_j = s * sum over valid i of (1/V - [t_i = j]) x_i
    ref = np.zeros((V, H))
    for i in range(N):
        if labels[i] == -100:
            continue
        ref += X[i][None, :] / V
        ref[labels[i]] -= X[i]
    np.testing.assert_allclose(dW, s * ref, rtol=1e-12, atol=1e-15)


def test_two_class_is_logistic_loss():
    N, H = 30, 7
    X, W, labels = _rand(N, H, 2, 2, ignore_frac=0.2)
    f = oracle.forward(X, W, labels)
    valid = labels != -100
    z = X @ W.T
    t = np.where(valid, labels, 0)
    d = z[np.arange(N), 1 - t] - z[np.arange(N), t]
    softplus = np.logaddexp(0.0, d)
    assert f["loss"] == pytest.approx(softplus[valid].mean(), rel=1e-13)
    sig = 1.0 / (1.0 + np.exp(-d))
    dX, dW = oracle.backward(X, W, labels)
    s = 1.0 / valid.sum()
    ref = s * sig[:, None] * (W[1 - t] - W[t]) * valid[:, None]
    np.testing.assert_allclose(dX, ref, rtol=1e-12, atol=1e-15)


# --------------------------------------------------------------------------
# finite differences
# --------------------------------------------------------------------------

@pytest.mark.parametrize("reduction,shift", [("mean", True), ("sum", False)])
def test_central_finite_differences(reduction, shift):
    N, H, V = 6, 8, 16
    X, W, labels = _rand(N, H, V, 3, ignore_frac=0.2)
    kw = dict(seq_len=3, shift=shift, reduction=reduction)
    dX, dW = oracle.backward(X, W, labels, **kw)
    eps = 1e-6

    def L(Xp, Wp):
        return oracle.forward(Xp, Wp, labels, **kw)["loss"]

    fdX = np.zeros_like(X)
    for i in range(N):
        for h in range(H):
            Xp, Xm = X.copy(), X.copy()
            Xp[i, h] += eps
            Xm[i, h] -= eps
            fdX[i, h] = (L(Xp, W) - L(Xm, W)) / (2 * eps)
    fdW = np.zeros_like(W)
    for j in range(V):
        for h in range(H):
            Wp, Wm = W.copy(), W.copy()
            Wp[j, h] += eps
            Wm[j, h] -= eps
            fdW[j, h] = (L(X, Wp) - L(X, Wm)) / (2 * eps)
    scale = max(np.abs(dX).max(), np.abs(dW).max())
    assert np.abs(dX - fdX).max() <= 1e-7 * scale + 1e-9
    assert np.abs(dW - fdW).max() <= 1e-7 * scale + 1e-9


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

def test_grad_logit_rows_sum_to_zero():
    N, H, V = 50, 10, 70
    X, W, labels = _rand(N, H, V, 4)
    dX, dW = oracle.backward(X, W, labels)
    # each valid row of dZ sums to 0, so the vocab rows of dW sum to the zero vector
    assert np.abs(dW.sum(axis=0)).max() <= 1e-13 * np.abs(dW).max()
    t, valid, n, _ = oracle.effective_targets(labels, V)
    Z = X @ W.T
    lse = oracle.forward(X, W, labels)["lse"]
    dZ = oracle.grad_logits(Z, lse, t, valid, 1.0)
    np.testing.assert_allclose(dZ.sum(axis=1), 0.0, atol=1e-14)


def _cos(a, b):
    return float((a * b).sum() / np.sqrt((a * a).sum() * (b * b).sum()))


def test_chunked_equals_global_rows():
    """Row chunks of 2048 with grad_weight accumulated chunk by chunk (PR #9784,
    sections What this PR does and Mathematical Equivalence) equal the global
    computation: gradient cosine 1.000000."""
    N, H, V = 5000, 12, 40
    X, W, labels = _rand(N, H, V, 5)
    t, valid, n, _ = oracle.effective_targets(labels, V)
    dX, dW = oracle.backward(X, W, labels)
    loss = oracle.forward(X, W, labels)["loss"]
    dXc, dWc, lc = np.zeros_like(X), np.zeros_like(W), 0.0
    for c0 in range(0, N, 2048):
        c1 = min(N, c0 + 2048)
        # the mean is over the whole call: each chunk is a sum scaled by 1/n
        a, b = oracle.backward(X[c0:c1], W, labels[c0:c1], reduction="sum", grad_loss=1.0 / n)
        dXc[c0:c1] = a
        dWc += b
        lc += oracle.forward(X[c0:c1], W, labels[c0:c1], reduction="sum")["loss"] / n
    assert round(_cos(dW, dWc), 6) == 1.0 and round(_cos(dX, dXc), 6) == 1.0
    assert np.abs(dW - dWc).max() <= 1e-12 and np.abs(dX - dXc).max() <= 1e-12
    assert lc == pytest.approx(loss, rel=1e-12)


def test_chunked_equals_global_vocab():
    """Vocab split (Megatron-LM PR #2739, section 2): per-slice log-sum-exp merged
    over slices gives lse; d_hidden summed over slices, d_logits_slice times
    weight_slice, gives dX."""
    N, H, V = 64, 10, 301
    X, W, labels = _rand(N, H, V, 6)
    f = oracle.forward(X, W, labels)
    dX, _ = oracle.backward(X, W, labels)
    slices = [(0, 100), (100, 256), (256, 301)]
    part = np.stack([oracle.forward(X, W[a:b], np.full(N, -100))["lse"] for a, b in slices])
    np.testing.assert_allclose(np.logaddexp.reduce(part, axis=0), f["lse"], rtol=1e-14)
    t, valid, n, _ = oracle.effective_targets(labels, V)
    dZ = oracle.grad_logits(X @ W.T, f["lse"], t, valid, 1.0 / n)
    acc = np.zeros_like(X)
    for a, b in slices:
        acc += dZ[:, a:b] @ W[a:b]
    assert round(_cos(acc, dX), 6) == 1.0
    np.testing.assert_allclose(acc, dX, rtol=1e-12, atol=1e-15)


def test_ignored_rows_are_inert():
    N, H, V = 24, 9, 31
    X, W, labels = _rand(N, H, V, 7, ignore_frac=0.4)
    ign = np.nonzero(labels == -100)[0]
    assert len(ign) > 2
    f = oracle.forward(X, W, labels)
    dX, dW = oracle.backward(X, W, labels)
    assert np.all(dX[ign] == 0.0)
    X2 = X.copy()
    X2[ign] *= -37.0
    f2 = oracle.forward(X2, W, labels)
    _, dW2 = oracle.backward(X2, W, labels)
    assert f2["loss"] == f["loss"]
    np.testing.assert_array_equal(dW2, dW)
    # with the shift on, a sequence's first label is never a target
    lab3 = labels.copy()
    lab3[0] = (labels[0] + 5) % V
    a = oracle.forward(X, W, labels, shift=True, seq_len=N)
    b = oracle.forward(X, W, lab3, shift=True, seq_len=N)
    assert a["loss"] == b["loss"]


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_rows_without_a_target_drop_out(reduction):
    """Loss, lse and dW over all rows equal those over the rows that have a
    target alone (gathered in order, the shift applied first), and their dX
    rows are the same; the other rows' dX is exactly 0.  The mean's
    denominator counts the same rows either way.  (What lets a backward run on
    the rows with a target only.)"""
    B, S, H, V = 2, 40, 11, 37
    X, W, labels = _rand(B * S, H, V, 21, ignore_frac=0.45)
    t, valid, n_valid, _ = oracle.effective_targets(labels, V, seq_len=S, shift=True)
    rows = np.nonzero(valid)[0]
    assert 0 < len(rows) < B * S
    full = oracle.forward(X, W, labels, seq_len=S, shift=True, reduction=reduction)
    dX, dW = oracle.backward(X, W, labels, seq_len=S, shift=True, reduction=reduction,
                             grad_loss=0.7)
    dense = oracle.forward(X[rows], W, t[rows], reduction=reduction)
    dXd, dWd = oracle.backward(X[rows], W, t[rows], reduction=reduction, grad_loss=0.7)
    assert dense["n_valid"] == full["n_valid"] == n_valid == len(rows)
    assert dense["loss"] == pytest.approx(full["loss"], rel=1e-13)
    np.testing.assert_allclose(dense["lse"], full["lse"][rows], rtol=1e-14)
    np.testing.assert_allclose(dWd, dW, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dXd, dX[rows], rtol=1e-12, atol=1e-15)
    assert np.all(dX[~valid] == 0.0)


def test_shift_has_no_leak_across_sequences():
    B, S, H, V = 3, 7, 5, 19
    X, W, labels = _rand(B * S, H, V, 8, ignore_frac=0.1)
    a = oracle.forward(X, W, labels, shift=True, seq_len=S)
    lab = labels.reshape(B, S)
    manual = np.concatenate([lab[:, 1:], np.full((B, 1), -100)], axis=1).reshape(-1)
    b = oracle.forward(X, W, manual, shift=False)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-15)
    # changing the first label of sequence 1 only moves the last row of sequence 0? no:
    # the last row of sequence 0 is ignored, so nothing moves
    lab2 = labels.copy()
    lab2[S] = (lab2[S] + 1) % V
    c = oracle.forward(X, W, lab2, shift=True, seq_len=S)
    assert c["loss"] == a["loss"]


def test_reduction_and_grad_scaling():
    N, H, V = 33, 6, 25
    X, W, labels = _rand(N, H, V, 9)
    m = oracle.forward(X, W, labels, reduction="mean")
    s = oracle.forward(X, W, labels, reduction="sum")
    assert s["loss"] == pytest.approx(m["n_valid"] * m["loss"], rel=1e-14)
    dXm, dWm = oracle.backward(X, W, labels, reduction="mean", grad_loss=1.0)
    dXs, dWs = oracle.backward(X, W, labels, reduction="sum", grad_loss=1.0)
    np.testing.assert_allclose(dXs, m["n_valid"] * dXm, rtol=1e-12, atol=1e-14 * np.abs(dXs).max())
    dX3, dW3 = oracle.backward(X, W, labels, reduction="mean", grad_loss=-2.5)
    np.testing.assert_allclose(dW3, -2.5 * dWm, rtol=1e-12, atol=1e-14 * np.abs(dWm).max())


def test_vocab_permutation_equivariance():
    N, H, V = 20, 8, 29
    X, W, labels = _rand(N, H, V, 10)
    perm = np.random.default_rng(0).permutation(V)   # new row k holds old row perm[k]
    inv = np.argsort(perm)
    lab2 = np.where(labels == -100, -100, inv[np.where(labels == -100, 0, labels)])
    a, b = oracle.forward(X, W, labels), oracle.forward(X, W[perm], lab2)
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-13)
    np.testing.assert_allclose(b["lse"], a["lse"], rtol=1e-13)
    dXa, dWa = oracle.backward(X, W, labels)
    dXb, dWb = oracle.backward(X, W[perm], lab2)
    np.testing.assert_allclose(dXb, dXa, rtol=1e-11, atol=1e-15)
    np.testing.assert_allclose(dWb, dWa[perm], rtol=1e-11, atol=1e-15)


def test_row_permutation_equivariance():
    N, H, V = 20, 8, 29
    X, W, labels = _rand(N, H, V, 11)
    p = np.random.default_rng(1).permutation(N)
    a, b = oracle.forward(X, W, labels), oracle.forward(X[p], W, labels[p])
    np.testing.assert_allclose(b["lse"], a["lse"][p], rtol=1e-14)
    dXa, dWa = oracle.backward(X, W, labels)
    dXb, dWb = oracle.backward(X[p], W, labels[p])
    np.testing.assert_allclose(dXb, dXa[p], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dWb, dWa, rtol=1e-11, atol=1e-15)


def test_huge_logit_offset_is_stable():
    """Adding c to every logit (an extra hidden column of 1s in X and c in W)
    moves lse by c and leaves loss and gradients unchanged: this fails if the
    max is not subtracted before exponentiating."""
    N, H, V = 16, 6, 23
    X, W, labels = _rand(N, H, V, 12)
    c = 5000.0
    X1 = np.concatenate([X, np.ones((N, 1))], 1)
    W1 = np.concatenate([W, np.full((V, 1), c)], 1)
    a, b = oracle.forward(X, W, labels), oracle.forward(X1, W1, labels)
    np.testing.assert_allclose(b["lse"] - c, a["lse"], atol=1e-9)
    assert b["loss"] == pytest.approx(a["loss"], abs=1e-9)
    dXa, _ = oracle.backward(X, W, labels)
    dXb, _ = oracle.backward(X1, W1, labels)
    np.testing.assert_allclose(dXb[:, :H], dXa, atol=1e-9)


# --------------------------------------------------------------------------
# brute force and a library routine
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shift,reduction", [(False, "mean"), (True, "mean"), (True, "sum")])
def test_brute_force_equals_blas(shift, reduction):
    B, S, H, V = 2, 4, 5, 9
    X, W, labels = _rand(B * S, H, V, 13, ignore_frac=0.2)
    kw = dict(seq_len=S, shift=shift, reduction=reduction)
    loss, lse, n, dX, dW = oracle.brute_force(X.tolist(), W.tolist(), labels.tolist(),
                                              grad_loss=1.3, **kw)
    f = oracle.forward(X, W, labels, **kw)
    a, b = oracle.backward(X, W, labels, grad_loss=1.3, **kw)
    assert n == f["n_valid"]
    assert loss == pytest.approx(f["loss"], rel=1e-13)
    np.testing.assert_allclose(lse, f["lse"], rtol=1e-14)
    np.testing.assert_allclose(dX, a, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dW, b, rtol=1e-12, atol=1e-15)
    # the one-pass form used at full size, against the loops directly
    fb = oracle.forward_backward(X, W, labels, grad_loss=1.3, row_block=3, **kw)
    assert fb["n_valid"] == n
    assert fb["loss"] == pytest.approx(loss, rel=1e-13)
    np.testing.assert_allclose(fb["lse"], lse, rtol=1e-14)
    np.testing.assert_allclose(fb["dX"], dX, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(fb["dW"], dW, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_matches_torch_cross_entropy_float64(reduction):
    N, H, V = 48, 16, 57
    X, W, labels = _rand(N, H, V, 14)
    Xt = torch.tensor(X, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(Xt @ Wt.T, torch.tensor(labels),
                                             ignore_index=-100, reduction=reduction)
    loss.backward()
    f = oracle.forward(X, W, labels, reduction=reduction)
    dX, dW = oracle.backward(X, W, labels, reduction=reduction)
    assert f["loss"] == pytest.approx(loss.item(), rel=1e-13)
    np.testing.assert_allclose(dX, Xt.grad.numpy(), rtol=1e-11, atol=1e-15)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=1e-11, atol=1e-15)


# --------------------------------------------------------------------------
# degenerate cases and the sampled helpers used at full size
# --------------------------------------------------------------------------

def test_no_valid_rows():
    N, H, V = 8, 4, 10
    X, W, _ = _rand(N, H, V, 15)
    labels = np.full(N, -100)
    for red in ("mean", "sum"):
        f = oracle.forward(X, W, labels, reduction=red)
        assert f["loss"] == 0.0 and f["n_valid"] == 0
        dX, dW = oracle.backward(X, W, labels, reduction=red)
        assert not dX.any() and not dW.any()


def test_out_of_range_targets_are_flagged_and_ignored():
    N, H, V = 6, 4, 10
    X, W, _ = _rand(N, H, V, 16)
    labels = np.array([1, 10, -3, 2, -100, 9])
    t, valid, n, oor = oracle.effective_targets(labels, V)
    assert oor.tolist() == [False, True, True, False, False, False]
    assert valid.tolist() == [True, False, False, True, False, True] and n == 3
    # an ignore_index inside [0, V) wins over being a class id
    t, valid, n, oor = oracle.effective_targets(np.array([3, 4, 3]), V, ignore_index=3)
    assert valid.tolist() == [False, True, False] and not oor.any()


@pytest.mark.parametrize("row_block", [1, 7, 64, 4096])
def test_one_pass_equals_forward_and_backward(row_block):
    """forward_backward (one pass, used for whole-matrix checks at full size)
    is forward() + backward() whatever the row blocking, ragged last block
    included."""
    B, S, H, V = 3, 41, 10, 131
    X, W, labels = _rand(B * S, H, V, 18)
    for kw in (dict(seq_len=S, shift=True, reduction="mean"), dict(reduction="sum")):
        f = oracle.forward(X, W, labels, **kw)
        dX, dW = oracle.backward(X, W, labels, grad_loss=0.7, **kw)
        fb = oracle.forward_backward(X, W, labels, grad_loss=0.7, row_block=row_block, **kw)
        assert fb["n_valid"] == f["n_valid"]
        assert fb["loss"] == pytest.approx(f["loss"], rel=1e-13)
        np.testing.assert_allclose(fb["lse"], f["lse"], rtol=1e-14)
        np.testing.assert_array_equal(fb["valid"], f["valid"])
        np.testing.assert_allclose(fb["dX"], dX, rtol=1e-12, atol=1e-16)
        np.testing.assert_allclose(fb["dW"], dW, rtol=1e-11, atol=1e-16)


def test_sampled_helpers_equal_full():
    B, S, H, V = 2, 40, 9, 77
    X, W, labels = _rand(B * S, H, V, 17)
    kw = dict(seq_len=S, shift=True, reduction="mean", grad_loss=0.9)
    f = oracle.forward(X, W, labels, seq_len=S, shift=True)
    dX, dW = oracle.backward(X, W, labels, **kw)
    rows = [0, 5, 39, 40, 79]
    r = oracle.rows_forward_backward(X, W, labels, rows, **kw)
    np.testing.assert_allclose(r["lse"], f["lse"][rows], rtol=1e-14)
    np.testing.assert_allclose(r["dX"], dX[rows], rtol=1e-12, atol=1e-16)
    js = [0, 3, 76]
    np.testing.assert_allclose(oracle.vocab_rows_dW(X, W, labels, f["lse"], js, **kw),
                               dW[js], rtol=1e-11, atol=1e-16)
    rt = oracle.rows_forward_backward(torch.tensor(X), torch.tensor(W),
                                      torch.tensor(labels), rows, **kw)
    np.testing.assert_allclose(rt["dX"], r["dX"], rtol=1e-15)
