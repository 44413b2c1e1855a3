"""Pins of the vocabulary-parallel oracle (shard forward, merge, shard
backward) to the unsharded oracle and to closed forms.

The unsharded oracle is itself pinned (closed forms, finite differences,
brute force, a library routine); splitting the vocabulary must reproduce it to
float64 rounding, whatever the split.  The closed forms catch a merge that
averages instead of log-sum-exp-ing, a z that is taken from the wrong shard or
counted twice, and validity judged against the shard instead of the whole
vocabulary.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import vocab_parallel as vp


def _rand(N, H, V, seed, ignore_frac=0.2, w_std=0.5):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((N, H))
    W = rng.standard_normal((V, H)) * w_std
    labels = rng.integers(0, V, N)
    labels[rng.random(N) < ignore_frac] = -100
    return X, W, labels


def _sharded(X, W, labels, sizes, *, seq_len=None, shift=False, reduction="mean", grad=1.0):
    V = W.shape[0]
    bounds = vp.split_bounds(V, sizes)
    lse_p, z_p = [], []
    for v0, n in bounds:
        l, z, nv, valid = vp.shard_forward(X, W[v0:v0 + n], labels, v0, V, seq_len=seq_len,
                                           shift=shift)
        lse_p.append(l)
        z_p.append(z)
    loss, lse = vp.merge_shards(lse_p, z_p, valid, nv, reduction)
    dX = np.zeros_like(X)
    dWs = []
    for v0, n in bounds:
        dx, dw = vp.shard_backward(X, W[v0:v0 + n], labels, v0, V, lse, seq_len=seq_len,
                                   shift=shift, reduction=reduction, grad_loss=grad)
        dX += dx
        dWs.append(dw)
    return loss, lse, nv, dX, np.concatenate(dWs), lse_p, z_p


@pytest.mark.parametrize("sizes,shift,reduction", [
    ([97], False, "mean"),                 # one shard: the unsharded call
    ([40, 57], True, "mean"),
    ([1, 30, 66], False, "sum"),           # a one-column shard
    ([25, 24, 24, 24], True, "sum"),
])
def test_shards_reproduce_unsharded(sizes, shift, reduction):
    X, W, labels = _rand(48, 12, 97, seed=sum(sizes) + len(sizes))
    S = 12 if shift else None
    loss, lse, nv, dX, dW, _, _ = _sharded(X, W, labels, sizes, seq_len=S, shift=shift,
                                           reduction=reduction, grad=0.7)
    ref = oracle.forward(X, W, labels, seq_len=S, shift=shift, reduction=reduction)
    rdX, rdW = oracle.backward(X, W, labels, seq_len=S, shift=shift, reduction=reduction,
                               grad_loss=0.7)
    assert nv == ref["n_valid"]
    assert loss == pytest.approx(ref["loss"], rel=1e-13)
    np.testing.assert_allclose(lse, ref["lse"], rtol=1e-13)
    np.testing.assert_allclose(dX, rdX, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(dW, rdW, rtol=1e-11, atol=1e-14)


def test_w_zero_closed_form_per_shard():
    # W = 0: every logit is 0, so lse_r = ln V_r, z_r = 0, the merged lse is
    # ln V and the loss is ln V (mean)
    N, H, sizes = 20, 8, [3, 5, 8]
    V = sum(sizes)
    X, _, labels = _rand(N, H, V, seed=3)
    W = np.zeros((V, H))
    loss, lse, nv, dX, dW, lse_p, z_p = _sharded(X, W, labels, sizes)
    for (v0, n), l, z in zip(vp.split_bounds(V, sizes), lse_p, z_p):
        np.testing.assert_allclose(l, math.log(n), rtol=1e-15)
        assert not z.any()
    np.testing.assert_allclose(lse, math.log(V), rtol=1e-15)
    assert loss == pytest.approx(math.log(V), rel=1e-15)
    assert not dX.any()


def test_two_one_column_shards_are_the_logistic_loss():
    # V = 2 split as [1, 1]: lse_r is that column's logit; the merge gives
    # softplus(z_other - z_target) per valid row
    rng = np.random.default_rng(4)
    X = rng.standard_normal((9, 4))
    W = rng.standard_normal((2, 4))
    labels = np.array([0, 1, 1, -100, 0, 1, 0, 0, 1])
    loss, lse, nv, dX, dW, lse_p, z_p = _sharded(X, W, labels, [1, 1], reduction="sum")
    Z = X @ W.T
    np.testing.assert_allclose(lse_p[0], Z[:, 0], rtol=1e-14)
    np.testing.assert_allclose(lse_p[1], Z[:, 1], rtol=1e-14)
    valid = labels >= 0
    t = np.where(valid, labels, 0)
    margin = Z[np.arange(9), 1 - t] - Z[np.arange(9), t]
    expect = np.sum(np.where(valid, np.logaddexp(0.0, margin), 0.0))
    assert loss == pytest.approx(expect, rel=1e-14)


def test_target_counted_once_and_validity_is_global():
    X, W, labels = _rand(30, 6, 40, seed=5, ignore_frac=0.0)
    labels[:] = 25  # every target in the second shard of [20, 20]
    labels[3] = 19  # ... except one, the last column of the first shard
    labels[4] = 20  # ... and the first column of the second
    l0, z0, nv0, _ = vp.shard_forward(X, W[:20], labels, 0, 40)
    l1, z1, nv1, _ = vp.shard_forward(X, W[20:], labels, 20, 40)
    assert nv0 == nv1 == 30  # rows whose target is elsewhere still count
    Z = X @ W.T
    assert np.count_nonzero(z0) == 1 and z0[3] == Z[3, 19]
    assert z1[3] == 0.0 and z1[4] == Z[4, 20] and z1[0] == Z[0, 25]
    # the backward of the first shard has softmax terms on every row but a
    # one-hot term only on row 3
    _, lse = vp.merge_shards([l0, l1], [z0, z1], np.ones(30, bool), 30, "sum")
    _, dW0 = vp.shard_backward(X, W[:20], labels, 0, 40, lse, reduction="sum")
    P = np.exp(Z - lse[:, None])
    P[3, 19] -= 1.0
    np.testing.assert_allclose(dW0, P[:, :20].T @ X, rtol=1e-12)


def test_split_bounds_must_cover_the_vocabulary():
    assert vp.split_bounds(10, [4, 6]) == [(0, 4), (4, 6)]
    with pytest.raises(ValueError):
        vp.split_bounds(10, [4, 5])
