"""Property checks of the oracle over many random small cases (hypothesis):
identities that must hold for any input, so that a mistake that only shows on
some shapes or label patterns is caught."""
import math

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from oracle import vocab_parallel as ovp  # noqa: E402


@st.composite
def cases(draw):
    B = draw(st.integers(1, 3))
    S = draw(st.integers(1, 6))
    H = draw(st.integers(1, 6))
    V = draw(st.integers(1, 9))
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((B * S, H))
    W = rng.standard_normal((V, H)) * draw(st.sampled_from([0.0, 0.3, 2.0]))
    labels = rng.integers(0, V, B * S)
    labels[rng.random(B * S) < draw(st.sampled_from([0.0, 0.3, 1.0]))] = -100
    return X, W, labels, S


SETTINGS = settings(max_examples=60, deadline=None, derandomize=True)


@SETTINGS
@given(cases())
def test_lse_bounds_and_loss_sign(c):
    X, W, labels, S = c
    f = oracle.forward(X, W, labels, reduction="sum")
    Z = X @ W.T
    V = W.shape[0]
    assert np.all(f["lse"] >= Z.max(1) - 1e-12)
    assert np.all(f["lse"] <= Z.max(1) + math.log(V) + 1e-12)
    assert np.all(f["row_loss"] >= -1e-12)  # -log p >= 0


@SETTINGS
@given(cases())
def test_shift_is_a_per_sequence_roll(c):
    X, W, labels, S = c
    rolled = labels.reshape(-1, S).copy()
    rolled[:, :-1] = rolled[:, 1:].copy()
    rolled[:, -1] = -100
    a = oracle.forward(X, W, labels, seq_len=S, shift=True)
    b = oracle.forward(X, W, rolled.reshape(-1))
    assert a["n_valid"] == b["n_valid"]
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-12, abs=1e-12)
    dXa, dWa = oracle.backward(X, W, labels, seq_len=S, shift=True)
    dXb, dWb = oracle.backward(X, W, rolled.reshape(-1))
    np.testing.assert_allclose(dXa, dXb, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dWa, dWb, rtol=1e-12, atol=1e-14)


@SETTINGS
@given(cases(), st.floats(-3, 3))
def test_sum_is_n_valid_times_mean_and_grads_are_linear_in_g(c, g):
    X, W, labels, S = c
    m = oracle.forward(X, W, labels, reduction="mean")
    s = oracle.forward(X, W, labels, reduction="sum")
    assert s["loss"] == pytest.approx(m["n_valid"] * m["loss"], rel=1e-12, abs=1e-12)
    dXm, dWm = oracle.backward(X, W, labels, reduction="mean", grad_loss=g)
    dXs, dWs = oracle.backward(X, W, labels, reduction="sum", grad_loss=g)
    n = m["n_valid"]
    if n:
        np.testing.assert_allclose(dXs, n * dXm, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dWs, n * dWm, rtol=1e-10, atol=1e-12)
    else:
        assert not dXm.any() and not dWs.any()


@SETTINGS
@given(cases(), st.data())
def test_any_vocabulary_split_reproduces_the_whole(c, data):
    X, W, labels, S = c
    V = W.shape[0]
    cuts = sorted(set(data.draw(st.lists(st.integers(1, max(1, V - 1)), max_size=3)))) if V > 1 else []
    bounds = [(a, b - a) for a, b in zip([0] + cuts, cuts + [V])]
    lse_p, z_p = [], []
    for v0, n in bounds:
        l, z, nv, valid = ovp.shard_forward(X, W[v0:v0 + n], labels, v0, V)
        lse_p.append(l)
        z_p.append(z)
    loss, lse = ovp.merge_shards(lse_p, z_p, valid, nv, "mean")
    ref = oracle.forward(X, W, labels)
    assert loss == pytest.approx(ref["loss"], rel=1e-12, abs=1e-12)
    np.testing.assert_allclose(lse, ref["lse"], rtol=1e-12)
    dX = sum(ovp.shard_backward(X, W[v0:v0 + n], labels, v0, V, lse)[0] for v0, n in bounds)
    rdX, _ = oracle.backward(X, W, labels)
    np.testing.assert_allclose(dX, rdX, rtol=1e-10, atol=1e-12)
