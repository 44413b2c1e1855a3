"""Brute-force loop version of the oracle, for tiny shapes only.

TEST INFRASTRUCTURE ONLY (see ``oracle/flce_oracle.py``).  It writes the same
definition as ``flce_oracle`` with explicit Python loops and ``math`` functions
instead of BLAS and numpy reductions, so the two can check each other: every
dot product, max, exp, log and sum is spelled out one element at a time.
Definition: Z = X W^T, per-row cross-entropy with ignore_index, optional
per-sequence one-position shift, mean or sum; dX = dZ W, dW = dZ^T X
(ms-swift PR #9784, section Mathematical Equivalence).
"""
from __future__ import annotations

import math


def brute_force(X, W, labels, *, seq_len=None, shift=False, ignore_index=-100,
                reduction="mean", grad_loss=1.0):
    """X, W: nested lists of floats; labels: list of ints.
    Returns (loss, lse list, n_valid, dX nested list, dW nested list)."""
    N, V, H = len(X), len(W), len(W[0]) if W else 0
    S = N if not seq_len else seq_len
    # targets after the shift, sequence by sequence
    t = []
    for i in range(N):
        if shift:
            pos = i % S
            t.append(labels[i + 1] if pos + 1 < S else ignore_index)
        else:
            t.append(labels[i])
    valid = [ti != ignore_index and 0 <= ti < V for ti in t]
    n_valid = sum(1 for v in valid if v)

    Z = [[sum(X[i][h] * W[j][h] for h in range(H)) for j in range(V)] for i in range(N)]
    lse = []
    for i in range(N):
        m = max(Z[i])
        lse.append(m + math.log(sum(math.exp(z - m) for z in Z[i])))
    total = 0.0
    for i in range(N):
        if valid[i]:
            total += lse[i] - Z[i][t[i]]
    if reduction == "mean":
        loss = total / n_valid if n_valid else 0.0
        s = grad_loss / n_valid if n_valid else 0.0
    else:
        loss = total
        s = grad_loss

    dZ = [[0.0] * V for _ in range(N)]
    for i in range(N):
        if not valid[i]:
            continue
        for j in range(V):
            p = math.exp(Z[i][j] - lse[i])
            dZ[i][j] = s * (p - (1.0 if j == t[i] else 0.0))
    dX = [[sum(dZ[i][j] * W[j][h] for j in range(V)) for h in range(H)] for i in range(N)]
    dW = [[sum(dZ[i][j] * X[i][h] for i in range(N)) for h in range(H)] for j in range(V)]
    return loss, lse, n_valid, dX, dW
