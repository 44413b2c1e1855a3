"""flce_logits, the no-label path: bf16 logits Z = X W^T against the oracle's
float64 product, on ragged shapes and a Qwen2-7B-sized vocabulary."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import to_np

pytestmark = pytest.mark.gpu

flce = pytest.importorskip("lm_head_linear_flce_gb300")

# bf16 output: each element carries a rounding error of at most 2^-9 relative
LOGITS_RTOL = 4e-3


@pytest.mark.parametrize("N,H,V", [(300, 200, 1000), (1, 64, 7), (513, 256, 4099),
                                   (1024, 512, 152064),
                                   (2800, 8192, 3000)])  # row bands of 6 and 5 tiles
def test_logits_match_float64_product(N, H, V):
    X, W, _ = workloads.random_case(N, H, V, seed=60 + N, w_std=0.1)
    dev = torch.device("cuda")
    Z = flce.flce_logits(X.to(dev), W.to(dev))
    torch.cuda.synchronize()
    assert Z.shape == (N, V) and Z.dtype == torch.bfloat16
    rows = np.arange(N) if N * V <= 1024 * 152064 else np.random.default_rng(0).choice(
        N, 256, replace=False)
    ref = oracle.logits_rows(X, W, rows)
    got = to_np(Z)[rows]
    err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= LOGITS_RTOL, err
    assert np.abs(got - ref).max() <= 2e-2 * np.abs(ref).max() + 1e-6


def test_linear_cross_entropy_without_labels_returns_logits():
    X, W, _ = workloads.random_case(64, 128, 500, seed=61)
    dev = torch.device("cuda")
    Z = flce.linear_cross_entropy(X.to(dev).view(2, 32, 128), W.to(dev), None)
    assert Z.shape == (2, 32, 500)
    ref = oracle.logits_rows(X, W, np.arange(64)).reshape(2, 32, 500)
    assert np.linalg.norm(to_np(Z) - ref) / np.linalg.norm(ref) <= LOGITS_RTOL
