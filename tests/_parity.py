"""Shared comparison helpers for the GPU parity tests (tolerances of the
fused linear cross-entropy spec: loss rel. error <= 1e-4, lse abs. error
<= 2e-3, gradients rel. Frobenius error <= 1e-2 with cosine >= 0.9999,
n_valid exact)."""
import numpy as np

LOSS_RTOL = 1e-4
LSE_ATOL = 2e-3
GRAD_RTOL = 1e-2
GRAD_COS = 0.9999


def to_np(t):
    return t.detach().double().cpu().numpy()


def grad_metrics(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nr = np.linalg.norm(ref)
    ng = np.linalg.norm(got)
    if nr == 0.0:
        return (0.0 if ng == 0.0 else np.inf), (1.0 if ng == 0.0 else 0.0)
    rel = float(np.linalg.norm(got - ref) / nr)
    cos = float((got * ref).sum() / (nr * ng)) if ng > 0 else 0.0
    return rel, cos


def assert_grad(name, got, ref):
    rel, cos = grad_metrics(got, ref)
    assert rel <= GRAD_RTOL and cos >= GRAD_COS, f"{name}: rel {rel:.3e} cos {cos:.7f}"


def assert_loss(got, ref):
    if ref == 0.0:
        assert got == 0.0, got
    else:
        assert abs(got - ref) <= LOSS_RTOL * abs(ref), (got, ref)


def assert_lse(got, ref):
    err = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))
    assert err.max() <= LSE_ATOL, f"lse max abs err {err.max():.3e}"


# Oracle forward results of the full-size workloads, kept for the rest of the
# test session (loss, lse, n_valid: small) so that a later test on the same
# workload need not redo minutes of host work.  Filled by whichever test
# computes them first; oracle_forward_cached computes them when absent, so
# every test also runs on its own.
_ORACLE_FORWARD = {}


def remember_oracle_forward(name, ref):
    _ORACLE_FORWARD[name] = {k: ref[k] for k in ("loss", "lse", "n_valid", "valid")}


def oracle_forward_cached(name, X, W, labels, **kw):
    if name not in _ORACLE_FORWARD:
        import oracle
        remember_oracle_forward(name, oracle.forward(X, W, labels, **kw))
    return _ORACLE_FORWARD[name]
