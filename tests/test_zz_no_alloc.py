"""flce_forward_noalloc: the forward for callers that cannot allocate device
memory -- a plugin inside a host framework that owns every device allocation
and hands the plugin only its input and output buffers, or a latency-critical
path where the device-synchronising cudaMalloc / cudaFree are not allowed.

The entry point keeps its scratch in a fixed 16 MiB array inside the library
(shared by every call, keeping the last call's contents), so these tests check
its outputs against the CPU float64 oracle -- the loss, the lse of every row
and the exact valid count -- on calls in a row of different shapes (each over
the previous call's leftovers), at the full Qwen2-7B forward size, and on a
clean call right after a call that raised a device error; that a call made
with every output preallocated moves neither the device's free memory nor
torch's allocator; that the wait limit set by flce_set_wait_limit_ns reaches
its launch; and that problems too large for the array are refused before
anything runs.  This file sorts last so that a stop-at-first-failure run has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import assert_loss, assert_lse, oracle_forward_cached

pytestmark = pytest.mark.gpu

flce = pytest.importorskip("lm_head_linear_flce_gb300")

_RED = {"mean": 0, "sum": 1}


def _c_noalloc():
    fn = flce.library().flce_forward_noalloc
    c_i64, c_p, c_int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [c_p, c_p, c_p, c_i64, c_i64, c_i64, c_i64, c_i64, c_int, c_int,
                   c_p, c_p, c_p, c_p, c_p]
    fn.restype = c_int
    return fn


def _call(bufs, N, H, V, seq_len=0, shift=False, reduction="mean", ignore_index=-100):
    """One flce_forward_noalloc through the C ABI into preallocated outputs."""
    X, W, L, loss, lse, nv, derr = bufs
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = _c_noalloc()(p(X), p(W), p(L), N, H, V, seq_len, ignore_index, int(shift),
                      _RED[reduction], p(loss), p(lse), p(nv), p(derr),
                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def _buffers(X, W, L):
    dev = torch.device("cuda")
    N = X.shape[0]
    return (X.to(dev), W.to(dev), L.to(dev), torch.empty(1, dtype=torch.float32, device=dev),
            torch.empty(N, dtype=torch.float32, device=dev),
            torch.empty(1, dtype=torch.int64, device=dev),
            torch.empty(1, dtype=torch.int32, device=dev))


def _check_against_oracle(bufs, ref):
    torch.cuda.synchronize()
    _, _, _, loss, lse, nv, derr = bufs
    assert int(derr.item()) == 0
    assert int(nv.item()) == ref["n_valid"]
    assert_loss(loss.item(), ref["loss"])
    assert_lse(lse.cpu().numpy(), ref["lse"])


CASES = [  # (N, H, V, seed, ignore_frac, kwargs): ragged tiles, shift, sum, and a
    # vocabulary of more than 512 tiles (work units of 5 tiles, not 4)
    (1000, 200, 3000, 21, 0.1, dict(seq_len=250, shift=True)),
    (384, 136, 1500, 22, 0.5, dict(reduction="sum")),
    (300, 64, 140000, 24, 0.1, dict(reduction="mean")),
]


def test_calls_in_a_row_match_the_oracle():
    for N, H, V, seed, frac, kw in CASES + CASES[:1]:
        X, W, L = workloads.random_case(N, H, V, seed=seed, ignore_frac=frac)
        bufs = _buffers(X, W, L)
        assert _call(bufs, N, H, V, **kw) == 0
        _check_against_oracle(bufs, oracle.forward(X, W, L, **kw))


def test_full_qwen2_7b_forward_fits_and_matches_twice():
    wl = workloads.get("qwen2_7b")
    X, W, L = workloads.make_inputs(wl)
    kw = dict(seq_len=wl.S, shift=wl.shift, reduction=wl.reduction)
    ref = oracle_forward_cached(wl.name, X, W, L, **kw)
    bufs = _buffers(X, W, L)
    for _ in range(2):
        bufs[4].fill_(float("nan"))
        assert _call(bufs, wl.N, wl.H, wl.V, **kw) == 0
        _check_against_oracle(bufs, ref)


def test_a_call_with_preallocated_outputs_allocates_nothing():
    N, H, V = 2048, 512, 20000
    X, W, L = workloads.random_case(N, H, V, seed=25)
    bufs = _buffers(X, W, L)
    assert _call(bufs, N, H, V) == 0  # first call on the device: one-time set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_stats()["allocation.all.allocated"]
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(2):
        assert _call(bufs, N, H, V) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_stats()["allocation.all.allocated"] == alloc0
    assert torch.cuda.memory_reserved() == reserved0
    _check_against_oracle(bufs, oracle.forward(X, W, L))


def test_clean_call_after_a_device_error():
    N, H, V = 256, 64, 500
    X, W, L = workloads.random_case(N, H, V, seed=23)
    bad = L.clone()
    bad[3] = 999  # outside [0, V) and not ignore_index
    bufs = _buffers(X, W, bad)
    assert _call(bufs, N, H, V) == 0
    torch.cuda.synchronize()
    assert int(bufs[6].item()) == 1  # label out of range, reported through device_error
    ref_bad = oracle.forward(X, W, bad)  # the bad row counts as ignored
    assert int(bufs[5].item()) == ref_bad["n_valid"]
    assert_loss(bufs[3].item(), ref_bad["loss"])
    bufs[2].copy_(L.cuda())
    assert _call(bufs, N, H, V) == 0  # the next call starts from a clear error word
    _check_against_oracle(bufs, oracle.forward(X, W, L))


def test_wait_limit_reaches_the_launch():
    N, H, V = 512, 128, 3000
    X, W, L = workloads.random_case(N, H, V, seed=26)
    bufs = _buffers(X, W, L)
    try:
        flce.flce_set_wait_limit_ns(3_000_000_007)
        assert _call(bufs, N, H, V) == 0
        assert flce.flce_last_launch_wait_limit_ns() == 3_000_000_007
    finally:
        flce.flce_set_wait_limit_ns(0)  # back to the default
    assert _call(bufs, N, H, V) == 0
    assert flce.flce_last_launch_wait_limit_ns() == 2_000_000_000
    _check_against_oracle(bufs, oracle.forward(X, W, L))


def test_problem_larger_than_the_scratch_is_refused():
    dev = torch.device("cuda")
    N, H, V = 32768, 8, 151936  # needs about 31 MB of scratch
    X = torch.zeros(N, H, dtype=torch.bfloat16, device=dev)
    W = torch.zeros(V, H, dtype=torch.bfloat16, device=dev)
    L = torch.zeros(N, dtype=torch.int64, device=dev)
    with pytest.raises(flce.FlceError) as e:
        flce.flce_forward_noalloc(X, W, L)
    assert e.value.status == 3  # FLCE_ERR_WORKSPACE_TOO_SMALL
    # and a problem that fits runs afterwards as usual
    Xs, Ws, Ls = workloads.random_case(256, 64, 777, seed=27)
    bufs = _buffers(Xs, Ws, Ls)
    assert _call(bufs, 256, 64, 777) == 0
    _check_against_oracle(bufs, oracle.forward(Xs, Ws, Ls))
    assert np.isfinite(bufs[4].cpu().numpy()).all()
