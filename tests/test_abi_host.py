"""The C ABI without a GPU: the library loads, exports every symbol declared in
include/flce.h, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flce.h")

flce = pytest.importorskip("lm_head_linear_flce_gb300")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(flce.library_path):
        from lm_head_linear_flce_gb300 import _build
        _build.build()
    return flce.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flce_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("flce_workspace_size", "flce_forward", "flce_backward", "flce_get_error",
                 "flce_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in flce.STATUS.items():
        assert lib.flce_status_string(code).decode() == name


def test_workspace_size_is_bounded(lib):
    # O(N*H + Vb*H + N*V/1024), far below the N x V logits it replaces
    for N, H, V in [(8192, 3584, 152064), (32768, 2048, 151936), (4096, 8192, 128256),
                    (16384, 4096, 151936), (256, 256, 4096)]:
        ws = lib.flce_workspace_size(N, H, V)
        assert ws > 0
        assert ws < 0.2 * N * V * 2 + (N + 8192) * H * 4 + 64 * 2**20, (N, H, V, ws)
    assert lib.flce_workspace_size(8, 12, 100) == 0     # H % 8 != 0
    assert lib.flce_workspace_size(8, 0, 100) == 0
    assert lib.flce_workspace_size(-1, 64, 100) == 0
    assert lib.flce_workspace_size(0, 64, 100) > 0      # an empty batch is allowed


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def test_forward_rejects_bad_arguments_on_host(lib):
    ws_need = lib.flce_workspace_size(64, 64, 100)
    args = dict(X=_fake(), W=_fake(), labels=_fake(), N=64, H=64, V=100, seq_len=0,
                ignore=-100, shift=0, red=0, loss=_fake(), lse=_fake(), nv=_fake(),
                ws=_fake(0x100000), wsb=ws_need, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return lib.flce_forward(a["X"], a["W"], a["labels"], a["N"], a["H"], a["V"],
                                a["seq_len"], a["ignore"], a["shift"], a["red"], a["loss"],
                                a["lse"], a["nv"], a["ws"], a["wsb"], a["stream"])

    assert call(X=None) == 1
    assert call(H=12) == 2
    assert call(V=0) == 1
    assert call(red=7) == 1
    assert call(wsb=ws_need - 1) == 3
    assert call(ws=_fake(0x100010)) == 1               # workspace not 256-byte aligned
    assert call(X=_fake(0x10008)) == 1                 # X not 16-byte aligned
    assert call(shift=1, seq_len=48) == 1              # N % seq_len != 0


def test_backward_rejects_bad_arguments_on_host(lib):
    ws_need = lib.flce_workspace_size(64, 64, 100)
    f = lib.flce_backward
    base = [_fake(), _fake(), _fake(), 64, 64, 100, 0, -100, 0, 0, _fake(), _fake(), _fake(),
            _fake(), _fake(), _fake(0x100000), ws_need, None]
    assert f(*base[:12], None, *base[13:]) == 1       # no grad_loss
    b = list(base)
    b[16] = ws_need - 256
    assert f(*b) == 3


def test_plan_blocks_follow_the_tuning_knob(lib):
    a = lib.flce_workspace_size(4096, 1024, 50000)
    lib.flce_set_backward_block(128, 128 * 256)
    try:
        b = lib.flce_workspace_size(4096, 1024, 50000)
    finally:
        lib.flce_set_backward_block(0, 0)
    assert lib.flce_workspace_size(4096, 1024, 50000) == a
    assert b != a


def test_vocab_shard_entry_points_reject_bad_arguments_on_host(lib):
    N, H, V, Vt = 64, 64, 100, 300
    ws_need = lib.flce_workspace_size(N, H, V)
    i64, c_int = ctypes.c_int64, ctypes.c_int

    def fwd(v_offset=100, V_total=Vt, Vs=V, z=_fake(), wsb=ws_need):
        return lib.flce_forward_vocab_shard(_fake(), _fake(), _fake(), i64(N), i64(H), i64(Vs),
                                            i64(v_offset), i64(V_total), i64(0), i64(-100),
                                            c_int(0), _fake(), z, _fake(), _fake(0x100000),
                                            ctypes.c_size_t(wsb), None)

    assert fwd(v_offset=-1) == 1
    assert fwd(v_offset=201) == 1                 # shard runs past the vocabulary
    assert fwd(V_total=0) == 1
    assert fwd(z=None) == 1
    assert fwd(wsb=ws_need - 1) == 3

    def bwd(v_offset=0, V_total=Vt, dx=_fake(0x200000), dw=_fake(0x300000)):
        return lib.flce_backward_vocab_shard(_fake(), _fake(), _fake(), i64(N), i64(H), i64(V),
                                             i64(v_offset), i64(V_total), i64(0), i64(-100),
                                             c_int(0), c_int(0), _fake(), _fake(), _fake(), dx,
                                             dw, _fake(0x100000), ctypes.c_size_t(ws_need), None)

    assert bwd(v_offset=250) == 1
    assert bwd(dx=_fake(0x200004)) == 1          # FP32 buffer not 16-byte aligned

    def merge(P=2, red=0, wsb=1 << 20, ws=_fake(0x100000)):
        return lib.flce_merge_vocab_shards(_fake(), _fake(), i64(P), _fake(), i64(N), i64(Vt),
                                           i64(0), i64(-100), c_int(0), c_int(red), _fake(),
                                           _fake(), _fake(), ws, ctypes.c_size_t(wsb), None)

    assert merge(P=0) == 1
    assert merge(red=3) == 1
    assert merge(wsb=256) == 3
    assert merge(ws=_fake(0x100008)) == 1

    def down(count=64, src=_fake(0x200000)):
        return lib.flce_downcast_bf16(src, _fake(0x300000), i64(count), None)

    assert down(count=12) == 1
    assert down(count=0) == 0
    assert down(src=_fake(0x200008)) == 1


def _noalloc_need(N, V):
    """Scratch bytes of flce_forward_noalloc, as the header states them."""
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    T = -(-V // 256)
    U = -(-T // max(4, -(-T // 128)))
    assert U <= 128
    return 256 + 2 * up(4 * N) + up(8 * N * U) + up(8 * (-(-N // 32) + 1)) + 256


@pytest.mark.parametrize("V", [4096, 32768, 151936, 152064, 262144, 1 << 22])
def test_noalloc_scratch_formula(lib, V):
    """The largest N the header's formula lets into the 16 MiB scratch passes
    the size check and one more row is refused, before anything is enqueued."""
    import torch
    cap = 16 << 20
    lo, hi = 1, 1 << 20
    while lo < hi:  # largest N with need(N) <= cap
        mid = (lo + hi + 1) // 2
        lo, hi = (mid, hi) if _noalloc_need(mid, V) <= cap else (lo, mid - 1)
    n_max = lo
    i64, c_int = ctypes.c_int64, ctypes.c_int
    fn = lib.flce_forward_noalloc
    fn.argtypes = [ctypes.c_void_p] * 3 + [i64] * 5 + [c_int, c_int] + [ctypes.c_void_p] * 5
    fn.restype = c_int

    def call(N):
        return fn(_fake(), _fake(), _fake(), N, 8, V, 0, -100, 0, 0, _fake(), _fake(), _fake(),
                  None, None)

    assert call(n_max + 1) == 3
    if not torch.cuda.is_available():
        # passes the size check, then stops at the device query (no GPU here)
        assert call(n_max) not in (0, 3)


def test_forward_partials_do_not_grow_with_the_vocabulary(lib):
    # at most 128 (max, sum-exp) partials per row whatever V is: with a
    # vocabulary past 512 tiles the noalloc size limit no longer moves
    assert _noalloc_need(8192, 1 << 22) == _noalloc_need(8192, 1 << 24)
    assert _noalloc_need(8192, 152064) < _noalloc_need(8192, 1 << 22)


def test_large_blocks_grow_until_a_launch_holds_enough_dw_tiles(lib):
    """Above 8192 rows, with every row in one block, the automatic dZ block
    doubles (up to 2^27 elements) while it would hold fewer than 76 dW tiles of
    256 x 256 (include/flce.h, flce_set_backward_block): at N = 32768 and
    H = 2048 a 64 Mi-element block has 2048 vocab columns (8 x 8 = 64 dW
    tiles), so it grows to 4096 columns: both dZ slots gain 32768 x 2048
    bf16 elements over the same plan with the cap set to 64 Mi by hand."""
    N, H, V = 32768, 2048, 151936
    auto = lib.flce_workspace_size(N, H, V)
    lib.flce_set_backward_block(0, 64 << 20)
    try:
        capped = lib.flce_workspace_size(N, H, V)
    finally:
        lib.flce_set_backward_block(0, 0)
    # (the per-launch counters shrink a little with half as many blocks)
    assert abs((auto - capped) - 2 * N * 2048 * 2) <= 64 * 1024, auto - capped
    # enough dW tiles already (H = 4096: 16 x 16 at 4096 columns): no growth
    lib.flce_set_backward_block(0, 64 << 20)
    try:
        capped = lib.flce_workspace_size(16384, 4096, V)
    finally:
        lib.flce_set_backward_block(0, 0)
    assert lib.flce_workspace_size(16384, 4096, V) == capped


def test_w_block_kept_within_64_mib(lib):
    """The automatic block's vocab width is capped so that its W rows (Vb x H
    bf16) take at most 64 MiB (include/flce.h, flce_set_backward_block).  At
    N = 4096 and H = 8192 the 32 Mi-element cap alone gives 8192 columns
    (128 MiB of W rows), so the width drops to 4096: the plan is the one a
    16 Mi-element cap set by hand gives, and both dZ slots shrink by 4096 x
    4096 bf16 elements against the 32 Mi-element cap set by hand (which the
    W-row cap leaves alone).  At H = 3584 it does not bind."""
    N, H, V = 4096, 8192, 128256
    auto = lib.flce_workspace_size(N, H, V)
    try:
        lib.flce_set_backward_block(0, 16 << 20)
        narrow = lib.flce_workspace_size(N, H, V)
        lib.flce_set_backward_block(0, 32 << 20)
        wide = lib.flce_workspace_size(N, H, V)
        lib.flce_set_backward_block(0, 32 << 20)
        qwen2_by_hand = lib.flce_workspace_size(8192, 3584, 152064)
    finally:
        lib.flce_set_backward_block(0, 0)
    assert auto == narrow
    # (the per-launch counters grow a little with twice as many blocks)
    assert abs((wide - auto) - 2 * N * 4096 * 2) <= 64 * 1024, wide - auto
    assert lib.flce_workspace_size(8192, 3584, 152064) == qwen2_by_hand


def test_backward_blocking_of_the_five_workloads(lib):
    """flce_backward_blocking reports the automatic dZ block (include/flce.h,
    flce_set_backward_block): every row in one token block for all five
    workloads; 4096 vocab columns where V spans several blocks (the 32 Mi /
    64 Mi element caps, the 76-dW-tile growth at 32K rows, the 64 MiB W-row
    cap at H = 8192); the whole 4096-column vocabulary of the tiny workload in
    one block, which keeps it on token tiles rather than dense rows."""
    import ctypes
    fn = lib.flce_backward_blocking
    fn.argtypes = [ctypes.c_int64] * 3 + [ctypes.POINTER(ctypes.c_int64)] * 2
    fn.restype = ctypes.c_int
    want = {(256, 256, 4096): (256, 4096), (8192, 3584, 152064): (8192, 4096),
            (16384, 4096, 151936): (16384, 4096), (32768, 2048, 151936): (32768, 4096),
            (4096, 8192, 128256): (4096, 4096)}
    for (N, H, V), blk in want.items():
        nb, vb = ctypes.c_int64(), ctypes.c_int64()
        assert fn(N, H, V, ctypes.byref(nb), ctypes.byref(vb)) == 0
        assert (nb.value, vb.value) == blk, (N, H, V, nb.value, vb.value)
    nb, vb = ctypes.c_int64(), ctypes.c_int64()
    assert fn(8192, 3583, 152064, ctypes.byref(nb), ctypes.byref(vb)) != 0  # H % 8 != 0


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="made-up device addresses: only where no kernel can run")
def test_backward_refuses_outputs_that_overlap_on_the_host(lib):
    """No output may overlap an input, the workspace or another output
    (include/flce.h, flce_backward): refused with FLCE_ERR_INVALID_ARG on the
    host, before anything is enqueued.  Made-up, suitably aligned addresses
    stand in for device buffers."""
    N, H, V = 512, 64, 1000
    nh = N * H * 2
    base = 1 << 40
    X, W = base, base + (1 << 30)
    labels, lse, nv, g = base + (2 << 30), base + (3 << 30), base + (4 << 30), base + (5 << 30)
    ws, wsn = base + (6 << 30), lib.flce_workspace_size(N, H, V)
    dX, dW = base + (8 << 30), base + (9 << 30)
    fn = lib.flce_backward
    P = ctypes.c_void_p

    def call(dx, dw):
        return fn(P(X), P(W), P(labels), N, H, V, 0, -100, 0, 0, P(lse), P(nv), P(g),
                  P(dx), P(dw), P(ws), wsn, None)

    for dx, dw in [(X, None), (X + nh - 16, None), (W, None), (None, W + 256),
                   (dX, dX + nh - 16), (dW + 4096, dW), (ws + 256, None), (None, ws),
                   (lse - 16 * 64, None), (None, labels)]:
        assert call(dx, dw) == 1, (dx, dw)
