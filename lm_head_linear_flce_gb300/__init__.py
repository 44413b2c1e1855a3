"""Fused linear cross-entropy for one GB300 GPU.

A thin Python binding over the C ABI in ``include/flce.h`` (``libflce.so``).
It only marshals arguments: tensors become device pointers, the stream is
torch's current stream, and the workspace comes from torch's caching
allocator.  Every step of the computation runs in the library's kernels; there
is no fallback path.  If the library has not been built, every call raises.

The user-facing call mirrors ``linear_cross_entropy(hidden, weight, labels,
ignore_index=-100, shift=True, reduction="mean")`` from the Qwen3.5-35B-A3B
LoRA SFT blog post (listing `_patch_model_with_cce`), with W stored
(vocab, hidden).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "FlceError", "library", "library_path", "workspace_size", "flce_forward", "flce_backward",
    "flce_get_error", "flce_selftest_wait_timeout", "flce_set_wait_limit_ns",
    "flce_set_backward_block", "flce_backward_blocking", "flce_kernel_launch_count",
    "flce_last_launch_wait_limit_ns",
    "flce_profile_enable",
    "flce_profile_collect", "PROFILE_KINDS", "flce_forward_noalloc", "flce_backward_accumulate",
    "flce_logits", "flce_forward_vocab_shard", "flce_merge_vocab_shards",
    "flce_backward_vocab_shard", "flce_downcast_bf16",
    "linear_cross_entropy", "STATUS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "_lib", "libflce.so")

STATUS = {
    0: "FLCE_OK", 1: "FLCE_ERR_INVALID_ARG", 2: "FLCE_ERR_UNSUPPORTED_SHAPE",
    3: "FLCE_ERR_WORKSPACE_TOO_SMALL", 4: "FLCE_ERR_LABEL_OUT_OF_RANGE", 5: "FLCE_ERR_TIMEOUT",
    6: "FLCE_ERR_CUDA", 7: "FLCE_ERR_UNSUPPORTED_DEVICE",
}
_REDUCTION = {"mean": 0, "sum": 1}


class FlceError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


_lib = None


def library() -> ctypes.CDLL:
    """The loaded libflce.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise RuntimeError(
            f"{library_path} is missing: build it with lm_head_linear_flce_gb300._build.build() "
            "(nvcc, sm_103a); there is no fallback implementation")
    lib = ctypes.CDLL(library_path)
    c_i64, c_sz, c_p, c_int = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
    lib.flce_workspace_size.argtypes = [c_i64, c_i64, c_i64]
    lib.flce_workspace_size.restype = c_sz
    lib.flce_forward.argtypes = [c_p, c_p, c_p, c_i64, c_i64, c_i64, c_i64, c_i64, c_int, c_int,
                                 c_p, c_p, c_p, c_p, c_sz, c_p]
    lib.flce_forward.restype = c_int
    lib.flce_backward.argtypes = [c_p, c_p, c_p, c_i64, c_i64, c_i64, c_i64, c_i64, c_int, c_int,
                                  c_p, c_p, c_p, c_p, c_p, c_p, c_sz, c_p]
    lib.flce_backward.restype = c_int
    lib.flce_get_error.argtypes = [c_p, c_p]
    lib.flce_get_error.restype = c_int
    lib.flce_status_string.argtypes = [c_int]
    lib.flce_status_string.restype = ctypes.c_char_p
    lib.flce_set_wait_limit_ns.argtypes = [c_i64]
    lib.flce_set_wait_limit_ns.restype = None
    lib.flce_set_backward_block.argtypes = [c_i64, c_i64]
    lib.flce_set_backward_block.restype = None
    lib.flce_backward_blocking.argtypes = [c_i64, c_i64, c_i64, ctypes.POINTER(c_i64),
                                           ctypes.POINTER(c_i64)]
    lib.flce_backward_blocking.restype = c_int
    lib.flce_kernel_launch_count.argtypes = []
    lib.flce_kernel_launch_count.restype = c_i64
    lib.flce_profile_enable.argtypes = [c_int]
    lib.flce_profile_enable.restype = None
    lib.flce_profile_collect.argtypes = [c_p, c_p]
    lib.flce_profile_collect.restype = c_int
    lib.flce_selftest_wait_timeout.argtypes = [c_i64, c_p, c_sz, c_p]
    lib.flce_selftest_wait_timeout.restype = c_int
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(status: int, where: str) -> None:
    if status != 0:
        raise FlceError(status, where)


def workspace_size(N: int, H: int, V: int) -> int:
    return int(library().flce_workspace_size(N, H, V))


def _workspace(N, H, V, device, workspace):
    need = workspace_size(N, H, V)
    if need == 0:
        raise FlceError(2, "flce_workspace_size")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    return workspace


def _check_inputs(X, W, labels):
    for name, t, dt in (("hidden", X, torch.bfloat16), ("weight", W, torch.bfloat16),
                        ("labels", labels, torch.int64)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != dt:
            raise ValueError(f"{name} must be {dt}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if X.dim() != 2 or W.dim() != 2 or labels.dim() != 1:
        raise ValueError("expected X [N,H], W [V,H], labels [N]")
    if X.shape[1] != W.shape[1] or labels.shape[0] != X.shape[0]:
        raise ValueError("shape mismatch between X, W and labels")


def flce_forward(X, W, labels, *, seq_len=None, ignore_index=-100, shift=False,
                 reduction="mean", workspace=None):
    """Calls flce_forward; returns (loss [1] f32, lse [N] f32, n_valid [1] i64, workspace)."""
    _check_inputs(X, W, labels)
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    ws = _workspace(N, H, V, dev, workspace)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    n_valid = torch.empty(1, dtype=torch.int64, device=dev)
    st = library().flce_forward(_ptr(X), _ptr(W), _ptr(labels), N, H, V, int(seq_len or 0),
                                int(ignore_index), int(bool(shift)), _REDUCTION[reduction],
                                _ptr(loss), _ptr(lse), _ptr(n_valid), _ptr(ws), ws.numel(),
                                _stream(dev))
    _check(st, "flce_forward")
    return loss, lse, n_valid, ws


def flce_backward(X, W, labels, lse, n_valid, grad_loss, *, seq_len=None, ignore_index=-100,
                  shift=False, reduction="mean", need_dX=True, need_dW=True, workspace=None,
                  dX=None, dW=None):
    """Calls flce_backward; returns (dX or None, dW or None, workspace)."""
    _check_inputs(X, W, labels)
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    ws = _workspace(N, H, V, dev, workspace)
    if need_dX and dX is None:
        dX = torch.empty_like(X)
    if need_dW and dW is None:
        dW = torch.empty_like(W)
    g = grad_loss.to(device=dev, dtype=torch.float32).reshape(1).contiguous()
    st = library().flce_backward(_ptr(X), _ptr(W), _ptr(labels), N, H, V, int(seq_len or 0),
                                 int(ignore_index), int(bool(shift)), _REDUCTION[reduction],
                                 _ptr(lse), _ptr(n_valid), _ptr(g),
                                 _ptr(dX if need_dX else None), _ptr(dW if need_dW else None),
                                 _ptr(ws), ws.numel(), _stream(dev))
    _check(st, "flce_backward")
    return (dX if need_dX else None), (dW if need_dW else None), ws


def flce_backward_accumulate(X, W, labels, lse, n_valid, grad_loss, dW_acc, *, seq_len=None,
                             ignore_index=-100, shift=False, reduction="mean", need_dX=True,
                             workspace=None, dX=None):
    """Calls flce_backward_accumulate: dW_acc (float32 [V, H], modified in place)
    += the weight gradient; returns (dX or None, workspace)."""
    _check_inputs(X, W, labels)
    N, H = X.shape
    V = W.shape[0]
    if dW_acc.dtype != torch.float32 or tuple(dW_acc.shape) != (V, H) or not dW_acc.is_contiguous():
        raise ValueError("dW_acc must be a contiguous float32 [V, H] tensor")
    dev = X.device
    ws = _workspace(N, H, V, dev, workspace)
    if need_dX and dX is None:
        dX = torch.empty_like(X)
    g = grad_loss.to(device=dev, dtype=torch.float32).reshape(1).contiguous()
    lib = library()
    fn = lib.flce_backward_accumulate
    c_i64, c_p, c_int, c_sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    fn.argtypes = [c_p, c_p, c_p, c_i64, c_i64, c_i64, c_i64, c_i64, c_int, c_int,
                   c_p, c_p, c_p, c_p, c_p, c_p, c_sz, c_p]
    fn.restype = c_int
    st = fn(_ptr(X), _ptr(W), _ptr(labels), N, H, V, int(seq_len or 0), int(ignore_index),
            int(bool(shift)), _REDUCTION[reduction], _ptr(lse), _ptr(n_valid), _ptr(g),
            _ptr(dX if need_dX else None), _ptr(dW_acc), _ptr(ws), ws.numel(), _stream(dev))
    _check(st, "flce_backward_accumulate")
    return (dX if need_dX else None), ws


def flce_logits(X, W):
    """Calls flce_logits: bf16 logits [N, V] = X W^T (no labels, no loss)."""
    for name, t in (("hidden", X), ("weight", W)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 2:
            raise ValueError(f"{name} must be a contiguous 2-D bf16 CUDA tensor")
    N, H = X.shape
    V = W.shape[0]
    if W.shape[1] != H:
        raise ValueError("shape mismatch between X and W")
    ld = (V + 7) // 8 * 8
    out = torch.empty(N, ld, dtype=torch.bfloat16, device=X.device)
    lib = library()
    fn = lib.flce_logits
    c_i64, c_p = ctypes.c_int64, ctypes.c_void_p
    fn.argtypes = [c_p, c_p, c_i64, c_i64, c_i64, c_p, c_i64, c_p]
    fn.restype = ctypes.c_int
    _check(fn(_ptr(X), _ptr(W), N, H, V, _ptr(out), ld, _stream(X.device)), "flce_logits")
    return out[:, :V] if ld != V else out


def _fn(name, argtypes):
    fn = getattr(library(), name)
    fn.argtypes = argtypes
    fn.restype = ctypes.c_int
    return fn


_I64, _P, _INT, _SZ = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t


def flce_forward_vocab_shard(X, W_shard, labels, v_offset, V_total, *, seq_len=None,
                             ignore_index=-100, shift=False, workspace=None):
    """Calls flce_forward_vocab_shard for the vocabulary rows W_shard =
    W[v_offset : v_offset + V]; returns (lse_shard [N] f32, z_shard [N] f32,
    n_valid [1] i64, workspace)."""
    _check_inputs(X, W_shard, labels)
    N, H = X.shape
    V = W_shard.shape[0]
    dev = X.device
    ws = _workspace(N, H, V, dev, workspace)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    z = torch.empty(N, dtype=torch.float32, device=dev)
    n_valid = torch.empty(1, dtype=torch.int64, device=dev)
    fn = _fn("flce_forward_vocab_shard", [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I64,
                                          _INT, _P, _P, _P, _P, _SZ, _P])
    st = fn(_ptr(X), _ptr(W_shard), _ptr(labels), N, H, V, int(v_offset), int(V_total),
            int(seq_len or 0), int(ignore_index), int(bool(shift)), _ptr(lse), _ptr(z),
            _ptr(n_valid), _ptr(ws), ws.numel(), _stream(dev))
    _check(st, "flce_forward_vocab_shard")
    return lse, z, n_valid, ws


def flce_merge_vocab_shards(lse_parts, z_parts, labels, V_total, *, seq_len=None,
                            ignore_index=-100, shift=False, reduction="mean", workspace):
    """Calls flce_merge_vocab_shards on the gathered float32 [P, N] shard
    outputs; returns (loss [1] f32, lse [N] f32, n_valid [1] i64)."""
    for name, t in (("lse_parts", lse_parts), ("z_parts", z_parts)):
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous() or t.dim() != 2:
            raise ValueError(f"{name} must be a contiguous float32 [P, N] CUDA tensor")
    if lse_parts.shape != z_parts.shape or labels.shape != (lse_parts.shape[1],):
        raise ValueError("lse_parts, z_parts and labels disagree in shape")
    P, N = lse_parts.shape
    dev = lse_parts.device
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    n_valid = torch.empty(1, dtype=torch.int64, device=dev)
    fn = _fn("flce_merge_vocab_shards", [_P, _P, _I64, _P, _I64, _I64, _I64, _I64, _INT, _INT,
                                         _P, _P, _P, _P, _SZ, _P])
    st = fn(_ptr(lse_parts), _ptr(z_parts), P, _ptr(labels), N, int(V_total), int(seq_len or 0),
            int(ignore_index), int(bool(shift)), _REDUCTION[reduction], _ptr(loss), _ptr(lse),
            _ptr(n_valid), _ptr(workspace), workspace.numel(), _stream(dev))
    _check(st, "flce_merge_vocab_shards")
    return loss, lse, n_valid


def flce_backward_vocab_shard(X, W_shard, labels, v_offset, V_total, lse, n_valid, grad_loss,
                              dX_acc=None, *, seq_len=None, ignore_index=-100, shift=False,
                              reduction="mean", need_dW=True, workspace=None, dW=None):
    """Calls flce_backward_vocab_shard: dX_acc (float32 [N, H] or None, modified
    in place) += this shard's part of dX; returns (dW_shard or None, workspace)."""
    _check_inputs(X, W_shard, labels)
    N, H = X.shape
    V = W_shard.shape[0]
    if dX_acc is not None and (dX_acc.dtype != torch.float32 or tuple(dX_acc.shape) != (N, H)
                               or not dX_acc.is_contiguous()):
        raise ValueError("dX_acc must be a contiguous float32 [N, H] tensor")
    dev = X.device
    ws = _workspace(N, H, V, dev, workspace)
    if need_dW and dW is None:
        dW = torch.empty_like(W_shard)
    g = grad_loss.to(device=dev, dtype=torch.float32).reshape(1).contiguous()
    fn = _fn("flce_backward_vocab_shard", [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I64,
                                           _INT, _INT, _P, _P, _P, _P, _P, _P, _SZ, _P])
    st = fn(_ptr(X), _ptr(W_shard), _ptr(labels), N, H, V, int(v_offset), int(V_total),
            int(seq_len or 0), int(ignore_index), int(bool(shift)), _REDUCTION[reduction],
            _ptr(lse), _ptr(n_valid), _ptr(g), _ptr(dX_acc), _ptr(dW if need_dW else None),
            _ptr(ws), ws.numel(), _stream(dev))
    _check(st, "flce_backward_vocab_shard")
    return (dW if need_dW else None), ws


def flce_downcast_bf16(src, out=None):
    """Calls flce_downcast_bf16: a bf16 copy of a float32 CUDA tensor (numel a
    multiple of 8)."""
    if not src.is_cuda or src.dtype != torch.float32 or not src.is_contiguous():
        raise ValueError("src must be a contiguous float32 CUDA tensor")
    if out is None:
        out = torch.empty(src.shape, dtype=torch.bfloat16, device=src.device)
    fn = _fn("flce_downcast_bf16", [_P, _P, _I64, _P])
    _check(fn(_ptr(src), _ptr(out), src.numel(), _stream(src.device)), "flce_downcast_bf16")
    return out


def flce_get_error(workspace) -> int:
    """Synchronises the current stream and returns the workspace's error status."""
    return int(library().flce_get_error(_ptr(workspace), _stream(workspace.device)))


def flce_set_wait_limit_ns(limit_ns: int) -> None:
    library().flce_set_wait_limit_ns(int(limit_ns))


def flce_set_backward_block(max_rows: int = 0, max_block_elems: int = 0) -> None:
    """Caps the backward's dZ block (0 restores the defaults); see include/flce.h."""
    library().flce_set_backward_block(int(max_rows), int(max_block_elems))


def flce_backward_blocking(N: int, H: int, V: int) -> tuple[int, int]:
    """The backward's dZ block (token rows, vocab columns) for these sizes."""
    nb, vb = ctypes.c_int64(), ctypes.c_int64()
    _check(library().flce_backward_blocking(int(N), int(H), int(V), ctypes.byref(nb),
                                            ctypes.byref(vb)), "flce_backward_blocking")
    return nb.value, vb.value


def flce_kernel_launch_count() -> int:
    return int(library().flce_kernel_launch_count())


def flce_last_launch_wait_limit_ns() -> int:
    """The wait limit (ns) the most recent tensor-core launch was given."""
    fn = library().flce_last_launch_wait_limit_ns
    fn.argtypes = []
    fn.restype = ctypes.c_int64
    return int(fn())


def flce_profile_enable(enable: bool) -> None:
    library().flce_profile_enable(int(bool(enable)))


PROFILE_KINDS = ("forward", "backward")


def flce_profile_collect() -> dict:
    """{kind: (total_ms, launches)} of the tensor-core launches recorded since
    profiling was enabled or last collected; waits for them to finish."""
    ms = (ctypes.c_double * 4)()
    n = (ctypes.c_int64 * 4)()
    _check(library().flce_profile_collect(ctypes.cast(ms, ctypes.c_void_p),
                                          ctypes.cast(n, ctypes.c_void_p)),
           "flce_profile_collect")
    return {k: (ms[i], int(n[i])) for i, k in enumerate(PROFILE_KINDS)}


def flce_selftest_wait_timeout(limit_ns: int, workspace) -> int:
    return int(library().flce_selftest_wait_timeout(int(limit_ns), _ptr(workspace),
                                                    workspace.numel(),
                                                    _stream(workspace.device)))


def flce_forward_noalloc(X, W, labels, *, seq_len=None, ignore_index=-100, shift=False,
                         reduction="mean"):
    """flce_forward without a workspace (C entry point flce_forward_noalloc).

    For callers that cannot allocate device memory: the library keeps a fixed
    16 MiB scratch array in its device image and uses it instead (problems
    needing more are refused with FLCE_ERR_WORKSPACE_TOO_SMALL).  Returns
    (loss [1] f32, lse [N] f32, n_valid [1] i64, device_error [1] i32).  Calls
    share the scratch; serialise calls that could overlap on the GPU.
    """
    _check_inputs(X, W, labels)
    lib = library()
    fn = lib.flce_forward_noalloc
    c_i64, c_p, c_int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [c_p, c_p, c_p, c_i64, c_i64, c_i64, c_i64, c_i64, c_int, c_int,
                   c_p, c_p, c_p, c_p, c_p]
    fn.restype = c_int
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    n_valid = torch.empty(1, dtype=torch.int64, device=dev)
    derr = torch.empty(1, dtype=torch.int32, device=dev)
    st = fn(_ptr(X), _ptr(W), _ptr(labels), N, H, V, int(seq_len or 0), int(ignore_index),
            int(bool(shift)), _REDUCTION[reduction], _ptr(loss), _ptr(lse), _ptr(n_valid),
            _ptr(derr), _stream(dev))
    _check(st, "flce_forward_noalloc")
    return loss, lse, n_valid, derr


class _FusedLinearCE(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, W, labels, seq_len, ignore_index, shift, reduction):
        loss, lse, n_valid, _ = flce_forward(X, W, labels, seq_len=seq_len,
                                             ignore_index=ignore_index, shift=shift,
                                             reduction=reduction)
        ctx.save_for_backward(X, W, labels, lse, n_valid)
        ctx.cfg = (seq_len, ignore_index, shift, reduction)
        return loss.reshape(())

    @staticmethod
    def backward(ctx, grad):
        X, W, labels, lse, n_valid = ctx.saved_tensors
        seq_len, ignore_index, shift, reduction = ctx.cfg
        dX, dW, _ = flce_backward(X, W, labels, lse, n_valid, grad.detach(), seq_len=seq_len,
                                  ignore_index=ignore_index, shift=shift, reduction=reduction,
                                  need_dX=ctx.needs_input_grad[0],
                                  need_dW=ctx.needs_input_grad[1])
        return dX, dW, None, None, None, None, None


def linear_cross_entropy(hidden, weight, labels, ignore_index=-100, shift=False,
                         reduction="mean", seq_len=None):
    """Cross-entropy of hidden @ weight.T against labels, without the logits.

    hidden: bf16 [B, S, H] or [N, H]; weight: bf16 [V, H]; labels: int64 [B, S]
    or [N].  With shift=True, position s of each sequence is scored against
    labels[s+1] and the last position is ignored (for 3-D hidden the sequence
    length is S; for 2-D, seq_len or one sequence).  Returns a 0-dim float32
    loss that back-propagates to hidden and weight.  With labels=None it
    returns the bf16 logits hidden @ weight.T instead (no gradient).
    """
    if labels is None:
        # no labels: the plain LM head (inference); returns bf16 logits
        lead = hidden.shape[:-1]
        Z = flce_logits(hidden.reshape(-1, hidden.shape[-1]).contiguous(), weight.contiguous())
        return Z.reshape(*lead, weight.shape[0])
    if reduction not in _REDUCTION:
        raise ValueError(f"reduction must be 'mean' or 'sum', got {reduction!r}")
    if hidden.dim() == 3:
        B, S, H = hidden.shape
        seq_len = S
        hidden = hidden.reshape(B * S, H)
        labels = labels.reshape(B * S)
    return _FusedLinearCE.apply(hidden.contiguous(), weight.contiguous(), labels.contiguous(),
                                seq_len, ignore_index, shift, reduction)
