"""Peak extra device memory of a forward + backward through the autograd call,
at every workload's full size.

The library allocates nothing: its only scratch is the workspace the binding
takes from torch's allocator.  So the peak of the bytes requested from torch's
allocator during the step, minus the inputs and the outputs (loss, lse,
n_valid, dX, dW) and the 4-byte upstream gradient, is the workspace and nothing
more; the device's free memory moves only by what torch itself reserved; and
the workspace stays within its documented bound (FP32 dX, at most one FP32 dW
band, two bounded dZ blocks, at most 128 partials per row) -- far below the
N x V logits the method avoids.

Requested bytes, not allocated bytes: the caching allocator hands out a cached
block whole when the leftover would be under its 1 MiB split threshold, so
each large block (workspace, dX, dW) may count up to 1 MiB more than was asked
for in the allocated-bytes statistics.
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

flce = pytest.importorskip("lm_head_linear_flce_gb300")

MiB = 1 << 20


def documented_bound(N, H, V):
    """Upper bound of flce_workspace_size from the layout in include/flce.h:
    FP32 dX [N][H]; an FP32 dW band of at most 2^27 / 256 vocab rows; two dZ
    blocks of at most 2^27 bf16 elements plus 64 padding columns per row; 128
    (max, sum-exp) pairs per row; 16 bytes per row of targets and dense-row
    maps; 1 MiB of counters and flags."""
    return (4 * N * H + 4 * H * min(V, (1 << 27) // 256) + 2 * 2 * ((1 << 27) + 64 * N)
            + 8 * 128 * N + 16 * N + MiB)


def device_inputs(wl):
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(wl.seed)
    X = (torch.randn(wl.N, wl.H, device=dev, generator=g) * wl.x_std).to(torch.bfloat16)
    W = (torch.randn(wl.V, wl.H, device=dev, generator=g) * wl.w_std).to(torch.bfloat16)
    L = torch.randint(0, wl.V, (wl.N,), device=dev, generator=g)
    L[torch.rand(wl.N, device=dev, generator=g) < wl.mask_frac] = -100
    return X, W, L


@pytest.mark.parametrize("name", [w.name for w in workloads.WORKLOADS])
def test_peak_extra_memory_is_the_workspace(name):
    wl = workloads.get(name)
    N, H, V = wl.N, wl.H, wl.V
    X, W, L = device_inputs(wl)
    kw = dict(shift=wl.shift, reduction=wl.reduction, seq_len=wl.S)

    def step():
        xg = X.detach().requires_grad_(True)
        wg = W.detach().requires_grad_(True)
        loss = flce.linear_cross_entropy(xg, wg, L, **kw)
        loss.backward()
        return loss, xg, wg

    step()  # loads the kernels; torch's allocator keeps its caches
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_stats()["requested_bytes.all.current"]
    base_alloc = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    loss, xg, wg = step()
    torch.cuda.synchronize()
    peak = torch.cuda.memory_stats()["requested_bytes.all.peak"] - base
    peak_alloc = torch.cuda.max_memory_allocated() - base_alloc
    free1, _ = torch.cuda.mem_get_info()
    reserved1 = torch.cuda.memory_reserved()
    assert torch.isfinite(loss).item()

    # dX, dW, lse, loss, n_valid, and the upstream gradient of the scalar loss
    outputs = X.numel() * 2 + W.numel() * 2 + N * 4 + 4 + 8 + 4
    ws = flce.workspace_size(N, H, V)
    extra = peak - outputs
    print(f"\n{name}: peak extra {extra} B (workspace {ws} B = {ws / MiB:.1f} MiB, "
          f"bf16 logits {N * V * 2 / MiB:.0f} MiB)")
    # exactly the workspace: nothing else is requested while it is live
    assert extra == ws, (extra, ws)
    # the allocated-bytes view: up to 1 MiB of block rounding for each of the
    # three large blocks, and 512-byte rounding of the small ones
    assert ws <= peak_alloc - outputs <= ws + 3 * MiB + 4 * 512, (peak_alloc - outputs, ws)
    assert ws <= documented_bound(N, H, V), (ws, documented_bound(N, H, V))
    # nothing outside torch's allocator: free memory moved only by torch's
    # reserve (up to the CUDA driver's own bookkeeping for new mappings)
    assert abs((free0 - free1) - (reserved1 - reserved0)) <= 8 * MiB, (free0 - free1,
                                                                       reserved1 - reserved0)
    if N * V >= 1 << 30:  # the Qwen-sized workloads: far below the logits
        assert ws < 0.15 * N * V * 2, (ws, N * V * 2)
