"""Throughput of the fused linear cross-entropy (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload qwen2_7b]
                    [--impl ours|reference]

One step is flce_forward + flce_backward (loss, lse, n_valid, dX, dW) over one
batch of the workload, inputs resident in HBM.  The workload's weight matrix
alone (V x H bf16, >= 1 GB) is larger than the 129 MB L2, so no flush is
needed between steps.  Prints one JSON line (rank 0).

--impl reference times the CPU float64 oracle on the host cores instead (a
bounded sample of rows per step), reported in the same metric and unit.

With several ranks (torchrun) every rank runs its own replica of the workload
on its own GPU ("replicas only": the method has no exchange step here); value
is the tokens of all ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "fused linear-CE fwd+bwd tokens/s and TFLOP/s (% bf16 peak), peak extra HBM"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic_qwen2_7b.md")
KERNEL_SOURCES = [os.path.join(ROOT, "lm_head_linear_flce_gb300", "csrc", f)
                  for f in ("flce_gemm.cu", "flce_api.cu", "flce_device.cuh", "flce_internal.h")]
# Dense bf16 tensor-core rate of one SM per clock: 4096 FMAs (8192 FLOPs).  At
# this rate the 152-SM GB300 reaches its nominal 2.25 PFLOP/s dense bf16 at
# about 1.81 GHz, and the measured sustained cuBLAS figure (1754.5 TFLOP/s at a
# median 1507 MHz) is 0.935 of it -- a library GEMM cannot exceed it.
BF16_FLOP_PER_CLK_PER_SM = 8192


def _code_only(text: str) -> str:
    """C++ source with comments and blank or trailing space removed (the sources
    hold no string literal containing a comment marker)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_digest() -> str:
    """sha256 (first 16 hex) of the kernel and launch sources, comments aside."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def load_traffic(workload: str, kind: str):
    """DRAM bytes per launch of `kind` from the committed ncu capture, or None
    when the capture is for another workload or the kernel sources changed."""
    try:
        with open(TRAFFIC_FILE) as f:
            text = f.read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        line = line.strip().strip("`")
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("workload") != workload or vals.get("sources") != kernel_source_digest():
        return None
    try:
        return int(float(vals[f"{kind}_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def reduce_max(x: float, world: int, device) -> float:
    """Maximum of x over all ranks (identity for one rank)."""
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(tokens_per_step: int, steps: int, elapsed_ms_local: float, world: int,
                         device) -> tuple[float, float]:
    """(value, max elapsed ms): tokens of all ranks over the slowest rank's time."""
    worst = reduce_max(elapsed_ms_local, world, device)
    return world * tokens_per_step * steps / (worst / 1e3), worst


class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons, kept only
    while the timed region runs (each sample carries nvidia-smi's timestamp;
    `window(t0, t1)` gives the host-clock bounds of the region)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "-i", str(self.gpu),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def window(self, t0: float, t1: float):
        self.t0, self.t1 = t0, t1

    @staticmethod
    def _when(stamp: str):
        import datetime
        try:
            return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((self._when(parts[0]), float(parts[1]), float(parts[2]),
                             float(parts[3]), parts[4:8]))
            except ValueError:
                continue
        if self.t0 is not None:
            inside = [r for r in rows if r[0] is not None and self.t0 <= r[0] <= self.t1]
            if not inside:  # a region shorter than the sampling period: nearest samples
                inside = [r for r in rows
                          if r[0] is not None and self.t0 - 0.1 <= r[0] <= self.t1 + 0.1]
            rows = inside
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for name, v in zip(self.NAMES, r[4]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in rows),
                "sm_min_mhz": min(r[1] for r in rows),
                "sm_max_mhz": max(r[2] for r in rows),
                "power_w": round(statistics.median(r[3] for r in rows), 1),
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import lm_head_linear_flce_gb300 as flce

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = workloads.get(args.workload)
    if args.tokens or args.vocab:
        # a reduced case of the same workload (profiling captures)
        import dataclasses
        n = args.tokens or wl.N
        wl = dataclasses.replace(wl, name=f"{wl.name}_N{n}_V{args.vocab or wl.V}", B=1, S=n,
                                 V=args.vocab or wl.V)
    N, H, V = wl.N, wl.H, wl.V
    Xh, Wh, Lh = workloads.make_inputs(wl)
    Xh, Wh, Lh = Xh.pin_memory(), Wh.pin_memory(), Lh.pin_memory()
    X, W, L = Xh.to(dev), Wh.to(dev), Lh.to(dev)
    kw = dict(seq_len=wl.S, shift=wl.shift, reduction=wl.reduction)
    grad = torch.ones(1, dtype=torch.float32, device=dev)
    dX = torch.empty_like(X)
    dW = torch.empty_like(W)
    ws = torch.empty(flce.workspace_size(N, H, V), dtype=torch.uint8, device=dev)

    def step():
        loss, lse, nv, _ = flce.flce_forward(X, W, L, workspace=ws, **kw)
        flce.flce_backward(X, W, L, lse, nv, grad, workspace=ws, dX=dX, dW=dW, **kw)
        return loss

    # peak extra device memory of one step: everything beyond inputs and outputs
    torch.cuda.synchronize()
    del ws
    torch.cuda.empty_cache()
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    ws = torch.empty(flce.workspace_size(N, H, V), dtype=torch.uint8, device=dev)
    loss = step()
    torch.cuda.synchronize()
    out_bytes = 4 + N * 4 + 8  # loss, lse, n_valid (dX, dW were allocated before `base`)
    extra = torch.cuda.max_memory_allocated(dev) - base - out_bytes

    for _ in range(args.warmup):
        step()
    if flce.flce_get_error(ws) != 0:
        raise RuntimeError(f"device error after warm-up: {flce.STATUS[flce.flce_get_error(ws)]}")

    stream = torch.cuda.current_stream(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    flce.flce_profile_collect()
    flce.flce_profile_enable(True)
    n0 = flce.flce_kernel_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    h0 = time.time()
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    clocks.window(h0, time.time())
    barrier(world)
    clk = clocks.stop()
    launches = flce.flce_kernel_launch_count() - n0
    flce.flce_profile_enable(False)
    prof = flce.flce_profile_collect()
    status = flce.flce_get_error(ws)
    if status != 0:
        raise RuntimeError(f"device error in timed region: {flce.STATUS[status]}")
    elapsed = t0.elapsed_time(t1)
    value, worst = aggregate_throughput(N, args.steps, elapsed, world, dev)
    ms_step = worst / args.steps

    # End to end through the public autograd call.  Every step copies its inputs
    # from pinned host memory and reads the loss back; the copy of step i+1 runs
    # on a second stream while step i computes (double-buffered device inputs),
    # as a training loop that prefetches its next batch would.
    e2e = None
    if not args.no_e2e:
        del ws
        torch.cuda.empty_cache()
        bufs = [(torch.empty_like(X), torch.empty_like(W), torch.empty_like(L)) for _ in range(2)]
        loss_h = torch.empty(max(1, args.steps), dtype=torch.float32).pin_memory()
        copy_stream = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]
        # the same K steps as the device-timed region; the first step's copy,
        # which nothing before it can hide, is inside the timed region
        e_steps = max(1, args.steps)

        def issue_copy(i):
            b = i % 2
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(consumed[b])
                for d, h in zip(bufs[b], (Xh, Wh, Lh)):
                    d.copy_(h, non_blocking=True)
                copied[b].record(copy_stream)

        def e2e_run(n):
            for b in range(2):
                consumed[b].record(stream)
            issue_copy(0)
            for i in range(n):
                b = i % 2
                stream.wait_event(copied[b])
                if i + 1 < n:
                    issue_copy(i + 1)
                Xd, Wd, Ld = bufs[b]
                xg = Xd.detach().requires_grad_(True)
                wg = Wd.detach().requires_grad_(True)
                lo = flce.linear_cross_entropy(xg, wg, Ld, shift=wl.shift,
                                               reduction=wl.reduction, seq_len=wl.S)
                lo.backward()
                loss_h[i].copy_(lo.detach(), non_blocking=True)
                consumed[b].record(stream)

        e2e_run(2)
        torch.cuda.synchronize()
        barrier(world)
        e_clocks = ClockSampler(local)  # the clock this later region ran at
        e_clocks.start()
        time.sleep(0.3)
        eh0 = time.time()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(e_steps)
        e1.record(stream)
        torch.cuda.synchronize()
        e_clocks.window(eh0, time.time())
        e_clk = e_clocks.stop()
        e_val, _ = aggregate_throughput(N, e_steps, e0.elapsed_time(e1), world, dev)
        h2d = X.numel() * 2 + W.numel() * 2 + L.numel() * 8
        e2e = {"value": round(e_val, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": 4, "steps": e_steps,
               "api": "lm_head_linear_flce_gb300.linear_cross_entropy + backward",
               "copies": "inputs of step i+1 copied on a second stream during step i",
               "clocks": e_clk}

    peaks, src = load_peaks()
    flops = wl.flops
    # FLOPs actually executed per step (reported beside the algorithmic
    # 8*N*H*V, and the basis of the backward's roofline)
    active_rows = backward_rows(wl, Lh)
    exec_flops = 2 * N * H * V + 6 * active_rows * H * V
    tflops = flops / (ms_step / 1e3) / 1e12 * 1.0
    tflops_all = world * tflops
    # dominant tensor-core kernel of the step: forward launch (2NHV) or the
    # backward launches (recompute + dX + dW: 6 x H x V per row they run on)
    kind_flops = {"forward": 2 * N * H * V, "backward": 6 * active_rows * H * V}
    kinds = {k: v for k, v in prof.items() if v[1] > 0}
    dom = max(kinds, key=lambda k: kinds[k][0])
    dom_ms, dom_n = kinds[dom]
    achieved = kind_flops[dom] * args.steps / (dom_ms / 1e3) / 1e12
    burst, sustained = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # the dense rate at the SM clock sampled inside the timed region
    clock_peak = (sms * BF16_FLOP_PER_CLK_PER_SM * clk["sm_mhz"] * 1e6 / 1e12
                  if clk and clk.get("sm_mhz") else None)
    step_ms_total = sum(v[0] for v in kinds.values())
    roofline = {
        "kernel": dom, "bound": "tensor", "achieved": round(achieved, 1), "peak": burst,
        "unit": "TFLOP/s", "frac": round(achieved / burst, 4),
        "traffic": load_traffic(wl.name, dom),
        "peak_source": f"bf16_tflops, burst cuBLAS GEMM ({src})",
        "frac_burst": round(achieved / burst, 4),
        "frac_sustained": round(achieved / sustained, 4),
        "sustained_peak": sustained,
        "sustained_peak_source": f"bf16_tflops_sustained, cuBLAS GEMM looped for seconds ({src})",
        "frac_per_clock": round(achieved / clock_peak, 4) if clock_peak else None,
        "per_clock_peak": round(clock_peak, 1) if clock_peak else None,
        "per_clock_peak_basis": (f"{sms} SMs x {BF16_FLOP_PER_CLK_PER_SM} bf16 FLOP/clk/SM x "
                                 "median SM MHz sampled in the timed region"),
        "launches_per_step": dom_n / args.steps,
        "avg_launch_ms": dom_ms / dom_n,
        "flops_per_launch": kind_flops[dom] * args.steps / dom_n,
        "flops_basis": ("forward: 2*N*H*V; backward: 6*H*V per row it runs on "
                        f"({active_rows} of N={N}: the rows with a valid target, in 256-row tiles)"),
        "share_of_step": round(dom_ms / (ms_step * args.steps), 4),
        "per_kind_ms_per_step": {k: round(v[0] / args.steps, 3) for k, v in kinds.items()},
        "per_kind_tflops": {k: round(kind_flops[k] * args.steps / (v[0] / 1e3) / 1e12, 1)
                            for k, v in kinds.items()},
        "tensor_kernels_ms_per_step": round(step_ms_total / args.steps, 3),
    }

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, Xh, Wh, Lh, rows=args.cpu_rows)

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "N": N, "H": H, "V": V, "B": wl.B, "seq_len": wl.S,
                   "shift": wl.shift, "reduction": wl.reduction,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2 (W is %.2f GB); no flush" % (V * H * 2 / 1e9)},
        "tflops": round(tflops_all, 1),
        "executed_tflops": round(world * exec_flops / (ms_step / 1e3) / 1e12, 1),
        "executed_flops_per_step": exec_flops,
        "pct_bf16_peak": round(100 * tflops / burst, 2),
        "pct_bf16_peak_basis": f"bf16_tflops (burst) {burst} ({src}), 8*N*H*V per step",
        "pct_bf16_peak_sustained": round(100 * tflops / sustained, 2),
        "pct_bf16_peak_per_clock": round(100 * tflops / clock_peak, 2) if clock_peak else None,
        "peak_extra_hbm_bytes": int(extra),
        "logits_bytes_avoided": {"bf16": N * V * 2, "fp32": N * V * 4},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clk,
        "loss": float(loss.item()),
    }
    if rank == 0:
        print(json.dumps(result), flush=True)


# ---------------------------------------------------------------- CPU oracle
def cpu_baseline(wl, X, W, L, rows: int):
    """The float64 oracle, as it stands, on the host cores: forward + backward of
    `rows` token rows of the workload (their full vocabulary of logits, their dX
    rows and their contribution to dW)."""
    import numpy as np

    import oracle
    t, valid, n_valid, _ = oracle.effective_targets(L, wl.V, seq_len=wl.S, shift=wl.shift)
    idx = np.arange(rows) * max(1, wl.N // rows)
    tgt = torch.tensor(np.where(valid[idx], t[idx], -100))
    Xs = X[torch.as_tensor(idx)]
    t0 = time.perf_counter()
    f = oracle.forward(Xs, W, tgt, reduction=wl.reduction)
    oracle.backward(Xs, W, tgt, reduction="sum",
                    grad_loss=(1.0 / n_valid if wl.reduction == "mean" else 1.0), lse=f["lse"])
    dt = time.perf_counter() - t0
    return {"value": round(rows / dt, 3), "unit": "tokens/s", "cores": os.cpu_count(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"{rows} token rows of {wl.name} (every {max(1, wl.N // rows)}th), "
                      "float64 forward + backward incl. their dW contribution"}


# ------------------------------------------------- the other rows of the path
ROWS = ("main", "dx_only", "accumulate", "logits", "vocab_shard4", "phases")


def run_row(args, world, rank, local):
    """One of the path's other entry points on the workload, timed like the
    main step: dx_only (forward + backward without dW), accumulate (forward +
    backward adding dW into an FP32 gradient), logits (plain bf16 logits, no
    labels), vocab_shard4 (one rank of a four-way vocabulary split: shard
    forward, merge, shard backward into an FP32 dX buffer; the all-gather and
    all-reduce of a real group are not part of one GPU's step)."""
    import lm_head_linear_flce_gb300 as flce

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = workloads.get(args.workload)
    N, H, V = wl.N, wl.H, wl.V
    X, W, L = (t.to(dev) for t in workloads.make_inputs(wl))
    kw = dict(seq_len=wl.S, shift=wl.shift, reduction=wl.reduction)
    g = torch.ones(1, dtype=torch.float32, device=dev)
    if args.row == "vocab_shard4":
        from lm_head_linear_flce_gb300.vocab_parallel import vocab_shard_bounds
        v0, Vr = vocab_shard_bounds(V, 4)[0]
        Wr = W[v0:v0 + Vr].contiguous()
        del W
        ws = torch.empty(flce.workspace_size(N, H, Vr), dtype=torch.uint8, device=dev)
        dX_acc = torch.empty(N, H, dtype=torch.float32, device=dev)
        dWr = torch.empty_like(Wr)
        flops = 8 * N * H * Vr

        def step():
            lse_r, z_r, _, _ = flce.flce_forward_vocab_shard(X, Wr, L, v0, V, workspace=ws,
                                                             seq_len=wl.S, shift=wl.shift)
            # the gathered rows of four ranks (this rank's, four times: same cost)
            loss, lse, nv = flce.flce_merge_vocab_shards(
                lse_r.expand(4, N).contiguous(), z_r.expand(4, N).contiguous(), L, V,
                workspace=ws, **kw)
            dX_acc.zero_()
            flce.flce_backward_vocab_shard(X, Wr, L, v0, V, lse, nv, g, dX_acc, workspace=ws,
                                           dW=dWr, **kw)
    else:
        ws = torch.empty(flce.workspace_size(N, H, V), dtype=torch.uint8, device=dev)
        dX = torch.empty_like(X)
        rows = backward_rows(wl, L.cpu())  # the backward runs on these rows only
        if args.row == "dx_only":
            flops = 2 * N * H * V + 4 * rows * H * V

            def step():
                _, lse, nv, _ = flce.flce_forward(X, W, L, workspace=ws, **kw)
                flce.flce_backward(X, W, L, lse, nv, g, workspace=ws, dX=dX, need_dW=False, **kw)
        elif args.row == "accumulate":
            flops = 2 * N * H * V + 6 * rows * H * V
            dW_acc = torch.zeros(V, H, dtype=torch.float32, device=dev)

            def step():
                _, lse, nv, _ = flce.flce_forward(X, W, L, workspace=ws, **kw)
                flce.flce_backward_accumulate(X, W, L, lse, nv, g, dW_acc, workspace=ws, dX=dX,
                                              **kw)
        else:  # logits
            flops = 2 * N * H * V
            del ws

            def step():
                flce.flce_logits(X, W)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = flce.flce_kernel_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    launches = flce.flce_kernel_launch_count() - n0
    value, worst = aggregate_throughput(N, args.steps, t0.elapsed_time(t1), world, dev)
    ms_step = worst / args.steps
    peaks, src = load_peaks()
    tfl = flops / (ms_step / 1e3) / 1e12
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "row": args.row, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "N": N, "H": H, "V": V, "row": args.row},
            "roofline": {"kernel": "step", "bound": "tensor", "achieved": round(tfl, 1),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(tfl / peaks["bf16_tflops"], 4),
                         "frac_sustained": round(tfl / peaks["bf16_tflops_sustained"], 4),
                         "traffic": None, "flops_per_step": flops,
                         "peak_source": f"bf16_tflops, burst ({src})"},
            **({"exchange": "unmeasured (no multi-GPU run): the all-gather of 2*N floats "
                            "per rank and the FP32 all-reduce of N*H*4 bytes that a real "
                            "group adds are not in this step"}
               if args.row == "vocab_shard4" else {}),
            "gpu_launches": launches}), flush=True)


def backward_rows(wl, labels):
    """Rows the backward runs on: those with a valid target, gathered into dense
    256-row tiles when V spans several dZ blocks (a backward with dX), else
    the 256-row token tiles that hold one (include/flce.h, flce_backward)."""
    import lm_head_linear_flce_gb300 as flce
    N, H, V = wl.N, wl.H, wl.V
    tgt = torch.full((N,), -100, dtype=torch.int64)
    if wl.shift:
        lab = labels.view(-1, wl.S)
        tgt.view(-1, wl.S)[:, :-1] = lab[:, 1:]
    else:
        tgt.copy_(labels)
    has = (tgt != -100).view(-1)
    _, Vb = flce.flce_backward_blocking(N, H, V)
    if V > Vb:
        return min(N, -(-int(has.sum()) // 256) * 256)
    pad = (-N) % 256
    tiles = torch.cat([has, torch.zeros(pad, dtype=torch.bool)]).view(-1, 256).any(1)
    return min(N, int(tiles.sum()) * 256)


def run_phases(args, world, rank, local):
    """Steady state of each kernel alone: the forward looped for --seconds, then
    the backward, then a cuBLAS bf16 8192^3 GEMM (torch.matmul, the pool's
    measured-peak method) as the reference, twice each, with the SM clock and
    board power sampled during each loop.  At the board's power limit this
    compares the kernels with cuBLAS on the same GPU at the same moment."""
    import lm_head_linear_flce_gb300 as flce

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = workloads.get(args.workload)
    N, H, V = wl.N, wl.H, wl.V
    X, W, L = (t.to(dev) for t in workloads.make_inputs(wl))
    kw = dict(seq_len=wl.S, shift=wl.shift, reduction=wl.reduction)
    g = torch.ones(1, dtype=torch.float32, device=dev)
    ws = torch.empty(flce.workspace_size(N, H, V), dtype=torch.uint8, device=dev)
    dX, dW = torch.empty_like(X), torch.empty_like(W)
    _, lse, nv, _ = flce.flce_forward(X, W, L, workspace=ws, **kw)
    lse, nv = lse.clone(), nv.clone()
    A = torch.randn(8192, 8192, device=dev).to(torch.bfloat16)
    B = torch.randn(8192, 8192, device=dev).to(torch.bfloat16)
    C = torch.empty(8192, 8192, device=dev, dtype=torch.bfloat16)
    phases = {
        "forward": (lambda: flce.flce_forward(X, W, L, workspace=ws, **kw), 2 * N * H * V),
        "backward": (lambda: flce.flce_backward(X, W, L, lse, nv, g, workspace=ws, dX=dX, dW=dW,
                                                **kw), 6 * backward_rows(wl, L.cpu()) * H * V),
        "cublas_bf16_gemm": (lambda: torch.matmul(A, B, out=C), 2 * 8192 ** 3),
    }
    for fn, _ in phases.values():
        for _ in range(args.warmup):
            fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    out = {}
    for rnd in range(2):
        for name, (fn, flops) in phases.items():
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            n = max(3, int(args.seconds * 1e3 / e0.elapsed_time(e1)))
            clocks = ClockSampler(local)
            clocks.start()
            time.sleep(0.3)
            h0 = time.time()
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            h1 = time.time()
            # the second half of the loop (after the power controller settled)
            clocks.window(0.5 * (h0 + h1), h1)
            clk = clocks.stop()
            ms = e0.elapsed_time(e1) / n
            tfl = flops / (ms / 1e3) / 1e12
            rec = {"ms": round(ms, 4), "tflops": round(tfl, 1), "clocks": clk}
            if clk and clk.get("sm_mhz"):
                sms = torch.cuda.get_device_properties(dev).multi_processor_count
                rec["per_clock"] = round(tfl * 1e12 / (sms * BF16_FLOP_PER_CLK_PER_SM *
                                                       clk["sm_mhz"] * 1e6), 4)
                rec["watts_per_tflops"] = round(clk["power_w"] / tfl, 4)
            out.setdefault(name, []).append(rec)
    best = {k: max(v, key=lambda r: r["tflops"]) for k, v in out.items()}
    ref = best["cublas_bf16_gemm"]["tflops"]
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "row": "phases", "unit": "TFLOP/s", "workload": wl.name,
            "seconds_per_loop": args.seconds, "phases": out,
            "vs_cublas_same_run": {k: round(v["tflops"] / ref, 4) for k, v in best.items()},
            "dtype": "bf16", "data": "synthetic"}), flush=True)


def run_reference(args, world, rank):
    if rank != 0:
        return
    wl = workloads.get(args.workload)
    X, W, L = workloads.make_inputs(wl)
    rows = args.ref_rows
    for _ in range(args.warmup):
        cpu_baseline(wl, X, W, L, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cb = cpu_baseline(wl, X, W, L, rows)
    dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    res = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * dt / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "N": wl.N, "H": wl.H, "V": wl.V, "B": wl.B,
                   "seq_len": wl.S, "shift": wl.shift, "reduction": wl.reduction,
                   "parallelism": "single"},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": cb["sample"]},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--workload", default="qwen2_7b", choices=sorted(workloads.BY_NAME))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-rows", type=int, default=1024)
    p.add_argument("--ref-rows", type=int, default=8)
    p.add_argument("--tokens", type=int, default=0, help="override N (profiling cases)")
    p.add_argument("--vocab", type=int, default=0, help="override V (profiling cases)")
    p.add_argument("--seconds", type=float, default=3.0,
                   help="--row phases: length of each kernel's steady-state loop")
    p.add_argument("--row", default="main", choices=ROWS,
                   help="main: the fused forward + backward step; phases: each kernel's "
                        "steady state beside a cuBLAS GEMM; the others time the path's other "
                        "entry points")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        elif args.row == "phases":
            run_phases(args, world, rank, local)
        elif args.row != "main":
            run_row(args, world, rank, local)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1 and torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
