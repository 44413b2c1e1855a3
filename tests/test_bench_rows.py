"""The rows the backward runs on, as bench.py counts them for the executed
FLOPs and the backward's roofline, against a direct count from each
workload's labels (include/flce.h, flce_backward: with dX and several vocab
blocks, the rows with a valid target gathered into dense 256-row tiles;
otherwise the 256-row token tiles that hold one).  The labels are drawn with
H = 8 (the workload's own label distribution, a lighter draw); the blocking
is queried at the workload's real sizes."""
import math

import pytest
import torch

import bench
import workloads

flce = pytest.importorskip("lm_head_linear_flce_gb300")


def targets(wl, labels):
    t = labels.clone()
    if wl.shift:
        t = t.view(-1, wl.S)
        t = torch.cat([t[:, 1:], torch.full((t.shape[0], 1), -100)], dim=1).reshape(-1)
    return t


@pytest.mark.parametrize("name,dense", [("qwen2_7b", True), ("qwen3_8b", True),
                                        ("long_ctx", True), ("stress", True), ("tiny", False)])
def test_rows_the_backward_runs_on(name, dense):
    wl = workloads.get(name)
    _, _, labels = workloads.make_inputs(wl, H=8)
    got = bench.backward_rows(wl, labels)
    valid = targets(wl, labels) != -100
    _, Vb = flce.flce_backward_blocking(wl.N, wl.H, wl.V)
    assert (wl.V > Vb) == dense
    if dense:
        assert got == min(wl.N, math.ceil(int(valid.sum()) / 256) * 256)
    else:
        assert got == 256 * sum(bool(valid[i:i + 256].any()) for i in range(0, wl.N, 256))
    assert 0 < got <= wl.N
