"""The boundary used from C: a C99 program (tests/c/abi_gpu_run.c) allocates
device memory with the CUDA runtime, runs flce_forward and flce_backward
through include/flce.h and writes the results to files; they must match the
oracle like the Python binding's results do."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import assert_grad, assert_loss, assert_lse

pytestmark = pytest.mark.gpu

flce = pytest.importorskip("lm_head_linear_flce_gb300")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bf16_from_bits(a, shape):
    return torch.from_numpy(a.astype(np.int16)).view(torch.bfloat16).reshape(shape).double().numpy()


@pytest.mark.parametrize("N,H,V,S,shift,red", [(700, 136, 1500, 350, 1, 0), (256, 64, 3000, 0, 0, 1)])
def test_c_program_matches_the_oracle(tmp_path, N, H, V, S, shift, red):
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if cc is None or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime_api.h")):
        pytest.skip("no C compiler or CUDA runtime headers")
    libdir = os.path.dirname(flce.library_path)
    cudalib = next((d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                    if os.path.isdir(d)), None)
    exe = tmp_path / "abi_gpu_run"
    cmd = [cc, "-std=c99", "-O1", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c", "abi_gpu_run.c"),
           "-L", libdir, "-lflce", f"-Wl,-rpath,{libdir}", "-L", cudalib, "-lcudart",
           f"-Wl,-rpath,{cudalib}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    X, W, labels = workloads.random_case(N, H, V, seed=N + V, w_std=0.08)
    inp, out = tmp_path / "in", tmp_path / "out"
    inp.mkdir()
    out.mkdir()
    X.view(torch.int16).numpy().tofile(inp / "X.bin")
    W.view(torch.int16).numpy().tofile(inp / "W.bin")
    labels.numpy().astype(np.int64).tofile(inp / "labels.bin")
    r = subprocess.run([str(exe), str(N), str(H), str(V), str(S), str(shift), str(red), str(inp),
                        str(out)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    kw = dict(seq_len=S or None, shift=bool(shift), reduction="sum" if red else "mean")
    ref = oracle.forward(X, W, labels, **kw)
    dX, dW = oracle.backward(X, W, labels, lse=ref["lse"], **kw)
    assert int(np.fromfile(out / "n_valid.bin", np.int64)[0]) == ref["n_valid"]
    assert_loss(float(np.fromfile(out / "loss.bin", np.float32)[0]), ref["loss"])
    assert_lse(np.fromfile(out / "lse.bin", np.float32), ref["lse"])
    assert_grad("dX", _bf16_from_bits(np.fromfile(out / "dX.bin", np.int16), (N, H)), dX)
    assert_grad("dW", _bf16_from_bits(np.fromfile(out / "dW.bin", np.int16), (V, H)), dW)
