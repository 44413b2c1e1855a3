"""The boundary from C: a C99 program that includes include/flce.h, links
libflce.so and calls the host-only entry points (sizes, status strings,
argument checks).  Runs without a GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

flce = pytest.importorskip("lm_head_linear_flce_gb300")


def test_c_program_compiles_links_and_runs(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(flce.library_path):
        from lm_head_linear_flce_gb300 import _build
        _build.build()
    exe = tmp_path / "abi_host_check"
    libdir = os.path.dirname(flce.library_path)
    cmd = [cc, "-std=c99", "-Wall", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_host_check.c"),
           "-L", libdir, "-lflce", f"-Wl,-rpath,{libdir}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok ")
    assert int(r.stdout.split()[1]) == flce.workspace_size(8192, 3584, 152064)
