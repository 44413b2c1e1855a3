"""Without the built library every entry point of the binding raises; nothing
falls back to another implementation (the oracle is never imported by the
product package)."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
import lm_head_linear_flce_gb300 as flce
flce.library_path = "/nonexistent/libflce.so"
flce._lib = None
import torch
calls = [
    lambda: flce.workspace_size(8, 8, 8),
    lambda: flce.flce_set_wait_limit_ns(0),
    lambda: flce.flce_kernel_launch_count(),
]
for c in calls:
    try:
        c()
    except RuntimeError as e:
        assert "no fallback" in str(e), e
    else:
        sys.exit("a call succeeded without the library")
assert "oracle" not in sys.modules, "the product package imported the oracle"
import lm_head_linear_flce_gb300.vocab_parallel  # noqa: F401
assert "oracle" not in sys.modules, "the vocabulary-parallel module imported the oracle"
print("ok")
"""


def test_calls_raise_without_the_library():
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")
