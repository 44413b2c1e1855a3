"""CPU float64 oracle for fused linear cross-entropy (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path.
"""
from .flce_oracle import (IGNORE_INDEX, as_f64, as_i64, backward, effective_targets,
                          forward, forward_backward, grad_logits, grad_scale, logits_rows,
                          rows_forward_backward, vocab_rows_dW)
from .brute import brute_force

__all__ = ["IGNORE_INDEX", "as_f64", "as_i64", "backward", "effective_targets", "forward",
           "forward_backward", "grad_logits", "grad_scale", "logits_rows", "rows_forward_backward",
           "vocab_rows_dW", "brute_force"]
