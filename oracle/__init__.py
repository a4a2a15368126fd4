"""fp64 CPU oracle for exact attention -- test infrastructure only.

Imported by the tests, the smoke check and the benchmark's CPU-baseline leg;
never by the library.  See ``oracle/attention.py`` for what it computes and
which passages each function follows.
"""
from .attention import (backward, backward_gqa, bf16_bits_to_f64, causal_visible, e4m3_to_f64,
                        forward, forward_gqa, head_backward, head_backward_rows, head_forward,
                        kv_head_of, scores, softmax_rows, window_visible)

__all__ = ["backward", "backward_gqa", "bf16_bits_to_f64", "causal_visible", "e4m3_to_f64",
           "forward", "forward_gqa", "head_backward", "head_backward_rows", "head_forward",
           "kv_head_of", "scores", "softmax_rows", "window_visible"]
