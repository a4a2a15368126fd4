"""Exact softmax attention for GB300 (sm_103a): forward, backward and FP8 forward.

The compute runs in ``libattn_sm103a.so`` (hand-written CUDA behind a C ABI,
declared in ``include/attn_sm103a.h``); ``exact_attention_52_gb300.api`` is the
thin Python binding over it.  Importing this package loads nothing: the
library is opened on the first call, and a missing or unbuilt library raises.
"""

__all__ = ["api", "inputs", "roofline"]
