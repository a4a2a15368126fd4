"""Work and traffic conventions used to turn kernel times into roofline figures.

FLOPs: two matrix products of 2*N*N*d each per head in the forward pass,
i.e. ``4*B*H*N^2*d`` (the multiply-add convention 2*M*N*K of the GEMM items
on the GPU-programming topic page); this reproduces the FlashAttention-3
ablation figures (Table 2: 3.538 ms <-> 661 TFLOP/s at B=4, H=16, N=8448,
d=128).  Causal masking halves it.  The backward pass counts five products
(S recomputed, dP, dV, dK, dQ): 2.5x the forward.

Algorithmic HBM bytes: what one pass must move at least once.
  forward bf16: read Q, K, V (2 B/elem), write O (2 B) and LSE (4 B/row);
  forward fp8 : read Q, K, V (1 B/elem), write O (2 B) and LSE (4 B/row);
  backward    : read Q, K, V, O, dO, write dQ, dK, dV (2 B each), read LSE
                and D, plus the fp32 dQ accumulator written once and read
                once (4 + 4 B/elem).
  backward main kernel alone: read Q, K, V, dO (2 B each), write dK, dV
                (2 B each), read LSE and D (4 B/row each), and read + write
                the fp32 dQ accumulator once (8 B/elem).
"""

from __future__ import annotations


def attn_flops(B: int, H: int, N: int, d: int, causal: bool, pass_: str = "fwd") -> float:
    f = 4.0 * B * H * N * N * d
    if causal:
        f *= 0.5
    if pass_ == "bwd":
        f *= 2.5
    return f


def attn_bytes(B: int, H: int, N: int, d: int, pass_: str = "fwd") -> float:
    rows = B * H * N
    elems = rows * d
    if pass_ == "fwd":
        return 8.0 * elems + 4.0 * rows
    if pass_ == "fwd_fp8":
        return 5.0 * elems + 4.0 * rows
    if pass_ == "bwd":
        return 16.0 * elems + 8.0 * elems + 8.0 * rows
    if pass_ == "bwd_main":
        return 12.0 * elems + 8.0 * elems + 8.0 * rows
    raise ValueError(pass_)
