"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws random numbers and packs them into the storage formats
the kernels read (bf16 bit patterns, OCP FP8 E4M3 bytes with a per-tensor
scale).  It holds none of the attention arithmetic: the oracle and the CUDA
path each decode these bytes on their own.

Recipe (the workloads of the FlashAttention pages: i.i.d. N(0,1) Q/K/V/dO):
  * ``numpy.random.Generator(PCG64(seed))``, seed 0 unless stated;
  * draw order Q, K, V, dO, each ``standard_normal`` float32 of shape
    ``[B, H, N, d]``;
  * optional "outlier keys": per (b, h) a set of ``round(frac * N)`` distinct
    key rows chosen with ``Generator.choice(..., replace=False)`` (drawn after
    dO, heads in (b, h) order) is multiplied by a factor in float32 before any
    rounding; with factor 8 this is exact in bf16;
  * bf16: round-to-nearest-even of the float32 value, stored as uint16 bits;
  * FP8 E4M3 (OCP "e4m3fn", max finite 448): per-tensor scale
    ``s = amax(|x|) / 448``; codes = saturating round-to-nearest-even of
    ``x / s``.  The value the kernels see is ``s * decode(code)``.
"""

from __future__ import annotations

import dataclasses

import numpy as np

E4M3_MAX = 448.0


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return uint16 bits.

    Inputs are finite normal draws, so no NaN handling is needed here; the
    function refuses non-finite input instead of guessing.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("bf16 packing expects finite inputs")
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return rounded.astype(np.uint16)


def f32_to_e4m3(x: np.ndarray) -> tuple[np.ndarray, float]:
    """Per-tensor FP8 E4M3 packing: returns (uint8 codes, fp32 scale s).

    ``s = amax(|x|)/448`` so the largest magnitude lands on the largest
    finite code.  The float8 conversion of PyTorch's CPU backend does the
    round-to-nearest-even encoding; values are clamped to +-448 first so that
    nothing can overflow to the NaN code.
    """
    import torch

    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    s = np.float32(amax / E4M3_MAX) if amax > 0 else np.float32(1.0)
    y = np.clip(x / s, -E4M3_MAX, E4M3_MAX).astype(np.float32)
    codes = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes.copy(), float(s)


@dataclasses.dataclass
class AttnInputs:
    """One seeded problem.  ``*_bits`` are bf16 uint16 patterns, ``[B,H,N,d]``."""

    B: int
    H: int
    N: int
    d: int
    q_bits: np.ndarray
    k_bits: np.ndarray
    v_bits: np.ndarray
    do_bits: np.ndarray | None
    seed: int
    outlier_rows: np.ndarray | None  # [B*H, n_out] key rows scaled, or None


@dataclasses.dataclass
class AttnInputsFP8:
    """One seeded FP8 problem: E4M3 codes ``[B,H,N,d]`` and per-tensor scales."""

    B: int
    H: int
    N: int
    d: int
    q8: np.ndarray
    k8: np.ndarray
    v8: np.ndarray
    sq: float
    sk: float
    sv: float
    seed: int


def _draw(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def make_inputs(B: int, H: int, N: int, d: int, *, seed: int = 0,
                with_grad: bool = False, outlier_frac: float = 0.0,
                outlier_factor: float = 8.0) -> AttnInputs:
    """Draw Q, K, V (and dO) as described in the module docstring."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = (B, H, N, d)
    q = _draw(rng, shape)
    k = _draw(rng, shape)
    v = _draw(rng, shape)
    do = _draw(rng, shape) if with_grad else None
    rows = None
    if outlier_frac > 0.0:
        n_out = int(round(outlier_frac * N))
        rows = np.zeros((B * H, n_out), dtype=np.int64)
        kf = k.reshape(B * H, N, d)
        for bh in range(B * H):
            sel = rng.choice(N, size=n_out, replace=False)
            rows[bh] = np.sort(sel)
            kf[bh, sel, :] *= np.float32(outlier_factor)
    return AttnInputs(B, H, N, d, f32_to_bf16_bits(q), f32_to_bf16_bits(k),
                      f32_to_bf16_bits(v),
                      f32_to_bf16_bits(do) if do is not None else None,
                      seed, rows)


def make_inputs_gqa(B: int, H: int, Hk: int, N: int, d: int, *, seed: int = 0,
                    with_grad: bool = False) -> AttnInputs:
    """Grouped-query inputs: Q and dO ``[B, H, N, d]``, K and V ``[B, Hk, N, d]``,
    drawn in the order Q, K, V, dO like ``make_inputs``."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _draw(rng, (B, H, N, d))
    k = _draw(rng, (B, Hk, N, d))
    v = _draw(rng, (B, Hk, N, d))
    do = _draw(rng, (B, H, N, d)) if with_grad else None
    return AttnInputs(B, H, N, d, f32_to_bf16_bits(q), f32_to_bf16_bits(k), f32_to_bf16_bits(v),
                      f32_to_bf16_bits(do) if do is not None else None, seed, None)


def make_inputs_fp8(B: int, H: int, N: int, d: int, *, seed: int = 0) -> AttnInputsFP8:
    """Draw Q, K, V ~ N(0,1) in float32 and pack each to E4M3 with its own scale."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = (B, H, N, d)
    q = _draw(rng, shape)
    k = _draw(rng, shape)
    v = _draw(rng, shape)
    q8, sq = f32_to_e4m3(q)
    k8, sk = f32_to_e4m3(k)
    v8, sv = f32_to_e4m3(v)
    return AttnInputsFP8(B, H, N, d, q8, k8, v8, sq, sk, sv, seed)


# The five workloads the benchmark and the full-size parity tests use.  Each
# entry: (name, B, H, N, d, causal, passes, options).
WORKLOADS = {
    "fwd_b1_h1_n128_d64": dict(B=1, H=1, N=128, d=64, causal=False, passes=("fwd",)),
    "fwd_b4_h16_n1024_d64": dict(B=4, H=16, N=1024, d=64, causal=False, passes=("fwd",)),
    "fwdbwd_causal_b2_h16_n4096_d128": dict(B=2, H=16, N=4096, d=128, causal=True,
                                            passes=("fwd", "bwd")),
    "fwdbwd_b1_h32_n8192_d128_outlierK": dict(B=1, H=32, N=8192, d=128, causal=False,
                                              passes=("fwd", "bwd"), outlier_frac=0.01,
                                              outlier_factor=8.0),
    "fp8fwd_causal_b1_h16_n16384_d128": dict(B=1, H=16, N=16384, d=128, causal=True,
                                             passes=("fwd_fp8",)),
}


def workload_inputs(name: str, *, seed: int = 0):
    """Inputs of one named workload (bf16 ``AttnInputs`` or ``AttnInputsFP8``)."""
    w = WORKLOADS[name]
    if "fwd_fp8" in w["passes"]:
        return make_inputs_fp8(w["B"], w["H"], w["N"], w["d"], seed=seed)
    return make_inputs(w["B"], w["H"], w["N"], w["d"], seed=seed,
                       with_grad="bwd" in w["passes"],
                       outlier_frac=w.get("outlier_frac", 0.0),
                       outlier_factor=w.get("outlier_factor", 8.0))
