"""Shared test helpers: comparison metrics, host<->device packing of the seeded
inputs, and oracle calls on decoded inputs."""

import numpy as np

import oracle

# Tolerances the parity tests enforce (bf16 O max-abs beyond the output's own
# rounding, LSE absolute, gradient relative Frobenius, FP8 O relative Frobenius).
TOL_O_MAXABS = 1e-2
TOL_LSE_ABS = 1e-3
TOL_GRAD_RELFRO = 2e-2
TOL_FP8_RELFRO = 6e-2


def max_abs(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def bf16_half_ulp(x):
    """Half the spacing of bfloat16 numbers at |x| (8 significant bits)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 0.5 * 2.0 ** (e - 7), 0.0)


def bf16_out_err(gpu, ref):
    """Max over elements of |gpu - ref| beyond the rounding of ref itself to
    bfloat16: the part of the error the computation adds on top of storing the
    exact result in the output format."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if not gpu.size:
        return 0.0
    return float(np.max(np.abs(gpu - ref) - bf16_half_ulp(ref)))


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))


def row_blocks(n, tile=128):
    """[start, stop) blocks of ``tile`` rows covering n rows; a ragged last block
    shorter than tile / 2 is merged into the block before it, so that no block
    is so short that the output's own rounding noise decides its error (one row
    with two visible keys can be 3 % off its own norm from bf16 rounding)."""
    starts = list(range(0, n, tile))
    if len(starts) > 1 and n - starts[-1] < tile // 2:
        starts.pop()
    return [(a, starts[i + 1] if i + 1 < len(starts) else n) for i, a in enumerate(starts)]


def grad_rel_err(gpu, ref, tile=128):
    """Largest relative Frobenius error of a gradient over the whole tensor and
    over every block of about ``tile`` consecutive rows (second-to-last axis)
    of every head: a single wrong row, ragged tail or mis-indexed tile moves its
    own block's error by O(1) even where the whole-tensor figure hides it."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    worst = rel_fro(gpu, ref)
    n = ref.shape[-2] if ref.ndim >= 2 else ref.shape[0]
    g2 = gpu.reshape((-1,) + gpu.shape[-2:]) if gpu.ndim >= 2 else gpu.reshape(1, -1, 1)
    r2 = ref.reshape((-1,) + ref.shape[-2:]) if ref.ndim >= 2 else ref.reshape(1, -1, 1)
    for i in range(r2.shape[0]):
        for a, b in row_blocks(n, tile):
            worst = max(worst, rel_fro(g2[i, a:b], r2[i, a:b]))
    return worst


def bf16_to_device(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def u8_to_device(codes):
    import torch
    return torch.from_numpy(np.ascontiguousarray(codes)).cuda()


def device_bf16_to_f64(t):
    import torch
    bits = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return oracle.bf16_bits_to_f64(bits)


def device_f32_to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def decoded(inp):
    """fp64 Q, K, V (and dO) exactly as the GPU reads them."""
    q = oracle.bf16_bits_to_f64(inp.q_bits)
    k = oracle.bf16_bits_to_f64(inp.k_bits)
    v = oracle.bf16_bits_to_f64(inp.v_bits)
    do = oracle.bf16_bits_to_f64(inp.do_bits) if inp.do_bits is not None else None
    return q, k, v, do


def decoded_fp8(inp):
    return (oracle.e4m3_to_f64(inp.q8, inp.sq), oracle.e4m3_to_f64(inp.k8, inp.sk),
            oracle.e4m3_to_f64(inp.v8, inp.sv))
