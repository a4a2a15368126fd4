"""Shared test helpers: comparison metrics, host<->device packing of the seeded
inputs, and oracle calls on decoded inputs."""

import numpy as np

import oracle

# Tolerances the parity tests enforce (bf16 O max-abs, LSE absolute, gradient
# relative Frobenius, FP8 O relative Frobenius).
TOL_O_MAXABS = 1e-2
TOL_LSE_ABS = 1e-3
TOL_GRAD_RELFRO = 2e-2
TOL_FP8_RELFRO = 6e-2


def max_abs(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))


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
