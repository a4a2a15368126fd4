"""FP8 (E4M3, per-tensor scales) forward parity vs the oracle run on the
dequantised inputs s * decode(code)."""

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import AttnInputsFP8, f32_to_e4m3, make_inputs_fp8

from .helpers import (TOL_FP8_RELFRO, TOL_LSE_ABS, decoded_fp8, device_bf16_to_f64,
                      device_f32_to_f64, max_abs, rel_fro, u8_to_device)

pytestmark = pytest.mark.gpu


def run_fp8(inp, causal):
    q8, k8, v8 = (u8_to_device(x) for x in (inp.q8, inp.k8, inp.v8))
    o, lse = api.fwd_fp8(q8, k8, v8, inp.sq, inp.sk, inp.sv, causal=causal)
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    return device_bf16_to_f64(o), device_f32_to_f64(lse)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 100, 128, 300, 1024])
def test_fp8_fwd_matches_oracle(N, causal):
    inp = make_inputs_fp8(1, 2, N, 128, seed=N + int(causal))
    o, lse = run_fp8(inp, causal)
    q, k, v = decoded_fp8(inp)
    o_ref, lse_ref = oracle.forward(q, k, v, 1.0 / np.sqrt(128), causal)
    assert np.all(np.isfinite(o))
    assert rel_fro(o, o_ref) <= TOL_FP8_RELFRO, rel_fro(o, o_ref)
    # scores are exact fp32 sums of E4M3 products: the log-sum-exp stays tight
    assert max_abs(lse, lse_ref) <= TOL_LSE_ABS, max_abs(lse, lse_ref)


def test_fp8_fwd_persistent_many_items():
    """Without a mask the FP8 forward runs persistent CTAs: 2 x 24 heads x 8
    query-tile pairs = 384 items, two or three per CTA, each with a ragged last
    tile, so barrier phases, the key/value ring position and the output
    accumulators carry over between items.  Sampled heads against the oracle."""
    B, H, N, d = 2, 24, 2000, 128
    inp = make_inputs_fp8(B, H, N, d, seed=11)
    o, lse = run_fp8(inp, False)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    q, k, v = decoded_fp8(inp)
    scale = 1.0 / np.sqrt(d)
    for (b, h) in [(0, 0), (B - 1, H - 1), (B // 2, H // 2)]:
        o_ref, lse_ref, _ = oracle.head_forward(q[b, h], k[b, h], v[b, h], scale, False)
        assert rel_fro(o[b, h], o_ref) <= TOL_FP8_RELFRO, (b, h, rel_fro(o[b, h], o_ref))
        assert max_abs(lse[b, h], lse_ref) <= TOL_LSE_ABS, (b, h)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_fwd_growing_scores_exercise_rescale(causal):
    """Keys that grow along a direction shared with the queries make every row's
    maximum rise by more than the lazy threshold (2^8 in log2 units) from one key
    tile to the next: without a mask every row rescales its output accumulator at
    each of the 7 key tiles after the first (counted on the CPU with the same
    rule), so the FP8 rescale path runs throughout."""
    B, H, N, d = 1, 2, 1024, 128
    rng = np.random.Generator(np.random.PCG64(21))
    base = rng.standard_normal(d).astype(np.float32)
    q = (base + 0.5 * rng.standard_normal((B, H, N, d))).astype(np.float32)
    ramp = (6.0 * np.arange(N) / N).astype(np.float32)[None, None, :, None]
    k = (ramp * base + 0.5 * rng.standard_normal((B, H, N, d))).astype(np.float32)
    v = rng.standard_normal((B, H, N, d)).astype(np.float32)
    (q8, sq), (k8, sk), (v8, sv) = f32_to_e4m3(q), f32_to_e4m3(k), f32_to_e4m3(v)
    inp = AttnInputsFP8(B, H, N, d, q8, k8, v8, sq, sk, sv, 21)
    o, lse = run_fp8(inp, causal)
    qd, kd, vd = decoded_fp8(inp)
    o_ref, lse_ref = oracle.forward(qd, kd, vd, 1.0 / np.sqrt(d), causal)
    assert np.all(np.isfinite(o))
    assert rel_fro(o, o_ref) <= TOL_FP8_RELFRO, rel_fro(o, o_ref)
    assert max_abs(lse, lse_ref) <= TOL_LSE_ABS, max_abs(lse, lse_ref)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [100, 300, 2000])
def test_fp8_fwd_exp2_offload_matches_oracle(N, causal):
    """attn_set_exp2_offload(1): one group of four exponentials in eight is
    computed on the FMA pipe (2^n times a cubic for 2^r).  The outputs must
    meet the same FP8 tolerances, and differ from the MUFU path only by the
    polynomial's relative error (7.5e-5) passed through the E4M3 rounding of P."""
    inp = make_inputs_fp8(2, 2, N, 128, seed=70 + N + int(causal))
    o_ref_gpu, lse_ref_gpu = run_fp8(inp, causal)
    api.set_exp2_offload(True)
    try:
        o, lse = run_fp8(inp, causal)
    finally:
        api.set_exp2_offload(False)
    q, k, v = decoded_fp8(inp)
    o_ref, lse_ref = oracle.forward(q, k, v, 1.0 / np.sqrt(128), causal)
    assert rel_fro(o, o_ref) <= TOL_FP8_RELFRO, rel_fro(o, o_ref)
    assert max_abs(lse, lse_ref) <= TOL_LSE_ABS, max_abs(lse, lse_ref)
    # the two GPU paths: P rounded to E4M3 can flip by one code where the
    # polynomial lands on the other side of a rounding boundary
    assert rel_fro(o, o_ref_gpu) <= 1e-2
    assert max_abs(lse, lse_ref_gpu) <= 1e-4
