"""A seeded sweep of problem shapes the other files do not enumerate: sequence
lengths anywhere in 1..900 (ragged tails of every size), both head dims, one
or two batches, grouped heads (H = G * Hk), and every mask the library offers
(none, causal, sliding windows with one or two bounds, windows narrower than a
tile or wider than the sequence).  Each case runs the forward and the backward
on the GPU and compares O, LSE and dQ/dK/dV with the fp64 oracle at the stated
tolerances; FP8 cases compare O.  The shapes come from a fixed generator, so
every run checks the same cases."""

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import make_inputs_fp8, make_inputs_gqa

from .helpers import (TOL_FP8_RELFRO, TOL_GRAD_RELFRO, TOL_LSE_ABS, TOL_O_MAXABS, bf16_out_err,
                      bf16_to_device, decoded, decoded_fp8, device_bf16_to_f64, device_f32_to_f64,
                      grad_rel_err, max_abs, rel_fro, u8_to_device)

pytestmark = pytest.mark.gpu


def _cases(n_cases, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for i in range(n_cases):
        d = int(rng.choice([64, 128]))
        B = int(rng.integers(1, 3))
        Hk = int(rng.integers(1, 4))
        G = int(rng.integers(1, 4))
        N = int(rng.integers(1, 901))
        kind = ("none", "causal", "window")[int(rng.integers(0, 3))]
        window = None
        if kind == "window":
            left = int(rng.choice([-1, int(rng.integers(0, N + 130))]))
            right = int(rng.choice([-1, 0, int(rng.integers(0, N + 130))]))
            window = (left, right)
        out.append((i, B, G * Hk, Hk, N, d, kind, window))
    return out


@pytest.mark.parametrize("case", _cases(24, 2026), ids=lambda c: f"c{c[0]}-B{c[1]}H{c[2]}Hk{c[3]}N{c[4]}d{c[5]}-{c[6]}")
def test_random_shapes_fwd_bwd(case):
    i, B, H, Hk, N, d, kind, window = case
    inp = make_inputs_gqa(B, H, Hk, N, d, seed=9000 + i, with_grad=True)
    q, k, v, do = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    causal = kind == "causal"
    if kind == "window":
        o, lse = api.fwd_window(q, k, v, *window)
        dq, dk, dv = api.bwd_window(q, k, v, o, do, lse, *window)
    else:
        o, lse = api.fwd(q, k, v, causal=causal)
        dq, dk, dv = api.bwd(q, k, v, o, do, lse, causal=causal)
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    qf, kf, vf, dof = decoded(inp)
    scale = 1.0 / np.sqrt(d)
    o_ref, lse_ref = oracle.forward_gqa(qf, kf, vf, scale, causal, window=window)
    assert bf16_out_err(device_bf16_to_f64(o), o_ref) <= TOL_O_MAXABS
    assert max_abs(device_f32_to_f64(lse), lse_ref) <= TOL_LSE_ABS
    ref = oracle.backward_gqa(qf, kf, vf, dof, scale, causal, window=window)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        g = device_bf16_to_f64(g)
        assert np.all(np.isfinite(g)), name
        err = grad_rel_err(g, r)
        assert err <= TOL_GRAD_RELFRO, (name, err)


@pytest.mark.parametrize("N,causal", [(1, False), (77, True), (129, False), (383, True), (640, False)])
def test_random_lengths_fp8(N, causal):
    f8 = make_inputs_fp8(1, 2, N, 128, seed=700 + N)
    q8, k8, v8 = (u8_to_device(x) for x in (f8.q8, f8.k8, f8.v8))
    o, lse = api.fwd_fp8(q8, k8, v8, f8.sq, f8.sk, f8.sv, causal=causal)
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    o_ref, _ = oracle.forward(*decoded_fp8(f8), 1.0 / np.sqrt(128), causal)
    assert rel_fro(device_bf16_to_f64(o), o_ref) <= TOL_FP8_RELFRO
