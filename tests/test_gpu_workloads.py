"""Parity at the five benchmark workloads' full sizes, in the launch
configuration the benchmark uses.  The small workloads are compared element
by element; the large ones on sampled heads (forward and backward, all rows
of the head) or sampled query rows (FP8), which the oracle computes one by
one, plus properties that must hold everywhere."""

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import workload_inputs, WORKLOADS

from .helpers import (bf16_half_ulp, bf16_out_err, TOL_FP8_RELFRO, TOL_GRAD_RELFRO, TOL_LSE_ABS, TOL_O_MAXABS, bf16_to_device,
                      decoded, decoded_fp8, device_bf16_to_f64, device_f32_to_f64, max_abs,
                      rel_fro, u8_to_device)

pytestmark = pytest.mark.gpu


def _bf16_run(name):
    w = WORKLOADS[name]
    inp = workload_inputs(name)
    q, k, v = (bf16_to_device(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits))
    o, lse = api.fwd(q, k, v, causal=w["causal"])
    grads = None
    if "bwd" in w["passes"]:
        do = bf16_to_device(inp.do_bits)
        grads = api.bwd(q, k, v, o, do, lse, causal=w["causal"])
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    return w, inp, o, lse, grads


@pytest.mark.parametrize("name", ["fwd_b1_h1_n128_d64", "fwd_b4_h16_n1024_d64"])
def test_small_workloads_every_element(name):
    w, inp, o, lse, _ = _bf16_run(name)
    q, k, v, _ = decoded(inp)
    o_ref, lse_ref = oracle.forward(q, k, v, 1.0 / np.sqrt(w["d"]), w["causal"])
    assert bf16_out_err(device_bf16_to_f64(o), o_ref) <= TOL_O_MAXABS
    assert max_abs(device_f32_to_f64(lse), lse_ref) <= TOL_LSE_ABS


@pytest.mark.parametrize("name,heads", [
    ("fwdbwd_causal_b2_h16_n4096_d128", [(0, 0), (1, 15)]),
    ("fwdbwd_b1_h32_n8192_d128_outlierK", [(0, 0), (0, 31)]),
])
def test_large_bf16_workloads_sampled_heads(name, heads):
    w, inp, o, lse, grads = _bf16_run(name)
    og, lg = device_bf16_to_f64(o), device_f32_to_f64(lse)
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg))
    gg = [device_bf16_to_f64(t) for t in grads]
    for t in gg:
        assert np.all(np.isfinite(t))
    q, k, v, do = decoded(inp)
    scale = 1.0 / np.sqrt(w["d"])
    for (b, h) in heads:
        o_ref, lse_ref, _ = oracle.head_forward(q[b, h], k[b, h], v[b, h], scale, w["causal"])
        assert bf16_out_err(og[b, h], o_ref) <= TOL_O_MAXABS, (b, h)
        assert max_abs(lg[b, h], lse_ref) <= TOL_LSE_ABS, (b, h)
        ref = oracle.head_backward(q[b, h], k[b, h], v[b, h], do[b, h], scale, w["causal"])
        for nm, g, r in zip(("dq", "dk", "dv"), gg, ref[:3]):
            assert rel_fro(g[b, h], r) <= TOL_GRAD_RELFRO, (nm, b, h, rel_fro(g[b, h], r))
    # every head and row: LSE_i >= ln(1) + max score >= max over the sampled
    # diagonal score, and LSE_i <= max score + ln(#visible keys)
    qs = q.reshape(-1, w["N"], w["d"])
    ks = k.reshape(-1, w["N"], w["d"])
    diag = scale * np.einsum("hnd,hnd->hn", qs, ks)
    assert np.all(lg.reshape(diag.shape) >= diag - TOL_LSE_ABS)
    # every head and row: O is a convex combination of the head's V rows, so each
    # element lies within that head's range of the V column (up to the tolerance
    # and the output's own rounding)
    vmin = v.min(axis=2, keepdims=True)
    vmax = v.max(axis=2, keepdims=True)
    slack = TOL_O_MAXABS + bf16_half_ulp(np.maximum(np.abs(vmin), np.abs(vmax)))
    assert np.all(og >= vmin - slack) and np.all(og <= vmax + slack)


def test_fp8_workload_sampled_rows():
    name = "fp8fwd_causal_b1_h16_n16384_d128"
    w = WORKLOADS[name]
    inp = workload_inputs(name)
    q8, k8, v8 = (u8_to_device(x) for x in (inp.q8, inp.k8, inp.v8))
    o, lse = api.fwd_fp8(q8, k8, v8, inp.sq, inp.sk, inp.sv, causal=True)
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    og, lg = device_bf16_to_f64(o), device_f32_to_f64(lse)
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg))
    q, k, v = decoded_fp8(inp)
    rng = np.random.Generator(np.random.PCG64(1))
    rows = np.unique(np.concatenate([np.arange(0, 130), np.arange(w["N"] - 130, w["N"]),
                                     rng.choice(w["N"], 256, replace=False)]))
    scale = 1.0 / np.sqrt(w["d"])
    for h in (0, 7, 15):
        o_ref, lse_ref, _ = oracle.head_forward(q[0, h], k[0, h], v[0, h], scale, True, rows=rows)
        assert rel_fro(og[0, h][rows], o_ref) <= TOL_FP8_RELFRO, h
        assert max_abs(lg[0, h][rows], lse_ref) <= TOL_LSE_ABS, h
