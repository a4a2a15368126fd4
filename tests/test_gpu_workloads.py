"""Parity at the five benchmark workloads' full sizes, in the launch
configuration the benchmark uses.  The small workloads are compared element
by element.  The large ones are compared on sampled query rows of EVERY head
(O, LSE and dQ rows, which the oracle computes one by one), on whole heads for
dK and dV (four heads each, block by block), and on properties that must hold
for every row of every head: the log-sum-exp lies between the row's largest
score and that score plus ln(number of visible keys), and O is a convex
combination of the head's V rows."""

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import workload_inputs, WORKLOADS

from .helpers import (bf16_half_ulp, bf16_out_err, TOL_FP8_RELFRO, TOL_GRAD_RELFRO, TOL_LSE_ABS,
                      TOL_O_MAXABS, bf16_to_device, decoded, decoded_fp8, device_bf16_to_f64,
                      device_f32_to_f64, grad_rel_err, max_abs, rel_fro, u8_to_device)

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


def sampled_rows(N, seed, n_random=48):
    """Rows of the first and last tiles, two tile boundaries and random rows."""
    rng = np.random.Generator(np.random.PCG64(seed))
    fixed = [0, 1, 2, 63, 64, 126, 127, 128, 129, N // 2 - 1, N // 2, N - 129, N - 128, N - 2, N - 1]
    return np.unique(np.concatenate([np.array(fixed), rng.choice(N, n_random, replace=False)]))


def row_max_scores(q, k, scale, causal, block=1024):
    """max_j scale * q_i . k_j over the visible keys of every row, per head
    ([heads, N, d] fp64 inputs), in float32 blocks (error ~1e-6 relative)."""
    hs, N, _ = q.shape
    out = np.empty((hs, N))
    for h in range(hs):
        kt = np.ascontiguousarray(k[h].T.astype(np.float32))
        for r0 in range(0, N, block):
            s = (q[h, r0:r0 + block].astype(np.float32) @ kt) * np.float32(scale)
            if causal:
                rows = np.arange(r0, min(N, r0 + block))[:, None]
                s = np.where(np.arange(N)[None, :] <= rows, s, -np.inf)
            out[h, r0:r0 + block] = s.max(axis=1)
    return out


def assert_lse_bounds(lse, q, k, scale, causal):
    """max score <= LSE <= max score + ln(#visible keys), every row of every head."""
    N = q.shape[-2]
    qs = q.reshape(-1, N, q.shape[-1])
    ks = k.reshape(-1, N, k.shape[-1])
    mx = row_max_scores(qs, ks, scale, causal)
    n_vis = np.arange(1, N + 1, dtype=np.float64) if causal else np.full(N, float(N))
    lg = lse.reshape(mx.shape)
    slack = TOL_LSE_ABS + 1e-5 * np.abs(mx)
    assert np.all(lg >= mx - slack), float(np.max(mx - lg))
    assert np.all(lg <= mx + np.log(n_vis)[None, :] + slack), float(np.max(lg - mx - np.log(n_vis)))


@pytest.mark.parametrize("name", ["fwd_b1_h1_n128_d64", "fwd_b4_h16_n1024_d64"])
def test_small_workloads_every_element(name):
    w, inp, o, lse, _ = _bf16_run(name)
    q, k, v, _ = decoded(inp)
    o_ref, lse_ref = oracle.forward(q, k, v, 1.0 / np.sqrt(w["d"]), w["causal"])
    assert bf16_out_err(device_bf16_to_f64(o), o_ref) <= TOL_O_MAXABS
    assert max_abs(device_f32_to_f64(lse), lse_ref) <= TOL_LSE_ABS


# B1 H32 N8192: 2048 key-tile items for 152 CTAs, the last 72 (key tiles 56-63 of
# head 30 and all of head 31) split into two parts each, so head 31's dK and dV
# come entirely from summed partials
@pytest.mark.parametrize("name,full_heads", [
    ("fwdbwd_causal_b2_h16_n4096_d128", [(0, 0), (0, 9), (1, 4), (1, 15)]),
    ("fwdbwd_b1_h32_n8192_d128_outlierK", [(0, 0), (0, 11), (0, 22), (0, 31)]),
])
def test_large_bf16_workloads(name, full_heads):
    w, inp, o, lse, grads = _bf16_run(name)
    og, lg = device_bf16_to_f64(o), device_f32_to_f64(lse)
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg))
    dqg, dkg, dvg = (device_bf16_to_f64(t) for t in grads)
    for t in (dqg, dkg, dvg):
        assert np.all(np.isfinite(t))
    q, k, v, do = decoded(inp)
    scale = 1.0 / np.sqrt(w["d"])
    B, H, N = w["B"], w["H"], w["N"]
    # every head: sampled rows of O, LSE and dQ
    for b in range(B):
        for h in range(H):
            rows = sampled_rows(N, seed=1000 * b + h)
            o_ref, lse_ref, _ = oracle.head_forward(q[b, h], k[b, h], v[b, h], scale, w["causal"],
                                                    rows=rows)
            assert bf16_out_err(og[b, h][rows], o_ref) <= TOL_O_MAXABS, (b, h)
            assert max_abs(lg[b, h][rows], lse_ref) <= TOL_LSE_ABS, (b, h)
            dq_ref, _ = oracle.head_backward_rows(q[b, h], k[b, h], v[b, h], do[b, h], scale,
                                                  w["causal"], rows)
            err = rel_fro(dqg[b, h][rows], dq_ref)
            assert err <= TOL_GRAD_RELFRO, ("dq rows", b, h, err)
    # four whole heads: dQ, dK, dV against the oracle, whole and per 128-row block
    for (b, h) in full_heads:
        ref = oracle.head_backward(q[b, h], k[b, h], v[b, h], do[b, h], scale, w["causal"])
        for nm, g, r in zip(("dq", "dk", "dv"), (dqg, dkg, dvg), ref[:3]):
            err = grad_rel_err(g[b, h], r)
            assert err <= TOL_GRAD_RELFRO, (nm, b, h, err)
    # every head and row
    assert_lse_bounds(lg, q, k, scale, w["causal"])
    vmin = v.min(axis=2, keepdims=True)
    vmax = v.max(axis=2, keepdims=True)
    slack = TOL_O_MAXABS + bf16_half_ulp(np.maximum(np.abs(vmin), np.abs(vmax)))
    assert np.all(og >= vmin - slack) and np.all(og <= vmax + slack)


def test_fp8_workload_every_head():
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
    scale = 1.0 / np.sqrt(w["d"])
    for h in range(w["H"]):
        rows = sampled_rows(w["N"], seed=77 + h, n_random=160)
        o_ref, lse_ref, _ = oracle.head_forward(q[0, h], k[0, h], v[0, h], scale, True, rows=rows)
        assert rel_fro(og[0, h][rows], o_ref) <= TOL_FP8_RELFRO, h
        assert max_abs(lg[0, h][rows], lse_ref) <= TOL_LSE_ABS, h
    assert_lse_bounds(lg, q, k, scale, True)
