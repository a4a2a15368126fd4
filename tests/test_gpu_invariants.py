"""Properties of attention that hold at any size, checked at N = 8192 (d = 128,
eight heads: 512 backward CTAs and 128 forward items, several waves), where
the oracle can afford only sampled rows:

* a joint permutation of the key and value rows leaves O, LSE and dQ
  unchanged and permutes dK and dV the same way (no mask: the sum over keys
  does not depend on their order);
* Q = 0 makes every score 0, so P is uniform over the visible keys and the
  results have closed forms in V and dO alone:
  O_i = mean of the visible V rows, LSE_i = ln(#visible keys),
  dK = 0, dV_j = sum over the rows i that see key j of dO_i / n_i, and
  dQ_i = scale * (1/n_i) sum_j (dO_i . (V_j - O_i)) K_j over the visible j;
* value rows that are all equal to one vector v give O_i = v for any Q, K;
* two runs on the same inputs give bit-identical O, LSE, dK and dV (dQ is
  summed by fp32 reductions whose order may change: compared within the
  rounding of its bf16 output).
The closed forms are evaluated here in fp64 from the definitions; they share
nothing with the CUDA path."""

import numpy as np
import pytest

from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import f32_to_bf16_bits, make_inputs

from .helpers import (TOL_GRAD_RELFRO, TOL_LSE_ABS, TOL_O_MAXABS, bf16_out_err, bf16_to_device,
                      decoded, device_bf16_to_f64, device_f32_to_f64, grad_rel_err, max_abs, rel_fro)

pytestmark = pytest.mark.gpu

B, H, N, D = 1, 8, 8192, 128
SCALE = 1.0 / np.sqrt(D)


def _run(q_bits, k_bits, v_bits, do_bits, causal):
    q, k, v, do = (bf16_to_device(x) for x in (q_bits, k_bits, v_bits, do_bits))
    o, lse = api.fwd(q, k, v, scale=SCALE, causal=causal)
    dq, dk, dv = api.bwd(q, k, v, o, do, lse, scale=SCALE, causal=causal)
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    return (device_bf16_to_f64(o), device_f32_to_f64(lse), device_bf16_to_f64(dq),
            device_bf16_to_f64(dk), device_bf16_to_f64(dv))


@pytest.fixture(scope="module")
def inputs():
    return make_inputs(B, H, N, D, seed=8192, with_grad=True)


def test_key_value_permutation_equivariance(inputs):
    rng = np.random.Generator(np.random.PCG64(3))
    perm = rng.permutation(N)
    a = _run(inputs.q_bits, inputs.k_bits, inputs.v_bits, inputs.do_bits, False)
    b = _run(inputs.q_bits, inputs.k_bits[:, :, perm], inputs.v_bits[:, :, perm], inputs.do_bits,
             False)
    o_a, lse_a, dq_a, dk_a, dv_a = a
    o_b, lse_b, dq_b, dk_b, dv_b = b
    # each run is within the tolerance of the exact result, so they are within
    # twice of each other (O: beyond the output rounding of both)
    assert bf16_out_err(o_b, o_a) <= 2 * TOL_O_MAXABS + float(np.max(_half_ulp(o_a)))
    assert max_abs(lse_b, lse_a) <= 2 * TOL_LSE_ABS
    assert grad_rel_err(dq_b, dq_a) <= 2 * TOL_GRAD_RELFRO
    # dK, dV of the permuted run, row p, belong to original key perm[p]
    assert grad_rel_err(dk_b, dk_a[:, :, perm]) <= 2 * TOL_GRAD_RELFRO
    assert grad_rel_err(dv_b, dv_a[:, :, perm]) <= 2 * TOL_GRAD_RELFRO


def _half_ulp(x):
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 0.5 * 2.0 ** (e - 7), 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_closed_forms(inputs, causal):
    zero = np.zeros_like(inputs.q_bits)  # bf16 +0.0
    o, lse, dq, dk, dv = _run(zero, inputs.k_bits, inputs.v_bits, inputs.do_bits, causal)
    _, k, v, do = decoded(inputs)
    n = np.arange(1, N + 1, dtype=np.float64) if causal else np.full(N, float(N))
    if causal:
        o_ref = np.cumsum(v, axis=2) / n[:, None]
    else:
        o_ref = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
    assert bf16_out_err(o, o_ref) <= TOL_O_MAXABS
    assert max_abs(lse, np.broadcast_to(np.log(n), lse.shape)) <= TOL_LSE_ABS
    assert np.all(dk == 0.0)
    # dV_j = sum_{i sees j} dO_i / n_i
    w = do / n[:, None]
    if causal:
        dv_ref = np.flip(np.cumsum(np.flip(w, axis=2), axis=2), axis=2)
    else:
        dv_ref = np.broadcast_to(w.sum(axis=2, keepdims=True), do.shape)
    assert grad_rel_err(dv, dv_ref) <= TOL_GRAD_RELFRO
    # dQ_i = scale / n_i * sum_{j visible} (dO_i . (V_j - O_i)) K_j
    #      = scale / n_i * (sum_j K_j V_j^T - (sum_j K_j) O_i^T) dO_i   (visible j)
    dq_ref = np.empty_like(do)
    for b in range(B):
        for h in range(H):
            kk, vv, dd = k[b, h], v[b, h], do[b, h]
            if causal:
                # running sums over the keys j <= i
                acc = np.zeros((D, D))
                ksum = np.zeros(D)
                for i in range(N):
                    acc += np.outer(kk[i], vv[i])
                    ksum += kk[i]
                    dq_ref[b, h, i] = SCALE / n[i] * ((acc - np.outer(ksum, o_ref[b, h, i])) @ dd[i])
            else:
                m = kk.T @ vv - np.outer(kk.sum(axis=0), o_ref[b, h, 0])
                dq_ref[b, h] = SCALE / N * (dd @ m.T)
    assert grad_rel_err(dq, dq_ref) <= TOL_GRAD_RELFRO


def test_identical_value_rows(inputs):
    import oracle
    rng = np.random.Generator(np.random.PCG64(11))
    vrow = rng.standard_normal((B, H, 1, D), dtype=np.float32)
    v_bits = np.ascontiguousarray(np.broadcast_to(f32_to_bf16_bits(vrow), inputs.v_bits.shape))
    o, _, _, _, dv = _run(inputs.q_bits, inputs.k_bits, v_bits, inputs.do_bits, False)
    assert bf16_out_err(o, oracle.bf16_bits_to_f64(v_bits)) <= TOL_O_MAXABS
    assert np.all(np.isfinite(dv))


@pytest.mark.parametrize("causal", [False, True])
def test_run_to_run_bitwise(inputs, causal):
    a = _run(inputs.q_bits, inputs.k_bits, inputs.v_bits, inputs.do_bits, causal)
    b = _run(inputs.q_bits, inputs.k_bits, inputs.v_bits, inputs.do_bits, causal)
    for nm, x, y in zip(("o", "lse", "dk", "dv"), (a[0], a[1], a[3], a[4]), (b[0], b[1], b[3], b[4])):
        assert np.array_equal(x, y), nm
    assert rel_fro(a[2], b[2]) <= 1e-4  # dQ: fp32 reduction order only
