"""Forward parity: CUDA path vs the fp64 oracle, element by element, on seeded
inputs spanning several 128-row tiles, ragged tails and the degenerate N=1."""

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import AttnInputs, f32_to_bf16_bits, make_inputs

from .helpers import (bf16_out_err, TOL_LSE_ABS, TOL_O_MAXABS, bf16_to_device, decoded, device_bf16_to_f64,
                      device_f32_to_f64, max_abs)

pytestmark = pytest.mark.gpu

SHAPES = [1, 17, 128, 129, 255, 256, 257, 640, 1000]


def run_fwd(inp, causal, scale=None):
    q, k, v = (bf16_to_device(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits))
    o, lse = api.fwd(q, k, v, scale=scale, causal=causal)
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    return device_bf16_to_f64(o), device_f32_to_f64(lse)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", SHAPES)
def test_fwd_matches_oracle(N, d, causal):
    inp = make_inputs(1, 2, N, d, seed=N * 7 + d + int(causal))
    o, lse = run_fwd(inp, causal)
    q, k, v, _ = decoded(inp)
    o_ref, lse_ref = oracle.forward(q, k, v, 1.0 / np.sqrt(d), causal)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    assert bf16_out_err(o, o_ref) <= TOL_O_MAXABS, bf16_out_err(o, o_ref)
    assert max_abs(lse, lse_ref) <= TOL_LSE_ABS, max_abs(lse, lse_ref)


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_many_heads_and_batches(causal):
    inp = make_inputs(3, 5, 300, 64, seed=11)
    o, lse = run_fwd(inp, causal)
    q, k, v, _ = decoded(inp)
    o_ref, lse_ref = oracle.forward(q, k, v, 0.125, causal)
    assert bf16_out_err(o, o_ref) <= TOL_O_MAXABS
    assert max_abs(lse, lse_ref) <= TOL_LSE_ABS


def test_fwd_outlier_keys_exercise_rescale():
    """A few keys scaled x8 raise a row's scores far above its first tile's
    maximum mid-sequence: P exceeds 1 by up to about 2^35 on those tiles (bf16
    rows exponentiate against the stored maximum)."""
    inp = make_inputs(1, 4, 1024, 128, seed=3, outlier_frac=0.01, outlier_factor=8.0)
    o, lse = run_fwd(inp, False)
    q, k, v, _ = decoded(inp)
    o_ref, lse_ref = oracle.forward(q, k, v, 1.0 / np.sqrt(128), False)
    assert bf16_out_err(o, o_ref) <= TOL_O_MAXABS
    assert max_abs(lse, lse_ref) <= TOL_LSE_ABS


@pytest.mark.parametrize("scale", [0.02, 0.5])
def test_fwd_other_scales(scale):
    inp = make_inputs(1, 2, 384, 64, seed=5)
    o, lse = run_fwd(inp, True, scale=scale)
    q, k, v, _ = decoded(inp)
    o_ref, lse_ref = oracle.forward(q, k, v, scale, True)
    assert bf16_out_err(o, o_ref) <= TOL_O_MAXABS
    assert max_abs(lse, lse_ref) <= TOL_LSE_ABS


def test_fwd_is_deterministic():
    inp = make_inputs(1, 3, 700, 128, seed=9)
    a = run_fwd(inp, True)
    b = run_fwd(inp, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_fwd_identical_value_rows():
    """Every V row equal to v: O = v for any Q, K (up to bf16 rounding of v itself)."""
    inp = make_inputs(1, 2, 333, 64, seed=12)
    inp.v_bits[:] = inp.v_bits[:, :, :1, :]
    o, _ = run_fwd(inp, False)
    v = oracle.bf16_bits_to_f64(inp.v_bits)
    assert max_abs(o, v) <= 1e-2


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_score_jumps_redo_tiles(causal, d):
    """Keys that grow along a direction shared with the queries, so that a row's
    scores rise by tens of log2 units from one 128-key tile to the next: bf16
    tiles whose row sum against the stored maximum passes 2^60 are redone with
    their own maximum and the output is rescaled (d = 128: up to 7 redos per row,
    counted on the CPU with the same rule), and the tiles in between carry P up
    to about 2^58."""
    B, H, N = 1, 2, 1024
    rng = np.random.Generator(np.random.PCG64(31))
    base = rng.standard_normal(d).astype(np.float32)
    q = (base + 0.5 * rng.standard_normal((B, H, N, d))).astype(np.float32)
    ramp = (32.0 * np.arange(N) / N).astype(np.float32)[None, None, :, None]
    k = (ramp * base + 0.5 * rng.standard_normal((B, H, N, d))).astype(np.float32)
    v = rng.standard_normal((B, H, N, d)).astype(np.float32)
    inp = AttnInputs(B, H, N, d, f32_to_bf16_bits(q), f32_to_bf16_bits(k), f32_to_bf16_bits(v),
                     None, 31, None)
    o, lse = run_fwd(inp, causal)
    qd, kd, vd, _ = decoded(inp)
    o_ref, lse_ref = oracle.forward(qd, kd, vd, 1.0 / np.sqrt(d), causal)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    assert bf16_out_err(o, o_ref) <= TOL_O_MAXABS
    assert max_abs(lse, lse_ref) <= TOL_LSE_ABS, max_abs(lse, lse_ref)
