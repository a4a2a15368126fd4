"""Long sequences: two heads at N = 65499 (511 full 128-row tiles and a ragged
last one), forward and backward, with and without the causal mask.  The oracle
computes sampled query rows of O, LSE and dQ one by one (a row needs only its
own row of S, P and dP); every dK and dV element must be finite."""

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import make_inputs

from .helpers import (TOL_GRAD_RELFRO, TOL_LSE_ABS, TOL_O_MAXABS, bf16_out_err, bf16_to_device,
                      decoded, device_bf16_to_f64, device_f32_to_f64, max_abs, rel_fro)

pytestmark = pytest.mark.gpu

N_LONG = 65499
# first tile, a tile boundary, the middle, and the rows of the ragged last tile
ROWS = np.array([0, 1, 127, 128, 32749, 65370, 65497, 65498])


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_sampled_rows(causal):
    d = 128
    inp = make_inputs(1, 2, N_LONG, d, seed=4242 + int(causal), with_grad=True)
    q, k, v, do = (bf16_to_device(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    o, lse = api.fwd(q, k, v, causal=causal)
    dq, dk, dv = api.bwd(q, k, v, o, do, lse, causal=causal)
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    og, lg, dqg = device_bf16_to_f64(o), device_f32_to_f64(lse), device_bf16_to_f64(dq)
    assert np.all(np.isfinite(device_bf16_to_f64(dk))) and np.all(np.isfinite(device_bf16_to_f64(dv)))
    qd, kd, vd, dod = decoded(inp)
    scale = 1.0 / np.sqrt(d)
    for h in range(2):
        o_ref, lse_ref, _ = oracle.head_forward(qd[0, h], kd[0, h], vd[0, h], scale, causal, rows=ROWS)
        assert bf16_out_err(og[0, h][ROWS], o_ref) <= TOL_O_MAXABS, h
        assert max_abs(lg[0, h][ROWS], lse_ref) <= TOL_LSE_ABS, h
        dq_ref, _ = oracle.head_backward_rows(qd[0, h], kd[0, h], vd[0, h], dod[0, h], scale, causal,
                                              ROWS)
        err = rel_fro(dqg[0, h][ROWS], dq_ref)
        assert err <= TOL_GRAD_RELFRO, (h, err)
