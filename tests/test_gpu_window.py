"""Sliding-window attention (attn_fwd_window / attn_bwd_window): key j visible
to query i iff i - left <= j <= i + right.  Forward and backward against the
oracle's window mask, including windows narrower than a tile, windows that
span several tiles, one-sided windows and grouped heads."""

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import make_inputs_gqa

from .helpers import (TOL_GRAD_RELFRO, TOL_LSE_ABS, TOL_O_MAXABS, bf16_out_err, bf16_to_device,
                      decoded, device_bf16_to_f64, device_f32_to_f64, max_abs, grad_rel_err)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("window", [(64, 0), (200, 50), (0, 0), (-1, 100), (300, -1), (-1, 0),
                                    (1, 1)])
@pytest.mark.parametrize("N,H,Hk", [(700, 2, 2), (513, 4, 2)])
def test_window_fwd_bwd_match_oracle(window, N, H, Hk, d):
    inp = make_inputs_gqa(1, H, Hk, N, d, seed=N + d + window[0] + 3 * window[1], with_grad=True)
    q, k, v, do = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    o, lse = api.fwd_window(q, k, v, *window)
    dq, dk, dv = api.bwd_window(q, k, v, o, do, lse, *window)
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    qf, kf, vf, dof = decoded(inp)
    scale = 1.0 / np.sqrt(d)
    o_ref, lse_ref = oracle.forward_gqa(qf, kf, vf, scale, False, window=window)
    assert bf16_out_err(device_bf16_to_f64(o), o_ref) <= TOL_O_MAXABS
    assert max_abs(device_f32_to_f64(lse), lse_ref) <= TOL_LSE_ABS
    ref = oracle.backward_gqa(qf, kf, vf, dof, scale, False, window=window)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        err = grad_rel_err(device_bf16_to_f64(g), r)
        assert err <= TOL_GRAD_RELFRO, (name, err)


def test_window_rejects_bounds_below_minus_one():
    import torch
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.AttnError):
        api.fwd_window(q, q, q, -2, 0)
