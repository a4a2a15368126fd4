"""Grouped-query attention (Hk key/value heads shared by H query heads, MQA when
Hk = 1): forward and backward through attn_fwd_gqa / attn_bwd_gqa against the
oracle's grouped forward and backward."""

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import make_inputs_gqa

from .helpers import (TOL_GRAD_RELFRO, TOL_LSE_ABS, TOL_O_MAXABS, bf16_out_err, bf16_to_device,
                      decoded, device_bf16_to_f64, device_f32_to_f64, max_abs, grad_rel_err)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hk,N", [(8, 2, 300), (4, 1, 257), (6, 3, 128), (4, 4, 200)])
def test_gqa_fwd_bwd_match_oracle(H, Hk, N, d, causal):
    B = 2
    inp = make_inputs_gqa(B, H, Hk, N, d, seed=H * 10 + Hk + N + d, with_grad=True)
    q, k, v, do = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    o, lse = api.fwd(q, k, v, causal=causal)
    dq, dk, dv = api.bwd(q, k, v, o, do, lse, causal=causal)
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    assert tuple(dk.shape) == (B, Hk, N, d) and tuple(dv.shape) == (B, Hk, N, d)
    qf, kf, vf, dof = decoded(inp)
    scale = 1.0 / np.sqrt(d)
    o_ref, lse_ref = oracle.forward_gqa(qf, kf, vf, scale, causal)
    assert bf16_out_err(device_bf16_to_f64(o), o_ref) <= TOL_O_MAXABS
    assert max_abs(device_f32_to_f64(lse), lse_ref) <= TOL_LSE_ABS
    ref = oracle.backward_gqa(qf, kf, vf, dof, scale, causal)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        err = grad_rel_err(device_bf16_to_f64(g), r)
        assert err <= TOL_GRAD_RELFRO, (name, err)


def test_gqa_rejects_bad_grouping():
    import torch
    q = torch.zeros(1, 6, 128, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 4, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.AttnError):
        api.fwd(q, k, k)
