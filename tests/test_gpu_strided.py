"""Strided layouts through attn_fwd_strided / attn_bwd_strided: [B, N, H, d]
tensors (the layout a fused QKV projection produces) and padded views, with
grouped heads and windows, against the oracle."""

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import make_inputs_gqa

from .helpers import (TOL_GRAD_RELFRO, TOL_LSE_ABS, TOL_O_MAXABS, bf16_out_err, bf16_to_device,
                      decoded, device_bf16_to_f64, device_f32_to_f64, max_abs, grad_rel_err)

pytestmark = pytest.mark.gpu


def to_bnhd(t):
    """[B, H, N, d] device tensor -> a [B, N, H, d] contiguous tensor."""
    return t.permute(0, 2, 1, 3).contiguous()


def from_bnhd(t):
    return t.permute(0, 2, 1, 3)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hk,N,window", [(4, 4, 300, (-1, -1)), (8, 2, 513, (-1, 0)),
                                           (4, 1, 200, (64, 16))])
def test_bnhd_layout_matches_oracle(H, Hk, N, window, d):
    B = 2
    inp = make_inputs_gqa(B, H, Hk, N, d, seed=H + Hk + N + d, with_grad=True)
    q, k, v, do = (to_bnhd(bf16_to_device(x)) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    o, lse = api.fwd_strided(q, k, v, layout="bnhd", window=window)
    dq, dk, dv = api.bwd_strided(q, k, v, o, do, lse, layout="bnhd", window=window)
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    assert o.shape == q.shape and dk.shape == k.shape
    qf, kf, vf, dof = decoded(inp)
    scale = 1.0 / np.sqrt(d)
    o_ref, lse_ref = oracle.forward_gqa(qf, kf, vf, scale, False, window=window)
    assert bf16_out_err(device_bf16_to_f64(from_bnhd(o)), o_ref) <= TOL_O_MAXABS
    assert max_abs(device_f32_to_f64(lse), lse_ref) <= TOL_LSE_ABS
    ref = oracle.backward_gqa(qf, kf, vf, dof, scale, False, window=window)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        err = grad_rel_err(device_bf16_to_f64(from_bnhd(g)), r)
        assert err <= TOL_GRAD_RELFRO, (name, err)


def test_padded_views_match_dense_call():
    """Q, K, V as column slices of one wider [B, N, 3, H, d] buffer (a packed QKV
    projection): the strided call must equal the dense call bit for bit."""
    import torch
    B, H, N, d = 1, 4, 384, 128
    inp = make_inputs_gqa(B, H, H, N, d, seed=7, with_grad=False)
    q, k, v = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits))
    qkv = torch.stack([to_bnhd(q), to_bnhd(k), to_bnhd(v)], dim=2)  # [B, N, 3, H, d]
    qv, kv_, vv = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    assert not qv.is_contiguous()
    o_s, lse_s = api.fwd_strided(qv, kv_, vv, layout="bnhd", window=(-1, 0))
    o_d, lse_d = api.fwd(q, k, v, causal=True)
    assert torch.equal(from_bnhd(o_s), o_d) and torch.equal(lse_s, lse_d)


def test_bad_strides_rejected():
    import torch
    q = torch.zeros(1, 128, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        api.fwd_strided(q[..., ::2], q[..., ::2], q[..., ::2], layout="bnhd")
