"""Output rows that start on a 16-byte but not a 32-byte boundary.  The forward's
O rows and the backward's dK/dV rows go out as 32-byte stores when every row of
the output starts on a 32-byte boundary, else as 16-byte stores; the API asks
only for 16 bytes.  Outputs placed 16 bytes into an allocation take the second
path: their bits must equal those written to aligned outputs (the forward and
dK/dV are deterministic; dQ's fp32 summation order may differ run to run)."""

import numpy as np
import pytest

from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import make_inputs_fp8, make_inputs_gqa

from .helpers import bf16_to_device, rel_fro, u8_to_device

pytestmark = pytest.mark.gpu


def _offset_like(t, offset_elems=8):
    """An uninitialised tensor shaped like t whose data starts offset_elems
    elements (16 bytes for bf16) into its allocation."""
    import torch
    buf = torch.empty(t.numel() + offset_elems, dtype=t.dtype, device=t.device)
    return buf[offset_elems:].view(t.shape)


@pytest.mark.parametrize("d,causal,N", [(128, True, 1000), (128, False, 640), (64, False, 777)])
def test_forward_offset_output_matches_aligned(d, causal, N):
    import torch
    inp = make_inputs_gqa(2, 3, 3, N, d, seed=31 + d + N)
    q, k, v = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits))
    o_a, lse_a = api.fwd(q, k, v, causal=causal)
    o_off = _offset_like(o_a)
    assert o_off.data_ptr() % 32 == 16
    o_b, lse_b = api.fwd(q, k, v, causal=causal, o=o_off)
    assert torch.equal(o_a.view(torch.int16), o_b.view(torch.int16))
    assert torch.equal(lse_a, lse_b)


def test_fp8_forward_offset_output_matches_aligned():
    import torch
    inp = make_inputs_fp8(1, 2, 900, 128, seed=41)
    q8, k8, v8 = (u8_to_device(x) for x in (inp.q8, inp.k8, inp.v8))
    o_a, lse_a = api.fwd_fp8(q8, k8, v8, inp.sq, inp.sk, inp.sv, causal=True)
    o_off = _offset_like(o_a)
    o_b, lse_b = api.fwd_fp8(q8, k8, v8, inp.sq, inp.sk, inp.sv, causal=True, o=o_off)
    assert torch.equal(o_a.view(torch.int16), o_b.view(torch.int16))
    assert torch.equal(lse_a, lse_b)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_offset_dk_dv_match_aligned(causal):
    import torch
    B, H, N, d = 2, 4, 1000, 128
    inp = make_inputs_gqa(B, H, H, N, d, seed=51, with_grad=True)
    q, k, v, do = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    o, lse = api.fwd(q, k, v, causal=causal)
    dq_a, dk_a, dv_a = api.bwd(q, k, v, o, do, lse, causal=causal)
    dk_off, dv_off = _offset_like(dk_a), _offset_like(dv_a)
    assert dk_off.data_ptr() % 32 == 16 and dv_off.data_ptr() % 32 == 16
    dq_b, dk_b, dv_b = api.bwd(q, k, v, o, do, lse, causal=causal, dk=dk_off, dv=dv_off)
    assert torch.equal(dk_a.view(torch.int16), dk_b.view(torch.int16))
    assert torch.equal(dv_a.view(torch.int16), dv_b.view(torch.int16))
    assert rel_fro(dq_b.float().cpu().numpy().astype(np.float64),
                   dq_a.float().cpu().numpy().astype(np.float64)) < 1e-2
