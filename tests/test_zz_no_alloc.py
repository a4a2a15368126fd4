"""attn_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (code handed only its input and output tensors by a framework that owns
all device memory).  It runs on a fixed scratch array inside the library.

Checked through the C ABI against attn_bwd (which takes a caller-allocated
workspace) on four calls in a row with different inputs and sizes -- a small
one, two that use nearly all of the 64 MiB scratch, then a small one again --
so that anything left in the shared scratch by an earlier call would show up
in a later one:
  * dK and dV come from the same deterministic kernels and must be
    bit-identical to attn_bwd's where the workspace layout of attn_bwd fits in
    the scratch (B1 H10 N8192, whose last round of key tiles is split into
    parts); where it does not (B1 H15 N8192) the call runs without the split
    last round, and the rows of those key tiles are summed in another order:
    compared within the rounding of their bf16 output;
  * dQ is summed by fp32 reductions in an order that may differ between the
    two calls, so it is compared within the rounding of its bf16 output;
  * all three gradients are also compared with the fp64 oracle.
This file is collected last so that a failure here cannot hide other tests; it
also passes when run alone in a fresh process."""

import ctypes

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import make_inputs

from .helpers import (TOL_GRAD_RELFRO, bf16_to_device, decoded, device_bf16_to_f64, grad_rel_err,
                      rel_fro)

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20


def _call_noalloc(lib, q, k, v, o, do, lse, causal):
    import torch
    B, H, N, d = q.shape
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    rc = lib.attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                              lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N,
                              d, 1.0 / np.sqrt(d), int(causal),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, api.STATUS_NAMES.get(rc, rc)
    return dq, dk, dv


# (B, H, N, d, oracle heads): the middle calls need 60 MiB (with the split last
# round's partials) and 61 MiB (without them) of scratch
CALLS = [(1, 3, 700, 128, None), (1, 10, 8192, 128, [(0, 9)]), (1, 15, 8192, 128, [(0, 7)]),
         (2, 2, 513, 64, None)]


@pytest.mark.parametrize("causal", [False, True])
def test_noalloc_matches_workspace_backward_three_calls(causal):
    lib = api.load_library()
    for call, (B, H, N, d, heads) in enumerate(CALLS):
        same_layout = lib.attn_bwd_workspace_bytes(B, H, N, d) <= SCRATCH_BYTES
        assert same_layout or (B, H, N, d) == (1, 15, 8192, 128)
        inp = make_inputs(B, H, N, d, seed=40 + call + 10 * int(causal), with_grad=True)
        q, k, v, do = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
        o, lse = api.fwd(q, k, v, causal=causal)
        ref = api.bwd(q, k, v, o, do, lse, causal=causal)
        got = _call_noalloc(lib, q, k, v, o, do, lse, causal)
        rc, site = api.check_device_error()
        assert rc == 0, f"device error {rc} at site {site:#x}"
        dq_g, dk_g, dv_g = (device_bf16_to_f64(t) for t in got)
        dq_r, dk_r, dv_r = (device_bf16_to_f64(t) for t in ref)
        if same_layout:
            assert np.array_equal(dk_g, dk_r), (call, "dk")
            assert np.array_equal(dv_g, dv_r), (call, "dv")
        else:
            assert rel_fro(dk_g, dk_r) <= 1e-3, (call, "dk", rel_fro(dk_g, dk_r))
            assert rel_fro(dv_g, dv_r) <= 1e-3, (call, "dv", rel_fro(dv_g, dv_r))
        assert rel_fro(dq_g, dq_r) <= 1e-4, (call, rel_fro(dq_g, dq_r))
        qd, kd, vd, dod = decoded(inp)
        scale = 1.0 / np.sqrt(d)
        if heads is None:
            refs = oracle.backward(qd, kd, vd, dod, scale, causal)
            for name, g, r in zip(("dq", "dk", "dv"), (dq_g, dk_g, dv_g), refs):
                assert grad_rel_err(g, r) <= TOL_GRAD_RELFRO, (call, name)
        else:
            for (b, h) in heads:
                refs = oracle.head_backward(qd[b, h], kd[b, h], vd[b, h], dod[b, h], scale, causal)
                for name, g, r in zip(("dq", "dk", "dv"), (dq_g, dk_g, dv_g), refs[:3]):
                    assert grad_rel_err(g[b, h], r) <= TOL_GRAD_RELFRO, (call, name, b, h)


def test_noalloc_rejects_problems_larger_than_its_scratch():
    lib = api.load_library()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size checks come first
    args = [fake] * 9
    # B*H*Npad*d*4 bytes for the fp32 accumulator alone exceeds 64 MiB here
    assert lib.attn_bwd_noalloc(*args, 1, 32, 8192, 128, 0.088, 0, None) == -2
    # an unsupported head dim gets attn_bwd's own status, before the size limit
    assert lib.attn_bwd_noalloc(*args, 1, 1, 128, 96, 0.1, 0, None) == -2
    # invalid sizes and flags: ATTN_ERR_INVALID, as attn_bwd
    assert lib.attn_bwd_noalloc(*args, 0, 1, 128, 128, 0.1, 0, None) == -1
    assert lib.attn_bwd_noalloc(*args, 1, 1, 128, 128, 0.1, 2, None) == -1
    assert lib.attn_bwd_noalloc(*args, 1, 1, 128, 128, -1.0, 0, None) == -1
