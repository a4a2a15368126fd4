"""attn_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (code handed only its input and output tensors by a framework that owns
all device memory).  It runs on a fixed scratch array inside the library.

Checked through the C ABI against attn_bwd (which takes a caller-allocated
workspace) on two calls in a row with different inputs, so that anything left
in the shared scratch by the first call would show up in the second.  This
file is collected last so that a failure here cannot hide other tests; it also
passes when run alone in a fresh process."""

import ctypes

import numpy as np
import pytest

from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import make_inputs

from .helpers import TOL_GRAD_RELFRO, bf16_to_device, device_bf16_to_f64, rel_fro

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("causal", [False, True])
def test_noalloc_matches_workspace_backward_twice(causal):
    lib = api.load_library()
    for call, (B, H, N, d) in enumerate([(1, 3, 700, 128), (2, 2, 513, 64)]):
        inp = make_inputs(B, H, N, d, seed=40 + call, with_grad=True)
        q, k, v, do = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
        o, lse = api.fwd(q, k, v, causal=causal)
        ref = api.bwd(q, k, v, o, do, lse, causal=causal)
        got = _call_noalloc(lib, q, k, v, o, do, lse, causal)
        rc, site = api.check_device_error()
        assert rc == 0, f"device error {rc} at site {site:#x}"
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            err = rel_fro(device_bf16_to_f64(g), device_bf16_to_f64(r))
            assert err <= TOL_GRAD_RELFRO, (call, name, err)


def test_noalloc_rejects_problems_larger_than_its_scratch():
    lib = api.load_library()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    args = [fake] * 9
    # B*H*Npad*d*4 bytes for the fp32 accumulator alone exceeds 64 MiB here
    assert lib.attn_bwd_noalloc(*args, 1, 32, 8192, 128, 0.088, 0, None) == -2
