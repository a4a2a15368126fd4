"""The range-checked build (libattn_sm103a_debug.so, compiled with
ATTN_DEBUG_CHECKS): every TMA box coordinate and every tensor-memory access or
MMA operand address is checked on the device, and a failed check would skip
the access and set the device error word (never a trap).  Compute-sanitizer
is not available on this machine, so this build stands in for its memory
checker: the parity shapes below -- ragged tails, one-row problems, both
masks, both head dims, grouped heads, windows, split-KV, FP8 -- run through
every kernel of the debug library and must leave the error word clear and
still match the fp64 oracle."""

import contextlib

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import make_inputs, make_inputs_fp8, make_inputs_gqa

from .helpers import (TOL_FP8_RELFRO, TOL_GRAD_RELFRO, TOL_LSE_ABS, TOL_O_MAXABS, bf16_out_err,
                      bf16_to_device, decoded, decoded_fp8, device_bf16_to_f64, device_f32_to_f64,
                      grad_rel_err, max_abs, rel_fro, u8_to_device)

pytestmark = pytest.mark.gpu


@contextlib.contextmanager
def debug_library():
    """Route the binding's calls to the range-checked library for the block."""
    lib = api.load_library(api.DEBUG_LIB_PATH)
    assert lib.attn_build_flags() & 1, "debug library built without range checks"
    saved = api._lib
    api._lib = lib
    try:
        yield lib
    finally:
        api._lib = saved


def _assert_clean():
    rc, site = api.check_device_error()
    assert rc == 0, f"range check failed at site {site:#x} (status {rc})"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 300])
def test_debug_build_fwd_bwd(N, d, causal):
    inp = make_inputs(2, 2, N, d, seed=500 + N + d + int(causal), with_grad=True)
    with debug_library():
        q, k, v, do = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
        o, lse = api.fwd(q, k, v, causal=causal)
        dq, dk, dv = api.bwd(q, k, v, o, do, lse, causal=causal)
        _assert_clean()
    qf, kf, vf, dof = decoded(inp)
    scale = 1.0 / np.sqrt(d)
    o_ref, lse_ref = oracle.forward(qf, kf, vf, scale, causal)
    assert bf16_out_err(device_bf16_to_f64(o), o_ref) <= TOL_O_MAXABS
    assert max_abs(device_f32_to_f64(lse), lse_ref) <= TOL_LSE_ABS
    refs = oracle.backward(qf, kf, vf, dof, scale, causal)
    for g, r in zip((dq, dk, dv), refs):
        assert grad_rel_err(device_bf16_to_f64(g), r) <= TOL_GRAD_RELFRO


@pytest.mark.parametrize("window", [(64, 0), (1, 1), (-1, 100)])
def test_debug_build_grouped_heads_and_windows(window):
    inp = make_inputs_gqa(1, 4, 2, 513, 128, seed=77 + window[0], with_grad=True)
    with debug_library():
        q, k, v, do = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
        o, lse = api.fwd_window(q, k, v, *window)
        dq, dk, dv = api.bwd_window(q, k, v, o, do, lse, *window)
        _assert_clean()
    qf, kf, vf, dof = decoded(inp)
    scale = 1.0 / np.sqrt(128)
    o_ref, _ = oracle.forward_gqa(qf, kf, vf, scale, False, window=window)
    assert bf16_out_err(device_bf16_to_f64(o), o_ref) <= TOL_O_MAXABS
    refs = oracle.backward_gqa(qf, kf, vf, dof, scale, False, window=window)
    for g, r in zip((dq, dk, dv), refs):
        assert grad_rel_err(device_bf16_to_f64(g), r) <= TOL_GRAD_RELFRO


def test_debug_build_splitkv_and_fp8():
    import torch
    inp = make_inputs(1, 1, 1000, 128, seed=9)
    f8 = make_inputs_fp8(1, 2, 300, 128, seed=10)
    with debug_library() as lib:
        q, k, v = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits))
        ws = torch.empty(lib.attn_fwd_splitkv_workspace_bytes(1, 1, 1000, 128, 4), dtype=torch.uint8,
                         device="cuda")
        o, lse = api.fwd_splitkv(q, k, v, num_splits=4, workspace=ws)
        q8, k8, v8 = (u8_to_device(x) for x in (f8.q8, f8.k8, f8.v8))
        o8, _ = api.fwd_fp8(q8, k8, v8, f8.sq, f8.sk, f8.sv, causal=True)
        _assert_clean()
    qf, kf, vf, _ = decoded(inp)
    o_ref, _ = oracle.forward(qf, kf, vf, 1.0 / np.sqrt(128), False)
    assert bf16_out_err(device_bf16_to_f64(o), o_ref) <= TOL_O_MAXABS
    o8_ref, _ = oracle.forward(*decoded_fp8(f8), 1.0 / np.sqrt(128), True)
    assert rel_fro(device_bf16_to_f64(o8), o8_ref) <= TOL_FP8_RELFRO


def test_debug_build_split_last_round():
    """d = 128 without a mask, 160 key-tile items of 32 steps for 152 CTAs: the
    last round's 8 items are split into 2 parts each, whose partials meet in the
    workspace."""
    inp = make_inputs_gqa(1, 20, 10, 2048, 128, seed=91, with_grad=True)
    with debug_library():
        q, k, v, do = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
        o, lse = api.fwd(q, k, v, causal=False)
        dq, dk, dv = api.bwd(q, k, v, o, do, lse, causal=False)
        _assert_clean()
    qf, kf, vf, dof = decoded(inp)
    refs = oracle.backward_gqa(qf, kf, vf, dof, 1.0 / np.sqrt(128), False)
    for g, r in zip((dq, dk, dv), refs):
        assert grad_rel_err(device_bf16_to_f64(g), r) <= TOL_GRAD_RELFRO


def test_debug_build_causal_dealt():
    """Causal, one key/value head for 8 query heads at N = 2048: 16 items of up
    to 128 steps, each split in two and dealt from per-CTA lists."""
    inp = make_inputs_gqa(1, 8, 1, 2048, 128, seed=92, with_grad=True)
    with debug_library():
        q, k, v, do = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
        o, lse = api.fwd(q, k, v, causal=True)
        dq, dk, dv = api.bwd(q, k, v, o, do, lse, causal=True)
        _assert_clean()
    qf, kf, vf, dof = decoded(inp)
    refs = oracle.backward_gqa(qf, kf, vf, dof, 1.0 / np.sqrt(128), True)
    for g, r in zip((dq, dk, dv), refs):
        assert grad_rel_err(device_bf16_to_f64(g), r) <= TOL_GRAD_RELFRO
