"""The d = 128 backward's split items: the last round of a launch without a mask
(or its only round, with fewer items than SMs), and the longest items of causal
launches with grouped heads.

Split last round.  With G persistent CTAs and n = R G + r
key-tile items (0 < r, no mask), the last round's r items are dealt as
P = G / r parts each (contiguous ranges of their query steps); every part leaves
an fp32 dV/dK partial in the workspace and the last part to finish a 32-row slice
adds them up in part order.  These shapes put every kind of part on the GPU and
compare dQ, dK and dV with the fp64 oracle, block by block:
  * grouped heads, where a part's steps run across query heads of the group and
    may start inside one;
  * a ragged N, whose last key tile has rows past the sequence end;
  * fewer items than SMs, where every item is split.
The split also runs at B1 H32 N8192 d128 in the workload and invariant tests.

Causal grouped heads.  A key tile's item visits every query head of its group, so
causal items run from G n_q steps down to G; when the longest reach the per-CTA
mean, the host splits them in two and deals parts and whole items longest first
from per-CTA lists passed to the kernel (only when the longest item has at least
64 steps).  The causal shapes below take that path (one or two key/value heads,
ragged N included).

Causal head groups.  When the launch's Q, dO and fp32 dQ accumulator pass 64 MiB
and no item is split, the same per-CTA lists deal the items group by group of
key/value heads (longest first within a group); the grouped shapes below take
that path (grouped query heads and a ragged N included).

With 152 SMs (GB300) the shapes below split; on another SM count they may not,
and the comparison with the oracle holds either way."""

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import make_inputs_gqa

from .helpers import TOL_GRAD_RELFRO, bf16_to_device, decoded, device_bf16_to_f64, grad_rel_err

pytestmark = pytest.mark.gpu


def _run(B, H, Hk, N, seed, causal=False):
    inp = make_inputs_gqa(B, H, Hk, N, 128, seed=seed, with_grad=True)
    q, k, v, do = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    o, lse = api.fwd(q, k, v, causal=causal)
    grads = api.bwd(q, k, v, o, do, lse, causal=causal)
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    return inp, (q, k, v, o, do, lse), grads


# (B, H, Hk, N): items B*Hk*ceil(N/128) against 152 CTAs; a part keeps 16 steps
# at least (steps of an item: (H / Hk) * ceil(N/128))
SHAPES = [
    (2, 32, 8, 1280),    # 160 items of 40 steps: r = 8, P = 2 parts of 20
    (1, 20, 10, 2048),   # 160 items of 32 steps: r = 8, P = 2 parts of 16
    # fewer items than SMs: every item in parts, on P times as many CTAs
    (1, 1, 1, 4096),     # 32 items of 32 steps: P = 2
    (2, 24, 4, 1024),    # 64 items of 48 steps over 6 query heads: P = 2
    (1, 6, 1, 1536),     # 12 items of 72 steps: P = 4 parts of 18 (parts start mid-head)
    (1, 32, 4, 1000),    # 32 items of 64 steps, ragged last key tile: P = 4
]


@pytest.mark.parametrize("B,H,Hk,N", SHAPES)
def test_split_last_round_matches_oracle(B, H, Hk, N):
    inp, _, grads = _run(B, H, Hk, N, seed=B * 1000 + H * 10 + N)
    qf, kf, vf, dof = decoded(inp)
    ref = oracle.backward_gqa(qf, kf, vf, dof, 1.0 / np.sqrt(128), False)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        g = device_bf16_to_f64(g)
        assert np.all(np.isfinite(g)), name
        err = grad_rel_err(g, r)
        assert err <= TOL_GRAD_RELFRO, (name, err)


def test_split_last_round_is_deterministic():
    """dK and dV of split items are summed in part order, whichever part ends
    last: two calls give the same bits."""
    _, args, first = _run(2, 24, 4, 1024, seed=5)
    second = api.bwd(*args, causal=False)
    for name, a, b in zip(("dk", "dv"), first[1:], second[1:]):
        assert np.array_equal(device_bf16_to_f64(a), device_bf16_to_f64(b)), name


def test_split_last_round_bnhd_layout():
    """A split last round writing dK and dV through [B, N, H, d] strides (rows of
    a key tile 8 heads apart) with grouped heads: 2 x 4 kv heads x 20 key tiles
    = 160 items of 40 steps, the last 8 in 2 parts."""
    B, H, Hk, N = 2, 8, 4, 2560
    inp = make_inputs_gqa(B, H, Hk, N, 128, seed=606, with_grad=True)

    def to_bnhd(t):
        return t.permute(0, 2, 1, 3).contiguous()

    q, k, v, do = (to_bnhd(bf16_to_device(x)) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    o, lse = api.fwd_strided(q, k, v, layout="bnhd", window=(-1, -1))
    grads = api.bwd_strided(q, k, v, o, do, lse, layout="bnhd", window=(-1, -1))
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    qf, kf, vf, dof = decoded(inp)
    ref = oracle.backward_gqa(qf, kf, vf, dof, 1.0 / np.sqrt(128), False)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        err = grad_rel_err(device_bf16_to_f64(g.permute(0, 2, 1, 3)), r)
        assert err <= TOL_GRAD_RELFRO, (name, err)


# (B, H, Hk, N): causal, 16 / 64 / 11 items of up to 128 / 64 / 66 steps (items
# shorter than 64 steps are never dealt)
CAUSAL_SHAPES = [(1, 8, 1, 2048), (2, 8, 2, 2048), (1, 6, 1, 1400)]


@pytest.mark.parametrize("B,H,Hk,N", CAUSAL_SHAPES)
def test_causal_long_items_dealt_match_oracle(B, H, Hk, N):
    inp, _, grads = _run(B, H, Hk, N, seed=7000 + N + H, causal=True)
    qf, kf, vf, dof = decoded(inp)
    ref = oracle.backward_gqa(qf, kf, vf, dof, 1.0 / np.sqrt(128), True)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        g = device_bf16_to_f64(g)
        assert np.all(np.isfinite(g)), name
        err = grad_rel_err(g, r)
        assert err <= TOL_GRAD_RELFRO, (name, err)


def test_causal_dealt_is_deterministic():
    _, args, first = _run(2, 8, 2, 2048, seed=8, causal=True)
    second = api.bwd(*args, causal=True)
    for name, a, b in zip(("dk", "dv"), first[1:], second[1:]):
        assert np.array_equal(device_bf16_to_f64(a), device_bf16_to_f64(b)), name


def test_causal_dealt_full_size_mqa_batch0():
    """The dealt launch at full size, B4 H16 Hk1 N4096 causal (128 items of up to
    512 steps, the 80 longest split in two): every gradient of batch 0 (dQ of its
    16 query heads, dK and dV of its key/value head) against the oracle, block by
    block; the other batches' gradients finite."""
    B, H, Hk, N = 4, 16, 1, 4096
    inp, _, grads = _run(B, H, Hk, N, seed=4242, causal=True)
    qf, kf, vf, dof = decoded(inp)
    ref = oracle.backward_gqa(qf[:1], kf[:1], vf[:1], dof[:1], 1.0 / np.sqrt(128), True)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        g = device_bf16_to_f64(g)
        assert np.all(np.isfinite(g)), name
        err = grad_rel_err(g[:1], r)
        assert err <= TOL_GRAD_RELFRO, (name, err)


def _sweep_cases(n_cases, seed):
    """Seeded shapes around the split and deal thresholds of 152 SMs, ragged N:
    even cases without a mask (key-tile items = B * Hk * ceil(N/128) from a few
    dozen to a few hundred, items of (H/Hk) * ceil(N/128) steps from 8 to 160),
    odd cases causal with 8 or 16 query heads per key/value head (longest items
    of 64 steps or more, so that the deal is considered)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for i in range(n_cases):
        if i % 2 == 0:
            B = int(rng.integers(1, 3))
            Hk = int(rng.choice([1, 2, 4, 8]))
            G = int(rng.choice([1, 2, 4, 8]))
            N = int(rng.integers(300, 2561))
            causal = False
        else:
            B = 1
            Hk = int(rng.choice([1, 2]))
            G = int(rng.choice([8, 16]))
            N = int(rng.integers(1025, 2561))
            causal = True
        out.append((i, B, G * Hk, Hk, N, causal))
    return out


@pytest.mark.parametrize("case", _sweep_cases(16, 4077),
                         ids=lambda c: f"s{c[0]}-B{c[1]}H{c[2]}Hk{c[3]}N{c[4]}-{'causal' if c[5] else 'full'}")
def test_split_and_deal_sweep_matches_oracle(case):
    i, B, H, Hk, N, causal = case
    inp, _, grads = _run(B, H, Hk, N, seed=5000 + i, causal=causal)
    qf, kf, vf, dof = decoded(inp)
    ref = oracle.backward_gqa(qf, kf, vf, dof, 1.0 / np.sqrt(128), causal)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        g = device_bf16_to_f64(g)
        assert np.all(np.isfinite(g)), name
        err = grad_rel_err(g, r)
        assert err <= TOL_GRAD_RELFRO, (name, err)


def test_causal_head_groups_match_oracle():
    """B4 H8 Hk4 N2100 causal (16 key/value heads of 17 key tiles, items of 2 to
    34 steps, 71 MB of Q, dO and dQ accumulator): dealt in groups of key/value
    heads; every gradient of every head against the oracle, block by block."""
    B, H, Hk, N = 4, 8, 4, 2100
    inp, _, grads = _run(B, H, Hk, N, seed=9100, causal=True)
    qf, kf, vf, dof = decoded(inp)
    ref = oracle.backward_gqa(qf, kf, vf, dof, 1.0 / np.sqrt(128), True)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        err = grad_rel_err(device_bf16_to_f64(g), r)
        assert err <= TOL_GRAD_RELFRO, (name, err)


def test_causal_head_groups_ragged_heads_sampled():
    """B1 H16 N4500 causal (ragged last key tile, 74 MB): heads 0, 7 and 15 (the
    first and last groups and one between) against the oracle, block by block;
    every gradient finite."""
    B, H, N = 1, 16, 4500
    inp, _, grads = _run(B, H, H, N, seed=9200, causal=True)
    qf, kf, vf, dof = decoded(inp)
    heads = [0, 7, 15]
    ref = oracle.backward_gqa(qf[:, heads], kf[:, heads], vf[:, heads], dof[:, heads],
                              1.0 / np.sqrt(128), True)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        g = device_bf16_to_f64(g)
        assert np.all(np.isfinite(g)), name
        err = grad_rel_err(g[:, heads], r)
        assert err <= TOL_GRAD_RELFRO, (name, err)


def test_causal_head_groups_deterministic():
    _, args, first = _run(4, 8, 4, 2100, seed=11, causal=True)
    second = api.bwd(*args, causal=True)
    for name, a, b in zip(("dk", "dv"), first[1:], second[1:]):
        assert np.array_equal(device_bf16_to_f64(a), device_bf16_to_f64(b)), name


def test_causal_head_groups_full_size_sampled_heads():
    """B4 H32 N4096 causal: 4096 key-tile items (an 8192-entry deal table) in groups
    of 8 heads, 512 MB of Q, dO and dQ accumulator.  Heads (0, 0), (1, 13) and
    (3, 31) (first, middle and last group) against the oracle block by block; every
    gradient finite (checked on the device)."""
    import torch
    B, H, N = 4, 32, 4096
    inp, _, grads = _run(B, H, H, N, seed=9300, causal=True)
    for name, g in zip(("dq", "dk", "dv"), grads):
        assert bool(torch.isfinite(g.float()).all()), name
    scale = 1.0 / np.sqrt(128)
    for b, h in ((0, 0), (1, 13), (3, 31)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        q, k, v, do = (oracle.bf16_bits_to_f64(x[sl]) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
        ref = oracle.backward_gqa(q, k, v, do, scale, True)
        for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
            err = grad_rel_err(device_bf16_to_f64(g[sl]), r)
            assert err <= TOL_GRAD_RELFRO, (name, b, h, err)
