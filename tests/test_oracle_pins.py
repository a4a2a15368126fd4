"""Pins for the fp64 oracle: it is checked against facts fixed by the pages and
by mathematics, never against itself or the CUDA path.

* online-softmax merge identity (FlashAttention digest, section 2: running max
  and running sum of exponentials of two halves combine to the full softmax);
* every row of P sums to one; Q = 0 gives column (prefix) means of V and
  LSE = ln(#visible keys); identical V rows are returned unchanged;
* N = 1 and N = 2 closed forms (the N = 2 case is a logistic sigmoid);
* brute force with Python floats and ``math.fsum`` on tiny shapes;
* finite differences of L = sum(dO * O) against the analytic backward;
* D_i = sum_j P_ij dP_ij equals sum_k dO_ik O_ik (the identity the GPU's
  backward preprocess relies on);
* invariance of (O, LSE) under a joint permutation of K and V rows;
* the README's 5-query / 2-key bottom-right causal example (golden file);
* bf16 and E4M3 decoders against PyTorch's own conversions;
* the FLOP convention against the FlashAttention-3 ablation table and the
  H200 scalar-kernel sweep (golden files).
Each pin is chosen so that a plausible mistake (dropped scale, wrong sign,
transposed operand, off-by-one mask) fails at least one of them; the
mutation tests at the end plant such mistakes and check that they are caught.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand(shape, seed):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


# ---------------------------------------------------------------------------
# Forward pins
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_P_sum_to_one(causal):
    q, k = rand((37, 16), 1), rand((37, 16), 2)
    p, lse = A.softmax_rows(A.scores(q, k, 0.3, causal))
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    assert np.all(p >= 0)
    if causal:
        assert np.all(p[np.triu_indices(37, 1)] == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_merge_identity_equals_full_softmax(causal):
    """Split the keys into two random halves, run the oracle on each half and
    combine (O, LSE) with the running-max / running-sum rule; the result must be
    the oracle on all keys."""
    N, d = 48, 8
    q, k, v = rand((N, d), 3), rand((N, d), 4), rand((N, d), 5)
    scale = 0.7
    perm = np.random.Generator(np.random.PCG64(6)).permutation(N)
    h1, h2 = np.sort(perm[: N // 2]), np.sort(perm[N // 2:])
    vis = A.causal_visible(N, N) if causal else np.ones((N, N), bool)

    def half(idx):
        s = scale * (q @ k[idx].T)
        s = np.where(vis[:, idx], s, -np.inf)
        p, lse = A.softmax_rows(s)
        # a half with no visible key has running sum 0: log-sum-exp -inf
        return p @ v[idx], np.where(np.isposinf(lse), -np.inf, lse)

    o1, l1 = half(h1)
    o2, l2 = half(h2)
    o_full, lse_full, _ = A.head_forward(q, k, v, scale, causal)
    # m(x) = max(m1, m2); l(x) = e^{m1-m} l1 + e^{m2-m} l2 with l_i = e^{LSE_i - m_i}
    m = np.maximum(l1, l2)
    m = np.where(np.isfinite(m), m, 0.0)
    w1 = np.exp(l1 - m)
    w2 = np.exp(l2 - m)
    lse_merged = m + np.log(w1 + w2)
    o_merged = (w1[:, None] * o1 + w2[:, None] * o2) / (w1 + w2)[:, None]
    assert np.all(np.isfinite(o_merged))
    np.testing.assert_allclose(lse_merged, lse_full, rtol=0, atol=1e-13)
    np.testing.assert_allclose(o_merged, o_full, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_column_means(causal):
    N, d = 33, 8
    q = np.zeros((N, d))
    k, v = rand((N, d), 7), rand((N, d), 8)
    o, lse, _ = A.head_forward(q, k, v, 0.25, causal)
    if causal:
        expect = np.cumsum(v, axis=0) / np.arange(1, N + 1)[:, None]
        np.testing.assert_allclose(lse, np.log(np.arange(1, N + 1)), atol=1e-14)
    else:
        expect = np.broadcast_to(v.mean(axis=0), (N, d))
        np.testing.assert_allclose(lse, np.log(N), atol=1e-14)
    np.testing.assert_allclose(o, expect, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_value_rows_are_returned(causal):
    N, d = 29, 8
    q, k = rand((N, d), 9), rand((N, d), 10)
    row = rand((d,), 11)
    v = np.tile(row, (N, 1))
    o, _, _ = A.head_forward(q, k, v, 1.3, causal)
    np.testing.assert_allclose(o, np.broadcast_to(row, (N, d)), atol=1e-13)


def test_single_key_closed_form():
    q, k, v = rand((1, 8), 12), rand((1, 8), 13), rand((1, 8), 14)
    o, lse, _ = A.head_forward(q, k, v, 0.4, False)
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, 0.4 * float(q[0] @ k[0]), atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_two_keys_is_a_sigmoid(causal):
    q, k, v = rand((2, 8), 15), rand((2, 8), 16), rand((2, 8), 17)
    scale = 0.9
    o, lse, _ = A.head_forward(q, k, v, scale, causal)
    for i in range(2):
        s0, s1 = scale * q[i] @ k[0], scale * q[i] @ k[1]
        if causal and i == 0:
            np.testing.assert_allclose(o[0], v[0], atol=1e-15)
            np.testing.assert_allclose(lse[0], s0, atol=1e-14)
            continue
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        np.testing.assert_allclose(o[i], w0 * v[0] + (1 - w0) * v[1], atol=1e-14)
        np.testing.assert_allclose(lse[i], max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))),
                                   atol=1e-14)


def brute_force_forward(q, k, v, scale, causal):
    """Pure-Python definition: visible scores, exp, fsum, divide, weighted fsum."""
    nq, nk, d = len(q), len(k), len(v[0])
    o = [[0.0] * d for _ in range(nq)]
    lse = [0.0] * nq
    for i in range(nq):
        vis = [j for j in range(nk) if (not causal) or j <= i + (nk - nq)]
        if not vis:
            lse[i] = math.inf
            continue
        s = {j: scale * math.fsum(q[i][t] * k[j][t] for t in range(len(q[i]))) for j in vis}
        mx = max(s.values())
        e = {j: math.exp(s[j] - mx) for j in vis}
        z = math.fsum(e.values())
        lse[i] = mx + math.log(z)
        for c in range(d):
            o[i][c] = math.fsum(e[j] * v[j][c] for j in vis) / z
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("nq,nk,causal", [(5, 5, False), (9, 9, True), (16, 16, True),
                                          (7, 3, True), (3, 7, True), (16, 11, False)])
def test_brute_force_tiny(nq, nk, causal):
    d = 6
    q, k, v = rand((nq, d), 20 + nq), rand((nk, d), 40 + nk), rand((nk, 5), 60 + nk)
    o_bf, lse_bf = brute_force_forward(q.tolist(), k.tolist(), v.tolist(), 0.37, causal)
    o, lse, _ = A.head_forward(q, k, v, 0.37, causal)
    np.testing.assert_allclose(o, o_bf, atol=1e-13)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(lse_bf))
    fin = np.isfinite(lse_bf)
    np.testing.assert_allclose(lse[fin], lse_bf[fin], atol=1e-13)


def test_causal_bottom_right_golden():
    spec = {}
    mask = []
    with open(os.path.join(GOLDEN, "causal_bottom_right_5q2k.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "mask":
                mask.append([int(x) for x in vals])
            else:
                spec[key] = [int(x) for x in vals]
    nq, nk = spec["nq"][0], spec["nk"][0]
    np.testing.assert_array_equal(A.causal_visible(nq, nk), np.array(mask, bool))
    q, k, v = rand((nq, 4), 70), rand((nk, 4), 71), rand((nk, 4), 72)
    o, lse, _ = A.head_forward(q, k, v, 0.5, True)
    for r in spec["zero_rows"]:
        assert np.all(o[r] == 0.0) and lse[r] == np.inf
    assert np.all(np.isfinite(o)) and not np.any(np.isnan(lse))
    np.testing.assert_allclose(o[3], v[0], atol=1e-15)  # one visible key


def test_permutation_equivariance():
    N, d = 40, 8
    q, k, v = rand((N, d), 80), rand((N, d), 81), rand((N, d), 82)
    perm = np.random.Generator(np.random.PCG64(83)).permutation(N)
    o1, l1, _ = A.head_forward(q, k, v, 0.5, False)
    o2, l2, _ = A.head_forward(q, k[perm], v[perm], 0.5, False)
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(l1, l2, atol=1e-14)


def test_batched_forward_matches_per_head_and_sampled_rows():
    B, H, N, d = 2, 3, 20, 8
    q, k, v = rand((B, H, N, d), 90), rand((B, H, N, d), 91), rand((B, H, N, d), 92)
    o, lse = oracle.forward(q, k, v, 0.3, True)
    rows = np.array([0, 7, 19])
    sampled = oracle.forward(q, k, v, 0.3, True, heads=[(1, 2)], rows=rows)
    o_s, lse_s = sampled[(1, 2)]
    np.testing.assert_array_equal(o_s, o[1, 2][rows])
    np.testing.assert_array_equal(lse_s, lse[1, 2][rows])


# ---------------------------------------------------------------------------
# Backward pins
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(6, 6), (8, 8), (5, 3)])
def test_backward_matches_finite_differences(causal, nq, nk):
    d = 4
    q, k, v = rand((nq, d), 100), rand((nk, d), 101), rand((nk, 3), 102)
    do = rand((nq, 3), 103)
    scale = 0.8
    dq, dk, dv, _ = A.head_backward(q, k, v, do, scale, causal)

    def loss(qq, kk, vv):
        o, _, _ = A.head_forward(qq, kk, vv, scale, causal)
        return float(np.sum(do * o))

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"])
                        - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        err = np.linalg.norm(num - g) / max(np.linalg.norm(num), 1e-300)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_rows_match_finite_differences(causal):
    """dQ of selected rows against central differences of L = sum(dO * O) in
    those rows of Q (one is the first row, which sees a single key when causal)."""
    nq, nk, d = 9, 9, 4
    q, k, v = rand((nq, d), 130), rand((nk, d), 131), rand((nk, 3), 132)
    do = rand((nq, 3), 133)
    scale = 0.7
    rows = np.array([0, 4, 8])
    dq_rows, _ = A.head_backward_rows(q, k, v, do, scale, causal, rows)

    def loss(qq):
        o, _, _ = A.head_forward(qq, k, v, scale, causal)
        return float(np.sum(do * o))

    h = 1e-6
    num = np.zeros((len(rows), d))
    for a, i in enumerate(rows):
        for c in range(d):
            qp, qm = q.copy(), q.copy()
            qp[i, c] += h
            qm[i, c] -= h
            num[a, c] = (loss(qp) - loss(qm)) / (2 * h)
    err = np.linalg.norm(num - dq_rows) / np.linalg.norm(num)
    assert err < 1e-6, err


def test_backward_rows_agree_with_full_backward():
    N, d = 40, 8
    q, k, v, do = (rand((N, d), s) for s in (140, 141, 142, 143))
    dq, _, _, dsum = A.head_backward(q, k, v, do, 0.4, True, window=(6, 0))
    rows = np.array([0, 7, 39])
    dq_rows, d_rows = A.head_backward_rows(q, k, v, do, 0.4, True, rows, window=(6, 0))
    np.testing.assert_allclose(dq_rows, dq[rows], rtol=0, atol=1e-13)
    np.testing.assert_allclose(d_rows, dsum[rows], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_D_identity(causal):
    N, d = 30, 8
    q, k, v, do = (rand((N, d), s) for s in (110, 111, 112, 113))
    o, _, _ = A.head_forward(q, k, v, 0.6, causal)
    _, _, _, dsum = A.head_backward(q, k, v, do, 0.6, causal)
    np.testing.assert_allclose(dsum, np.sum(do * o, axis=1), atol=1e-12)


def test_batched_backward_matches_per_head():
    B, H, N, d = 1, 2, 12, 4
    q, k, v, do = (rand((B, H, N, d), s) for s in (120, 121, 122, 123))
    dq, dk, dv = oracle.backward(q, k, v, do, 0.5, True)
    per = oracle.backward(q, k, v, do, 0.5, True, heads=[(0, 1)])
    for a, b in zip((dq[0, 1], dk[0, 1], dv[0, 1]), per[(0, 1)]):
        np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------------------
# Storage decoders
# ---------------------------------------------------------------------------


def test_bf16_decoder_matches_torch():
    torch = pytest.importorskip("torch")
    bits = np.arange(0, 1 << 16, 7, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = A.bf16_bits_to_f64(bits)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert np.all(same)


def test_e4m3_decoder_matches_torch_on_all_codes():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = A.e4m3_to_f64(codes)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert np.all(same)
    # OCP E4M3: 0x7E is the largest finite value, 0x01 the smallest subnormal.
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF]) and got[0xB8] == -1.0


def test_input_packing_round_trips():
    from exact_attention_52_gb300 import inputs as I
    inp = I.make_inputs(1, 2, 33, 8, seed=0, with_grad=True, outlier_frac=0.1)
    q = A.bf16_bits_to_f64(inp.q_bits)
    assert q.shape == (1, 2, 33, 8) and np.all(np.isfinite(q))
    # outlier rows are exactly 8x the bf16 value they would otherwise have had
    inp0 = I.make_inputs(1, 2, 33, 8, seed=0, with_grad=True)
    k0 = A.bf16_bits_to_f64(inp0.k_bits).reshape(2, 33, 8)
    k1 = A.bf16_bits_to_f64(inp.k_bits).reshape(2, 33, 8)
    for bh in range(2):
        rows = inp.outlier_rows[bh]
        assert len(rows) == round(0.1 * 33)
        np.testing.assert_array_equal(k1[bh, rows], 8.0 * k0[bh, rows])
        rest = np.setdiff1d(np.arange(33), rows)
        np.testing.assert_array_equal(k1[bh, rest], k0[bh, rest])
    f8 = I.make_inputs_fp8(1, 1, 50, 16, seed=0)
    x = A.e4m3_to_f64(f8.q8, f8.sq)
    assert np.all(np.isfinite(x)) and abs(np.max(np.abs(x)) - 448.0 * f8.sq) < 1e-6


# ---------------------------------------------------------------------------
# FLOP convention (host logic used by the benchmark)
# ---------------------------------------------------------------------------


def test_flop_convention_reproduces_fa3_table2():
    from exact_attention_52_gb300.roofline import attn_flops
    g = json.load(open(os.path.join(GOLDEN, "fa3_table2_ablation.json")))
    w = g["workload"]
    for row in g["rows"]:
        tf = attn_flops(w["B"], w["H"], w["N"], w["d"], w["causal"]) / (row["ms"] * 1e-3) / 1e12
        assert abs(tf - row["tflops"]) < 1.0, (row, tf)


def test_flop_convention_reproduces_h200_sweep():
    from exact_attention_52_gb300.roofline import attn_flops
    g = json.load(open(os.path.join(GOLDEN, "h200_scalar_sweep.json")))
    w = g["workload"]
    f = attn_flops(w["B"], w["H"], w["N"], w["d"], w["causal"])
    for row in g["rows"]:
        gf = f / (row["ms"] * 1e-3) / 1e9
        assert abs(gf / row["gflops"] - 1.0) < 4e-3, (row, gf)


# ---------------------------------------------------------------------------
# Mutation checks: plant a mistake in a copy of the oracle, on the CPU, and
# check that the pins above would have caught it.
# ---------------------------------------------------------------------------


def _mutant_forward(kind):
    def fwd(q, k, v, scale, causal):
        if kind == "transposed_k":
            s = scale * (q @ k)  # wrong operand orientation (square d == N case)
        elif kind == "scale_missing_in_lse":
            s = q @ k.T
        else:
            s = scale * (q @ k.T)
        if causal:
            shift = 1 if kind == "mask_off_by_one" else 0
            s = np.where(A.causal_visible(len(q), len(k)) | (np.eye(len(q), len(k), shift) > 0),
                         s, -np.inf) if shift else np.where(A.causal_visible(len(q), len(k)), s, -np.inf)
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        p = e / e.sum(axis=1)[:, None]
        if kind == "scale_missing_in_lse":
            p = np.exp(scale * s - (scale * s).max(1)[:, None])
            p /= p.sum(1)[:, None]
        lse = m + np.log(e.sum(axis=1))
        return p @ v, lse
    return fwd


@pytest.mark.parametrize("kind", ["transposed_k", "scale_missing_in_lse", "mask_off_by_one"])
def test_pins_catch_planted_mistakes(kind):
    fwd = _mutant_forward(kind)
    d = N = 8
    q, k, v = rand((N, d), 130), rand((N, d), 131), rand((N, d), 132)
    causal = kind == "mask_off_by_one"
    o_m, lse_m = fwd(q, k, v, 0.5, causal)
    o_bf, lse_bf = brute_force_forward(q.tolist(), k.tolist(), v.tolist(), 0.5, causal)
    caught = (not np.allclose(o_m, o_bf, atol=1e-10)) or (not np.allclose(lse_m, lse_bf, atol=1e-10))
    assert caught


# ---------------------------------------------------------------------------
# Grouped-query attention pins
# ---------------------------------------------------------------------------


def test_gqa_with_one_kv_head_per_query_head_is_mha():
    B, H, N, d = 1, 3, 10, 4
    q, k, v, do = (rand((B, H, N, d), s) for s in (140, 141, 142, 143))
    o1, l1 = oracle.forward(q, k, v, 0.5, True)
    o2, l2 = oracle.forward_gqa(q, k, v, 0.5, True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    for a, b in zip(oracle.backward(q, k, v, do, 0.5, True), oracle.backward_gqa(q, k, v, do, 0.5, True)):
        np.testing.assert_allclose(a, b, atol=1e-15)


def test_gqa_head_mapping_contiguous_groups():
    """Query heads 0..G-1 read key/value head 0, heads G..2G-1 read head 1 (the
    layout of a K projection with Hk heads repeated G times along the head axis)."""
    assert [oracle.kv_head_of(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [oracle.kv_head_of(h, 6, 1) for h in range(6)] == [0] * 6
    B, H, Hk, N, d = 1, 4, 2, 7, 3
    q = rand((B, H, N, d), 150)
    k, v = rand((B, Hk, N, d), 151), rand((B, Hk, N, d), 152)
    o, _ = oracle.forward_gqa(q, k, v, 0.9, False)
    # the same thing written with an explicitly repeated K/V along the head axis
    o_rep, _ = oracle.forward(q, np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1), 0.9, False)
    np.testing.assert_allclose(o, o_rep, atol=1e-15)
    o_bf, _ = brute_force_forward(q[0, 3].tolist(), k[0, 1].tolist(), v[0, 1].tolist(), 0.9, False)
    np.testing.assert_allclose(o[0, 3], o_bf, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_backward_matches_finite_differences(causal):
    B, H, Hk, N, d = 1, 4, 2, 5, 3
    q = rand((B, H, N, d), 160)
    k, v = rand((B, Hk, N, d), 161), rand((B, Hk, N, d), 162)
    do = rand((B, H, N, d), 163)
    scale = 0.7
    dq, dk, dv = oracle.backward_gqa(q, k, v, do, scale, causal)

    def loss(qq, kk, vv):
        o, _ = oracle.forward_gqa(qq, kk, vv, scale, causal)
        return float(np.sum(do * o))

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"])
                        - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        err = np.linalg.norm(num - g) / np.linalg.norm(num)
        assert err < 1e-6, (name, err)


# ---------------------------------------------------------------------------
# Sliding-window pins
# ---------------------------------------------------------------------------


def test_window_special_cases_are_causal_and_full():
    np.testing.assert_array_equal(A.window_visible(9, 9, (-1, 0)), A.causal_visible(9, 9))
    assert A.window_visible(9, 9, (-1, -1)).all()
    np.testing.assert_array_equal(A.window_visible(5, 2, (-1, 0)), A.causal_visible(5, 2))
    # window (1, 2) on 6 rows: row i sees i-1 .. i+2
    expect = np.array([[abs(j - i) <= 2 and j >= i - 1 for j in range(6)] for i in range(6)])
    np.testing.assert_array_equal(A.window_visible(6, 6, (1, 2)), expect)


def test_window_zero_returns_own_value_row():
    N, d = 11, 4
    q, k, v = rand((N, d), 170), rand((N, d), 171), rand((N, d), 172)
    o, lse, _ = A.head_forward(q, k, v, 0.6, False, window=(0, 0))
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, 0.6 * np.sum(q * k, axis=1), atol=1e-14)


def test_window_one_left_is_a_sigmoid_of_two_keys():
    N, d = 7, 4
    q, k, v = rand((N, d), 173), rand((N, d), 174), rand((N, d), 175)
    o, _, _ = A.head_forward(q, k, v, 0.5, False, window=(1, 0))
    for i in range(1, N):
        s0, s1 = 0.5 * q[i] @ k[i - 1], 0.5 * q[i] @ k[i]
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        np.testing.assert_allclose(o[i], w0 * v[i - 1] + (1 - w0) * v[i], atol=1e-14)


def brute_force_window(q, k, v, scale, left, right):
    n = len(q)
    o = []
    for i in range(n):
        vis = [j for j in range(n) if (right < 0 or j <= i + right) and (left < 0 or j >= i - left)]
        s = {j: scale * math.fsum(a * b for a, b in zip(q[i], k[j])) for j in vis}
        m = max(s.values())
        e = {j: math.exp(s[j] - m) for j in vis}
        z = math.fsum(e.values())
        o.append([math.fsum(e[j] * v[j][c] for j in vis) / z for c in range(len(v[0]))])
    return np.array(o)


@pytest.mark.parametrize("window", [(2, 1), (0, 3), (4, -1), (-1, 2)])
def test_window_brute_force(window):
    N, d = 12, 5
    q, k, v = rand((N, d), 180), rand((N, d), 181), rand((N, d), 182)
    o, _, _ = A.head_forward(q, k, v, 0.4, False, window=window)
    np.testing.assert_allclose(o, brute_force_window(q.tolist(), k.tolist(), v.tolist(), 0.4, *window),
                               atol=1e-13)


@pytest.mark.parametrize("window", [(2, 1), (1, 0)])
def test_window_backward_matches_finite_differences(window):
    N, d = 6, 3
    q, k, v, do = (rand((N, d), s) for s in (190, 191, 192, 193))
    dq, dk, dv, _ = A.head_backward(q, k, v, do, 0.8, False, window=window)

    def loss(qq, kk, vv):
        o, _, _ = A.head_forward(qq, kk, vv, 0.8, False, window=window)
        return float(np.sum(do * o))

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            a = {"q": q, "k": k, "v": v}
            b = dict(a)
            a[name], b[name] = xp, xm
            num[idx] = (loss(a["q"], a["k"], a["v"]) - loss(b["q"], b["k"], b["v"])) / (2 * h)
        assert np.linalg.norm(num - g) / np.linalg.norm(num) < 1e-6, name
