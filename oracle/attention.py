"""fp64 CPU oracle for exact softmax attention (forward and backward).

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
benchmark's CPU-baseline leg may import this module; the library itself never
does, and this module imports nothing from the library.

What it computes, per (batch, head), materialising S and P in full:

* scores ``S = scale * Q K^T`` (FlashAttention paper page, standard
  attention, section 1: S and P are N x N matrices), with the causal mask
  aligned to the bottom-right corner when query and key lengths differ
  (FlashAttention README item, "Causal-Mask and Small-Query Behavior"):
  query row ``i`` may see key ``j`` iff ``j <= i + (Nk - Nq)``;
* ``P = softmax(S)`` row-wise, with the row maximum subtracted first
  (online-normalizer item: running max ``m`` and sum ``d``);
* ``O = P V`` and ``LSE_i = m_i + ln(sum_j exp(S_ij - m_i))`` -- the natural
  log-sum-exp of the scaled scores, i.e. the "normalization statistics" the
  backward pass reuses (FlashAttention item 58);
* a row with no visible key gives ``O_i = 0`` (README example: fully masked
  rows have zero output) and ``LSE_i = +inf`` so that ``exp(S - LSE) = 0``
  there (CUDA softmax item: no -inf - -inf, no divide by zero);
* sliding-window (local) attention: key j visible to query i iff
  i - left <= j <= i + right, a negative bound meaning none (FlashAttention-3
  tuning page, window sizes); (-1, 0) is the causal mask;
* grouped-query attention: ``Hk`` key/value heads shared by ``H`` query heads
  (FlashAttention-3 walkthrough: ``num_heads_k`` runtime parameter, GQA/MQA
  feature list); query head ``h`` reads key/value head ``h // (H // Hk)``, and
  the gradient of a shared key/value head is the sum over its query heads;
* backward of ``O = softmax(scale Q K^T) V`` for a given ``dO``, written from
  the calculus of that definition (the pages cut off before printing it):
  ``dV = P^T dO``, ``dP = dO V^T``, ``D_i = sum_j P_ij dP_ij``,
  ``dS = P * (dP - D)``, ``dQ = scale dS K``, ``dK = scale dS^T Q``.

Inputs are the exact values the GPU reads: bf16 bit patterns or FP8 E4M3
codes are decoded here by this module's own decoders.

Pins: every function is checked by ``tests/test_oracle_pins.py`` against
closed forms, brute force, finite differences and the pages' examples.
"""

from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# Storage decoders
# ---------------------------------------------------------------------------


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 is the top half of an IEEE binary32: shift left 16 and reinterpret."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):  # NaN payloads widen to NaN
        return b.view(np.float32).astype(np.float64)


def _e4m3_table() -> np.ndarray:
    """Value of every OCP FP8 E4M3 ("fn") code: 1 sign, 4 exponent (bias 7), 3 mantissa
    bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities."""
    t = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            t[code] = math.nan
        elif e == 0:
            t[code] = sign * (m / 8.0) * 2.0 ** (-6)
        else:
            t[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return t


_E4M3 = _e4m3_table()


def e4m3_to_f64(codes: np.ndarray, scale: float = 1.0) -> np.ndarray:
    """Decode E4M3 codes and multiply by the per-tensor scale (x = s * q8)."""
    return _E4M3[np.asarray(codes, dtype=np.uint8)] * float(scale)


# ---------------------------------------------------------------------------
# Forward
# ---------------------------------------------------------------------------


def causal_visible(nq: int, nk: int, rows: np.ndarray | None = None) -> np.ndarray:
    """Boolean [len(rows), nk] mask: True where query row i sees key j (bottom-right)."""
    i = np.arange(nq) if rows is None else np.asarray(rows)
    j = np.arange(nk)
    return j[None, :] <= (i[:, None] + (nk - nq))


def window_visible(nq: int, nk: int, window: tuple[int, int],
                   rows: np.ndarray | None = None) -> np.ndarray:
    """Boolean [len(rows), nk] mask of a local (sliding-window) attention:
    key j is visible to query i iff i' - left <= j <= i' + right, where
    i' = i + (nk - nq) aligns the last query with the last key (as the causal
    rule does) and a negative bound is no bound (FlashAttention-3 tuning page:
    window_size_left / window_size_right)."""
    left, right = window
    i = (np.arange(nq) if rows is None else np.asarray(rows)) + (nk - nq)
    j = np.arange(nk)
    vis = np.ones((len(i), nk), dtype=bool)
    if right >= 0:
        vis &= j[None, :] <= i[:, None] + right
    if left >= 0:
        vis &= j[None, :] >= i[:, None] - left
    return vis


def scores(q: np.ndarray, k: np.ndarray, scale: float, causal: bool,
           rows: np.ndarray | None = None, window: tuple[int, int] | None = None) -> np.ndarray:
    """S = scale * Q K^T for one head ([Nq, d] x [Nk, d]); masked entries are -inf.
    ``window`` (left, right), when given, replaces the causal flag."""
    qq = q if rows is None else q[rows]
    s = float(scale) * (qq @ k.T)
    if window is not None:
        s = np.where(window_visible(q.shape[0], k.shape[0], window, rows), s, -np.inf)
    elif causal:
        s = np.where(causal_visible(q.shape[0], k.shape[0], rows), s, -np.inf)
    return s


def softmax_rows(s: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Row softmax of S with the row max subtracted; returns (P, LSE).

    Rows that are entirely -inf give P = 0 and LSE = +inf.
    """
    m = np.max(s, axis=1)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe[:, None])
    l = np.sum(e, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(empty[:, None], 0.0, e / np.where(empty, 1.0, l)[:, None])
        lse = np.where(empty, np.inf, m_safe + np.log(np.where(empty, 1.0, l)))
    return p, lse


def head_forward(q, k, v, scale, causal, rows=None, window=None):
    """One head: returns (O [rows, d], LSE [rows], P [rows, Nk])."""
    p, lse = softmax_rows(scores(q, k, scale, causal, rows, window))
    return p @ v, lse, p


def forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
            causal: bool, heads=None, rows=None):
    """Attention forward on fp64 arrays ``[B, H, N, d]``.

    ``heads``: optional list of (b, h) to evaluate (others are skipped);
    ``rows``: optional query-row indices.  Returns dict (b, h) -> (O, LSE)
    when ``heads`` or ``rows`` is given, else full arrays (O [B,H,Nq,d],
    LSE [B,H,Nq]).
    """
    B, H = q.shape[0], q.shape[1]
    if heads is None and rows is None:
        o = np.zeros(q.shape[:3] + (v.shape[3],), dtype=np.float64)
        lse = np.zeros(q.shape[:3], dtype=np.float64)
        for b in range(B):
            for h in range(H):
                o[b, h], lse[b, h], _ = head_forward(q[b, h], k[b, h], v[b, h],
                                                     scale, causal)
        return o, lse
    out = {}
    for (b, h) in (heads if heads is not None else
                   [(b, h) for b in range(B) for h in range(H)]):
        o_bh, lse_bh, _ = head_forward(q[b, h], k[b, h], v[b, h], scale, causal, rows)
        out[(b, h)] = (o_bh, lse_bh)
    return out


# ---------------------------------------------------------------------------
# Backward
# ---------------------------------------------------------------------------


def head_backward(q, k, v, do, scale, causal, window=None):
    """One head: gradients of O = softmax(scale Q K^T) V for upstream dO.

    Returns (dQ, dK, dV, D) with D_i = sum_j P_ij dP_ij.
    """
    o, _, p = head_forward(q, k, v, scale, causal, window=window)
    dv = p.T @ do
    dp = do @ v.T
    dsum = np.sum(p * dp, axis=1)
    ds = p * (dp - dsum[:, None])
    dq = float(scale) * (ds @ k)
    dk = float(scale) * (ds.T @ q)
    return dq, dk, dv, dsum


def head_backward_rows(q, k, v, do, scale, causal, rows, window=None):
    """dQ for the query rows ``rows`` only, by the same calculus as
    ``head_backward``: each row of dQ needs only that row of P, dP and D, so long
    sequences can be checked row by row (``dQ_i = scale * sum_j dS_ij K_j`` with
    ``dS_i = P_i * (dP_i - D_i)``, ``dP_i = dO_i V^T``, ``D_i = sum_j P_ij dP_ij``).

    Returns (dQ [rows, d], D [rows]).
    """
    rows = np.asarray(rows)
    _, _, p = head_forward(q, k, v, scale, causal, rows=rows, window=window)
    dp = do[rows] @ v.T
    dsum = np.sum(p * dp, axis=1)
    ds = p * (dp - dsum[:, None])
    return float(scale) * (ds @ k), dsum


def backward(q, k, v, do, scale, causal, heads=None):
    """Backward on fp64 ``[B, H, N, d]`` arrays.

    Returns full (dQ, dK, dV) arrays, or dict (b, h) -> (dQ, dK, dV) when
    ``heads`` is given.
    """
    B, H = q.shape[0], q.shape[1]
    if heads is None:
        dq = np.zeros_like(q)
        dk = np.zeros_like(k)
        dv = np.zeros_like(v)
        for b in range(B):
            for h in range(H):
                dq[b, h], dk[b, h], dv[b, h], _ = head_backward(
                    q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
        return dq, dk, dv
    out = {}
    for (b, h) in heads:
        dq, dk, dv, _ = head_backward(q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
        out[(b, h)] = (dq, dk, dv)
    return out


# ---------------------------------------------------------------------------
# Grouped-query attention
# ---------------------------------------------------------------------------


def kv_head_of(h: int, H: int, Hk: int) -> int:
    """Key/value head read by query head h."""
    return h // (H // Hk)


def forward_gqa(q, k, v, scale, causal, window=None):
    """Forward with k, v of shape [B, Hk, N, d]: every query head h attends with
    key/value head kv_head_of(h).  Returns (O [B,H,N,d], LSE [B,H,N])."""
    B, H = q.shape[0], q.shape[1]
    Hk = k.shape[1]
    o = np.zeros(q.shape[:3] + (v.shape[3],), dtype=np.float64)
    lse = np.zeros(q.shape[:3], dtype=np.float64)
    for b in range(B):
        for h in range(H):
            g = kv_head_of(h, H, Hk)
            o[b, h], lse[b, h], _ = head_forward(q[b, h], k[b, g], v[b, g], scale, causal,
                                                 window=window)
    return o, lse


def backward_gqa(q, k, v, do, scale, causal, window=None):
    """Backward with shared key/value heads: dQ per query head; dK, dV per
    key/value head, summed over the query heads that read it."""
    B, H = q.shape[0], q.shape[1]
    Hk = k.shape[1]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            g = kv_head_of(h, H, Hk)
            dq[b, h], dkh, dvh, _ = head_backward(q[b, h], k[b, g], v[b, g], do[b, h], scale, causal,
                                                  window=window)
            dk[b, g] += dkh
            dv[b, g] += dvh
    return dq, dk, dv
