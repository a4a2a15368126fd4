"""Forward launches with many more work items than SMs, so that each persistent
CTA walks several items (barrier phases, the key/value ring position and the
output accumulators all carry over from one item to the next).  A ragged
sequence length gives every item a partial last tile; grouped heads and a
sliding window change the per-item key ranges.  Sampled heads are compared with
the oracle; every output must be finite."""

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import make_inputs_gqa

from .helpers import (TOL_LSE_ABS, TOL_O_MAXABS, bf16_out_err, bf16_to_device, device_bf16_to_f64,
                      device_f32_to_f64, max_abs)

pytestmark = pytest.mark.gpu

SCALE_D = 128


def _decode(bits):
    return oracle.bf16_bits_to_f64(bits)


@pytest.mark.parametrize("B,H,Hk,N,window", [
    (2, 24, 24, 2000, None),      # 24 * 2 * 8 = 384 items of ragged tiles, 2-3 per CTA
    (1, 48, 12, 3001, None),      # grouped heads, 48 * 12 = 576 items
    (3, 16, 16, 1500, (300, 0)),  # sliding window: short, item-dependent key ranges
])
def test_persistent_forward_many_items(B, H, Hk, N, window):
    d = SCALE_D
    inp = make_inputs_gqa(B, H, Hk, N, d, seed=7)
    q, k, v = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits))
    if window is None:
        o, lse = api.fwd(q, k, v)
    else:
        o, lse = api.fwd_window(q, k, v, *window)
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    og, lg = device_bf16_to_f64(o), device_f32_to_f64(lse)
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg))
    qd, kd, vd = _decode(inp.q_bits), _decode(inp.k_bits), _decode(inp.v_bits)
    G = H // Hk
    scale = 1.0 / np.sqrt(d)
    # first, last and a middle head: items early, late and in the middle of the walk
    for (b, h) in [(0, 0), (B - 1, H - 1), (B // 2, H // 2)]:
        o_ref, lse_ref, _ = oracle.head_forward(qd[b, h], kd[b, h // G], vd[b, h // G], scale, False,
                                                window=window)
        assert bf16_out_err(og[b, h], o_ref) <= TOL_O_MAXABS, (b, h)
        assert max_abs(lg[b, h], lse_ref) <= TOL_LSE_ABS, (b, h)
