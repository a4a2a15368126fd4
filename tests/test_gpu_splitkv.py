"""Split-KV forward: key tiles divided among CTAs, partial (O, LSE) merged by
the combine kernel with the running-max / running-sum rule.  Checked against
the oracle and against the single-pass forward."""

import numpy as np
import pytest

import oracle
from exact_attention_52_gb300 import api
from exact_attention_52_gb300.inputs import make_inputs

from .helpers import (TOL_LSE_ABS, TOL_O_MAXABS, bf16_out_err, bf16_to_device, decoded,
                      device_bf16_to_f64, device_f32_to_f64, max_abs)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,splits", [(300, 2), (1000, 3), (2048, 0), (1500, 16), (128, 4), (5, 2)])
def test_splitkv_matches_oracle(N, splits, d, causal):
    inp = make_inputs(1, 2, N, d, seed=N + splits + d)
    q, k, v = (bf16_to_device(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits))
    o, lse = api.fwd_splitkv(q, k, v, num_splits=splits, causal=causal)
    o1, lse1 = api.fwd(q, k, v, causal=causal)
    rc, site = api.check_device_error()
    assert rc == 0, f"device error {rc} at site {site:#x}"
    qf, kf, vf, _ = decoded(inp)
    o_ref, lse_ref = oracle.forward(qf, kf, vf, 1.0 / np.sqrt(d), causal)
    og, lg = device_bf16_to_f64(o), device_f32_to_f64(lse)
    assert bf16_out_err(og, o_ref) <= TOL_O_MAXABS
    assert max_abs(lg, lse_ref) <= TOL_LSE_ABS
    # same answer as the single-pass kernel up to rounding
    assert max_abs(og, device_bf16_to_f64(o1)) <= 2e-2
    assert max_abs(lg, device_f32_to_f64(lse1)) <= 2e-5 * np.max(np.abs(lse_ref)) + 1e-5


def test_splitkv_rejects_bad_split_count():
    import torch
    q = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        api.fwd_splitkv(q, q, q, num_splits=17)
