"""The comparison helpers used by the parity tests, checked against PyTorch's
own bfloat16 rounding (CPU only)."""

import numpy as np
import pytest

from .helpers import bf16_half_ulp, bf16_out_err, max_abs, rel_fro


def test_bf16_half_ulp_bounds_round_to_nearest():
    torch = pytest.importorskip("torch")
    x32 = (np.random.Generator(np.random.PCG64(0)).standard_normal(100000) * 3.0).astype(np.float32)
    x = x32.astype(np.float64)  # single rounding float32 -> bf16 below
    xb = torch.from_numpy(x32).to(torch.bfloat16).double().numpy()
    assert np.all(np.abs(xb - x) <= bf16_half_ulp(x) * (1 + 1e-12))
    assert bf16_out_err(xb, x) <= 1e-12
    # one spacing off is an error of about half a spacing beyond rounding
    assert bf16_out_err(np.array([4.0 + 2 ** -5]), np.array([4.0])) == pytest.approx(2 ** -6)
    assert bf16_half_ulp(np.array([1.0, 4.13, 0.0])).tolist() == [2 ** -8, 2 ** -6, 0.0]


def test_metrics():
    a = np.array([1.0, 2.0, 3.0])
    assert max_abs(a, a + [0, 0.5, 0]) == 0.5
    assert rel_fro(a * 1.01, a) == pytest.approx(0.01)


def test_grad_rel_err_catches_one_wrong_row():
    from .helpers import grad_rel_err
    rng = np.random.Generator(np.random.PCG64(1))
    ref = rng.standard_normal((2, 8192, 128))
    gpu = ref * (1 + 1e-3 * rng.standard_normal(ref.shape))
    assert grad_rel_err(gpu, ref) < 2e-3
    bad = gpu.copy()
    bad[1, 5000] = 0.0  # one row lost
    assert rel_fro(bad, ref) < 2e-2  # the whole-tensor figure alone would pass
    assert grad_rel_err(bad, ref) > 0.05  # its 128-row block does not
    tail = gpu[:, :8000].copy()
    tail[0, -3:] *= -1.0  # a ragged last block with a sign error
    assert grad_rel_err(tail, ref[:, :8000]) > 0.1


def test_row_blocks_merge_short_tails():
    from .helpers import row_blocks
    assert row_blocks(1) == [(0, 1)]
    assert row_blocks(128) == [(0, 128)]
    assert row_blocks(513) == [(0, 128), (128, 256), (256, 384), (384, 513)]
    assert row_blocks(8000)[-1] == (7936, 8000)  # 64 rows: kept as a block of its own
    assert row_blocks(300) == [(0, 128), (128, 300)]
