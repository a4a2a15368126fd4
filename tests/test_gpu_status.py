"""Device error path, exercised without any fault: a kernel waits on a barrier
that nothing completes, gives up after a short limit, and the host reads the
error word."""

import pytest

from exact_attention_52_gb300 import api

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout():
    api.set_wait_limit_ns(2_000_000)  # 2 ms
    try:
        api.selftest_wait_timeout()
        rc, site = api.check_device_error()
    finally:
        api.set_wait_limit_ns(0)
    assert rc == -4 and site in (0x901, 0x902)
    # the word is cleared by the read, and the context is still usable
    assert api.check_device_error() == (0, 0)


def test_wrong_device_dtype_rejected_by_binding():
    import torch
    q = torch.zeros(1, 1, 128, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        api.fwd(q, q, q)
