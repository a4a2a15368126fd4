"""Host-side checks of the C ABI (no GPU needed, no kernel launched): the
library loads, exports every function include/attn_sm103a.h declares, and
rejects bad arguments before touching the device."""

import ctypes
import os
import re

import pytest

from exact_attention_52_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_sm103a.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(api.LIB_PATH):
        pytest.skip("library not built (run __graft_entry__.build())")
    return api.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_bytes", "attn_fwd_fp8",
               "attn_check_device_error", "attn_status_string"):
        assert fn in names
    assert set(names) == set(api.SIGNATURES), "binding and header disagree"


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in api.STATUS_NAMES.items():
        assert lib.attn_status_string(code).decode() == name


def test_workspace_bytes(lib):
    # fp32 dQ accumulator over padded rows + two fp32 vectors, 256-byte rounded;
    # d = 128 adds the counters (160 x 8 words) and fp32 dV/dK partials of split
    # items: min(160, items * min(10, tiles)) parts of 2 x 128 x d floats,
    # tiles = ceil(N/128), items = B*H*tiles
    r256 = lambda x: (x + 255) // 256 * 256
    for B, H, N, d in ((2, 3, 200, 128), (2, 3, 200, 64), (1, 1, 128, 128), (1, 32, 8192, 128)):
        npad = (N + 127) // 128 * 128
        rows = B * H * npad
        base = r256(rows * d * 4) + 2 * r256(rows * 4)
        tiles = npad // 128
        cap = min(160, B * H * tiles * min(10, tiles)) if d == 128 else 0
        split = r256(160 * 8 * 4) + r256(cap * 2 * 128 * d * 4) if cap > 0 else 0
        assert lib.attn_bwd_workspace_bytes(B, H, N, d) == base + split, (B, H, N, d)
    assert lib.attn_bwd_workspace_bytes(0, 1, 1, 64) == 0
    assert lib.attn_bwd_workspace_bytes(1, 1, 1, 96) == 0


def test_splitkv_workspace_bytes(lib):
    B, H, N, d = 1, 2, 1000, 128
    rows = B * H * N
    r256 = lambda x: (x + 255) // 256 * 256
    for S in (1, 3, 16):
        assert lib.attn_fwd_splitkv_workspace_bytes(B, H, N, d, S) == r256(S * rows * d * 4) + r256(S * rows * 4)
    assert lib.attn_fwd_splitkv_workspace_bytes(B, H, N, d, 0) == lib.attn_fwd_splitkv_workspace_bytes(B, H, N, d, 16)
    assert lib.attn_fwd_splitkv_workspace_bytes(B, H, N, d, 17) == 0
    assert lib.attn_fwd_splitkv_workspace_bytes(B, H, N, 96, 2) == 0


def test_smem_budget(lib):
    for which, d in ((0, 64), (0, 128), (1, 128), (2, 64), (2, 128)):
        b = lib.attn_kernel_smem_bytes(which, d)
        assert 0 < b <= 232448, (which, d, b)
    assert lib.attn_kernel_smem_bytes(1, 64) == 0


def test_invalid_arguments_are_rejected_before_launch(lib):
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    null = ctypes.c_void_p(0)
    INVALID, UNSUP = -1, -2
    # null pointers
    assert lib.attn_fwd(null, fake, fake, fake, fake, 1, 1, 128, 64, 0.125, 0, None) == INVALID
    # sizes
    assert lib.attn_fwd(fake, fake, fake, fake, fake, 0, 1, 128, 64, 0.125, 0, None) == INVALID
    assert lib.attn_fwd(fake, fake, fake, fake, fake, 1, 1, 0, 64, 0.125, 0, None) == INVALID
    assert lib.attn_fwd(fake, fake, fake, fake, fake, 1, 1, 128, 96, 0.125, 0, None) == UNSUP
    # scale and causal flag
    assert lib.attn_fwd(fake, fake, fake, fake, fake, 1, 1, 128, 64, 0.0, 0, None) == INVALID
    assert lib.attn_fwd(fake, fake, fake, fake, fake, 1, 1, 128, 64, float("nan"), 0, None) == INVALID
    assert lib.attn_fwd(fake, fake, fake, fake, fake, 1, 1, 128, 64, 0.1, 2, None) == INVALID
    # misaligned pointer
    mis = ctypes.c_void_p((1 << 20) + 8)
    assert lib.attn_fwd(mis, fake, fake, fake, fake, 1, 1, 128, 64, 0.125, 0, None) == INVALID
    # fp8: d = 64 is not built; non-positive scales rejected
    assert lib.attn_fwd_fp8(fake, fake, fake, 1.0, 1.0, 1.0, fake, fake, 1, 1, 128, 64, 0.1, 0,
                            None) == UNSUP
    assert lib.attn_fwd_fp8(fake, fake, fake, 0.0, 1.0, 1.0, fake, fake, 1, 1, 128, 128, 0.1, 0,
                            None) == INVALID
    # backward: workspace must be 256-byte aligned and present
    args = [fake] * 9
    assert lib.attn_bwd(*args, null, 1, 1, 128, 64, 0.1, 0, None) == INVALID
    assert lib.attn_bwd(*args, ctypes.c_void_p((1 << 20) + 16), 1, 1, 128, 64, 0.1, 0,
                        None) == INVALID


def test_binding_raises_when_library_missing(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        api.load_library(str(tmp_path / "libattn_sm103a.so"))


def test_noalloc_checks_the_problem_before_its_scratch_limit(lib):
    """attn_bwd_noalloc gives attn_bwd's status for a bad problem, and rejects a
    valid one that needs more than its 64 MiB scratch, before touching the
    device (no GPU here: any device call would fail with ATTN_ERR_CUDA)."""
    fake = ctypes.c_void_p(1 << 20)
    args = [fake] * 9
    INVALID, UNSUP = -1, -2
    assert lib.attn_bwd_noalloc(*args, 1, 1, 128, 96, 0.1, 0, None) == UNSUP
    assert lib.attn_bwd_noalloc(*args, 0, 1, 128, 128, 0.1, 0, None) == INVALID
    assert lib.attn_bwd_noalloc(*args, 1, 1, 128, 128, 0.1, 2, None) == INVALID
    assert lib.attn_bwd_noalloc(*args, 1, 1, 128, 128, float("inf"), 0, None) == INVALID
    assert lib.attn_bwd_noalloc(*args, 1, 32, 8192, 128, 0.088, 0, None) == UNSUP
    # without the split last round's partials (which it leaves out when they do
    # not fit) B1 H15 N8192 d128 fits the scratch and B1 H32 N8192 does not
    r256 = lambda x: (x + 255) // 256 * 256
    unsplit = lambda H: r256(H * 8192 * 128 * 4) + 2 * r256(H * 8192 * 4)
    assert unsplit(15) <= 64 << 20 < unsplit(32)
