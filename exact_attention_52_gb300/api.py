"""Python binding of libattn_sm103a.so (ctypes): argument marshalling only.

Every function here checks dtypes, shapes and devices, allocates outputs with
PyTorch when the caller did not pass them, and calls the C ABI declared in
``include/attn_sm103a.h`` on the current PyTorch CUDA stream.  All arithmetic
runs in the library's CUDA kernels; there is no fallback path.  If the shared
library is missing, every call raises ``RuntimeError``.
"""

from __future__ import annotations

import ctypes
import math
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn_sm103a.so")
# The same library built with device-side range checks (see attn_build_flags).
DEBUG_LIB_PATH = os.path.join(_PKG, "libattn_sm103a_debug.so")

ATTN_OK = 0
STATUS_NAMES = {0: "ATTN_OK", -1: "ATTN_ERR_INVALID", -2: "ATTN_ERR_UNSUPPORTED",
                -3: "ATTN_ERR_CUDA", -4: "ATTN_ERR_TIMEOUT"}



class Strides(ctypes.Structure):
    """attn_strides_t: element strides (b, h, n) of a [B, heads, N, d] view."""
    _fields_ = [("b", ctypes.c_int64), ("h", ctypes.c_int64), ("n", ctypes.c_int64)]


# Every symbol the header declares, with (restype, argtypes).
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_st = Strides
SIGNATURES = {
    "attn_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
    "attn_bwd_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "attn_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
    "attn_bwd_preprocess": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "attn_bwd_main": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
    "attn_bwd_dq_convert": (_i, [_vp, _vp, _i, _i, _i, _i, _f, _vp]),
    "attn_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i,
                              _vp]),
    "attn_fwd_gqa": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "attn_bwd_gqa": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f,
                          _i, _vp]),
    "attn_fwd_splitkv_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "attn_fwd_splitkv": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "attn_fwd_window": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "attn_bwd_window": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                             _f, _i, _i, _vp]),
    "attn_fwd_strided": (_i, [_vp, _st, _vp, _st, _vp, _st, _vp, _st, _vp, _i, _i, _i, _i, _i, _f,
                              _i, _i, _vp]),
    "attn_bwd_strided": (_i, [_vp, _st, _vp, _st, _vp, _st, _vp, _st, _vp, _st, _vp, _vp, _st, _vp,
                              _st, _vp, _st, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "attn_fwd_fp8": (_i, [_vp, _vp, _vp, _f, _f, _f, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
    "attn_check_device_error": (_i, [_vp, ctypes.POINTER(ctypes.c_uint)]),
    "attn_set_wait_limit_ns": (None, [ctypes.c_ulonglong]),
    "attn_set_exp2_offload": (None, [_i]),
    "attn_selftest_wait_timeout": (_i, [_vp]),
    "attn_status_string": (ctypes.c_char_p, [_i]),
    "attn_kernel_smem_bytes": (_i, [_i, _i]),
    "attn_build_flags": (_i, []),
}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Open the shared library and declare every C signature (no GPU needed)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{os.path.basename(path)} is not built; run "
                           "`python -m exact_attention_52_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


def _check(fn: str, status: int) -> None:
    if status != ATTN_OK:
        raise AttnError(fn, status)


def _stream_handle(stream) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check_qkv(name, t, shape, dtype):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous [B, H, N, d]")


def fwd(q, k, v, scale: float | None = None, causal: bool = False, o=None, lse=None,
        stream=None):
    """Forward pass on bf16 CUDA tensors [B, H, N, d]; returns (O bf16, LSE fp32 [B, H, N])."""
    import torch
    B, H, N, d = q.shape
    Hk = k.shape[1] if getattr(k, "dim", lambda: 0)() == 4 else H
    _check_qkv("q", q, (B, H, N, d), torch.bfloat16)
    for name, t in (("k", k), ("v", v)):
        _check_qkv(name, t, (B, Hk, N, d), torch.bfloat16)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_qkv("o", o, (B, H, N, d), torch.bfloat16)
    _check_qkv("lse", lse, (B, H, N), torch.float32)
    lib = load_library()
    if Hk == H:
        _check("attn_fwd", lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                        lse.data_ptr(), B, H, N, d, scale, int(bool(causal)),
                                        _stream_handle(stream)))
    else:
        _check("attn_fwd_gqa", lib.attn_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                o.data_ptr(), lse.data_ptr(), B, H, Hk, N, d, scale,
                                                int(bool(causal)), _stream_handle(stream)))
    return o, lse


def fwd_splitkv(q, k, v, num_splits: int = 0, scale: float | None = None, causal: bool = False,
                o=None, lse=None, workspace=None, stream=None):
    """Split-KV forward (bf16, Hk = H): returns (O, LSE) like ``fwd``."""
    import torch
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_qkv(name, t, (B, H, N, d), torch.bfloat16)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    lib = load_library()
    need = int(lib.attn_fwd_splitkv_workspace_bytes(B, H, N, d, int(num_splits)))
    if need == 0:
        raise ValueError("invalid sizes or num_splits")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check("attn_fwd_splitkv", lib.attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                    o.data_ptr(), lse.data_ptr(),
                                                    workspace.data_ptr(), B, H, N, d, scale,
                                                    int(bool(causal)), int(num_splits),
                                                    _stream_handle(stream)))
    return o, lse


def fwd_window(q, k, v, window_left: int, window_right: int, scale: float | None = None,
               o=None, lse=None, stream=None):
    """Sliding-window forward: key j visible to query i iff
    i - window_left <= j <= i + window_right (-1: unbounded side)."""
    import torch
    B, H, N, d = q.shape
    Hk = k.shape[1]
    _check_qkv("q", q, (B, H, N, d), torch.bfloat16)
    for name, t in (("k", k), ("v", v)):
        _check_qkv(name, t, (B, Hk, N, d), torch.bfloat16)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check("attn_fwd_window", load_library().attn_fwd_window(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Hk, N, d,
        scale, int(window_left), int(window_right), _stream_handle(stream)))
    return o, lse


def bwd_window(q, k, v, o, dout, lse, window_left: int, window_right: int,
               scale: float | None = None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Sliding-window backward; dK, dV have K's head count."""
    import torch
    B, H, N, d = q.shape
    Hk = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("q", q), ("o", o), ("dout", dout), ("dq", dq)):
        _check_qkv(name, t, (B, H, N, d), torch.bfloat16)
    for name, t in (("k", k), ("v", v), ("dk", dk), ("dv", dv)):
        _check_qkv(name, t, (B, Hk, N, d), torch.bfloat16)
    need = bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check("attn_bwd_window", load_library().attn_bwd_window(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(), B, H, Hk, N, d, scale,
        int(window_left), int(window_right), _stream_handle(stream)))
    return dq, dk, dv


def bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().attn_bwd_workspace_bytes(B, H, N, d))


def bwd(q, k, v, o, dout, lse, scale: float | None = None, causal: bool = False,
        dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward pass; returns (dQ, dK, dV) bf16 [B, H, N, d]."""
    import torch
    B, H, N, d = q.shape
    Hk = k.shape[1] if getattr(k, "dim", lambda: 0)() == 4 else H
    for name, t in (("q", q), ("o", o), ("dout", dout)):
        _check_qkv(name, t, (B, H, N, d), torch.bfloat16)
    for name, t in (("k", k), ("v", v)):
        _check_qkv(name, t, (B, Hk, N, d), torch.bfloat16)
    _check_qkv("lse", lse, (B, H, N), torch.float32)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_qkv("dq", dq, (B, H, N, d), torch.bfloat16)
    for name, t in (("dk", dk), ("dv", dv)):
        _check_qkv(name, t, (B, Hk, N, d), torch.bfloat16)
    need = bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace needs {need} bytes")
    lib = load_library()
    if Hk == H:
        _check("attn_bwd", lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                        dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                        dv.data_ptr(), workspace.data_ptr(), B, H, N, d, scale,
                                        int(bool(causal)), _stream_handle(stream)))
    else:
        _check("attn_bwd_gqa", lib.attn_bwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                                                dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                                workspace.data_ptr(), B, H, Hk, N, d, scale,
                                                int(bool(causal)), _stream_handle(stream)))
    return dq, dk, dv


def fwd_fp8(q8, k8, v8, sq: float, sk: float, sv: float, scale: float | None = None,
            causal: bool = False, o=None, lse=None, stream=None):
    """FP8 forward: uint8 E4M3 codes [B, H, N, d] with per-tensor scales; returns (O bf16, LSE)."""
    import torch
    B, H, N, d = q8.shape
    for name, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        _check_qkv(name, t, (B, H, N, d), torch.uint8)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    _check_qkv("o", o, (B, H, N, d), torch.bfloat16)
    _check_qkv("lse", lse, (B, H, N), torch.float32)
    lib = load_library()
    _check("attn_fwd_fp8", lib.attn_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(),
                                            float(sq), float(sk), float(sv), o.data_ptr(),
                                            lse.data_ptr(), B, H, N, d, scale,
                                            int(bool(causal)), _stream_handle(stream)))
    return o, lse


def check_device_error(stream=None) -> tuple[int, int]:
    """Synchronise and read/clear the device error word: (status, site)."""
    site = ctypes.c_uint(0)
    rc = load_library().attn_check_device_error(_stream_handle(stream), ctypes.byref(site))
    return int(rc), int(site.value)


def set_wait_limit_ns(ns: int) -> None:
    load_library().attn_set_wait_limit_ns(int(ns))


def set_exp2_offload(on: bool) -> None:
    """FP8 forward: compute one group of exponentials in eight on the FMA pipe."""
    load_library().attn_set_exp2_offload(int(bool(on)))


def selftest_wait_timeout(stream=None) -> None:
    _check("attn_selftest_wait_timeout",
           load_library().attn_selftest_wait_timeout(_stream_handle(stream)))


def bwd_stages(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale: float, causal: bool,
               stream=None, events=None):
    """attn_bwd as its three C-ABI stages; ``events`` (4 CUDA events, optional)
    are recorded before, between and after them on the same stream."""
    B, H, N, d = q.shape
    lib = load_library()
    h = _stream_handle(stream)
    c = int(bool(causal))
    ev = events or [None] * 4
    if ev[0] is not None:
        ev[0].record(stream)
    _check("attn_bwd_preprocess", lib.attn_bwd_preprocess(o.data_ptr(), dout.data_ptr(),
                                                          lse.data_ptr(), workspace.data_ptr(),
                                                          B, H, N, d, h))
    if ev[1] is not None:
        ev[1].record(stream)
    _check("attn_bwd_main", lib.attn_bwd_main(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                              dout.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                              workspace.data_ptr(), B, H, N, d, float(scale), c, h))
    if ev[2] is not None:
        ev[2].record(stream)
    _check("attn_bwd_dq_convert", lib.attn_bwd_dq_convert(dq.data_ptr(), workspace.data_ptr(),
                                                          B, H, N, d, float(scale), h))
    if ev[3] is not None:
        ev[3].record(stream)
    return dq, dk, dv


def _bhnd_strides(t, layout):
    """Strides of a 4-D CUDA tensor seen as [B, heads, N, d]: layout "bhnd" (the
    tensor is [B, heads, N, d]) or "bnhd" (the tensor is [B, N, heads, d])."""
    sb, s1, s2, sd = t.stride()
    if sd != 1:
        raise ValueError("the last (d) dimension must be contiguous")
    if layout == "bhnd":
        return Strides(sb, s1, s2)
    if layout == "bnhd":
        return Strides(sb, s2, s1)
    raise ValueError(f"unknown layout {layout!r}")


def _bhnd_shape(t, layout):
    B, a, b, d = t.shape
    return (B, a, b, d) if layout == "bhnd" else (B, b, a, d)


def fwd_strided(q, k, v, layout: str = "bnhd", scale: float | None = None, window=(-1, -1),
                o=None, lse=None, stream=None):
    """Forward on bf16 tensors of any strides with a contiguous last dimension.
    ``layout`` says how the 4 dimensions are ordered ("bnhd": [B, N, H, d] as
    produced by most projections; "bhnd": [B, H, N, d]).  Returns (O in the same
    layout as q, LSE [B, H, N])."""
    import torch
    B, H, N, d = _bhnd_shape(q, layout)
    Hk = _bhnd_shape(k, layout)[1]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be a bf16 CUDA tensor")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check("attn_fwd_strided", load_library().attn_fwd_strided(
        q.data_ptr(), _bhnd_strides(q, layout), k.data_ptr(), _bhnd_strides(k, layout),
        v.data_ptr(), _bhnd_strides(v, layout), o.data_ptr(), _bhnd_strides(o, layout),
        lse.data_ptr(), B, H, Hk, N, d, scale, int(window[0]), int(window[1]),
        _stream_handle(stream)))
    return o, lse


def bwd_strided(q, k, v, o, dout, lse, layout: str = "bnhd", scale: float | None = None,
                window=(-1, -1), dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward counterpart of ``fwd_strided``; gradients take the layout of
    their inputs (dq like q, dk like k, dv like v)."""
    import torch
    B, H, N, d = _bhnd_shape(q, layout)
    Hk = _bhnd_shape(k, layout)[1]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = lambda t: _bhnd_strides(t, layout)
    _check("attn_bwd_strided", load_library().attn_bwd_strided(
        q.data_ptr(), st(q), k.data_ptr(), st(k), v.data_ptr(), st(v), o.data_ptr(), st(o),
        dout.data_ptr(), st(dout), lse.data_ptr(), dq.data_ptr(), st(dq), dk.data_ptr(), st(dk),
        dv.data_ptr(), st(dv), workspace.data_ptr(), B, H, Hk, N, d, scale, int(window[0]),
        int(window[1]), _stream_handle(stream)))
    return dq, dk, dv
