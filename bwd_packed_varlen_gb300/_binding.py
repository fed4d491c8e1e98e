"""ctypes binding of libteattn.so: argument marshalling only.

Names mirror the C ABI (``te_attn_fwd_thd`` -> :func:`fwd`, ``te_attn_bwd_thd`` ->
:func:`bwd`). Tensors are passed by ``data_ptr()``; the current torch CUDA stream
is passed as the launch stream; output and workspace buffers are allocated with
torch when the caller does not supply them.
"""

from __future__ import annotations

import contextlib
import ctypes
import os

import torch

MASK_PADDING = 1
MASK_PADDING_CAUSAL = 2
MASK_PADDING_CAUSAL_BOTTOM_RIGHT = 3
_MASK_NAMES = {"padding": MASK_PADDING, "padding_causal": MASK_PADDING_CAUSAL,
               "padding_causal_bottom_right": MASK_PADDING_CAUSAL_BOTTOM_RIGHT}
_DTYPES = {torch.float16: 0, torch.bfloat16: 1}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "lib", "libteattn.so")
_LIB_DEBUG_PATH = os.path.join(_HERE, "lib", "libteattn_debug.so")
_libs = {}
_use_debug = False


class TeAttnError(RuntimeError):
    """A libteattn call returned a nonzero status."""

    def __init__(self, code: int, msg: str):
        super().__init__(f"libteattn error {code}: {msg}")
        self.code = code


def library_path(debug: bool = False) -> str:
    return _LIB_DEBUG_PATH if debug else _LIB_PATH


@contextlib.contextmanager
def debug_build():
    """Within this block every call goes to ``libteattn_debug.so``, the build that
    bounds-checks each computed global offset and records a bad one as
    ``TE_STATUS_OUT_OF_BOUNDS`` (bit 4) in the call's status word."""
    global _use_debug
    old = _use_debug
    _use_debug = True
    try:
        yield library(debug=True)
    finally:
        _use_debug = old


def library(debug: bool = None) -> ctypes.CDLL:
    """Load libteattn.so, or its debug build (raises if it has not been built).
    ``debug=None`` picks the build selected by :func:`debug_build`."""
    debug = _use_debug if debug is None else bool(debug)
    if debug in _libs:
        return _libs[debug]
    path = library_path(debug)
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; "
            "g.build()'` (or python bwd_packed_varlen_gb300/build.py)")
    L = ctypes.CDLL(path)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.te_attn_version.restype = i32
    L.te_attn_version.argtypes = []
    for name in ("te_attn_fwd_workspace_size", "te_attn_bwd_workspace_size",
                 "te_attn_bwd_fused_workspace_size"):
        fn = getattr(L, name)
        fn.restype = sz
        fn.argtypes = [i32] * 6
    L.te_attn_fwd_thd.restype = i32
    L.te_attn_fwd_thd.argtypes = [vp] * 5 + [vp] * 4 + [i32] * 8 + [f32, i32, i32, vp, sz, vp]
    L.te_attn_bwd_thd.restype = i32
    L.te_attn_bwd_thd.argtypes = [vp] * 9 + [vp] * 4 + [i32] * 8 + [f32, i32, i32, vp, sz, vp]
    L.te_attn_bwd_thd_fused.restype = i32
    L.te_attn_bwd_thd_fused.argtypes = [vp] * 9 + [vp] * 4 + [i32] * 8 + [f32, i32, i32, vp, sz, vp]
    L.te_attn_bwd_thd_ev.restype = i32
    L.te_attn_bwd_thd_ev.argtypes = [vp] * 9 + [vp] * 4 + [i32] * 8 + [f32, i32, i32, vp, sz, vp, vp]
    L.te_attn_bwd_thd_noalloc.restype = i32
    L.te_attn_bwd_thd_noalloc.argtypes = [vp] * 9 + [vp] * 4 + [i32] * 8 + [f32, i32, i32, vp]
    L.te_attn_fwd_sbhd.restype = i32
    L.te_attn_fwd_sbhd.argtypes = [vp] * 5 + [vp] * 2 + [i32] * 6 + [f32, i32, i32, vp, sz, vp]
    L.te_attn_bwd_sbhd.restype = i32
    L.te_attn_bwd_sbhd.argtypes = [vp] * 9 + [vp] * 2 + [i32] * 6 + [f32, i32, i32, vp, sz, vp]
    L.te_attn_fwd_e4m3_workspace_size.restype = sz
    L.te_attn_fwd_e4m3_workspace_size.argtypes = [i32] * 6
    L.te_attn_fwd_thd_e4m3.restype = i32
    L.te_attn_fwd_thd_e4m3.argtypes = ([vp] * 5 + [vp] * 4 + [i32] * 8 + [f32] * 4 +
                                        [i32, vp, sz, vp])
    L.te_attn_read_status.restype = i32
    L.te_attn_read_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int), vp]
    L.te_attn_last_error.restype = ctypes.c_char_p
    L.te_attn_last_error.argtypes = []
    L.te_attn_profile_enable.restype = i32
    L.te_attn_profile_enable.argtypes = [i32]
    L.te_attn_profile_read.restype = i32
    L.te_attn_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]
    L.te_attn_read_status_noalloc.restype = i32
    L.te_attn_read_status_noalloc.argtypes = [ctypes.POINTER(ctypes.c_int), vp]
    L.te_attn_selftest_wait_timeout.restype = i32
    L.te_attn_selftest_wait_timeout.argtypes = [vp, sz, ctypes.c_uint, vp]
    _libs[debug] = L
    return L


def version() -> int:
    return int(library().te_attn_version())


def _mask(mask_type) -> int:
    if isinstance(mask_type, str):
        if mask_type not in _MASK_NAMES:
            raise ValueError(f"unknown mask_type {mask_type!r}")
        return _MASK_NAMES[mask_type]
    return int(mask_type)


def _check(rc: int):
    if rc != 0:
        raise TeAttnError(rc, library().te_attn_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _on(t):
    """Make t's device current for the call: the library launches on, and looks up
    per-device state of, the current device."""
    return torch.cuda.device(t.device)


def _need_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (there is no CPU path)")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")


def _cu(*cus):
    for c in cus:
        if c.dtype != torch.int32:
            raise ValueError("cu_seqlens tensors must be int32")


def fwd_workspace_size(batch, total_q, total_kv, hq, hkv, d) -> int:
    return int(library().te_attn_fwd_workspace_size(batch, total_q, total_kv, hq, hkv, d))


def bwd_workspace_size(batch, total_q, total_kv, hq, hkv, d) -> int:
    return int(library().te_attn_bwd_workspace_size(batch, total_q, total_kv, hq, hkv, d))


def bwd_fused_workspace_size(batch, total_q, total_kv, hq, hkv, d) -> int:
    """Workspace bytes of ``te_attn_bwd_thd_fused`` (0 for head dims above 128)."""
    return int(library().te_attn_bwd_fused_workspace_size(batch, total_q, total_kv, hq, hkv, d))


def fwd(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded,
        attn_scale, mask_type="padding", max_seqlen_q=0, max_seqlen_kv=0, out=None, lse=None,
        workspace=None, stream=None):
    """``te_attn_fwd_thd``: returns ``(out, lse)``; out ``[T_q, hq, d]`` in q's dtype,
    lse ``[T_q, hq]`` fp32."""
    L = library()
    _need_cuda(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
               cu_seqlens_kv_padded, out, lse, workspace)
    _cu(cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded)
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype, float16 or bfloat16")
    Tq, hq, d = q.shape
    Tk, hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Tq, hq), dtype=torch.float32, device=q.device)
    need = fwd_workspace_size(B, Tq, Tk, hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    with _on(q):
        rc = L.te_attn_fwd_thd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
            _ptr(cu_seqlens_kv), _ptr(cu_seqlens_q_padded), _ptr(cu_seqlens_kv_padded), B, Tq, Tk,
            int(max_seqlen_q), int(max_seqlen_kv), hq, hkv, d, float(attn_scale), _mask(mask_type),
            _DTYPES[q.dtype], _ptr(workspace), workspace.numel(), ctypes.c_void_p(st))
    _check(rc)
    return out, lse


def bwd(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
        cu_seqlens_kv_padded, attn_scale, mask_type="padding", max_seqlen_q=0,
        max_seqlen_kv=0, dq=None, dk=None, dv=None, workspace=None, stream=None,
        dq_done=None, fused=False):
    """``te_attn_bwd_thd``: returns ``(dq, dk, dv)`` in q's dtype. With ``dq_done``
    (a ``torch.cuda.Event``) it calls ``te_attn_bwd_thd_ev`` instead, which records
    that event on the stream as soon as dq is final (before dk/dv are computed).
    ``fused=True`` calls ``te_attn_bwd_thd_fused`` (head dims up to 128)."""
    L = library()
    _need_cuda(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
               cu_seqlens_kv_padded, dq, dk, dv, workspace)
    _cu(cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded)
    if q.dtype not in _DTYPES or any(t.dtype != q.dtype for t in (k, v, out, dout)):
        raise ValueError("q, k, v, out, dout must share one dtype, float16 or bfloat16")
    if lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    Tq, hq, d = q.shape
    Tk, hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if fused and dq_done is not None:
        raise ValueError("the fused backward records no dq hand-over event")
    need = (bwd_fused_workspace_size if fused else bwd_workspace_size)(B, Tq, Tk, hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
            _ptr(dv), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), _ptr(cu_seqlens_q_padded),
            _ptr(cu_seqlens_kv_padded), B, Tq, Tk, int(max_seqlen_q), int(max_seqlen_kv), hq, hkv,
            d, float(attn_scale), _mask(mask_type), _DTYPES[q.dtype], _ptr(workspace),
            workspace.numel(), ctypes.c_void_p(st))
    with _on(q):
        if fused:
            rc = L.te_attn_bwd_thd_fused(*args)
        elif dq_done is None:
            rc = L.te_attn_bwd_thd(*args)
        else:
            if dq_done.cuda_event == 0:  # torch creates the CUDA event on its first record
                dq_done.record(torch.cuda.ExternalStream(st) if stream is not None
                               else torch.cuda.current_stream(q.device))
            rc = L.te_attn_bwd_thd_ev(*args, ctypes.c_void_p(dq_done.cuda_event))
    _check(rc)
    return dq, dk, dv


def fwd_e4m3(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded,
             attn_scale, q_descale, k_descale, v_descale, mask_type="padding", max_seqlen_q=0,
             max_seqlen_kv=0, out=None, lse=None, workspace=None, stream=None):
    """``te_attn_fwd_thd_e4m3``: q, k, v ``torch.float8_e4m3fn`` (packed layout) with
    per-tensor descale factors; returns ``(out bf16 [T_q, hq, d], lse [T_q, hq])``."""
    L = library()
    _need_cuda(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
               cu_seqlens_kv_padded, out, lse, workspace)
    _cu(cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded)
    f8 = getattr(torch, "float8_e4m3fn", None)
    if f8 is None or any(t.dtype != f8 for t in (q, k, v)):
        raise ValueError("q, k, v must be torch.float8_e4m3fn")
    Tq, hq, d = q.shape
    Tk, hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    out = torch.empty((Tq, hq, d), dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty((Tq, hq), dtype=torch.float32, device=q.device) if lse is None else lse
    need = int(L.te_attn_fwd_e4m3_workspace_size(B, Tq, Tk, hq, hkv, d))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    with _on(q):
        _check(L.te_attn_fwd_thd_e4m3(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv),
            _ptr(cu_seqlens_q_padded), _ptr(cu_seqlens_kv_padded), B, Tq, Tk, int(max_seqlen_q),
            int(max_seqlen_kv), hq, hkv, d, float(attn_scale), float(q_descale), float(k_descale),
            float(v_descale), _mask(mask_type), _ptr(workspace), workspace.numel(),
            ctypes.c_void_p(st)))
    return out, lse


def fwd_sbhd(q, k, v, cu_seqlens_q, cu_seqlens_kv, attn_scale, mask_type="padding", out=None,
             lse=None, workspace=None, stream=None):
    """``te_attn_fwd_sbhd``: q ``[S_q, B, hq, d]``, k/v ``[S_kv, B, hkv, d]``, real
    lengths from ``cu_seqlens_q/kv``; returns ``(out [S_q, B, hq, d], lse [S_q, B, hq])``."""
    L = library()
    _need_cuda(q, k, v, cu_seqlens_q, cu_seqlens_kv, out, lse, workspace)
    _cu(cu_seqlens_q, cu_seqlens_kv)
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype, float16 or bfloat16")
    Sq, B, hq, d = q.shape
    Sk, Bk, hkv, _ = k.shape
    if Bk != B or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q, k, v must be [S, B, h, d] with one batch size; v shaped like k")
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((Sq, B, hq), dtype=torch.float32, device=q.device) if lse is None else lse
    need = fwd_workspace_size(B, Sq * B, Sk * B, hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    with _on(q):
        _check(L.te_attn_fwd_sbhd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv),
            B, Sq, Sk, hq, hkv, d, float(attn_scale), _mask(mask_type), _DTYPES[q.dtype],
            _ptr(workspace), workspace.numel(), ctypes.c_void_p(st)))
    return out, lse


def bwd_sbhd(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_kv, attn_scale,
             mask_type="padding", dq=None, dk=None, dv=None, workspace=None, stream=None):
    """``te_attn_bwd_sbhd``: returns ``(dq, dk, dv)`` in the shapes of q, k, v."""
    L = library()
    _need_cuda(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_kv, dq, dk, dv, workspace)
    _cu(cu_seqlens_q, cu_seqlens_kv)
    if q.dtype not in _DTYPES or any(t.dtype != q.dtype for t in (k, v, out, dout)):
        raise ValueError("q, k, v, out, dout must share one dtype, float16 or bfloat16")
    if lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    Sq, B, hq, d = q.shape
    Sk, Bk, hkv, _ = k.shape
    if Bk != B or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q, k, v must be [S, B, h, d] with one batch size; v shaped like k")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = bwd_workspace_size(B, Sq * B, Sk * B, hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    with _on(q):
        _check(L.te_attn_bwd_sbhd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
            _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), B, Sq, Sk, hq, hkv, d, float(attn_scale),
            _mask(mask_type), _DTYPES[q.dtype], _ptr(workspace), workspace.numel(), ctypes.c_void_p(st)))
    return dq, dk, dv


def read_status(workspace, stream=None) -> int:
    """Synchronise and return the device status word of the last call that used
    ``workspace`` (0 clean; bit 1 inconsistent cu_seqlens; bit 2 wait timeout)."""
    L = library()
    st = stream if stream is not None else torch.cuda.current_stream(workspace.device).cuda_stream
    val = ctypes.c_int(0)
    with _on(workspace):
        _check(L.te_attn_read_status(_ptr(workspace), ctypes.byref(val), ctypes.c_void_p(st)))
    return int(val.value)


KERNELS = ("schedule", "fwd", "zero_fill", "delta", "dkdv", "dq", "widen_e4m3", "bwd_fused",
           "dq_convert")


def profile_enable(on: bool = True) -> None:
    """Bracket every later launch with CUDA events on its stream (te_attn_profile_enable)."""
    _check(library().te_attn_profile_enable(1 if on else 0))


def profile_read() -> dict:
    """Per-kernel ``{name: (total_ms, launches)}`` since the last read (te_attn_profile_read)."""
    n = len(KERNELS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int * n)()
    _check(library().te_attn_profile_read(ms, cnt))
    return {KERNELS[i]: (float(ms[i]), int(cnt[i])) for i in range(n)}


def bwd_noalloc(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                cu_seqlens_kv_padded, attn_scale, mask_type="padding", max_seqlen_q=0,
                max_seqlen_kv=0, dq=None, dk=None, dv=None, stream=None):
    """``te_attn_bwd_thd_noalloc``: the backward pass with the library's built-in
    scratch array instead of a workspace, for callers that cannot allocate device
    memory (the outputs here are still allocated by torch when not supplied)."""
    L = library()
    _need_cuda(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
               cu_seqlens_kv_padded, dq, dk, dv)
    _cu(cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded)
    if q.dtype not in _DTYPES or any(t.dtype != q.dtype for t in (k, v, out, dout)):
        raise ValueError("q, k, v, out, dout must share one dtype, float16 or bfloat16")
    Tq, hq, d = q.shape
    Tk, hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    st = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    with _on(q):
        rc = L.te_attn_bwd_thd_noalloc(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
            _ptr(dv), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), _ptr(cu_seqlens_q_padded),
            _ptr(cu_seqlens_kv_padded), B, Tq, Tk, int(max_seqlen_q), int(max_seqlen_kv), hq, hkv,
            d, float(attn_scale), _mask(mask_type), _DTYPES[q.dtype], ctypes.c_void_p(st))
    _check(rc)
    return dq, dk, dv


def read_status_noalloc(device=None, stream=None) -> int:
    """``te_attn_read_status_noalloc``: synchronise and return the status word of the
    last :func:`bwd_noalloc` call on ``device`` (default: the current device)."""
    L = library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        st = stream if stream is not None else torch.cuda.current_stream(dev).cuda_stream
        val = ctypes.c_int(0)
        _check(L.te_attn_read_status_noalloc(ctypes.byref(val), ctypes.c_void_p(st)))
    return int(val.value)


def selftest_wait_timeout(workspace, limit_us: int = 1000, stream=None) -> None:
    """``te_attn_selftest_wait_timeout``: launch the bounded-wait unwind self-test on
    ``workspace`` (a CUDA uint8 tensor of at least 256 bytes); read the outcome with
    :func:`read_status` and the workspace's header words 8..11."""
    L = library()
    _need_cuda(workspace)
    with _on(workspace):
        st = stream if stream is not None else torch.cuda.current_stream(workspace.device).cuda_stream
        _check(L.te_attn_selftest_wait_timeout(_ptr(workspace), workspace.numel(), int(limit_us),
                                               ctypes.c_void_p(st)))
