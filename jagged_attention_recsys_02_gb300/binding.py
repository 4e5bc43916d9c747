"""Thin Python binding of libgdpa.so (include/gdpa.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  Tensors are torch CUDA tensors (device memory and
streams come from PyTorch); their data pointers and the current stream are
handed to the library.  If the library cannot be loaded the calls raise: no
other implementation stands in for it.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

ACT_SOFTMAX, ACT_SILU, ACT_GELU_TANH, ACT_IDENTITY, ACT_GELU_ERF = 0, 1, 2, 3, 4
ACT_BY_NAME = {"softmax": ACT_SOFTMAX, "silu": ACT_SILU, "gelu_tanh": ACT_GELU_TANH,
               "identity": ACT_IDENTITY, "gelu_erf": ACT_GELU_ERF}
BIAS_NONE, BIAS_RELPOS, BIAS_DENSE = 0, 1, 2

STATUS_NAMES = {0: "GDPA_OK", 1: "GDPA_ERR_INVALID_ARG", 2: "GDPA_ERR_UNSUPPORTED",
                3: "GDPA_ERR_WORKSPACE", 4: "GDPA_ERR_CUDA", 5: "GDPA_ERR_TIMEOUT",
                6: "GDPA_ERR_BAD_OFFSETS"}

# Every symbol include/gdpa.h declares.
EXPORTS = ("gdpa_fwd_workspace_size", "gdpa_fwd", "gdpa_bwd_workspace_size", "gdpa_bwd",
           "gdpa_get_device_status", "gdpa_status_string", "gdpa_last_launch_count",
           "gdpa_timing_enable", "gdpa_timing_collect", "gdpa_fwd_noalloc",
           "gdpa_mxfp8_scale_bytes", "gdpa_quantize_mxfp8", "gdpa_fwd_mxfp8",
           "gdpa_fwd_window", "gdpa_bwd_window", "gdpa_fwd_mxfp8_window",
           "gdpa_block_workspace_size", "gdpa_block_fwd", "gdpa_block_bwd",
           "gdpa_bwd_mxfp8_workspace_size", "gdpa_bwd_mxfp8", "gdpa_bwd_mxfp8_window",
           "gdpa_bwd_rope", "gdpa_selftest_timeout", "gdpa_block_bwd_dbias",
           "gdpa_bwd_mxfp8_rope")
MX_ALONG_CHANNELS, MX_ALONG_TOKENS, MX_NOSAT = 0, 1, 2


class GdpaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")


class gdpa_bias(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("table", ctypes.c_void_p), ("max_rel", ctypes.c_int),
                ("offsets", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libgdpa.so (building it first if asked and needed)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise OSError(f"{path} is missing; run jagged_attention_recsys_02_gb300.build.build()")
            _build.build()
        lib = ctypes.CDLL(path)
        vp, i64, I, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        sz = ctypes.c_size_t
        lib.gdpa_fwd_workspace_size.argtypes = [I, I, I, i64, i64]
        lib.gdpa_fwd_workspace_size.restype = sz
        lib.gdpa_bwd_workspace_size.argtypes = [I, I, I, i64, i64]
        lib.gdpa_bwd_workspace_size.restype = sz
        lib.gdpa_fwd.argtypes = [vp, vp, vp, vp, vp, I, I, I, i64, i64,
                                 ctypes.POINTER(gdpa_bias), I, I, F, vp, vp, vp, sz, vp]
        lib.gdpa_fwd.restype = I
        lib.gdpa_fwd_window.argtypes = [vp, vp, vp, vp, vp, I, I, I, i64, i64,
                                        ctypes.POINTER(gdpa_bias), I, I, I, F, vp, vp, vp, sz, vp]
        lib.gdpa_fwd_window.restype = I
        lib.gdpa_bwd.argtypes = [vp, vp, vp, vp, vp, I, I, I, i64, i64,
                                 ctypes.POINTER(gdpa_bias), I, I, F, vp, vp, vp, vp, vp, vp,
                                 vp, sz, vp]
        lib.gdpa_bwd.restype = I
        lib.gdpa_bwd_window.argtypes = [vp, vp, vp, vp, vp, I, I, I, i64, i64,
                                        ctypes.POINTER(gdpa_bias), I, I, I, F, vp, vp, vp, vp, vp,
                                        vp, vp, vp, sz, vp]
        lib.gdpa_bwd_window.restype = I
        lib.gdpa_bwd_rope.argtypes = [vp, vp, vp, vp, vp, I, I, I, i64, i64,
                                      ctypes.POINTER(gdpa_bias), I, I, I, F, F, vp, vp, vp, vp, vp,
                                      vp, vp, vp, sz, vp]
        lib.gdpa_bwd_rope.restype = I
        lib.gdpa_selftest_timeout.argtypes = [I, vp]
        lib.gdpa_selftest_timeout.restype = I
        lib.gdpa_get_device_status.argtypes = [vp]
        lib.gdpa_get_device_status.restype = I
        lib.gdpa_status_string.argtypes = [I]
        lib.gdpa_status_string.restype = ctypes.c_char_p
        lib.gdpa_last_launch_count.argtypes = []
        lib.gdpa_last_launch_count.restype = I
        lib.gdpa_timing_enable.argtypes = [I]
        lib.gdpa_timing_enable.restype = I
        lib.gdpa_timing_collect.argtypes = [ctypes.POINTER(ctypes.c_float),
                                            ctypes.POINTER(ctypes.c_int), I]
        lib.gdpa_timing_collect.restype = I
        lib.gdpa_mxfp8_scale_bytes.argtypes = [I, I, I, i64, I]
        lib.gdpa_mxfp8_scale_bytes.restype = sz
        lib.gdpa_quantize_mxfp8.argtypes = [vp, vp, I, I, I, i64, I, vp, vp, vp]
        lib.gdpa_quantize_mxfp8.restype = I
        lib.gdpa_fwd_mxfp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, i64, i64,
                                       ctypes.POINTER(gdpa_bias), I, I, F, vp, vp, vp, sz, vp]
        lib.gdpa_fwd_mxfp8.restype = I
        lib.gdpa_fwd_mxfp8_window.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, i64, i64,
                                              ctypes.POINTER(gdpa_bias), I, I, I, F, vp, vp, vp,
                                              sz, vp]
        lib.gdpa_fwd_mxfp8_window.restype = I
        lib.gdpa_block_workspace_size.argtypes = [I, I, I, i64]
        lib.gdpa_block_workspace_size.restype = sz
        lib.gdpa_block_fwd.argtypes = [vp, vp, vp, vp, I, I, I, i64, ctypes.POINTER(gdpa_bias), I,
                                       I, F, vp, vp, sz, vp]
        lib.gdpa_block_fwd.restype = I
        lib.gdpa_block_bwd.argtypes = [vp, vp, vp, vp, I, I, I, i64, ctypes.POINTER(gdpa_bias), I,
                                       I, F, F, vp, vp, vp, vp, vp, sz, vp]
        lib.gdpa_block_bwd.restype = I
        lib.gdpa_block_bwd_dbias.argtypes = [vp, vp, vp, vp, I, I, I, i64,
                                             ctypes.POINTER(gdpa_bias), I, I, F, F, vp, vp, vp, vp,
                                             vp, vp, sz, vp]
        lib.gdpa_block_bwd_dbias.restype = I
        lib.gdpa_bwd_mxfp8_workspace_size.argtypes = [I, I, I, i64, i64]
        lib.gdpa_bwd_mxfp8_workspace_size.restype = sz
        lib.gdpa_bwd_mxfp8.argtypes = list(lib.gdpa_bwd.argtypes)
        lib.gdpa_bwd_mxfp8.restype = I
        lib.gdpa_bwd_mxfp8_window.argtypes = [vp, vp, vp, vp, vp, I, I, I, i64, i64,
                                              ctypes.POINTER(gdpa_bias), I, I, I, F, vp, vp, vp,
                                              vp, vp, vp, vp, sz, vp]
        lib.gdpa_bwd_mxfp8_window.restype = I
        lib.gdpa_bwd_mxfp8_rope.argtypes = list(lib.gdpa_bwd_rope.argtypes)
        lib.gdpa_bwd_mxfp8_rope.restype = I
        _lib = lib
        return lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _bias(bias, max_rel):
    """bias: None, a relative-position table [H, 2*max_rel-1] fp32, or a dense
    jagged bias given as (values fp32 [sum_b H*Lq_b*Lkv_b], offsets int64 [B+1])."""
    if bias is None:
        return None
    if isinstance(bias, tuple):
        values, offsets = bias
        return ctypes.byref(gdpa_bias(BIAS_DENSE, values.data_ptr(), 0, offsets.data_ptr()))
    return ctypes.byref(gdpa_bias(BIAS_RELPOS, bias.data_ptr(), int(max_rel), None))


def _act(act) -> int:
    return ACT_BY_NAME[act] if isinstance(act, str) else int(act)


def _check(code: int, where: str):
    if code != 0:
        raise GdpaError(code, where)


def fwd_workspace_size(B, H, d, Tq, Tkv) -> int:
    return int(load().gdpa_fwd_workspace_size(B, H, d, Tq, Tkv))


def bwd_workspace_size(B, H, d, Tq, Tkv) -> int:
    return int(load().gdpa_bwd_workspace_size(B, H, d, Tq, Tkv))


def gdpa_fwd(q, q_offsets, k, v, kv_offsets, *, act, causal=False, scale, bias=None, max_rel=0,
             window=0, out=None, lse=None, workspace=None, stream=None):
    """Forward pass through the C ABI (gdpa_fwd, or gdpa_fwd_window when
    window > 0).  Returns (out, lse)."""
    lib = load()
    Tq, H, d = q.shape
    Tkv = k.shape[0]
    B = q_offsets.numel() - 1
    a = _act(act)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and a == ACT_SOFTMAX:
        lse = torch.empty((H, Tq), device=q.device, dtype=torch.float32)
    if workspace is None:
        workspace = torch.empty(fwd_workspace_size(B, H, d, Tq, Tkv), device=q.device,
                                dtype=torch.uint8)
    head = (_ptr(q), _ptr(q_offsets), _ptr(k), _ptr(v), _ptr(kv_offsets), B, H, d, Tq, Tkv,
            _bias(bias, max_rel), a, int(bool(causal)))
    tail = (float(scale), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
            _stream(stream))
    if window:
        rc = lib.gdpa_fwd_window(*head, int(window), *tail)
    else:
        rc = lib.gdpa_fwd(*head, *tail)
    _check(rc, "gdpa_fwd_window" if window else "gdpa_fwd")
    return out, lse


def gdpa_bwd(q, q_offsets, k, v, kv_offsets, out, lse, dout, *, act, causal=False, scale,
             bias=None, max_rel=0, window=0, dq=None, dk=None, dv=None, dbias=None,
             rope_base=0.0, workspace=None, stream=None):
    """Backward pass through the C ABI (gdpa_bwd, or gdpa_bwd_window when
    window > 0 or a bias gradient `dbias` fp32 is given, which is added to: the
    table's [H, 2*max_rel-1], or a dense bias's values' layout; gdpa_bwd_rope
    when rope_base > 0, dq and dk then going back through the rotary
    embedding).  Returns (dq, dk, dv)."""
    lib = load()
    Tq, H, d = q.shape
    Tkv = k.shape[0]
    B = q_offsets.numel() - 1
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(bwd_workspace_size(B, H, d, Tq, Tkv), device=q.device,
                                dtype=torch.uint8)
    head = (_ptr(q), _ptr(q_offsets), _ptr(k), _ptr(v), _ptr(kv_offsets), B, H, d, Tq, Tkv,
            _bias(bias, max_rel), _act(act), int(bool(causal)))
    tail = (float(scale), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv))
    ws = (_ptr(workspace), workspace.numel(), _stream(stream))
    if rope_base:
        rc = lib.gdpa_bwd_rope(*head, int(window), float(scale), float(rope_base), *tail[1:],
                               _ptr(dbias), *ws)
        _check(rc, "gdpa_bwd_rope")
    elif window or dbias is not None:
        rc = lib.gdpa_bwd_window(*head, int(window), *tail, _ptr(dbias), *ws)
        _check(rc, "gdpa_bwd_window")
    else:
        rc = lib.gdpa_bwd(*head, *tail, *ws)
        _check(rc, "gdpa_bwd")
    return dq, dk, dv


def selftest_timeout(limit_us: int = 2000, stream=None) -> None:
    """Launch the failure-detection self-test (a wait that times out after
    limit_us and records GDPA_ERR_TIMEOUT in the device status word)."""
    _check(load().gdpa_selftest_timeout(int(limit_us), _stream(stream)), "gdpa_selftest_timeout")


def bwd_mxfp8_workspace_size(B, H, d, Tq, Tkv) -> int:
    return int(load().gdpa_bwd_mxfp8_workspace_size(B, H, d, Tq, Tkv))


def gdpa_bwd_mxfp8(q, q_offsets, k, v, kv_offsets, out, lse, dout, *, causal=False, scale,
                   bias=None, max_rel=0, window=0, dq=None, dk=None, dv=None, dbias=None,
                   rope_base=0.0, workspace=None, stream=None):
    """MXFP8 backward through the C ABI (gdpa_bwd_mxfp8, gdpa_bwd_mxfp8_window
    when window > 0, gdpa_bwd_mxfp8_rope when rope_base > 0 or the bias's
    gradient `dbias` is given, which is added to: the table's layout or a
    dense bias's) on the bf16 tensors of gdpa_bwd, softmax, d = 128.  Returns
    (dq, dk, dv)."""
    lib = load()
    Tq, H, d = q.shape
    Tkv = k.shape[0]
    B = q_offsets.numel() - 1
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(bwd_mxfp8_workspace_size(B, H, d, Tq, Tkv), device=q.device,
                                dtype=torch.uint8)
    head = (_ptr(q), _ptr(q_offsets), _ptr(k), _ptr(v), _ptr(kv_offsets), B, H, d, Tq, Tkv,
            _bias(bias, max_rel), ACT_SOFTMAX, int(bool(causal)))
    tail = (float(scale), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
            _ptr(workspace), workspace.numel(), _stream(stream))
    if rope_base or dbias is not None:
        rc = lib.gdpa_bwd_mxfp8_rope(*head, int(window), float(scale), float(rope_base), *tail[1:7],
                                     _ptr(dbias), *tail[7:])
        _check(rc, "gdpa_bwd_mxfp8_rope")
    elif window:
        rc = lib.gdpa_bwd_mxfp8_window(*head, int(window), *tail)
        _check(rc, "gdpa_bwd_mxfp8_window")
    else:
        rc = lib.gdpa_bwd_mxfp8(*head, *tail)
        _check(rc, "gdpa_bwd_mxfp8")
    return dq, dk, dv


def block_workspace_size(B, H, d, T) -> int:
    return int(load().gdpa_block_workspace_size(B, H, d, T))


def gdpa_block_fwd(q, offsets, k, v, *, act, causal=False, scale, bias=None, max_rel=0, out=None,
                   workspace=None, stream=None):
    """Block-aligned attention forward (64-token blocks) through the C ABI.
    Returns out."""
    lib = load()
    T, H, d = q.shape
    B = offsets.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = torch.empty(block_workspace_size(B, H, d, T), device=q.device,
                                dtype=torch.uint8)
    rc = lib.gdpa_block_fwd(_ptr(q), _ptr(offsets), _ptr(k), _ptr(v), B, H, d, T,
                            _bias(bias, max_rel), _act(act), int(bool(causal)), float(scale),
                            _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "gdpa_block_fwd")
    return out


def gdpa_block_bwd(q, offsets, k, v, dout, *, act, causal=False, scale, bias=None, max_rel=0,
                   rope_base=0.0, dq=None, dk=None, dv=None, dbias=None, workspace=None,
                   stream=None):
    """Block-aligned attention backward through the C ABI (gdpa_block_bwd, or
    gdpa_block_bwd_dbias when the bias's gradient `dbias` fp32 is given, which
    is added to: the table's [H, 2*max_rel-1], or a dense bias's values'
    layout).  Returns (dq, dk, dv); with rope_base > 0, dq and dk are gradients
    of the un-rotated q and k."""
    lib = load()
    T, H, d = q.shape
    B = offsets.numel() - 1
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(block_workspace_size(B, H, d, T), device=q.device,
                                dtype=torch.uint8)
    head = (_ptr(q), _ptr(offsets), _ptr(k), _ptr(v), B, H, d, T, _bias(bias, max_rel), _act(act),
            int(bool(causal)), float(scale), float(rope_base), _ptr(dout), _ptr(dq), _ptr(dk),
            _ptr(dv))
    ws = (_ptr(workspace), workspace.numel(), _stream(stream))
    if dbias is not None:
        rc = lib.gdpa_block_bwd_dbias(*head, _ptr(dbias), *ws)
        _check(rc, "gdpa_block_bwd_dbias")
    else:
        rc = lib.gdpa_block_bwd(*head, *ws)
        _check(rc, "gdpa_block_bwd")
    return dq, dk, dv


def device_status(stream=None) -> int:
    return int(load().gdpa_get_device_status(_stream(stream)))


def last_launch_count() -> int:
    return int(load().gdpa_last_launch_count())


def timing_enable(on: bool = True) -> None:
    load().gdpa_timing_enable(1 if on else 0)


def timing_collect(max_n: int = 4096):
    """Per-launch durations (ms) of the main kernels recorded while timing was
    enabled: returns (fwd_ms list, bwd_ms list)."""
    ms = (ctypes.c_float * max_n)()
    kind = (ctypes.c_int * max_n)()
    n = load().gdpa_timing_collect(ms, kind, max_n)
    if n < 0:
        raise GdpaError(4, "gdpa_timing_collect")
    f = [ms[i] for i in range(n) if kind[i] == 0]
    b = [ms[i] for i in range(n) if kind[i] == 1]
    return f, b


def quantize_mxfp8(x, offsets=None, *, mode, nosat=False, codes=None, scales=None, stream=None):
    """MXFP8 block quantisation through the C ABI (nosat: the saturation-free
    block scale, GDPA_MX_NOSAT).  Returns (codes u8, scales u8)."""
    lib = load()
    T, H, d = x.shape
    B = offsets.numel() - 1 if offsets is not None else 0
    mode = int(mode) | (MX_NOSAT if nosat else 0)
    if codes is None:
        codes = torch.empty((T, H, d), device=x.device, dtype=torch.uint8)
    if scales is None:
        n = lib.gdpa_mxfp8_scale_bytes(max(B, 0), H, d, T, mode)
        shape = (T, H, d // 32) if not mode & MX_ALONG_TOKENS else (n // (H * d), H, d)
        scales = torch.empty(shape, device=x.device, dtype=torch.uint8)
    rc = lib.gdpa_quantize_mxfp8(_ptr(x), _ptr(offsets), B, H, d, T, mode, _ptr(codes),
                                 _ptr(scales), _stream(stream))
    _check(rc, "gdpa_quantize_mxfp8")
    return codes, scales


def gdpa_fwd_mxfp8(q_codes, q_scales, q_offsets, k_codes, k_scales, v_codes, v_scales, kv_offsets,
                   *, causal=False, scale, bias=None, max_rel=0, window=0, out=None, lse=None,
                   workspace=None, stream=None):
    """MXFP8 forward (softmax) through the C ABI (gdpa_fwd_mxfp8, or
    gdpa_fwd_mxfp8_window when window > 0).  Returns (out bf16, lse)."""
    lib = load()
    Tq, H, d = q_codes.shape
    Tkv = k_codes.shape[0]
    B = q_offsets.numel() - 1
    if out is None:
        out = torch.empty((Tq, H, d), device=q_codes.device, dtype=torch.bfloat16)
    if lse is None:
        lse = torch.empty((H, Tq), device=q_codes.device, dtype=torch.float32)
    if workspace is None:
        workspace = torch.empty(fwd_workspace_size(B, H, d, Tq, Tkv), device=q_codes.device,
                                dtype=torch.uint8)
    head = (_ptr(q_codes), _ptr(q_scales), _ptr(q_offsets), _ptr(k_codes), _ptr(k_scales),
            _ptr(v_codes), _ptr(v_scales), _ptr(kv_offsets), B, H, d, Tq, Tkv,
            _bias(bias, max_rel), ACT_SOFTMAX, int(bool(causal)))
    tail = (float(scale), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
            _stream(stream))
    if window:
        rc = lib.gdpa_fwd_mxfp8_window(*head, int(window), *tail)
    else:
        rc = lib.gdpa_fwd_mxfp8(*head, *tail)
    _check(rc, "gdpa_fwd_mxfp8_window" if window else "gdpa_fwd_mxfp8")
    return out, lse
