"""ctypes front end of the fp64 oracle (test infrastructure only), plus the
rotary embedding (RoPE) in numpy float64.

All inputs are converted to float64 numpy arrays before the call; the bf16
values the GPU sees convert to float64 exactly, so the oracle works on the
same numbers.  Layouts: q/out [Tq, H, d], k/v [Tkv, H, d], lse [H, Tq],
bias table [H, 2*max_rel-1], offsets int32 [B+1].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

ACT_SOFTMAX, ACT_SILU, ACT_GELU_TANH, ACT_IDENTITY, ACT_GELU_ERF = 0, 1, 2, 3, 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdpa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gdpa_oracle.c into a shared object (gcc, OpenMP, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-D_DEFAULT_SOURCE",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        up = ctypes.POINTER(ctypes.c_uint8)
        I, D = ctypes.c_int, ctypes.c_double
        lp = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_fwd.argtypes = [dp, ip, dp, dp, ip, I, I, I, dp, I, I, I, I, I, D, dp, dp, dp, lp]
        lib.oracle_fwd.restype = I
        lib.oracle_bwd.argtypes = [dp, ip, dp, dp, ip, I, I, I, dp, I, I, I, I, I, D, dp, dp, dp, dp, dp,
                                   dp, lp]
        lib.oracle_bwd.restype = I
        lib.oracle_e4m3_encode.argtypes = [D]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = D
        lib.oracle_e8m0_scale.argtypes = [D]
        lib.oracle_e8m0_scale.restype = ctypes.c_uint8
        lib.oracle_quant_rows.argtypes = [dp, ctypes.c_long, I, I, I, up, up]
        lib.oracle_quant_rows.restype = None
        lib.oracle_quant_cols.argtypes = [dp, ip, I, I, I, I, up, up]
        lib.oracle_quant_cols.restype = None
        lib.oracle_e8m0_nosat.argtypes = [D]
        lib.oracle_e8m0_nosat.restype = ctypes.c_uint8
        lib.oracle_round_blocks_2d.argtypes = [dp, ctypes.c_long, ctypes.c_long]
        lib.oracle_round_blocks_2d.restype = None
        lib.oracle_bwd_mx.argtypes = [dp, dp, dp, dp, dp, dp, dp, ip, ip, I, I, I, dp, I, I, I, D,
                                      dp, dp, I, dp, dp, dp, dp, lp]
        lib.oracle_bwd_mx.restype = I
        _lib = lib
        return lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _p(a: np.ndarray, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _bias_arg(bias, H, max_rel):
    if bias is None:
        return None, ctypes.POINTER(ctypes.c_double)()
    b = _f64(bias)
    assert b.shape == (H, 2 * max_rel - 1), b.shape
    return b, _p(b, ctypes.c_double)


def dense_bias_offsets(q_offsets, kv_offsets, H: int) -> np.ndarray:
    """Element offset of each sample's [H][Lq][Lkv] block in a dense jagged
    bias: H * prefix sums of Lq_b * Lkv_b (int64 [B+1])."""
    qo, ko = _i32(q_offsets).astype(np.int64), _i32(kv_offsets).astype(np.int64)
    o = np.zeros(len(qo), dtype=np.int64)
    o[1:] = np.cumsum(H * np.diff(qo) * np.diff(ko))
    return o


def _dense_arg(dense_bias, qo, ko, H):
    if dense_bias is None:
        return None, ctypes.POINTER(ctypes.c_double)(), ctypes.POINTER(ctypes.c_int64)()
    dv = _f64(dense_bias).reshape(-1)
    off = np.ascontiguousarray(dense_bias_offsets(qo, ko, H))
    assert dv.size == off[-1], (dv.size, off[-1])
    return (dv, off), _p(dv, ctypes.c_double), _p(off, ctypes.c_int64)


def fwd(q, q_offsets, k, v, kv_offsets, *, act: int, causal: bool = False, scale: float,
        bias=None, max_rel: int = 0, window: int = 0, block: int = 0, dense_bias=None):
    """Forward pass.  Returns (out [Tq,H,d] float64, lse [H,Tq] float64).

    lse is the natural-log row logsumexp for softmax (-inf for a row with no
    key) and 0 for the GDPA activations.  window > 0 keeps only the pairs
    with |i - j| < window (sliding-window attention; needs Lq == Lkv).
    block > 0 keeps only the pairs inside one block of `block` tokens, the
    blocks starting at each sample's first token (block-aligned attention;
    needs Lq == Lkv).  dense_bias, instead of the table, gives one bias value
    per (head, query, key): the samples' [H][Lq_b][Lkv_b] blocks one after
    another (dense_bias_offsets)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    qo, ko = _i32(q_offsets), _i32(kv_offsets)
    Tq, H, d = q.shape
    B = len(qo) - 1
    assert k.shape[1:] == (H, d) and v.shape == k.shape
    assert qo[-1] == Tq and ko[-1] == k.shape[0]
    out = np.zeros((Tq, H, d), dtype=np.float64)
    lse = np.zeros((H, Tq), dtype=np.float64)
    keep, bp = _bias_arg(bias, H, max_rel)
    keep_d, dp_, op_ = _dense_arg(dense_bias, qo, ko, H)
    rc = _load().oracle_fwd(_p(q, ctypes.c_double), _p(qo, ctypes.c_int32),
                            _p(k, ctypes.c_double), _p(v, ctypes.c_double),
                            _p(ko, ctypes.c_int32), B, H, d, bp, int(max_rel), int(act),
                            int(bool(causal)), int(window), int(block), float(scale),
                            _p(out, ctypes.c_double), _p(lse, ctypes.c_double), dp_, op_)
    if rc != 0:
        raise ValueError("oracle_fwd rejected its arguments")
    del keep
    return out, lse


def bwd(q, q_offsets, k, v, kv_offsets, dout, *, act: int, causal: bool = False, scale: float,
        bias=None, max_rel: int = 0, window: int = 0, block: int = 0, want_dbias: bool = False,
        dense_bias=None):
    """Backward pass.  Returns (dq, dk, dv) as float64 arrays, and with
    want_dbias also the bias's gradient: the table's [H, 2*max_rel-1], or with
    a dense bias one value per pair in its layout (dS): (dq, dk, dv, dbias)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    qo, ko = _i32(q_offsets), _i32(kv_offsets)
    Tq, H, d = q.shape
    B = len(qo) - 1
    assert do.shape == q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    if want_dbias and dense_bias is not None:  # the dense bias's gradient: ds, same layout
        dbias = np.zeros(int(dense_bias_offsets(qo, ko, H)[-1]), dtype=np.float64)
    else:
        dbias = np.zeros((H, 2 * max(int(max_rel), 1) - 1), dtype=np.float64) if want_dbias else None
    keep, bp = _bias_arg(bias, H, max_rel)
    keep_d, dp_, op_ = _dense_arg(dense_bias, qo, ko, H)
    rc = _load().oracle_bwd(_p(q, ctypes.c_double), _p(qo, ctypes.c_int32),
                            _p(k, ctypes.c_double), _p(v, ctypes.c_double),
                            _p(ko, ctypes.c_int32), B, H, d, bp, int(max_rel), int(act),
                            int(bool(causal)), int(window), int(block), float(scale),
                            _p(do, ctypes.c_double), _p(dq, ctypes.c_double),
                            _p(dk, ctypes.c_double), _p(dv, ctypes.c_double),
                            _p(dbias, ctypes.c_double) if dbias is not None
                            else ctypes.POINTER(ctypes.c_double)(), dp_, op_)
    if rc != 0:
        raise ValueError("oracle_bwd rejected its arguments")
    del keep
    return (dq, dk, dv, dbias) if want_dbias else (dq, dk, dv)


def e4m3_encode(x: float) -> int:
    return int(_load().oracle_e4m3_encode(float(x)))


def e4m3_decode(c: int) -> float:
    return float(_load().oracle_e4m3_decode(int(c) & 0xFF))


def e8m0_scale(amax: float) -> int:
    return int(_load().oracle_e8m0_scale(float(amax)))


def quant_rows(x, nosat: bool = False):
    """MXFP8 along the channel axis: x [T,H,d] -> (codes u8 [T,H,d], scales u8 [T,H,d/32]).

    Block scale: the OCP one, 2^(floor(log2 amax) - 8), or with nosat the
    saturation-free one (smallest power of two X with amax / X <= 448)."""
    x = _f64(x)
    T, H, d = x.shape
    assert d % 32 == 0
    codes = np.zeros((T, H, d), dtype=np.uint8)
    scales = np.zeros((T, H, d // 32), dtype=np.uint8)
    _load().oracle_quant_rows(_p(x, ctypes.c_double), T, H, d, int(bool(nosat)),
                              _p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8))
    return codes, scales


def quant_cols(x, offsets, nosat: bool = False):
    """MXFP8 along tokens, in 32-token blocks aligned to each sample's start
    (block scale as in quant_rows).

    x [T,H,d] -> (codes u8 [T,H,d], scales u8 [NB,H,d]) with NB = sum ceil(L_b/32)."""
    x = _f64(x)
    o = _i32(offsets)
    T, H, d = x.shape
    B = len(o) - 1
    nb = int(sum((int(o[b + 1]) - int(o[b]) + 31) // 32 for b in range(B)))
    codes = np.zeros((T, H, d), dtype=np.uint8)
    scales = np.zeros((max(nb, 0), H, d), dtype=np.uint8)
    _load().oracle_quant_cols(_p(x, ctypes.c_double), _p(o, ctypes.c_int32), B, H, d,
                              int(bool(nosat)), _p(codes, ctypes.c_uint8),
                              _p(scales, ctypes.c_uint8))
    return codes, scales


def e8m0_nosat(amax: float) -> int:
    """E8M0 code of the smallest power of two X with amax / X <= 448."""
    return int(_load().oracle_e8m0_nosat(float(amax)))


def round_blocks_2d(m):
    """m [R, C] rounded to E4M3 in 32 x 32 blocks from (0, 0), each block with
    the scale e8m0_nosat(block amax); returns a new float64 array."""
    m = np.array(_f64(m), dtype=np.float64, copy=True, order="C")
    assert m.ndim == 2
    _load().oracle_round_blocks_2d(_p(m, ctypes.c_double), m.shape[0], m.shape[1])
    return m


_E4M3 = None


def _e4m3_table():
    global _E4M3
    if _E4M3 is None:
        _E4M3 = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return _E4M3


def dequant_rows(x, nosat: bool = False):
    """x quantised along channels (quant_rows) and decoded back to float64."""
    codes, scales = quant_rows(x, nosat)
    return _e4m3_table()[codes] * np.exp2(scales.astype(np.float64) - 127).repeat(32, axis=2)


def dequant_cols(x, offsets, nosat: bool = False):
    """x quantised along tokens (quant_cols) and decoded back to float64."""
    o = _i32(offsets)
    codes, scales = quant_cols(x, o, nosat)
    dec = _e4m3_table()[codes]
    out = np.zeros_like(dec)
    k = 0
    for b in range(len(o) - 1):
        for r in range((int(o[b + 1]) - int(o[b]) + 31) // 32):
            t0 = int(o[b]) + 32 * r
            t1 = min(t0 + 32, int(o[b + 1]))
            out[t0:t1] = dec[t0:t1] * np.exp2(scales[k].astype(np.float64) - 127)[None]
            k += 1
    return out


def bwd_mx_operands(qd, qt, kd, kt, vd, dod, dot, q_offsets, kv_offsets, lse, delta, *,
                    causal: bool = False, scale: float, bias=None, max_rel: int = 0,
                    window: int = 0, round_ps: bool = True, dense_bias=None):
    """Softmax backward with each product on its own operand version (the
    definition at the MXFP8 backward section of gdpa_oracle.c): qd, kd, vd, dod
    feed the channel contractions (S, dP), qt, kt, dot the token contractions
    (dK, dQ, dV); lse and delta [H, Tq] are given.  P and dS are rounded to
    E4M3 in 32 x 32 blocks when round_ps.  dense_bias (in the layout of
    dense_bias_offsets) replaces the table.  Returns (dq, dk, dv) float64."""
    arrs = [_f64(a) for a in (qd, qt, kd, kt, vd, dod, dot)]
    qo, ko = _i32(q_offsets), _i32(kv_offsets)
    Tq, H, d = arrs[0].shape
    B = len(qo) - 1
    lse_a, delta_a = _f64(lse), _f64(delta)
    assert lse_a.shape == (H, Tq) and delta_a.shape == (H, Tq)
    dq = np.zeros((Tq, H, d))
    dk = np.zeros(arrs[2].shape)
    dv = np.zeros(arrs[2].shape)
    keep, bp = _bias_arg(bias, H, max_rel)
    keep_d, dp_, op_ = _dense_arg(dense_bias, qo, ko, H)
    rc = _load().oracle_bwd_mx(*[_p(a, ctypes.c_double) for a in arrs], _p(qo, ctypes.c_int32),
                               _p(ko, ctypes.c_int32), B, H, d, bp, int(max_rel),
                               int(bool(causal)), int(window), float(scale),
                               _p(lse_a, ctypes.c_double),
                               _p(delta_a, ctypes.c_double), int(bool(round_ps)),
                               _p(dq, ctypes.c_double), _p(dk, ctypes.c_double),
                               _p(dv, ctypes.c_double), dp_, op_)
    if rc != 0:
        raise ValueError("oracle_bwd_mx rejected its arguments")
    del keep, keep_d
    return dq, dk, dv


def bwd_mxfp8(q, q_offsets, k, v, kv_offsets, out, dout, lse, *, causal: bool = False,
              scale: float, bias=None, max_rel: int = 0, window: int = 0, dense_bias=None):
    """The MXFP8 softmax backward on bf16 inputs: Q, K, dO quantised along
    channels and along tokens, V along channels (quant_rows / quant_cols,
    decoded), delta = rowsum(dO * O) of the given values, P and dS rounded in
    32 x 32 blocks.  Returns (dq, dk, dv) float64."""
    q, k, v, out, dout = (_f64(a) for a in (q, k, v, out, dout))
    qo, ko = _i32(q_offsets), _i32(kv_offsets)
    delta = np.einsum("thc,thc->ht", dout, out)
    return bwd_mx_operands(dequant_rows(q), dequant_cols(q, qo), dequant_rows(k),
                           dequant_cols(k, ko), dequant_rows(v), dequant_rows(dout),
                           dequant_cols(dout, qo), qo, ko, lse, delta, causal=causal,
                           scale=scale, bias=bias, max_rel=max_rel, window=window, round_ps=True,
                           dense_bias=dense_bias)


# ------------------------------------------------------------------ rotary embedding
def _rope_angles(offsets, d: int, base: float):
    """Angle [T, d/2] of channel pair c at each token: pos * base^(-2c/d), pos the
    token's position within its sample."""
    o = _i32(offsets)
    pos = np.concatenate([np.arange(int(o[b + 1]) - int(o[b]), dtype=np.float64)
                          for b in range(len(o) - 1)] or [np.zeros(0)])
    inv = float(base) ** (-2.0 * np.arange(d // 2, dtype=np.float64) / d)
    return pos[:, None] * inv[None, :]


def rope_fwd(x, offsets, base: float):
    """Rotary position embedding (rotate-half form): channel pairs (c, c + d/2)
    rotated by pos * base^(-2c/d).  x [T,H,d] -> float64 [T,H,d]."""
    x = _f64(x)
    d = x.shape[2]
    a = _rope_angles(offsets, d, base)[:, None, :]
    c, s = np.cos(a), np.sin(a)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def rope_bwd(g, offsets, base: float):
    """Gradient through rope_fwd: the transposed rotation R(pos)^T applied to g."""
    g = _f64(g)
    d = g.shape[2]
    a = _rope_angles(offsets, d, base)[:, None, :]
    c, s = np.cos(a), np.sin(a)
    g1, g2 = g[..., : d // 2], g[..., d // 2:]
    return np.concatenate([g1 * c + g2 * s, -g1 * s + g2 * c], axis=-1)
