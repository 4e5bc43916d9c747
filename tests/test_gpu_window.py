"""GPU parity of sliding-window attention (gdpa_fwd_window, gdpa_bwd_window,
gdpa_fwd_mxfp8_window) against the fp64 oracle, through the C ABI.

A window W keeps the pairs with |i - j| < W (and j <= i when causal); the
kernels skip every key / query tile outside that band.  Lengths and windows
are chosen so that bands start and end inside tiles, a 256-row forward item's
two halves begin on different key tiles, and samples are shorter and longer
than the window.  Tolerances are those of the unwindowed paths: abs 1e-2 +
rel 1e-2 (bf16 forward), abs 3e-2 + rel 3e-2 (bf16 backward), abs 6e-2 + rel
6e-2 (MXFP8 forward, against the oracle on the MXFP8-decoded operands).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_common import (BWD_TOL, FWD_TOL, MXFP8_TOL, assert_close, check_guards, guarded,
                        offsets, oracle_fwd_samples, rand_bf16, run_fwd, to_np)
from jagged_attention_recsys_02_gb300 import binding
from jagged_attention_recsys_02_gb300.workloads import ACTS, make_tensors, make_workload

pytestmark = pytest.mark.gpu

DEV = "cuda"
LENGTHS = [1, 63, 128, 129, 255, 256, 257, 300, 0, 513, 700, 1000]


def _inputs(lengths, H, d, max_rel, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    T = sum(lengths)
    q, k, v, do = (rand_bf16((T, H, d), g, DEV) for _ in range(4))
    o = offsets(lengths)
    bias = torch.randn(H, 2 * max_rel - 1, generator=g, device=DEV) * 0.5 if max_rel else None
    return q, k, v, do, o, torch.from_numpy(o).to(DEV), bias


def _np_bias(bias):
    return None if bias is None else bias.cpu().double().numpy()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("act", ["softmax", "silu", "gelu_tanh", "gelu_erf"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("window", [1, 77, 128, 200, 384])
def test_window_fwd_parity(d, act, causal, window):
    H, max_rel = 2, (300 if act == "softmax" else 0)
    q, k, v, _, o, od, bias = _inputs(LENGTHS, H, d, max_rel, seed=window + d)
    scale = 1.0 / math.sqrt(d)
    out, lse = run_fwd(q, od, k, v, od, act, causal, scale, bias, max_rel, window=window)
    ref = oracle_fwd_samples(to_np(q), to_np(k), to_np(v), o, o, range(len(LENGTHS)), act, causal,
                             scale, _np_bias(bias), max_rel, window=window)
    got = to_np(out)
    for rows, ro, rl in ref:
        assert_close(got[rows], ro, FWD_TOL, f"{act} W={window} out")
        if act == "softmax":
            assert_close(to_np(lse)[:, rows], rl, FWD_TOL, f"{act} W={window} lse")


def _run_bwd(q, k, v, do, od, act, causal, scale, bias, max_rel, window):
    a = ACTS[act]
    out, lse = binding.gdpa_fwd(q, od, k, v, od, act=a, causal=causal, scale=scale, bias=bias,
                                max_rel=max_rel, window=window)
    T, H, d = q.shape
    bufs = [guarded(T, H, d, DEV) for _ in range(3)]
    binding.gdpa_bwd(q, od, k, v, od, out, lse, do, act=a, causal=causal, scale=scale, bias=bias,
                     max_rel=max_rel, window=window, dq=bufs[0][1], dk=bufs[1][1], dv=bufs[2][1])
    assert binding.device_status() == 0
    for b, _ in bufs:
        check_guards(b)
    return [x for _, x in bufs]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("act", ["softmax", "silu"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("window", [1, 100, 128, 300])
def test_window_bwd_parity(d, act, causal, window):
    H, max_rel = 2, (200 if act == "softmax" else 0)
    q, k, v, do, o, od, bias = _inputs(LENGTHS, H, d, max_rel, seed=7 * window + d)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = _run_bwd(q, k, v, do, od, act, causal, scale, bias, max_rel, window)
    tb = _np_bias(bias)
    for b in range(len(LENGTHS)):
        s0, s1 = int(o[b]), int(o[b + 1])
        if s1 == s0:
            continue
        ob = np.array([0, s1 - s0], dtype=np.int32)
        rq, rk, rv = oracle.bwd(to_np(q[s0:s1]), ob, to_np(k[s0:s1]), to_np(v[s0:s1]), ob,
                                to_np(do[s0:s1]), act=ACTS[act], causal=causal, scale=scale,
                                bias=tb, max_rel=max_rel, window=window)
        what = f"{act} d={d} W={window} causal={causal} sample {b}"
        assert_close(to_np(dq[s0:s1]), rq, BWD_TOL, what + " dq")
        assert_close(to_np(dk[s0:s1]), rk, BWD_TOL, what + " dk")
        assert_close(to_np(dv[s0:s1]), rv, BWD_TOL, what + " dv")


@pytest.mark.parametrize("act", ["softmax", "silu"])
@pytest.mark.parametrize("causal", [True, False])
def test_window_as_long_as_the_samples_is_bit_identical(act, causal):
    """A window no shorter than every sample masks nothing: the kernels must
    visit the same tiles with the same masks and give bit-identical out, lse,
    dK and dV (rows of samples that the unwindowed call sends to the
    short-query kernels, or to the short-key forward, agree within the parity
    tolerances).  dQ sums the key blocks' contributions in whatever order the
    CTAs reach the fp32 accumulator, so two runs agree only up to that order:
    within a bf16 rounding step of the value plus fp32 rounding of partial
    sums that cancel (bounded here by 1e-4 of the tensor's largest entry)."""
    H, d = 2, 128
    q, k, v, do, o, od, bias = _inputs(LENGTHS, H, d, 0, seed=3)
    a, scale = ACTS[act], 1.0 / math.sqrt(d)
    wide = max(LENGTHS)
    res = []
    for window in (0, wide):
        out, lse = binding.gdpa_fwd(q, od, k, v, od, act=a, causal=causal, scale=scale,
                                    window=window)
        grads = binding.gdpa_bwd(q, od, k, v, od, out, lse, do, act=a, causal=causal, scale=scale,
                                 window=window)
        assert binding.device_status() == 0
        res.append(dict(out=out, lse=lse, dq=grads[0], dk=grads[1], dv=grads[2]))
    # Without a window, samples of at most 32 queries take the short-query
    # kernels (keys as TMEM lanes), and in the GDPA forward samples with more
    # queries and at most 256 keys the short-key kernel; their sums run in
    # another order, so those rows agree within the parity tolerances, every
    # other row bit for bit.
    o_np = offsets(LENGTHS)
    short = torch.zeros(sum(LENGTHS), dtype=torch.bool, device=DEV)
    short_fwd = torch.zeros_like(short)
    if not causal:
        for b, L in enumerate(LENGTHS):
            rows = slice(int(o_np[b]), int(o_np[b + 1]))
            if 1 <= L <= 32:
                short[rows] = True
                short_fwd[rows] = True
            elif act != "softmax" and 32 < L <= 256:
                short_fwd[rows] = True
    for name in ("out", "lse", "dk", "dv"):
        x, y = res[0][name], res[1][name]
        if x is None:
            continue
        sel = short_fwd if name in ("out", "lse") else short
        rows = sel if name != "lse" else sel[None, :].expand_as(x)
        tol = FWD_TOL if name in ("out", "lse") else BWD_TOL
        assert_close(to_np(x[rows]), to_np(y[rows]), tol, name + " (short-query / short-key samples)")
        x, y = x[~rows], y[~rows]
        if x.dtype == torch.bfloat16:
            x, y = x.view(torch.int16), y.view(torch.int16)
        assert torch.equal(x, y), name
    x, y = res[0]["dq"].float(), res[1]["dq"].float()
    tol = 2.0 ** -7 * torch.maximum(x.abs(), y.abs()) + 1e-4 * x.abs().max()
    tol[short] += BWD_TOL[0] + BWD_TOL[1] * x.abs()[short]
    assert torch.all((x - y).abs() <= tol), "dq"


def test_window_needs_equal_lengths():
    H, d = 1, 64
    g = torch.Generator(device=DEV).manual_seed(0)
    q = rand_bf16((10, H, d), g, DEV)
    k = rand_bf16((12, H, d), g, DEV)
    qo = torch.tensor([0, 4, 10], dtype=torch.int32, device=DEV)
    ko = torch.tensor([0, 6, 12], dtype=torch.int32, device=DEV)
    binding.gdpa_fwd(q, qo, k, k, ko, act="silu", scale=0.1, window=3)
    assert binding.device_status() == 6  # GDPA_ERR_BAD_OFFSETS
    with pytest.raises(binding.GdpaError):
        binding.gdpa_fwd(q, qo, q, q, qo, act="silu", scale=0.1, window=-1)


def _dequant(x, offs=None):
    if offs is None:
        codes, scales = oracle.quant_rows(x)
        dec = _DEC[codes]
        return dec * np.exp2(scales.astype(np.float64) - 127).repeat(32, axis=2)
    codes, scales = oracle.quant_cols(x, offs)
    dec = _DEC[codes]
    out = np.zeros_like(dec)
    r = 0
    for b in range(len(offs) - 1):
        for blk in range((int(offs[b + 1]) - int(offs[b]) + 31) // 32):
            t0 = int(offs[b]) + 32 * blk
            t1 = min(t0 + 32, int(offs[b + 1]))
            out[t0:t1] = dec[t0:t1] * np.exp2(scales[r].astype(np.float64) - 127)[None]
            r += 1
    return out


_DEC = np.array([oracle.e4m3_decode(c) for c in range(256)])


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("window", [50, 96, 250])
def test_window_mxfp8_fwd_parity(causal, window):
    H, d, max_rel = 2, 128, 256
    q, k, v, _, o, od, bias = _inputs(LENGTHS, H, d, max_rel, seed=window)
    scale = 1.0 / math.sqrt(d)
    qc, qs = binding.quantize_mxfp8(q, mode=binding.MX_ALONG_CHANNELS)
    kc, ks = binding.quantize_mxfp8(k, mode=binding.MX_ALONG_CHANNELS)
    vc, vs = binding.quantize_mxfp8(v, od, mode=binding.MX_ALONG_TOKENS)
    buf, out = guarded(sum(LENGTHS), H, d, DEV)
    lse = torch.full((H, sum(LENGTHS)), float("nan"), device=DEV)
    binding.gdpa_fwd_mxfp8(qc, qs, od, kc, ks, vc, vs, od, causal=causal, scale=scale, bias=bias,
                           max_rel=max_rel, window=window, out=out, lse=lse)
    assert binding.device_status() == 0
    check_guards(buf)
    ref = oracle_fwd_samples(_dequant(to_np(q)), _dequant(to_np(k)), _dequant(to_np(v), o), o, o,
                             range(len(LENGTHS)), "softmax", causal, scale, _np_bias(bias),
                             max_rel, window=window)
    got, gl = to_np(out), to_np(lse)
    for rows, ro, rl in ref:
        assert_close(got[rows], ro, MXFP8_TOL, f"mxfp8 W={window} out")
        assert_close(gl[:, rows], rl, MXFP8_TOL, f"mxfp8 W={window} lse")


def test_window_long_sequence_workload_sampled():
    """The long-sequence sliding-window workload at full size, in the launch
    configuration the benchmark times: forward and backward over every sample,
    checked on the two shortest samples whole and on row ranges of the longest.
    A causal window of W makes rows [r0, r1) of out / lse / dq / dk / dv depend
    only on rows [r0 - W + 1, r1 + W - 1) of the sample (the relative-position
    bias depends on i - j alone), so the oracle runs on that slice."""
    w = make_workload("swa_causal_relpos")
    t = make_tensors(w, device=DEV)
    kw = dict(act=ACTS[w.act], causal=w.causal, scale=w.scale, bias=t["bias"], max_rel=w.max_rel,
              window=w.window)
    out, lse = binding.gdpa_fwd(t["q"], t["qo"], t["k"], t["v"], t["ko"], **kw)
    dq, dk, dv = binding.gdpa_bwd(t["q"], t["qo"], t["k"], t["v"], t["ko"], out, lse, t["dout"],
                                  **kw)
    assert binding.device_status() == 0
    o, _ = w.offsets()
    tb = t["bias"].cpu().double().numpy()
    W = w.window
    order = np.argsort(w.lq, kind="stable")
    longest = int(order[-1])
    L = int(w.lq[longest])
    checks = [(int(b), 0, int(w.lq[b])) for b in order[:2]]
    checks += [(longest, L // 2 + 37, L // 2 + 337), (longest, L - 200, L)]
    for b, r0, r1 in checks:
        a, e = max(0, r0 - W + 1), min(int(w.lq[b]), r1 + W - 1)
        g0 = int(o[b])
        sl = slice(g0 + a, g0 + e)
        n = e - a
        ob = np.array([0, n], dtype=np.int32)
        args = (to_np(t["q"][sl]), ob, to_np(t["k"][sl]), to_np(t["v"][sl]), ob)
        okw = dict(act=0, causal=True, scale=w.scale, bias=tb, max_rel=w.max_rel, window=W)
        ro, rl = oracle.fwd(*args, **okw)
        rq, rk, rv = oracle.bwd(*args, to_np(t["dout"][sl]), **okw)
        keep = slice(r0 - a, r1 - a)
        rows = slice(g0 + r0, g0 + r1)
        what = f"swa sample {b} rows [{r0},{r1})"
        assert_close(to_np(out[rows]), ro[keep], FWD_TOL, what + " out")
        assert_close(to_np(lse[:, rows]), rl[:, keep], FWD_TOL, what + " lse")
        assert_close(to_np(dq[rows]), rq[keep], BWD_TOL, what + " dq")
        assert_close(to_np(dk[rows]), rk[keep], BWD_TOL, what + " dk")
        assert_close(to_np(dv[rows]), rv[keep], BWD_TOL, what + " dv")
