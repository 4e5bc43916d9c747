"""GPU parity of block-aligned attention (gdpa_block_fwd, gdpa_block_bwd)
against the fp64 oracle, through the C ABI.

Blocks of 64 tokens start at each sample's first token; a row attends to the
keys of its own block.  The lengths cover full and partial last blocks, odd
block counts (so a kernel tile pairs the last block of one sample with the
first of the next), empty and single-token samples.  Outputs land in
NaN-filled buffers with guard rows.  Tolerances are those of the jagged
paths: abs 1e-2 + rel 1e-2 (bf16 forward), abs 3e-2 + rel 3e-2 (bf16
backward).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_common import (BWD_TOL, FWD_TOL, assert_close, check_guards, ds_pair_bounds, guarded,
                        offsets, rand_bf16, to_np)
from jagged_attention_recsys_02_gb300 import binding
from jagged_attention_recsys_02_gb300.workloads import ACTS, make_tensors, make_workload

pytestmark = pytest.mark.gpu

DEV = "cuda"
BLOCK = 64
LENGTHS = [1, 63, 64, 65, 127, 128, 129, 0, 200, 256, 300, 7, 513]


def _inputs(lengths, H, d, max_rel, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    T = sum(lengths)
    q, k, v, do = (rand_bf16((T, H, d), g, DEV) for _ in range(4))
    o = offsets(lengths)
    bias = torch.randn(H, 2 * max_rel - 1, generator=g, device=DEV) * 0.5 if max_rel else None
    return q, k, v, do, o, torch.from_numpy(o).to(DEV), bias


def _np_bias(bias):
    return None if bias is None else bias.cpu().double().numpy()


def _oracle_fwd(q, k, v, o, act, causal, scale, bias, max_rel):
    out, _ = oracle.fwd(to_np(q), o, to_np(k), to_np(v), o, act=ACTS[act], causal=causal,
                        scale=scale, bias=_np_bias(bias), max_rel=max_rel, block=BLOCK)
    return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("act", ["softmax", "silu", "gelu_tanh", "identity", "gelu_erf"])
@pytest.mark.parametrize("causal", [False, True])
def test_block_fwd_parity(d, act, causal):
    H = 2
    max_rel = 100 if act in ("softmax", "silu") else 0
    q, k, v, _, o, od, bias = _inputs(LENGTHS, H, d, max_rel, seed=d + 3 * causal)
    scale = 1.0 / math.sqrt(d)
    buf, out = guarded(sum(LENGTHS), H, d, DEV)
    binding.gdpa_block_fwd(q, od, k, v, act=act, causal=causal, scale=scale, bias=bias,
                           max_rel=max_rel, out=out)
    assert binding.device_status() == 0
    check_guards(buf)
    ref = _oracle_fwd(q, k, v, o, act, causal, scale, bias, max_rel)
    assert_close(to_np(out), ref, FWD_TOL, f"block fwd {act} d={d} causal={causal}")


def test_block_fwd_single_sample_shapes():
    """One sample of every length around the tile edges (1..130 and a few long
    ones): the tile pairing and the partial last block."""
    H, d = 1, 128
    for L in list(range(1, 131, 7)) + [191, 192, 193, 1000]:
        q, k, v, _, o, od, _ = _inputs([L], H, d, 0, seed=L)
        scale = 1.0 / math.sqrt(d)
        buf, out = guarded(L, H, d, DEV)
        binding.gdpa_block_fwd(q, od, k, v, act="softmax", scale=scale, out=out)
        assert binding.device_status() == 0
        check_guards(buf)
        ref = _oracle_fwd(q, k, v, o, "softmax", False, scale, None, 0)
        assert_close(to_np(out), ref, FWD_TOL, f"block fwd L={L}")


def test_block_bad_offsets_are_reported():
    H, d = 1, 64
    g = torch.Generator(device=DEV).manual_seed(0)
    q = rand_bf16((10, H, d), g, DEV)
    od = torch.tensor([0, 6, 4, 10], dtype=torch.int32, device=DEV)  # not monotone
    out = torch.zeros_like(q)
    binding.gdpa_block_fwd(q, od, q, q, act="softmax", scale=0.1, out=out)
    assert binding.device_status() == 6  # GDPA_ERR_BAD_OFFSETS
    assert torch.all(out == 0)           # nothing was written


def test_block_long_sequence_workload_sampled():
    """The long-sequence block workload at full size, as the benchmark runs it;
    checked against the oracle on a few samples (every block of a sample is
    independent, so a sample's rows depend on that sample alone)."""
    w = make_workload("block_relpos")
    t = make_tensors(w, device=DEV)
    kw = dict(act=w.act, causal=w.causal, scale=w.scale, bias=t["bias"], max_rel=w.max_rel)
    out = binding.gdpa_block_fwd(t["q"], t["qo"], t["k"], t["v"], **kw)
    assert binding.device_status() == 0
    o, _ = w.offsets()
    order = np.argsort(w.lq, kind="stable")
    for b in [int(order[0]), int(order[1]), int(order[-1])]:
        s0, s1 = int(o[b]), int(o[b + 1])
        sl = slice(s0, s1)
        ob = np.array([0, s1 - s0], dtype=np.int32)
        ref, _ = oracle.fwd(to_np(t["q"][sl]), ob, to_np(t["k"][sl]), to_np(t["v"][sl]), ob, act=0,
                            scale=w.scale, bias=t["bias"].cpu().double().numpy(),
                            max_rel=w.max_rel, block=BLOCK)
        assert_close(to_np(out[sl]), ref, FWD_TOL, f"block_relpos sample {b}")


def _run_bwd(q, od, k, v, do, act, causal, scale, bias, max_rel):
    T, H, d = q.shape
    bufs = [guarded(T, H, d, DEV) for _ in range(3)]
    binding.gdpa_block_bwd(q, od, k, v, do, act=act, causal=causal, scale=scale, bias=bias,
                           max_rel=max_rel, dq=bufs[0][1], dk=bufs[1][1], dv=bufs[2][1])
    assert binding.device_status() == 0
    for b, _ in bufs:
        check_guards(b)
    return [x for _, x in bufs]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("act", ["softmax", "silu", "gelu_tanh", "gelu_erf"])
@pytest.mark.parametrize("causal", [False, True])
def test_block_bwd_parity(d, act, causal):
    H = 2
    max_rel = 100 if act in ("softmax", "gelu_tanh") else 0
    q, k, v, do, o, od, bias = _inputs(LENGTHS, H, d, max_rel, seed=11 * d + causal)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = _run_bwd(q, od, k, v, do, act, causal, scale, bias, max_rel)
    rq, rk, rv = oracle.bwd(to_np(q), o, to_np(k), to_np(v), o, to_np(do), act=ACTS[act],
                            causal=causal, scale=scale, bias=_np_bias(bias), max_rel=max_rel,
                            block=BLOCK)
    what = f"block bwd {act} d={d} causal={causal}"
    assert_close(to_np(dq), rq, BWD_TOL, what + " dq")
    assert_close(to_np(dk), rk, BWD_TOL, what + " dk")
    assert_close(to_np(dv), rv, BWD_TOL, what + " dv")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("act", ["softmax", "silu"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("max_rel", [100, 20])
def test_block_bwd_table_gradient(max_rel, causal, act, d):
    """gdpa_block_bwd_dbias: the relative-position table's gradient against the
    oracle's (summed per entry over the in-block pairs; max_rel 20 clamps), dq,
    dk, dv as without it, and the gradient added to what dbias held."""
    H = 2
    q, k, v, do, o, od, bias = _inputs(LENGTHS, H, d, max_rel, seed=40 + d + causal)
    scale = 1.0 / math.sqrt(d)
    base = torch.randn_like(bias)
    dbias = base.clone()
    kw = dict(act=act, causal=causal, scale=scale, bias=bias, max_rel=max_rel)
    dq, dk, dv = binding.gdpa_block_bwd(q, od, k, v, do, dbias=dbias, **kw)
    assert binding.device_status() == 0
    dq0, dk0, dv0 = binding.gdpa_block_bwd(q, od, k, v, do, **kw)
    assert binding.device_status() == 0
    assert torch.equal(dq, dq0) and torch.equal(dk, dk0) and torch.equal(dv, dv0)
    a = ACTS[act]
    tb = _np_bias(bias)
    qn, kn, vn, don = to_np(q), to_np(k), to_np(v), to_np(do)
    *_, ref = oracle.bwd(qn, o, kn, vn, o, don, act=a, causal=causal, scale=scale, bias=tb,
                         max_rel=max_rel, block=BLOCK, want_dbias=True)
    o_ref, _ = oracle.fwd(qn, o, kn, vn, o, act=0, causal=causal, scale=scale, bias=tb,
                          max_rel=max_rel, block=BLOCK)
    width = 2 * max_rel - 1
    tab = lambda i, j: np.clip(i - j + max_rel - 1, 0, width - 1)
    err = np.zeros_like(ref)
    for b, h, live, e in ds_pair_bounds(qn, o, kn, vn, o, don, o_ref, act=a, causal=causal,
                                        scale=scale, block=BLOCK,
                                        bias_of=lambda b, h, i, j: tb[h][tab(i, j)]):
        t = tab(np.arange(live.shape[0])[:, None], np.arange(live.shape[1])[None, :])
        np.add.at(err[h], t[live], e[live])
    got = (dbias - base).cpu().double().numpy()
    # the kernel's dS is fp32 (the per-pair bound covers the bf16 P it is formed
    # from), plus the fp32 rounding of adding to base and a floor of 1e-3 of
    # the largest entry
    bound = (1e-3 * np.abs(ref).max() + 1e-3 * np.abs(ref) + 4 * err +
             2.0 ** -23 * (np.abs(base.cpu().double().numpy()) + np.abs(ref)))
    assert np.all(np.abs(got - ref) <= bound), \
        f"block dbias {act}: worst err/bound {float((np.abs(got - ref) / bound).max()):.3f}"


def test_block_bwd_single_sample_shapes():
    H, d = 1, 128
    for L in [1, 2, 33, 64, 65, 100, 128, 129, 190, 193]:
        q, k, v, do, o, od, _ = _inputs([L], H, d, 0, seed=100 + L)
        scale = 1.0 / math.sqrt(d)
        dq, dk, dv = _run_bwd(q, od, k, v, do, "softmax", False, scale, None, 0)
        rq, rk, rv = oracle.bwd(to_np(q), o, to_np(k), to_np(v), o, to_np(do), act=0,
                                scale=scale, block=BLOCK)
        for got, ref, nm in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
            assert_close(to_np(got), ref, BWD_TOL, f"block bwd L={L} {nm}")


def test_block_bwd_long_sequence_workload_sampled():
    w = make_workload("block_relpos")
    t = make_tensors(w, device=DEV)
    kw = dict(act=w.act, causal=w.causal, scale=w.scale, bias=t["bias"], max_rel=w.max_rel)
    dq, dk, dv = binding.gdpa_block_bwd(t["q"], t["qo"], t["k"], t["v"], t["dout"], **kw)
    assert binding.device_status() == 0
    o, _ = w.offsets()
    order = np.argsort(w.lq, kind="stable")
    for b in [int(order[0]), int(order[1]), int(order[-1])]:
        s0, s1 = int(o[b]), int(o[b + 1])
        sl = slice(s0, s1)
        ob = np.array([0, s1 - s0], dtype=np.int32)
        rq, rk, rv = oracle.bwd(to_np(t["q"][sl]), ob, to_np(t["k"][sl]), to_np(t["v"][sl]), ob,
                                to_np(t["dout"][sl]), act=0, scale=w.scale,
                                bias=t["bias"].cpu().double().numpy(), max_rel=w.max_rel,
                                block=BLOCK)
        for got, ref, nm in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
            assert_close(to_np(got[sl]), ref, BWD_TOL, f"block_relpos sample {b} {nm}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("act", ["softmax", "silu"])
def test_block_bwd_fused_rope(d, act):
    """q and k arrive rotary-embedded; with rope_base the kernel returns dq, dk
    for the un-rotated inputs: the oracle's attention backward on the rotated
    inputs followed by its rotary backward.  dv is unchanged by the rotation."""
    H, base = 2, 10000.0
    q, k, v, do, o, od, _ = _inputs(LENGTHS, H, d, 0, seed=23 + d)
    scale = 1.0 / math.sqrt(d)
    bufs = [guarded(sum(LENGTHS), H, d, DEV) for _ in range(3)]
    binding.gdpa_block_bwd(q, od, k, v, do, act=act, scale=scale, rope_base=base,
                           dq=bufs[0][1], dk=bufs[1][1], dv=bufs[2][1])
    assert binding.device_status() == 0
    for b, _ in bufs:
        check_guards(b)
    rq, rk, rv = oracle.bwd(to_np(q), o, to_np(k), to_np(v), o, to_np(do), act=ACTS[act],
                            scale=scale, block=BLOCK)
    rq, rk = oracle.rope_bwd(rq, o, base), oracle.rope_bwd(rk, o, base)
    what = f"block bwd rope {act} d={d}"
    assert_close(to_np(bufs[0][1]), rq, BWD_TOL, what + " dq")
    assert_close(to_np(bufs[1][1]), rk, BWD_TOL, what + " dk")
    assert_close(to_np(bufs[2][1]), rv, BWD_TOL, what + " dv")


def test_block_bwd_fused_rope_long_positions():
    """Positions up to 16k (large rotation angles): rows [15360, 16000) of one
    16,000-token sample, whose blocks depend on themselves only."""
    H, d, L, a, base = 1, 128, 16000, 15360, 10000.0
    q, k, v, do, o, od, _ = _inputs([L], H, d, 0, seed=99)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = binding.gdpa_block_bwd(q, od, k, v, do, act="softmax", scale=scale,
                                        rope_base=base)
    assert binding.device_status() == 0
    ob = np.array([0, L - a], dtype=np.int32)
    sl = slice(a, L)
    rq, rk, rv = oracle.bwd(to_np(q[sl]), ob, to_np(k[sl]), to_np(v[sl]), ob, to_np(do[sl]), act=0,
                            scale=scale, block=BLOCK)

    def rope_at(g):  # rotary backward at positions a .. L-1
        pad = np.zeros((L, H, d))
        pad[a:] = g
        return oracle.rope_bwd(pad, np.array([0, L], dtype=np.int32), base)[a:]

    assert_close(to_np(dq[sl]), rope_at(rq), BWD_TOL, "rope dq at long positions")
    assert_close(to_np(dk[sl]), rope_at(rk), BWD_TOL, "rope dk at long positions")
    assert_close(to_np(dv[sl]), rv, BWD_TOL, "dv")
