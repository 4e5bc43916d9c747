"""GPU parity of the dense jagged bias (one fp32 value per head, query and key
of each sample) against the oracle: forward for every activation, the softmax
and GDPA backward, the bias's gradient, causal and not, ragged lengths,
malformed bias offsets; with a sliding window, the fused rotary backward and
the block-aligned kernels."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import (BWD_TOL, FWD_TOL, assert_close, check_dense_gradient, check_guards,
                        dense_ref_kw, guarded, offsets, rand_bf16, to_np)
from jagged_attention_recsys_02_gb300 import binding
from jagged_attention_recsys_02_gb300.workloads import ACTS

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _case(lq, lkv, H, d, act, causal, seed, std=1.0, window=0, block=0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    q = rand_bf16((sum(lq), H, d), g, DEV)
    k = rand_bf16((sum(lkv), H, d), g, DEV)
    v = rand_bf16((sum(lkv), H, d), g, DEV)
    do = rand_bf16((sum(lq), H, d), g, DEV)
    qo_np, ko_np = offsets(lq), offsets(lkv)
    off_np = oracle.dense_bias_offsets(qo_np, ko_np, H)
    vals = torch.randn(int(off_np[-1]), generator=g, device=DEV) * std
    qo, ko = torch.from_numpy(qo_np).to(DEV), torch.from_numpy(ko_np).to(DEV)
    off = torch.from_numpy(off_np).to(DEV)
    return dict(q=q, k=k, v=v, do=do, qo=qo, ko=ko, qo_np=qo_np, ko_np=ko_np, vals=vals, off=off,
                act=ACTS[act], causal=causal, scale=1.0 / np.sqrt(d), window=window, block=block)


def _fwd(c):
    Tq, H, d = c["q"].shape
    buf, out = guarded(Tq, H, d, DEV)
    lse = torch.full((H, Tq), float("nan"), device=DEV) if c["act"] == 0 else None
    binding.gdpa_fwd(c["q"], c["qo"], c["k"], c["v"], c["ko"], act=c["act"], causal=c["causal"],
                     scale=c["scale"], bias=(c["vals"], c["off"]), out=out, lse=lse,
                     window=c["window"])
    assert binding.device_status() == 0
    check_guards(buf)
    return out, lse


_ref_kw = dense_ref_kw


CASES = [
    ([1, 31, 64, 65, 200, 0, 300, 129], [7, 32, 1, 96, 128, 5, 191, 300], False),
    ([1, 64, 65, 128, 129, 300, 0, 257], None, True),
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("act", ["softmax", "silu", "gelu_tanh", "gelu_erf"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_dense_bias_forward(case, act, d):
    lq, lkv, causal = CASES[case]
    c = _case(lq, lkv or lq, 2, d, act, causal, seed=10 + case)
    out, lse = _fwd(c)
    ro, rl = oracle.fwd(to_np(c["q"]), c["qo_np"], to_np(c["k"]), to_np(c["v"]), c["ko_np"],
                        **_ref_kw(c))
    assert_close(to_np(out), ro, FWD_TOL, f"dense {act} out")
    if lse is not None:
        assert_close(lse.cpu().double().numpy(), rl, FWD_TOL, f"dense {act} lse")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("act", ["softmax", "silu", "gelu_tanh"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_dense_bias_backward(case, act, d):
    lq, lkv, causal = CASES[case]
    c = _case(lq, lkv or lq, 2, d, act, causal, seed=20 + case)
    out, lse = _fwd(c)
    Tq, H, _ = c["q"].shape
    Tkv = c["k"].shape[0]
    bq, dq = guarded(Tq, H, d, DEV)
    bk, dk = guarded(Tkv, H, d, DEV)
    bv, dv = guarded(Tkv, H, d, DEV)
    binding.gdpa_bwd(c["q"], c["qo"], c["k"], c["v"], c["ko"], out, lse, c["do"], act=c["act"],
                     causal=c["causal"], scale=c["scale"], bias=(c["vals"], c["off"]), dq=dq, dk=dk,
                     dv=dv)
    assert binding.device_status() == 0
    for b_ in (bq, bk, bv):
        check_guards(b_)
    ref = oracle.bwd(to_np(c["q"]), c["qo_np"], to_np(c["k"]), to_np(c["v"]), c["ko_np"],
                     to_np(c["do"]), **_ref_kw(c))
    for name, got, r in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        assert_close(to_np(got), r, BWD_TOL, f"dense {act} {name}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("act", ["softmax", "silu", "gelu_tanh"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_dense_bias_gradient(case, act, d):
    """The dense bias's gradient (dbias with a dense bias): each unmasked
    pair's entry gets its dS added, the other entries are left as they are;
    dq, dk, dv are those of the call without it."""
    lq, lkv, causal = CASES[case]
    c = _case(lq, lkv or lq, 2, d, act, causal, seed=30 + case)
    out, lse = _fwd(c)
    Tq, H, _ = c["q"].shape
    g = torch.Generator(device=DEV).manual_seed(7)
    base = torch.randn(c["vals"].numel(), generator=g, device=DEV)
    dbias = base.clone()
    kw = dict(act=c["act"], causal=c["causal"], scale=c["scale"], bias=(c["vals"], c["off"]),
              window=c["window"])
    dq, dk, dv = binding.gdpa_bwd(c["q"], c["qo"], c["k"], c["v"], c["ko"], out, lse, c["do"],
                                  dbias=dbias, **kw)
    assert binding.device_status() == 0
    check_dense_gradient(c, dbias, base, f"dense {act} d={d} dbias")
    dq0, dk0, dv0 = binding.gdpa_bwd(c["q"], c["qo"], c["k"], c["v"], c["ko"], out, lse, c["do"],
                                     **kw)
    assert binding.device_status() == 0
    assert torch.equal(dk, dk0) and torch.equal(dv, dv0)
    torch.testing.assert_close(dq, dq0, rtol=2 ** -7, atol=1e-3)  # (dQ reduce order)


@pytest.mark.parametrize("act", ["softmax", "silu"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_dense_bias_with_fused_rope(case, act):
    """gdpa_bwd_rope with a dense bias and its gradient: dq, dk through the
    rotary backward (queries and keys at their own positions), dv and the
    bias's gradient as without it."""
    lq, lkv, causal = CASES[case]
    d, base = 128, 10000.0
    c = _case(lq, lkv or lq, 2, d, act, causal, seed=40 + case)
    out, lse = _fwd(c)
    g = torch.Generator(device=DEV).manual_seed(8)
    bias0 = torch.randn(c["vals"].numel(), generator=g, device=DEV)
    dbias = bias0.clone()
    dq, dk, dv = binding.gdpa_bwd(c["q"], c["qo"], c["k"], c["v"], c["ko"], out, lse, c["do"],
                                  act=c["act"], causal=c["causal"], scale=c["scale"],
                                  bias=(c["vals"], c["off"]), dbias=dbias, rope_base=base)
    assert binding.device_status() == 0
    ref = oracle.bwd(to_np(c["q"]), c["qo_np"], to_np(c["k"]), to_np(c["v"]), c["ko_np"],
                     to_np(c["do"]), **_ref_kw(c))
    what = f"dense+rope {act}"
    assert_close(to_np(dq), oracle.rope_bwd(ref[0], c["qo_np"], base), BWD_TOL, what + " dq")
    assert_close(to_np(dk), oracle.rope_bwd(ref[1], c["ko_np"], base), BWD_TOL, what + " dk")
    assert_close(to_np(dv), ref[2], BWD_TOL, what + " dv")
    check_dense_gradient(c, dbias, bias0, what + " dbias")


@pytest.mark.parametrize("act", ["softmax", "silu"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_bias_with_window(causal, d, act):
    """A dense bias under a sliding window (self-attention): forward, backward
    and the bias's gradient against the oracle; entries outside the band keep
    their value.  The window crosses the 128-key tiles."""
    L = [1, 64, 130, 300, 0, 257, 129]
    c = _case(L, L, 2, d, act, causal, seed=50 + d, window=100)
    out, lse = _fwd(c)
    ro, rl = oracle.fwd(to_np(c["q"]), c["qo_np"], to_np(c["k"]), to_np(c["v"]), c["ko_np"],
                        **_ref_kw(c))
    what = f"dense+window {act} d={d} causal={causal}"
    assert_close(to_np(out), ro, FWD_TOL, what + " out")
    if lse is not None:
        assert_close(lse.cpu().double().numpy(), rl, FWD_TOL, what + " lse")
    g = torch.Generator(device=DEV).manual_seed(9)
    base = torch.randn(c["vals"].numel(), generator=g, device=DEV)
    dbias = base.clone()
    dq, dk, dv = binding.gdpa_bwd(c["q"], c["qo"], c["k"], c["v"], c["ko"], out, lse, c["do"],
                                  act=c["act"], causal=c["causal"], scale=c["scale"],
                                  bias=(c["vals"], c["off"]), window=c["window"], dbias=dbias)
    assert binding.device_status() == 0
    ref = oracle.bwd(to_np(c["q"]), c["qo_np"], to_np(c["k"]), to_np(c["v"]), c["ko_np"],
                     to_np(c["do"]), **_ref_kw(c))
    for name, got, r in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        assert_close(to_np(got), r, BWD_TOL, f"{what} {name}")
    check_dense_gradient(c, dbias, base, what + " dbias")


def test_dense_bias_bad_offsets_are_reported():
    """Offsets that do not step by H * Lq * Lkv are reported through the device
    status word, and nothing is computed."""
    c = _case([5, 40], [9, 3], 2, 64, "softmax", False, seed=3)
    bad = c["off"].clone()
    bad[1] += 1
    out = torch.zeros_like(c["q"])
    lse = torch.zeros((2, c["q"].shape[0]), device=DEV)
    binding.gdpa_fwd(c["q"], c["qo"], c["k"], c["v"], c["ko"], act=0, scale=c["scale"],
                     bias=(c["vals"], bad), out=out, lse=lse)
    assert binding.device_status() == 6   # GDPA_ERR_BAD_OFFSETS


BLOCK = 64
BLOCK_LENS = [1, 64, 65, 128, 129, 300, 0, 257, 200]  # blocks and tiles across samples


def _block_fwd(c):
    T, H, d = c["q"].shape
    buf, out = guarded(T, H, d, DEV)
    binding.gdpa_block_fwd(c["q"], c["qo"], c["k"], c["v"], act=c["act"], causal=c["causal"],
                           scale=c["scale"], bias=(c["vals"], c["off"]), out=out)
    assert binding.device_status() == 0
    check_guards(buf)
    return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("act", ["softmax", "silu", "gelu_tanh", "gelu_erf", "identity"])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_bias_block_forward(causal, act, d):
    """The block-aligned forward with a dense bias: only the pairs inside a
    64-token block are read; against the oracle with the same blocks."""
    c = _case(BLOCK_LENS, BLOCK_LENS, 2, d, act, causal, seed=60 + d, block=BLOCK)
    out = _block_fwd(c)
    ro, _ = oracle.fwd(to_np(c["q"]), c["qo_np"], to_np(c["k"]), to_np(c["v"]), c["ko_np"],
                       **_ref_kw(c))
    assert_close(to_np(out), ro, FWD_TOL, f"dense+block {act} d={d} causal={causal} out")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("act", ["softmax", "silu", "gelu_tanh"])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_bias_block_backward_and_gradient(causal, act, d):
    """The block-aligned backward with a dense bias: dq, dk, dv against the
    oracle; with dbias the entry of every pair inside a block gets its dS
    added (the other entries are left as they are) and dq, dk, dv are those
    of the call without it, bit for bit (each tile writes its rows once)."""
    c = _case(BLOCK_LENS, BLOCK_LENS, 2, d, act, causal, seed=70 + d, block=BLOCK)
    T, H, _ = c["q"].shape
    kw = dict(act=c["act"], causal=c["causal"], scale=c["scale"], bias=(c["vals"], c["off"]))
    bufs = [guarded(T, H, d, DEV) for _ in range(3)]
    binding.gdpa_block_bwd(c["q"], c["qo"], c["k"], c["v"], c["do"], dq=bufs[0][1],
                           dk=bufs[1][1], dv=bufs[2][1], **kw)
    assert binding.device_status() == 0
    for b_, _ in bufs:
        check_guards(b_)
    ref = oracle.bwd(to_np(c["q"]), c["qo_np"], to_np(c["k"]), to_np(c["v"]), c["ko_np"],
                     to_np(c["do"]), **_ref_kw(c))
    what = f"dense+block {act} d={d} causal={causal}"
    for name, (_, got), r in zip(("dq", "dk", "dv"), bufs, ref):
        assert_close(to_np(got), r, BWD_TOL, f"{what} {name}")
    g = torch.Generator(device=DEV).manual_seed(9)
    base = torch.randn(c["vals"].numel(), generator=g, device=DEV)
    dbias = base.clone()
    dq, dk, dv = binding.gdpa_block_bwd(c["q"], c["qo"], c["k"], c["v"], c["do"], dbias=dbias, **kw)
    assert binding.device_status() == 0
    for got, (_, want) in zip((dq, dk, dv), bufs):
        assert torch.equal(got, want), f"{what}: the gradient call changed dq / dk / dv"
    check_dense_gradient(c, dbias, base, what + " dbias")


def test_dense_bias_block_bad_offsets_are_reported():
    """A dense bias whose per-sample sizes are not H * L_b^2 is refused on the
    device by the block kernels too: GDPA_ERR_BAD_OFFSETS, nothing written."""
    c = _case(BLOCK_LENS, BLOCK_LENS, 2, 64, "softmax", False, seed=80, block=BLOCK)
    bad = c["off"].clone()
    bad[3] += 1  # samples 2 and 3 no longer hold H * L^2 values
    out = torch.zeros_like(c["q"])
    binding.gdpa_block_fwd(c["q"], c["qo"], c["k"], c["v"], act=c["act"], scale=c["scale"],
                           bias=(c["vals"], bad), out=out)
    assert binding.device_status() == 6   # GDPA_ERR_BAD_OFFSETS
    assert torch.all(out == 0)
