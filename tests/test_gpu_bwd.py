"""GPU parity of the backward pass against the fp64 oracle (through the C ABI).

Tolerance: |gpu - oracle| <= 3e-2 + 3e-2 |oracle| elementwise (bf16 backward)
for dQ, dK and dV.  Gradients are written into NaN-filled buffers with guard
rows on both sides.  The forward outputs fed to the backward (out, lse) come
from the library's own forward.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_common import (BWD_TOL, assert_close, check_guards, check_table_gradient, guarded,
                        offsets, pick_samples, rand_bf16, to_np)
from jagged_attention_recsys_02_gb300 import binding
from jagged_attention_recsys_02_gb300.workloads import ACTS, make_tensors, make_workload

pytestmark = pytest.mark.gpu

DEV = "cuda"


def run_bwd(q, qo, k, v, ko, do, act, causal, scale, bias=None, max_rel=0, guard=3):
    a = ACTS[act] if isinstance(act, str) else act
    out, lse = binding.gdpa_fwd(q, qo, k, v, ko, act=a, causal=causal, scale=scale, bias=bias,
                                max_rel=max_rel)
    Tq, H, d = q.shape
    Tkv = k.shape[0]
    bq, dq = guarded(Tq, H, d, q.device, guard)
    bk, dk = guarded(Tkv, H, d, q.device, guard)
    bv, dv = guarded(Tkv, H, d, q.device, guard)
    binding.gdpa_bwd(q, qo, k, v, ko, out, lse, do, act=a, causal=causal, scale=scale, bias=bias,
                     max_rel=max_rel, dq=dq, dk=dk, dv=dv)
    st = binding.device_status()
    assert st == 0, f"device status {st}"
    for b in (bq, bk, bv):
        check_guards(b, guard)
    return dq, dk, dv


def _check_samples(q, k, v, do, qo, ko, samples, act, causal, scale, bias, max_rel, dq, dk, dv,
                   what):
    a = ACTS[act]
    tb = None if bias is None else bias.cpu().double().numpy()
    for b in samples:
        q0, q1, k0, k1 = int(qo[b]), int(qo[b + 1]), int(ko[b]), int(ko[b + 1])
        rq, rk, rv = oracle.bwd(to_np(q[q0:q1]), np.array([0, q1 - q0]), to_np(k[k0:k1]),
                                to_np(v[k0:k1]), np.array([0, k1 - k0]), to_np(do[q0:q1]), act=a,
                                causal=causal, scale=scale, bias=tb, max_rel=max_rel)
        if q1 > q0:
            assert_close(to_np(dq[q0:q1]), rq, BWD_TOL, f"{what} dq sample {b}")
        if k1 > k0:
            assert_close(to_np(dk[k0:k1]), rk, BWD_TOL, f"{what} dk sample {b}")
            assert_close(to_np(dv[k0:k1]), rv, BWD_TOL, f"{what} dv sample {b}")


def _case(lq, lkv, H, d, act, causal=False, max_rel=0, seed=0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    q = rand_bf16((sum(lq), H, d), g, DEV)
    k = rand_bf16((sum(lkv), H, d), g, DEV)
    v = rand_bf16((sum(lkv), H, d), g, DEV)
    do = rand_bf16((sum(lq), H, d), g, DEV)
    qo_np, ko_np = offsets(lq), offsets(lkv)
    qo = torch.from_numpy(qo_np).to(DEV)
    ko = torch.from_numpy(ko_np).to(DEV)
    bias = torch.randn(H, 2 * max_rel - 1, generator=g, device=DEV) * 0.5 if max_rel else None
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = run_bwd(q, qo, k, v, ko, do, act, causal, scale, bias, max_rel)
    _check_samples(q, k, v, do, qo_np, ko_np, range(len(lq)), act, causal, scale, bias, max_rel,
                   dq, dk, dv, f"{act} d={d}")
    return dq, dk, dv


RAGGED_Q = [1, 63, 64, 65, 127, 128, 129, 0, 300, 513, 7]
RAGGED_KV = [5, 128, 0, 129, 200, 256, 384, 3, 1, 513, 700]


@pytest.mark.parametrize("act", ["softmax", "silu", "gelu_tanh", "identity", "gelu_erf"])
@pytest.mark.parametrize("d", [64, 128])
def test_bwd_ragged(act, d):
    _case(RAGGED_Q, RAGGED_KV, 2, d, act)


@pytest.mark.parametrize("act", ["softmax", "silu"])
@pytest.mark.parametrize("d", [64, 128])
def test_bwd_causal_relpos(act, d):
    L = [1, 64, 65, 128, 129, 300, 0, 511, 200]
    _case(L, L, 2, d, act, causal=True, max_rel=150)


@pytest.mark.parametrize("act", ["softmax", "silu"])
def test_bwd_causal_no_bias(act):
    L = [1, 64, 65, 128, 129, 300, 0, 511, 1000]
    _case(L, L, 2, 128, act, causal=True)


@pytest.mark.parametrize("act", ["softmax", "gelu_tanh"])
def test_bwd_bias_noncausal(act):
    _case([5, 300, 129], [260, 7, 500], 3, 128, act, max_rel=64)


# At most 32 queries: the short-query backward (keys as TMEM lanes, dQ kept in
# TMEM across the sample's keys and stored once).  All-short batches write dq
# directly in bf16; with a longer sample in the call, the short samples' dQ
# rows pass through the fp32 accumulator and its conversion like the others.
SHORTQ_Q = [32, 1, 31, 17, 32, 2, 5, 32]
SHORTQ_KV = [700, 1, 128, 0, 129, 256, 513, 64]


@pytest.mark.parametrize("act", ["softmax", "silu", "gelu_tanh", "identity", "gelu_erf"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mixed", [False, True])
def test_bwd_short_queries(act, d, mixed):
    lq = SHORTQ_Q + ([300] if mixed else [])
    lkv = SHORTQ_KV + ([200] if mixed else [])
    dq, dk, dv = _case(lq, lkv, 3, d, act)
    z = sum(SHORTQ_Q[:3])
    assert torch.all(dq[z:z + SHORTQ_Q[3]] == 0)  # the sample with no key


# GDPA samples whose keys fit one 128-key block get dQ written once in bf16 by
# the main kernel (their accumulator rows are neither zeroed nor converted);
# the others go through the fp32 accumulator.  One call mixes both with
# short-query samples (their own kernel), samples without keys (zero dQ rows)
# and without queries; query counts cross the 64-row tiles and the 16-row
# store pieces, key counts the 128-key block.
DIRECT_Q = [300, 65, 7, 129, 400, 33, 0, 250, 64, 1000, 20]
DIRECT_KV = [128, 1, 90, 129, 0, 64, 50, 256, 127, 700, 40]


@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_direct_dq_rows(causal, d, act):
    lq = DIRECT_Q
    lkv = [x for x in lq] if causal else DIRECT_KV
    dq, dk, dv = _case(lq, lkv, 3, d, act, causal=causal, seed=5)
    if not causal:
        z = sum(DIRECT_Q[:4])
        assert torch.all(dq[z:z + DIRECT_Q[4]] == 0)  # the sample with no key


@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
@pytest.mark.parametrize("d", [64, 128])
def test_bwd_direct_dq_ignores_a_stale_workspace(d, act):
    """With the workspace filled with NaN bit patterns the gradients still match
    the oracle: the direct dQ rows never read the accumulator, and the rows of
    the samples that reduce into it (more than 128 keys) are zeroed by the
    helper first."""
    lq, lkv = DIRECT_Q, DIRECT_KV
    H = 3
    g = torch.Generator(device=DEV).manual_seed(9)
    q = rand_bf16((sum(lq), H, d), g, DEV)
    k = rand_bf16((sum(lkv), H, d), g, DEV)
    v = rand_bf16((sum(lkv), H, d), g, DEV)
    do = rand_bf16((sum(lq), H, d), g, DEV)
    qo_np, ko_np = offsets(lq), offsets(lkv)
    qo, ko = torch.from_numpy(qo_np).to(DEV), torch.from_numpy(ko_np).to(DEV)
    scale = 1.0 / math.sqrt(d)
    a = ACTS[act]
    out, lse = binding.gdpa_fwd(q, qo, k, v, ko, act=a, scale=scale)
    B = len(lq)
    ws = torch.full((binding.bwd_workspace_size(B, H, d, sum(lq), sum(lkv)),), 0xFF,
                    dtype=torch.uint8, device=DEV)
    dq, dk, dv = binding.gdpa_bwd(q, qo, k, v, ko, out, lse, do, act=a, scale=scale, workspace=ws)
    assert binding.device_status() == 0
    _check_samples(q, k, v, do, qo_np, ko_np, range(B), act, False, scale, None, 0, dq, dk, dv,
                   f"stale workspace {act} d={d}")


def test_bwd_empty_sides():
    # no keys: dq rows are zero; no queries: dk/dv rows are zero
    dq, dk, dv = _case([3, 0, 130, 5], [0, 9, 0, 140], 2, 128, "softmax")
    assert torch.all(dq[:3] == 0) and torch.all(dq[3:133] == 0)
    assert torch.all(dk[:9] == 0) and torch.all(dv[:9] == 0)


def test_bwd_tiny_config():
    w = make_workload("tiny_silu")
    t = make_tensors(w, device=DEV)
    dq, dk, dv = run_bwd(t["q"], t["qo"], t["k"], t["v"], t["ko"], t["dout"], w.act, w.causal,
                         w.scale)
    qo, ko = w.offsets()
    _check_samples(t["q"], t["k"], t["v"], t["dout"], qo, ko, range(w.B), w.act, w.causal,
                   w.scale, None, 0, dq, dk, dv, "tiny")


def _key_rows(L):
    """Key rows of a long sample on both sides of 64- and 128-row tile edges."""
    rows = {0, 1, 63, 64, 127, 128, 129, 255, 256, L // 2, L // 2 + 1, L - 129, L - 128, L - 2,
            L - 1}
    return np.array(sorted(r for r in rows if 0 <= r < L))


def _check_key_rows(t, w, b, dk, dv, what):
    """dK and dV of a subset of key rows of sample b (non-causal, no bias) against
    the oracle.  GDPA: a key's gradients depend on that key and every query only,
    so the oracle backward on (all queries, the chosen keys) is exact for them.
    Softmax: the oracle forward of the whole sample gives lse and D = rowsum(dO O);
    the backward of the chosen keys is then the oracle's operand-form backward
    on unquantised operands without rounding (the plain softmax backward)."""
    qo, ko = w.offsets()
    q0, q1, k0, k1 = int(qo[b]), int(qo[b + 1]), int(ko[b]), int(ko[b + 1])
    keys = _key_rows(k1 - k0)
    sel = torch.from_numpy(k0 + keys).to(DEV)
    qn, don = to_np(t["q"][q0:q1]), to_np(t["dout"][q0:q1])
    kn, vn = to_np(t["k"][sel]), to_np(t["v"][sel])
    oq, ok = np.array([0, q1 - q0]), np.array([0, len(keys)])
    if w.act == "softmax":
        o_full, lse = oracle.fwd(qn, oq, to_np(t["k"][k0:k1]), to_np(t["v"][k0:k1]),
                                 np.array([0, k1 - k0]), act=oracle.ACT_SOFTMAX, scale=w.scale)
        delta = np.einsum("thc,thc->ht", don, o_full)
        _, rk, rv = oracle.bwd_mx_operands(qn, qn, kn, kn, vn, don, don, oq, ok, lse, delta,
                                           scale=w.scale, round_ps=False)
    else:
        _, rk, rv = oracle.bwd(qn, oq, kn, vn, ok, don, act=ACTS[w.act], scale=w.scale)
    assert_close(to_np(dk[sel]), rk, BWD_TOL, f"{what} dk key rows of sample {b} (L={k1 - k0})")
    assert_close(to_np(dv[sel]), rv, BWD_TOL, f"{what} dv key rows of sample {b} (L={k1 - k0})")


def _full_config(name, act=None, budget=3e6, softmax_rows_max=8192):
    """The full workload in the benchmark's launch configuration.  Every gradient
    element of a deterministic subset of samples (up to `budget` query-key
    pairs each); the longest sample in full when the workload is causal or has a
    bias (the oracle backward of a 4096-token causal sample takes seconds);
    otherwise dQ rows and dK / dV key rows of the longest sample (softmax: the
    longest up to `softmax_rows_max` tokens, whose whole oracle forward is
    needed for lse and D)."""
    w = make_workload(name, act=act)
    t = make_tensors(w, device=DEV)
    dq, dk, dv = run_bwd(t["q"], t["qo"], t["k"], t["v"], t["ko"], t["dout"], w.act, w.causal,
                         w.scale, t["bias"], w.max_rel)
    qo, ko = w.offsets()
    pairs = w.lq * w.lkv
    samples = [b for b in pick_samples(w.lq, w.lkv, budget_pairs=budget) if pairs[b] <= budget]
    longest = int(np.argmax(pairs))
    plain = not w.causal and t["bias"] is None
    if not plain:
        samples.append(longest)
    if not samples:
        samples = [int(np.argmin(pairs))]
    _check_samples(t["q"], t["k"], t["v"], t["dout"], qo, ko, sorted(set(samples)), w.act,
                   w.causal, w.scale, t["bias"], w.max_rel, dq, dk, dv, name)
    if plain:
        # longest sample: dQ rows are independent given all keys, so check a row subset
        b = longest
        q0, k0, k1 = int(qo[b]), int(ko[b]), int(ko[b + 1])
        L = int(w.lq[b])
        rows = np.array(sorted({0, 1, L // 3, L // 2, L - 2, L - 1}))
        rows = rows[(rows >= 0) & (rows < L)]
        sel = torch.from_numpy(q0 + rows).to(DEV)
        rq, _, _ = oracle.bwd(to_np(t["q"][sel]), np.array([0, len(rows)]), to_np(t["k"][k0:k1]),
                              to_np(t["v"][k0:k1]), np.array([0, k1 - k0]),
                              to_np(t["dout"][sel]), act=ACTS[w.act], causal=False,
                              scale=w.scale)
        assert_close(to_np(dq[sel]), rq, BWD_TOL, f"{name} dq rows of longest sample")
        # dK / dV key rows of the longest sample (softmax: the longest that fits the cap)
        if w.act == "softmax":
            fit = np.flatnonzero(w.lq <= softmax_rows_max)
            b = int(fit[np.argmax(pairs[fit])])
        if pairs[b] > budget:
            _check_key_rows(t, w, b, dk, dv, name)


def test_bwd_full_jfa_causal_relpos():
    _full_config("jfa_causal_relpos", budget=4e6)


def test_bwd_full_gdpa_cross_gelu():
    _full_config("gdpa_cross_gelu")


def test_bwd_full_gdpa_pma_silu():
    _full_config("gdpa_pma_silu")


@pytest.mark.parametrize("act", ["softmax", "silu"])
def test_bwd_full_heavy_tail(act):
    _full_config("heavy_tail", act=act, budget=1.5e6)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("variant", ["full", "causal", "window", "clamped"])
@pytest.mark.parametrize("act", ["softmax", "silu", "gelu_tanh"])
def test_dbias(act, d, variant):
    """Gradient of the relative-position table against the oracle's; it is
    added to, so a second call doubles it."""
    H = 2
    a = ACTS[act]
    causal = variant in ("causal", "window")
    window = 150 if variant == "window" else 0
    max_rel = 40 if variant == "clamped" else 600
    lq = [1, 129, 300, 0, 257, 64, 511]
    lkv = lq if causal else [5, 200, 128, 3, 300, 64, 400]
    g = torch.Generator(device=DEV).manual_seed(50 + d)
    q = rand_bf16((sum(lq), H, d), g, DEV)
    k = rand_bf16((sum(lkv), H, d), g, DEV)
    v = rand_bf16((sum(lkv), H, d), g, DEV)
    do = rand_bf16((sum(lq), H, d), g, DEV)
    bias = torch.randn(H, 2 * max_rel - 1, generator=g, device=DEV) * 0.5
    qo_np, ko_np = offsets(lq), offsets(lkv)
    qo, ko = torch.from_numpy(qo_np).to(DEV), torch.from_numpy(ko_np).to(DEV)
    scale = 1.0 / math.sqrt(d)
    kw = dict(act=a, causal=causal, scale=scale, bias=bias, max_rel=max_rel, window=window)
    out, lse = binding.gdpa_fwd(q, qo, k, v, ko, **kw)
    dbias = torch.zeros_like(bias)
    binding.gdpa_bwd(q, qo, k, v, ko, out, lse, do, dbias=dbias, **kw)
    assert binding.device_status() == 0
    check_table_gradient(q, qo_np, k, v, ko_np, do, bias, dbias, act=a, causal=causal,
                         scale=scale, max_rel=max_rel, window=window,
                         what=f"dbias {variant} d={d}")
    first = dbias.clone()
    binding.gdpa_bwd(q, qo, k, v, ko, out, lse, do, dbias=dbias, **kw)
    assert binding.device_status() == 0
    # (the fp32 atomics add in a different order each call: only the last bits differ)
    torch.testing.assert_close(dbias, 2 * first, rtol=1e-3, atol=1e-4 * float(first.abs().max()))


@pytest.mark.parametrize("act", ["softmax", "silu"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_fused_rope(causal, d, act):
    """gdpa_bwd_rope: q and k arrive rotary-embedded; dq and dk come back for
    the un-rotated q, k (the oracle's rotary backward applied to its gradients,
    queries and keys at their own positions), dv unchanged."""
    lq = [1, 64, 65, 200, 0, 300, 129]
    lkv = lq if causal else [7, 1, 130, 64, 5, 257, 3]
    H, base = 2, 10000.0
    g = torch.Generator(device="cuda").manual_seed(77 + d)
    q = rand_bf16((sum(lq), H, d), g, "cuda")
    k = rand_bf16((sum(lkv), H, d), g, "cuda")
    v = rand_bf16((sum(lkv), H, d), g, "cuda")
    do = rand_bf16((sum(lq), H, d), g, "cuda")
    qo_np, ko_np = offsets(lq), offsets(lkv)
    qo, ko = torch.from_numpy(qo_np).cuda(), torch.from_numpy(ko_np).cuda()
    scale = 1.0 / math.sqrt(d)
    a = ACTS[act]
    out, lse = binding.gdpa_fwd(q, qo, k, v, ko, act=a, causal=causal, scale=scale)
    bq, dq = guarded(sum(lq), H, d, q.device)
    bk, dk = guarded(sum(lkv), H, d, q.device)
    bv, dv = guarded(sum(lkv), H, d, q.device)
    binding.gdpa_bwd(q, qo, k, v, ko, out, lse, do, act=a, causal=causal, scale=scale,
                     rope_base=base, dq=dq, dk=dk, dv=dv)
    assert binding.device_status() == 0
    for b_ in (bq, bk, bv):
        check_guards(b_)
    rq, rk, rv = oracle.bwd(to_np(q), qo_np, to_np(k), to_np(v), ko_np, to_np(do), act=a,
                            causal=causal, scale=scale)
    what = f"rope bwd {act} d={d} causal={causal}"
    assert_close(to_np(dq), oracle.rope_bwd(rq, qo_np, base), BWD_TOL, what + " dq")
    assert_close(to_np(dk), oracle.rope_bwd(rk, ko_np, base), BWD_TOL, what + " dk")
    assert_close(to_np(dv), rv, BWD_TOL, what + " dv")


@pytest.mark.parametrize("act", ["softmax", "silu"])
def test_bwd_fused_rope_with_window(act):
    """gdpa_bwd_rope with a sliding window (the windowed instantiation)."""
    L = [1, 64, 65, 200, 300, 129]
    H, d, base, window = 2, 128, 500.0, 100
    g = torch.Generator(device="cuda").manual_seed(91)
    q, k, v, do = (rand_bf16((sum(L), H, d), g, "cuda") for _ in range(4))
    o_np = offsets(L)
    o = torch.from_numpy(o_np).cuda()
    scale = 1.0 / math.sqrt(d)
    a = ACTS[act]
    out, lse = binding.gdpa_fwd(q, o, k, v, o, act=a, causal=True, scale=scale, window=window)
    dq, dk, dv = binding.gdpa_bwd(q, o, k, v, o, out, lse, do, act=a, causal=True, scale=scale,
                                  window=window, rope_base=base)
    assert binding.device_status() == 0
    rq, rk, rv = oracle.bwd(to_np(q), o_np, to_np(k), to_np(v), o_np, to_np(do), act=a,
                            causal=True, scale=scale, window=window)
    what = f"rope+window bwd {act}"
    assert_close(to_np(dq), oracle.rope_bwd(rq, o_np, base), BWD_TOL, what + " dq")
    assert_close(to_np(dk), oracle.rope_bwd(rk, o_np, base), BWD_TOL, what + " dk")
    assert_close(to_np(dv), rv, BWD_TOL, what + " dv")


@pytest.mark.parametrize("act", ["softmax", "silu"])
@pytest.mark.parametrize("window", [0, 100])
def test_bwd_fused_rope_with_table_gradient(window, act):
    """gdpa_bwd_rope with a relative-position table and its gradient: dq, dk
    through the rotary backward, the table's gradient unchanged by it."""
    lq = [1, 64, 65, 200, 0, 300, 129]
    H, d, base, max_rel = 2, 128, 10000.0, 150
    g = torch.Generator(device="cuda").manual_seed(93 + window)
    q, k, v, do = (rand_bf16((sum(lq), H, d), g, "cuda") for _ in range(4))
    bias = torch.randn(H, 2 * max_rel - 1, generator=g, device="cuda") * 0.5
    o_np = offsets(lq)
    o = torch.from_numpy(o_np).cuda()
    scale = 1.0 / math.sqrt(d)
    a = ACTS[act]
    kw = dict(act=a, causal=True, scale=scale, bias=bias, max_rel=max_rel, window=window)
    out, lse = binding.gdpa_fwd(q, o, k, v, o, **kw)
    dbias = torch.zeros_like(bias)
    dq, dk, dv = binding.gdpa_bwd(q, o, k, v, o, out, lse, do, rope_base=base, dbias=dbias, **kw)
    assert binding.device_status() == 0
    rq, rk, rv = oracle.bwd(to_np(q), o_np, to_np(k), to_np(v), o_np, to_np(do), act=a,
                            causal=True, scale=scale, bias=bias.cpu().double().numpy(),
                            max_rel=max_rel, window=window)
    what = f"rope+table gradient {act} window={window}"
    assert_close(to_np(dq), oracle.rope_bwd(rq, o_np, base), BWD_TOL, what + " dq")
    assert_close(to_np(dk), oracle.rope_bwd(rk, o_np, base), BWD_TOL, what + " dk")
    assert_close(to_np(dv), rv, BWD_TOL, what + " dv")
    check_table_gradient(q, o_np, k, v, o_np, do, bias, dbias, act=a, causal=True, scale=scale,
                         max_rel=max_rel, window=window, what=what + " dbias")


# Epilogues store rows with 32-byte stores when every output base is 32-byte
# aligned and with 16-byte stores otherwise: outputs that start 16 bytes into
# an allocation must give the same results, for the forward and for every
# backward kernel family (softmax, GDPA, short-query samples).
@pytest.mark.parametrize("act", ["softmax", "silu"])
def test_outputs_at_16_byte_offsets(act):
    lq, lkv = [300, 20, 129, 1], [260, 700, 5, 129]
    H, d = 2, 128
    g = torch.Generator(device=DEV).manual_seed(3)
    q = rand_bf16((sum(lq), H, d), g, DEV)
    k = rand_bf16((sum(lkv), H, d), g, DEV)
    v = rand_bf16((sum(lkv), H, d), g, DEV)
    do = rand_bf16((sum(lq), H, d), g, DEV)
    qo = torch.from_numpy(offsets(lq)).to(DEV)
    ko = torch.from_numpy(offsets(lkv)).to(DEV)
    a = ACTS[act]
    scale = 1.0 / math.sqrt(d)

    def shifted(like):  # a view that starts 16 bytes into its allocation
        buf = torch.empty(like.numel() + 8, device=DEV, dtype=torch.bfloat16)
        view = buf[8:].view(like.shape)
        assert view.data_ptr() % 32 == 16
        return view

    out, lse = binding.gdpa_fwd(q, qo, k, v, ko, act=a, scale=scale)
    out16 = shifted(out)
    _, lse16 = binding.gdpa_fwd(q, qo, k, v, ko, act=a, scale=scale, out=out16)
    assert torch.equal(out16, out)
    if lse is not None:
        assert torch.equal(lse16, lse)
    grads = binding.gdpa_bwd(q, qo, k, v, ko, out, lse, do, act=a, scale=scale)
    g16 = [shifted(t) for t in grads]
    binding.gdpa_bwd(q, qo, k, v, ko, out, lse, do, act=a, scale=scale, dq=g16[0], dk=g16[1],
                     dv=g16[2])
    assert binding.device_status() == 0
    # dK and dV rows are written once each: same bits.  dQ is summed by
    # reduce-adds in whatever order the key blocks finish (its conversion
    # always uses 16-byte stores): equal up to the last bf16 bit.
    assert torch.equal(grads[1], g16[1]) and torch.equal(grads[2], g16[2])
    torch.testing.assert_close(g16[0], grads[0], rtol=2 ** -7, atol=1e-3)
