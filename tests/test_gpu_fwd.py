"""GPU parity of the forward pass against the fp64 oracle (through the C ABI).

Tolerance: |gpu - oracle| <= 1e-2 + 1e-2 |oracle| elementwise (bf16 forward).
Outputs are written into NaN-filled buffers with guard rows on both sides:
every valid row must be finite and every guard row untouched.
"""
import math

import numpy as np
import pytest
import torch

from gpu_common import (FWD_TOL, assert_close, offsets, oracle_fwd_samples, pick_samples,
                        rand_bf16, run_fwd, to_np)
from jagged_attention_recsys_02_gb300.workloads import make_tensors, make_workload

pytestmark = pytest.mark.gpu

DEV = "cuda"

# Lengths crossing every tile boundary (128-row kv tiles, 256-row query items).
RAGGED_Q = [1, 127, 128, 129, 255, 256, 257, 0, 300, 513, 64, 7]
RAGGED_KV = [5, 128, 0, 129, 200, 256, 384, 3, 1, 513, 700, 64]


def _case(lq, lkv, H, d, act, causal=False, max_rel=0, seed=0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    q = rand_bf16((sum(lq), H, d), g, DEV)
    k = rand_bf16((sum(lkv), H, d), g, DEV)
    v = rand_bf16((sum(lkv), H, d), g, DEV)
    qo = torch.from_numpy(offsets(lq)).to(DEV)
    ko = torch.from_numpy(offsets(lkv)).to(DEV)
    bias = None
    if max_rel:
        bias = torch.randn(H, 2 * max_rel - 1, generator=g, device=DEV) * 0.5
    scale = 1.0 / math.sqrt(d)
    out, lse = run_fwd(q, qo, k, v, ko, act, causal, scale, bias, max_rel)
    ref = oracle_fwd_samples(to_np(q), to_np(k), to_np(v), offsets(lq), offsets(lkv),
                             range(len(lq)), act, causal, scale,
                             None if bias is None else bias.cpu().double().numpy(), max_rel)
    got = to_np(out)
    got_lse = lse.cpu().double().numpy() if lse is not None else None
    for rows, o, l in ref:
        assert_close(got[rows], o, FWD_TOL, f"out rows {rows[0]}..{rows[-1]}")
        if got_lse is not None:
            assert_close(got_lse[:, rows], l, FWD_TOL, "lse")
    return out


@pytest.mark.parametrize("act", ["softmax", "silu", "gelu_tanh", "identity", "gelu_erf"])
@pytest.mark.parametrize("d", [64, 128])
def test_fwd_ragged(act, d):
    _case(RAGGED_Q, RAGGED_KV, 2, d, act)


@pytest.mark.parametrize("act", ["softmax", "silu"])
@pytest.mark.parametrize("d", [64, 128])
def test_fwd_causal_relpos(act, d):
    L = [1, 128, 129, 300, 0, 511, 64, 257]
    _case(L, L, 2, d, act, causal=True, max_rel=200)


@pytest.mark.parametrize("act", ["softmax", "silu"])
def test_fwd_causal_no_bias(act):
    L = [1, 128, 129, 300, 0, 511, 64, 257, 1000]
    _case(L, L, 2, 128, act, causal=True)


@pytest.mark.parametrize("act", ["softmax", "gelu_tanh"])
def test_fwd_bias_noncausal(act):
    _case([5, 300, 129], [260, 7, 500], 3, 128, act, max_rel=64)


# Relative-position tables whose entries span 0.3, 40 and 100 (natural units)
# against scores twice the usual size: the running maximum and the rescaling
# of the softmax must keep every row exact when the bias, not the score,
# decides which key dominates.
@pytest.mark.parametrize("span", [0.3, 40.0, 100.0])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_bias_span(span, causal):
    L = [1, 130, 300, 0, 511, 257]
    H, d, max_rel = 2, 128, 300
    g = torch.Generator(device=DEV).manual_seed(7)
    q = rand_bf16((sum(L), H, d), g, DEV) * 2.0
    k = rand_bf16((sum(L), H, d), g, DEV)
    v = rand_bf16((sum(L), H, d), g, DEV)
    o = torch.from_numpy(offsets(L)).to(DEV)
    table = torch.rand(H, 2 * max_rel - 1, generator=g, device=DEV) * span - span / 2
    scale = 1.0 / math.sqrt(d)
    out, lse = run_fwd(q, o, k, v, o, "softmax", causal, scale, table, max_rel)
    ref = oracle_fwd_samples(to_np(q), to_np(k), to_np(v), offsets(L), offsets(L), range(len(L)),
                             "softmax", causal, scale, table.cpu().double().numpy(), max_rel)
    got, got_lse = to_np(out), lse.cpu().double().numpy()
    for rows, ro, rl in ref:
        assert_close(got[rows], ro, FWD_TOL, f"out rows {rows[0]}..{rows[-1]}")
        assert_close(got_lse[:, rows], rl, FWD_TOL, "lse")


# At most 32 queries: the short-query kernel (keys as TMEM lanes, the queries
# as the MMA's N); the 300-query sample of the same call takes the row-tile
# kernel.  Key counts cross the 128-key tiles, and one short sample has none.
SHORT_Q = [32, 1, 31, 0, 17, 32, 2, 5, 32, 300]
SHORT_KV = [700, 1, 128, 9, 0, 129, 256, 513, 64, 200]


@pytest.mark.parametrize("act", ["silu", "gelu_tanh", "identity", "gelu_erf"])
@pytest.mark.parametrize("d", [64, 128])
def test_fwd_short_queries(act, d):
    out = _case(SHORT_Q, SHORT_KV, 3, d, act)
    assert torch.all(out[sum(SHORT_Q[:4]):sum(SHORT_Q[:5])] == 0)  # the sample with no key


# Short-key samples (more than 32 queries, 1..256 keys, GDPA without mask or
# bias: the cross-attention shape) take the kernel that keeps a sample's K and
# V in shared memory and streams its queries in 128-row tiles, in items of up
# to 2048 queries.  Key counts cross the 16-key MMA steps, the 32-key
# activation chunks and the 128-key boundary between two S buffers and one;
# query counts cross the 128-row tiles and the 2048-query items.  One sample
# has 257 keys (the general kernel), the last has none.
SHORT_KV_Q = [33, 2049, 129, 40, 300, 128, 4100, 77, 2048, 500, 64, 1000, 35]
SHORT_KV_KV = [1, 16, 17, 31, 33, 127, 128, 129, 200, 255, 256, 257, 0]


@pytest.mark.parametrize("act", ["silu", "gelu_tanh", "identity", "gelu_erf"])
@pytest.mark.parametrize("d", [64, 128])
def test_fwd_short_keys(act, d):
    out = _case(SHORT_KV_Q, SHORT_KV_KV, 3, d, act)
    assert torch.all(out[-SHORT_KV_Q[-1]:] == 0)  # the sample with no key


def test_fwd_empty_keys_and_queries():
    # samples with no keys give zero rows (lse = -inf for softmax); empty query samples write nothing
    out = _case([3, 0, 130, 5], [0, 9, 0, 140], 2, 128, "softmax")
    assert torch.all(out[:3] == 0) and torch.all(out[3:133] == 0)


def test_fwd_all_empty_keys_gdpa():
    out = _case([4, 9], [0, 0], 1, 64, "silu")
    assert torch.all(out == 0)


def test_fwd_tiny_config():
    w = make_workload("tiny_silu")
    t = make_tensors(w, device=DEV)
    out, _ = run_fwd(t["q"], t["qo"], t["k"], t["v"], t["ko"], w.act, w.causal, w.scale)
    qo, ko = w.offsets()
    ref = oracle_fwd_samples(to_np(t["q"]), to_np(t["k"]), to_np(t["v"]), qo, ko, range(w.B),
                             w.act, w.causal, w.scale)
    got = to_np(out)
    for rows, o, _ in ref:
        assert_close(got[rows], o, FWD_TOL, "tiny")


def test_fwd_deterministic():
    g = torch.Generator(device=DEV).manual_seed(3)
    lq = [700, 33, 1000]
    q = rand_bf16((sum(lq), 2, 128), g, DEV)
    k = rand_bf16((sum(lq), 2, 128), g, DEV)
    v = rand_bf16((sum(lq), 2, 128), g, DEV)
    o = torch.from_numpy(offsets(lq)).to(DEV)
    a, _ = run_fwd(q, o, k, v, o, "silu", False, 0.1)
    b, _ = run_fwd(q, o, k, v, o, "silu", False, 0.1)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ------------------------------------------------------------------ full-size workloads
def _full_config(name, act=None, row_sample=False):
    w = make_workload(name, act=act)
    t = make_tensors(w, device=DEV, with_dout=False)
    bias = t["bias"]
    out, lse = run_fwd(t["q"], t["qo"], t["k"], t["v"], t["ko"], w.act, w.causal, w.scale,
                       bias, w.max_rel)
    qo, ko = w.offsets()
    samples = pick_samples(w.lq, w.lkv, budget_pairs=4e6 if not row_sample else 2e5)
    rows = None
    if row_sample:
        # query rows are independent when there is no mask and no bias: check the
        # first, last and tile-boundary rows of each chosen sample
        rows = {}
        for b in samples:
            L = int(w.lq[b])
            cand = {0, 1, L - 1, L // 2}
            for t_ in range(128, L, 128 * 7):
                cand.update({t_ - 1, t_})
            rows[b] = np.array(sorted(x for x in cand if 0 <= x < L))
    sel_q = sorted({int(x) for b in samples for x in range(int(qo[b]), int(qo[b + 1]))})
    # copy only the needed slices to the host
    qh, kh, vh = t["q"], t["k"], t["v"]
    ref = []
    for b in samples:
        q0, q1, k0, k1 = int(qo[b]), int(qo[b + 1]), int(ko[b]), int(ko[b + 1])
        sub = oracle_fwd_samples(to_np(qh[q0:q1]), to_np(kh[k0:k1]), to_np(vh[k0:k1]),
                                 np.array([0, q1 - q0]), np.array([0, k1 - k0]), [0], w.act,
                                 w.causal, w.scale,
                                 None if bias is None else bias.cpu().double().numpy(), w.max_rel,
                                 rows={0: rows[b]} if rows else None)
        for r, o, l in sub:
            ref.append((r + q0, o, l))
    del sel_q
    for rows_g, o, l in ref:
        got = to_np(out[torch.from_numpy(rows_g).to(DEV)])
        assert_close(got, o, FWD_TOL, f"{name} rows {rows_g[0]}..{rows_g[-1]}")
        if lse is not None:
            got_l = lse[:, torch.from_numpy(rows_g).to(DEV)].cpu().double().numpy()
            assert_close(got_l, l, FWD_TOL, f"{name} lse")


def test_fwd_full_jfa_causal_relpos():
    _full_config("jfa_causal_relpos")


def test_fwd_full_gdpa_cross_gelu():
    _full_config("gdpa_cross_gelu")


def test_fwd_full_gdpa_pma_silu():
    _full_config("gdpa_pma_silu")


@pytest.mark.parametrize("act", ["softmax", "silu"])
def test_fwd_full_heavy_tail(act):
    _full_config("heavy_tail", act=act, row_sample=True)
