"""Helpers shared by the GPU parity tests (no test functions here)."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from jagged_attention_recsys_02_gb300 import binding
from jagged_attention_recsys_02_gb300.workloads import ACTS

FWD_TOL = (1e-2, 1e-2)     # (abs, rel) for the bf16 forward
BWD_TOL = (3e-2, 3e-2)     # (abs, rel) for the bf16 backward
MXFP8_TOL = (6e-2, 6e-2)   # (abs, rel) for the MXFP8 forward

BF16_NAN = 0x7FC0


def offsets(lengths):
    o = np.zeros(len(lengths) + 1, dtype=np.int32)
    o[1:] = np.cumsum(lengths)
    return o


def rand_bf16(shape, gen, device):
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def guarded(rows, H, d, device, guard=3):
    """A bf16 [rows, H, d] view into a NaN-filled buffer with `guard` extra rows
    on each side; returns (buffer, view)."""
    buf = torch.empty((rows + 2 * guard, H, d), device=device, dtype=torch.bfloat16)
    buf.view(torch.int16).fill_(BF16_NAN)
    return buf, buf[guard:guard + rows]


def check_guards(buf, guard=3):
    raw = buf.view(torch.int16)
    assert torch.all(raw[:guard] == BF16_NAN), "write before the output rows"
    assert torch.all(raw[raw.shape[0] - guard:] == BF16_NAN), "write after the output rows"


def assert_close(got, ref, tol, what):
    """Elementwise |got - ref| <= abs + rel * |ref| (ref = oracle, float64)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    # an infinite reference (lse of a row with no key) must be matched exactly
    inf = np.isinf(ref)
    assert np.array_equal(got[inf], ref[inf]), f"{what}: infinite entries differ"
    got, ref = got[~inf], ref[~inf]
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    bound = tol[0] + tol[1] * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.flatnonzero(bad)[:5]
        worst = float((err / bound).max())
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance "
                             f"(worst err/bound {worst:.3f}); first flat indices {idx.tolist()}: "
                             f"got {got[idx[0]]} ref {ref[idx[0]]}")
    return float((err / bound).max()) if err.size else 0.0


def run_fwd(q, qo, k, v, ko, act, causal, scale, bias=None, max_rel=0, guard=3, window=0):
    Tq, H, d = q.shape
    buf, out = guarded(Tq, H, d, q.device, guard)
    a = ACTS[act] if isinstance(act, str) else act
    lse = torch.full((H, Tq), float("nan"), device=q.device) if a == 0 else None
    binding.gdpa_fwd(q, qo, k, v, ko, act=a, causal=causal, scale=scale, bias=bias,
                     max_rel=max_rel, window=window, out=out, lse=lse)
    st = binding.device_status()
    assert st == 0, f"device status {st}"
    check_guards(buf, guard)
    return out, lse


def oracle_fwd_samples(q, k, v, qo, ko, samples, act, causal, scale, bias=None, max_rel=0,
                       rows=None, window=0, block=0):
    """Oracle forward on a subset of samples (and optionally a subset of query
    rows per sample: rows[b] = array of local row indices; only for
    non-causal, bias-free problems, where rows are position-independent).
    Returns a list of (global_row_indices, out[rows, H, d], lse[H, rows])."""
    a = ACTS[act] if isinstance(act, str) else act
    res = []
    for b in samples:
        q0, q1 = int(qo[b]), int(qo[b + 1])
        k0, k1 = int(ko[b]), int(ko[b + 1])
        if q1 == q0:
            continue
        if rows is not None and rows.get(b) is not None:
            assert not causal and bias is None
            sel = np.asarray(rows[b])
            qs = q[q0 + sel]
            glob = q0 + sel
        else:
            qs = q[q0:q1]
            glob = np.arange(q0, q1)
        o, l = oracle.fwd(qs, np.array([0, len(qs)], dtype=np.int32), k[k0:k1], v[k0:k1],
                          np.array([0, k1 - k0], dtype=np.int32), act=a, causal=causal,
                          scale=scale, bias=bias, max_rel=max_rel, window=window, block=block)
        res.append((glob, o, l))
    return res


def pick_samples(lq, lkv, budget_pairs=3e6, always=()):
    """Deterministic parity subset: shortest and longest sample, then every
    k-th sample while the pair budget lasts."""
    pairs = np.asarray(lq, dtype=np.int64) * np.asarray(lkv, dtype=np.int64)
    order = np.argsort(pairs, kind="stable")
    chosen = [int(order[0]), int(order[-1]), *always]
    total = int(sum(pairs[c] for c in set(chosen)))
    B = len(lq)
    step = max(1, B // 16)
    for b in range(0, B, step):
        if total + pairs[b] > budget_pairs:
            continue
        chosen.append(b)
        total += int(pairs[b])
    return sorted(set(chosen))


def to_np(t):
    return t.detach().float().cpu().double().numpy()


def scale_for(d):
    return 1.0 / math.sqrt(d)


def ds_pair_bounds(qn, qo, kn, vn, ko, don, o_ref, *, act, causal, scale, window=0,
                   bias_of=None, block=0):
    """Per (sample, head) of a backward problem: the unmasked pairs and a bound
    on the kernels' rounding in each pair's dS, from fp64 quantities of the
    same inputs.  Softmax: the kernel's D = rowsum(dO * O) uses the
    bf16-rounded O (relative error <= 2^-9 per element) and dS is formed from
    bf16 P and dP - D and rounded to bf16 (2^-9 each); per pair about
    |P| 2^-8 (|dP - D| + sum_c |dO_c O_c|).  GDPA: dS = act'(s) dP in fp32
    from fp32 scores; per pair at most 1.2 |dP| 2^-8 (|act'| <= 1.2 for SiLU
    and GELU).  bias_of(b, h, i, j) returns the bias of sample b, head h at
    local query / key grids i, j (None: no bias); block > 0 keeps only the
    pairs inside one block of that many tokens.  Yields (b, h, live, bound)
    with [Lq_b, Lkv_b] arrays."""
    a = ACTS[act] if isinstance(act, str) else act
    H = qn.shape[1]
    for b in range(len(qo) - 1):
        q0, q1, k0, k1 = int(qo[b]), int(qo[b + 1]), int(ko[b]), int(ko[b + 1])
        if q1 == q0 or k1 == k0:
            continue
        i = np.arange(q1 - q0)[:, None]
        j = np.arange(k1 - k0)[None, :]
        live = np.ones((q1 - q0, k1 - k0), bool)
        if causal:
            live &= j <= i
        if window:
            live &= np.abs(i - j) < window
        if block:
            live &= (i // block) == (j // block)
        for h in range(H):
            s0 = scale * qn[q0:q1, h] @ kn[k0:k1, h].T
            if bias_of is not None:
                s0 = s0 + bias_of(b, h, i, j)
            dp = don[q0:q1, h] @ vn[k0:k1, h].T
            if a == 0:
                s_ = np.where(live, s0, -np.inf)
                pm = np.exp(s_ - s_.max(1, keepdims=True))
                pm /= pm.sum(1, keepdims=True)
                dd = (don[q0:q1, h] * o_ref[q0:q1, h]).sum(1, keepdims=True)
                od = np.abs(don[q0:q1, h] * o_ref[q0:q1, h]).sum(1, keepdims=True)
                e = pm * 2.0 ** -8 * (np.abs(dp - dd) + od)
            else:
                e = 1.2 * 2.0 ** -8 * np.abs(dp)
            yield b, h, live, e


def check_table_gradient(q, qo_np, k, v, ko_np, do, bias, dbias, *, act, causal, scale, max_rel,
                         window, what):
    """The relative-position table's gradient against the oracle's.  Each
    table entry sums dS over many pairs, so the per-pair rounding
    (ds_pair_bounds) adds up.  Tolerance: the elementwise bound plus 4 times
    the per-pair bounds summed over the entry's pairs."""
    tb = bias.cpu().double().numpy()
    qn, kn, vn, don = to_np(q), to_np(k), to_np(v), to_np(do)
    *_, ref = oracle.bwd(qn, qo_np, kn, vn, ko_np, don, act=act, causal=causal, scale=scale,
                         bias=tb, max_rel=max_rel, window=window, want_dbias=True)
    o_ref, _ = oracle.fwd(qn, qo_np, kn, vn, ko_np, act=0, causal=causal, scale=scale, bias=tb,
                          max_rel=max_rel, window=window)
    width = 2 * max_rel - 1
    tab = lambda i, j: np.clip(i - j + max_rel - 1, 0, width - 1)
    err = np.zeros_like(ref)
    for b, h, live, e in ds_pair_bounds(qn, qo_np, kn, vn, ko_np, don, o_ref, act=act,
                                        causal=causal, scale=scale, window=window,
                                        bias_of=lambda b, h, i, j: tb[h][tab(i, j)]):
        t = tab(np.arange(live.shape[0])[:, None], np.arange(live.shape[1])[None, :])
        np.add.at(err[h], t[live], e[live])
    got = dbias.cpu().double().numpy()
    bound = BWD_TOL[0] + BWD_TOL[1] * np.abs(ref) + 4 * err
    assert np.all(np.abs(got - ref) <= bound), \
        f"{what}: worst err/bound {float((np.abs(got - ref) / bound).max()):.3f}"


def dense_ref_kw(c):
    """Oracle keyword arguments of a dense-bias case: a dict with act, causal,
    scale, window, block and the bias values vals (torch, on any device)."""
    return dict(act=c["act"], causal=c["causal"], scale=c["scale"], window=c["window"],
                block=c["block"], dense_bias=c["vals"].double().cpu().numpy())


def check_dense_gradient(c, got, base, what):
    """got = base + the kernel's dS of every unmasked pair, in the dense bias's
    layout: against the oracle's gradient within the per-pair rounding bound
    (times 4) plus the fp32 rounding of the addition to base; masked entries
    keep base bit for bit."""
    Tq, H, d = c["q"].shape
    qn, kn, vn, don = to_np(c["q"]), to_np(c["k"]), to_np(c["v"]), to_np(c["do"])
    *_, ref = oracle.bwd(qn, c["qo_np"], kn, vn, c["ko_np"], don, want_dbias=True, **dense_ref_kw(c))
    o_ref, _ = oracle.fwd(qn, c["qo_np"], kn, vn, c["ko_np"], **dense_ref_kw(c))
    vals = c["vals"].double().cpu().numpy()
    off = oracle.dense_bias_offsets(c["qo_np"], c["ko_np"], H)
    got = got.cpu()
    base = base.cpu()
    live_all = np.zeros(int(off[-1]), bool)
    pair = np.zeros(int(off[-1]))
    for b, h, live, e in ds_pair_bounds(qn, c["qo_np"], kn, vn, c["ko_np"], don, o_ref,
                                        act=c["act"], causal=c["causal"], scale=c["scale"],
                                        window=c["window"], block=c["block"],
                                        bias_of=lambda b, h, i, j: vals[
                                            off[b] + (h * i.shape[0] + i) * j.shape[1] + j]):
        n = live.size
        s = slice(int(off[b]) + h * n, int(off[b]) + (h + 1) * n)
        live_all[s] = live.reshape(-1)
        pair[s] = e.reshape(-1)
    assert torch.equal(got[~torch.from_numpy(live_all)], base[~torch.from_numpy(live_all)]), \
        f"{what}: a masked entry changed"
    g, b0 = got.double().numpy()[live_all], base.double().numpy()[live_all]
    r = ref[live_all]
    bound = 4 * pair[live_all] + 2.0 ** -23 * (np.abs(b0) + np.abs(r)) + 1e-7 * np.abs(r).max()
    err = np.abs(g - b0 - r)
    assert np.all(err <= bound), \
        f"{what}: {int((err > bound).sum())} of {err.size} out, worst err/bound {(err / bound).max():.3f}"
    # the softmax kernel rounds dS to bf16, the others keep it in fp32: both
    # sit far inside the bound above; the bound itself is not vacuous
    assert np.median(bound) < 1e-2 * np.abs(r).max()
