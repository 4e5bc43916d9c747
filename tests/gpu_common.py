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
