"""The varlen tile scheduler's work list, read back from the workspace.

"GEM Training ..." JFA paragraph: with jagged inputs, short sequences finish
early and leave SMs idle.  The library's scheduler kernel turns the offsets
into a list of (sample, head, block) items that persistent CTAs pull in
order; it writes the item count at byte 0 of the caller's workspace and the
items, one int2 {sample, (block << 8) | head} each, from byte 256.  These
tests run gdpa_fwd / gdpa_bwd (forward: blocks of 256 query rows over
128-key tiles; backward: blocks of 128 keys over 64-query tiles) and check
the list against a host count made row by row from the mask's definition
(samples with at most 32 queries and no mask or bias go to a second list,
one {sample, head} item each, for the short-query kernels; in the GDPA
forward without mask or bias, samples with more queries and 1..256 keys go
to a third list, one {sample, (chunk << 8) | head} item per 2048-query chunk,
for the short-key kernel):

  * every (sample, head, block) with rows appears exactly once, and nothing else;
  * a sample's items are contiguous, heads innermost, and without a window
    its blocks come in descending cost;
  * the samples' total costs do not increase along the list (exactly below
    1024 inner tiles, in 64-tile steps above, the scheduler's histogram);
  * a block's cost is 1 + the number of inner tiles holding a key (query)
    that some row of the block sees under the causal / sliding-window band.
"""
import math

import numpy as np
import pytest
import torch

from gpu_common import offsets, rand_bf16
from jagged_attention_recsys_02_gb300 import binding
from jagged_attention_recsys_02_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _visible(i, Lkv, causal, window):
    """Keys [lo, hi) that query rows i (an array) see."""
    lo = np.maximum(0, i - window + 1) if window else np.zeros_like(i)
    hi = np.minimum(Lkv, i + 1) if causal else (np.minimum(Lkv, i + window) if window
                                                 else np.full_like(i, Lkv))
    return lo, hi


def _fwd_cost(Lq, Lkv, blk, causal, window):
    i = np.arange(blk * 256, min(Lq, blk * 256 + 256))
    lo, hi = _visible(i, Lkv, causal, window)
    tiles = set()
    for a, b in zip(lo[hi > lo] // 128, (hi[hi > lo] - 1) // 128):
        tiles.update(range(int(a), int(b) + 1))
    return len(tiles) + 1


def _bwd_cost(Lq, Lkv, blk, causal, window):
    i = np.arange(Lq)
    lo, hi = _visible(i, Lkv, causal, window)
    sees = np.maximum(lo, blk * 128) < np.minimum(hi, blk * 128 + 128)  # row i sees the block
    return len(np.unique(i[sees] // 64)) + 1


def _bucket(total):
    return total if total < 1024 else 1024 + (total - 1024) // 64


def _align(n):
    return (n + 255) // 256 * 256


def _read_list(ws, short_at):
    """Main list (count at byte 0, items from byte 256) and the short-query
    list (count at byte 8, items from byte short_at, one {sample, head} each)."""
    raw = ws.cpu().numpy()
    n = int(raw[:4].view(np.int32)[0])
    items = raw[256:256 + 8 * n].view(np.int32).reshape(n, 2)
    main = (items[:, 0].astype(np.int64), (items[:, 1] >> 8).astype(np.int64),
            (items[:, 1] & 0xFF).astype(np.int64))
    ns = int(raw[8:12].view(np.int32)[0])
    short = raw[short_at:short_at + 8 * ns].view(np.int32).reshape(ns, 2).astype(np.int64)
    all_short = int(raw[16:20].view(np.int32)[0])
    return main, short, all_short


def _check_short(lq, lkv, H, short_set, short, all_short, n_main):
    """Short-query samples: one item per head, longest (most key tiles) first."""
    got = [tuple(x) for x in short.tolist()]
    assert len(got) == len(set(got)), "a short item appears twice"
    assert set(got) == {(b, h) for b in short_set for h in range(H)}, "short items missing or extra"
    costs = [_bucket(1 + math.ceil(lkv[b] / 128)) for b, _ in got]
    assert all(x >= y for x, y in zip(costs, costs[1:])), "short items not longest first"
    assert all_short == (1 if (n_main == 0 and len(got) > 0) else 0)


def _read_kv_list(ws, kv_at):
    raw = ws.cpu().numpy()
    n = int(raw[20:24].view(np.int32)[0])
    items = raw[kv_at:kv_at + 8 * n].view(np.int32).reshape(n, 2).astype(np.int64)
    return items[:, 0], items[:, 1] >> 8, items[:, 1] & 0xFF


def _check_kv(lq, lkv, H, kv_set, samples, chunks, heads):
    """Short-key samples: one item per head and 2048-query chunk, heads
    innermost, items in non-increasing cost (query tiles x 32-key columns)."""
    got = list(zip(samples.tolist(), chunks.tolist(), heads.tolist()))
    assert len(got) == len(set(got)), "a short-key item appears twice"
    want = {(b, ch, h) for b in kv_set for ch in range(math.ceil(lq[b] / 2048)) for h in range(H)}
    assert set(got) == want, "short-key items missing or extra"
    costs = []
    for i in range(0, len(got), H):
        unit = got[i:i + H]
        assert [u[2] for u in unit] == list(range(H)), "heads not innermost"
        assert all(u[:2] == unit[0][:2] for u in unit)
        b, ch = unit[0][:2]
        rows = min(2048, lq[b] - 2048 * ch)
        costs.append(math.ceil(rows / 128) * math.ceil(lkv[b] / 32))
    assert all(x >= y for x, y in zip(costs, costs[1:])), "short-key items not longest first"


def _check(lq, lkv, H, causal, window, mode, samples, blocks, heads, short_set=()):
    rows = lq if mode == "fwd" else lkv
    per = 256 if mode == "fwd" else 128
    cost_fn = _fwd_cost if mode == "fwd" else _bwd_cost
    # every (sample, head, block) with rows exactly once, nothing else (samples of
    # the short-query list have no blocks here)
    want = {(b, blk, h) for b in range(len(lq)) if b not in short_set
            for blk in range(math.ceil(rows[b] / per)) for h in range(H)}
    got = list(zip(samples.tolist(), blocks.tolist(), heads.tolist()))
    assert len(got) == len(set(got)), "an item appears twice"
    assert set(got) == want, "items missing or extra"
    # contiguous samples, heads innermost, blocks in descending cost
    order = []
    for i, (b, blk, h) in enumerate(got):
        if i % H == 0:
            assert [g[2] for g in got[i:i + H]] == list(range(H)), "heads not innermost"
            assert all(g[:2] == (b, blk) for g in got[i:i + H])
            if not order or order[-1][0] != b:
                assert b not in [o[0] for o in order], f"sample {b} is not contiguous"
                order.append((b, []))
            order[-1][1].append(blk)
    totals = []
    for b, blks in order:
        costs = [cost_fn(lq[b], lkv[b], blk, causal, window) for blk in blks]
        if not window:  # a window makes the costs nearly flat; the order is then the plain one
            assert all(x >= y for x, y in zip(costs, costs[1:])), f"sample {b}: blocks not by cost"
        totals.append(sum(costs))
    buckets = [_bucket(t) for t in totals]
    assert all(x >= y for x, y in zip(buckets, buckets[1:])), "samples not longest first"
    return totals


def _run(lq, lkv, H, causal=False, window=0, act="softmax", seed=0):
    d = 64
    g = torch.Generator(device=DEV).manual_seed(seed)
    Tq, Tkv = sum(lq), sum(lkv)
    q, do = rand_bf16((Tq, H, d), g, DEV), rand_bf16((Tq, H, d), g, DEV)
    k, v = rand_bf16((Tkv, H, d), g, DEV), rand_bf16((Tkv, H, d), g, DEV)
    qo = torch.from_numpy(offsets(lq)).to(DEV)
    ko = torch.from_numpy(offsets(lkv)).to(DEV)
    a = binding.ACT_BY_NAME[act]
    ws_f = torch.zeros(binding.fwd_workspace_size(len(lq), H, d, Tq, Tkv), device=DEV,
                       dtype=torch.uint8)
    out, lse = binding.gdpa_fwd(q, qo, k, v, ko, act=a, causal=causal, scale=0.125,
                                window=window, workspace=ws_f)
    ws_b = torch.zeros(binding.bwd_workspace_size(len(lq), H, d, Tq, Tkv), device=DEV,
                       dtype=torch.uint8)
    binding.gdpa_bwd(q, qo, k, v, ko, out, lse, do, act=a, causal=causal, scale=0.125,
                     window=window, workspace=ws_b)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    B = len(lq)
    # workspace layout: short list after the main list (forward), after the main
    # list, the fp32 dQ accumulator and D (backward)
    f_short_at = 256 + _align(H * (Tq // 256 + B) * 8)
    f_kv_at = f_short_at + _align(B * H * 8)
    b_short_at = 256 + _align(H * (Tkv // 128 + B) * 8) + _align(Tq * H * d * 4) + _align(Tq * H * 4)
    (f, fs, fa), (b, bs, ba) = _read_list(ws_f, f_short_at), _read_list(ws_b, b_short_at)
    lq, lkv = np.asarray(lq), np.asarray(lkv)
    # samples with 1..32 queries take the short-query kernels when there is no
    # mask or bias (forward: GDPA activations only)
    plain = not causal and not window
    short = {i for i in range(B) if 1 <= lq[i] <= 32} if plain else set()
    f_short = short if act != "softmax" else set()
    # GDPA forward without mask or bias: more than 32 queries and 1..256 keys
    f_kv = ({i for i in range(B) if lq[i] > 32 and 1 <= lkv[i] <= 256}
            if plain and act != "softmax" else set())
    _check_short(lq, lkv, H, f_short, fs, fa, len(f[0]))
    _check_short(lq, lkv, H, short, bs, ba, len(b[0]))
    _check_kv(lq, lkv, H, f_kv, *_read_kv_list(ws_f, f_kv_at))
    return (_check(lq, lkv, H, causal, window, "fwd", *f, short_set=f_short | f_kv),
            _check(lq, lkv, H, causal, window, "bwd", *b, short_set=short))


RAGGED_Q = [1, 300, 0, 129, 513, 64, 255, 256, 257, 1000, 7, 0, 2048, 5000, 4097]
RAGGED_KV = [7, 256, 5, 0, 700, 64, 128, 129, 1, 300, 3000, 0, 200, 100, 31]


@pytest.mark.parametrize("act", ["silu", "softmax"])
def test_worklist_ragged_cross(act):
    _run(RAGGED_Q, RAGGED_KV, 3, act=act)


def test_worklist_all_short():
    """Every sample short: the main lists are empty and the flag is set."""
    _run([32, 1, 7, 20], [700, 0, 129, 5], 2, act="silu")


def test_worklist_causal():
    L = [1, 300, 0, 129, 513, 64, 255, 256, 257, 1000, 2048, 4096, 17]
    _run(L, L, 2, causal=True)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [1, 100, 300])
def test_worklist_sliding_window(causal, window):
    L = [1, 300, 0, 129, 513, 64, 255, 256, 257, 1000, 2048, 17]
    _run(L, L, 2, causal=causal, window=window)


def test_worklist_heavy_tail_lengths():
    """The heavy-tailed length mix (1024 samples, up to 16384 tokens): totals
    beyond 1024 inner tiles are ordered in the histogram's 64-tile steps."""
    w = make_workload("heavy_tail")
    lq = w.lq[:300].tolist()
    fwd_totals, bwd_totals = _run(lq, lq, 1, act="silu")
    assert max(bwd_totals) > 1024  # the coarse buckets are exercised
