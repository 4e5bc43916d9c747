"""Host-side logic that needs no GPU: the seeded workload recipes and the
benchmark's aggregation over ranks (world_size 2 over gloo on CPU)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from jagged_attention_recsys_02_gb300.workloads import (CONFIG_NAMES, custom_workload, make_tensors,
                                                        make_workload)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("causal", [False, True])
def test_window_pair_counts_match_the_mask(causal):
    """Non-padded pair counts of sliding-window workloads (the FLOP count of
    every windowed measurement) equal the number of kept entries of the band
    mask |i - j| < W (and j <= i when causal), counted by brute force."""
    lengths = [0, 1, 2, 5, 64, 129, 300]
    for W in (1, 2, 7, 128, 400):
        w = custom_workload(lengths, lengths, 1, 64, causal=causal, window=W)
        for L, got in zip(lengths, w.sample_pairs()):
            i, j = np.arange(L)[:, None], np.arange(L)[None, :]
            keep = np.abs(i - j) < W
            if causal:
                keep &= j <= i
            assert got == keep.sum(), (L, W, causal)
    w = make_workload("swa_causal_relpos")
    assert w.window == 1024 and w.causal and w.max_rel == 1024 and w.B == 64
    assert w.pairs() < int(np.sum(w.lq * (w.lq + 1) // 2))


@pytest.mark.parametrize("causal", [False, True])
def test_block_and_plain_pair_counts_match_the_mask(causal):
    """Non-padded pair counts (the FLOP count of every measurement) for block
    attention, plain causal and asymmetric non-causal workloads against brute
    force over the mask; forward FLOPs are 4 H d per pair."""
    lengths = [0, 1, 2, 5, 63, 64, 65, 200]
    for K in (1, 3, 64):
        w = custom_workload(lengths, lengths, 1, 64, causal=causal, block=K)
        for L, got in zip(lengths, w.sample_pairs()):
            i, j = np.arange(L)[:, None], np.arange(L)[None, :]
            keep = (i // K) == (j // K)
            if causal:
                keep &= j <= i
            assert got == keep.sum(), (L, K, causal)
    lkv = lengths if causal else [3, 0, 9, 5, 1, 64, 2, 7]
    w = custom_workload(lengths, lkv, 2, 128, causal=causal)
    brute = sum(int(((np.arange(a)[:, None] >= np.arange(b)[None, :]) if causal
                     else np.ones((a, b), bool)).sum()) for a, b in zip(lengths, lkv))
    assert w.pairs() == brute and w.fwd_flops() == 4.0 * 2 * 128 * brute


def test_workload_recipes():
    w = make_workload("tiny_silu")
    assert list(w.lq) == [1, 7, 33, 64] and (w.H, w.d, w.act) == (2, 64, "silu")
    w = make_workload("jfa_causal_relpos")
    assert w.B == 32 and w.causal and w.max_rel == 4096 and np.array_equal(w.lq, w.lkv)
    assert w.lq.min() >= 1 and w.lq.max() <= 4096
    assert w.pairs() == int(np.sum(w.lq * (w.lq + 1) // 2))
    w = make_workload("gdpa_cross_gelu")
    assert w.lq.min() >= 64 and w.lq.max() <= 8192 and w.lkv.min() >= 32 and w.lkv.max() <= 256
    w = make_workload("gdpa_pma_silu")
    assert np.all(w.lq == 32) and w.pma_seeds == 32 and w.H == 8
    assert w.lkv.min() >= 16 and w.lkv.max() <= 16384
    w = make_workload("heavy_tail")
    assert w.B == 1024 and w.lq.min() >= 16 and w.lq.max() <= 16384
    # log-normal around 1024: the median sits near 1024
    assert 700 < np.median(w.lq) < 1400


def test_workloads_are_seeded():
    for name in CONFIG_NAMES:
        a, b = make_workload(name, seed=0), make_workload(name, seed=0)
        assert np.array_equal(a.lq, b.lq) and np.array_equal(a.lkv, b.lkv)
    assert not np.array_equal(make_workload("heavy_tail", seed=0).lq,
                              make_workload("heavy_tail", seed=1).lq)


def test_tensors_shapes_and_pma_sharing():
    w = make_workload("tiny_silu")
    t = make_tensors(w, device="cpu")
    assert t["q"].shape == (105, 2, 64) and t["q"].dtype == torch.bfloat16
    assert t["qo"].tolist() == [0, 1, 8, 41, 105]
    t2 = make_tensors(w, device="cpu")
    assert torch.equal(t["q"], t2["q"]) and torch.equal(t["dout"], t2["dout"])
    w = make_workload("gdpa_pma_silu")
    w.lkv = np.full(w.B, 16)  # shrink for the test
    t = make_tensors(w, device="cpu", with_dout=False)
    q = t["q"].view(w.B, 32, w.H, w.d)
    assert torch.equal(q[0], q[-1])  # seed queries are shared by every sample


def test_dense_bias_workload_layout():
    """jfa_causal_dense: jfa_causal_relpos's lengths, no table, and a dense bias
    whose per-sample blocks step by H * Lq * Lkv (checked on two samples)."""
    from jagged_attention_recsys_02_gb300.workloads import first_samples

    a, w = make_workload("jfa_causal_relpos"), make_workload("jfa_causal_dense")
    assert np.array_equal(a.lq, w.lq) and w.dense and w.max_rel == 0 and w.causal
    w2 = first_samples(w, 2)
    w2.lq = w2.lkv = np.array([3, 5])
    t = make_tensors(w2, device="cpu")
    vals, off = t["bias"]
    assert off.tolist() == [0, 4 * 9, 4 * 9 + 4 * 25] and vals.numel() == off[-1]
    assert vals.dtype == torch.float32 and float(vals.std()) < 0.1


def test_reference_arm_line_on_a_tiny_workload():
    """bench.py --impl reference prints one JSON line with the contract's keys
    (the oracle on the host cores; runs here, no GPU)."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_silu", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


_WORKER = r'''
import os, sys, json
sys.path.insert(0, sys.argv[1])
import torch.distributed as dist
import bench
rank = int(sys.argv[2])
dist.init_process_group("gloo", init_method="tcp://127.0.0.1:" + sys.argv[3], rank=rank,
                        world_size=2)
ms, flops = bench.reduce_over_ranks(1.5 + rank, 10.0 * (rank + 1))
print(json.dumps({"rank": rank, "ms": ms, "flops": flops}))
dist.destroy_process_group()
'''


def test_reduce_over_ranks_gloo_world2(tmp_path):
    import socket

    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    script = tmp_path / "worker.py"
    script.write_text(_WORKER)
    procs = [subprocess.Popen([sys.executable, str(script), ROOT, str(r), str(port)],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    res = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
    for r in res:
        assert r["ms"] == 2.5 and r["flops"] == 30.0


def test_reduce_over_ranks_single_process():
    import bench

    assert bench.reduce_over_ranks(3.0, 7.0) == (3.0, 7.0)


def test_traffic_table_is_well_formed():
    """profiles/dram_traffic.json: every entry names an existing kernel source
    and a 16-hex-digit hash prefix; the benchmark reports an entry only while
    that source is unchanged."""
    sys.path.insert(0, ROOT)
    import bench

    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        table = json.load(f)
    csrc = os.path.join(ROOT, "jagged_attention_recsys_02_gb300", "csrc")
    for key, e in table.items():
        if "/" not in key:
            continue
        assert os.path.exists(os.path.join(csrc, e["source"])), key
        assert len(e["sha256_16"]) == 16 and int(e["sha256_16"], 16) >= 0, key
        assert e["bytes"] > 0, key
    valid = bench.load_traffic()
    assert set(valid) <= set(table)
    assert all(valid[k] == table[k]["bytes"] for k in valid)


def test_roofline_arithmetic_of_the_per_workload_lines():
    """The per-workload roofline: algorithmic bytes counted from the tensors a
    pass must read and write, and min(tensor peak, intensity x HBM)."""
    sys.path.insert(0, ROOT)
    import bench

    w = make_workload("gdpa_pma_silu")
    row = w.H * w.d * 2
    f, b = bench.algorithmic_bytes(w)
    assert f == row * (2 * w.Tq + 2 * w.Tkv)               # q, k, v read; out written
    assert b == row * (4 * w.Tq + 4 * w.Tkv)               # q, k, v, out, dout; dq, dk, dv
    ws = make_workload("jfa_causal_relpos")
    f2, b2 = bench.algorithmic_bytes(ws)
    assert f2 == ws.H * ws.d * 2 * 4 * ws.Tq + 4 * ws.H * ws.Tq   # + lse
    fm, _ = bench.algorithmic_bytes(ws, mx=True)
    assert fm < f2                                          # one-byte operands
    # HBM-bound: 1e12 FLOP over 1e10 bytes at 1000 GB/s -> 100 TFLOP/s ceiling
    r = bench.roofline_for(1e12, 1e10, 20.0, tensor_peak=2000.0, hbm_gbs=1000.0)
    assert r["bound"] == "hbm" and abs(r["roofline_tflops"] - 100.0) < 1e-9
    assert abs(r["achieved_tflops"] - 50.0) < 1e-9 and abs(r["frac"] - 0.5) < 1e-12
    r = bench.roofline_for(1e12, 1e8, 1.0, tensor_peak=2000.0, hbm_gbs=1000.0)
    assert r["bound"] == "tensor" and r["roofline_tflops"] == 2000.0
