#!/usr/bin/env python
"""Benchmark of the jagged attention hot path on GB300.

A step is one forward plus one backward pass of jagged attention over one
batch of synthetic input (default workload: causal softmax self-attention
with a relative-position bias, B=32, lengths ~ U[1,4096] (fill 0.5), H=4,
d=128), run through the C ABI.  The metric is TFLOPS counted on non-padded
work only: forward 4*H*d*sum(unmasked query-key pairs), backward 2.5x that.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdpa|reference]

Prints one JSON line (rank 0).  With N > 1 (torchrun, one rank per GPU) each
rank runs an independent replica on its own seed (the attention has no
exchange step): value = total FLOPs of all ranks / max time over ranks.
`--impl reference` times the fp64 CPU oracle instead (rank 0 only), on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "jagged attn fwd/bwd TFLOPS (non-padded FLOPs) & % of GB300 BF16 tensor peak"
UNIT = "TFLOPS"
BWD_FLOP_FACTOR = 2.5
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic():
    """DRAM bytes per launch from the committed ncu summary, keyed
    "<workload>/<act>/<fwd|bwd>".  An entry is dropped (reported as null) when
    its kernel's source has changed since the counters were taken."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return {}
    csrc = os.path.join(ROOT, "jagged_attention_recsys_02_gb300", "csrc")
    out = {}
    for key, e in d.items():
        if "/" not in key or not isinstance(e, dict):
            continue
        try:
            with open(os.path.join(csrc, e["source"]), "rb") as f:
                h = hashlib.sha256(f.read()).hexdigest()[:16]
        except (OSError, KeyError):
            continue
        if h == e.get("sha256_16"):
            out[key] = e["bytes"]
    return out


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        with open(self.tmp.name) as f:
            lines = [ln.strip() for ln in f if ln.strip()]
        os.unlink(self.tmp.name)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": float(np.median(busy)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ ranks
def reduce_over_ranks(ms, flops, device=None):
    """Max of the timed duration and sum of the work over all ranks (a no-op
    without an initialised process group of more than one rank)."""
    import torch
    import torch.distributed as dist

    if not dist.is_initialized() or dist.get_world_size() == 1:
        return float(ms), float(flops)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    f = torch.tensor([float(flops)], dtype=torch.float64, device=device)
    dist.all_reduce(f, op=dist.ReduceOp.SUM)
    return float(t.item()), float(f.item())


def resolve_steps(args, step, world, device, target_s=1.2, min_steps=20):
    """--steps when given; otherwise enough steps for a timed region of about
    target_s seconds (one warmed-up step timed with CUDA events, the slowest
    rank's estimate shared by all)."""
    if args.steps is not None:
        return args.steps
    import torch

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    step()
    e1.record()
    torch.cuda.synchronize()
    ms, _ = reduce_over_ranks(e0.elapsed_time(e1), 0.0, device)
    return max(min_steps, int(np.ceil(target_s * 1e3 / max(ms, 1e-3))))


# ------------------------------------------------------------------ workload
def workload_flops(w):
    f = w.fwd_flops()
    return f, BWD_FLOP_FACTOR * f


def measure_padded_sdpa(w, t, dev, iters=5, max_gb=40.0):
    """torch's scaled_dot_product_attention, forward + backward, on zero-padded
    [B, H, Lmax, d] copies of the same inputs, on the same GPU, timed with CUDA
    events.  Its TFLOPS count the same non-padded FLOPs as the jagged path.

    Softmax self-attention gets the exact mask (causal and rel-pos bias folded
    into one additive [1, H, Lmax, Lmax] tensor; with equal lengths causality
    also hides every padded key from every real query).  Other workloads run
    mask-free softmax SDPA, a time-only lower bound on the padded cost (torch
    has no fused SiLU/GELU attention and no cheap key-padding mask at Lmax)."""
    import torch
    import torch.nn.functional as F

    B, H, d = w.B, w.H, w.d
    lq_max, lkv_max = int(w.lq.max()), int(w.lkv.max())
    exact = w.act == "softmax" and (w.causal or np.array_equal(w.lq, w.lkv))
    gb = (4 * B * H * lq_max * d + 4 * B * H * lkv_max * d) * 2 / 1e9
    if exact:
        gb += H * lq_max * lkv_max * 2 / 1e9
    if gb > max_gb:
        return {"value": None, "skipped": f"padded copies would need {gb:.0f} GB"}
    qo, ko = w.offsets()

    def pad(x, offs, lmax):
        y = torch.zeros((B, lmax, H, d), device=dev, dtype=x.dtype)
        for b in range(B):
            n = int(offs[b + 1] - offs[b])
            if n:
                y[b, :n] = x[int(offs[b]):int(offs[b + 1])]
        return y.transpose(1, 2).contiguous()

    q = pad(t["q"], qo, lq_max).requires_grad_(True)
    k = pad(t["k"], ko, lkv_max).requires_grad_(True)
    v = pad(t["v"], ko, lkv_max).requires_grad_(True)
    do = pad(t["dout"], qo, lq_max)
    mask = None
    if exact and (w.causal or w.max_rel or w.window or w.block):
        i = torch.arange(lq_max, device=dev)[:, None]
        j = torch.arange(lkv_max, device=dev)[None, :]
        if w.max_rel:
            idx = (i - j + (w.max_rel - 1)).clamp(0, 2 * w.max_rel - 2)
            mask = t["bias"][:, idx].to(torch.bfloat16)[None]
        else:
            mask = torch.zeros((1, H, lq_max, lkv_max), device=dev, dtype=torch.bfloat16)
        if w.causal:
            mask = mask.masked_fill((j > i)[None, None], float("-inf"))
        if w.window:
            mask = mask.masked_fill(((i - j).abs() >= w.window)[None, None], float("-inf"))
        if w.block:
            mask = mask.masked_fill((i // w.block != j // w.block)[None, None], float("-inf"))

    def once():
        o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=w.scale)
        o.backward(do)
        q.grad = k.grad = v.grad = None

    def timed(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / iters

    ms = timed(once)
    fwd, bwd = workload_flops(w)
    # The fastest padded call torch offers for this shape: no additive mask (so
    # the flash / cuDNN kernels run), causal through is_causal, the bias dropped.
    # It computes less than the jagged path (no bias), so it is a lower bound on
    # the padded cost, and the speed-up against it the conservative one.
    lb = None
    if w.act == "softmax" and not w.window and not w.block:
        def fast():
            o = F.scaled_dot_product_attention(q, k, v, is_causal=bool(w.causal), scale=w.scale)
            o.backward(do)
            q.grad = k.grad = v.grad = None

        ms_lb = timed(fast)
        lb = {"value": (fwd + bwd) / (ms_lb * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms_lb,
              "call": f"scaled_dot_product_attention(is_causal={bool(w.causal)}), no attn_mask",
              "note": "lower bound on padded cost: the bias is omitted"}
    return {"value": (fwd + bwd) / (ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms,
            "lower_bound": lb,
            "inputs": f"zero-padded [B={B}, H={H}, Lmax, d={d}] bf16",
            "mask": (" + ".join(x for x, on in (("causal", w.causal),
                                                 (f"window {w.window}", w.window),
                                                 (f"blocks of {w.block}", w.block),
                                                 ("rel-pos bias", w.max_rel)) if on)
                     + " as one additive bf16 mask" if mask is not None else
                     "none (exact for equal lengths without causal)" if exact else
                     "none: mask-free softmax lower bound on padded cost"),
            "steps": iters}


def pick_cpu_sample(w, target_pairs, seed=0):
    """Deterministic subset of samples whose pair count is close to target_pairs."""
    order = np.random.default_rng(seed + 12345).permutation(w.B)
    pairs = w.sample_pairs()
    chosen, tot = [], 0
    for b in order:
        if pairs[b] == 0:
            continue
        if tot > 0 and tot + pairs[b] > target_pairs:
            continue
        chosen.append(int(b))
        tot += int(pairs[b])
        if tot >= 0.9 * target_pairs:
            break
    return sorted(chosen), tot


def oracle_step(w, tensors, samples):
    """One oracle forward + backward over the given samples (host float64)."""
    import oracle

    from jagged_attention_recsys_02_gb300.workloads import ACTS

    qo, ko = w.offsets()
    a = ACTS[w.act]
    bias = tensors.get("bias_np")
    dense = tensors.get("dense_np", {})
    for b in samples:
        q0, q1, k0, k1 = int(qo[b]), int(qo[b + 1]), int(ko[b]), int(ko[b + 1])
        sq = tensors["q_np"][q0:q1]
        sk = tensors["k_np"][k0:k1]
        sv = tensors["v_np"][k0:k1]
        sd = tensors["do_np"][q0:q1]
        oq = np.array([0, q1 - q0], dtype=np.int32)
        ok = np.array([0, k1 - k0], dtype=np.int32)
        kw = dict(act=a, causal=w.causal, scale=w.scale, bias=bias, max_rel=w.max_rel,
                  window=w.window, block=w.block, dense_bias=dense.get(b))
        oracle.fwd(sq, oq, sk, sv, ok, **kw)
        oracle.bwd(sq, oq, sk, sv, ok, sd, **kw)


def host_sample_tensors(w, samples, device_tensors=None, seed=0):
    """float64 host copies of the chosen samples (other rows left zero)."""
    import torch

    out = {}
    if device_tensors is not None:
        src = device_tensors
    else:
        from jagged_attention_recsys_02_gb300.workloads import make_tensors

        src = make_tensors(w, device="cpu", seed=seed)
    qo, ko = w.offsets()
    for name, key, offs in (("q_np", "q", qo), ("do_np", "dout", qo), ("k_np", "k", ko),
                            ("v_np", "v", ko)):
        t = src[key]
        arr = np.zeros(tuple(t.shape), dtype=np.float64)
        for b in samples:
            a0, a1 = int(offs[b]), int(offs[b + 1])
            arr[a0:a1] = t[a0:a1].float().cpu().double().numpy()
        out[name] = arr
    if w.dense:  # the chosen samples' [H][Lq][Lkv] blocks of the dense bias
        vals, off = src["bias"]
        off = off.cpu().numpy()
        out["dense_np"] = {b: vals[int(off[b]):int(off[b + 1])].cpu().double().numpy()
                           for b in samples}
    elif src.get("bias") is not None:
        out["bias_np"] = src["bias"].cpu().double().numpy()
    del torch
    return out


def cpu_cores():
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.isdigit():
        n = min(n, int(env))
    return int(n)


def measure_oracle(w, seconds, device_tensors=None, seed=0):
    """Time the oracle on a bounded sample sized to take about `seconds`.
    Returns (tflops, sample_desc, wall_seconds)."""
    import oracle

    oracle.build()
    # calibrate on a small sample
    cal, cal_pairs = pick_cpu_sample(w, 2e5, seed)
    t_host = host_sample_tensors(w, cal, device_tensors, seed)
    t0 = time.perf_counter()
    oracle_step(w, t_host, cal)
    dt = max(time.perf_counter() - t0, 1e-3)
    rate = cal_pairs / dt
    samples, pairs = pick_cpu_sample(w, max(cal_pairs, rate * seconds), seed)
    t_host = host_sample_tensors(w, samples, device_tensors, seed)
    t0 = time.perf_counter()
    oracle_step(w, t_host, samples)
    dt = time.perf_counter() - t0
    flops = (1.0 + BWD_FLOP_FACTOR) * 4.0 * w.H * w.d * pairs
    desc = (f"{len(samples)} of {w.B} samples ({pairs} of {w.pairs()} non-padded query-key "
            f"pairs), forward + backward, fp64")
    return flops / dt / 1e12, desc, dt


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    from jagged_attention_recsys_02_gb300.workloads import make_workload

    if rank != 0:
        return 0
    w = make_workload(args.workload, act=args.act)
    if args.steps is None:
        args.steps = 20
    budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    import oracle

    oracle.build()
    cal, cal_pairs = pick_cpu_sample(w, 2e5, 0)
    t_host = host_sample_tensors(w, cal, None, 0)
    t0 = time.perf_counter()
    oracle_step(w, t_host, cal)
    rate = cal_pairs / max(time.perf_counter() - t0, 1e-3)
    samples, pairs = pick_cpu_sample(w, max(cal_pairs, rate * budget), 0)
    t_host = host_sample_tensors(w, samples, None, 0)
    for _ in range(args.warmup):
        oracle_step(w, t_host, samples)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, t_host, samples)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    flops = (1.0 + BWD_FLOP_FACTOR) * 4.0 * w.H * w.d * pairs
    value = flops / dt / 1e12
    desc = (f"{len(samples)} of {w.B} samples ({pairs} of {w.pairs()} non-padded query-key "
            f"pairs) per step, forward + backward, fp64")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, "oracle on host cores"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, l2_note, rope_base=0.0):
    extra = {"rope_base": rope_base} if rope_base else {}
    return {**extra, "workload": w.name, "B": w.B, "H": w.H, "d": w.d, "act": w.act,
            "causal": w.causal,
            "window": w.window, "block": w.block,
            "bias": (f"relpos table [{w.H},{2 * w.max_rel - 1}]" if w.max_rel else
                     (f"dense jagged fp32 [{w.H * int((w.lq * w.lkv).sum())}]" if w.dense
                      else "none")),
            "Tq": w.Tq, "Tkv": w.Tkv, "pairs_non_padded": w.pairs(),
            "pairs_full_square": w.full_pairs(), "step": "forward + backward", "l2": l2_note}


# ------------------------------------------------------------------ per-workload lines
# (workload, activation, MXFP8 forward) measured beside the headline workload
PER_WORKLOAD = (("gdpa_cross_gelu", None, False), ("gdpa_pma_silu", None, False),
                ("heavy_tail", "softmax", False), ("heavy_tail", "silu", False),
                ("heavy_tail", "softmax", True))


def algorithmic_bytes(w, mx=False):
    """Bytes a pass must move at least: forward reads q, k, v and writes out
    (plus lse for softmax); backward reads q, k, v, out, dout (plus lse and D)
    and writes dq, dk, dv.  bf16 rows of H*d elements; MXFP8 operands are one
    byte per element plus one scale byte per 32."""
    row = w.H * w.d * 2
    stats = 4 * w.H * w.Tq if w.act == "softmax" else 0
    op = (w.H * w.d * 33 // 32) if mx else row
    fwd = op * (w.Tq + 2 * w.Tkv) + row * w.Tq + stats
    bwd = row * (4 * w.Tq + 4 * w.Tkv) + 2 * stats
    return fwd, bwd


def roofline_for(flops, nbytes, ms, tensor_peak, hbm_gbs):
    """min(tensor peak, arithmetic intensity x HBM bandwidth) and the fraction
    of it reached."""
    achieved = flops / (ms * 1e-3) / 1e12
    bound_hbm = flops / nbytes * hbm_gbs / 1e3
    peak = min(tensor_peak, bound_hbm)
    return {"achieved_tflops": achieved, "roofline_tflops": peak,
            "bound": "tensor" if tensor_peak <= bound_hbm else "hbm",
            "ai_flop_per_byte": flops / nbytes, "algorithmic_bytes": nbytes,
            "frac": achieved / peak}


def measure_workload(name, act, mx, dev, gpu_index, steps, warmup):
    """Forward and backward (MXFP8: quantise + forward) of one workload through
    the C ABI: per-kernel CUDA-event times, TFLOPS on non-padded FLOPs and the
    fraction of the workload's roofline; clocks sampled during the timing."""
    import torch

    from jagged_attention_recsys_02_gb300 import binding
    from jagged_attention_recsys_02_gb300.workloads import ACTS, make_tensors, make_workload

    w = make_workload(name, act=act)
    t = make_tensors(w, device=dev, with_dout=not mx)
    H, d, Tq, Tkv = w.H, w.d, w.Tq, w.Tkv
    out = torch.empty_like(t["q"])
    lse = torch.empty((H, Tq), device=dev, dtype=torch.float32)
    ws_f = torch.empty(binding.fwd_workspace_size(w.B, H, d, Tq, Tkv), device=dev,
                       dtype=torch.uint8)
    kw = dict(act=ACTS[w.act], causal=w.causal, scale=w.scale, bias=t["bias"], max_rel=w.max_rel)
    if mx:
        qc, qs = binding.quantize_mxfp8(t["q"], mode=binding.MX_ALONG_CHANNELS, nosat=True)
        kc, ks = binding.quantize_mxfp8(t["k"], mode=binding.MX_ALONG_CHANNELS, nosat=True)
        vc, vs = binding.quantize_mxfp8(t["v"], t["ko"], mode=binding.MX_ALONG_TOKENS, nosat=True)

        def step():
            binding.quantize_mxfp8(t["q"], mode=binding.MX_ALONG_CHANNELS, nosat=True, codes=qc,
                                   scales=qs)
            binding.quantize_mxfp8(t["k"], mode=binding.MX_ALONG_CHANNELS, nosat=True, codes=kc,
                                   scales=ks)
            binding.quantize_mxfp8(t["v"], t["ko"], mode=binding.MX_ALONG_TOKENS, nosat=True,
                                   codes=vc, scales=vs)
            binding.gdpa_fwd_mxfp8(qc, qs, t["qo"], kc, ks, vc, vs, t["ko"], causal=w.causal,
                                   scale=w.scale, out=out, lse=lse, workspace=ws_f)
    else:
        dq, dk, dv = (torch.empty_like(t[n_]) for n_ in ("q", "k", "v"))
        ws_b = torch.empty(binding.bwd_workspace_size(w.B, H, d, Tq, Tkv), device=dev,
                           dtype=torch.uint8)

        def step():
            binding.gdpa_fwd(t["q"], t["qo"], t["k"], t["v"], t["ko"], out=out, lse=lse,
                             workspace=ws_f, **kw)
            binding.gdpa_bwd(t["q"], t["qo"], t["k"], t["v"], t["ko"], out, lse, t["dout"],
                             dq=dq, dk=dk, dv=dv, workspace=ws_b, **kw)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if binding.device_status() != 0:
        raise RuntimeError(f"device status after warm-up of {name}")
    clocks = ClockSampler(gpu_index)
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    binding.timing_enable(True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    binding.timing_enable(False)
    clk = clocks.stop()
    if binding.device_status() != 0:
        raise RuntimeError(f"device status after timing {name}")
    fwd_ms, bwd_ms = binding.timing_collect()
    peaks, src = load_peaks()
    bf16 = float(peaks["bf16_tflops"])
    hbm = float(peaks["hbm_gbs"])
    fwd_flops, bwd_flops = workload_flops(w)
    fb, bb = algorithmic_bytes(w, mx)
    res = {"config": workload_config(w, "inputs larger than L2 (no flush)"),
           "ms_per_step": e0.elapsed_time(e1) / steps, "steps": steps, "warmup": warmup,
           "clocks": clk, "peaks": f"{src}: bf16 {bf16} TFLOP/s"
                                   f"{' (x2 for FP8)' if mx else ''}, HBM {hbm} GB/s"}
    f_avg = float(np.mean(fwd_ms))
    res["fwd"] = dict(kernel_ms=f_avg, **roofline_for(fwd_flops, fb, f_avg,
                                                      2 * bf16 if mx else bf16, hbm))
    if not mx:
        b_avg = float(np.mean(bwd_ms))
        res["bwd"] = dict(kernel_ms=b_avg, **roofline_for(bwd_flops, bb, b_avg, bf16, hbm))
        res["step_tflops"] = (fwd_flops + bwd_flops) / (res["ms_per_step"] * 1e-3) / 1e12
    else:
        res["step_tflops"] = fwd_flops / (res["ms_per_step"] * 1e-3) / 1e12
        res["config"]["step"] = "MXFP8 quantise Q,K,V (saturation-free scales) + forward"
    return res


# ------------------------------------------------------------------ GPU arm
def run_gpu(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from jagged_attention_recsys_02_gb300 import binding
    from jagged_attention_recsys_02_gb300.workloads import (ACTS, first_samples, make_tensors,
                                                            make_workload)

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=dev)
    binding.load()
    w = make_workload(args.workload, act=args.act)
    if args.samples:
        w = first_samples(w, args.samples)
    skipped = None
    if w.dense:
        # the dense bias (GBs) is an input: an end-to-end step would mostly time its
        # host copy, and the padded SDPA comparison has no mask builder for it
        args.no_e2e = args.no_sdpa = True
        skipped = "dense bias: e2e and padded SDPA not run for this workload"
    t = make_tensors(w, device=dev, seed=rank)
    a = ACTS[w.act]
    H, d, Tq, Tkv = w.H, w.d, w.Tq, w.Tkv
    out = torch.empty_like(t["q"])
    lse = torch.empty((H, Tq), device=dev, dtype=torch.float32)
    dq = torch.empty_like(t["q"])
    dk = torch.empty_like(t["k"])
    dv = torch.empty_like(t["v"])
    ws_f = torch.empty(binding.fwd_workspace_size(w.B, H, d, Tq, Tkv), device=dev, dtype=torch.uint8)
    ws_b = torch.empty(binding.bwd_workspace_size(w.B, H, d, Tq, Tkv), device=dev, dtype=torch.uint8)
    kw = dict(act=a, causal=w.causal, scale=w.scale, bias=t["bias"], max_rel=w.max_rel,
              window=w.window)
    fwd_flops, bwd_flops = workload_flops(w)
    if w.block:
        # block-aligned attention: its own entry points (no lse, no D pass)
        ws_k = torch.empty(binding.block_workspace_size(w.B, H, d, Tq), device=dev,
                           dtype=torch.uint8)
        kw.pop("window")

    def run_fwd(q, qo, k, v, ko, out_, lse_, **kw_):
        if w.block:
            binding.gdpa_block_fwd(q, qo, k, v, out=out_, workspace=ws_k, **kw_)
        else:
            binding.gdpa_fwd(q, qo, k, v, ko, out=out_, lse=lse_, workspace=ws_f, **kw_)

    def run_bwd(q, qo, k, v, ko, out_, lse_, do, dq_, dk_, dv_, **kw_):
        if args.rope_base:  # q and k taken as rotary-embedded: the fused rotary backward
            kw_ = dict(kw_, rope_base=args.rope_base)
        if w.block:
            binding.gdpa_block_bwd(q, qo, k, v, do, dq=dq_, dk=dk_, dv=dv_, workspace=ws_k, **kw_)
        else:
            binding.gdpa_bwd(q, qo, k, v, ko, out_, lse_, do, dq=dq_, dk=dk_, dv=dv_,
                             workspace=ws_b, **kw_)

    def step(q, qo, k, v, ko, do):
        run_fwd(q, qo, k, v, ko, out, lse, **kw)
        n = binding.last_launch_count()
        run_bwd(q, qo, k, v, ko, out, lse, do, dq, dk, dv, **kw)
        return n + binding.last_launch_count()

    args_dev = (t["q"], t["qo"], t["k"], t["v"], t["ko"], t["dout"])
    for _ in range(args.warmup):
        step(*args_dev)
    torch.cuda.synchronize()
    st = binding.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")
    args.steps = resolve_steps(args, lambda: step(*args_dev), world, dev)

    clocks = ClockSampler(local_rank)
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    binding.timing_enable(True)
    launches = 0
    e0.record()
    for _ in range(args.steps):
        launches += step(*args_dev)
    e1.record()
    torch.cuda.synchronize()
    binding.timing_enable(False)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    fwd_ms, bwd_ms = binding.timing_collect()
    st = binding.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region")

    # max time over ranks, total FLOPs over ranks
    ms, tot_flops = reduce_over_ranks(ms, (fwd_flops + bwd_flops) * args.steps, dev)
    value = tot_flops / (ms * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    region_s = ms * 1e-3
    sustained = region_s > 2.0
    peak = float(peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"])
    f_avg = float(np.mean(fwd_ms)) if fwd_ms else float("nan")
    b_avg = float(np.mean(bwd_ms)) if bwd_ms else float("nan")
    f_tf = fwd_flops / (f_avg * 1e-3) / 1e12
    b_tf = bwd_flops / (b_avg * 1e-3) / 1e12
    dominant = "bwd" if sum(bwd_ms) >= sum(fwd_ms) else "fwd"
    achieved = b_tf if dominant == "bwd" else f_tf
    traffic = load_traffic().get(f"{w.name}/{w.act}/{dominant}")
    hbm = None
    if w.dense:
        # bound by reading the dense bias: algorithmic bytes are the bias (fp32,
        # once per pass) plus q, k, v read and out written (forward) or q, k, v,
        # out, dO read and dq, dk, dv written (backward), bf16
        row_bytes = H * d * 2
        bias_bytes = int(t["bias"][0].numel()) * 4
        f_bytes = bias_bytes + 4 * Tq * row_bytes
        b_bytes = bias_bytes + 8 * Tq * row_bytes
        hbm = {"fwd_gbs": f_bytes / (f_avg * 1e-3) / 1e9, "bwd_gbs": b_bytes / (b_avg * 1e-3) / 1e9,
               "fwd_bytes": f_bytes, "bwd_bytes": b_bytes}
    if w.block:
        # 64 x 64 problems are bound by HBM traffic: algorithmic bytes are q, k, v
        # read and out written once (forward), q, k, v, dO read and dq, dk, dv
        # written once (backward), bf16
        row_bytes = H * d * 2
        f_bytes, b_bytes = 4 * Tq * row_bytes, 7 * Tq * row_bytes
        hbm = {"fwd_gbs": f_bytes / (f_avg * 1e-3) / 1e9, "bwd_gbs": b_bytes / (b_avg * 1e-3) / 1e9,
               "fwd_bytes": f_bytes, "bwd_bytes": b_bytes}

    # ---------------- end to end through host buffers
    # Every step copies its inputs from pinned host memory, runs forward and
    # backward, and copies its outputs back.  Steps are pipelined over two
    # buffer slots on three streams (host->device, compute, device->host), so
    # the copies of one step overlap the compute of its neighbours.
    e2e = None
    if not args.no_e2e:
        names_in = ("q", "k", "v", "dout", "qo", "ko")
        pin = {k_: t[k_].cpu().pin_memory() for k_ in names_in}
        hbias = t["bias"].cpu().pin_memory() if t["bias"] is not None else None
        outs = [dict(out=torch.empty_like(out), lse=torch.empty_like(lse), dq=torch.empty_like(dq),
                     dk=torch.empty_like(dk), dv=torch.empty_like(dv)) for _ in range(2)]
        if w.block:  # the block forward writes no logsumexp
            for o_ in outs:
                del o_["lse"]
        host_out = [{k_: torch.empty(tuple(x.shape), dtype=x.dtype, pin_memory=True)
                     for k_, x in o.items()} for o in outs]
        dev_in = [{k_: torch.empty_like(t[k_]) for k_ in names_in} for _ in range(2)]
        dbias = [torch.empty_like(t["bias"]) if hbias is not None else None for _ in range(2)]
        h2d = sum(x.numel() * x.element_size() for x in pin.values())
        h2d += hbias.numel() * hbias.element_size() if hbias is not None else 0
        d2h = sum(x.numel() * x.element_size() for x in host_out[0].values())
        s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_cmp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        for sl in range(2):  # nothing pending on either slot yet
            for ev in (ev_cmp[sl], ev_out[sl]):
                ev.record(torch.cuda.current_stream(dev))

        def e2e_step(k_step):
            sl = k_step % 2
            di, o, ho = dev_in[sl], outs[sl], host_out[sl]
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_cmp[sl])  # the compute two steps back read this slot
                for k_, x in pin.items():
                    di[k_].copy_(x, non_blocking=True)
                if hbias is not None:
                    dbias[sl].copy_(hbias, non_blocking=True)
                ev_in[sl].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[sl])
                s_cmp.wait_event(ev_out[sl])  # outputs of two steps back have been read
                kw_e = dict(kw, bias=dbias[sl], stream=s_cmp)
                run_fwd(di["q"], di["qo"], di["k"], di["v"], di["ko"], o["out"], o.get("lse"),
                        **kw_e)
                run_bwd(di["q"], di["qo"], di["k"], di["v"], di["ko"], o["out"], o.get("lse"),
                        di["dout"], o["dq"], o["dk"], o["dv"], **kw_e)
                ev_cmp[sl].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[sl])
                for k_, x in o.items():
                    ho[k_].copy_(x, non_blocking=True)
                ev_out[sl].record(s_out)

        for k_step in range(2):
            e2e_step(k_step)
        torch.cuda.synchronize()
        n_e2e = max(4, args.steps // 2)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        main = torch.cuda.current_stream(dev)
        e0.record(main)
        for st_ in (s_in, s_cmp, s_out):
            st_.wait_event(e0)
        for k_step in range(n_e2e):
            e2e_step(k_step)
        for st_ in (s_in, s_cmp, s_out):
            done = torch.cuda.Event()
            done.record(st_)
            main.wait_event(done)
        e1.record(main)
        torch.cuda.synchronize()
        st = binding.device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} after the end-to-end steps")
        ms_e, _ = reduce_over_ranks(e0.elapsed_time(e1), 0.0, dev)
        e2e = {"value": tot_flops / args.steps * n_e2e / (ms_e * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": ms_e / n_e2e, "steps": n_e2e,
               "pipeline": "2 buffer slots; host->device, compute and device->host streams"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, desc, secs = measure_oracle(w, args.cpu_seconds, device_tensors=t, seed=rank)
        cpu = {"value": tf, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": desc,
               "seconds": secs}

    # Sliding window: the same step without the window on the same inputs (the
    # full causal attention the window replaces), for the latency reduction.
    swa = None
    if rank == 0 and world == 1 and w.window > 0:
        kw_full = dict(kw, window=0)

        def step_full():
            binding.gdpa_fwd(*args_dev[:5], out=out, lse=lse, workspace=ws_f, **kw_full)
            binding.gdpa_bwd(*args_dev, out, lse, dq=dq, dk=dk, dv=dv, workspace=ws_b, **kw_full)

        for _ in range(2):
            step_full()
        n_full = max(3, args.steps // 4)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n_full):
            step_full()
        e1.record()
        torch.cuda.synchronize()
        if binding.device_status() != 0:
            raise RuntimeError("device status after the full-attention comparison")
        full_ms = e0.elapsed_time(e1) / n_full
        swa = {"window": w.window, "swa_ms_per_step": ms / args.steps,
               "full_causal_ms_per_step": full_ms,
               "latency_reduction": 1.0 - (ms / args.steps) / full_ms, "full_steps": n_full}

    sdpa = None
    if rank == 0 and world == 1 and not args.no_sdpa:
        sdpa = measure_padded_sdpa(w, t, dev)
        if sdpa.get("value"):
            sdpa["jagged_over_padded"] = value / sdpa["value"]
        if sdpa.get("lower_bound"):
            sdpa["jagged_over_padded_lower_bound"] = value / sdpa["lower_bound"]["value"]


    in_bytes = sum(x.numel() * x.element_size() for x in (t["q"], t["k"], t["v"], t["dout"]))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 inputs, lengths per workload recipe)",
        "config": workload_config(
            w, f"inputs larger than L2: {in_bytes / 2**20:.0f} MiB of q,k,v,dO per step "
               f"(no flush)", args.rope_base),
        "pct_of_peak": {"value": 100.0 * value / peak, "peak_tflops": peak,
                        "peak": ("bf16_tflops_sustained" if sustained else "bf16_tflops")
                        + f" of {peak_src}"},
        "fwd": {"tflops": f_tf, "kernel_ms": f_avg, "flops_per_launch": fwd_flops},
        "bwd": {"tflops": b_tf, "kernel_ms": b_avg, "flops_per_launch": bwd_flops},
        "roofline": ({"bound": "tensor", "kernel": f"{dominant} main kernel",
                      "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                      "frac": achieved / peak, "traffic": traffic,
                      "peak_source": ("bf16_tflops_sustained" if sustained else "bf16_tflops")
                      + f" of {peak_src}"} if hbm is None else
                     {"bound": "hbm",
                      "kernel": f"{'dense-bias' if w.dense else 'block'} {dominant} kernel",
                      "achieved": hbm[f"{dominant}_gbs"], "peak": float(peaks["hbm_gbs"]),
                      "unit": "GB/s", "frac": hbm[f"{dominant}_gbs"] / float(peaks["hbm_gbs"]),
                      "traffic": traffic, "algorithmic_bytes": hbm[f"{dominant}_bytes"],
                      "peak_source": f"hbm_gbs of {peak_src}"}),
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": e2e,
        "hbm": hbm,
        **({"skipped": skipped} if skipped else {}),
        "cpu_baseline": cpu,
        "padded_sdpa": sdpa,
    }
    # Every other configuration of the benchmark suite, timed on the same GPU
    # in the same run (default workload only, one GPU).
    if rank == 0 and world == 1 and args.per_workload:
        del t, args_dev
        torch.cuda.empty_cache()
        per_workload = {}
        for name, act, mx in PER_WORKLOAD:
            per_workload[f"{name}/{'mxfp8' if mx else act}"] = measure_workload(
                name, act, mx, dev, local_rank, steps=5, warmup=3)
            torch.cuda.empty_cache()
        line["per_workload"] = per_workload
    if swa is not None:
        line["swa_vs_full"] = swa
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ MXFP8 forward
def run_gpu_mxfp8(args, rank, world, local_rank):
    """Forward on MXFP8 operands: a step quantises Q, K, V (E4M3 + E8M0 block
    scales) and runs the block-scaled forward (softmax); with --mxfp8-bwd the
    step also runs the MXFP8 backward (which quantises Q, K, V, dO itself).
    FLOPs are the non-padded 4*H*d*pairs forward (2.5x that for the backward);
    the peak is the FP8 one (2x the measured bf16 peak, the nominal FP8 : BF16
    ratio of the part)."""
    import torch
    import torch.distributed as dist

    from jagged_attention_recsys_02_gb300 import binding
    from jagged_attention_recsys_02_gb300.workloads import first_samples, make_tensors, make_workload

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=dev)
    w = make_workload(args.workload or "heavy_tail", act="softmax")
    if args.samples:
        w = first_samples(w, args.samples)
    train = args.mxfp8_bwd
    t = make_tensors(w, device=dev, seed=rank, with_dout=train)
    H, d, Tq, Tkv = w.H, w.d, w.Tq, w.Tkv
    out = torch.empty_like(t["q"])
    lse = torch.empty((H, Tq), device=dev, dtype=torch.float32)
    ws = torch.empty(binding.fwd_workspace_size(w.B, H, d, Tq, Tkv), device=dev, dtype=torch.uint8)
    if train:
        ws_b = torch.empty(binding.bwd_mxfp8_workspace_size(w.B, H, d, Tq, Tkv), device=dev,
                           dtype=torch.uint8)
        dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
    # the saturation-free block scale (GDPA_MX_NOSAT), the recipe the forward is tested with
    qc, qs = binding.quantize_mxfp8(t["q"], mode=binding.MX_ALONG_CHANNELS, nosat=True)
    kc, ks = binding.quantize_mxfp8(t["k"], mode=binding.MX_ALONG_CHANNELS, nosat=True)
    vc, vs = binding.quantize_mxfp8(t["v"], t["ko"], mode=binding.MX_ALONG_TOKENS, nosat=True)

    def step():
        n = 0
        binding.quantize_mxfp8(t["q"], mode=binding.MX_ALONG_CHANNELS, nosat=True, codes=qc,
                               scales=qs)
        n += binding.last_launch_count()
        binding.quantize_mxfp8(t["k"], mode=binding.MX_ALONG_CHANNELS, nosat=True, codes=kc,
                               scales=ks)
        n += binding.last_launch_count()
        binding.quantize_mxfp8(t["v"], t["ko"], mode=binding.MX_ALONG_TOKENS, nosat=True, codes=vc,
                               scales=vs)
        n += binding.last_launch_count()
        binding.gdpa_fwd_mxfp8(qc, qs, t["qo"], kc, ks, vc, vs, t["ko"], causal=w.causal,
                               scale=w.scale, bias=t["bias"], max_rel=w.max_rel, window=w.window,
                               out=out, lse=lse, workspace=ws)
        n += binding.last_launch_count()
        if train:
            binding.gdpa_bwd_mxfp8(t["q"], t["qo"], t["k"], t["v"], t["ko"], out, lse, t["dout"],
                                   causal=w.causal, scale=w.scale, bias=t["bias"],
                                   max_rel=w.max_rel, window=w.window, dq=dq, dk=dk, dv=dv,
                                   workspace=ws_b)
            n += binding.last_launch_count()
        return n

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if binding.device_status() != 0:
        raise RuntimeError("device status after warm-up")
    args.steps = resolve_steps(args, step, world, dev)
    clocks = ClockSampler(local_rank)
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    binding.timing_enable(True)
    launches = 0
    e0.record()
    for _ in range(args.steps):
        launches += step()
    e1.record()
    torch.cuda.synchronize()
    binding.timing_enable(False)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    fwd_ms, bwd_ms = binding.timing_collect()
    fwd_flops = w.fwd_flops()
    bwd_flops = 2.5 * fwd_flops if train else 0.0
    flops = fwd_flops + bwd_flops
    ms, tot = reduce_over_ranks(e0.elapsed_time(e1), flops * args.steps, dev)
    value = tot / (ms * 1e-3) / 1e12
    peaks, src = load_peaks()
    fp8_peak = 2.0 * float(peaks["bf16_tflops"])
    f_ms = float(np.mean(fwd_ms))
    kernels = {"fwd": {"tflops": fwd_flops / (f_ms * 1e-3) / 1e12, "kernel_ms": f_ms,
                       "flops_per_launch": fwd_flops}}
    if train:
        b_ms = float(np.mean(bwd_ms))
        kernels["bwd"] = {"tflops": bwd_flops / (b_ms * 1e-3) / 1e12, "kernel_ms": b_ms,
                          "flops_per_launch": bwd_flops}
    # the dominant kernel: the one with the larger share of the step
    dom = "bwd" if train and kernels["bwd"]["kernel_ms"] > f_ms else "fwd"
    achieved = kernels[dom]["tflops"]
    line = {
        "metric": ("jagged attn MXFP8 fwd+bwd TFLOPS (non-padded FLOPs) & % of GB300 FP8 tensor peak"
                   if train else
                   "jagged attn MXFP8 fwd TFLOPS (non-padded FLOPs) & % of GB300 FP8 tensor peak"),
        "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (E8M0 block scales), fp32 accumulate",
        "data": "synthetic (seeded N(0,1) bf16 inputs, quantised every step)",
        "config": dict(workload_config(w, "inputs larger than L2 (no flush)"),
                       step=("MXFP8 quantise Q,K,V + forward + backward (quantise Q,K,V,dO inside)"
                             if train else "MXFP8 quantise Q,K,V + forward")),
        **kernels,
        "roofline": {"bound": "tensor",
                     "kernel": "MXFP8 backward kernel" if dom == "bwd" else "MXFP8 forward kernel",
                     "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": achieved / fp8_peak,
                     "traffic": load_traffic().get(f"{w.name}/mxfp8/{dom}"),
                     "peak_source": f"2 x bf16_tflops of {src} (nominal FP8:BF16 = 2)"},
        "gpu_launches": launches, "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for a timed region of about 1.2 s)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gdpa", choices=["gdpa", "reference"])
    ap.add_argument("--workload", default=None,
                    help="default: jfa_causal_relpos (heavy_tail with --mxfp8)")
    ap.add_argument("--act", default=None, help="override the workload's activation")
    ap.add_argument("--samples", type=int, default=0,
                    help="keep only the workload's first N samples (small profiler captures; "
                         "not a benchmark configuration)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sdpa", action="store_true",
                    help="skip the padded torch SDPA comparison")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-per-workload", dest="per_workload", action="store_false",
                    help="skip the other configurations' forward / backward lines")
    ap.add_argument("--rope-base", type=float, default=0.0,
                    help="run the backward with the fused rotary-embedding backward (q, k taken "
                         "as rotary-embedded with this base)")
    ap.add_argument("--mxfp8", action="store_true",
                    help="time the MXFP8 forward path (quantise + block-scaled forward) instead")
    ap.add_argument("--mxfp8-bwd", action="store_true",
                    help="time the MXFP8 training step (forward + backward, all block-scaled)")
    args = ap.parse_args()
    args.mxfp8 = args.mxfp8 or args.mxfp8_bwd
    # the other configurations are measured beside the default workload only
    args.per_workload = args.per_workload and args.workload is None and not args.samples
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        args.workload = args.workload or "jfa_causal_relpos"
        return run_reference(args, rank, world)
    if args.mxfp8:
        return run_gpu_mxfp8(args, rank, world, local_rank)
    args.workload = args.workload or "jfa_causal_relpos"
    return run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
