"""Seeded synthetic jagged-attention workloads.

This module only draws inputs; it holds none of the attention arithmetic.
Both the CUDA path (tests, benchmark) and the fp64 oracle are fed from it.

Sequence lengths come from ``numpy.random.default_rng(seed)``; tensor values
from ``torch.Generator(device).manual_seed(seed + 1)`` in float32, rounded to
bf16, drawn in the fixed order q, k, v, dout, bias.  The pages ("GEM
Training ..." JFA paragraph) describe production sequences only as jagged,
"varying from hundreds to tens of thousands of tokens per sample", at
sparsity 0.5; these workloads stand in for that traffic:

  tiny_silu          B=4, q=kv lengths {1,7,33,64}, H=2, d=64, SiLU
  jfa_causal_relpos  B=32, L~U[1,4096], H=4, d=128, softmax, causal,
                     per-head relative-position bias table [H, 8191] ~ N(0, 0.02)
  gdpa_cross_gelu    B=256, Lq~U[64,8192], Lkv~U[32,256], H=4, d=128, GELU(tanh)
  gdpa_pma_silu      32 shared seed queries, B=512, Lkv~U[16,16384], H=8,
                     d=128, SiLU (queries expanded to [B*32, H, d])
  heavy_tail         B=1024, L=round(exp(N(ln 1024, 1))) clipped to [16,16384],
                     H=4, d=128, softmax or SiLU
  swa_causal_relpos  sliding-window self-attention over long sequences ("GEM
                     Training ..." SWA paragraph): B=64, L~U[1,16384], H=4,
                     d=128, softmax, causal, window 1024, relative-position
                     bias table [H, 2047] ~ N(0, 0.02)
  block_relpos       block-aligned attention over the same long sequences
                     (same paragraph): B=64, L~U[1,16384], H=4, d=128,
                     softmax, 64-token blocks, relative-position bias table
                     [H, 127] ~ N(0, 0.02)
  jfa_causal_dense   jfa_causal_relpos's lengths and settings with a dense
                     jagged bias instead of the table: one fp32 value
                     ~ N(0, 0.02) per (head, query, key) of each sample
                     (the JFA paragraph's custom biases in general form)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

ACTS = {"softmax": 0, "silu": 1, "gelu_tanh": 2, "identity": 3, "gelu_erf": 4}

CONFIG_NAMES = ("tiny_silu", "jfa_causal_relpos", "gdpa_cross_gelu", "gdpa_pma_silu", "heavy_tail")
EXTRA_NAMES = ("swa_causal_relpos", "block_relpos", "jfa_causal_dense")


@dataclass
class Workload:
    name: str
    B: int
    H: int
    d: int
    act: str
    causal: bool
    lq: np.ndarray            # int64 [B]
    lkv: np.ndarray           # int64 [B]
    max_rel: int = 0          # >0: relative-position bias table [H, 2*max_rel-1]
    pma_seeds: int = 0        # >0: queries are this many seeds shared by all samples
    window: int = 0           # >0: sliding window, pairs with |i - j| < window
    block: int = 0            # >0: block-aligned attention in blocks of this many tokens
    dense: bool = False       # dense jagged bias [sum_b H*Lq_b*Lkv_b] instead of a table
    scale: float = 0.0
    extra: dict = field(default_factory=dict)

    @property
    def Tq(self) -> int:
        return int(self.lq.sum())

    @property
    def Tkv(self) -> int:
        return int(self.lkv.sum())

    def offsets(self):
        qo = np.zeros(self.B + 1, dtype=np.int32)
        ko = np.zeros(self.B + 1, dtype=np.int32)
        qo[1:] = np.cumsum(self.lq)
        ko[1:] = np.cumsum(self.lkv)
        return qo, ko

    def sample_pairs(self) -> np.ndarray:
        """Per-sample query-key pairs that are not masked (int64 [B])."""
        L, W = self.lq, self.window
        if self.block > 0:
            K = self.block
            full, rest = L // K, L % K
            per = (lambda n: n * (n + 1) // 2) if self.causal else (lambda n: n * n)
            return full * per(K) + per(rest)
        if W <= 0:
            return self.lq * (self.lq + 1) // 2 if self.causal else self.lq * self.lkv
        # causal window: row i sees min(i + 1, W) keys
        m = np.minimum(L, W)
        causal = m * (m + 1) // 2 + (L - m) * W
        if self.causal:
            return causal
        # symmetric window: add the keys ahead of each row, min(L - 1 - i, W - 1)
        return causal + causal - L

    def pairs(self) -> int:
        """Query-key pairs that are not masked (the non-padded work)."""
        return int(np.sum(self.sample_pairs()))

    def full_pairs(self) -> int:
        return int(np.sum(self.lq * self.lkv))

    def fwd_flops(self) -> float:
        return 4.0 * self.H * self.d * self.pairs()


def make_workload(name: str, seed: int = 0, act: str | None = None) -> Workload:
    rng = np.random.default_rng(seed)
    if name == "tiny_silu":
        L = np.array([1, 7, 33, 64], dtype=np.int64)
        w = Workload(name, 4, 2, 64, "silu", False, L.copy(), L.copy())
    elif name in ("jfa_causal_relpos", "jfa_causal_dense"):
        L = rng.integers(1, 4096, size=32, endpoint=True).astype(np.int64)
        dense = name == "jfa_causal_dense"
        w = Workload(name, 32, 4, 128, "softmax", True, L.copy(), L.copy(),
                     max_rel=0 if dense else 4096, dense=dense)
    elif name == "gdpa_cross_gelu":
        lq = rng.integers(64, 8192, size=256, endpoint=True).astype(np.int64)
        lkv = rng.integers(32, 256, size=256, endpoint=True).astype(np.int64)
        w = Workload(name, 256, 4, 128, "gelu_tanh", False, lq, lkv)
    elif name == "gdpa_pma_silu":
        lkv = rng.integers(16, 16384, size=512, endpoint=True).astype(np.int64)
        w = Workload(name, 512, 8, 128, "silu", False, np.full(512, 32, dtype=np.int64), lkv,
                     pma_seeds=32)
    elif name == "heavy_tail":
        x = np.exp(rng.normal(math.log(1024.0), 1.0, size=1024))
        L = np.clip(np.round(x), 16, 16384).astype(np.int64)
        w = Workload(name, 1024, 4, 128, "softmax", False, L.copy(), L.copy())
    elif name == "swa_causal_relpos":
        L = rng.integers(1, 16384, size=64, endpoint=True).astype(np.int64)
        w = Workload(name, 64, 4, 128, "softmax", True, L.copy(), L.copy(), max_rel=1024,
                     window=1024)
    elif name == "block_relpos":
        L = rng.integers(1, 16384, size=64, endpoint=True).astype(np.int64)
        w = Workload(name, 64, 4, 128, "softmax", False, L.copy(), L.copy(), max_rel=64,
                     block=64)
    else:
        raise KeyError(name)
    if act is not None:
        w.act = act
    w.scale = 1.0 / math.sqrt(w.d)
    return w


def first_samples(w: Workload, n: int) -> Workload:
    """The workload restricted to its first n samples (same lengths and
    settings; small cases of a recipe for profiler captures)."""
    n = max(1, min(int(n), w.B))
    return Workload(f"{w.name}[:{n}]", n, w.H, w.d, w.act, w.causal, w.lq[:n].copy(),
                    w.lkv[:n].copy(), max_rel=w.max_rel, pma_seeds=w.pma_seeds, window=w.window,
                    block=w.block, dense=w.dense, scale=w.scale, extra=dict(w.extra))


def custom_workload(lq, lkv, H, d, act="softmax", causal=False, max_rel=0, name="custom",
                    window=0, block=0):
    lq = np.asarray(lq, dtype=np.int64)
    lkv = np.asarray(lkv, dtype=np.int64)
    w = Workload(name, len(lq), H, d, act, causal, lq, lkv, max_rel=max_rel, window=window,
                 block=block)
    w.scale = 1.0 / math.sqrt(d)
    return w


def make_tensors(w: Workload, device="cpu", seed: int = 0, with_dout: bool = True,
                 dtype=torch.bfloat16) -> dict:
    """Draw q, k, v (and dout, bias) for workload `w` on `device`."""
    g = torch.Generator(device=device)
    g.manual_seed(seed + 1)
    H, d = w.H, w.d

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dtype)

    if w.pma_seeds:
        seeds = randn(w.pma_seeds, H, d)
        q = seeds.repeat(w.B, 1, 1)
    else:
        q = randn(w.Tq, H, d)
    k = randn(w.Tkv, H, d)
    v = randn(w.Tkv, H, d)
    dout = randn(w.Tq, H, d) if with_dout else None
    bias = None
    if w.max_rel:
        bias = (torch.randn(H, 2 * w.max_rel - 1, generator=g, device=device,
                            dtype=torch.float32) * 0.02)
    elif w.dense:
        # sample b's [H][Lq_b][Lkv_b] block starts at element off[b]
        off = np.zeros(w.B + 1, dtype=np.int64)
        off[1:] = np.cumsum(H * w.lq.astype(np.int64) * w.lkv.astype(np.int64))
        vals = torch.randn(int(off[-1]), generator=g, device=device, dtype=torch.float32) * 0.02
        bias = (vals, torch.from_numpy(off).to(device))
    qo, ko = w.offsets()
    return dict(q=q, k=k, v=v, dout=dout, bias=bias,
                qo=torch.from_numpy(qo).to(device), ko=torch.from_numpy(ko).to(device))
