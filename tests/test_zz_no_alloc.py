"""The allocation-free forward entry point, gdpa_fwd_noalloc.

Callers that cannot allocate device memory (for example a plugin inside a
framework that has already claimed the GPU's memory for its own pool) use
gdpa_fwd_noalloc, which takes its scratch from a fixed 1 MiB array inside the
library instead of a caller-provided workspace.  These checks call it through
the C ABI several times in a row -- a larger problem, then a smaller one, so a
work list left in the shared array by the first call would show in the
second -- and compare every result with the fp64 oracle (within the forward
tolerance of the other parity tests) and with the regular gdpa_fwd on the same
inputs bit for bit (the same kernels run on the same work items; a forward
item writes its own rows only, so the order of the list cannot change them).

This file is named so that pytest collects it last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from gpu_common import (FWD_TOL, assert_close, check_guards, guarded, offsets,
                        oracle_fwd_samples, rand_bf16, to_np)
from jagged_attention_recsys_02_gb300 import binding

pytestmark = pytest.mark.gpu

DEV = "cuda"
GDPA_ERR_WORKSPACE = 3


def _noalloc(lib):
    fn = lib.gdpa_fwd_noalloc
    vp, i64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, I, I, I, i64, i64, ctypes.POINTER(binding.gdpa_bias), I, I,
                   ctypes.c_float, vp, vp, vp]
    fn.restype = I
    return fn


def _problem(lq, lkv, H, d, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    q = rand_bf16((sum(lq), H, d), g, DEV)
    k = rand_bf16((sum(lkv), H, d), g, DEV)
    v = rand_bf16((sum(lkv), H, d), g, DEV)
    qo_np, ko_np = offsets(lq), offsets(lkv)
    return q, k, v, qo_np, ko_np


LARGE = ([1, 300, 0, 129, 513, 64, 2000, 77], [7, 256, 5, 0, 700, 64, 1500, 77])
SMALL = ([5, 0, 200], [9, 3, 130])


@pytest.mark.parametrize("act", [0, 1])  # softmax, SiLU
def test_noalloc_matches_oracle_and_workspace_call(act):
    lib = binding.load()
    fn = _noalloc(lib)
    H, d = 2, 128
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream().cuda_stream
    # larger problem, smaller problem, larger again: each call reuses the array
    for n, (lq, lkv) in enumerate((LARGE, SMALL, LARGE)):
        q, k, v, qo_np, ko_np = _problem(lq, lkv, H, d, seed=11 + n)
        qo, ko = torch.from_numpy(qo_np).to(DEV), torch.from_numpy(ko_np).to(DEV)
        buf, out = guarded(sum(lq), H, d, DEV)
        lse = torch.full((H, sum(lq)), float("nan"), device=DEV) if act == 0 else None
        rc = fn(q.data_ptr(), qo.data_ptr(), k.data_ptr(), v.data_ptr(), ko.data_ptr(), len(lq),
                H, d, sum(lq), sum(lkv), None, act, 0, scale, out.data_ptr(),
                lse.data_ptr() if lse is not None else None, stream)
        assert rc == 0, binding.STATUS_NAMES.get(rc, rc)
        assert binding.device_status() == 0
        check_guards(buf)
        # the fp64 oracle, every sample
        for rows, o, l in oracle_fwd_samples(to_np(q), to_np(k), to_np(v), qo_np, ko_np,
                                             range(len(lq)), act, False, scale):
            assert_close(to_np(out[torch.from_numpy(rows).to(DEV)]), o, FWD_TOL,
                         f"gdpa_fwd_noalloc out (call {n})")
            if act == 0:
                assert_close(lse[:, torch.from_numpy(rows).to(DEV)].cpu().double().numpy(), l,
                             FWD_TOL, f"gdpa_fwd_noalloc lse (call {n})")
        # the workspace entry point on the same inputs: identical bits
        ref_out, ref_lse = binding.gdpa_fwd(q, qo, k, v, ko, act=act, scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), f"call {n}: out"
        if act == 0:
            assert torch.equal(lse, ref_lse), f"call {n}: lse"


def test_noalloc_refuses_problems_beyond_its_scratch():
    lib = binding.load()
    fn = _noalloc(lib)
    # 1 MiB of scratch holds about 131k work items; this problem needs far more.
    B, H, d, T = 200000, 8, 128, 200000
    assert lib.gdpa_fwd_workspace_size(B, H, d, T, T) > (1 << 20)
    dummy = torch.zeros(16, device=DEV, dtype=torch.bfloat16)
    p = dummy.data_ptr()
    rc = fn(p, p, p, p, p, B, H, d, T, T, None, 1, 0, 0.1, p, None,
            torch.cuda.current_stream().cuda_stream)
    assert rc == GDPA_ERR_WORKSPACE
