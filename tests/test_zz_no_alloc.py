"""The allocation-free forward entry point, gdpa_fwd_noalloc.

Callers that cannot allocate device memory (for example a plugin inside a
framework that has already claimed the GPU's memory for its own pool) use
gdpa_fwd_noalloc, which takes its scratch from a fixed 1 MiB array inside the
library instead of a caller-provided workspace.  These checks call it through
the C ABI twice in a row and compare each result with the regular gdpa_fwd
on the same inputs, within the forward tolerance the other parity tests use.

This file is named so that pytest collects it last.
"""
import ctypes
import math

import pytest
import torch

from gpu_common import FWD_TOL, assert_close, check_guards, guarded, offsets, rand_bf16, to_np
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


@pytest.mark.parametrize("act", [0, 1])  # softmax, SiLU
def test_noalloc_matches_workspace_call(act):
    lib = binding.load()
    fn = _noalloc(lib)
    g = torch.Generator(device=DEV).manual_seed(11)
    lq = [1, 300, 0, 129, 513, 64]
    lkv = [7, 256, 5, 0, 700, 64]
    H, d = 2, 128
    q = rand_bf16((sum(lq), H, d), g, DEV)
    k = rand_bf16((sum(lkv), H, d), g, DEV)
    v = rand_bf16((sum(lkv), H, d), g, DEV)
    qo = torch.from_numpy(offsets(lq)).to(DEV)
    ko = torch.from_numpy(offsets(lkv)).to(DEV)
    scale = 1.0 / math.sqrt(d)
    ref_out, ref_lse = binding.gdpa_fwd(q, qo, k, v, ko, act=act, scale=scale)
    torch.cuda.synchronize()
    ref = to_np(ref_out)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # two calls in a row share (and reuse) the static scratch
        buf, out = guarded(sum(lq), H, d, DEV)
        lse = torch.full((H, sum(lq)), float("nan"), device=DEV) if act == 0 else None
        rc = fn(q.data_ptr(), qo.data_ptr(), k.data_ptr(), v.data_ptr(), ko.data_ptr(), len(lq), H,
                d, sum(lq), sum(lkv), None, act, 0, scale, out.data_ptr(),
                lse.data_ptr() if lse is not None else None, stream)
        assert rc == 0, binding.STATUS_NAMES.get(rc, rc)
        assert binding.device_status() == 0
        check_guards(buf)
        assert_close(to_np(out), ref, FWD_TOL, "gdpa_fwd_noalloc out")
        if act == 0:
            assert_close(lse.cpu().double().numpy(), ref_lse.cpu().double().numpy(), FWD_TOL,
                         "gdpa_fwd_noalloc lse")


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
