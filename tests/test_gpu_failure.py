"""Failure detection without a GPU fault: a pipeline wait that cannot complete
gives up after its limit, the kernel records GDPA_ERR_TIMEOUT in the device
status word and returns; the host reads (and clears) it, and the context stays
usable for the next call."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_common import FWD_TOL, assert_close, offsets, rand_bf16, to_np
from jagged_attention_recsys_02_gb300 import binding

pytestmark = pytest.mark.gpu

TIMEOUT = 5  # GDPA_ERR_TIMEOUT


def test_timeout_is_reported_cleared_and_the_context_survives():
    assert binding.device_status() == 0
    binding.selftest_timeout(2000)           # a 2 ms wait that nothing completes
    assert binding.device_status() == TIMEOUT
    assert binding.device_status() == 0      # reading the word clears it
    # the context still works: a small forward matches the oracle
    lengths = [3, 40, 0, 17]
    H, d = 2, 64
    g = torch.Generator(device="cuda").manual_seed(5)
    q, k, v = (rand_bf16((sum(lengths), H, d), g, "cuda") for _ in range(3))
    o_np = offsets(lengths)
    o = torch.from_numpy(o_np).cuda()
    out, _ = binding.gdpa_fwd(q, o, k, v, o, act="silu", scale=1.0 / math.sqrt(d))
    assert binding.device_status() == 0
    ref, _ = oracle.fwd(to_np(q), o_np, to_np(k), to_np(v), o_np, act=oracle.ACT_SILU,
                        scale=1.0 / math.sqrt(d))
    assert_close(to_np(out), ref, FWD_TOL, "forward after a reported timeout")


def test_the_first_error_is_kept():
    """The status word keeps the first error until it is read."""
    binding.selftest_timeout(500)
    binding.selftest_timeout(500)
    assert binding.device_status() == TIMEOUT
    assert binding.device_status() == 0
