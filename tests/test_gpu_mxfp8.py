"""GPU MXFP8 quantiser against the oracle's quantiser: codes and scales must
match bit for bit (integer / byte work), including empty and partial blocks,
all-zero blocks, signed zeros, subnormal bf16 inputs and saturation."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import offsets, to_np
from jagged_attention_recsys_02_gb300 import binding

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs(T, H, d, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn(T, H, d, generator=g, device=DEV)
    # per-row magnitudes spread over many binades, plus special values
    x = x * torch.exp2(torch.randint(-20, 20, (T, H, 1), generator=g, device=DEV).float())
    x = x.to(torch.bfloat16)
    flat = x.view(-1)
    n = flat.numel()
    if n > 4096:
        flat[0:32] = 0.0                                   # all-zero block
        flat[32:64] = -0.0
        flat[64:96] = torch.tensor(1e-40, dtype=torch.bfloat16)  # bf16 subnormals
        flat[96] = 3.0e38                                   # huge amax
        flat[128:160] = torch.linspace(-500, 500, 32, device=DEV).to(torch.bfloat16)
        flat[160:192] = 1.0 + 1.0 / 16                      # E4M3 ties
        flat[192] = 1.0
    return x


@pytest.mark.parametrize("d", [64, 128])
def test_quant_rows_bit_exact(d):
    T, H = 300, 3
    x = _inputs(T, H, d, 1)
    codes, scales = binding.quantize_mxfp8(x, mode=binding.MX_ALONG_CHANNELS)
    rc, rs = oracle.quant_rows(to_np(x))
    np.testing.assert_array_equal(scales.cpu().numpy(), rs)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("lengths", [[5, 40, 33, 0, 64, 1, 97], [300, 0, 31, 32, 33]])
def test_quant_tokens_bit_exact(lengths):
    H, d = 2, 128
    T = sum(lengths)
    x = _inputs(T, H, d, 2)
    o = offsets(lengths)
    off = torch.from_numpy(o).to(DEV)
    codes, scales = binding.quantize_mxfp8(x, off, mode=binding.MX_ALONG_TOKENS)
    rc, rs = oracle.quant_cols(to_np(x), o)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)
    # map the oracle's compact block rows onto the library's row index b + floor(o_b/32) + r
    got = scales.cpu().numpy()
    k = 0
    for b, L in enumerate(lengths):
        for r in range((L + 31) // 32):
            np.testing.assert_array_equal(got[b + o[b] // 32 + r], rs[k])
            k += 1
    assert k == rs.shape[0]


def test_quant_full_size_v_and_q():
    """heavy-tail-like shapes: V along tokens, Q along channels (sampled rows)."""
    rng = np.random.default_rng(0)
    L = np.clip(np.round(np.exp(rng.normal(np.log(1024.0), 1.0, 64))), 16, 16384).astype(int)
    H, d = 4, 128
    o = offsets(L)
    x = _inputs(int(o[-1]), H, d, 3)
    off = torch.from_numpy(o).to(DEV)
    vc, vs = binding.quantize_mxfp8(x, off, mode=binding.MX_ALONG_TOKENS)
    qc, qs = binding.quantize_mxfp8(x, mode=binding.MX_ALONG_CHANNELS)
    for b in (0, int(np.argmax(L)), 17):
        sl = slice(int(o[b]), int(o[b + 1]))
        rc, rs = oracle.quant_cols(to_np(x[sl]), np.array([0, L[b]]))
        np.testing.assert_array_equal(vc[sl].cpu().numpy(), rc)
        base = b + int(o[b]) // 32
        np.testing.assert_array_equal(vs[base:base + rs.shape[0]].cpu().numpy(), rs)
        rc, rs = oracle.quant_rows(to_np(x[sl]))
        np.testing.assert_array_equal(qc[sl].cpu().numpy(), rc)
        np.testing.assert_array_equal(qs[sl].cpu().numpy(), rs)
