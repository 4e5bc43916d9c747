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


@pytest.mark.parametrize("nosat", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_quant_rows_bit_exact(d, nosat):
    T, H = 300, 3
    x = _inputs(T, H, d, 1)
    codes, scales = binding.quantize_mxfp8(x, mode=binding.MX_ALONG_CHANNELS, nosat=nosat)
    rc, rs = oracle.quant_rows(to_np(x), nosat)
    np.testing.assert_array_equal(scales.cpu().numpy(), rs)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("nosat", [False, True])
@pytest.mark.parametrize("lengths", [[5, 40, 33, 0, 64, 1, 97], [300, 0, 31, 32, 33]])
def test_quant_tokens_bit_exact(lengths, nosat):
    H, d = 2, 128
    T = sum(lengths)
    x = _inputs(T, H, d, 2)
    o = offsets(lengths)
    off = torch.from_numpy(o).to(DEV)
    codes, scales = binding.quantize_mxfp8(x, off, mode=binding.MX_ALONG_TOKENS, nosat=nosat)
    rc, rs = oracle.quant_cols(to_np(x), o, nosat)
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


# ------------------------------------------------------------------ MXFP8 forward
from gpu_common import (MXFP8_TOL, assert_close, check_dense_gradient, check_guards,  # noqa: E402
                        check_table_gradient, dense_ref_kw, guarded, oracle_fwd_samples,
                        rand_bf16)
from jagged_attention_recsys_02_gb300.workloads import make_tensors, make_workload  # noqa: E402


def _mx_fwd(q, qo, k, v, ko, causal, scale, bias=None, max_rel=0):
    """The MXFP8 forward on operands quantised with the saturation-free block
    scale (GDPA_MX_NOSAT), the recipe the forward is specified with."""
    qc, qs = binding.quantize_mxfp8(q, mode=binding.MX_ALONG_CHANNELS, nosat=True)
    kc, ks = binding.quantize_mxfp8(k, mode=binding.MX_ALONG_CHANNELS, nosat=True)
    vc, vs = binding.quantize_mxfp8(v, ko, mode=binding.MX_ALONG_TOKENS, nosat=True)
    Tq, H, d = q.shape
    buf, out = guarded(Tq, H, d, q.device)
    lse = torch.full((H, Tq), float("nan"), device=q.device)
    binding.gdpa_fwd_mxfp8(qc, qs, qo, kc, ks, vc, vs, ko, causal=causal, scale=scale, bias=bias,
                           max_rel=max_rel, out=out, lse=lse)
    assert binding.device_status() == 0
    check_guards(buf)
    return out, lse


def _mx_reference(q, k, v, qo, ko, samples, causal, scale, bias, max_rel, rows=None):
    """fp64 oracle attention twice: on the MXFP8 operands (the bf16 inputs
    quantised by the oracle's own saturation-free quantiser and decoded again,
    so only P's rounding is left to the kernel), and exactly, on the
    unquantised inputs (the comparison the tolerance is stated for)."""
    qd = oracle.dequant_rows(q, nosat=True)
    kd = oracle.dequant_rows(k, nosat=True)
    vd = oracle.dequant_cols(v, ko, nosat=True)
    mx = oracle_fwd_samples(qd, kd, vd, qo, ko, samples, "softmax", causal, scale, bias, max_rel,
                            rows=rows)
    exact = oracle_fwd_samples(q, k, v, qo, ko, samples, "softmax", causal, scale, bias, max_rel,
                               rows=rows)
    return mx, exact


def _assert_exact(pairs, what, max_frac, max_worst):
    """The MXFP8 output against the exact fp64 forward on the unquantised bf16
    inputs, at abs 6e-2 + rel 6e-2.  E4M3 keeps 3 mantissa bits, so at d = 128
    the scores carry a rounding error of about 0.05 (one standard deviation);
    on rows with a handful of keys the softmax turns that into output errors
    near the bound, and a few elements pass it.  The assertion: at most
    `max_frac` of the elements outside the bound and none beyond `max_worst`
    times it.  Returns (fraction outside, worst err/bound)."""
    bad = tot = 0
    worst = 0.0
    for got, ref in pairs:
        r = np.abs(got - ref) / (MXFP8_TOL[0] + MXFP8_TOL[1] * np.abs(ref))
        bad += int((r > 1.0).sum())
        tot += r.size
        worst = max(worst, float(r.max()) if r.size else 0.0)
    frac = bad / max(tot, 1)
    print(f"{what}: against the unquantised inputs {bad} of {tot} elements outside "
          f"abs/rel 6e-2 (fraction {frac:.2e}), worst err/bound {worst:.3f}")
    assert frac <= max_frac and worst <= max_worst, \
        f"{what}: {bad} of {tot} elements outside the bound, worst {worst:.3f}"
    return frac, worst


# Short-key edge cases (1 to 3 keys, a bias of scale 0.5): at most 0.2% of the
# elements may pass the bound, none by more than 3x.  The heavy-tailed
# workload: at most 1e-5 of them, none by more than 1.5x.
EDGE_BUDGET = (2e-3, 3.0)
WORKLOAD_BUDGET = (1e-5, 1.5)


def _mx_case(lq, lkv, H, causal=False, max_rel=0, seed=0):
    d = 128
    g = torch.Generator(device=DEV).manual_seed(seed)
    q = rand_bf16((sum(lq), H, d), g, DEV)
    k = rand_bf16((sum(lkv), H, d), g, DEV)
    v = rand_bf16((sum(lkv), H, d), g, DEV)
    qo_np, ko_np = offsets(lq), offsets(lkv)
    qo, ko = torch.from_numpy(qo_np).to(DEV), torch.from_numpy(ko_np).to(DEV)
    bias = torch.randn(H, 2 * max_rel - 1, generator=g, device=DEV) * 0.5 if max_rel else None
    scale = 1.0 / np.sqrt(d)
    out, lse = _mx_fwd(q, qo, k, v, ko, causal, scale, bias, max_rel)
    ref, exact = _mx_reference(to_np(q), to_np(k), to_np(v), qo_np, ko_np, range(len(lq)), causal,
                               scale, None if bias is None else bias.cpu().double().numpy(),
                               max_rel)
    got = to_np(out)
    got_lse = lse.cpu().double().numpy()
    for rows, o, l in ref:
        assert_close(got[rows], o, MXFP8_TOL, f"mxfp8 out rows {rows[0]}..{rows[-1]}")
        assert_close(got_lse[:, rows], l, MXFP8_TOL, "mxfp8 lse")
    _assert_exact([(got[r_], o) for r_, o, _ in exact], "mxfp8 case", *EDGE_BUDGET)


def test_mxfp8_fwd_ragged():
    # lengths crossing the 32-token scale blocks and the 96-row key tiles
    _mx_case([1, 31, 32, 33, 95, 96, 97, 200, 0, 300, 513, 64],
             [7, 32, 31, 96, 97, 1, 200, 3, 5, 191, 700, 64], 2)


def test_mxfp8_fwd_causal_relpos():
    L = [1, 96, 97, 128, 300, 0, 511, 257]
    _mx_case(L, L, 2, causal=True, max_rel=300)


def test_mxfp8_fwd_empty_keys():
    _mx_case([3, 0, 130, 5], [0, 9, 0, 140], 2)


@pytest.mark.parametrize("causal", [False, True])
def test_mxfp8_fwd_dense_bias(causal):
    """The MXFP8 forward with a dense jagged bias (fp32 values added to the
    fp32 scores): against the oracle on the decoded operands at the MXFP8
    tolerance, and against the exact forward on the unquantised inputs within
    the edge-case budget."""
    lq = [1, 31, 96, 97, 200, 0, 300, 129]
    lkv = lq if causal else [7, 32, 1, 96, 128, 5, 191, 300]
    H, d = 2, 128
    g = torch.Generator(device=DEV).manual_seed(11 + causal)
    q = rand_bf16((sum(lq), H, d), g, DEV)
    k = rand_bf16((sum(lkv), H, d), g, DEV)
    v = rand_bf16((sum(lkv), H, d), g, DEV)
    qo_np, ko_np = offsets(lq), offsets(lkv)
    qo, ko = torch.from_numpy(qo_np).to(DEV), torch.from_numpy(ko_np).to(DEV)
    off_np = oracle.dense_bias_offsets(qo_np, ko_np, H)
    vals = torch.randn(int(off_np[-1]), generator=g, device=DEV) * 0.5
    scale = 1.0 / np.sqrt(d)
    out, lse = _mx_fwd(q, qo, k, v, ko, causal, scale, bias=(vals, torch.from_numpy(off_np).to(DEV)))
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    kw = dict(act=0, causal=causal, scale=scale, dense_bias=vals.double().cpu().numpy())
    ro, rl = oracle.fwd(oracle.dequant_rows(qn, nosat=True), qo_np,
                        oracle.dequant_rows(kn, nosat=True),
                        oracle.dequant_cols(vn, ko_np, nosat=True), ko_np, **kw)
    got = to_np(out)
    assert_close(got, ro, MXFP8_TOL, f"mxfp8 dense causal={causal} out")
    assert_close(lse.cpu().double().numpy(), rl, MXFP8_TOL, f"mxfp8 dense causal={causal} lse")
    ex, _ = oracle.fwd(qn, qo_np, kn, vn, ko_np, **kw)
    _assert_exact([(got, ex)], f"mxfp8 dense causal={causal}", *EDGE_BUDGET)


def test_mxfp8_rejects_gdpa_and_d64():
    lib = binding.load()
    p = torch.zeros(64, device=DEV, dtype=torch.uint8).data_ptr()
    o = torch.zeros(2, device=DEV, dtype=torch.int32).data_ptr()
    common = (p, p, o, p, p, p, p, o, 1, 1)
    assert lib.gdpa_fwd_mxfp8(*common, 128, 1, 1, None, 1, 0, 0.1, p, p, p, 1 << 20, None) == 2
    assert lib.gdpa_fwd_mxfp8(*common, 64, 1, 1, None, 0, 0, 0.1, p, p, p, 1 << 20, None) == 2


def test_mxfp8_fwd_full_heavy_tail():
    """The production-like heavy-tailed mix (B=1024, log-normal lengths), softmax,
    the workload the MXFP8 forward's tolerance is stated on.  Sampled samples:
    every row of those up to 2048 tokens, the first, last and tile-boundary rows
    of longer ones; against the quantisation-mirroring oracle elementwise, and
    against the exact forward on the unquantised inputs."""
    w = make_workload("heavy_tail", act="softmax")
    t = make_tensors(w, device=DEV, with_dout=False)
    out, lse = _mx_fwd(t["q"], t["qo"], t["k"], t["v"], t["ko"], False, w.scale)
    qo, ko = w.offsets()
    pairs = w.lq * w.lkv
    rng = np.random.default_rng(5)
    samples = sorted({int(np.argmin(pairs)), int(np.argmax(pairs)),
                      *np.argsort(pairs)[:6].tolist(),
                      *rng.choice(w.B, 24, replace=False).tolist()})
    exact_pairs = []
    for b in samples:
        q0, q1, k0, k1 = int(qo[b]), int(qo[b + 1]), int(ko[b]), int(ko[b + 1])
        L = q1 - q0
        if L <= 2048:
            rows = np.arange(L)
        else:
            rows = np.array(sorted({0, 1, L // 2, L - 1, *range(95, L, 96 * 5)}))
        ref, exact = _mx_reference(to_np(t["q"][q0:q1]), to_np(t["k"][k0:k1]),
                                   to_np(t["v"][k0:k1]), np.array([0, L]),
                                   np.array([0, k1 - k0]), [0], False, w.scale, None, 0,
                                   rows={0: rows})
        sel = torch.from_numpy(q0 + rows).to(DEV)
        got = to_np(out[sel])
        for r, o, l in ref:
            assert_close(got, o, MXFP8_TOL, f"heavy_tail mxfp8 sample {b}")
            assert_close(lse[:, sel].cpu().double().numpy(), l, MXFP8_TOL, "heavy_tail mxfp8 lse")
        exact_pairs += [(got, o) for _, o, _ in exact]
    _assert_exact(exact_pairs, "heavy_tail mxfp8", *WORKLOAD_BUDGET)


def test_quant_tokens_zeroes_tokens_outside_samples():
    """Codes of tokens before the first or after the last sample are 0, whatever
    the buffer held (a tile that runs past a sample's end reads them)."""
    H, d, T = 2, 128, 70
    x = _inputs(T, H, d, 4)
    o = offsets([5, 40])                       # samples cover tokens 0..44
    off = torch.from_numpy(o).to(DEV)
    codes = torch.full((T, H, d), 0x7F, device=DEV, dtype=torch.uint8)  # E4M3 NaN codes
    codes, scales = binding.quantize_mxfp8(x, off, mode=binding.MX_ALONG_TOKENS, codes=codes)
    got = codes.cpu().numpy()
    assert np.all(got[45:] == 0)
    rc, _ = oracle.quant_cols(to_np(x[:45]), o)
    np.testing.assert_array_equal(got[:45], rc)


# ------------------------------------------------------------------ MXFP8 backward
# The reference is the oracle's MXFP8 backward: the operands quantised by the
# oracle's own quantisers, P and dS rounded in 32 x 32 blocks the same way.
# What is left differs only by fp32 accumulation order, ex2.approx in P, the
# bf16 rounding of the outputs (2^-9) and, rarely, an element sitting within
# fp32 rounding of an E4M3 rounding boundary: (2e-2, 2e-2) covers them.
MXBWD_TOL = (2e-2, 2e-2)


def _mx_bwd_run(q, qo, k, v, ko, out, lse, dout, causal, scale, bias, max_rel, window=0):
    Tq, H, d = q.shape
    Tkv = k.shape[0]
    bq, dq = guarded(Tq, H, d, q.device)
    bk, dk = guarded(Tkv, H, d, q.device)
    bv, dv = guarded(Tkv, H, d, q.device)
    ws = torch.full((binding.bwd_mxfp8_workspace_size(qo.numel() - 1, H, d, Tq, Tkv),), 0xFF,
                    device=q.device, dtype=torch.uint8)  # stale bytes must not matter
    binding.gdpa_bwd_mxfp8(q, qo, k, v, ko, out, lse, dout, causal=causal, scale=scale, bias=bias,
                           max_rel=max_rel, window=window, dq=dq, dk=dk, dv=dv, workspace=ws)
    assert binding.device_status() == 0
    for b in (bq, bk, bv):
        check_guards(b)
    return dq, dk, dv


def _mx_bwd_case(lq, lkv, H, causal=False, max_rel=0, seed=0, window=0):
    """Random bf16 inputs; out and lse from the oracle's forward (the backward's
    inputs, as a training step passes them); every gradient element checked."""
    d = 128
    g = torch.Generator(device=DEV).manual_seed(seed)
    Tq, Tkv = sum(lq), sum(lkv)
    q = rand_bf16((Tq, H, d), g, DEV)
    k = rand_bf16((Tkv, H, d), g, DEV)
    v = rand_bf16((Tkv, H, d), g, DEV)
    dout = rand_bf16((Tq, H, d), g, DEV)
    qo_np, ko_np = offsets(lq), offsets(lkv)
    qo, ko = torch.from_numpy(qo_np).to(DEV), torch.from_numpy(ko_np).to(DEV)
    bias = torch.randn(H, 2 * max_rel - 1, generator=g, device=DEV) * 0.5 if max_rel else None
    bias_np = None if bias is None else bias.cpu().double().numpy()
    scale = 1.0 / np.sqrt(d)
    nq, nk = sum(lq), sum(lkv)
    o_ref, l_ref = oracle.fwd(to_np(q[:nq]), qo_np, to_np(k[:nk]), to_np(v[:nk]), ko_np,
                              act=oracle.ACT_SOFTMAX, causal=causal, scale=scale, bias=bias_np,
                              max_rel=max_rel, window=window)
    out = torch.zeros((Tq, H, d), device=DEV, dtype=torch.bfloat16)
    out[:nq] = torch.from_numpy(o_ref).to(DEV).to(torch.bfloat16)
    lse = torch.zeros((H, Tq), device=DEV, dtype=torch.float32)
    lse[:, :nq] = torch.from_numpy(np.where(np.isinf(l_ref), 0.0, l_ref)).to(DEV).float()
    dq, dk, dv = _mx_bwd_run(q, qo, k, v, ko, out, lse, dout, causal, scale, bias, max_rel,
                             window=window)
    ref = oracle.bwd_mxfp8(to_np(q[:nq]), qo_np, to_np(k[:nk]), to_np(v[:nk]), ko_np,
                           to_np(out[:nq]), to_np(dout[:nq]), lse[:, :nq].cpu().double().numpy(),
                           causal=causal, scale=scale, bias=bias_np, max_rel=max_rel,
                           window=window)
    for name, got, r in (("dq", dq[:nq], ref[0]), ("dk", dk[:nk], ref[1]), ("dv", dv[:nk], ref[2])):
        assert_close(to_np(got), r, MXBWD_TOL, f"mxfp8 bwd {name}")
    exact = oracle.bwd(to_np(q[:nq]), qo_np, to_np(k[:nk]), to_np(v[:nk]), ko_np, to_np(dout[:nq]),
                       act=oracle.ACT_SOFTMAX, causal=causal, scale=scale, bias=bias_np,
                       max_rel=max_rel, window=window)
    for name, got, r in (("dq", dq[:nq], exact[0]), ("dk", dk[:nk], exact[1]), ("dv", dv[:nk], exact[2])):
        e = np.abs(to_np(got) - r)
        print(f"mxfp8 bwd {name}: relative RMS error against the unquantised backward "
              f"{np.sqrt((e ** 2).mean() / max((r ** 2).mean(), 1e-300)):.4f}")
    return dq, dk, dv


def test_mxfp8_bwd_ragged():
    # lengths crossing the 32-token scale blocks, the 64-query tiles and the 128-key blocks
    _mx_bwd_case([1, 31, 32, 33, 63, 64, 65, 200, 0, 300, 129, 7],
                 [7, 32, 31, 96, 128, 1, 129, 3, 5, 191, 300, 64], 2)


def test_mxfp8_bwd_causal_relpos():
    L = [1, 64, 65, 128, 129, 300, 0, 511, 257]
    _mx_bwd_case(L, L, 2, causal=True, max_rel=300)


@pytest.mark.parametrize("causal", [False, True])
def test_mxfp8_bwd_sliding_window(causal):
    # windows shorter and longer than a 64-query tile / 128-key block, band edges inside tiles
    L = [1, 64, 65, 130, 300, 0, 511]
    for window in (7, 100, 200):
        _mx_bwd_case(L, L, 2, causal=causal, max_rel=64, window=window, seed=window)


def _e4m3_exact(shape, g):
    """bf16 values that E4M3 holds exactly under any power-of-two block scale
    the quantisers pick: k / 8 for integers |k| <= 12 (three significand bits),
    so every product of the backward runs on exact operands."""
    k = torch.randint(-12, 13, shape, generator=g, device=DEV)
    return (k.float() / 8.0).to(torch.bfloat16)


@pytest.mark.parametrize("causal", [False, True])
def test_mxfp8_bwd_table_gradient(causal):
    """gdpa_bwd_mxfp8_rope with dbias: the gradient is summed from the fp32 dS
    before its E4M3 rounding.  On inputs the quantisers hold exactly, the
    scores and dP are exact, so the table gradient must match the unquantised
    oracle's within the per-pair bounds of the bf16 backward (P from ex2.approx,
    D from the bf16 forward output); dq, dk, dv still match the oracle's MXFP8
    backward."""
    L = [1, 64, 65, 130, 300, 0, 257]
    lkv = L if causal else [7, 1, 128, 129, 200, 3, 300]
    H, d, max_rel = 2, 128, 150
    g = torch.Generator(device=DEV).manual_seed(17 + causal)
    q, do = _e4m3_exact((sum(L), H, d), g), _e4m3_exact((sum(L), H, d), g)
    k, v = _e4m3_exact((sum(lkv), H, d), g), _e4m3_exact((sum(lkv), H, d), g)
    bias = torch.randn(H, 2 * max_rel - 1, generator=g, device=DEV) * 0.5
    qo_np, ko_np = offsets(L), offsets(lkv)
    qo, ko = torch.from_numpy(qo_np).to(DEV), torch.from_numpy(ko_np).to(DEV)
    scale = 1.0 / np.sqrt(d)
    bias_np = bias.cpu().double().numpy()
    o_ref, l_ref = oracle.fwd(to_np(q), qo_np, to_np(k), to_np(v), ko_np, act=oracle.ACT_SOFTMAX,
                              causal=causal, scale=scale, bias=bias_np, max_rel=max_rel)
    out = torch.from_numpy(o_ref).to(DEV).to(torch.bfloat16)
    lse = torch.from_numpy(np.where(np.isinf(l_ref), 0.0, l_ref)).to(DEV).float()
    dbias = torch.zeros_like(bias)
    dq, dk, dv = binding.gdpa_bwd_mxfp8(q, qo, k, v, ko, out, lse, do, causal=causal, scale=scale,
                                        bias=bias, max_rel=max_rel, dbias=dbias)
    assert binding.device_status() == 0
    check_table_gradient(q, qo_np, k, v, ko_np, do, bias, dbias, act=oracle.ACT_SOFTMAX,
                         causal=causal, scale=scale, max_rel=max_rel, window=0,
                         what=f"mxfp8 dbias causal={causal}")
    ref = oracle.bwd_mxfp8(to_np(q), qo_np, to_np(k), to_np(v), ko_np, to_np(out), to_np(do),
                           lse.cpu().double().numpy(), causal=causal, scale=scale, bias=bias_np,
                           max_rel=max_rel)
    for name, got, r in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        assert_close(to_np(got), r, MXBWD_TOL, f"mxfp8 bwd with dbias {name}")


@pytest.mark.parametrize("window", [0, 100])
@pytest.mark.parametrize("causal", [False, True])
def test_mxfp8_bwd_dense_bias(causal, window):
    """The MXFP8 backward with a dense jagged bias: dq, dk, dv against the
    oracle's MXFP8 backward with that bias on random bf16 inputs (with and
    without a sliding window); then on inputs the quantisers hold exactly, the
    dense bias's gradient (dbias, from the fp32 dS) against the unquantised
    oracle's within the per-pair bounds, masked entries untouched."""
    L = [1, 64, 65, 130, 300, 0, 257]
    lkv = L if (causal or window) else [7, 1, 128, 129, 200, 3, 300]
    H, d = 2, 128
    g = torch.Generator(device=DEV).manual_seed(29 + causal + window)
    qo_np, ko_np = offsets(L), offsets(lkv)
    qo, ko = torch.from_numpy(qo_np).to(DEV), torch.from_numpy(ko_np).to(DEV)
    off_np = oracle.dense_bias_offsets(qo_np, ko_np, H)
    off = torch.from_numpy(off_np).to(DEV)
    vals = torch.randn(int(off_np[-1]), generator=g, device=DEV) * 0.5
    scale = 1.0 / np.sqrt(d)
    what = f"mxfp8 dense causal={causal} window={window}"
    for exact_inputs in (False, True):
        if exact_inputs:
            q, do = _e4m3_exact((sum(L), H, d), g), _e4m3_exact((sum(L), H, d), g)
            k, v = _e4m3_exact((sum(lkv), H, d), g), _e4m3_exact((sum(lkv), H, d), g)
        else:
            q, do = rand_bf16((sum(L), H, d), g, DEV), rand_bf16((sum(L), H, d), g, DEV)
            k, v = rand_bf16((sum(lkv), H, d), g, DEV), rand_bf16((sum(lkv), H, d), g, DEV)
        c = dict(q=q, k=k, v=v, do=do, qo_np=qo_np, ko_np=ko_np, vals=vals, act=oracle.ACT_SOFTMAX,
                 causal=causal, scale=scale, window=window, block=0)
        o_ref, l_ref = oracle.fwd(to_np(q), qo_np, to_np(k), to_np(v), ko_np, **dense_ref_kw(c))
        out = torch.from_numpy(o_ref).to(DEV).to(torch.bfloat16)
        lse = torch.from_numpy(np.where(np.isinf(l_ref), 0.0, l_ref)).to(DEV).float()
        base = torch.randn(vals.numel(), generator=g, device=DEV) if exact_inputs else None
        dbias = base.clone() if exact_inputs else None
        dq, dk, dv = binding.gdpa_bwd_mxfp8(q, qo, k, v, ko, out, lse, do, causal=causal,
                                            scale=scale, bias=(vals, off), window=window,
                                            dbias=dbias)
        assert binding.device_status() == 0
        ref = oracle.bwd_mxfp8(to_np(q), qo_np, to_np(k), to_np(v), ko_np, to_np(out), to_np(do),
                               lse.cpu().double().numpy(), causal=causal, scale=scale,
                               window=window, dense_bias=vals.double().cpu().numpy())
        for name, got, r in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
            assert_close(to_np(got), r, MXBWD_TOL, f"{what} exact_inputs={exact_inputs} {name}")
        if exact_inputs:
            check_dense_gradient(c, dbias, base, what + " dbias")


@pytest.mark.parametrize("causal", [False, True])
def test_mxfp8_bwd_fused_rope(causal):
    """gdpa_bwd_mxfp8_rope with rope_base > 0: dq, dk are the oracle's MXFP8
    gradients sent back through the rotary embedding (queries and keys at
    their own positions), dv unchanged."""
    L = [1, 64, 65, 130, 300, 0, 257]
    lkv = L if causal else [7, 1, 128, 129, 200, 3, 300]
    H, d, base = 2, 128, 10000.0
    g = torch.Generator(device=DEV).manual_seed(29 + causal)
    q, do = rand_bf16((sum(L), H, d), g, DEV), rand_bf16((sum(L), H, d), g, DEV)
    k, v = rand_bf16((sum(lkv), H, d), g, DEV), rand_bf16((sum(lkv), H, d), g, DEV)
    qo_np, ko_np = offsets(L), offsets(lkv)
    qo, ko = torch.from_numpy(qo_np).to(DEV), torch.from_numpy(ko_np).to(DEV)
    scale = 1.0 / np.sqrt(d)
    o_ref, l_ref = oracle.fwd(to_np(q), qo_np, to_np(k), to_np(v), ko_np, act=oracle.ACT_SOFTMAX,
                              causal=causal, scale=scale)
    out = torch.from_numpy(o_ref).to(DEV).to(torch.bfloat16)
    lse = torch.from_numpy(np.where(np.isinf(l_ref), 0.0, l_ref)).to(DEV).float()
    dq, dk, dv = binding.gdpa_bwd_mxfp8(q, qo, k, v, ko, out, lse, do, causal=causal, scale=scale,
                                        rope_base=base)
    assert binding.device_status() == 0
    ref = oracle.bwd_mxfp8(to_np(q), qo_np, to_np(k), to_np(v), ko_np, to_np(out), to_np(do),
                           lse.cpu().double().numpy(), causal=causal, scale=scale)
    what = f"mxfp8 rope causal={causal}"
    assert_close(to_np(dq), oracle.rope_bwd(ref[0], qo_np, base), MXBWD_TOL, what + " dq")
    assert_close(to_np(dk), oracle.rope_bwd(ref[1], ko_np, base), MXBWD_TOL, what + " dk")
    assert_close(to_np(dv), ref[2], MXBWD_TOL, what + " dv")


def test_mxfp8_bwd_empty_sides():
    _mx_bwd_case([3, 0, 130, 5], [0, 9, 0, 140], 2)


def test_mxfp8_bwd_rejects_offsets_short_of_the_tensor():
    """Offsets must end at the tensor's last row: a mismatch is reported through
    the device status word (and the kernels do no work)."""
    H, d = 1, 128
    g = torch.Generator(device=DEV).manual_seed(3)
    q = rand_bf16((150, H, d), g, DEV)
    qo = torch.from_numpy(offsets([70, 30])).to(DEV)
    lse = torch.zeros((H, 150), device=DEV)
    binding.gdpa_bwd_mxfp8(q, qo, q, q, qo, q, lse, q, causal=True, scale=0.1)
    assert binding.device_status() == 6  # GDPA_ERR_BAD_OFFSETS


def test_mxfp8_bwd_rejects_gdpa_and_d64():
    lib = binding.load()
    p = torch.zeros(64, device=DEV, dtype=torch.uint8).data_ptr()
    o = torch.zeros(2, device=DEV, dtype=torch.int32).data_ptr()
    common = (p, o, p, p, o, 1, 1)
    tail = (p, p, p, p, p, p, p, 1 << 20, None)
    assert lib.gdpa_bwd_mxfp8(*common, 128, 1, 1, None, 1, 0, 0.1, *tail) == 2
    assert lib.gdpa_bwd_mxfp8(*common, 64, 1, 1, None, 0, 0, 0.1, *tail) == 2


def test_mxfp8_bwd_full_jfa_causal_relpos():
    """The full causal rel-pos workload (B=32, L~U[1,4096], H=4) in the launch
    configuration the benchmark times, every gradient element of three samples
    (the shortest, a middle one, the longest) against the oracle.  The other
    samples get out = 0 and lse = 30 (finite, P tiny): samples are independent."""
    w = make_workload("jfa_causal_relpos")
    t = make_tensors(w, device=DEV, with_dout=True)
    qo, ko = w.offsets()
    order = np.argsort(w.lq)
    samples = [int(order[0]), int(order[len(order) // 2]), int(order[-1])]
    out = torch.zeros_like(t["q"])
    lse = torch.full((w.H, w.Tq), 30.0, device=DEV, dtype=torch.float32)
    bias_np = t["bias"].cpu().double().numpy()
    for b in samples:
        s0, s1 = int(qo[b]), int(qo[b + 1])
        o_ref, l_ref = oracle.fwd(to_np(t["q"][s0:s1]), np.array([0, s1 - s0]),
                                  to_np(t["k"][s0:s1]), to_np(t["v"][s0:s1]),
                                  np.array([0, s1 - s0]), act=oracle.ACT_SOFTMAX, causal=True,
                                  scale=w.scale, bias=bias_np, max_rel=w.max_rel)
        out[s0:s1] = torch.from_numpy(o_ref).to(DEV).to(torch.bfloat16)
        lse[:, s0:s1] = torch.from_numpy(l_ref).to(DEV).float()
    dq, dk, dv = _mx_bwd_run(t["q"], t["qo"], t["k"], t["v"], t["ko"], out, lse, t["dout"], True,
                             w.scale, t["bias"], w.max_rel)
    for b in samples:
        s0, s1 = int(qo[b]), int(qo[b + 1])
        one = np.array([0, s1 - s0])
        ref = oracle.bwd_mxfp8(to_np(t["q"][s0:s1]), one, to_np(t["k"][s0:s1]),
                               to_np(t["v"][s0:s1]), one, to_np(out[s0:s1]),
                               to_np(t["dout"][s0:s1]), lse[:, s0:s1].cpu().double().numpy(),
                               causal=True, scale=w.scale, bias=bias_np, max_rel=w.max_rel)
        for name, got, r in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
            assert_close(to_np(got[s0:s1]), r, MXBWD_TOL, f"jfa mxfp8 bwd {name} sample {b}")
