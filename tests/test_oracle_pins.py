"""Pins of the fp64 oracle against things other than itself (CPU only).

Each pin checks the oracle against an independent fact: a hand-derived worked
example, a closed form, a library routine (torch's fp64 SDPA, logsumexp,
SiLU/GELU, float8 conversion), an algebraic identity evaluated in a different
order, an invariant, or central finite differences of the oracle's own
forward (which pins every backward formula).  They are chosen so that a
dropped term, a wrong sign or index, or a transposed operand in the oracle
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import ACT_GELU_ERF, ACT_GELU_TANH, ACT_IDENTITY, ACT_SILU, ACT_SOFTMAX

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ACT_NAMES = {ACT_SOFTMAX: "softmax", ACT_SILU: "silu", ACT_GELU_TANH: "gelu", ACT_IDENTITY: "identity",
             ACT_GELU_ERF: "gelu_erf"}


def _bf16_randn(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16).double().numpy()


def _offsets(lengths):
    o = np.zeros(len(lengths) + 1, dtype=np.int32)
    o[1:] = np.cumsum(lengths)
    return o


def _relpos_mask(table_h, Lq, Lkv, max_rel):
    i = np.arange(Lq)[:, None]
    j = np.arange(Lkv)[None, :]
    idx = np.clip(i - j + max_rel - 1, 0, 2 * max_rel - 2)
    return table_h[idx]


# --------------------------------------------------------------- golden cases
def _expr(s):
    return eval(s, {"log": math.log, "sqrt": math.sqrt})  # literal arithmetic from the fixture


def _golden_cases():
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_hand_worked_examples(oracle_mod, case):
    q = np.array(case["q"], dtype=np.float64)
    k = np.array(_expr(case["k_expr"]) if "k_expr" in case else case["k"], dtype=np.float64)
    v = np.array(case["v"], dtype=np.float64)
    qo, ko = _offsets(case["lq"]), _offsets(case["lkv"])
    bias = np.array(case["bias_table"]) if "bias_table" in case else None
    out, lse = oracle_mod.fwd(q, qo, k, v, ko, act=case["act"], causal=case["causal"],
                              scale=_expr(case["scale_expr"]), bias=bias,
                              max_rel=case.get("max_rel", 0))
    exp_out = np.array(_expr(case["out_expr"]) if "out_expr" in case else case["out"])
    np.testing.assert_allclose(out, exp_out, rtol=1e-13, atol=1e-13)
    if "lse" in case:
        exp_lse = np.array([[float(x) for x in row] for row in case["lse"]])
        np.testing.assert_allclose(lse, exp_lse, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------- library pins
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_softmax_matches_torch_sdpa(oracle_mod, with_bias, causal):
    H, d, max_rel = 2, 16, 8
    lq = [5, 0, 17, 1, 12]
    lkv = lq if causal else [9, 3, 12, 0, 20]
    q = _bf16_randn((sum(lq), H, d), 1)
    k = _bf16_randn((sum(lkv), H, d), 2)
    v = _bf16_randn((sum(lkv), H, d), 3)
    table = np.random.default_rng(4).normal(0, 0.5, size=(H, 2 * max_rel - 1)) if with_bias else None
    qo, ko = _offsets(lq), _offsets(lkv)
    scale = 1 / math.sqrt(d)
    out, lse = oracle_mod.fwd(q, qo, k, v, ko, act=ACT_SOFTMAX, causal=causal, scale=scale,
                              bias=table, max_rel=max_rel)
    for b in range(len(lq)):
        Lq, Lkv = lq[b], lkv[b]
        if Lq == 0:
            continue
        qb = torch.from_numpy(q[qo[b]:qo[b + 1]]).permute(1, 0, 2)[None]
        kb = torch.from_numpy(k[ko[b]:ko[b + 1]]).permute(1, 0, 2)[None]
        vb = torch.from_numpy(v[ko[b]:ko[b + 1]]).permute(1, 0, 2)[None]
        if Lkv == 0:
            np.testing.assert_array_equal(out[qo[b]:qo[b + 1]], 0.0)
            assert np.all(np.isneginf(lse[:, qo[b]:qo[b + 1]]))
            continue
        mask = np.zeros((H, Lq, Lkv))
        if with_bias:
            mask += np.stack([_relpos_mask(table[h], Lq, Lkv, max_rel) for h in range(H)])
        if causal:
            mask += np.where(np.arange(Lkv)[None, :] > np.arange(Lq)[:, None], -np.inf, 0.0)[None]
        m = torch.from_numpy(mask)[None]
        ref = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=m, scale=scale)
        ref = ref[0].permute(1, 0, 2).numpy()
        np.testing.assert_allclose(out[qo[b]:qo[b + 1]], ref, rtol=1e-11, atol=1e-12)
        logits = scale * torch.einsum("bhqd,bhkd->bhqk", qb, kb) + m
        ref_lse = torch.logsumexp(logits, dim=-1)[0].numpy()
        np.testing.assert_allclose(lse[:, qo[b]:qo[b + 1]], ref_lse, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", [ACT_SILU, ACT_GELU_TANH, ACT_IDENTITY, ACT_GELU_ERF])
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_gdpa_activation_via_onehot_values(oracle_mod, act, with_bias, causal):
    """With v_j = e_j (one-hot rows) the output row is the activated score row,
    so the oracle's activation and masking meet torch's fp64 SiLU/GELU."""
    H, d, max_rel = 2, 32, 6
    lq = [7, 3, 20] if not causal else [7, 3, 20]
    lkv = [11, 1, 32] if not causal else lq
    q = _bf16_randn((sum(lq), H, d), 5)
    k = _bf16_randn((sum(lkv), H, d), 6, scale=0.7)
    v = np.zeros((sum(lkv), H, d))
    qo, ko = _offsets(lq), _offsets(lkv)
    for b in range(len(lq)):
        for j in range(lkv[b]):
            v[ko[b] + j, :, j] = 1.0
    table = np.random.default_rng(7).normal(0, 0.3, size=(H, 2 * max_rel - 1)) if with_bias else None
    scale = 0.37
    out, _ = oracle_mod.fwd(q, qo, k, v, ko, act=act, causal=causal, scale=scale, bias=table,
                            max_rel=max_rel)
    tact = {ACT_SILU: F.silu, ACT_GELU_TANH: lambda x: F.gelu(x, approximate="tanh"),
            ACT_IDENTITY: lambda x: x, ACT_GELU_ERF: lambda x: F.gelu(x, approximate="none")}[act]
    for b in range(len(lq)):
        qb = torch.from_numpy(q[qo[b]:qo[b + 1]])
        kb = torch.from_numpy(k[ko[b]:ko[b + 1]])
        s = scale * torch.einsum("qhd,khd->hqk", qb, kb)
        if with_bias:
            s = s + torch.from_numpy(np.stack([_relpos_mask(table[h], lq[b], lkv[b], max_rel)
                                               for h in range(H)]))
        p = tact(s)
        if causal:
            p = p * (torch.arange(lkv[b])[None, :] <= torch.arange(lq[b])[:, None])
        got = out[qo[b]:qo[b + 1], :, :lkv[b]].transpose(1, 0, 2)
        np.testing.assert_allclose(got, p.numpy(), rtol=1e-12, atol=1e-13)
        np.testing.assert_array_equal(out[qo[b]:qo[b + 1], :, lkv[b]:], 0.0)


def test_identity_activation_associativity(oracle_mod):
    """Identity activation: O = (scale Q K^T) V must equal scale Q (K^T V)."""
    H, d = 3, 24
    lq, lkv = [9, 4, 30], [14, 25, 6]
    q = _bf16_randn((sum(lq), H, d), 8)
    k = _bf16_randn((sum(lkv), H, d), 9)
    v = _bf16_randn((sum(lkv), H, d), 10)
    qo, ko = _offsets(lq), _offsets(lkv)
    out, _ = oracle_mod.fwd(q, qo, k, v, ko, act=ACT_IDENTITY, scale=0.125)
    for b in range(3):
        for h in range(H):
            Q = q[qo[b]:qo[b + 1], h]
            K = k[ko[b]:ko[b + 1], h]
            V = v[ko[b]:ko[b + 1], h]
            ref = 0.125 * (Q @ (K.T @ V))
            np.testing.assert_allclose(out[qo[b]:qo[b + 1], h], ref, rtol=1e-12, atol=1e-11)


# --------------------------------------------------------------- closed forms
@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_SILU, ACT_GELU_TANH])
def test_zero_keys(oracle_mod, act):
    """K = 0, no bias: softmax gives the mean of V; SiLU/GELU give act(0) = 0."""
    H, d = 2, 8
    lq, lkv = [3, 5], [4, 7]
    q = _bf16_randn((8, H, d), 11)
    k = np.zeros((11, H, d))
    v = _bf16_randn((11, H, d), 12)
    qo, ko = _offsets(lq), _offsets(lkv)
    out, lse = oracle_mod.fwd(q, qo, k, v, ko, act=act, scale=0.3)
    for b in range(2):
        if act == ACT_SOFTMAX:
            mean = v[ko[b]:ko[b + 1]].mean(axis=0)
            np.testing.assert_allclose(out[qo[b]:qo[b + 1]], np.broadcast_to(mean, (lq[b], H, d)),
                                       rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(lse[:, qo[b]:qo[b + 1]], math.log(lkv[b]), rtol=1e-14)
        else:
            np.testing.assert_array_equal(out[qo[b]:qo[b + 1]], 0.0)


def test_single_key_and_constant_values(oracle_mod):
    H, d = 2, 8
    q = _bf16_randn((6, H, d), 13)
    k = _bf16_randn((6, H, d), 14)
    v = _bf16_randn((6, H, d), 15)
    # one key per sample: softmax output is that key's value row exactly
    out, _ = oracle_mod.fwd(q, _offsets([4, 2]), k[:2], v[:2], _offsets([1, 1]), act=ACT_SOFTMAX,
                            scale=1.0)
    np.testing.assert_array_equal(out[:4], np.broadcast_to(v[0], (4, H, d)))
    np.testing.assert_array_equal(out[4:], np.broadcast_to(v[1], (2, H, d)))
    # constant value rows: softmax output equals that row for any scores
    vc = np.broadcast_to(v[3], (6, H, d)).copy()
    out, _ = oracle_mod.fwd(q, _offsets([6]), k, vc, _offsets([6]), act=ACT_SOFTMAX, scale=2.0)
    np.testing.assert_allclose(out, vc, rtol=1e-13, atol=1e-14)
    # scale 0: uniform weights
    out, lse = oracle_mod.fwd(q, _offsets([6]), k, v, _offsets([6]), act=ACT_SOFTMAX, scale=0.0)
    np.testing.assert_allclose(out, np.broadcast_to(v.mean(0), (6, H, d)), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(6), rtol=1e-14)


def test_causal_closed_form(oracle_mod):
    """K = 0 and one-hot V under the causal mask: o_ij = 1/(i+1) for j <= i."""
    L, H, d = 9, 1, 16
    q = _bf16_randn((L, H, d), 16)
    k = np.zeros((L, H, d))
    v = np.zeros((L, H, d))
    for j in range(L):
        v[j, 0, j] = 1.0
    out, lse = oracle_mod.fwd(q, _offsets([L]), k, v, _offsets([L]), act=ACT_SOFTMAX, causal=True,
                              scale=1.0)
    ref = np.tril(np.ones((L, L))) / np.arange(1, L + 1)[:, None]
    np.testing.assert_allclose(out[:, 0, :L], ref, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse[0], np.log(np.arange(1, L + 1)), rtol=1e-14, atol=1e-15)


def test_relpos_index_closed_form(oracle_mod):
    """q = k = 0, identity act, one-hot V: o_ij = table[clamp(i - j + max_rel - 1)]."""
    max_rel, L = 5, 12
    table = np.arange(2 * max_rel - 1, dtype=np.float64)[None, :] * 10.0 + 1.0
    q = np.zeros((L, 1, L))
    k = np.zeros((L, 1, L))
    v = np.eye(L)[:, None, :]
    out, _ = oracle_mod.fwd(q, _offsets([L]), k, v, _offsets([L]), act=ACT_IDENTITY, scale=1.0,
                            bias=table, max_rel=max_rel)
    for i in range(L):
        for j in range(L):
            idx = min(max(i - j + max_rel - 1, 0), 2 * max_rel - 2)
            assert out[i, 0, j] == 10.0 * idx + 1.0


def test_softmax_rows_sum_to_one(oracle_mod):
    H, d = 2, 8
    lq, lkv = [5, 9, 2], [7, 3, 16]
    q = _bf16_randn((sum(lq), H, d), 17, scale=3.0)
    k = _bf16_randn((sum(lkv), H, d), 18, scale=3.0)
    v = np.ones((sum(lkv), H, d))
    table = np.random.default_rng(0).normal(size=(H, 15))
    out, _ = oracle_mod.fwd(q, _offsets(lq), k, v, _offsets(lkv), act=ACT_SOFTMAX, scale=0.5,
                            bias=table, max_rel=8)
    np.testing.assert_allclose(out, 1.0, rtol=1e-13)


# --------------------------------------------------------------- invariants
@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_SILU])
def test_sample_permutation_and_per_sample_equality(oracle_mod, act):
    H, d = 2, 16
    lq, lkv = [6, 0, 13, 3], [4, 9, 0, 11]
    q = _bf16_randn((sum(lq), H, d), 19)
    k = _bf16_randn((sum(lkv), H, d), 20)
    v = _bf16_randn((sum(lkv), H, d), 21)
    qo, ko = _offsets(lq), _offsets(lkv)
    out, lse = oracle_mod.fwd(q, qo, k, v, ko, act=act, scale=0.25)
    # each sample alone equals its slice of the jagged result
    for b in range(4):
        ob, lb = oracle_mod.fwd(q[qo[b]:qo[b + 1]], _offsets([lq[b]]), k[ko[b]:ko[b + 1]],
                                v[ko[b]:ko[b + 1]], _offsets([lkv[b]]), act=act, scale=0.25)
        np.testing.assert_array_equal(out[qo[b]:qo[b + 1]], ob)
        np.testing.assert_array_equal(lse[:, qo[b]:qo[b + 1]], lb)
    # permuting samples permutes the outputs
    perm = [2, 0, 3, 1]
    qp = np.concatenate([q[qo[b]:qo[b + 1]] for b in perm])
    kp = np.concatenate([k[ko[b]:ko[b + 1]] for b in perm])
    vp = np.concatenate([v[ko[b]:ko[b + 1]] for b in perm])
    op, _ = oracle_mod.fwd(qp, _offsets([lq[b] for b in perm]), kp, vp,
                           _offsets([lkv[b] for b in perm]), act=act, scale=0.25)
    np.testing.assert_array_equal(op, np.concatenate([out[qo[b]:qo[b + 1]] for b in perm]))


def test_zero_length_writes_nothing(oracle_mod):
    """A sample with no keys (GDPA) gives zero rows; samples with no queries
    leave every other row untouched."""
    H, d = 1, 8
    lq, lkv = [3, 0, 2], [0, 5, 4]
    q = _bf16_randn((5, H, d), 22)
    k = _bf16_randn((9, H, d), 23)
    v = _bf16_randn((9, H, d), 24)
    out, _ = oracle_mod.fwd(q, _offsets(lq), k, v, _offsets(lkv), act=ACT_SILU, scale=0.3)
    np.testing.assert_array_equal(out[:3], 0.0)
    o2, _ = oracle_mod.fwd(q[3:], _offsets([2]), k[5:], v[5:], _offsets([4]), act=ACT_SILU,
                           scale=0.3)
    np.testing.assert_array_equal(out[3:], o2)


def test_rejects_bad_offsets(oracle_mod):
    q = np.zeros((3, 1, 4))
    with pytest.raises(ValueError):
        oracle_mod.fwd(q, np.array([0, 2, 1, 3], dtype=np.int32), q, q,
                       np.array([0, 1, 2, 3], dtype=np.int32), act=0, scale=1.0)
    with pytest.raises(ValueError):  # causal needs equal lengths
        oracle_mod.fwd(q, np.array([0, 1, 3], dtype=np.int32), q, q,
                       np.array([0, 2, 3], dtype=np.int32), act=0, causal=True, scale=1.0)


# --------------------------------------------------------------- backward (finite differences)
@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_SILU, ACT_GELU_TANH, ACT_IDENTITY, ACT_GELU_ERF])
@pytest.mark.parametrize("variant", ["plain", "bias", "causal_bias"])
def test_backward_matches_central_differences(oracle_mod, act, variant):
    H, d, max_rel = 2, 6, 3
    causal = variant == "causal_bias"
    lq = [3, 4, 0]
    lkv = lq if causal else [5, 2, 3]
    rng = np.random.default_rng(100 + act)
    q = rng.normal(size=(sum(lq), H, d))
    k = rng.normal(size=(sum(lkv), H, d))
    v = rng.normal(size=(sum(lkv), H, d))
    do = rng.normal(size=(sum(lq), H, d))
    table = rng.normal(0, 0.5, size=(H, 2 * max_rel - 1)) if variant != "plain" else None
    qo, ko = _offsets(lq), _offsets(lkv)
    kw = dict(act=act, causal=causal, scale=0.45, bias=table, max_rel=max_rel)
    dq, dk, dv = oracle_mod.bwd(q, qo, k, v, ko, do, **kw)

    def loss(qq, kk, vv):
        o, _ = oracle_mod.fwd(qq, qo, kk, vv, ko, **kw)
        return float(np.sum(o * do))

    h = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(num - g).max() / max(1.0, np.abs(num).max())
        assert err < 1e-7, f"d{name}: {err}"


# --------------------------------------------------------------- MXFP8 (OCP)
def test_e4m3_spec_values(oracle_mod):
    enc = oracle_mod.e4m3_encode
    assert enc(0.0) == 0x00
    assert enc(1.0) == 0x38            # exponent field 7, mantissa 0
    assert enc(448.0) == 0x7E          # largest normal S.1111.110
    assert enc(-448.0) == 0xFE
    assert enc(2.0 ** -6) == 0x08      # smallest normal
    assert enc(2.0 ** -9) == 0x01      # smallest subnormal
    assert enc(1.0 + 1 / 16) == 0x38   # tie between 1 and 1.125 -> even (1.0)
    assert enc(1.0 + 3 / 16) == 0x3A   # tie between 1.125 and 1.25 -> even (1.25)
    assert enc(1000.0) == 0x7E         # saturates
    assert enc(-1e30) == 0xFE
    assert enc(float("nan")) == 0x7F
    assert enc(2.0 ** -11) == 0x00     # below half the smallest subnormal rounds to 0
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            assert math.isnan(oracle_mod.e4m3_decode(c))
        elif c != 0x80:
            assert enc(oracle_mod.e4m3_decode(c)) == c


def test_e4m3_matches_torch_float8(oracle_mod):
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.normal(0, 50, 4000), rng.normal(0, 0.01, 2000),
                        rng.uniform(-448, 448, 2000), np.linspace(-448, 448, 4097)])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.e4m3_encode(t) for t in x], dtype=np.uint8)
    # torch keeps the sign of a value that rounds to zero; so does the oracle
    np.testing.assert_array_equal(got, ref)


def test_e8m0_scale_closed_forms(oracle_mod):
    s = oracle_mod.e8m0_scale
    assert s(1.0) == 127 - 8
    assert s(3.0) == 127 + 1 - 8
    assert s(448.0) == 127
    assert s(511.9) == 127 + 8 - 8
    assert s(512.0) == 127 + 9 - 8
    assert s(2.0 ** -3) == 127 - 3 - 8
    assert s(0.0) == 0
    assert s(2.0 ** -140) == 0
    assert s(2.0 ** 200) == 254


def test_quant_rows_roundtrip_and_blocks(oracle_mod):
    T, H, d = 5, 2, 64
    x = _bf16_randn((T, H, d), 30) * np.exp2(np.arange(d) // 32)[None, None, :] * 3
    codes, scales = oracle_mod.quant_rows(x)
    assert scales.shape == (T, H, 2)
    dec = np.vectorize(oracle_mod.e4m3_decode)(codes)
    X = np.exp2(scales.astype(np.float64) - 127).repeat(32, axis=2)
    xr = dec * X
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 on normals, plus half a
    # subnormal step.  The scale 2^(floor(log2 amax) - 8) maps a block's largest
    # magnitude into [256, 512), so scaled values above 448 saturate to 448.
    sat = np.abs(x) / X > 448.0
    np.testing.assert_array_equal(np.abs(xr[sat]), 448.0 * X[sat])
    ok = np.abs(xr - x) <= 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * X
    assert np.all(ok | sat)
    amax = np.abs(x).reshape(T, H, 2, 32).max(-1)
    np.testing.assert_array_equal(scales, np.floor(np.log2(amax)).astype(int) - 8 + 127)


def test_quant_cols_sample_aligned_blocks(oracle_mod):
    """V blocks start at each sample's first token: sample b is filled with
    +-2^b so every one of its blocks must carry scale code b - 8 + 127, and
    a block straddling two samples would show the wrong code."""
    lengths = [5, 40, 33, 0, 64]
    H, d = 2, 4
    o = _offsets(lengths)
    x = np.zeros((sum(lengths), H, d))
    rng = np.random.default_rng(1)
    for b, L in enumerate(lengths):
        x[o[b]:o[b + 1]] = rng.choice([-1.0, 1.0], size=(L, H, d)) * 2.0 ** b
    codes, scales = oracle_mod.quant_cols(x, o)
    nb = [(L + 31) // 32 for L in lengths]
    assert scales.shape[0] == sum(nb)
    r = 0
    for b in range(len(lengths)):
        for _ in range(nb[b]):
            np.testing.assert_array_equal(scales[r], b - 8 + 127)
            r += 1
    dec = np.vectorize(oracle_mod.e4m3_decode)(codes)
    # every element is +-2^b = +-2^8 * 2^(b-8): code 256 -> 0x78 with sign
    np.testing.assert_array_equal(np.abs(dec), 256.0)


def _nosat_exponent(amax):
    """Least integer e with amax <= 448 * 2^e, from frexp (amax = f 2^k, f in
    [0.5, 1)): 448 2^e = 0.875 2^(e+9), so e = k - 9 when f <= 0.875, else k - 8."""
    f, k = np.frexp(amax)
    return np.where(f <= 0.875, k - 9, k - 8)


def test_quant_rows_nosat_against_torch_float8(oracle_mod):
    """The saturation-free quantiser along channels: each 32-channel block is
    divided by 2^e with e the least exponent keeping its maximum at or below
    448, then rounded as torch's float8_e4m3fn conversion rounds; no element
    saturates, and the scale is the OCP one or one step above it."""
    T, H, d = 7, 3, 64
    x = _bf16_randn((T, H, d), 31) * np.exp2(np.arange(d) // 32 * 3)[None, None, :]
    x[0, 0, :32] = 1.875 * 2.0 ** 4                    # mantissa above 1.75: OCP would clip
    x[1, 1, 32:] = 0.0                                 # all-zero block
    codes, scales = oracle_mod.quant_rows(x, nosat=True)
    blocks = x.reshape(T, H, 2, 32)
    amax = np.abs(blocks).max(-1)
    e = np.where(amax > 0, _nosat_exponent(np.where(amax > 0, amax, 1.0)), -127)
    np.testing.assert_array_equal(scales.astype(int), e + 127)
    X = np.exp2(e)[..., None]
    ref = torch.from_numpy(blocks / X).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes, ref.reshape(T, H, d))
    assert np.all(np.abs(blocks / X) <= 448.0)
    _, ocp = oracle_mod.quant_rows(x)
    step = scales.astype(int) - ocp.astype(int)
    assert np.all((step == 0) | (step == 1)) and step[0, 0, 0] == 1
    # the clipped block decodes exactly with the saturation-free scale
    dec = np.vectorize(oracle_mod.e4m3_decode)(codes[0, 0, :32]) * 2.0 ** (int(scales[0, 0, 0]) - 127)
    np.testing.assert_array_equal(dec, x[0, 0, :32])


def test_quant_cols_nosat_against_torch_float8(oracle_mod):
    """Saturation-free quantiser along tokens: the same rule on 32-token blocks
    aligned to each sample's first token (the last block partial)."""
    lengths = [5, 40, 33, 0, 64]
    H, d = 2, 8
    o = _offsets(lengths)
    x = _bf16_randn((sum(lengths), H, d), 32) * 7.0
    codes, scales = oracle_mod.quant_cols(x, o, nosat=True)
    r = 0
    for b, L in enumerate(lengths):
        for t0 in range(int(o[b]), int(o[b + 1]), 32):
            blk = x[t0:min(t0 + 32, int(o[b + 1]))]
            amax = np.abs(blk).max(0)
            e = _nosat_exponent(amax)
            np.testing.assert_array_equal(scales[r].astype(int), e + 127)
            ref = torch.from_numpy(blk / np.exp2(e)).to(torch.float8_e4m3fn).view(torch.uint8)
            np.testing.assert_array_equal(codes[t0:t0 + len(blk)], ref.numpy())
            r += 1
    assert r == scales.shape[0]


# --------------------------------------------------------------- sliding window
def _band(L, window, causal):
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    keep = np.abs(i - j) < window
    if causal:
        keep &= j <= i
    return keep


@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [1, 3, 8])
def test_window_softmax_matches_torch_sdpa(oracle_mod, window, causal, with_bias):
    """The windowed softmax rows equal torch's fp64 SDPA under a band mask."""
    H, d, max_rel = 2, 16, 6
    lq = [5, 0, 17, 1, 12]
    q = _bf16_randn((sum(lq), H, d), 41)
    k = _bf16_randn((sum(lq), H, d), 42)
    v = _bf16_randn((sum(lq), H, d), 43)
    table = np.random.default_rng(44).normal(0, 0.5, size=(H, 2 * max_rel - 1)) if with_bias else None
    qo = _offsets(lq)
    scale = 1 / math.sqrt(d)
    out, lse = oracle_mod.fwd(q, qo, k, v, qo, act=ACT_SOFTMAX, causal=causal, scale=scale,
                              bias=table, max_rel=max_rel, window=window)
    for b, L in enumerate(lq):
        if L == 0:
            continue
        sl = slice(qo[b], qo[b + 1])
        qb, kb, vb = (torch.from_numpy(x[sl]).permute(1, 0, 2)[None] for x in (q, k, v))
        mask = np.where(_band(L, window, causal), 0.0, -np.inf)[None].repeat(H, 0)
        if with_bias:
            mask = mask + np.stack([_relpos_mask(table[h], L, L, max_rel) for h in range(H)])
        m = torch.from_numpy(mask)[None]
        ref = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=m, scale=scale)
        np.testing.assert_allclose(out[sl], ref[0].permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)
        ref_lse = torch.logsumexp(scale * torch.einsum("bhqd,bhkd->bhqk", qb, kb) + m, dim=-1)
        np.testing.assert_allclose(lse[:, sl], ref_lse[0].numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", [ACT_SILU, ACT_GELU_TANH, ACT_IDENTITY])
@pytest.mark.parametrize("causal", [False, True])
def test_window_gdpa_onehot_values(oracle_mod, act, causal):
    """One-hot values: output row i is act(s_ij) on the band and exactly 0 off it."""
    H, W, max_rel = 1, 4, 5
    L = d = 13
    q = _bf16_randn((L, H, d), 45)
    k = _bf16_randn((L, H, d), 46)
    v = np.eye(L)[:, None, :]
    table = np.random.default_rng(47).normal(0, 0.5, size=(H, 2 * max_rel - 1))
    out, _ = oracle_mod.fwd(q, _offsets([L]), k, v, _offsets([L]), act=act, causal=causal,
                            scale=0.3, bias=table, max_rel=max_rel, window=W)
    s = 0.3 * torch.einsum("qd,kd->qk", torch.from_numpy(q[:, 0]), torch.from_numpy(k[:, 0]))
    s = s + torch.from_numpy(_relpos_mask(table[0], L, L, max_rel))
    a = {ACT_SILU: F.silu, ACT_GELU_TANH: lambda x: F.gelu(x, approximate="tanh"),
         ACT_IDENTITY: lambda x: x}[act](s).numpy()
    ref = np.where(_band(L, W, causal), a, 0.0)
    np.testing.assert_allclose(out[:, 0, :], ref, rtol=1e-13, atol=1e-14)


def test_window_closed_forms(oracle_mod):
    """K = 0 and one-hot V: the causal window averages the last min(i+1, W)
    positions; window 1 returns v_i with lse = s_ii; a window at least as long
    as the sample changes nothing."""
    L, H, W = 11, 1, 4
    d = L
    q = _bf16_randn((L, H, d), 48)
    k = np.zeros((L, H, d))
    v = np.eye(L)[:, None, :]
    o = _offsets([L])
    out, lse = oracle_mod.fwd(q, o, k, v, o, act=ACT_SOFTMAX, causal=True, scale=1.0, window=W)
    ref = np.zeros((L, L))
    for i in range(L):
        n = min(i + 1, W)
        ref[i, i - n + 1:i + 1] = 1.0 / n
    np.testing.assert_allclose(out[:, 0, :], ref, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse[0], np.log(np.minimum(np.arange(1, L + 1), W)), rtol=1e-14)
    kk = _bf16_randn((L, H, d), 49)
    vv = _bf16_randn((L, H, d), 50)
    for causal in (False, True):
        o1, l1 = oracle_mod.fwd(q, o, kk, vv, o, act=ACT_SOFTMAX, causal=causal, scale=0.7,
                                window=1)
        np.testing.assert_array_equal(o1, vv)
        np.testing.assert_allclose(l1[0], 0.7 * np.einsum("id,id->i", q[:, 0], kk[:, 0]),
                                   rtol=1e-14, atol=1e-14)
        full, lf = oracle_mod.fwd(q, o, kk, vv, o, act=ACT_SOFTMAX, causal=causal, scale=0.7)
        wide, lw = oracle_mod.fwd(q, o, kk, vv, o, act=ACT_SOFTMAX, causal=causal, scale=0.7,
                                  window=L)
        np.testing.assert_array_equal(wide, full)
        np.testing.assert_array_equal(lw, lf)


def test_window_row_equals_causal_attention_over_its_slice(oracle_mod):
    """Row i of causal window W sees exactly keys i-W+1..i, so it equals the
    last row of plain causal attention over that slice of the sample (the
    relative-position bias depends on i - j only and is unchanged)."""
    L, H, d, W, max_rel = 20, 2, 8, 6, 4
    q = _bf16_randn((L, H, d), 51)
    k = _bf16_randn((L, H, d), 52)
    v = _bf16_randn((L, H, d), 53)
    table = np.random.default_rng(54).normal(0, 0.5, size=(H, 2 * max_rel - 1))
    o = _offsets([L])
    kw = dict(scale=0.4, bias=table, max_rel=max_rel)
    for act in (ACT_SOFTMAX, ACT_SILU):
        out, lse = oracle_mod.fwd(q, o, k, v, o, act=act, causal=True, window=W, **kw)
        for i in range(L):
            a = max(0, i - W + 1)
            n = i + 1 - a
            os_, ls = oracle_mod.fwd(q[a:i + 1], _offsets([n]), k[a:i + 1], v[a:i + 1],
                                     _offsets([n]), act=act, causal=True, **kw)
            np.testing.assert_allclose(out[i], os_[-1], rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(lse[:, i], ls[:, -1], rtol=1e-13, atol=1e-14)


def test_window_rejects_bad_arguments(oracle_mod):
    q = np.zeros((3, 1, 4))
    with pytest.raises(ValueError):  # a window needs equal lengths
        oracle_mod.fwd(q, np.array([0, 1, 3], dtype=np.int32), q, q,
                       np.array([0, 2, 3], dtype=np.int32), act=0, scale=1.0, window=2)
    with pytest.raises(ValueError):
        oracle_mod.fwd(q, _offsets([3]), q, q, _offsets([3]), act=0, scale=1.0, window=-1)


@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_SILU, ACT_GELU_TANH])
@pytest.mark.parametrize("causal", [False, True])
def test_window_backward_matches_central_differences(oracle_mod, act, causal):
    H, d, max_rel, W = 2, 5, 3, 2
    lq = [4, 5, 0]
    rng = np.random.default_rng(200 + act + 10 * causal)
    q = rng.normal(size=(sum(lq), H, d))
    k = rng.normal(size=(sum(lq), H, d))
    v = rng.normal(size=(sum(lq), H, d))
    do = rng.normal(size=(sum(lq), H, d))
    table = rng.normal(0, 0.5, size=(H, 2 * max_rel - 1))
    qo = _offsets(lq)
    kw = dict(act=act, causal=causal, scale=0.45, bias=table, max_rel=max_rel, window=W)
    dq, dk, dv = oracle_mod.bwd(q, qo, k, v, qo, do, **kw)

    def loss(qq, kk, vv):
        o, _ = oracle_mod.fwd(qq, qo, kk, vv, qo, **kw)
        return float(np.sum(o * do))

    h = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(num - g).max() / max(1.0, np.abs(num).max())
        assert err < 1e-7, f"d{name}: {err}"


# --------------------------------------------------------------- block-aligned attention
@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_SILU])
@pytest.mark.parametrize("causal", [False, True])
def test_blocks_equal_separate_samples(oracle_mod, act, causal):
    """Cutting every sample into blocks of K tokens from its first token and
    attending inside each block is the same as running each block as a sample
    of its own (the relative-position bias depends on i - j only)."""
    H, d, K, max_rel = 2, 8, 5, 4
    lq = [12, 0, 5, 1, 9]
    q = _bf16_randn((sum(lq), H, d), 61)
    k = _bf16_randn((sum(lq), H, d), 62)
    v = _bf16_randn((sum(lq), H, d), 63)
    table = np.random.default_rng(64).normal(0, 0.5, size=(H, 2 * max_rel - 1))
    o = _offsets(lq)
    kw = dict(act=act, causal=causal, scale=0.3, bias=table, max_rel=max_rel)
    out, lse = oracle_mod.fwd(q, o, k, v, o, block=K, **kw)
    pieces = [min(K, L - s) for L in lq for s in range(0, L, K)]
    ob = _offsets(pieces)
    ref, rl = oracle_mod.fwd(q, ob, k, v, ob, **kw)
    np.testing.assert_array_equal(out, ref)
    np.testing.assert_array_equal(lse, rl)


@pytest.mark.parametrize("causal", [False, True])
def test_blocks_softmax_matches_torch_sdpa(oracle_mod, causal):
    """Torch fp64 SDPA under a block-diagonal mask (blocks of 4 from the start)."""
    H, d, K, L = 2, 16, 4, 14
    q = _bf16_randn((L, H, d), 65)
    k = _bf16_randn((L, H, d), 66)
    v = _bf16_randn((L, H, d), 67)
    o = _offsets([L])
    out, lse = oracle_mod.fwd(q, o, k, v, o, act=ACT_SOFTMAX, causal=causal, scale=0.25, block=K)
    i, j = np.arange(L)[:, None], np.arange(L)[None, :]
    keep = (i // K) == (j // K)
    if causal:
        keep &= j <= i
    m = torch.from_numpy(np.where(keep, 0.0, -np.inf))[None, None].expand(1, H, L, L)
    qb, kb, vb = (torch.from_numpy(x).permute(1, 0, 2)[None] for x in (q, k, v))
    ref = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=m, scale=0.25)
    np.testing.assert_allclose(out, ref[0].permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)
    ref_lse = torch.logsumexp(0.25 * torch.einsum("bhqd,bhkd->bhqk", qb, kb) + m, dim=-1)
    np.testing.assert_allclose(lse, ref_lse[0].numpy(), rtol=1e-12, atol=1e-13)


def test_blocks_closed_forms(oracle_mod):
    """K = 0 and one-hot V: row i averages its block's keys (1/len of the block,
    the last block shorter); block 1 returns v_i; a block as long as the sample
    changes nothing; blocks of 64 on a 150-token sample end at 64, 128, 150."""
    L = 150
    H = 1
    q = _bf16_randn((L, H, L), 68)
    k = np.zeros((L, H, L))
    v = np.eye(L)[:, None, :]
    o = _offsets([L])
    out, lse = oracle_mod.fwd(q, o, k, v, o, act=ACT_SOFTMAX, scale=1.0, block=64)
    ref = np.zeros((L, L))
    for s, e in ((0, 64), (64, 128), (128, 150)):
        ref[s:e, s:e] = 1.0 / (e - s)
    np.testing.assert_allclose(out[:, 0, :], ref, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse[0], np.log(np.repeat([64, 64, 22], [64, 64, 22])), rtol=1e-14)
    kk = _bf16_randn((L, H, L), 69)
    vv = _bf16_randn((L, H, L), 70)
    o1, _ = oracle_mod.fwd(q, o, kk, vv, o, act=ACT_SOFTMAX, scale=0.1, block=1)
    np.testing.assert_array_equal(o1, vv)
    full, lf = oracle_mod.fwd(q, o, kk, vv, o, act=ACT_SILU, scale=0.1)
    wide, lw = oracle_mod.fwd(q, o, kk, vv, o, act=ACT_SILU, scale=0.1, block=L)
    np.testing.assert_array_equal(wide, full)


def test_blocks_reject_bad_arguments(oracle_mod):
    q = np.zeros((3, 1, 4))
    with pytest.raises(ValueError):
        oracle_mod.fwd(q, np.array([0, 1, 3], dtype=np.int32), q, q,
                       np.array([0, 2, 3], dtype=np.int32), act=0, scale=1.0, block=2)
    with pytest.raises(ValueError):
        oracle_mod.fwd(q, _offsets([3]), q, q, _offsets([3]), act=0, scale=1.0, block=-2)


@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_GELU_TANH])
@pytest.mark.parametrize("causal", [False, True])
def test_blocks_backward_matches_central_differences(oracle_mod, act, causal):
    H, d, max_rel, K = 2, 4, 3, 3
    lq = [7, 2]
    rng = np.random.default_rng(300 + act + 10 * causal)
    q = rng.normal(size=(sum(lq), H, d))
    k = rng.normal(size=(sum(lq), H, d))
    v = rng.normal(size=(sum(lq), H, d))
    do = rng.normal(size=(sum(lq), H, d))
    table = rng.normal(0, 0.5, size=(H, 2 * max_rel - 1))
    qo = _offsets(lq)
    kw = dict(act=act, causal=causal, scale=0.45, bias=table, max_rel=max_rel, block=K)
    dq, dk, dv = oracle_mod.bwd(q, qo, k, v, qo, do, **kw)

    def loss(qq, kk, vv):
        o_, _ = oracle_mod.fwd(qq, qo, kk, vv, qo, **kw)
        return float(np.sum(o_ * do))

    h = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(num - g).max() / max(1.0, np.abs(num).max())
        assert err < 1e-7, f"d{name}: {err}"


def test_gelu_forms_differ_and_match_their_definitions(oracle_mod):
    """Single key, one-hot value: the output is act(s) for the scalar score s,
    checked against math.erf / math.tanh directly; the two GELU forms differ by
    up to about 1e-3 (so a swapped form fails)."""
    xs = np.linspace(-6, 6, 49)
    d = 4
    q = np.zeros((len(xs), 1, d))
    q[:, 0, 0] = xs
    k = np.zeros((len(xs), 1, d))
    k[:, 0, 0] = 1.0
    v = np.zeros((len(xs), 1, d))
    v[:, 0, 1] = 1.0
    o = _offsets([1] * len(xs))
    out_e, _ = oracle_mod.fwd(q, o, k, v, o, act=ACT_GELU_ERF, scale=1.0)
    out_t, _ = oracle_mod.fwd(q, o, k, v, o, act=ACT_GELU_TANH, scale=1.0)
    ref_e = [0.5 * x * (1 + math.erf(x / math.sqrt(2))) for x in xs]
    ref_t = [0.5 * x * (1 + math.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3))) for x in xs]
    np.testing.assert_allclose(out_e[:, 0, 1], ref_e, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(out_t[:, 0, 1], ref_t, rtol=1e-14, atol=1e-15)
    assert np.abs(out_e - out_t).max() > 1e-4


# --------------------------------------------------------------- rotary embedding
def test_rope_closed_form_and_identities(oracle_mod):
    """d = 2: one pair rotated by exactly pos radians (theta_0 = 1); position 0 is
    the identity; the backward is the inverse (R is orthogonal), so it undoes the
    forward and keeps norms."""
    x = np.array([[[1.0, 0.0]], [[0.0, 1.0]], [[0.6, -0.8]], [[2.0, 3.0]]])
    o = _offsets([4])
    y = oracle_mod.rope_fwd(x, o, 10000.0)
    for p_, (a, b) in enumerate(x[:, 0]):
        np.testing.assert_allclose(y[p_, 0], [a * math.cos(p_) - b * math.sin(p_),
                                              a * math.sin(p_) + b * math.cos(p_)], rtol=1e-15, atol=1e-15)
    lengths = [5, 0, 9]
    z = _bf16_randn((sum(lengths), 3, 16), 80)
    oo = _offsets(lengths)
    rz = oracle_mod.rope_fwd(z, oo, 500.0)
    np.testing.assert_array_equal(rz[0], z[0])        # sample 0, position 0
    np.testing.assert_array_equal(rz[5], z[5])        # sample 2 restarts at position 0
    np.testing.assert_allclose(oracle_mod.rope_bwd(rz, oo, 500.0), z, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(np.linalg.norm(rz, axis=-1), np.linalg.norm(z, axis=-1), rtol=1e-13)


def test_rope_scores_depend_on_relative_position(oracle_mod):
    """RoPE's defining property: <R(m) q, R(n) k> depends on m - n only."""
    d, L = 32, 12
    q = _bf16_randn((1, 1, d), 81).repeat(L, 0)
    k = _bf16_randn((1, 1, d), 82).repeat(L, 0)
    o = _offsets([L])
    rq, rk = oracle_mod.rope_fwd(q, o, 10000.0), oracle_mod.rope_fwd(k, o, 10000.0)
    s = np.einsum("ic,jc->ij", rq[:, 0], rk[:, 0])
    for delta in range(-L + 1, L):
        diag = np.diagonal(s, offset=-delta)
        np.testing.assert_allclose(diag, diag[0], rtol=1e-12, atol=1e-12)


def test_rope_backward_is_the_gradient(oracle_mod):
    """<rope_fwd(x), g> differentiated by central differences equals rope_bwd(g)."""
    rng = np.random.default_rng(83)
    x = rng.normal(size=(7, 2, 8))
    g = rng.normal(size=(7, 2, 8))
    o = _offsets([3, 4])
    h = 1e-6
    num = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        xp = x.copy(); xp[idx] += h
        xm = x.copy(); xm[idx] -= h
        num[idx] = (np.sum(oracle_mod.rope_fwd(xp, o, 100.0) * g) -
                    np.sum(oracle_mod.rope_fwd(xm, o, 100.0) * g)) / (2 * h)
    np.testing.assert_allclose(oracle_mod.rope_bwd(g, o, 100.0), num, rtol=1e-8, atol=1e-8)


# --------------------------------------------------------------- bias table gradient
@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_SILU, ACT_GELU_TANH])
@pytest.mark.parametrize("variant", ["plain", "causal", "window", "clamped", "block"])
def test_dbias_matches_central_differences(oracle_mod, act, variant):
    """The bias table's gradient against central differences of the forward in
    every table entry (a 'clamped' table is shorter than the samples, so its end
    entries collect many offsets; 'block' keeps pairs inside 3-token blocks)."""
    H, d = 2, 5
    max_rel = 2 if variant == "clamped" else 6
    lq = [4, 6, 0]
    causal = variant == "causal"
    window = 3 if variant == "window" else 0
    block = 3 if variant == "block" else 0
    lkv = lq if (causal or window or block) else [5, 3, 2]
    rng = np.random.default_rng(400 + act)
    q = rng.normal(size=(sum(lq), H, d))
    k = rng.normal(size=(sum(lkv), H, d))
    v = rng.normal(size=(sum(lkv), H, d))
    do = rng.normal(size=(sum(lq), H, d))
    table = rng.normal(0, 0.5, size=(H, 2 * max_rel - 1))
    qo, ko = _offsets(lq), _offsets(lkv)
    kw = dict(act=act, causal=causal, window=window, block=block, scale=0.45, max_rel=max_rel)
    *_, db = oracle_mod.bwd(q, qo, k, v, ko, do, bias=table, want_dbias=True, **kw)
    h = 1e-6
    num = np.zeros_like(table)
    for idx in np.ndindex(*table.shape):
        tp = table.copy(); tp[idx] += h
        tm = table.copy(); tm[idx] -= h
        op, _ = oracle_mod.fwd(q, qo, k, v, ko, bias=tp, **kw)
        om, _ = oracle_mod.fwd(q, qo, k, v, ko, bias=tm, **kw)
        num[idx] = (np.sum(op * do) - np.sum(om * do)) / (2 * h)
    np.testing.assert_allclose(db, num, rtol=1e-7, atol=1e-8)


# --------------------------------------------------------------- MXFP8 backward
def test_e8m0_nosat_closed_forms(oracle_mod):
    """The saturation-free block scale: the smallest power of two X with
    amax / X <= 448, against hand values and against the OCP rule, which it
    exceeds by one step exactly when the mantissa of amax is above 1.75."""
    s = oracle_mod.e8m0_nosat
    assert s(0.0) == 0
    assert s(448.0) == 127
    assert s(np.nextafter(448.0, np.inf)) == 128
    assert s(1.75) == 119                      # 1.75 / 2^-8 = 448
    assert s(np.nextafter(1.75, np.inf)) == 120
    assert s(1.0) == 119                       # 2^-9 would give 512 > 448
    assert s(2.0 ** -140) == 0                 # below the smallest scale: clamped
    assert s(2.0 ** 200) == 254
    for e in range(-100, 100):
        assert s(448.0 * 2.0 ** e) == 127 + e
        assert s(449.0 * 2.0 ** e) == 128 + e
    rng = np.random.default_rng(3)
    for a in np.exp(rng.uniform(-40, 40, 2000)):
        m = a / 2.0 ** math.floor(math.log2(a))
        assert s(a) - oracle_mod.e8m0_scale(a) == (1 if m > 1.75 else 0), a


def test_round_blocks_2d_against_torch_float8(oracle_mod):
    """32 x 32 blocks from (0, 0), edge blocks partial; each block divided by
    its own scale and rounded as torch's float8_e4m3fn conversion rounds."""
    rng = np.random.default_rng(4)
    R, C = 70, 45
    m = rng.standard_normal((R, C)) * np.exp2(rng.integers(-12, 12, (R, C)))
    m[40:64, 32:45] = 0.0                      # an all-zero block part
    r = oracle_mod.round_blocks_2d(m)
    for r0 in range(0, R, 32):
        for c0 in range(0, C, 32):
            blk = m[r0:r0 + 32, c0:c0 + 32]
            X = 2.0 ** (oracle_mod.e8m0_nosat(np.abs(blk).max()) - 127)
            assert np.abs(blk).max() / X <= 448.0
            ref = torch.from_numpy(blk / X).to(torch.float8_e4m3fn).double().numpy() * X
            np.testing.assert_array_equal(r[r0:r0 + 32, c0:c0 + 32], ref)
    np.testing.assert_array_equal(oracle_mod.round_blocks_2d(-m), -r)


def test_round_blocks_2d_block_independence(oracle_mod):
    rng = np.random.default_rng(6)
    m = rng.standard_normal((64, 64))
    r = oracle_mod.round_blocks_2d(m)
    m2 = m.copy()
    m2[31, 31] = 1e4                           # last element of block (0, 0)
    r2 = oracle_mod.round_blocks_2d(m2)
    changed = r2 != r
    assert changed[:32, :32].any()
    assert not changed[32:, :].any() and not changed[:, 32:].any()
    # values already on a block's grid stay exact (amax 448 X, X = 2^-3)
    g = np.array([oracle_mod.e4m3_decode(c) for c in range(0x00, 0x7F)])
    blk = rng.choice(g, size=(32, 32)) * rng.choice([-1.0, 1.0], size=(32, 32))
    blk[0, 0] = 448.0
    np.testing.assert_array_equal(oracle_mod.round_blocks_2d(blk * 2.0 ** -3), blk * 2.0 ** -3)


def _mx_inputs(lq, lkv, H, d, seed, causal, with_bias, oracle_mod):
    qo, ko = _offsets(lq), _offsets(lkv)
    q = _bf16_randn((sum(lq), H, d), seed)
    k = _bf16_randn((sum(lkv), H, d), seed + 1)
    v = _bf16_randn((sum(lkv), H, d), seed + 2)
    do = _bf16_randn((sum(lq), H, d), seed + 3)
    max_rel = 20 if with_bias else 0
    bias = np.random.default_rng(seed).normal(0, 0.5, (H, 2 * max_rel - 1)) if with_bias else None
    scale = 1.0 / math.sqrt(d)
    out, lse = oracle_mod.fwd(q, qo, k, v, ko, act=ACT_SOFTMAX, causal=causal, scale=scale,
                              bias=bias, max_rel=max_rel)
    delta = np.einsum("thc,thc->ht", do, out)
    return q, k, v, do, qo, ko, bias, max_rel, scale, out, lse, delta


@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_mx_operands_reduce_to_the_backward(oracle_mod, causal, with_bias):
    """With every operand version equal to the unquantised tensor, no rounding
    of P and dS, and the forward's lse and rowsum(dO * O), the MXFP8 backward's
    definition is the softmax backward (itself pinned by finite differences)."""
    lq = [5, 0, 37, 70, 1] if causal else [5, 3, 37, 70, 0]
    lkv = lq if causal else [9, 0, 33, 64, 4]
    H, d = 2, 8
    q, k, v, do, qo, ko, bias, max_rel, scale, out, lse, delta = _mx_inputs(
        lq, lkv, H, d, 11, causal, with_bias, oracle_mod)
    got = oracle_mod.bwd_mx_operands(q, q, k, k, v, do, do, qo, ko, lse, delta, causal=causal,
                                     scale=scale, bias=bias, max_rel=max_rel, round_ps=False)
    ref = oracle_mod.bwd(q, qo, k, v, ko, do, act=ACT_SOFTMAX, causal=causal, scale=scale,
                         bias=bias, max_rel=max_rel)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_mx_operands_dense_bias_reduces_to_the_backward(oracle_mod, causal):
    """The same reduction with a dense jagged bias: the MXFP8 backward's
    definition reads the bias of each pair where the dense backward does (that
    one pinned by finite differences and by torch's SDPA with the bias as a
    mask); a transposed or shifted index fails it."""
    lq = [5, 0, 37, 70, 1] if causal else [5, 3, 37, 70, 0]
    lkv = lq if causal else [9, 0, 33, 64, 4]
    H, d = 2, 8
    qo, ko = _offsets(lq), _offsets(lkv)
    q = _bf16_randn((sum(lq), H, d), 21)
    k = _bf16_randn((sum(lkv), H, d), 22)
    v = _bf16_randn((sum(lkv), H, d), 23)
    do = _bf16_randn((sum(lq), H, d), 24)
    off = oracle_mod.dense_bias_offsets(qo, ko, H)
    dense = np.random.default_rng(5).normal(0, 1.0, int(off[-1]))
    kw = dict(causal=causal, scale=1.0 / math.sqrt(d), dense_bias=dense)
    out, lse = oracle_mod.fwd(q, qo, k, v, ko, act=ACT_SOFTMAX, **kw)
    delta = np.einsum("thc,thc->ht", do, out)
    got = oracle_mod.bwd_mx_operands(q, q, k, k, v, do, do, qo, ko, lse, delta, round_ps=False,
                                     **kw)
    ref = oracle_mod.bwd(q, qo, k, v, ko, do, act=ACT_SOFTMAX, **kw)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-12)
    # the bias matters here: without it the result moves well past the tolerance
    plain = oracle_mod.bwd(q, qo, k, v, ko, do, act=ACT_SOFTMAX, causal=causal,
                           scale=1.0 / math.sqrt(d))
    assert max(np.abs(g - r).max() for g, r in zip(got, plain)) > 1e-3


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [1, 5, 40])
def test_bwd_mx_operands_window_reduces_to_the_windowed_backward(oracle_mod, window, causal):
    """The same reduction with a sliding window: the mask matches the windowed
    backward's (pinned against torch's banded SDPA and finite differences)."""
    lq = [5, 37, 70, 1]
    H, d = 2, 8
    qo = _offsets(lq)
    q = _bf16_randn((sum(lq), H, d), 41)
    k = _bf16_randn((sum(lq), H, d), 42)
    v = _bf16_randn((sum(lq), H, d), 43)
    do = _bf16_randn((sum(lq), H, d), 44)
    bias = np.random.default_rng(2).normal(0, 0.5, (H, 39))
    scale = 1.0 / math.sqrt(d)
    kw = dict(causal=causal, scale=scale, bias=bias, max_rel=20, window=window)
    out, lse = oracle_mod.fwd(q, qo, k, v, qo, act=ACT_SOFTMAX, **kw)
    delta = np.einsum("thc,thc->ht", do, out)
    got = oracle_mod.bwd_mx_operands(q, q, k, k, v, do, do, qo, qo, lse, delta, round_ps=False, **kw)
    ref = oracle_mod.bwd(q, qo, k, v, qo, do, act=ACT_SOFTMAX, **kw)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-12)


def test_bwd_mx_operands_wiring(oracle_mod):
    """Each token-contraction operand feeds one gradient, linearly; the channel
    operands of dP reach dQ and dK but not dV; and dV with distinct versions is
    the plain backward's dV on (qd, kd) with dout = dOt."""
    lq = [40, 7, 66]
    H, d = 2, 16
    q, k, v, do, qo, ko, bias, max_rel, scale, out, lse, delta = _mx_inputs(
        lq, lq, H, d, 21, True, True, oracle_mod)
    rng = np.random.default_rng(8)
    alt = {n: x + 0.1 * rng.standard_normal(x.shape) for n, x in
           (("qt", q), ("kt", k), ("dot", do), ("vd", v), ("dod", do))}
    ops = dict(qd=q, qt=alt["qt"], kd=k, kt=alt["kt"], vd=alt["vd"], dod=alt["dod"], dot=alt["dot"])
    kw = dict(causal=True, scale=scale, bias=bias, max_rel=max_rel, round_ps=False)
    order = ["qd", "qt", "kd", "kt", "vd", "dod", "dot"]

    def run(**over):
        o = dict(ops, **over)
        return oracle_mod.bwd_mx_operands(*[o[n] for n in order], qo, qo, lse, delta, **kw)

    dq, dk, dv = run()
    for name, which in (("qt", 1), ("kt", 0), ("dot", 2)):
        res = run(**{name: 2.0 * ops[name]})
        for i, (a, b) in enumerate(zip(res, (dq, dk, dv))):
            np.testing.assert_allclose(a, 2.0 * b if i == which else b, rtol=1e-12, atol=1e-14)
    for name in ("vd", "dod"):
        res = run(**{name: ops[name] + 0.3})
        np.testing.assert_array_equal(res[2], dv)
        assert not np.allclose(res[0], dq) and not np.allclose(res[1], dk)
    ref_dv = oracle_mod.bwd(q, qo, k, v, qo, alt["dot"], act=ACT_SOFTMAX, causal=True,
                            scale=scale, bias=bias, max_rel=max_rel)[2]
    np.testing.assert_allclose(dv, ref_dv, rtol=1e-10, atol=1e-12)


def test_bwd_mx_rounding_bound(oracle_mod):
    """Rounding P and dS moves each gradient by at most 2^-4 of the sum of the
    magnitudes of its terms (E4M3 keeps 3 mantissa bits; no block saturates),
    plus a subnormal allowance."""
    lq = [64, 33]
    H, d = 1, 16
    q, k, v, do, qo, ko, bias, max_rel, scale, out, lse, delta = _mx_inputs(
        lq, lq, H, d, 31, True, False, oracle_mod)
    args = (q, q, k, k, v, do, do, qo, qo, lse, delta)
    exact = oracle_mod.bwd_mx_operands(*args, causal=True, scale=scale, round_ps=False)
    rounded = oracle_mod.bwd_mx_operands(*args, causal=True, scale=scale, round_ps=True)
    # sum of |terms| of dv: sum_i |p_ij| |do_i|; of dq, dk through |ds|: recompute p, ds
    for b in range(len(lq)):
        s0, s1 = int(qo[b]), int(qo[b + 1])
        L = s1 - s0
        S = scale * q[s0:s1, 0] @ k[s0:s1, 0].T
        P = np.where(np.tril(np.ones((L, L), bool)), np.exp(S - lse[0, s0:s1, None]), 0.0)
        dS = P * (do[s0:s1, 0] @ v[s0:s1, 0].T - delta[0, s0:s1, None])
        # an element in its block's subnormal range is off by at most 2^-10 X,
        # and X < amax / 224 under the saturation-free scale
        ep = 2.0 ** -4 * np.abs(P) + 2.0 ** -10 * np.abs(P).max() / 224
        es = 2.0 ** -4 * np.abs(dS) + 2.0 ** -10 * np.abs(dS).max() / 224
        bv = ep.T @ np.abs(do[s0:s1, 0])
        bq = scale * es @ np.abs(k[s0:s1, 0])
        bk = scale * es.T @ np.abs(q[s0:s1, 0])
        for g, e, bd in ((rounded[0], exact[0], bq), (rounded[1], exact[1], bk),
                         (rounded[2], exact[2], bv)):
            assert np.all(np.abs(g[s0:s1, 0] - e[s0:s1, 0]) <= bd * (1 + 1e-9))
        assert np.abs(rounded[2] - exact[2]).max() > 0   # the rounding does act


def test_bwd_mxfp8_on_exactly_representable_inputs(oracle_mod):
    """Inputs whose every 32-element block (along channels and along tokens)
    already lies on the E4M3 grid with scale 1 (magnitudes 256..448) are left
    unchanged by the operand quantisation, so the full MXFP8 backward equals
    the operand form with one version per tensor."""
    lq = [40, 64, 9]
    H, d = 2, 32
    rng = np.random.default_rng(12)
    grid = 256.0 * (1.0 + np.arange(7) / 8.0)          # 256 .. 448
    T = sum(lq)
    mk = lambda: rng.choice(grid, size=(T, H, d)) * rng.choice([-1.0, 1.0], size=(T, H, d))
    q, k, v, do = mk(), mk(), mk(), mk()
    qo = _offsets(lq)
    scale = 2.0 ** -22
    out, lse = oracle_mod.fwd(q, qo, k, v, qo, act=ACT_SOFTMAX, causal=True, scale=scale)
    for x in (q, k, v, do):
        np.testing.assert_array_equal(oracle_mod.dequant_rows(x), x)
        np.testing.assert_array_equal(oracle_mod.dequant_cols(x, qo), x)
    got = oracle_mod.bwd_mxfp8(q, qo, k, v, qo, out, do, lse, causal=True, scale=scale)
    delta = np.einsum("thc,thc->ht", do, out)
    ref = oracle_mod.bwd_mx_operands(q, q, k, k, v, do, do, qo, qo, lse, delta, causal=True,
                                     scale=scale, round_ps=True)
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(g, r)


# --------------------------------------------------------------- dense jagged bias
def _dense_from_table(table, lq, lkv, max_rel):
    """The relative-position table written out as a dense jagged bias."""
    parts = []
    for Lq, Lkv in zip(lq, lkv):
        for h in range(table.shape[0]):
            parts.append(_relpos_mask(table[h], Lq, Lkv, max_rel).reshape(-1))
    return np.concatenate(parts) if parts else np.zeros(0)


@pytest.mark.parametrize("causal", [False, True])
def test_dense_bias_matches_torch_sdpa(oracle_mod, causal):
    """Softmax forward with a random dense bias against torch's fp64 SDPA with
    that bias as the additive mask, sample by sample and head by head."""
    lq = [5, 1, 33, 17]
    lkv = lq if causal else [9, 4, 20, 1]
    H, d = 3, 8
    qo, ko = _offsets(lq), _offsets(lkv)
    q = _bf16_randn((sum(lq), H, d), 51)
    k = _bf16_randn((sum(lkv), H, d), 52)
    v = _bf16_randn((sum(lkv), H, d), 53)
    off = oracle_mod.dense_bias_offsets(qo, ko, H)
    dense = np.random.default_rng(9).normal(0, 1.0, int(off[-1]))
    scale = 1.0 / math.sqrt(d)
    out, lse = oracle_mod.fwd(q, qo, k, v, ko, act=ACT_SOFTMAX, causal=causal, scale=scale,
                              dense_bias=dense)
    for b in range(len(lq)):
        Lq, Lkv = lq[b], lkv[b]
        blk = dense[off[b]:off[b + 1]].reshape(H, Lq, Lkv)
        for h in range(H):
            mask = torch.from_numpy(blk[h].copy())
            if causal:
                mask = mask.masked_fill(torch.ones(Lq, Lkv).triu(1).bool(), float("-inf"))
            qs = torch.from_numpy(q[qo[b]:qo[b + 1], h].copy())[None, None]
            ks = torch.from_numpy(k[ko[b]:ko[b + 1], h].copy())[None, None]
            vs = torch.from_numpy(v[ko[b]:ko[b + 1], h].copy())[None, None]
            ref = F.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask, scale=scale)[0, 0]
            np.testing.assert_allclose(out[qo[b]:qo[b + 1], h], ref.numpy(), rtol=1e-12, atol=1e-12)
            s_ = scale * (qs[0, 0] @ ks[0, 0].T) + mask
            np.testing.assert_allclose(lse[h, qo[b]:qo[b + 1]], torch.logsumexp(s_, -1).numpy(),
                                       rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_SILU, ACT_GELU_TANH])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_bias_written_from_the_table_equals_the_table(oracle_mod, act, causal):
    """A dense bias holding the relative-position table's values gives the
    table's forward and backward (each pinned on its own): catches a swapped
    query / key index, a wrong head or a wrong sample offset."""
    lq = [6, 0, 40, 13]
    lkv = lq if causal else [3, 7, 21, 13]
    H, d, max_rel = 2, 8, 9
    qo, ko = _offsets(lq), _offsets(lkv)
    q = _bf16_randn((sum(lq), H, d), 61)
    k = _bf16_randn((sum(lkv), H, d), 62)
    v = _bf16_randn((sum(lkv), H, d), 63)
    do = _bf16_randn((sum(lq), H, d), 64)
    table = np.random.default_rng(4).normal(0, 0.7, (H, 2 * max_rel - 1))
    dense = _dense_from_table(table, lq, lkv, max_rel)
    kw = dict(act=act, causal=causal, scale=1.0 / math.sqrt(d))
    a = oracle_mod.fwd(q, qo, k, v, ko, bias=table, max_rel=max_rel, **kw)
    b = oracle_mod.fwd(q, qo, k, v, ko, dense_bias=dense, **kw)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    a = oracle_mod.bwd(q, qo, k, v, ko, do, bias=table, max_rel=max_rel, **kw)
    b = oracle_mod.bwd(q, qo, k, v, ko, do, dense_bias=dense, **kw)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_dense_bias_backward_matches_central_differences(oracle_mod):
    """The backward under a random (non-Toeplitz) dense bias against central
    differences of the forward."""
    lq, lkv = [4, 3], [5, 2]
    H, d = 2, 4
    qo, ko = _offsets(lq), _offsets(lkv)
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((sum(n), H, d)) for n in (lq, lkv, lkv))
    do = rng.standard_normal((sum(lq), H, d))
    dense = rng.normal(0, 1.0, int(oracle_mod.dense_bias_offsets(qo, ko, H)[-1]))
    for act in (ACT_SOFTMAX, ACT_SILU):
        kw = dict(act=act, scale=0.7, dense_bias=dense)
        dq, dk, dv = oracle_mod.bwd(q, qo, k, v, ko, do, **kw)
        loss = lambda q_, k_, v_: float((oracle_mod.fwd(q_, qo, k_, v_, ko, **kw)[0] * do).sum())
        h = 1e-6
        for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
            num = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = [q, k, v]
                args_m = [q, k, v]
                args_p[which], args_m[which] = xp, xm
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-7)


def test_dense_bias_rejects_a_wrong_size(oracle_mod):
    lq = [3, 2]
    qo = _offsets(lq)
    x = np.zeros((5, 1, 4))
    with pytest.raises(AssertionError):
        oracle_mod.fwd(x, qo, x, x, qo, act=ACT_SOFTMAX, scale=1.0, dense_bias=np.zeros(12))


# --------------------------------------------------------------- independent formulation
def _torch_act(act):
    return {ACT_SILU: F.silu, ACT_GELU_TANH: lambda x: F.gelu(x, approximate="tanh"),
            ACT_GELU_ERF: lambda x: F.gelu(x, approximate="none"), ACT_IDENTITY: lambda x: x}[act]


def _torch_reference(q, k, v, do, lq, lkv, act, causal, scale, table=None, max_rel=0, window=0,
                     block=0, dense=None):
    """Per-sample fp64 matrices (torch ops) and autograd: out, dq, dk, dv and the
    table's gradient, with no code shared with the oracle's loops."""
    H = q.shape[1]
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    tt = torch.tensor(table, dtype=torch.float64, requires_grad=True) if table is not None else None
    outs, qo, ko, doff = [], 0, 0, 0
    for Lq, Lkv in zip(lq, lkv):
        i = torch.arange(Lq)[:, None]
        j = torch.arange(Lkv)[None, :]
        keep = torch.ones(Lq, Lkv, dtype=torch.bool)
        if causal:
            keep &= j <= i
        if window:
            keep &= (i - j).abs() < window
        if block:
            keep &= (i // block) == (j // block)
        for h in range(H):
            s = scale * tq[qo:qo + Lq, h] @ tk[ko:ko + Lkv, h].T
            if tt is not None:
                s = s + tt[h][(i - j + max_rel - 1).clamp(0, 2 * max_rel - 2)]
            if dense is not None:
                s = s + torch.tensor(dense[doff:doff + Lq * Lkv].reshape(Lq, Lkv))
                doff += Lq * Lkv
            if act == ACT_SOFTMAX:
                p = torch.softmax(s.masked_fill(~keep, float("-inf")), dim=-1)
                p = torch.nan_to_num(p, nan=0.0)      # a row with no key attends to nothing
            else:
                p = _torch_act(act)(s) * keep
            outs.append((qo, h, p @ tv[ko:ko + Lkv, h]))
        qo, ko = qo + Lq, ko + Lkv
    out = torch.zeros_like(tq)
    for q0, h, o in outs:
        out[q0:q0 + o.shape[0], h] = o
    (out * torch.tensor(do)).sum().backward()
    return (out.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy(),
            tt.grad.numpy() if tt is not None else None)


@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_SILU, ACT_GELU_TANH, ACT_GELU_ERF, ACT_IDENTITY])
@pytest.mark.parametrize("variant", ["tiny", "causal_bias", "window", "block", "dense"])
def test_tiny_inputs_against_torch_autograd(oracle_mod, act, variant):
    """Tiny inputs (B <= 4, L <= 64) against torch fp64 matrices differentiated by
    autograd: the whole forward and every backward output, bias gradient too."""
    rng = np.random.default_rng(100 + act)
    H, d = 2, 8
    if variant == "tiny":          # the four-sample tiny workload's lengths
        lq = lkv = [1, 7, 33, 64]
    elif variant == "causal_bias":
        lq = lkv = [3, 5, 1]
    else:
        lq = lkv = [4, 5, 2] if variant != "block" else [9, 5, 12]
    if variant == "tiny":
        lkv = [2, 7, 5, 64]        # asymmetric lengths, no mask
    causal = variant in ("causal_bias", "window")
    max_rel = 4 if variant in ("causal_bias", "window", "block") else 0
    table = rng.normal(0, 0.5, (H, 2 * max_rel - 1)) if max_rel else None
    window = 2 if variant == "window" else 0
    block = 4 if variant == "block" else 0
    qo, ko = _offsets(lq), _offsets(lkv)
    q, do = (rng.standard_normal((sum(lq), H, d)) for _ in range(2))
    k, v = (rng.standard_normal((sum(lkv), H, d)) for _ in range(2))
    dense = None
    if variant == "dense":
        dense = rng.normal(0, 0.7, int(oracle_mod.dense_bias_offsets(qo, ko, H)[-1]))
        # the reference walks samples then heads: the oracle's layout is [b][h][i][j] too
    scale = 0.6
    kw = dict(act=act, causal=causal, scale=scale, window=window, block=block)
    if table is not None:
        kw.update(bias=table, max_rel=max_rel)
    if dense is not None:
        kw.update(dense_bias=dense)
    ro, rdq, rdk, rdv, rdb = _torch_reference(q, k, v, do, lq, lkv, act, causal, scale, table,
                                              max_rel, window, block, dense)
    out, _ = oracle_mod.fwd(q, qo, k, v, ko, **kw)
    np.testing.assert_allclose(out, ro, rtol=1e-11, atol=1e-12)
    got = oracle_mod.bwd(q, qo, k, v, ko, do, want_dbias=table is not None, **kw)
    for g, r in zip(got[:3], (rdq, rdk, rdv)):
        np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-11)
    if table is not None:
        np.testing.assert_allclose(got[3], rdb, rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_SILU])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_bias_gradient(oracle_mod, act, causal):
    """The dense bias's gradient (dS, in the bias's layout): central differences
    of the forward in sampled entries, zeros on masked pairs, and summed along
    the clamped relative positions it equals the (pinned) table gradient when
    the dense bias is the table written out."""
    lq = [4, 6, 1] if causal else [4, 6, 2]
    lkv = lq if causal else [3, 5, 4]
    H, d, max_rel = 2, 4, 3
    qo, ko = _offsets(lq), _offsets(lkv)
    rng = np.random.default_rng(11)
    q = rng.standard_normal((sum(lq), H, d))
    k, v = (rng.standard_normal((sum(lkv), H, d)) for _ in range(2))
    do = rng.standard_normal((sum(lq), H, d))
    table = rng.normal(0, 0.5, (H, 2 * max_rel - 1))
    dense = _dense_from_table(table, lq, lkv, max_rel)
    kw = dict(act=act, causal=causal, scale=0.8)
    *_, g = oracle_mod.bwd(q, qo, k, v, ko, do, want_dbias=True, dense_bias=dense, **kw)
    assert g.shape == dense.shape
    loss = lambda dn: float((oracle_mod.fwd(q, qo, k, v, ko, dense_bias=dn, **kw)[0] * do).sum())
    h = 1e-6
    for idx in rng.choice(dense.size, 25, replace=False):
        e = np.zeros_like(dense)
        e[idx] = h
        np.testing.assert_allclose(g[idx], (loss(dense + e) - loss(dense - e)) / (2 * h),
                                   rtol=1e-6, atol=1e-8)
    off = oracle_mod.dense_bias_offsets(qo, ko, H)
    table_grad = np.zeros_like(table)
    for b, (Lq, Lkv) in enumerate(zip(lq, lkv)):
        blk = g[off[b]:off[b + 1]].reshape(H, Lq, Lkv)
        i, j = np.arange(Lq)[:, None], np.arange(Lkv)[None, :]
        if causal:
            assert np.all(blk[:, j > i] == 0.0)
        idx = np.clip(i - j + max_rel - 1, 0, 2 * max_rel - 2)
        for hh in range(H):
            np.add.at(table_grad[hh], idx, blk[hh])
    ref = oracle_mod.bwd(q, qo, k, v, ko, do, want_dbias=True, bias=table, max_rel=max_rel, **kw)[3]
    np.testing.assert_allclose(table_grad, ref, rtol=1e-12, atol=1e-12)
