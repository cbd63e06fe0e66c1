"""Pins for the CPU oracle, against things other than the oracle itself:
hand-worked examples (tests/golden), exact rational arithmetic, library
routines (torch's bf16 cast, numpy's argsort/bincount/int64 einsum, float64
math), closed forms, invariants and brute force on tiny inputs."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import wq_oracle as O
from w8a8_int8_quantized_token_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def to_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def ulp_f32(x):
    x = np.abs(np.asarray(x, np.float32))
    return np.spacing(np.maximum(x, np.float32(np.finfo(np.float32).tiny)))


# ---------------------------------------------------------------- bf16
def test_bf16_cast_matches_torch():
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(20000, generator=g) * 10 ** torch.randint(-30, 30, (20000,), generator=g).float(),
                   torch.tensor([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.4e38, -3.4e38,
                                 float("inf"), float("-inf"), 1e-40, -1e-42])])
    got = O.f32_to_bf16(x.numpy())
    want = to_bf16_bits(x)
    assert np.array_equal(got, want)
    back = O.bf16_to_f32(want)
    assert np.array_equal(back, x.to(torch.bfloat16).float().numpy())


def test_bf16_nan_stays_nan():
    out = O.bf16_to_f32(O.f32_to_bf16(np.array([np.nan], np.float32)))
    assert np.isnan(out[0])


# ---------------------------------------------------------------- exp / silu
def test_exp_constants_split_ln2():
    hi = Fraction(float(O.LN2_HI))
    # at most 16 significant bits, so n*LN2_HI is exact for |n| < 2**8
    assert (hi * 2**16).denominator == 1 and hi * 2**16 < 2**16
    assert abs(float(O.LN2_HI) + float(O.LN2_LO) - math.log(2.0)) < 1e-13
    assert float(O.LOG2E) == float(np.float32(1 / math.log(2)))
    for i, c in enumerate(O.EXP_COEF):
        assert c == np.float32(1 / math.factorial(i))


def test_exp_error_within_2_ulp():
    x = np.concatenate([np.linspace(-103.0, 88.7, 400001, dtype=np.float32),
                        np.float32(np.random.default_rng(0).uniform(-20, 20, 200000))])
    got = O.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    normal = ref > np.finfo(np.float32).tiny
    err = np.abs(got - ref)[normal] / ulp_f32(ref[normal].astype(np.float32))
    assert err.max() <= 2.0, err.max()
    # subnormal range: absolute error within one least subnormal
    sub = ~normal
    assert np.all(np.abs(got - ref)[sub] <= 2 ** -149)


def test_exp_special_values():
    x = np.array([0.0, -0.0, 89.0, 1000.0, -104.0, -1e9, np.inf, -np.inf, np.nan, 88.7], np.float32)
    y = O.exp_f32(x)
    assert y[0] == 1.0 and y[1] == 1.0
    assert np.isinf(y[2]) and np.isinf(y[3]) and np.isinf(y[6])
    assert y[4] == 0.0 and y[5] == 0.0 and y[7] == 0.0
    assert np.isnan(y[8])
    assert np.isfinite(y[9])


def test_silu_matches_float64():
    g = np.float32(np.random.default_rng(1).normal(0, 6, 100000))
    got = O.silu_f32(g).astype(np.float64)
    gd = g.astype(np.float64)
    ref = gd / (1.0 + np.exp(-gd))
    assert np.all(np.abs(got - ref) <= 4 * ulp_f32(ref.astype(np.float32)) + 1e-37)
    assert O.silu_f32(np.float32([0.0]))[0] == 0.0
    big = O.silu_f32(np.float32([200.0, -200.0]))
    assert big[0] == 200.0 and big[1] == 0.0


# ---------------------------------------------------------------- quant
def test_quant_golden():
    G = golden("quant_worked.json")
    for case in G["per_token"]:
        x = O.f32_to_bf16(np.array([case["x"]], np.float32))
        q, s = O.quantize_per_token(x)
        assert q.tolist()[0] == case["q"]
        assert np.isclose(s[0], case["s"], rtol=1e-6, atol=0)
    pg = G["per_group_4"]
    x = O.f32_to_bf16(np.array([pg["x"]], np.float32))
    q, s = O.quantize_per_token_group(x, 4)
    assert q.tolist()[0] == pg["q"] and s.tolist()[0] == pg["s"]


def _round_half_even(fr: Fraction) -> int:
    fl = math.floor(fr)
    d = fr - fl
    if d > Fraction(1, 2) or (d == Fraction(1, 2) and fl % 2 == 1):
        return fl + 1
    return fl


def test_quant_against_exact_rationals():
    """Codes equal exact-rational round-half-even of x/s except where the
    float32 quotient sits within 2**-20 of a rounding midpoint."""
    x = synth.activations(6, 384, True, 11)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    q, s = O.quantize_per_token(xb)
    xf = O.bf16_to_f32(xb)
    for t in range(xf.shape[0]):
        a = np.max(np.abs(xf[t]))
        # s is the float32 quotient absmax / 127
        assert Fraction(float(s[t])) == Fraction(float(np.float32(a) / np.float32(127)))
        for j in range(0, xf.shape[1], 3):
            ex = Fraction(float(xf[t, j])) / Fraction(float(s[t]))
            frac = ex - math.floor(ex)
            if abs(frac - Fraction(1, 2)) < Fraction(1, 2**20):
                continue
            assert q[t, j] == max(-127, min(127, _round_half_even(ex)))


def test_quant_invariants():
    x = synth.activations(64, 1024, True, 2)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    for q, s, xx in [(*O.quantize_per_token(xb), O.bf16_to_f32(xb)),
                     ]:
        rec = q.astype(np.float64) * s[:, None].astype(np.float64)
        assert np.all(np.abs(rec - xx) <= s[:, None] / 2 * (1 + 2 ** -20))
        assert q.min() >= -127 and q.max() <= 127
        # every row reaches +-127 at its absmax element
        assert np.all(np.abs(q).max(axis=1) == 127)


def test_quant_integer_multiples_exact():
    # x = n * s with s a power of two: the codes are n
    n = np.arange(-127, 128, dtype=np.float32)
    for s in (0.25, 1.0, 8.0):
        x = O.f32_to_bf16((n * np.float32(s))[None, :])
        q, sc = O.quantize_per_token(x)
        assert sc[0] == np.float32(s)
        assert np.array_equal(q[0], n.astype(np.int8))


def test_group_quant_is_per_row_quant_of_groups():
    x = synth.activations(8, 512, True, 4)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    q, s = O.quantize_per_token_group(xb, 128)
    q2, s2 = O.quantize_per_token(xb.reshape(32, 128))
    assert np.array_equal(q.reshape(32, 128), q2) and np.array_equal(s.reshape(-1), s2)


def test_block_weight_quant():
    g = torch.Generator().manual_seed(5)
    w = (torch.randn(256, 384, generator=g) * 0.02).to(torch.bfloat16)
    wb = w.view(torch.int16).numpy().view(np.uint16)
    q, s = O.quantize_weight_block(wb)
    assert s.shape == (2, 3)
    for nb in range(2):
        for kb in range(3):
            blk = wb[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128].reshape(1, -1)
            qq, ss = O.quantize_per_token(blk)
            assert ss[0] == s[nb, kb]
            assert np.array_equal(qq.reshape(128, 128), q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128])
    const = O.f32_to_bf16(np.full((128, 128), -0.5, np.float32))
    qc, sc = O.quantize_weight_block(const)
    assert np.all(qc == -127)


def test_channel_weight_quant_is_per_row():
    g = torch.Generator().manual_seed(6)
    w = (torch.randn(64, 256, generator=g) * 0.02).to(torch.bfloat16)
    wb = w.view(torch.int16).numpy().view(np.uint16)
    q, s = O.quantize_weight_channel(wb)
    for n in range(64):
        a = np.max(np.abs(O.bf16_to_f32(wb[n])))
        assert s[n] == np.float32(a) / np.float32(127)


# ---------------------------------------------------------------- routing
def test_route_golden():
    for c in golden("route_worked.json")["cases"]:
        ids, w = O.route_topk(np.array([c["logits"]], np.float32), c["k"])
        assert ids.tolist()[0] == c["ids"]
        assert np.allclose(w[0], c["w"], rtol=2 ** -23, atol=0)


def test_route_selection_matches_stable_argsort():
    lg = synth.router_logits(50, 32, 3).numpy()
    lg[:, 5] = lg[:, 9]  # plant exact ties
    ids, w = O.route_topk(lg, 6)
    ref = np.argsort(-lg, axis=1, kind="stable")[:, :6]
    assert np.array_equal(ids, ref)


def test_route_all_experts_is_softmax():
    lg = synth.router_logits(20, 8, 4).numpy()
    ids, w = O.route_topk(lg, 8)
    ld = lg.astype(np.float64)
    p = np.exp(ld - ld.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    got = np.zeros_like(p)
    np.put_along_axis(got, ids, w.astype(np.float64), 1)
    assert np.allclose(got, p, rtol=1e-6, atol=1e-7)
    assert np.allclose(w.sum(1), 1.0, atol=1e-6)


def test_route_k1_weight_is_one():
    ids, w = O.route_topk(synth.router_logits(30, 16, 5).numpy(), 1)
    assert np.all(w == 1.0)


# ---------------------------------------------------------------- align / permute
def test_align_golden():
    G = golden("align_worked.json")
    ids = np.array(G["ids"], np.int32)
    for key, pad in (("tight", 1), ("padded", G["pad_m"])):
        counts, offsets, sp, p2r = O.moe_align(ids, G["E"], pad)
        want = G[key]
        assert counts.tolist() == want["counts"]
        assert offsets.tolist() == want["offsets"]
        assert sp.tolist() == want["sorted_pair"]
        assert p2r.tolist() == want["pair_to_row"]


def test_align_invariants():
    rng = np.random.default_rng(7)
    T, k, E = 300, 4, 37
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    ids[:, 0] = 3  # a hot expert
    counts, offsets, sp, p2r = O.moe_align(ids, E)
    assert np.array_equal(counts, np.bincount(ids.reshape(-1), minlength=E))
    assert counts.sum() == T * k and offsets[0] == 0 and offsets[-1] == T * k
    assert np.array_equal(sp[p2r], np.arange(T * k))
    flat = ids.reshape(-1)
    for e in range(E):
        seg = sp[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


def test_permute_is_gather_by_pair():
    rng = np.random.default_rng(8)
    T, k, E, K = 50, 3, 9, 64
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    q = rng.integers(-127, 128, (T, K), dtype=np.int8)
    s = rng.random(T).astype(np.float32)
    _, offs, sp, p2r = O.moe_align(ids, E)
    A, sa = O.moe_permute(q, s, sp, k)
    for p in range(T * k):
        assert np.array_equal(A[p2r[p]], q[p // k]) and sa[p2r[p]] == s[p // k]
    _, offs4, sp4, p2r4 = O.moe_align(ids, E, 4)
    A4, sa4 = O.moe_permute(q, s, sp4, k)
    assert np.all(A4[sp4 < 0] == 0) and np.all(sa4[sp4 < 0] == 0)


# ---------------------------------------------------------------- GEMM
def test_int_matmul_matches_int64_einsum():
    rng = np.random.default_rng(9)
    a = rng.integers(-127, 128, (33, 700), dtype=np.int8)
    w = rng.integers(-127, 128, (21, 700), dtype=np.int8)
    ref = np.einsum("mk,nk->mn", a.astype(np.int64), w.astype(np.int64))
    assert np.array_equal(O.int_matmul(a, w), ref)
    worst = np.full((2, 7168), 127, np.int8)
    neg = worst.copy()
    neg[1] = -127
    C = O.int_matmul(worst, neg)
    assert C[0, 0] == 127 * 127 * 7168 and C[0, 1] == -127 * 127 * 7168
    # an odd sum above 2**24 has no float32 representation: the matmul must be exact
    odd = worst[:1].copy()
    odd[0, 100] = 126
    assert O.int_matmul(worst[:1], odd)[0, 0] == 127 * 127 * 7168 - 127


def test_gemm_golden():
    G = golden("gemm_worked.json")
    A = np.array(G["A"], np.int8)
    W = np.array(G["W"], np.int8)
    assert O.int_matmul(A, W).tolist() == G["C"]
    out = O.grouped_gemm_w8a8(A, np.array(G["sa"], np.float32), W[None], np.array(G["sw"], np.float32)[None],
                              np.array([0, 2]), "channel", "i32")
    assert O.bf16_to_f32(out).tolist() == G["out"]


def _rand_gemm(seed, m=37, n=256, K=384):
    rng = np.random.default_rng(seed)
    A = rng.integers(-127, 128, (m, K), dtype=np.int8)
    W = rng.integers(-127, 128, (n, K), dtype=np.int8)
    return rng, A, W


def test_gemm_f32_tiles_equal_i32_when_partial_sums_exact():
    rng, A, W = _rand_gemm(10)
    sa = rng.random(A.shape[0]).astype(np.float32)
    sw = rng.random(W.shape[0]).astype(np.float32)
    v32 = O.gemm_dequant(A, sa, W, sw, "channel", "i32")
    vf = O.gemm_dequant(A, sa, W, sw, "channel", "f32")
    # |C| <= 127*127*384 < 2**24: every float partial sum is exact
    assert np.array_equal(v32, vf)


def test_gemm_f32_tiles_round_each_partial():
    # K = 7168 all-127: partials 2064512 each, the running float sum exceeds
    # 2**24 and rounds, unlike the int32 accumulator
    A = np.full((1, 7168), 127, np.int8)
    W = np.full((1, 7168), 127, np.int8)
    W[0, ::2] = 125
    one = np.ones(1, np.float32)
    acc = np.float32(0)
    for t in range(56):
        acc = np.float32(acc + np.float32(int(O.int_matmul(A[:, t*128:(t+1)*128], W[:, t*128:(t+1)*128])[0, 0])))
    assert O.gemm_dequant(A, one, W, one, "channel", "f32")[0, 0] == acc
    assert O.gemm_dequant(A, one, W, one, "channel", "i32")[0, 0] == np.float32(int(O.int_matmul(A, W)[0, 0]))


def test_gemm_block_with_power_of_two_scales_equals_channel():
    rng, A, W = _rand_gemm(11)
    sa = np.float32(2.0) ** rng.integers(-8, 0, A.shape[0]).astype(np.float32)
    sw = np.float32(2.0) ** rng.integers(-12, -6, W.shape[0] // 128).astype(np.float32)
    sa_b = np.repeat(sa[:, None], 3, 1)
    sw_b = np.repeat(sw[:, None], 3, 1)
    vb = O.gemm_dequant(A, sa_b, W, sw_b, "block", "f32")
    vc = O.gemm_dequant(A, sa, W, np.repeat(sw, 128), "channel", "i32")
    assert np.array_equal(vb, vc)


def test_gemm_matches_dequantize_then_float64_matmul():
    """Dequantize first, multiply in float64: a different decomposition of the
    same definition; catches transposed operands and wrong scale indices."""
    rng, A, W = _rand_gemm(12, m=29, n=256, K=384)
    sa = (rng.random(29) * 0.1).astype(np.float32)
    sw = (rng.random(256) * 0.01).astype(np.float32)
    ref = (A * sa[:, None].astype(np.float64)) @ (W * sw[:, None].astype(np.float64)).T
    for acc in ("i32", "f32"):
        got = O.gemm_dequant(A, sa, W, sw, "channel", acc).astype(np.float64)
        assert np.all(np.abs(got - ref) <= 4 * ulp_f32(ref.astype(np.float32)))
    sa_b = (rng.random((29, 3)) * 0.1).astype(np.float32)
    sw_b = (rng.random((2, 3)) * 0.01).astype(np.float32)
    Af = A * np.repeat(sa_b, 128, 1).astype(np.float64)
    Wf = W * np.repeat(np.repeat(sw_b, 128, 0), 128, 1).astype(np.float64)
    ref_b = Af @ Wf.T
    got_b = O.gemm_dequant(A, sa_b, W, sw_b, "block", "f32").astype(np.float64)
    bound = 8 * np.spacing(np.float32(np.abs(Af) @ np.abs(Wf).T))
    assert np.all(np.abs(got_b - ref_b) <= bound)


def test_grouped_gemm_segments():
    rng = np.random.default_rng(13)
    E, N, K = 4, 128, 256
    W = rng.integers(-127, 128, (E, N, K), dtype=np.int8)
    offsets = np.array([0, 5, 5, 17, 20])
    A = rng.integers(-127, 128, (20, K), dtype=np.int8)
    C = O.grouped_gemm_i32(A, W, offsets)
    for r in range(20):
        e = np.searchsorted(offsets, r, side="right") - 1
        assert np.array_equal(C[r], A[r].astype(np.int64) @ W[e].astype(np.int64).T)


# ---------------------------------------------------------------- activation / combine
def test_silu_mul_quant_definition():
    rng = np.random.default_rng(14)
    I = 256
    gu = O.f32_to_bf16(rng.normal(0, 3, (9, 2 * I)).astype(np.float32))
    hq, sh = O.silu_mul_quant(gu, I, 0)
    g = O.bf16_to_f32(gu[:, :I]).astype(np.float64)
    u = O.bf16_to_f32(gu[:, I:]).astype(np.float64)
    h = g / (1 + np.exp(-g)) * u
    # scale is absmax(h)/127 up to float32 rounding of h
    assert np.allclose(sh, np.abs(h).max(1) / 127, rtol=1e-6)
    assert np.all(np.abs(hq * sh[:, None].astype(np.float64) - h) <= sh[:, None] * (0.5 + 1e-4))
    hq_g, sh_g = O.silu_mul_quant(gu, I, 128)
    assert sh_g.shape == (9, 2)
    assert np.allclose(sh_g, np.abs(h).reshape(9, 2, 128).max(2) / 127, rtol=1e-6)


def test_combine_identity_and_float64():
    rng = np.random.default_rng(15)
    T, H = 12, 64
    y = O.f32_to_bf16(rng.normal(0, 2, (T, H)).astype(np.float32))
    perm = rng.permutation(T).astype(np.int32)
    out = O.moe_combine(y, perm, np.ones((T, 1), np.float32), 1)
    assert np.array_equal(out, y[perm])
    k = 4
    y4 = O.f32_to_bf16(rng.normal(0, 2, (T * k, H)).astype(np.float32))
    w = rng.random((T, k)).astype(np.float32)
    p2r = rng.permutation(T * k).astype(np.int32)
    out = O.bf16_to_f32(O.moe_combine(y4, p2r, w, k)).astype(np.float64)
    ref = (w[:, :, None].astype(np.float64) * O.bf16_to_f32(y4)[p2r.reshape(T, k)]).sum(1)
    mag = (np.abs(w[:, :, None].astype(np.float64)) * np.abs(O.bf16_to_f32(y4)[p2r.reshape(T, k)])).sum(1)
    # one bf16 rounding (half an ulp, at most 2**-8 relative) plus k float32 roundings
    assert np.all(np.abs(out - ref) <= 2.0 ** -8 * np.abs(ref) + 2 * k * 2.0 ** -24 * mag + 1e-30)


# ---------------------------------------------------------------- the layer
def _quantized_weights(cfg):
    q13, s13, q2, s2 = [], [], [], []
    for e in range(cfg.E):
        w13, w2 = synth.expert_weights(cfg, e)
        a, b, c, d = O.quantize_weights(w13.view(torch.int16).numpy().view(np.uint16),
                                        w2.view(torch.int16).numpy().view(np.uint16), cfg.scheme)
        q13.append(a); s13.append(b); q2.append(c); s2.append(d)
    return np.stack(q13), np.stack(s13), np.stack(q2), np.stack(s2)


@pytest.mark.parametrize("scheme,acc", [("channel", "i32"), ("channel", "f32"), ("block", "f32")])
def test_layer_equals_token_by_token_evaluation(scheme, acc):
    """Expert-major (align/permute/grouped GEMM/combine) equals evaluating each
    token on each of its experts directly."""
    cfg = synth.small_config(T=9, H=256, I=128, E=5, k=2, scheme=scheme, acc=acc)
    x, lg = synth.layer_inputs(cfg)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    W13, S13, W2, S2 = _quantized_weights(cfg)
    out = O.moe_forward(xb, lg.numpy(), W13, S13, W2, S2, cfg.k, scheme, acc)
    ids, w = O.route_topk(lg.numpy(), cfg.k)
    grp = 0 if scheme == "channel" else 128
    for t in range(cfg.T):
        if scheme == "channel":
            q, s = O.quantize_per_token(xb[t:t + 1])
        else:
            q, s = O.quantize_per_token_group(xb[t:t + 1], 128)
        acc_t = np.zeros(cfg.H, np.float32)
        for j in range(cfg.k):
            e = ids[t, j]
            gu = O.f32_to_bf16(O.gemm_dequant(q, s, W13[e], S13[e], scheme, acc))
            hq, sh = O.silu_mul_quant(gu, cfg.I, grp)
            y = O.f32_to_bf16(O.gemm_dequant(hq, sh, W2[e], S2[e], scheme, acc))
            acc_t = acc_t + w[t, j] * O.bf16_to_f32(y[0])
        assert np.array_equal(O.f32_to_bf16(acc_t), out[t]), t


def test_layer_single_expert_is_dense_ffn():
    cfg = synth.small_config(T=7, H=256, I=128, E=1, k=1)
    x, lg = synth.layer_inputs(cfg)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    W13, S13, W2, S2 = _quantized_weights(cfg)
    out = O.moe_forward(xb, lg.numpy(), W13, S13, W2, S2, 1)
    q, s = O.quantize_per_token(xb)
    gu = O.f32_to_bf16(O.gemm_dequant(q, s, W13[0], S13[0], "channel", "i32"))
    hq, sh = O.silu_mul_quant(gu, cfg.I)
    y = O.f32_to_bf16(O.gemm_dequant(hq, sh, W2[0], S2[0], "channel", "i32"))
    assert np.array_equal(out, y)


def test_masked_layout_matches_per_expert_layer():
    cfg = synth.small_config(T=0, H=256, I=128, E=4, k=1)
    rng = np.random.default_rng(16)
    Mmax = 24
    xm = synth.activations(cfg.E * Mmax, cfg.H, True, 3).view(torch.int16).numpy().view(np.uint16)
    q, s = O.quantize_per_token(xm)
    q = q.reshape(cfg.E, Mmax, cfg.H)
    s = s.reshape(cfg.E, Mmax)
    mm = np.array([5, 0, 24, 1], np.int32)
    W13, S13, W2, S2 = _quantized_weights(cfg)
    y, valid = O.moe_forward_masked(q, s, mm, W13, S13, W2, S2)
    assert valid.sum() == mm.sum()
    for e in range(cfg.E):
        m = mm[e]
        if m == 0:
            continue
        gu = O.grouped_gemm_w8a8(q[e, :m], s[e, :m], W13[e:e + 1], S13[e:e + 1], np.array([0, m]))
        hq, sh = O.silu_mul_quant(gu, cfg.I)
        ye = O.grouped_gemm_w8a8(hq, sh, W2[e:e + 1], S2[e:e + 1], np.array([0, m]))
        assert np.array_equal(y[e, :m], ye)


def test_linear_hand_worked():
    """A dense W8A8 linear worked by hand: x = [2, -1, 0.5, 0, ...] gives
    s = 2/127 and codes [127, -64 (-63.5, tie to even), 32 (31.75), 0, ...];
    channel codes [1, 2, 3, 0, ...] and [-1, 0, 4, 0, ...] with scales 0.5
    and 0.25 give C = 95 and 1, and v = (C * s) * sw rounded to float32 at
    each step, then to bf16."""
    from fractions import Fraction
    K = 128
    x = np.zeros((1, K), np.float32)
    x[0, :3] = [2.0, -1.0, 0.5]
    xb = O.f32_to_bf16(x)
    w = np.zeros((2, K), np.int8)
    w[0, :3] = [1, 2, 3]
    w[1, :3] = [-1, 0, 4]
    sw = np.array([0.5, 0.25], np.float32)
    got = O.bf16_to_f32(O.linear_w8a8(xb, w, sw, "channel", "i32"))[0]
    s = np.float32(2.0) / np.float32(127.0)
    q = [127, -64, 32]
    C = [sum(qi * wi for qi, wi in zip(q, (1, 2, 3))), sum(qi * wi for qi, wi in zip(q, (-1, 0, 4)))]
    assert C == [95, 1]

    want = []
    for c, swc in zip(C, sw):
        p = np.float32(float(Fraction(c) * Fraction(float(s))))
        want.append(np.float32(float(Fraction(float(p)) * Fraction(float(swc)))))
    want_bf = O.bf16_to_f32(O.f32_to_bf16(np.array(want, np.float32)))
    assert np.array_equal(got, want_bf), (got, want_bf)
    assert abs(float(got[0]) - 95 * 2 / 127 * 0.5) < 0.01 and abs(float(got[1]) - 2 / 127 * 0.25) < 1e-4


def test_linear_is_single_expert_grouped_gemm_on_quantized_rows():
    """The linear equals the oracle's grouped GEMM with one expert on the
    rows' own quantization, both schemes, and the float64 dequantized
    product within the float32 rounding bound."""
    rng = np.random.default_rng(17)
    T, K, N = 9, 256, 384
    x = (rng.standard_normal((T, K)) * 3).astype(np.float32)
    xb = O.f32_to_bf16(x)
    w = rng.integers(-127, 128, (N, K), dtype=np.int8)
    sw = (rng.random(N) * 1e-2).astype(np.float32)
    q, s = O.quantize_per_token(xb)
    got = O.linear_w8a8(xb, w, sw, "channel", "i32")
    assert np.array_equal(got, O.grouped_gemm_w8a8(q, s, w[None], sw[None], np.array([0, T]),
                                                   "channel", "i32"))
    ref = (q.astype(np.float64) * s[:, None].astype(np.float64)) @ (
        w.astype(np.float64) * sw[:, None].astype(np.float64)).T
    assert np.allclose(O.bf16_to_f32(got), ref, rtol=2 ** -7, atol=1e-6)
    swb = (rng.random((N // 128, K // 128)) * 1e-2).astype(np.float32)
    qb, sb = O.quantize_per_token_group(xb, 128)
    gotb = O.linear_w8a8(xb, w, swb, "block", "f32")
    assert np.array_equal(gotb, O.grouped_gemm_w8a8(qb, sb, w[None], swb[None], np.array([0, T]),
                                                    "block", "f32"))



def test_e4m3_decode_matches_torch_and_fixed_points():
    """Every one of the 256 e4m3 bytes decodes to torch's float8_e4m3fn value
    (a library conversion), and fixed points of the format hold: 0x38 = 1,
    0x7e = 448 (largest), 0x01 = 2^-9 (smallest subnormal), 0x08 = 2^-6,
    0x7f is NaN."""
    b = np.arange(256, dtype=np.uint8)
    got = O.e4m3_to_f32(b)
    want = torch.from_numpy(b).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert got[0x38] == 1.0 and got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9
    assert got[0x08] == 2.0 ** -6 and got[0xB8] == -1.0 and np.isnan(got[0x7F])


def test_fp8_dequant_and_conversion():
    """Dequantization = the byte's value times its block's scale, rounded to
    float32 then bf16 (checked against float64 products); the conversion's
    codes then follow the INT8 weight rules (a block whose bf16 values are
    already n * s quantizes back to n exactly)."""
    rng = np.random.default_rng(41)
    N, K = 256, 384
    w8 = rng.integers(0, 256, (N, K), dtype=np.uint8)
    w8[(w8 & 0x7F) == 0x7F] = 0x10  # no NaN bytes
    s8 = (rng.random((N // 128, K // 128)) * 1e-2 + 1e-4).astype(np.float32)
    bf = O.bf16_to_f32(O.dequant_fp8_block(w8, s8))
    v64 = O.e4m3_to_f32(w8).astype(np.float64) * np.repeat(np.repeat(s8, 128, 0), 128, 1)
    assert np.all(np.abs(bf - v64) <= np.abs(v64) * 2.0 ** -8 + 1e-30)
    q, s = O.convert_fp8_weights(w8, s8, "channel")
    q2, s2 = O.quantize_weight_channel(O.dequant_fp8_block(w8, s8))
    assert np.array_equal(q, q2) and np.array_equal(s, s2)
    # power-of-two block scale and codes of a single magnitude: values n * s
    w8b = np.full((128, 128), 0x38, np.uint8)  # 1.0 everywhere
    w8b[:, ::2] = 0xB8  # -1.0
    qb, sb = O.convert_fp8_weights(w8b, np.array([[0.25]], np.float32), "block")
    assert sb[0, 0] == np.float32(np.float32(0.25) / np.float32(127.0))
    assert np.all(np.abs(qb) == 127)


# ---------------------------------------------------------------------------
# W4A8 (int4 weights, int8 activations, masked layout)
# ---------------------------------------------------------------------------
def test_w4a8_golden():
    G = golden("w4a8_worked.json")
    u = G["unpack"]
    codes = O.unpack_int4(np.array(u["bytes"], np.uint8))
    assert codes.tolist() == u["codes"]
    assert O.pack_int4(codes).tolist() == u["bytes"]
    qg = G["quant"]
    w = np.array(qg["w"], np.float32)
    q, s = O.quantize_weight_int4(O.f32_to_bf16(w)[None, :])
    assert q[0].tolist() == qg["codes"] and float(s[0]) == qg["scale"]
    g = G["gemm"]
    a = np.array(g["a"], np.int8)[None]
    sa = np.array(g["sa"], np.float32)[None]
    W4 = np.array(g["w_bytes"], np.uint8)[None]
    assert O.pack_int4(np.array(g["w_codes"], np.int8)).tolist() == g["w_bytes"]
    out, valid = O.grouped_gemm_w4a8_masked(a, sa, np.array(g["masked_m"]), W4,
                                            np.array(g["s4"], np.float32)[None])
    m = g["masked_m"][0]
    assert valid[0].tolist() == [True] * m + [False] * (a.shape[1] - m)
    assert O.bf16_to_f32(out[0, :m, 0]).tolist() == g["out"]
    assert (O.int_matmul(a[0, :m], O.unpack_int4(W4[0])).reshape(-1)).tolist() == g["C"]


def test_int4_pack_round_trips():
    every = np.arange(256, dtype=np.uint8)
    codes = O.unpack_int4(every)
    assert codes.min() == -8 and codes.max() == 7
    assert np.array_equal(O.pack_int4(codes), every)
    pairs = np.array([(lo, hi) for lo in range(-8, 8) for hi in range(-8, 8)], np.int8)
    assert np.array_equal(O.unpack_int4(O.pack_int4(pairs)), pairs)


def test_quantize_weight_int4_invariants():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    w[3] = 0.0                      # a zero row
    w[4, :] = 0.01                  # an all-equal row
    wb = O.f32_to_bf16(w)
    wf = O.bf16_to_f32(wb)
    q, s = O.quantize_weight_int4(wb)
    assert q.dtype == np.int8 and np.abs(q).max() <= 7
    assert np.all(q[3] == 0) and s[3] == np.float32(1e-10) / np.float32(7.0)
    assert np.all(q[4] == 7)
    nz = np.abs(wf).max(1) > 0
    assert np.all(np.abs(q[nz]).max(1) == 7)  # the absmax element takes the end code
    # dequantization stays within half a scale step (plus float32 rounding)
    err = np.abs(s[:, None].astype(np.float64) * q - wf)
    assert np.all(err <= s[:, None] * (0.5 + 2.0 ** -20))
    # codes are the round-half-even of the exact quotient away from ties
    from fractions import Fraction
    for r in (0, 7, 63):
        for k in range(0, 256, 17):
            exact = Fraction(float(wf[r, k])) / Fraction(float(s[r]))
            if abs(abs(exact - int(exact)) - Fraction(1, 2)) > Fraction(1, 1 << 16):
                assert int(q[r, k]) == max(-7, min(7, round(exact)))


def test_w4a8_gemm_is_the_exact_integer_product():
    """The int4 GEMM's integer sums against an int64 einsum of the unpacked
    codes, and its outputs against the W8A8 masked GEMM on those codes
    (pinned in its own tests): a wrong nibble, sign or scale index fails."""
    rng = np.random.default_rng(6)
    E, Mmax, K, N = 3, 5, 64, 8
    a = rng.integers(-127, 128, (E, Mmax, K), dtype=np.int8)
    sa = (rng.random((E, Mmax)) * 0.05).astype(np.float32)
    codes = rng.integers(-7, 8, (E, N, K), dtype=np.int8)
    W4 = O.pack_int4(codes)
    S4 = (rng.random((E, N)) * 1e-2).astype(np.float32)
    mm = np.array([5, 0, 3])
    out, valid = O.grouped_gemm_w4a8_masked(a, sa, mm, W4, S4)
    for e in range(E):
        m = mm[e]
        C = np.einsum("rk,nk->rn", a[e, :m].astype(np.int64), codes[e].astype(np.int64))
        assert np.array_equal(O.int_matmul(a[e, :m], O.unpack_int4(W4[e])), C)
        want = O.f32_to_bf16(O.gemm_dequant(a[e, :m], sa[e, :m], codes[e], S4[e], "channel", "i32"))
        assert np.array_equal(out[e, :m], want)
    assert valid.sum() == mm.sum()
