"""Parity at the full DeepSeek-V3 layer sizes, in the launch configuration the
benchmark times (the one-call layer, all 256 experts resident).

Inputs are drawn on the GPU (the weights one expert at a time) and quantized
by the library.  Compared with the oracle:
  * in full: routing ids and weights, activation codes and scales, expert
    counts/offsets, the stable permutation and its inverse;
  * on sampled tokens, evaluated by the oracle one token at a time with its
    own quantization of those experts' bf16 weights: the int8 weights of the
    touched experts, the int32 accumulators of GEMM1 and the final bf16
    outputs (exactly, and against the stated tolerance)."""
import numpy as np
import pytest
import torch

from oracle import wq_oracle as O
from w8a8_int8_quantized_token_gb300 import binding as wq
from w8a8_int8_quantized_token_gb300 import synth
from wq_testutil import assert_bf16_equal, bits, np_, tolerance_report

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _init():
    from w8a8_int8_quantized_token_gb300 import build_lib
    build_lib.build()
    wq.init(0)


def gpu_weights(cfg):
    E, I, H = cfg.E, cfg.I, cfg.H
    blk = cfg.scheme == "block"
    W13 = torch.empty(E, 2 * I, H, dtype=torch.int8, device=DEV)
    W2 = torch.empty(E, H, I, dtype=torch.int8, device=DEV)
    S13 = torch.empty((E, 2 * I // 128, H // 128) if blk else (E, 2 * I), dtype=torch.float32, device=DEV)
    S2 = torch.empty((E, H // 128, I // 128) if blk else (E, H), dtype=torch.float32, device=DEV)
    for e in range(E):
        w13, w2 = synth.expert_weights(cfg, e, device=DEV)
        wq.quantize_weight(w13, cfg.scheme, W13[e], S13[e])
        wq.quantize_weight(w2, cfg.scheme, W2[e], S2[e])
    return W13, S13, W2, S2


def oracle_expert(cfg, e, cache):
    """The oracle's own quantization of expert e's bf16 weights (drawn by the
    same seeded generator on the GPU, copied to the host)."""
    if e not in cache:
        w13, w2 = synth.expert_weights(cfg, e, device=DEV)
        cache[e] = O.quantize_weights(bits(w13), bits(w2), cfg.scheme)
    return cache[e]


def check_expert_weights(gpu_w, oq, e):
    W13, S13, W2, S2 = gpu_w
    q13, s13, q2, s2 = oq
    assert np.array_equal(np_(W13[e]), q13) and np.array_equal(np_(S13[e]), s13)
    assert np.array_equal(np_(W2[e]), q2) and np.array_equal(np_(S2[e]), s2)


def token_output(cfg, x_row_bits, ids, w, oq_of):
    """Oracle value of one token: its k experts evaluated directly."""
    grp = 0 if cfg.scheme == "channel" else 128
    if cfg.scheme == "channel":
        q, s = O.quantize_per_token(x_row_bits[None])
    else:
        q, s = O.quantize_per_token_group(x_row_bits[None], 128)
    acc = np.zeros(cfg.H, np.float32)
    gemm1_i32 = []
    for j, e in enumerate(ids):
        q13, s13, q2, s2 = oq_of(int(e))
        gemm1_i32.append(O.int_matmul(q, q13)[0])
        gu = O.f32_to_bf16(O.gemm_dequant(q, s, q13, s13, cfg.scheme, cfg.acc))
        hq, sh = O.silu_mul_quant(gu, cfg.I, grp)
        y = O.f32_to_bf16(O.gemm_dequant(hq, sh, q2, s2, cfg.scheme, cfg.acc))
        acc = acc + w[j] * O.bf16_to_f32(y[0])
    return O.f32_to_bf16(acc), gemm1_i32


@pytest.mark.parametrize("name", ["decode", "prefill", "prefill_f32", "block"])
def test_layer_full_size(name):
    cfg = synth.CONFIGS[name]
    x, lg = synth.layer_inputs(cfg, device=DEV)
    gw = gpu_weights(cfg)
    st = wq.new_status()
    out = wq.moe_forward(x, lg, *gw, cfg.k, cfg.scheme, cfg.acc, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    xb, lgn = bits(x), np_(lg)

    # routing, codes and alignment, in full
    ids, w = wq.route_topk(lg, cfg.k)
    io, wo = O.route_topk(lgn, cfg.k)
    assert np.array_equal(np_(ids), io) and np.array_equal(np_(w), wo)
    if cfg.scheme == "channel":
        q, s = wq.quantize_per_token(x)
        qo, so = O.quantize_per_token(xb)
    else:
        q, s = wq.quantize_per_token_group(x, 128)
        qo, so = O.quantize_per_token_group(xb, 128)
    assert np.array_equal(np_(q), qo) and np.array_equal(np_(s), so)
    c, off, sp, p2r = wq.moe_align(ids, cfg.E)
    co, offo, spo, p2ro = O.moe_align(io, cfg.E)
    assert np.array_equal(np_(c), co) and np.array_equal(np_(off), offo)
    assert np.array_equal(np_(sp), spo) and np.array_equal(np_(p2r), p2ro)

    # GEMM1 int32 accumulators of the permuted rows (channel, int32 mode)
    A, sa = wq.moe_permute(q, s, sp, cfg.k)
    gemm1_raw = None
    if cfg.scheme == "channel" and cfg.acc == "i32":
        gemm1_raw = wq.grouped_gemm_w8a8(A, sa, gw[0], gw[1], off, "channel", "i32", out_type="i32")

    # final outputs of sampled tokens, evaluated token by token by the oracle
    rng = np.random.default_rng(11)
    toks = sorted({0, cfg.T - 1, *rng.choice(cfg.T, 2, replace=False).tolist()})
    cache = {}
    ob = bits(out)
    got, want = [], []
    for t in toks:
        for e in io[t]:
            check_expert_weights(gw, oracle_expert(cfg, int(e), cache), int(e))
        ref, g1 = token_output(cfg, xb[t], io[t], wo[t], lambda e: oracle_expert(cfg, e, cache))
        got.append(ob[t])
        want.append(ref)
        if gemm1_raw is not None:
            for j in range(cfg.k):
                row = int(p2ro[t * cfg.k + j])
                assert np.array_equal(np_(gemm1_raw[row]), g1[j].astype(np.int32)), (t, j)
    got, want = np.stack(got), np.stack(want)
    max_abs, rel = tolerance_report(got, want)
    assert max_abs <= 2e-2 and rel <= 1e-2, (max_abs, rel)
    assert_bf16_equal(got, want, f"{name} sampled tokens {toks}")


def test_masked_full_size():
    cfg = synth.CONFIGS["masked"]
    xm, mm = synth.masked_inputs(cfg, device=DEV)
    E, Mmax, H = cfg.E, cfg.Mmax, cfg.H
    a, sa = wq.quantize_per_token(xm.reshape(E * Mmax, H))
    gw = gpu_weights(cfg)
    y = torch.full((E, Mmax, H), 3.0, dtype=torch.bfloat16, device=DEV)
    st = wq.new_status()
    wq.moe_forward_masked(a.view(E, Mmax, H), sa.view(E, Mmax), torch.from_numpy(mm).to(DEV), *gw,
                          y=y, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert mm.sum() > 0
    yb = bits(y)
    # rows at or past the counts stay untouched
    for e in range(E):
        assert np.all(O.bf16_to_f32(yb[e, mm[e]:]) == 3.0)
    # sampled valid rows, evaluated by the oracle one row at a time
    rng = np.random.default_rng(5)
    experts = sorted({int(np.argmax(mm)), int(np.argmin(mm)), *rng.choice(E, 2, replace=False).tolist()})
    cache = {}
    got, want = [], []
    for e in experts:
        oq = oracle_expert(cfg, e, cache)
        check_expert_weights(gw, oq, e)
        rows = sorted({0, int(mm[e]) - 1})
        xr = bits(xm[e, rows])
        q, s = O.quantize_per_token(xr)
        gu = O.f32_to_bf16(O.gemm_dequant(q, s, oq[0], oq[1], "channel", "i32"))
        hq, sh = O.silu_mul_quant(gu, cfg.I)
        ref = O.f32_to_bf16(O.gemm_dequant(hq, sh, oq[2], oq[3], "channel", "i32"))
        got.append(yb[e, rows])
        want.append(ref)
    got, want = np.concatenate(got), np.concatenate(want)
    max_abs, rel = tolerance_report(got, want)
    assert max_abs <= 2e-2 and rel <= 1e-2, (max_abs, rel)
    assert_bf16_equal(got, want, "masked sampled rows")


@pytest.mark.parametrize("name", ["block", "prefill", "decode"])
def test_layer_repeatable(name):
    """The full-size layer run again and again on fresh copies of its inputs
    gives the same bits every time (a staging-ring hand-off that lets a copy
    land early shows up here as an occasional differing run)."""
    cfg = synth.CONFIGS[name]
    x, lg = synth.layer_inputs(cfg, device=DEV)
    gw = gpu_weights(cfg)
    st = wq.new_status()
    first = wq.moe_forward(x, lg, *gw, cfg.k, cfg.scheme, cfg.acc, status=st).clone()
    for i in range(12):
        out = wq.moe_forward(x.clone(), lg.clone(), *gw, cfg.k, cfg.scheme, cfg.acc, status=st)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), first.view(torch.int16)), f"run {i + 1} differs"
    assert int(st.item()) == 0


@pytest.mark.parametrize("T", [8192, 128])
def test_linear_full_size(T):
    """The dense W8A8 linear at a DeepSeek-V3 dense-MLP gate_up shape (K
    7168, N 36864): sampled rows against the oracle's linear on the same
    weights."""
    K, N = 7168, 36864
    g = torch.Generator(device=DEV).manual_seed(3)
    x = torch.randn(T, K, generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    Wq, sw = wq.quantize_weight(w, "channel")
    del w
    st = wq.new_status()
    out = wq.linear_w8a8(x, Wq, sw, "channel", "i32", status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = sorted({0, T - 1, T // 3})
    ref = O.linear_w8a8(bits(x[rows]), np_(Wq), np_(sw), "channel", "i32")
    got = bits(out[rows])
    max_abs, rel = tolerance_report(got, ref)
    assert max_abs <= 2e-2 and rel <= 1e-2
    assert_bf16_equal(got, ref, f"linear T{T} sampled rows {rows}")
