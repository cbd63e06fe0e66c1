"""Parity of every step of the CUDA path with the CPU oracle, through the C
ABI.  Integer results (codes, ids, offsets, permutations, int32
accumulators) are compared bit-exactly; bf16 and float results are compared
exactly too (the kernels follow the oracle's float32 operation order), and
the layer outputs also report the stated tolerance (max abs 2e-2, relative
Frobenius 1e-2)."""
import numpy as np
import pytest
import torch

from oracle import wq_oracle as O
from w8a8_int8_quantized_token_gb300 import binding as wq
from w8a8_int8_quantized_token_gb300 import synth
from wq_testutil import assert_bf16_equal, bits, np_, quantized_weights, stack_oracle, tolerance_report

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _init():
    from w8a8_int8_quantized_token_gb300 import build_lib
    build_lib.build()
    wq.init(0)


# ---------------------------------------------------------------- quantization
@pytest.mark.parametrize("T,K,outl", [(1, 8, False), (37, 384, True), (130, 7168, True),
                                      (5, 2048, False), (3, 65536, True)])
def test_quantize_per_token(T, K, outl):
    x = synth.activations(T, K, outl, seed=T + K)
    q, s = wq.quantize_per_token(x.to(DEV))
    qo, so = O.quantize_per_token(bits(x))
    assert np.array_equal(np_(q), qo)
    assert np.array_equal(np_(s), so)


def test_quantize_zero_and_constant_rows():
    x = torch.zeros(3, 256, dtype=torch.bfloat16)
    x[1] = -0.375
    x[2, 7] = 3.0
    q, s = wq.quantize_per_token(x.to(DEV))
    qo, so = O.quantize_per_token(bits(x))
    assert np.array_equal(np_(q), qo) and np.array_equal(np_(s), so)
    assert np.all(np_(q)[1] == -127) and np.all(np_(q)[0] == 0)


def test_quantize_exact_half_integer_quotients():
    """Rows whose scale is a power of two (absmax = 127 * 2^j) so that x / s
    is exactly every half-integer in (-127, 127) and every integer: the codes
    of the half-integers take the ties-to-even rule through the
    exact-quotient branch."""
    K = 512
    rows = []
    for j in (-3, 0, 2):
        h = (np.arange(-127, 127) + 0.5) * 2.0 ** j
        n = np.arange(-127, 128) * 2.0 ** j
        rows.append(np.resize(np.concatenate([[127 * 2.0 ** j], h, n]), K))
    x = torch.tensor(np.stack(rows), dtype=torch.float32)
    assert torch.equal(x.to(torch.bfloat16).float(), x)  # exact in bf16
    x = x.to(torch.bfloat16)
    q, s = wq.quantize_per_token(x.to(DEV))
    qo, so = O.quantize_per_token(bits(x))
    assert np.array_equal(np_(s), so) and np.all(so == 2.0 ** np.array([-3, 0, 2], np.float32))
    assert np.array_equal(np_(q), qo)
    assert qo[1, 1 + 127] == 0 and qo[1, 1 + 128] == 2  # 0.5 -> 0, 1.5 -> 2
    qg, sg = wq.quantize_per_token_group(x.to(DEV), 128)
    qgo, sgo = O.quantize_per_token_group(bits(x), 128)
    assert np.array_equal(np_(qg), qgo) and np.array_equal(np_(sg), sgo)


@pytest.mark.parametrize("group", [32, 64, 128, 256])
def test_quantize_per_token_group(group):
    x = synth.activations(19, 1024, True, seed=group)
    q, s = wq.quantize_per_token_group(x.to(DEV), group)
    qo, so = O.quantize_per_token_group(bits(x), group)
    assert np.array_equal(np_(q), qo) and np.array_equal(np_(s), so)


def test_quantize_weight_block():
    g = torch.Generator().manual_seed(4)
    w = (torch.randn(384, 640, generator=g) * 0.02).to(torch.bfloat16)
    q, s = wq.quantize_weight_block(w.to(DEV))
    qo, so = O.quantize_weight_block(bits(w))
    assert np.array_equal(np_(q), qo) and np.array_equal(np_(s), so)


# ---------------------------------------------------------------- routing / align / permute
@pytest.mark.parametrize("T,E,k", [(16, 8, 2), (200, 256, 8), (33, 1024, 32), (9, 5, 5), (7, 300, 1)])
def test_route_topk(T, E, k):
    lg = synth.router_logits(T, E, seed=E + k)
    lg[:, 3] = lg[:, 1]  # exact ties
    ids, w = wq.route_topk(lg.to(DEV), k)
    io, wo = O.route_topk(lg.numpy(), k)
    assert np.array_equal(np_(ids), io)
    assert np.array_equal(np_(w), wo)


@pytest.mark.parametrize("T,k,E,pad", [(3, 2, 4, 1), (3, 2, 4, 4), (1000, 8, 256, 1),
                                       (8192, 8, 256, 1), (77, 3, 4096, 1), (500, 6, 33, 128), (0, 2, 8, 1)])
def test_moe_align(T, k, E, pad):
    rng = np.random.default_rng(T + E)
    ids = np.array([rng.choice(E, k, replace=False) for _ in range(T)], np.int32).reshape(T, k)
    if T:
        ids[: T // 2, 0] = 1  # a hot expert
    c, o, sp, p2r = wq.moe_align(torch.from_numpy(ids).to(DEV), E, pad)
    co, oo, spo, p2ro = O.moe_align(ids, E, pad)
    assert np.array_equal(np_(c), co) and np.array_equal(np_(o), oo)
    n = int(oo[-1])
    assert np.array_equal(np_(sp)[:n], spo) and np.all(np_(sp)[n:] == -1)
    assert np.array_equal(np_(p2r), p2ro)


def test_moe_align_reports_bad_ids():
    ids = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32, device=DEV)
    st = wq.new_status()
    c, o, sp, p2r = wq.moe_align(ids, 4, 1, status=st)
    assert int(st.item()) == -6
    assert np_(p2r).tolist()[3] == -1 and np_(c).tolist() == [1, 1, 1, 0]


@pytest.mark.parametrize("groups", [1, 56])
def test_moe_permute(groups):
    T, k, E, K = 300, 8, 64, 7168
    rng = np.random.default_rng(groups)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    q = rng.integers(-127, 128, (T, K), dtype=np.int8)
    s = rng.random((T, groups) if groups > 1 else T).astype(np.float32)
    _, _, spo, _ = O.moe_align(ids, E, 4)
    A, sa = wq.moe_permute(torch.from_numpy(q).to(DEV), torch.from_numpy(s).to(DEV),
                           torch.from_numpy(spo).to(DEV), k)
    Ao, sao = O.moe_permute(q, s, spo, k)
    assert np.array_equal(np_(A), Ao) and np.array_equal(np_(sa), sao)


# ---------------------------------------------------------------- activation / combine
@pytest.mark.parametrize("R,I,group", [(70, 2048, 0), (5, 128, 0), (33, 2048, 128), (9, 256, 32),
                                       (3, 16384, 0)])
def test_silu_mul_quant(R, I, group):
    g = torch.Generator().manual_seed(R + I)
    gu = (torch.randn(R, 2 * I, generator=g) * 4).to(torch.bfloat16)
    gu[0, :4] = torch.tensor([0.0, -120.0, 95.0, -0.0])  # saturated exp paths
    hq, sh = wq.silu_mul_quant(gu.to(DEV), group)
    hqo, sho = O.silu_mul_quant(bits(gu), I, group)
    assert np.array_equal(np_(hq), hqo) and np.array_equal(np_(sh), sho)


@pytest.mark.parametrize("T,k,H", [(129, 8, 7168), (3, 8, 7168), (1, 1, 8), (64, 16, 512),
                                   (5, 32, 256), (200, 2, 1032)])
def test_moe_combine(T, k, H):
    """Every k up to 32 (register sets of 8, 16 and 32 rows), few tokens (rows
    split over several CTAs), odd widths; a -1 row contributes nothing."""
    rng = np.random.default_rng(3 + T + k)
    y = (torch.randn(T * k + 5, H, generator=torch.Generator().manual_seed(1)) * 3).to(torch.bfloat16)
    p2r = rng.permutation(T * k).astype(np.int32)
    p2r[min(5, T * k - 1)] = -1
    w = rng.random((T, k)).astype(np.float32)
    out = wq.moe_combine(y.to(DEV), torch.from_numpy(p2r).to(DEV), torch.from_numpy(w).to(DEV), k)
    yb = bits(y)
    # the oracle's combine takes the rows by index; a -1 row contributes nothing
    yz = np.concatenate([yb, np.zeros((1, H), np.uint16)])
    p2r_o = np.where(p2r < 0, yb.shape[0], p2r)
    assert_bf16_equal(bits(out), O.moe_combine(yz, p2r_o, w, k), "combine")


def test_moe_combine_refuses_k_above_32():
    y = torch.zeros(33, 8, dtype=torch.bfloat16, device=DEV)
    p2r = torch.arange(33, dtype=torch.int32, device=DEV)
    w = torch.ones(1, 33, device=DEV)
    with pytest.raises(wq.WQError):
        wq.moe_combine(y, p2r, w, 33)


# ---------------------------------------------------------------- grouped GEMM
def _gemm_case(seed, E, counts, N, K, scheme):
    rng = np.random.default_rng(seed)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offsets[-1])
    A = rng.integers(-127, 128, (R, K), dtype=np.int8)
    W = rng.integers(-127, 128, (E, N, K), dtype=np.int8)
    if scheme == "channel":
        sa = (rng.random(R) * 0.05).astype(np.float32)
        sw = (rng.random((E, N)) * 1e-3).astype(np.float32)
    else:
        sa = (rng.random((R, K // 128)) * 0.05).astype(np.float32)
        sw = (rng.random((E, N // 128, K // 128)) * 1e-3).astype(np.float32)
    return A, sa, W, sw, offsets


@pytest.mark.parametrize("scheme,acc", [("channel", "i32"), ("channel", "f32"), ("block", "f32")])
@pytest.mark.parametrize("counts,N,K", [([3, 0, 130, 1, 257], 256, 384),
                                         ([0, 0, 5], 128, 128),
                                         ([700, 64, 129], 512, 1024),
                                         ([300, 0, 1, 555], 768, 2304),
                                         # few rows per expert: the 64-row token tiles
                                         ([0, 1, 5, 16, 17, 63, 64, 65, 130, 3, 2, 0, 7, 9, 33, 40],
                                          256, 512)])
def test_grouped_gemm(scheme, acc, counts, N, K):
    E = len(counts)
    A, sa, W, sw, offs = _gemm_case(len(counts) + N + K, E, counts, N, K, scheme)
    t = lambda a: torch.from_numpy(a).to(DEV)
    st = wq.new_status()
    out = wq.grouped_gemm_w8a8(t(A), t(sa), t(W), t(sw), t(offs), scheme, acc, status=st)
    ref = O.grouped_gemm_w8a8(A, sa, W, sw, offs, scheme, acc)
    assert int(st.item()) == 0
    assert_bf16_equal(bits(out), ref, f"gemm {scheme}/{acc}")


@pytest.mark.parametrize("scheme,acc", [("channel", "i32"), ("channel", "f32"), ("block", "f32")])
def test_grouped_gemm_few_tokens_per_expert(scheme, acc):
    """Decode-like segments (0..16 rows, each size present) and small
    remainders of larger segments: the small-token engine's tiles of 1..16
    rows (token boxes 4, 8, 16); the channel-wise cases use a channel count
    that leaves idle lanes in the last 256-channel block."""
    counts = list(range(17)) + [33, 256 + 5, 128 + 16, 2 * 64 + 3]
    E, N, K = len(counts), 384 if scheme == "channel" else 512, 1024
    A, sa, W, sw, offs = _gemm_case(31, E, counts, N, K, scheme)
    t = lambda a: torch.from_numpy(a).to(DEV)
    st = wq.new_status()
    out = wq.grouped_gemm_w8a8(t(A), t(sa), t(W), t(sw), t(offs), scheme, acc, status=st)
    assert_bf16_equal(bits(out), O.grouped_gemm_w8a8(A, sa, W, sw, offs, scheme, acc),
                      f"few-token gemm {scheme}/{acc}")
    if scheme == "channel" and acc == "i32":
        C = wq.grouped_gemm_w8a8(t(A), t(sa), t(W), t(sw), t(offs), "channel", "i32",
                                 out_type="i32", status=st)
        assert np.array_equal(np_(C), O.grouped_gemm_i32(A, W, offs))
    assert int(st.item()) == 0


def test_grouped_gemm_int32_accumulators_and_extremes():
    E, counts, N, K = 3, [200, 1, 77], 256, 7168
    A, sa, W, sw, offs = _gemm_case(9, E, counts, N, K, "channel")
    A[0, :] = 127
    W[0, 0, :] = 127
    W[0, 1, :] = -127
    A[1, :] = -127
    t = lambda a: torch.from_numpy(a).to(DEV)
    st = wq.new_status()
    C = wq.grouped_gemm_w8a8(t(A), t(sa), t(W), t(sw), t(offs), "channel", "i32", out_type="i32",
                             status=st)
    Co = O.grouped_gemm_i32(A, W, offs)
    assert int(st.item()) == 0
    assert np.array_equal(np_(C), Co)
    assert Co[0, 0] == 127 * 127 * 7168 and Co[0, 1] == -127 * 127 * 7168


def test_grouped_gemm_f32_accumulator_extremes():
    """Float32-accumulator mode on rows whose sums exceed 2^24 (one of them
    odd): the single-pass engine cannot prove these tiles exact and the
    chunked recompute adds the 128-wide tile sums in order."""
    E, counts, N, K = 3, [200, 1, 77], 256, 7168
    A, sa, W, sw, offs = _gemm_case(10, E, counts, N, K, "channel")
    A[0, :] = 127
    W[0, 0, :] = 127
    W[0, 0, 5] = 126
    W[0, 1, :] = -127
    t = lambda a: torch.from_numpy(a).to(DEV)
    st = wq.new_status()
    out = wq.grouped_gemm_w8a8(t(A), t(sa), t(W), t(sw), t(offs), "channel", "f32", status=st)
    assert int(st.item()) == 0
    assert_bf16_equal(bits(out), O.grouped_gemm_w8a8(A, sa, W, sw, offs, "channel", "f32"),
                      "gemm channel/f32 extremes")


def test_grouped_gemm_leaves_rows_outside_segments():
    E, N, K = 2, 128, 256
    rng = np.random.default_rng(5)
    offs = np.array([0, 10, 20], np.int32)
    R = 32  # rows 20..31 belong to no expert
    A = rng.integers(-127, 128, (R, K), dtype=np.int8)
    W = rng.integers(-127, 128, (E, N, K), dtype=np.int8)
    sa = np.ones(R, np.float32)
    sw = np.full((E, N), 1e-3, np.float32)
    t = lambda a: torch.from_numpy(a).to(DEV)
    out = torch.full((R, N), 7.0, dtype=torch.bfloat16, device=DEV)
    wq.grouped_gemm_w8a8(t(A), t(sa), t(W), t(sw), t(offs), out=out)
    assert torch.all(out[20:] == 7.0)
    assert_bf16_equal(bits(out[:20]), O.grouped_gemm_w8a8(A[:20], sa[:20], W, sw, offs))


@pytest.mark.parametrize("scheme,acc", [("channel", "i32"), ("block", "f32")])
def test_grouped_gemm_masked(scheme, acc):
    E, Mmax, N, K = 5, 200, 256, 512
    mm = np.array([0, 1, 200, 129, 64], np.int32)
    rng = np.random.default_rng(6)
    A = rng.integers(-127, 128, (E, Mmax, K), dtype=np.int8)
    W = rng.integers(-127, 128, (E, N, K), dtype=np.int8)
    if scheme == "channel":
        sa = (rng.random((E, Mmax)) * 0.05).astype(np.float32)
        sw = (rng.random((E, N)) * 1e-3).astype(np.float32)
    else:
        sa = (rng.random((E, Mmax, K // 128)) * 0.05).astype(np.float32)
        sw = (rng.random((E, N // 128, K // 128)) * 1e-3).astype(np.float32)
    t = lambda a: torch.from_numpy(a).to(DEV)
    out = torch.full((E, Mmax, N), -3.0, dtype=torch.bfloat16, device=DEV)
    wq.grouped_gemm_w8a8_masked(t(A), t(sa), t(mm), t(W), t(sw), scheme, acc, out=out)
    ob = bits(out)
    for e in range(E):
        m = mm[e]
        ref = O.grouped_gemm_w8a8(A[e, :m], sa[e, :m], W[e:e + 1], sw[e:e + 1], np.array([0, m]),
                                  scheme, acc)
        assert_bf16_equal(ob[e, :m], ref, f"masked expert {e}")
        assert np.all(O.bf16_to_f32(ob[e, m:]) == -3.0)


def test_grouped_gemm_masked_norm_bound_fails():
    """Masked layout, channel scheme, 256-token tiles: the launch sums its
    valid rows' squared norms once for the int8-code engine's exactness
    check.  A row of 127s against a weight row of 127s with one 126 (an odd
    sum above 2^24) fails the bound, so the exact recompute must run: every
    int32 accumulator equals the oracle's."""
    E, Mmax, N, K = 3, 300, 256, 7168
    mm = np.array([300, 40, 5], np.int32)
    rng = np.random.default_rng(12)
    A = rng.integers(-127, 128, (E, Mmax, K), dtype=np.int8)
    W = rng.integers(-127, 128, (E, N, K), dtype=np.int8)
    A[0, 7, :] = 127
    W[0, 0, :] = 127
    W[0, 0, 5] = 126
    A[1, 3, :] = -127
    W[1, 1, :] = 127
    sa = (rng.random((E, Mmax)) * 0.05).astype(np.float32)
    sw = (rng.random((E, N)) * 1e-3).astype(np.float32)
    t = lambda a: torch.from_numpy(a).to(DEV)
    st = wq.new_status()
    out = torch.full((E, Mmax, N), -3, dtype=torch.int32, device=DEV)
    wq.grouped_gemm_w8a8_masked(t(A), t(sa), t(mm), t(W), t(sw), "channel", "i32", out_type="i32",
                                out=out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o = np_(out)
    for e in range(E):
        m = int(mm[e])
        Co = O.grouped_gemm_i32(A[e, :m], W[e:e + 1], np.array([0, m]))
        assert np.array_equal(o[e, :m], Co), f"masked expert {e}"
        assert np.all(o[e, m:] == -3)
    assert o[0, 7, 0] == 127 * (127 * (K - 1) + 126) and o[1, 3, 1] == -127 * 127 * K


# ---------------------------------------------------------------- the layer
def _layer_case(cfg):
    x, lg = synth.layer_inputs(cfg)
    (W13, S13, W2, S2), orc = quantized_weights(cfg, DEV)
    ow = stack_oracle(orc, cfg.E)
    for gpu, ref in zip((W13, S13, W2, S2), ow):
        assert np.array_equal(np_(gpu), ref), "weight quantization differs"
    return x, lg, (W13, S13, W2, S2), ow


@pytest.mark.parametrize("cfg", [
    synth.CONFIGS["tiny"],
    synth.small_config("small_i32", T=150, H=384, I=256, E=6, k=3),
    synth.small_config("small_f32", T=97, H=512, I=256, E=7, k=2, acc="f32"),
    synth.small_config("small_block", T=130, H=384, I=256, E=5, k=3, scheme="block", acc="f32"),
    # widths multiples of 256 and many rows per expert: the fp16-code block engine
    synth.small_config("small_block_f16", T=300, H=512, I=256, E=4, k=2, scheme="block", acc="f32"),
    synth.small_config("hot", T=300, H=256, I=128, E=4, k=1),
    # K >= 1024 with many rows per expert: GEMM1 on the tensor-memory-weights
    # pair engine within a small layer
    synth.small_config("small_k1024", T=300, H=1024, I=256, E=4, k=2),
    synth.small_config("small_k2048_f32", T=260, H=2048, I=256, E=3, k=2, acc="f32"),
], ids=lambda c: c.name)
def test_layer_forward(cfg):
    x, lg, w, ow = _layer_case(cfg)
    st = wq.new_status()
    out = wq.moe_forward(x.to(DEV), lg.to(DEV), *w, cfg.k, cfg.scheme, cfg.acc, status=st)
    ref = O.moe_forward(bits(x), lg.numpy(), *ow, cfg.k, cfg.scheme, cfg.acc)
    assert int(st.item()) == 0
    max_abs, rel = tolerance_report(bits(out), ref)
    assert max_abs <= 2e-2 and rel <= 1e-2
    assert_bf16_equal(bits(out), ref, f"layer {cfg.name}")


def test_layer_forward_host_equals_device():
    cfg = synth.small_config("host", T=64, H=256, I=128, E=8, k=2)
    x, lg, w, _ = _layer_case(cfg)
    dev_out = wq.moe_forward(x.to(DEV), lg.to(DEV), *w, cfg.k)
    xh, lh = x.pin_memory(), lg.pin_memory()
    host_out = wq.moe_forward_host(xh, lh, *w, cfg.k)
    torch.cuda.synchronize()
    assert torch.equal(host_out.view(torch.int16), dev_out.cpu().view(torch.int16))


def test_layer_forward_masked():
    cfg = synth.small_config("masked_small", T=0, H=256, I=128, E=4, k=1)
    Mmax = 150
    x = synth.activations(cfg.E * Mmax, cfg.H, True, 3)
    a, sa = wq.quantize_per_token(x.to(DEV))
    qo, so = O.quantize_per_token(bits(x))
    mm = np.array([150, 0, 1, 77], np.int32)
    (W13, S13, W2, S2), orc = quantized_weights(cfg, DEV)
    y = torch.full((cfg.E, Mmax, cfg.H), 5.0, dtype=torch.bfloat16, device=DEV)
    wq.moe_forward_masked(a.view(cfg.E, Mmax, cfg.H), sa.view(cfg.E, Mmax),
                          torch.from_numpy(mm).to(DEV), W13, S13, W2, S2, y=y)
    ref, valid = O.moe_forward_masked(qo.reshape(cfg.E, Mmax, cfg.H), so.reshape(cfg.E, Mmax), mm,
                                      *stack_oracle(orc, cfg.E))
    yb = bits(y)
    assert_bf16_equal(yb[valid], ref[valid], "masked layer")
    assert np.all(O.bf16_to_f32(yb[~valid]) == 5.0)


def test_layer_forward_masked_norm_bound_fails():
    """The masked layer hands the int8-code engine its rows' squared norms
    (computed once per launch) instead of having it sum them stage by stage.
    With every activation code at 127 and K = 7168 the exactness bound
    ||a||^2 ||w||^2 < 2^48 fails, so the gated exact recompute must run; the
    output still equals the oracle's, and so do the rows of the experts the
    small-token engine takes."""
    cfg = synth.small_config("masked_extreme", T=0, H=7168, I=256, E=3, k=1)
    Mmax = 300
    qo = np.full((cfg.E, Mmax, cfg.H), 127, np.int8)
    qo[1, :, ::7] = -127
    so = np.random.default_rng(5).random((cfg.E, Mmax)).astype(np.float32) * 1e-3 + 1e-4
    mm = np.array([300, 40, 5], np.int32)
    (W13, S13, W2, S2), orc = quantized_weights(cfg, DEV)
    y = torch.full((cfg.E, Mmax, cfg.H), 5.0, dtype=torch.bfloat16, device=DEV)
    st = wq.new_status()
    wq.moe_forward_masked(torch.from_numpy(qo).to(DEV), torch.from_numpy(so).to(DEV),
                          torch.from_numpy(mm).to(DEV), W13, S13, W2, S2, y=y, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref, valid = O.moe_forward_masked(qo, so, mm, *stack_oracle(orc, cfg.E))
    yb = bits(y)
    assert_bf16_equal(yb[valid], ref[valid], "masked layer, bound failing")
    assert np.all(O.bf16_to_f32(yb[~valid]) == 5.0)


@pytest.mark.parametrize("group", [0, 128])
@pytest.mark.parametrize("f16", [False, True])
def test_silu_mul_quant_every_bf16_gate(group, f16):
    """Every finite bf16 gate value g (65280 patterns: both signs, subnormals,
    zeros, the largest) through SiLU-mul + re-quantization: the kernel looks
    silu(g) up in a table for |g| in [2^-24, 89), either sign, and takes the
    formula elsewhere; codes and scales must equal the oracle's.  The
    patterns are sorted by magnitude so the values sharing a row (or a
    128-group) are alike and their codes carry information; |u| < 1 keeps
    every product finite."""
    I = 2048
    b = np.arange(65536, dtype=np.uint32)
    finite = (b & 0x7F80) != 0x7F80
    pats = b[finite].astype(np.uint16)
    pats = pats[np.argsort(O.bf16_to_f32(pats).astype(np.float64) ** 2, kind="stable")]
    R = (pats.size + I - 1) // I
    g = np.zeros(R * I, np.uint16)
    g[:pats.size] = pats
    rng = np.random.default_rng(31)
    u = O.f32_to_bf16((rng.random(R * I) * 1.8 - 0.9).astype(np.float32))
    gu = np.concatenate([g.reshape(R, I), u.reshape(R, I)], axis=1)
    gut = torch.from_numpy(gu.view(np.int16)).view(torch.bfloat16).to(DEV)
    hqo, sho = O.silu_mul_quant(gu, I, group)
    if f16:
        hq, sh, n2 = wq.silu_mul_quant_f16(gut, group)
        assert np.array_equal(np_(hq).astype(np.int32), hqo.astype(np.int32))
        if group == 0:
            assert np.array_equal(np_(n2), (hqo.astype(np.int64) ** 2).sum(1))
    else:
        hq, sh = wq.silu_mul_quant(gut, group)
        assert np.array_equal(np_(hq), hqo)
    assert np.array_equal(np_(sh).reshape(sho.shape), sho)


@pytest.mark.parametrize("R,I,group", [(1, 8, 0), (3, 24, 0), (2, 256, 32), (40, 1024, 64),
                                       (17, 2048, 256), (6, 1544, 0), (5, 1280, 128),
                                       (6000, 2048, 0), (5, 4096, 0), (4, 4096, 128)])
def test_silu_mul_quant_shapes(R, I, group):
    """Row widths around the table kernel's per-lane vector counts (1 to 4
    vectors of 8 per lane, partly filled last vectors), rows split between
    two warps (I > 1024, the second warp's part partly filled at I = 1544 and
    1280), more rows than the launch has row slots (R = 6000: each warp pair
    takes several rows, reusing its exchange slots), every group size, and
    rows too wide for it (I = 4096: the block-per-row kernels)."""
    g = torch.Generator().manual_seed(R * 7 + I)
    gu = (torch.randn(R, 2 * I, generator=g) * 3).to(torch.bfloat16)
    hq, sh = wq.silu_mul_quant(gu.to(DEV), group)
    hqo, sho = O.silu_mul_quant(bits(gu), I, group)
    assert np.array_equal(np_(hq), hqo)
    assert np.array_equal(np_(sh).reshape(sho.shape), sho)
    if group in (0, 32, 128):
        hq16, sh16, n2 = wq.silu_mul_quant_f16(gu.to(DEV), group)
        assert np.array_equal(np_(hq16).astype(np.int32), hqo.astype(np.int32))
        assert np.array_equal(np_(sh16).reshape(sho.shape), sho)


# ---------------------------------------------------------------- fp16-stored codes
@pytest.mark.parametrize("groups", [1, 56])
def test_moe_permute_f16(groups):
    T, k, E, K = 200, 8, 64, 7168
    rng = np.random.default_rng(21)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    q = rng.integers(-127, 128, (T, K), dtype=np.int8)
    s = rng.random(T).astype(np.float32) if groups == 1 else rng.random((T, groups)).astype(np.float32)
    _, _, spo, _ = O.moe_align(ids, E, 4)
    A16, sa, n2 = wq.moe_permute_f16(torch.from_numpy(q).to(DEV), torch.from_numpy(s).to(DEV),
                                     torch.from_numpy(spo).to(DEV), k)
    Ao, sao = O.moe_permute(q, s, spo, k)
    assert np.array_equal(np_(A16).astype(np.int32), Ao.astype(np.int32))
    assert np.array_equal(np_(sa), sao)
    assert np.array_equal(np_(n2), (Ao.astype(np.int64) ** 2).sum(1))


@pytest.mark.parametrize("f16", [True, False], ids=["f16", "i8"])
@pytest.mark.parametrize("T,K,k,E,group,pad", [(200, 7168, 8, 64, 0, 1), (200, 7168, 8, 64, 128, 1),
                                                (33, 256, 1, 4, 0, 1), (40, 512, 32, 64, 32, 1),
                                                (70, 2048, 4, 16, 0, 4), (5, 65536, 2, 4, 256, 1)])
def test_quantize_permute(T, K, k, E, group, pad, f16):
    """Quantization and permute in one pass (scatter form) against the
    oracle's quantization followed by its permute: every routed row's codes
    (fp16 or int8), scale(s) and, for fp16 codes, squared norm.  With padded
    alignment (pad 4) the padding rows, which no pair maps to, keep their
    previous contents."""
    rng = np.random.default_rng(T * 31 + K + k)
    x = (torch.randn(T, K, generator=torch.Generator().manual_seed(K + T)) * 2).to(torch.bfloat16)
    x[0, :3] = torch.tensor([0.0, 1e-30, -5e4])  # a zero, a tiny and a large value in one row
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    _, _, spo, p2r = O.moe_align(ids, E, pad)
    R = spo.size
    if group == 0:
        qo, so = O.quantize_per_token(bits(x))
    else:
        qo, so = O.quantize_per_token_group(bits(x), group)
    Ao, sao = O.moe_permute(qo, so, spo, k)
    sa = torch.full((R,) if group == 0 else (R, K // group), -3.0, device=DEV)
    valid = spo >= 0
    if f16:
        A = torch.full((R, K), 7.0, dtype=torch.float16, device=DEV)
        n2 = torch.full((R,), -5, dtype=torch.int32, device=DEV) if group == 0 else None
        wq.quantize_permute_f16(x.to(DEV), torch.from_numpy(p2r).to(DEV), k, R, group, out=(A, sa, n2))
        if group == 0:
            assert np.array_equal(np_(n2)[valid], (Ao[valid].astype(np.int64) ** 2).sum(1))
            assert bool((np_(n2)[~valid] == -5).all())
    else:
        A = torch.full((R, K), 7, dtype=torch.int8, device=DEV)
        wq.quantize_permute(x.to(DEV), torch.from_numpy(p2r).to(DEV), k, R, group, out=(A, sa))
    assert np.array_equal(np_(A)[valid].astype(np.int32), Ao[valid].astype(np.int32))
    assert np.array_equal(np_(sa)[valid], sao[valid])
    # padding rows untouched
    assert bool((np_(A)[~valid] == 7).all()) and bool((np_(sa)[~valid] == -3.0).all())


def test_quantize_permute_f16_skips_rows_outside():
    """Map entries outside [0, R) are skipped (no write anywhere)."""
    T, K, k, R = 4, 256, 2, 6
    x = (torch.randn(T, K, generator=torch.Generator().manual_seed(2))).to(torch.bfloat16)
    p2r = torch.tensor([0, 1, -1, 2, 6, 3, 1000, 5], dtype=torch.int32)
    A16 = torch.full((R, K), 7.0, dtype=torch.float16, device=DEV)
    sa = torch.full((R,), -3.0, device=DEV)
    n2 = torch.full((R,), -5, dtype=torch.int32, device=DEV)
    wq.quantize_permute_f16(x.to(DEV), p2r.to(DEV), k, R, 0, out=(A16, sa, n2))
    torch.cuda.synchronize()
    qo, so = O.quantize_per_token(bits(x))
    written = {0: 0, 1: 0, 2: 1, 3: 2, 5: 3}  # row -> token
    for r in range(R):
        if r in written:
            t = written[r]
            assert np.array_equal(np_(A16[r]).astype(np.int32), qo[t].astype(np.int32))
            assert float(sa[r]) == float(so[t])
        else:
            assert bool((A16[r] == 7.0).all()) and float(sa[r]) == -3.0 and int(n2[r]) == -5


@pytest.mark.parametrize("group", [0, 32, 128])
def test_silu_mul_quant_f16(group):
    R, I = 70, 2048
    g = torch.Generator().manual_seed(22)
    gu = (torch.randn(R, 2 * I, generator=g) * 4).to(torch.bfloat16)
    hq16, sh, n2 = wq.silu_mul_quant_f16(gu.to(DEV), group)
    hqo, sho = O.silu_mul_quant(bits(gu), I, group)
    assert np.array_equal(np_(hq16).astype(np.int32), hqo.astype(np.int32))
    assert np.array_equal(np_(sh).reshape(sho.shape), sho)
    if group == 0:
        assert np.array_equal(np_(n2), (hqo.astype(np.int64) ** 2).sum(1))


@pytest.mark.parametrize("K", [384, 2048])
def test_grouped_gemm_f16codes_block(K):
    """The block-wise CTA-pair engine (token tiles of up to 160 rows, per-K-
    block drains of a float32 running sum): segments around the tile size
    (0, 1, 16, 17, 159, 160, 161, 330 rows) against the oracle's block GEMM."""
    counts = [3, 0, 160, 1, 161, 330, 16, 17, 159]
    E, N = len(counts), 512
    rng = np.random.default_rng(29)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offs[-1])
    A = rng.integers(-127, 128, (R, K), dtype=np.int8)
    W = rng.integers(-127, 128, (E, N, K), dtype=np.int8)
    A[:3] = 127
    W[0, :2] = -127
    sa = (rng.random((R, K // 128)) * 0.05).astype(np.float32)
    sw = (rng.random((E, N // 128, K // 128)) * 1e-3).astype(np.float32)
    t = lambda a: torch.from_numpy(a).to(DEV)
    st = wq.new_status()
    out = torch.full((R, N), 5.0, dtype=torch.bfloat16, device=DEV)
    wq.grouped_gemm_w8a8_f16codes(t(A).to(torch.float16), None, t(sa), t(W), t(sw), t(offs),
                                  acc="f32", out=out, status=st, scheme="block")
    assert int(st.item()) == 0
    assert_bf16_equal(bits(out), O.grouped_gemm_w8a8(A, sa, W, sw, offs, "block", "f32"),
                      "f16 codes block gemm")


@pytest.mark.parametrize("K,I", [(384, 256), (2048, 384)])
def test_grouped_gemm_silu_quant_block(K, I):
    """GEMM1 with SiLU-and-mul and the per-128-group re-quantization in its
    epilogue (block scheme; the gate and up blocks of one 128-column group on
    the two CTAs of a pair, which trade halves of their token columns).  fp16
    codes and group scales bit-exact against the oracle's block GEMM followed
    by its SiLU-and-mul-quant; segments around the 160-token tile and its
    80- and 40-column splits; rows past the last segment stay untouched."""
    counts = [3, 0, 160, 1, 161, 330, 16, 17, 159, 41, 79]
    E = len(counts)
    rng = np.random.default_rng(31 + K + I)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offs[-1])
    Rt = R + 5
    A = rng.integers(-127, 128, (Rt, K), dtype=np.int8)
    W = rng.integers(-127, 128, (E, 2 * I, K), dtype=np.int8)
    A[:3] = 127
    W[2, :I] = -127  # saturated gate block: silu of large negatives
    sa = (rng.random((Rt, K // 128)) * 0.05).astype(np.float32)
    sw = (rng.random((E, 2 * I // 128, K // 128)) * 1e-3).astype(np.float32)
    t = lambda a: torch.from_numpy(a).to(DEV)
    st = wq.new_status()
    hq16 = torch.full((Rt, I), 7.0, dtype=torch.float16, device=DEV)
    sh = torch.full((Rt, I // 128), -1.0, dtype=torch.float32, device=DEV)
    wq.grouped_gemm_w8a8_silu_quant_f16codes(t(A).to(torch.float16), t(sa), t(W), t(sw), t(offs),
                                             hq16=hq16, sh=sh, status=st)
    assert int(st.item()) == 0
    gu = O.grouped_gemm_w8a8(A[:R], sa[:R], W, sw, offs, "block", "f32")
    hqo, sho = O.silu_mul_quant(gu, I, 128)
    got = np_(hq16)
    assert np.array_equal(got[:R].astype(np.int32), hqo.astype(np.int32))
    assert np.array_equal(np_(sh)[:R], sho.reshape(R, I // 128))
    assert np.all(got[R:] == 7.0) and np.all(np_(sh)[R:] == -1.0)


def test_grouped_gemm_silu_quant_channel_refused():
    """The channel scheme needs each row's maximum over all I columns, which
    no tile of the fused epilogue sees: the entry refuses it."""
    K, I, E = 256, 256, 1
    A16 = torch.zeros(4, K, dtype=torch.float16, device=DEV)
    W = torch.zeros(E, 2 * I, K, dtype=torch.int8, device=DEV)
    with pytest.raises(wq.WQError):
        wq.grouped_gemm_w8a8_silu_quant_f16codes(
            A16, torch.ones(4, device=DEV), W, torch.ones(E, 2 * I, device=DEV),
            torch.tensor([0, 4], dtype=torch.int32, device=DEV), scheme="channel")


@pytest.mark.parametrize("K,counts", [
    (512, [3, 0, 270, 1, 513]),    # K < 1024: shared-memory-weights pair engine
    (2048, [3, 0, 270, 1, 513]),   # tensor-memory weights, 320-token items with
    (4096, [3, 0, 270, 1, 513]),   #   output boxes (513 rows split at 320)
    (2048, [700, 5, 400]),         # experts average > 320 rows: 384-token items,
])                                 #   direct stores (700 rows split at 384)
@pytest.mark.parametrize("extreme", [False, True])
def test_grouped_gemm_f16codes(extreme, K, counts):
    """The CTA-pair engines (K < 1024: shared-memory weights; K >= 1024:
    weights in tensor memory, two MMAs for items above 256 tokens, 320-token
    items with shared-memory output boxes or 384-token items with direct
    stores) with codes in +-40 (the exactness check passes) and their exact
    recompute (all-127 rows: the check fails), int32 and bf16 outputs, both
    accumulator modes.  In the extreme case expert-0 rows sum to integers
    above 2^24 (one odd), so the exact recompute runs and takes each
    accumulator mode's own steps."""
    E, N = len(counts), 512
    rng = np.random.default_rng(23)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offs[-1])
    lim = 127 if extreme else 40
    A = rng.integers(-lim, lim + 1, (R, K), dtype=np.int8)
    W = rng.integers(-lim, lim + 1, (E, N, K), dtype=np.int8)
    if extreme:
        A[:5] = 127
        W[E - 1, :3] = -127
        W[0, :3] = 127
        W[0, 2, 5] = 126
    sa = (rng.random(R) * 0.05).astype(np.float32)
    sw = (rng.random((E, N)) * 1e-3).astype(np.float32)
    t = lambda a: torch.from_numpy(a).to(DEV)
    A16 = t(A).to(torch.float16)
    n2 = t((A.astype(np.int64) ** 2).sum(1).astype(np.int32))
    st = wq.new_status()
    C = wq.grouped_gemm_w8a8_f16codes(A16, n2, t(sa), t(W), t(sw), t(offs), out_type="i32", status=st)
    out = wq.grouped_gemm_w8a8_f16codes(A16, n2, t(sa), t(W), t(sw), t(offs), status=st)
    out32 = wq.grouped_gemm_w8a8_f16codes(A16, n2, t(sa), t(W), t(sw), t(offs), acc="f32", status=st)
    assert int(st.item()) == 0
    assert np.array_equal(np_(C), O.grouped_gemm_i32(A, W, offs))
    assert_bf16_equal(bits(out), O.grouped_gemm_w8a8(A, sa, W, sw, offs), "f16 codes gemm")
    assert_bf16_equal(bits(out32), O.grouped_gemm_w8a8(A, sa, W, sw, offs, "channel", "f32"),
                      "f16 codes gemm, float32 accumulator")


def _redo_flag(ws):
    """The exact-recompute flag a single-pass engine raises when a tile fails
    its exactness check: the last 256-byte piece of the grouped GEMM's
    workspace (the tile lists and their counts come first)."""
    return int(ws[-256:-252].view(torch.int32).item())


# K, engine: the single-pass engines on the exactness check's edge.  The rows
# are all +-127 and the channels all +-127 but for one 126, so
# max||a||^2 * max||w||^2 = (K*127^2) * (K*127^2) stays below 2^48 (the check
# passes and the single pass is trusted) while the sums reach odd integers in
# [2^23, 2^24): 127*127*(K-1) + 127*126.  A tensor pipe that dropped a low
# bit while adding a product to a partial sum near 2^24 would fail here.
@pytest.mark.parametrize("K,engine", [(1024, "tc5"), (768, "tc4"), (1024, "tc2")])
def test_single_pass_odd_sums_near_2_24(K, engine):
    counts = [40, 300, 3, 129]  # ragged token tiles, and a remainder of 3 rows
    E, N = len(counts), 512
    rng = np.random.default_rng(K + len(engine))
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offs[-1])
    sgn = lambda *shape: np.where(rng.random(shape) < 0.5, -1, 1)
    A = (127 * sgn(R, K)).astype(np.int8)
    A[offs[:-1]] = 127                         # each expert's first row: all +127
    W = (127 * sgn(E, N, K)).astype(np.int8)
    W[:, 0, :] = 127
    W[:, 1, :] = 127
    W[:, 1, 5] = 126                           # 127^2 (K-1) + 127*126: odd
    W[:, 2, :] = -127
    W[:, 2, K - 1] = -126
    n2a = (A.astype(np.int64) ** 2).sum(1)
    n2w = (W.astype(np.int64) ** 2).sum(2)
    assert int(n2a.max()) * int(n2w.max()) < 2 ** 48  # the engines' check passes
    sa = (rng.random(R) * 0.05).astype(np.float32)
    sw = (rng.random((E, N)) * 1e-3).astype(np.float32)
    Co = O.grouped_gemm_i32(A, W, offs)
    edge = Co[offs[:-1], 1]
    assert np.all(edge == 127 * 127 * (K - 1) + 127 * 126) and np.all(edge % 2 == 1)
    assert np.all((edge >= 2 ** 23) & (edge < 2 ** 24))
    t = lambda a: torch.from_numpy(a).to(DEV)
    st = wq.new_status()
    nws = wq.lib().wq_grouped_gemm_workspace_size(R, E)
    outs = {}
    for acc, out_type in (("i32", "i32"), ("i32", "bf16"), ("f32", "bf16")):
        ws = torch.zeros(nws, dtype=torch.uint8, device=DEV)
        if engine == "tc2":
            outs[acc, out_type] = wq.grouped_gemm_w8a8(t(A), t(sa), t(W), t(sw), t(offs), "channel", acc,
                                                       out_type, status=st, ws=ws)
        else:
            A16 = t(A).to(torch.float16)
            outs[acc, out_type] = wq.grouped_gemm_w8a8_f16codes(
                A16, t(n2a.astype(np.int32)), t(sa), t(W), t(sw), t(offs), acc=acc, out_type=out_type,
                status=st, ws=ws)
        torch.cuda.synchronize()
        assert _redo_flag(ws) == 0, "the exactness check failed: the recompute ran instead"
    assert int(st.item()) == 0
    assert np.array_equal(np_(outs["i32", "i32"]), Co)
    assert_bf16_equal(bits(outs["i32", "bf16"]), O.grouped_gemm_w8a8(A, sa, W, sw, offs),
                      f"{engine} K{K} int32 accumulator")
    assert_bf16_equal(bits(outs["f32", "bf16"]),
                      O.grouped_gemm_w8a8(A, sa, W, sw, offs, "channel", "f32"),
                      f"{engine} K{K} float32 accumulator")


def test_quantize_per_token_f16():
    """fp16-code quantization: the per-token codes, scales and squared row
    norms of the oracle (codes compared as the integers they hold)."""
    x = synth.activations(70, 7168, True, seed=41)
    x[3] = 0  # a zero row: zero codes, norm 0
    q16, s, n2 = wq.quantize_per_token_f16(x.to(DEV))
    qo, so = O.quantize_per_token(bits(x))
    assert np.array_equal(np_(q16).astype(np.int32), qo.astype(np.int32))
    assert np.array_equal(np_(s), so)
    assert np.array_equal(np_(n2), (qo.astype(np.int64) ** 2).sum(1))


# ---------------------------------------------------------------- dense linear
@pytest.mark.parametrize("T,K,N,scheme,acc", [
    (5, 256, 256, "channel", "i32"),      # few rows: the small-token engine
    (70, 384, 384, "channel", "i32"),     # N not a multiple of 256: int8 codes
    (300, 512, 512, "channel", "i32"),    # fp16 codes, shared-memory pair engine
    (300, 512, 512, "channel", "f32"),
    (300, 4096, 512, "channel", "i32"),   # fp16 codes, tensor-memory weights
    (300, 512, 512, "block", "f32"),      # fp16 codes, block-wise pair engine
    (40, 256, 384, "block", "f32"),       # int8 codes, block-wise
])
def test_linear_w8a8(T, K, N, scheme, acc):
    rng = np.random.default_rng(T + K + N)
    g = torch.Generator().manual_seed(T + N)
    x = (torch.randn(T, K, generator=g) * 2).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    Wq, sw = wq.quantize_weight(w.to(DEV), scheme)
    out = wq.linear_w8a8(x.to(DEV), Wq, sw, scheme, acc)
    torch.cuda.synchronize()
    ref = O.linear_w8a8(bits(x), np_(Wq), np_(sw), scheme, acc)
    max_abs, rel = tolerance_report(bits(out), ref)
    assert max_abs <= 2e-2 and rel <= 1e-2
    assert_bf16_equal(bits(out), ref, f"linear {scheme}/{acc} T{T} K{K} N{N}")


# ---------------------------------------------------------------- FP8 -> INT8 weights
@pytest.mark.parametrize("scheme", ["channel", "block"])
@pytest.mark.parametrize("N,K", [(128, 128), (384, 1024), (256, 7168)])
def test_convert_fp8_weights(scheme, N, K):
    w8, s8 = synth.fp8_block_weights(N, K, seed=N + K)
    w8[0, :17] = torch.arange(17, dtype=torch.uint8)       # zero and subnormal bytes
    w8[1, :8] = torch.tensor([0x7E, 0xFE, 0x38, 0xB8, 0x08, 0x88, 0x01, 0x81], dtype=torch.uint8)
    q, s = wq.convert_fp8_weights(w8.to(DEV), s8.to(DEV), scheme)
    qo, so = O.convert_fp8_weights(w8.numpy(), s8.numpy(), scheme)
    assert np.array_equal(np_(q), qo)
    assert np.array_equal(np_(s), so)



# ---------------------------------------------------------------------------
# W4A8: int4 weights (two codes a byte), int8 activations, masked layout
# ---------------------------------------------------------------------------
def test_quantize_weight_int4():
    g = torch.Generator().manual_seed(41)
    w = (torch.randn(300, 640, generator=g) * 0.02)
    w[3] = 0.0
    w[5, 7] = 0.5   # an outlier channel
    w = w.to(torch.bfloat16)
    q4, s = wq.quantize_weight_int4(w.to(DEV))
    qo, so = O.quantize_weight_int4(bits(w))
    assert np.array_equal(np_(q4), O.pack_int4(qo))
    assert np.array_equal(np_(s), so)


def _w4_problem(rng, counts, Mmax, N, K, extreme=False):
    E = len(counts)
    if extreme:
        a = np.where(rng.random((E, Mmax, K)) < 0.5, -127, 127).astype(np.int8)
        codes = np.where(rng.random((E, N, K)) < 0.5, -7, 7).astype(np.int8)
    else:
        a = rng.integers(-127, 128, (E, Mmax, K), dtype=np.int8)
        codes = rng.integers(-7, 8, (E, N, K), dtype=np.int8)
    sa = (rng.random((E, Mmax)) * 0.05).astype(np.float32)
    s4 = (rng.random((E, N)) * 1e-2).astype(np.float32)
    return a, sa, codes, O.pack_int4(codes), s4, np.array(counts, np.int32)


@pytest.mark.parametrize("K,N,counts,Mmax", [
    (512, 256, [0, 1, 17, 300, 257, 16], 300),   # 256-token tiles, short ones, an empty expert
    (2048, 384, [64, 3, 129], 160),
    (7168, 256, [5, 40], 48),                    # 64-token tiles (few rows per expert)
])
def test_grouped_gemm_w4a8_masked(K, N, counts, Mmax):
    rng = np.random.default_rng(K + N)
    a, sa, codes, W4, s4, mm = _w4_problem(rng, counts, Mmax, N, K)
    t = lambda x: torch.from_numpy(x).to(DEV)
    E = len(counts)
    for out_type in ("i32", "bf16"):
        fill = torch.full((E, Mmax, N), 7, dtype=torch.int32 if out_type == "i32" else torch.bfloat16,
                          device=DEV)
        st = wq.new_status()
        out = wq.grouped_gemm_w4a8_masked(t(a), t(sa), t(mm), t(W4), t(s4), out_type=out_type,
                                          out=fill, status=st)
        assert int(st.item()) == 0
        got = np_(out) if out_type == "i32" else O.bf16_to_f32(bits(out))
        for e in range(E):
            m = int(mm[e])
            if out_type == "i32":
                want = np.einsum("rk,nk->rn", a[e, :m].astype(np.int64), codes[e].astype(np.int64))
                assert np.array_equal(got[e, :m].astype(np.int64), want)
            assert np.all(got[e, m:].astype(np.float32) == 7)  # rows past the count untouched
        if out_type == "bf16":
            want, valid = O.grouped_gemm_w4a8_masked(a, sa, mm, W4, s4)
            assert_bf16_equal(bits(out)[valid], want[valid], "w4a8 masked gemm")


def test_grouped_gemm_w4a8_extreme_sums():
    """All codes +-7 against activations +-127 at K = 16384: sums reach
    127 * 7 * 16384 = 14.6 M, exact in the single float32 pass."""
    rng = np.random.default_rng(9)
    a, sa, codes, W4, s4, mm = _w4_problem(rng, [64, 20], 64, 128, 16384, extreme=True)
    a[0, 0] = 127
    codes[0, 0] = 7
    W4 = O.pack_int4(codes)
    t = lambda x: torch.from_numpy(x).to(DEV)
    st = wq.new_status()
    out = wq.grouped_gemm_w4a8_masked(t(a), t(sa), t(mm), t(W4), t(s4), out_type="i32", status=st)
    assert int(st.item()) == 0
    got = np_(out)
    assert got[0, 0, 0] == 127 * 7 * 16384
    for e in range(2):
        m = int(mm[e])
        want = np.einsum("rk,nk->rn", a[e, :m].astype(np.int64), codes[e].astype(np.int64))
        assert np.array_equal(got[e, :m].astype(np.int64), want)


def test_layer_forward_masked_w4a8():
    E, Mmax, H, I = 4, 80, 256, 256
    rng = np.random.default_rng(12)
    g = torch.Generator().manual_seed(12)
    w13 = (torch.randn(E, 2 * I, H, generator=g) * 0.02).to(torch.bfloat16)
    w2 = (torch.randn(E, H, I, generator=g) * 0.02).to(torch.bfloat16)
    x = torch.randn(E * Mmax, H, generator=g).to(torch.bfloat16)
    mm = np.array([80, 0, 33, 1], np.int32)
    W13 = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=DEV)
    W2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=DEV)
    S13 = torch.empty(E, 2 * I, device=DEV)
    S2 = torch.empty(E, H, device=DEV)
    for e in range(E):
        W13[e], S13[e] = wq.quantize_weight_int4(w13[e].to(DEV))
        W2[e], S2[e] = wq.quantize_weight_int4(w2[e].to(DEV))
    a, sa = wq.quantize_per_token(x.to(DEV))
    y = torch.full((E, Mmax, H), 3.0, dtype=torch.bfloat16, device=DEV)
    st = wq.new_status()
    wq.moe_forward_masked_w4a8(a.view(E, Mmax, H), sa.view(E, Mmax), torch.from_numpy(mm).to(DEV),
                               W13, S13, W2, S2, y=y, status=st)
    assert int(st.item()) == 0
    q13 = [O.quantize_weight_int4(bits(w13[e])) for e in range(E)]
    q2 = [O.quantize_weight_int4(bits(w2[e])) for e in range(E)]
    aq, as_ = O.quantize_per_token(bits(x))
    want, valid = O.moe_forward_masked_w4a8(
        aq.reshape(E, Mmax, H), as_.reshape(E, Mmax), mm,
        np.stack([O.pack_int4(q[0]) for q in q13]), np.stack([q[1] for q in q13]),
        np.stack([O.pack_int4(q[0]) for q in q2]), np.stack([q[1] for q in q2]))
    got = bits(y)
    assert_bf16_equal(got[valid], want[valid], "w4a8 masked layer")
    assert np.all(O.bf16_to_f32(got[~valid]) == 3.0)


@pytest.mark.parametrize("w4", [False, True])
@pytest.mark.parametrize("Mmax, counts", [
    (64, [64, 17, 16, 0, 1, 63]),     # 64-token plan: the engine widens its own tiles
    (65, [65, 17, 16, 0, 1, 64]),     # the smallest buffer of the fp16 token form
    (300, [300, 257, 17, 16, 0, 1]),  # two tiles (256 + 44, 256 + 1 to the small engine)
])
def test_layer_forward_masked_token_form_boundaries(w4, Mmax, counts):
    """The masked layer around the fp16 token form's limits: more than 64
    rows per expert buffer selects it; experts of 16 valid rows (or
    remainders of at most 16) go to the small-token engine, 17 to the
    tensor-core engine.  The workspace starts as 0xFF bytes, so every fp16
    token row past a valid count reads as NaN: such rows may only reach MMA
    columns that are never stored.  Outputs equal the oracle's bit for bit,
    rows past the counts stay untouched."""
    E, H, I = len(counts), 256, 256
    g = torch.Generator().manual_seed(Mmax + (7 if w4 else 0))
    w13 = (torch.randn(E, 2 * I, H, generator=g) * 0.02).to(torch.bfloat16)
    w2 = (torch.randn(E, H, I, generator=g) * 0.02).to(torch.bfloat16)
    x = synth.activations(E * Mmax, H, True, Mmax)
    mm = np.array(counts, np.int32)
    a, sa = wq.quantize_per_token(x.to(DEV))
    aq, as_ = O.quantize_per_token(bits(x))
    y = torch.full((E, Mmax, H), 3.0, dtype=torch.bfloat16, device=DEV)
    st = wq.new_status()
    if w4:
        W13 = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=DEV)
        W2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=DEV)
        S13 = torch.empty(E, 2 * I, device=DEV)
        S2 = torch.empty(E, H, device=DEV)
        for e in range(E):
            W13[e], S13[e] = wq.quantize_weight_int4(w13[e].to(DEV))
            W2[e], S2[e] = wq.quantize_weight_int4(w2[e].to(DEV))
        n = wq.lib().wq_moe_forward_masked_w4a8_workspace_size(E, Mmax, H, I)
        ws = torch.full((n,), 0xFF, dtype=torch.uint8, device=DEV)
        wq.moe_forward_masked_w4a8(a.view(E, Mmax, H), sa.view(E, Mmax),
                                   torch.from_numpy(mm).to(DEV), W13, S13, W2, S2, y=y, ws=ws,
                                   status=st)
        q13 = [O.quantize_weight_int4(bits(w13[e])) for e in range(E)]
        q2 = [O.quantize_weight_int4(bits(w2[e])) for e in range(E)]
        want, valid = O.moe_forward_masked_w4a8(
            aq.reshape(E, Mmax, H), as_.reshape(E, Mmax), mm,
            np.stack([O.pack_int4(q[0]) for q in q13]), np.stack([q[1] for q in q13]),
            np.stack([O.pack_int4(q[0]) for q in q2]), np.stack([q[1] for q in q2]))
    else:
        W13 = torch.empty(E, 2 * I, H, dtype=torch.int8, device=DEV)
        W2 = torch.empty(E, H, I, dtype=torch.int8, device=DEV)
        S13 = torch.empty(E, 2 * I, device=DEV)
        S2 = torch.empty(E, H, device=DEV)
        q = []
        for e in range(E):
            wq.quantize_weight(w13[e].to(DEV), "channel", W13[e], S13[e])
            wq.quantize_weight(w2[e].to(DEV), "channel", W2[e], S2[e])
            q.append(O.quantize_weights(bits(w13[e]), bits(w2[e]), "channel"))
        n = wq.lib().wq_moe_forward_masked_workspace_size(E, Mmax, H, I, 0)
        ws = torch.full((n,), 0xFF, dtype=torch.uint8, device=DEV)
        wq.moe_forward_masked(a.view(E, Mmax, H), sa.view(E, Mmax), torch.from_numpy(mm).to(DEV),
                              W13, S13, W2, S2, y=y, ws=ws, status=st)
        want, valid = O.moe_forward_masked(aq.reshape(E, Mmax, H), as_.reshape(E, Mmax), mm,
                                           np.stack([t[0] for t in q]), np.stack([t[1] for t in q]),
                                           np.stack([t[2] for t in q]), np.stack([t[3] for t in q]))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = bits(y)
    assert_bf16_equal(got[valid], want[valid], f"masked layer, Mmax {Mmax}, w4 {w4}")
    assert np.all(O.bf16_to_f32(got[~valid]) == 3.0)


def test_layer_forward_masked_wide_intermediate():
    """I = 2176 (more than the 2048 outputs the table SiLU pass takes): the
    masked layer re-quantizes h with the general SiLU kernel and widens h's
    rows for the fp16 token form in a separate pass.  Bit-exact."""
    cfg = synth.small_config("masked_wide", T=0, H=256, I=2176, E=3, k=1)
    Mmax = 80
    x = synth.activations(cfg.E * Mmax, cfg.H, True, 11)
    a, sa = wq.quantize_per_token(x.to(DEV))
    qo, so = O.quantize_per_token(bits(x))
    mm = np.array([80, 20, 5], np.int32)
    (W13, S13, W2, S2), orc = quantized_weights(cfg, DEV)
    y = torch.full((cfg.E, Mmax, cfg.H), 5.0, dtype=torch.bfloat16, device=DEV)
    st = wq.new_status()
    wq.moe_forward_masked(a.view(cfg.E, Mmax, cfg.H), sa.view(cfg.E, Mmax),
                          torch.from_numpy(mm).to(DEV), W13, S13, W2, S2, y=y, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref, valid = O.moe_forward_masked(qo.reshape(cfg.E, Mmax, cfg.H), so.reshape(cfg.E, Mmax), mm,
                                      *stack_oracle(orc, cfg.E))
    yb = bits(y)
    assert_bf16_equal(yb[valid], ref[valid], "masked layer, I = 2176")
    assert np.all(O.bf16_to_f32(yb[~valid]) == 5.0)


# ---------------------------------------------------------------- empty inputs
def test_empty_inputs_write_nothing():
    """Zero tokens, zero routed rows and all-zero masked counts: every entry
    returns success and leaves its outputs untouched."""
    H, I, E, k = 256, 128, 4, 2
    x0 = torch.empty(0, H, dtype=torch.bfloat16, device=DEV)
    q, s = wq.quantize_per_token(x0)
    assert q.shape == (0, H) and s.shape == (0,)
    q, s = wq.quantize_per_token_group(x0, 128)
    assert q.shape == (0, H)
    p2r0 = torch.empty(0, dtype=torch.int32, device=DEV)
    A16 = torch.full((4, H), 7.0, dtype=torch.float16, device=DEV)
    sa = torch.full((4,), -3.0, device=DEV)
    n2 = torch.full((4,), -5, dtype=torch.int32, device=DEV)
    wq.quantize_permute_f16(x0, p2r0, k, 4, 0, out=(A16, sa, n2))
    A8 = torch.full((4, H), 7, dtype=torch.int8, device=DEV)
    wq.quantize_permute(x0, p2r0, k, 4, 0, out=(A8, sa))
    gu0 = torch.empty(0, 2 * I, dtype=torch.bfloat16, device=DEV)
    hq, sh = wq.silu_mul_quant(gu0, 0)
    assert hq.shape == (0, I)
    hq16, sh16, hn = wq.silu_mul_quant_f16(gu0, 0)
    assert hq16.shape == (0, I)
    out = wq.moe_combine(torch.empty(0, H, dtype=torch.bfloat16, device=DEV), p2r0,
                         torch.empty(0, k, device=DEV), k)
    assert out.shape == (0, H)
    cfg = synth.small_config("empty", T=0, H=H, I=I, E=E, k=k)
    (W13, S13, W2, S2), _ = quantized_weights(cfg, DEV, experts=[])
    lg0 = torch.empty(0, E, dtype=torch.float32, device=DEV)
    assert wq.moe_forward(x0, lg0, W13, S13, W2, S2, k).shape == (0, H)
    # grouped GEMM with every expert empty
    offs = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    g = wq.grouped_gemm_w8a8(torch.empty(0, H, dtype=torch.int8, device=DEV),
                             torch.empty(0, device=DEV), W13, S13, offs)
    assert g.shape == (0, 2 * I)
    # masked layer with every count zero: y untouched
    Mmax = 16
    a = torch.ones(E, Mmax, H, dtype=torch.int8, device=DEV)
    sam = torch.ones(E, Mmax, device=DEV)
    y = torch.full((E, Mmax, H), 5.0, dtype=torch.bfloat16, device=DEV)
    wq.moe_forward_masked(a, sam, torch.zeros(E, dtype=torch.int32, device=DEV), W13, S13, W2, S2, y=y)
    torch.cuda.synchronize()
    assert bool((y == 5.0).all())
    assert bool((A16 == 7.0).all()) and bool((A8 == 7).all()) and bool((sa == -3.0).all())
    assert bool((n2 == -5).all())
