"""CPU oracle for the W8A8 INT8 fused Mixture-of-Experts layer.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
CPU-baseline leg may import this module.  The product path (the CUDA library
and its Python binding) never imports, calls or links it, and this module
imports nothing from the product path.

It is a plain, slow, obviously correct restatement of what the layer
computes, one function per step, in the order of the pages:

* "[Feature] DeepSeek V3/R1 INT8 Quantization (channel-wise)" (sglang pull
  request 3888), sections Modifications and Performance: the fused MoE with
  channel-wise INT8 weights and an int32 or fp32 accumulator;
* "老显卡福音！美团技术团队开源首发INT8无损满血版DeepSeek R1" (jiqizhixin,
  the Meituan INT8 DeepSeek R1 article), section 量化技术的探索 ("exploring
  the quantization techniques"): block-wise [128,128] weights with online
  per-token-group activation quantization, and channel-wise weights (one
  group per output column) with online per-token activation quantization and
  a single dequantization after the integer matmul;
* "[WIP] feat: support cutlass_moe_fp8 for deepepmoe" (sglang pull request
  8273), review comments: expert offsets are the cumulative sum of the
  per-expert counts with a leading zero; tokens are scattered by expert
  before the grouped GEMMs and gathered after them;
* "Support DeepSeek-R1 w4a8 low latency deepep" (sglang pull request 8311),
  Highlights: the masked low-latency layout with per-expert problem sizes,
  and its w4a8 weight path (int4 weights; the format is a reading, stated
  with the functions at the end of this module).

Precision.  The pages fix the data types of the method: int8 codes, float
scales, an int32 or fp32 accumulator, bf16 activations in and out.  Where a
float decides an integer (a quantized code) or feeds one (the activation
that is re-quantized), the oracle takes that decision in float32, the
precision of the kernels, with an operation order stated in each function.
The integer matmul is exact (a float64 BLAS matmul of integers whose partial
sums stay below 2**53).  Float32 arithmetic is numpy's IEEE float32
(every multiply, add and divide rounded to nearest even, never fused).

Readings where the pages are silent are listed in the function docstrings
and collected in the repository's design notes.

bf16 tensors are handled as numpy ``uint16`` bit patterns.
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32

# ---------------------------------------------------------------------------
# bf16 <-> float32
# ---------------------------------------------------------------------------


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    b = np.asarray(b).view(np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest, ties to even.

    NaN stays a (quiet) NaN; values that round past the largest finite bf16
    become infinity, as IEEE rounding to nearest requires."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


# ---------------------------------------------------------------------------
# exp and SiLU
# ---------------------------------------------------------------------------
# The activation between the two GEMMs needs exp.  Its result feeds a
# re-quantization, so both implementations must agree bit for bit; each side
# therefore implements the same published method rather than calling a
# library exp: Cody and Waite's argument reduction x = n*ln2 + r with ln2
# split into a short high part and a low part, followed by the degree-7
# Taylor polynomial of exp(r) in Horner form (|r| <= ln2/2, truncation error
# below 6e-9 relative), scaled by 2**n through two exact power-of-two
# factors.  Every operation is an individually rounded float32 operation.

LOG2E = F32(1.0 / math.log(2.0))                      # nearest float to 1/ln 2
LN2_HI = F32(math.floor(math.log(2.0) * 2**16) / 2**16)  # 16 significant bits
LN2_LO = F32(math.log(2.0) - float(LN2_HI))           # rest of ln 2
# Taylor coefficients 1/i!, i = 0..7, each rounded to the nearest float.
EXP_COEF = [F32(1.0 / math.factorial(i)) for i in range(8)]
EXP_HI = F32(89.0)     # x >= 89 overflows: +inf
EXP_LO = F32(-104.0)   # x <= -104 underflows below half the least subnormal: 0


def _pow2_f32(n: np.ndarray) -> np.ndarray:
    """Exact 2**n as float32 for integer n in [-126, 127]."""
    return ((n.astype(np.int32) + 127) << 23).astype(np.uint32).view(np.float32)


def exp_f32(x: np.ndarray) -> np.ndarray:
    """float32 exp by Cody-Waite reduction and a degree-7 Taylor polynomial.

    Steps (each a float32 operation, rounded to nearest even):
      n  = rint(x * LOG2E)
      r  = (x - n*LN2_HI) - n*LN2_LO
      p  = (((((((c7*r + c6)*r + c5)*r + c4)*r + c3)*r + c2)*r + c1)*r + c0)
      n1 = floor(n/2), n2 = n - n1
      y  = (p * 2**n1) * 2**n2
    x >= 89 gives +inf, x <= -104 gives 0, NaN propagates."""
    x = np.asarray(x, dtype=np.float32)
    out = np.empty_like(x)
    nan = np.isnan(x)
    hi = x >= EXP_HI
    lo = x <= EXP_LO
    mid = ~(nan | hi | lo)
    xm = x[mid]
    n = np.rint(xm * LOG2E)
    r = (xm - n * LN2_HI) - n * LN2_LO
    p = EXP_COEF[7]
    for c in EXP_COEF[6::-1]:
        p = p * r + c
    ni = n.astype(np.int32)
    n1 = ni >> 1
    n2 = ni - n1
    out[mid] = (p * _pow2_f32(n1)) * _pow2_f32(n2)
    out[hi] = np.inf
    out[lo] = 0.0
    out[nan] = x[nan]
    return out


def silu_f32(g: np.ndarray) -> np.ndarray:
    """silu(g) = g / (1 + exp(-g)), float32: t = exp_f32(-g); d = 1 + t; g / d."""
    g = np.asarray(g, dtype=np.float32)
    return g / (F32(1.0) + exp_f32(-g))


# ---------------------------------------------------------------------------
# Quantization (Meituan INT8 DeepSeek R1 article, 量化技术的探索)
# ---------------------------------------------------------------------------
QMAX = F32(127.0)
SCALE_EPS = F32(1e-10)


def quantize_rows(x: np.ndarray):
    """Symmetric int8 quantization, one scale per row of a float32 2-D array.

    a = max_j |x_j| (exact);  s = max(a, 1e-10) / 127  (float32 divide);
    q_j = clamp(rint(x_j / s), -127, 127)  (float32 divide, ties to even).

    Readings: the symmetric range [-127, 127] (-128 is never produced); the
    float scale is absmax/127 and codes come from dividing by it; a zero row
    gets the scale 1e-10/127 and all-zero codes."""
    x = np.asarray(x, dtype=np.float32)
    a = np.max(np.abs(x), axis=-1) if x.shape[-1] > 0 else np.zeros(x.shape[:-1], np.float32)
    s = np.maximum(a, SCALE_EPS) / QMAX
    q = np.clip(np.rint(x / s[..., None]), -127, 127).astype(np.int8)
    return q, s.astype(np.float32)


def quantize_per_token(x_bf16: np.ndarray):
    """Online per-token activation quantization (channel-wise scheme): one
    scale per token row of the bf16 activations.  Returns (q int8 [T,K],
    s float32 [T])."""
    return quantize_rows(bf16_to_f32(x_bf16))


def quantize_per_token_group(x_bf16: np.ndarray, group: int = 128):
    """Online per-token-group activation quantization (block-wise scheme):
    each token's embedding is cut into groups of ``group`` consecutive
    elements, one scale per group.  Returns (q int8 [T,K], s float32
    [T, K/group])."""
    x = bf16_to_f32(x_bf16)
    T, K = x.shape
    assert K % group == 0
    q, s = quantize_rows(x.reshape(T, K // group, group))
    return q.reshape(T, K), s


def quantize_weight_channel(w_bf16: np.ndarray):
    """Channel-wise weight quantization: one scale per output channel.
    Weights are stored [N, K] (one row per output channel), so this is the
    per-row rule.  Returns (q int8 [N,K], s float32 [N])."""
    return quantize_rows(bf16_to_f32(w_bf16))


def quantize_weight_block(w_bf16: np.ndarray, block: int = 128):
    """Block-wise weight quantization: one scale per [128, 128] block of the
    [N, K] weight.  Returns (q int8 [N,K], s float32 [N/128, K/128])."""
    w = bf16_to_f32(w_bf16)
    N, K = w.shape
    assert N % block == 0 and K % block == 0
    blocks = w.reshape(N // block, block, K // block, block).transpose(0, 2, 1, 3)
    q, s = quantize_rows(blocks.reshape(N // block, K // block, block * block))
    q = q.reshape(N // block, K // block, block, block).transpose(0, 2, 1, 3).reshape(N, K)
    return np.ascontiguousarray(q), s


# ---------------------------------------------------------------------------
# Routing
# ---------------------------------------------------------------------------


def route_topk(logits: np.ndarray, k: int):
    """Top-k routing with renormalized softmax weights.

    The pages consume ``topk_idx`` (cutlass_moe_fp8 review, ep_scatter call)
    but do not state the router; the layer's configurations ask for top-k of
    a softmax, renormalized over the chosen experts.  Readings:
      * selection by logit, descending; equal logits -> lower expert first;
      * softmax over all experts followed by renormalization over the k
        chosen ones equals the softmax over the chosen logits alone, which is
        what is computed:  m = l[id_0] (the largest logit);
        e_j = exp_f32(l[id_j] - m);  S = ((e_0 + e_1) + e_2) + ...;
        w_j = e_j / S   (float32, in j order).
    Returns (ids int32 [T,k], w float32 [T,k])."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    for t in range(T):
        row = logits[t]
        order = sorted(range(E), key=lambda i: (-float(row[i]), i))[:k]
        ids[t] = order
        m = row[order[0]]
        e = exp_f32(np.array([row[i] - m for i in order], np.float32))
        S = F32(0.0)
        for j in range(k):
            S = F32(S + e[j])
        w[t] = e / S
    return ids, w


# ---------------------------------------------------------------------------
# Align and permute (cutlass_moe_fp8 review: offsets, ep_scatter)
# ---------------------------------------------------------------------------


def moe_align(ids: np.ndarray, E: int, pad_m: int = 1):
    """Group the (token, slot) pairs by expert.

    Pair p = t*k + j routes token t to expert ids[t, j].
      counts[e]      = number of pairs routed to e;
      offsets        = [0, cumsum(ceil(counts/pad_m)*pad_m)]  (leading zero);
      sorted_pair[r] = the pair held by permuted row r, pairs of one expert in
                       ascending p (reading: stable order), -1 on padding rows;
      pair_to_row[p] = the permuted row of pair p (inverse of sorted_pair).
    """
    flat = np.asarray(ids, np.int64).reshape(-1)
    counts = np.zeros(E, np.int64)
    for e in flat:
        counts[e] += 1
    padded = (counts + pad_m - 1) // pad_m * pad_m
    offsets = np.zeros(E + 1, np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + padded[e]
    sorted_pair = np.full(int(offsets[E]), -1, np.int64)
    pair_to_row = np.empty(flat.size, np.int64)
    cursor = offsets[:E].copy()
    for p, e in enumerate(flat):
        sorted_pair[cursor[e]] = p
        pair_to_row[p] = cursor[e]
        cursor[e] += 1
    return (counts.astype(np.int32), offsets.astype(np.int32),
            sorted_pair.astype(np.int32), pair_to_row.astype(np.int32))


def moe_permute(q: np.ndarray, s: np.ndarray, sorted_pair: np.ndarray, k: int):
    """Scatter quantized tokens and their scales into expert order:
    A[r] = q[sorted_pair[r] // k], sa[r] = s[sorted_pair[r] // k]; padding
    rows (sorted_pair = -1) get zero codes and zero scales."""
    s2 = s.reshape(s.shape[0], -1)
    R = sorted_pair.size
    A = np.zeros((R, q.shape[1]), np.int8)
    sa = np.zeros((R, s2.shape[1]), np.float32)
    valid = sorted_pair >= 0
    tok = sorted_pair[valid] // k
    A[valid] = q[tok]
    sa[valid] = s2[tok]
    return A, (sa[:, 0].copy() if s.ndim == 1 else sa)


# ---------------------------------------------------------------------------
# Grouped INT8 GEMM with dequantization epilogue
# ---------------------------------------------------------------------------
KTILE = 128


def int_matmul(a: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Exact integer product a[m,K] @ w[n,K]^T as int64.  Computed with a
    float64 BLAS matmul: every product and partial sum is an integer below
    127*127*K <= 2**53, so float64 holds it exactly."""
    return (a.astype(np.float64) @ w.astype(np.float64).T).astype(np.int64)


def gemm_dequant(a: np.ndarray, sa: np.ndarray, w: np.ndarray, sw: np.ndarray,
                 scheme: str, acc: str) -> np.ndarray:
    """One expert's INT8 GEMM and dequantization, float32 result [m, n].

    channel, acc="i32" (one dequant after the int32 matmul):
        v = (float(C) * sa[r]) * sw[n]
    channel, acc="f32": C_t = int32 partial product over K tile t (128 wide),
        acc = 0; for t ascending: acc = acc + float(C_t);  v = (acc*sa[r])*sw[n]
        (reading: the pages name an fp32 accumulator but not its tile width;
        128 matches the block scheme's K blocks)
    block (weights [128,128] blocks, acts 128-groups, fp32 accumulation):
        acc = 0; for kb ascending:
            acc = acc + float(C_kb) * (sa[r,kb] * sw[n//128, kb]);   v = acc
    float(.) rounds an int to the nearest float32 (ties to even)."""
    m, K = a.shape
    n = w.shape[0]
    if scheme == "channel" and acc == "i32":
        C = int_matmul(a, w)
        return (C.astype(np.float32) * sa[:, None]) * sw[None, :]
    nt = K // KTILE
    assert K % KTILE == 0
    accum = np.zeros((m, n), np.float32)
    for t in range(nt):
        sl = slice(t * KTILE, (t + 1) * KTILE)
        Ct = int_matmul(a[:, sl], w[:, sl]).astype(np.float32)
        if scheme == "channel":
            accum = accum + Ct
        else:
            scale = sa[:, t][:, None] * np.repeat(sw[:, t], KTILE)[None, :n]
            accum = accum + Ct * scale
    if scheme == "channel":
        return (accum * sa[:, None]) * sw[None, :]
    return accum


def grouped_gemm_w8a8(A, sa, W, sw, offsets, scheme="channel", acc="i32"):
    """Grouped GEMM over experts: rows [offsets[e], offsets[e+1]) of A use
    expert e's weights.  Returns bf16 bit patterns [R, N]."""
    R = A.shape[0]
    E, N, K = W.shape
    out = np.zeros((R, N), np.float32)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            out[r0:r1] = gemm_dequant(A[r0:r1], sa[r0:r1], W[e], sw[e], scheme, acc)
    return f32_to_bf16(out)


def grouped_gemm_i32(A, W, offsets) -> np.ndarray:
    """The raw int32 accumulators of the grouped GEMM (C = A_e W_e^T)."""
    R = A.shape[0]
    E, N, K = W.shape
    out = np.zeros((R, N), np.int64)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            out[r0:r1] = int_matmul(A[r0:r1], W[e])
    return out.astype(np.int32)


# ---------------------------------------------------------------------------
# Activation with re-quantization, and combine
# ---------------------------------------------------------------------------


def silu_mul_quant(gu_bf16: np.ndarray, I: int, group: int = 0):
    """SiLU-and-mul of the gate_up output, then re-quantization.

    g = GU[:, :I], u = GU[:, I:2I] (reading: gate half first), both widened
    exactly from bf16 (reading: the GEMM1 output is rounded to bf16 first);
    h = silu_f32(g) * u  (float32);  h is quantized per row (group = 0,
    channel scheme) or per 128-group (block scheme) with the rule of
    ``quantize_rows``.  Returns (hq int8 [R, I], sh float32 [R] or [R, I/group])."""
    gu = bf16_to_f32(gu_bf16)
    g, u = gu[:, :I], gu[:, I:2 * I]
    h = silu_f32(g) * u
    if group == 0:
        return quantize_rows(h)
    R = h.shape[0]
    q, s = quantize_rows(h.reshape(R, I // group, group))
    return q.reshape(R, I), s


def moe_combine(y_bf16: np.ndarray, pair_to_row: np.ndarray, w: np.ndarray, k: int):
    """Top-k weighted combine: out[t] = bf16(sum_j w[t,j] * y[pair_to_row[t*k+j]]),
    float32, acc = 0; for j ascending: acc = acc + (w * y);  round once."""
    y = bf16_to_f32(y_bf16)
    T = w.shape[0]
    acc = np.zeros((T, y.shape[1]), np.float32)
    rows = pair_to_row.reshape(T, k)
    for j in range(k):
        acc = acc + w[:, j][:, None] * y[rows[:, j]]
    return f32_to_bf16(acc)


# ---------------------------------------------------------------------------
# The whole layer
# ---------------------------------------------------------------------------


def quantize_weights(w13_bf16, w2_bf16, scheme: str):
    """Offline weight quantization of one expert (channel or [128,128] block)."""
    f = quantize_weight_channel if scheme == "channel" else quantize_weight_block
    q13, s13 = f(w13_bf16)
    q2, s2 = f(w2_bf16)
    return q13, s13, q2, s2


def moe_forward(x_bf16, logits, W13, S13, W2, S2, k: int, scheme="channel", acc="i32",
                return_all=False):
    """Fused MoE: route -> quantize -> align -> permute -> GEMM1 (gate_up) ->
    SiLU-mul + re-quantize -> GEMM2 (down) -> weighted combine.  Weights are
    already quantized ([E,2I,H] int8 + scales, [E,H,I] int8 + scales)."""
    E, N1, H = W13.shape
    I = N1 // 2
    ids, w = route_topk(logits, k)
    if scheme == "channel":
        q, s = quantize_per_token(x_bf16)
    else:
        q, s = quantize_per_token_group(x_bf16, 128)
    counts, offsets, sorted_pair, pair_to_row = moe_align(ids, E)
    A, sa = moe_permute(q, s, sorted_pair, k)
    gu = grouped_gemm_w8a8(A, sa, W13, S13, offsets, scheme, acc)
    hq, sh = silu_mul_quant(gu, I, 0 if scheme == "channel" else 128)
    y = grouped_gemm_w8a8(hq, sh, W2, S2, offsets, scheme, acc)
    out = moe_combine(y, pair_to_row, w, k)
    if return_all:
        return dict(ids=ids, w=w, q=q, s=s, counts=counts, offsets=offsets,
                    sorted_pair=sorted_pair, pair_to_row=pair_to_row, A=A, sa=sa,
                    gu=gu, hq=hq, sh=sh, y=y, out=out)
    return out


def moe_forward_masked(a_q, a_s, masked_m, W13, S13, W2, S2, scheme="channel", acc="i32"):
    """Masked (expert-parallel low-latency) layout: a_q int8 [E, Mmax, H] with
    per-token scales a_s [E, Mmax] and per-expert valid counts masked_m[E].
    For each expert only rows < masked_m[e] are computed: GEMM1 -> SiLU-mul +
    re-quantize -> GEMM2.  Returns (y bf16 [E, Mmax, H], valid mask [E, Mmax]);
    rows at or past masked_m[e] are not defined by the layer."""
    E, Mmax, H = a_q.shape
    I = W13.shape[1] // 2
    y = np.zeros((E, Mmax, H), np.uint16)
    valid = np.zeros((E, Mmax), bool)
    for e in range(E):
        m = int(masked_m[e])
        if m <= 0:
            continue
        valid[e, :m] = True
        gu = f32_to_bf16(gemm_dequant(a_q[e, :m], a_s[e, :m], W13[e], S13[e], scheme, acc))
        hq, sh = silu_mul_quant(gu, I, 0 if scheme == "channel" else 128)
        y[e, :m] = f32_to_bf16(gemm_dequant(hq, sh, W2[e], S2[e], scheme, acc))
    return y, valid


def linear_w8a8(x_bits: np.ndarray, w: np.ndarray, sw: np.ndarray, scheme: str = "channel",
                acc: str = "i32") -> np.ndarray:
    """Dense W8A8 INT8 linear ("Norm Linear" in [Feature] DeepSeek V3/R1 INT8
    Quantization (channel-wise), Modifications: the non-MoE linears run as a
    w8a8 INT8 GEMM).  The activation quantization of the scheme (per token,
    or per token per 128-group), then the INT8 GEMM with its dequantization
    (gemm_dequant), rounded to bf16.  x_bits bf16 bits [T, K]; w int8 [N, K];
    sw [N] or [N/128, K/128].  Returns bf16 bits [T, N]."""
    if scheme == "channel":
        q, s = quantize_per_token(x_bits)
    else:
        q, s = quantize_per_token_group(x_bits, KTILE)
    return f32_to_bf16(gemm_dequant(q, s, w, sw, scheme, acc))


# ---------------------------------------------------------------------------
# FP8 (e4m3) block-scaled weights -> BF16 -> INT8 (offline conversion)
# ---------------------------------------------------------------------------
def e4m3_to_f32(b: np.ndarray) -> np.ndarray:
    """The value of FP8 e4m3 bytes (1 sign, 4 exponent bits with bias 7, 3
    mantissa bits; no infinities, S.1111.111 is NaN): exponent field 0 gives
    (m / 8) * 2^-6, otherwise (1 + m / 8) * 2^(e - 7).  Every value is exact
    in float32."""
    b = b.astype(np.uint8)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = ((b >> 3) & 0xF).astype(np.int64)
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return (sign * mag).astype(np.float32)


def dequant_fp8_block(w8: np.ndarray, s8: np.ndarray, block: int = 128) -> np.ndarray:
    """FP8 weights [N, K] with one float32 scale per [128, 128] block
    ([N/128, K/128]) to BF16, the first step of the conversion in the Meituan
    INT8 article (量化技术的探索: the released FP8 weights are dequantized to
    BF16 before INT8 quantization).  Reading: the product value * scale is
    one float32 multiplication rounded to nearest, then rounded to bf16.
    Returns bf16 bits [N, K]."""
    N, K = w8.shape
    sc = np.repeat(np.repeat(s8.astype(np.float32), block, axis=0), block, axis=1)[:N, :K]
    return f32_to_bf16((e4m3_to_f32(w8) * sc).astype(np.float32))


def convert_fp8_weights(w8: np.ndarray, s8: np.ndarray, scheme: str):
    """FP8 -> BF16 -> INT8: dequantize (dequant_fp8_block), then the INT8
    weight quantization of the scheme (per output channel, or per [128,128]
    block).  Returns (int8 codes [N, K], scales)."""
    bf = dequant_fp8_block(w8, s8)
    return quantize_weight_channel(bf) if scheme == "channel" else quantize_weight_block(bf)


# ---------------------------------------------------------------------------
# W4A8: int4 weights with int8 activations on the masked layout
# ("Support DeepSeek-R1 w4a8 low latency deepep" (sglang pull request 8311),
# Highlights and the forward_cutlass_w4a8_masked hunk: a w4a8 weight path for
# the masked low-latency layout with per-expert problem sizes)
# ---------------------------------------------------------------------------
# Readings.  The page names the path but states no format: neither the int4
# code range, group or scale layout, nor the activation type, nor how two
# codes share a byte.  This oracle takes the plainest reading that the rest
# of the method supports: the channel-wise rule of the INT8 weights with 7 in
# place of 127 (symmetric codes in [-7, 7], one float32 scale per output
# channel), activations quantized per token to int8 exactly as in the W8A8
# layer, and two codes per byte with code 2j in the low nibble and code 2j+1
# in the high nibble (two's complement nibbles).
Q4MAX = F32(7.0)


def quantize_weight_int4(w_bf16: np.ndarray):
    """Channel-wise symmetric int4 weight quantization, one scale per output
    channel (row of the [N, K] storage):
        a = max_k |w_k|;  s = max(a, 1e-10) / 7  (float32 divide);
        q_k = clamp(rint(w_k / s), -7, 7)  (float32 divide, ties to even).
    Returns (q int8 [N, K] with values in [-7, 7], s float32 [N])."""
    w = bf16_to_f32(w_bf16)
    a = np.max(np.abs(w), axis=-1) if w.shape[-1] > 0 else np.zeros(w.shape[:-1], np.float32)
    s = (np.maximum(a, SCALE_EPS) / Q4MAX).astype(np.float32)
    q = np.clip(np.rint(w / s[..., None]), -7, 7).astype(np.int8)
    return q, s


def pack_int4(q: np.ndarray) -> np.ndarray:
    """int4 codes [..., K] (K even, values in [-8, 7]) -> bytes [..., K/2]:
    code 2j in bits 0-3 and code 2j+1 in bits 4-7 of byte j."""
    q = np.asarray(q)
    assert q.shape[-1] % 2 == 0
    u = (q.astype(np.int16) & 0xF).astype(np.uint8)
    return (u[..., 0::2] | (u[..., 1::2] << 4)).astype(np.uint8)


def unpack_int4(b: np.ndarray) -> np.ndarray:
    """Bytes [..., K/2] -> int4 codes [..., K] as int8 (the inverse of
    pack_int4; a nibble n >= 8 is the code n - 16)."""
    b = np.asarray(b, dtype=np.uint8)
    lo = (b & 0xF).astype(np.int16)
    hi = (b >> 4).astype(np.int16)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), np.int8)
    out[..., 0::2] = np.where(lo >= 8, lo - 16, lo)
    out[..., 1::2] = np.where(hi >= 8, hi - 16, hi)
    return out


def grouped_gemm_w4a8_masked(a_q, a_s, masked_m, W4, S4):
    """The masked grouped GEMM with int4 weights: for expert e and rows
    r < masked_m[e],  C = sum_k a[e,r,k] * w[e,n,k]  (exact integers, |C| <=
    127 * 7 * K), then  v = (float(C) * sa[e,r]) * s4[e,n]  (the channel
    int32 epilogue), rounded to bf16.  a_q int8 [E, Mmax, K], a_s [E, Mmax],
    W4 packed uint8 [E, N, K/2], S4 [E, N].  Returns (out bf16 [E, Mmax, N],
    valid [E, Mmax]); rows at or past masked_m[e] are not defined."""
    E, Mmax, K = a_q.shape
    N = W4.shape[1]
    out = np.zeros((E, Mmax, N), np.uint16)
    valid = np.zeros((E, Mmax), bool)
    for e in range(E):
        m = min(int(masked_m[e]), Mmax)
        if m <= 0:
            continue
        valid[e, :m] = True
        out[e, :m] = f32_to_bf16(gemm_dequant(a_q[e, :m], a_s[e, :m], unpack_int4(W4[e]), S4[e],
                                              "channel", "i32"))
    return out, valid


def moe_forward_masked_w4a8(a_q, a_s, masked_m, W13_4, S13_4, W2_4, S2_4):
    """The masked layer with int4 weights: GEMM1 (gate_up) -> SiLU-mul +
    per-token int8 re-quantization -> GEMM2 (down), on the valid rows.  It is
    the W8A8 masked layer (channel scheme, int32 accumulator) applied to the
    unpacked int4 codes and their scales.  Returns (y bf16 [E, Mmax, H],
    valid [E, Mmax])."""
    return moe_forward_masked(a_q, a_s, masked_m, unpack_int4(W13_4), S13_4, unpack_int4(W2_4),
                              S2_4, "channel", "i32")
