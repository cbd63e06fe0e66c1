"""ctypes binding of libwq.so (include/wq.h): argument marshalling only.

Each function takes CUDA torch tensors, allocates the outputs with torch
(device memory is the only thing PyTorch provides here), passes raw device
pointers and the current stream to the C ABI, and raises ``WQError`` on a
non-zero return code.  Every step of the layer runs in the library's CUDA
kernels; there is no fallback: if the library is missing, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwq.so")

SCHEME = {"channel": 0, "block": 1}
ACC = {"i32": 0, "f32": 1}
OUT = {"bf16": 0, "i32": 1}


class WQError(RuntimeError):
    pass


_lib = None
_c = ctypes
_P = _c.c_void_p
_I = _c.c_int
_L = _c.c_int64
_S = _c.c_size_t

_SIGS = {
    "wq_init": (_I, [_I]),
    "wq_status_string": (_c.c_char_p, [_I]),
    "wq_kernel_launches": (_c.c_uint64, []),
    "wq_quantize_per_token": (_I, [_P, _L, _L, _L, _P, _P, _P]),
    "wq_quantize_per_token_group": (_I, [_P, _L, _L, _L, _I, _P, _P, _P]),
    "wq_quantize_weight_block": (_I, [_P, _L, _L, _P, _P, _P]),
    "wq_convert_fp8_weights": (_I, [_P, _P, _L, _L, _I, _P, _P, _P]),
    "wq_route_topk": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "wq_moe_align_workspace_size": (_S, [_I, _I, _I]),
    "wq_moe_align": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _S, _P, _P]),
    "wq_moe_permute": (_I, [_P, _P, _I, _I, _I, _L, _P, _L, _P, _P, _P]),
    "wq_grouped_gemm_workspace_size": (_S, [_L, _I]),
    "wq_grouped_gemm_w8a8": (_I, [_P, _P, _P, _P, _P, _I, _L, _L, _L, _I, _I, _I, _P, _P, _S, _P, _P]),
    "wq_grouped_gemm_w8a8_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _L, _L, _L, _I, _I, _I, _P, _P, _P]),
    "wq_moe_permute_f16": (_I, [_P, _P, _I, _I, _I, _L, _P, _L, _P, _P, _P, _P]),
    "wq_silu_mul_quant_f16": (_I, [_P, _L, _L, _I, _P, _P, _P, _P]),
    "wq_grouped_gemm_w8a8_f16codes": (_I, [_P, _P, _P, _P, _P, _P, _I, _L, _L, _L, _I, _I, _I, _P, _P, _S, _P, _P]),
    "wq_quantize_per_token_f16": (_I, [_P, _L, _L, _L, _P, _P, _P, _P]),
    "wq_quantize_permute_f16": (_I, [_P, _L, _L, _I, _P, _I, _L, _P, _P, _P, _P]),
    "wq_quantize_permute": (_I, [_P, _L, _L, _I, _P, _I, _L, _P, _P, _P]),
    "wq_grouped_gemm_silu_quant_workspace_size": (_S, [_L, _I]),
    "wq_quantize_weight_int4": (_I, [_P, _L, _L, _P, _P, _P]),
    "wq_grouped_gemm_w4a8_masked": (_I, [_P, _P, _P, _I, _I, _P, _P, _L, _L, _I, _P, _P, _S, _P, _P]),
    "wq_moe_forward_masked_w4a8_workspace_size": (_S, [_I, _I, _I, _I]),
    "wq_moe_forward_masked_w4a8": (_I, [_P, _P, _P, _I, _I, _P, _P, _P, _P, _I, _I, _P, _P, _S, _P, _P]),
    "wq_selftest_wait_timeout": (_I, [_P, _P, _P, _P, _P, _I, _L, _L, _L, _P, _P, _S, _P, _P]),
    "wq_grouped_gemm_w8a8_silu_quant_f16codes": (_I, [_P, _P, _P, _P, _P, _I, _L, _L, _L, _I, _P, _P, _P, _S, _P, _P]),
    "wq_grouped_gemm_masked_workspace_size": (_S, [_I, _I]),
    "wq_grouped_gemm_w8a8_masked": (_I, [_P, _P, _P, _I, _I, _P, _P, _L, _L, _I, _I, _I, _P, _P, _S, _P, _P]),
    "wq_silu_mul_quant": (_I, [_P, _L, _L, _I, _P, _P, _P]),
    "wq_moe_combine": (_I, [_P, _P, _P, _I, _I, _L, _P, _P]),
    "wq_moe_forward_workspace_size": (_S, [_I, _I, _I, _I, _I, _I]),
    "wq_moe_forward": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _S, _P, _P]),
    "wq_moe_forward_host_workspace_size": (_S, [_I, _I, _I, _I, _I, _I]),
    "wq_moe_forward_host": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _S, _P, _P]),
    "wq_moe_forward_masked_workspace_size": (_S, [_I, _I, _I, _I, _I]),
    "wq_linear_w8a8_workspace_size": (_S, [_L, _L, _L, _I]),
    "wq_linear_w8a8": (_I, [_P, _L, _L, _L, _P, _P, _L, _I, _I, _P, _P, _S, _P, _P]),
    "wq_moe_forward_masked": (_I, [_P, _P, _P, _I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _S, _P, _P]),
}


def exported_names():
    return list(_SIGS)


def lib():
    """Load libwq.so (once).  Raises if it has not been built, or if this
    process is one rank of a multi-process launch (WORLD_SIZE > 1): the
    library's pair GEMM engines share token tiles between the two CTAs of a
    cluster through TMA multicast, which it supports in one-GPU runs only."""
    global _lib
    if _lib is None:
        if int(os.environ.get("WORLD_SIZE", "1")) > 1:
            raise WQError("libwq.so serves one-GPU runs only; WORLD_SIZE > 1 is refused")
        if not os.path.exists(LIB_PATH):
            raise WQError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _lib = h
    return _lib


def _check(rc: int, what: str):
    if rc != 0:
        raise WQError(f"{what}: {lib().wq_status_string(rc).decode()} ({rc})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dev(t, dtype, name):
    if not t.is_cuda:
        raise WQError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise WQError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise WQError(f"{name} must be contiguous")
    return t


def new_status(device=None):
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def init(device: int = 0):
    _check(lib().wq_init(device), "wq_init")


# ---------------------------------------------------------------- quantization
def quantize_per_token(x):
    _dev(x, torch.bfloat16, "x")
    T, K = x.shape
    q = torch.empty(T, K, dtype=torch.int8, device=x.device)
    s = torch.empty(T, dtype=torch.float32, device=x.device)
    _check(lib().wq_quantize_per_token(_ptr(x), T, K, K, _ptr(q), _ptr(s), _stream()),
           "wq_quantize_per_token")
    return q, s


def quantize_per_token_group(x, group=128):
    _dev(x, torch.bfloat16, "x")
    T, K = x.shape
    q = torch.empty(T, K, dtype=torch.int8, device=x.device)
    s = torch.empty(T, max(K // group, 1), dtype=torch.float32, device=x.device)
    _check(lib().wq_quantize_per_token_group(_ptr(x), T, K, K, group, _ptr(q), _ptr(s), _stream()),
           "wq_quantize_per_token_group")
    return q, s


def quantize_weight_block(w):
    _dev(w, torch.bfloat16, "w")
    N, K = w.shape
    q = torch.empty(N, K, dtype=torch.int8, device=w.device)
    s = torch.empty(N // 128, K // 128, dtype=torch.float32, device=w.device)
    _check(lib().wq_quantize_weight_block(_ptr(w), N, K, _ptr(q), _ptr(s), _stream()),
           "wq_quantize_weight_block")
    return q, s


def convert_fp8_weights(w8, s8, scheme: str, q_out=None, s_out=None):
    """FP8 e4m3 weights (uint8 [N, K] bytes) with [N/128, K/128] block
    scales -> bf16 -> int8 codes and scales of the scheme."""
    _dev(w8, torch.uint8, "w8")
    _dev(s8, torch.float32, "s8")
    N, K = w8.shape
    q = q_out if q_out is not None else torch.empty(N, K, dtype=torch.int8, device=w8.device)
    if s_out is not None:
        s = s_out
    else:
        shape = (N,) if scheme == "channel" else (N // 128, K // 128)
        s = torch.empty(shape, dtype=torch.float32, device=w8.device)
    _check(lib().wq_convert_fp8_weights(_ptr(w8), _ptr(s8), N, K, SCHEME[scheme], _ptr(q), _ptr(s),
                                        _stream()), "wq_convert_fp8_weights")
    return q, s


def quantize_weight(w, scheme: str, q_out=None, s_out=None):
    """Offline weight quantization of one [N, K] bf16 matrix (channel or block),
    optionally into preallocated outputs."""
    N, K = w.shape
    if scheme == "channel":
        _dev(w, torch.bfloat16, "w")
        q = q_out if q_out is not None else torch.empty(N, K, dtype=torch.int8, device=w.device)
        s = s_out if s_out is not None else torch.empty(N, dtype=torch.float32, device=w.device)
        _check(lib().wq_quantize_per_token(_ptr(w), N, K, K, _ptr(q), _ptr(s), _stream()),
               "wq_quantize_per_token")
        return q, s
    _dev(w, torch.bfloat16, "w")
    q = q_out if q_out is not None else torch.empty(N, K, dtype=torch.int8, device=w.device)
    s = s_out if s_out is not None else torch.empty(N // 128, K // 128, dtype=torch.float32, device=w.device)
    _check(lib().wq_quantize_weight_block(_ptr(w), N, K, _ptr(q), _ptr(s), _stream()),
           "wq_quantize_weight_block")
    return q, s


# ---------------------------------------------------------------- routing / align / permute
def route_topk(logits, k):
    _dev(logits, torch.float32, "logits")
    T, E = logits.shape
    ids = torch.empty(T, k, dtype=torch.int32, device=logits.device)
    w = torch.empty(T, k, dtype=torch.float32, device=logits.device)
    _check(lib().wq_route_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _stream()), "wq_route_topk")
    return ids, w


def moe_align(ids, E, pad_m=1, status=None):
    _dev(ids, torch.int32, "ids")
    T, k = ids.shape
    dev = ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_pair = torch.empty(T * k + E * (pad_m - 1), dtype=torch.int32, device=dev)
    pair_to_row = torch.empty(T * k, dtype=torch.int32, device=dev)
    nws = lib().wq_moe_align_workspace_size(T, k, E)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=dev)
    st = status if status is not None else new_status(dev)
    _check(lib().wq_moe_align(_ptr(ids), T, k, E, pad_m, _ptr(counts), _ptr(offsets),
                              _ptr(sorted_pair), _ptr(pair_to_row), _ptr(ws), nws, _ptr(st),
                              _stream()), "wq_moe_align")
    return counts, offsets, sorted_pair, pair_to_row


def moe_permute(q, s, sorted_pair, k):
    _dev(q, torch.int8, "q")
    _dev(s, torch.float32, "s")
    _dev(sorted_pair, torch.int32, "sorted_pair")
    T, K = q.shape
    groups = 1 if s.dim() == 1 else s.shape[1]
    R = sorted_pair.numel()
    A = torch.empty(R, K, dtype=torch.int8, device=q.device)
    sa = torch.empty((R,) if s.dim() == 1 else (R, groups), dtype=torch.float32, device=q.device)
    _check(lib().wq_moe_permute(_ptr(q), _ptr(s), groups, T, k, K, _ptr(sorted_pair), R, _ptr(A),
                                _ptr(sa), _stream()), "wq_moe_permute")
    return A, sa


def moe_permute_f16(q, s, sorted_pair, k):
    """Permute into fp16-stored codes; returns (A16 as torch.float16, sa, norm2)."""
    _dev(q, torch.int8, "q")
    _dev(s, torch.float32, "s")
    _dev(sorted_pair, torch.int32, "sorted_pair")
    T, K = q.shape
    groups = 1 if s.dim() == 1 else s.shape[1]
    R = sorted_pair.numel()
    A16 = torch.empty(R, K, dtype=torch.float16, device=q.device)
    sa = torch.empty((R,) if s.dim() == 1 else (R, groups), dtype=torch.float32, device=q.device)
    n2 = torch.empty(R, dtype=torch.int32, device=q.device)
    _check(lib().wq_moe_permute_f16(_ptr(q), _ptr(s), groups, T, k, K, _ptr(sorted_pair), R,
                                    _ptr(A16), _ptr(sa), _ptr(n2), _stream()), "wq_moe_permute_f16")
    return A16, sa, n2


def silu_mul_quant_f16(gu, group=0):
    """SiLU-mul + re-quantization into fp16-stored codes: (hq16, sh, norm2);
    with a group, sh is [R, I/group] and norm2 is None."""
    _dev(gu, torch.bfloat16, "gu")
    R, I2 = gu.shape
    I = I2 // 2
    hq = torch.empty(R, I, dtype=torch.float16, device=gu.device)
    sh = torch.empty(R, I // group if group else 1, dtype=torch.float32, device=gu.device)
    n2 = torch.empty(R, dtype=torch.int32, device=gu.device) if group == 0 else None
    _check(lib().wq_silu_mul_quant_f16(_ptr(gu), R, I, group, _ptr(hq), _ptr(sh),
                                       _ptr(n2) if n2 is not None else None, _stream()),
           "wq_silu_mul_quant_f16")
    return hq, (sh.view(R) if group == 0 else sh), n2


def grouped_gemm_w8a8_f16codes(A16, a_norm2, sa, W, sw, offsets, acc="i32", out_type="bf16",
                               out=None, status=None, scheme="channel", ws=None):
    _dev(A16, torch.float16, "A16")
    if a_norm2 is not None:
        _dev(a_norm2, torch.int32, "a_norm2")
    _dev(sa, torch.float32, "sa")
    _dev(W, torch.int8, "W")
    _dev(sw, torch.float32, "sw")
    _dev(offsets, torch.int32, "offsets")
    R, K = A16.shape
    E, N, _ = W.shape
    if out is None:
        out = torch.empty(R, N, dtype=torch.bfloat16 if out_type == "bf16" else torch.int32,
                          device=A16.device)
    nws = lib().wq_grouped_gemm_workspace_size(R, E)
    if ws is None:
        ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=A16.device)
    st = status if status is not None else new_status(A16.device)
    _check(lib().wq_grouped_gemm_w8a8_f16codes(_ptr(A16), _ptr(a_norm2) if a_norm2 is not None else None,
                                               _ptr(sa), _ptr(W), _ptr(sw),
                                               _ptr(offsets), E, R, N, K, SCHEME[scheme], ACC[acc],
                                               OUT[out_type],
                                               _ptr(out),
                                               _ptr(ws), nws, _ptr(st), _stream()),
           "wq_grouped_gemm_w8a8_f16codes")
    return out


def grouped_gemm_w8a8_silu_quant_f16codes(A16, sa, W13, sw13, offsets, hq16=None, sh=None,
                                           status=None, scheme="block", ws=None):
    """Fused gate_up GEMM -> SiLU-and-mul -> per-128-group re-quantization
    (block scheme): (hq16 fp16 codes [R, I], sh [R, I/128])."""
    _dev(A16, torch.float16, "A16")
    _dev(sa, torch.float32, "sa")
    _dev(W13, torch.int8, "W13")
    _dev(sw13, torch.float32, "sw13")
    _dev(offsets, torch.int32, "offsets")
    R, K = A16.shape
    E, N2, _ = W13.shape
    I = N2 // 2
    if hq16 is None:
        hq16 = torch.empty(R, I, dtype=torch.float16, device=A16.device)
    if sh is None:
        sh = torch.empty(R, max(I // 128, 1), dtype=torch.float32, device=A16.device)
    nws = lib().wq_grouped_gemm_silu_quant_workspace_size(R, E)
    if ws is None:
        ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=A16.device)
    st = status if status is not None else new_status(A16.device)
    _check(lib().wq_grouped_gemm_w8a8_silu_quant_f16codes(
        _ptr(A16), _ptr(sa), _ptr(W13), _ptr(sw13), _ptr(offsets), E, R, I, K, SCHEME[scheme],
        _ptr(hq16), _ptr(sh), _ptr(ws), nws, _ptr(st), _stream()),
        "wq_grouped_gemm_w8a8_silu_quant_f16codes")
    return hq16, sh


def selftest_wait_timeout(A16, sa, W, sw, offsets, out, status):
    """Launch the block engine with a wait that nothing completes (failure-path
    test); the device writes WQ_ERR_TIMEOUT into `status` after 1 s."""
    R, K = A16.shape
    E, N, _ = W.shape
    nws = lib().wq_grouped_gemm_workspace_size(R, E)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=A16.device)
    _check(lib().wq_selftest_wait_timeout(_ptr(A16), _ptr(sa), _ptr(W), _ptr(sw), _ptr(offsets), E,
                                          R, N, K, _ptr(out), _ptr(ws), nws, _ptr(status),
                                          _stream()),
           "wq_selftest_wait_timeout")


def quantize_per_token_f16(x):
    """Per-token quantization into fp16 codes: (q16 fp16 [T, K], s [T], norm2 [T])."""
    _dev(x, torch.bfloat16, "x")
    T, K = x.shape
    q16 = torch.empty(T, K, dtype=torch.float16, device=x.device)
    s = torch.empty(T, dtype=torch.float32, device=x.device)
    n2 = torch.empty(T, dtype=torch.int32, device=x.device)
    _check(lib().wq_quantize_per_token_f16(_ptr(x), T, K, K, _ptr(q16), _ptr(s), _ptr(n2), _stream()),
           "wq_quantize_per_token_f16")
    return q16, s, n2


def quantize_permute_f16(x, pair_to_row, k, R, group=0, out=None):
    """Quantization and permute in one pass: (A16 fp16 [R, K], sa [R] or
    [R, K/group], norm2 [R] or None).  Rows no pair maps to keep the contents
    of `out` (a tuple of the three tensors) or are left uninitialised."""
    _dev(x, torch.bfloat16, "x")
    _dev(pair_to_row, torch.int32, "pair_to_row")
    T, K = x.shape
    if out is None:
        A16 = torch.empty(R, K, dtype=torch.float16, device=x.device)
        sa = torch.empty((R,) if group == 0 else (R, K // group), dtype=torch.float32, device=x.device)
        n2 = torch.empty(R, dtype=torch.int32, device=x.device) if group == 0 else None
    else:
        A16, sa, n2 = out
    _check(lib().wq_quantize_permute_f16(_ptr(x), T, K, group, _ptr(pair_to_row), k, R, _ptr(A16),
                                         _ptr(sa), _ptr(n2) if n2 is not None else None, _stream()),
           "wq_quantize_permute_f16")
    return A16, sa, n2


def quantize_permute(x, pair_to_row, k, R, group=0, out=None):
    """Quantization and permute in one pass, int8 codes: (A int8 [R, K], sa
    [R] or [R, K/group]).  Rows no pair maps to keep the contents of `out`
    (a tuple of the two tensors) or are left uninitialised."""
    _dev(x, torch.bfloat16, "x")
    _dev(pair_to_row, torch.int32, "pair_to_row")
    T, K = x.shape
    if out is None:
        A = torch.empty(R, K, dtype=torch.int8, device=x.device)
        sa = torch.empty((R,) if group == 0 else (R, K // group), dtype=torch.float32, device=x.device)
    else:
        A, sa = out
    _check(lib().wq_quantize_permute(_ptr(x), T, K, group, _ptr(pair_to_row), k, R, _ptr(A), _ptr(sa),
                                     _stream()), "wq_quantize_permute")
    return A, sa


# ---------------------------------------------------------------- GEMMs
def grouped_gemm_w8a8(A, sa, W, sw, offsets, scheme="channel", acc="i32", out_type="bf16",
                      out=None, status=None, ws=None):
    _dev(A, torch.int8, "A")
    _dev(sa, torch.float32, "sa")
    _dev(W, torch.int8, "W")
    _dev(sw, torch.float32, "sw")
    _dev(offsets, torch.int32, "offsets")
    R, K = A.shape
    E, N, K2 = W.shape
    if K2 != K:
        raise WQError("A and W disagree on K")
    if out is None:
        out = torch.empty(R, N, dtype=torch.bfloat16 if out_type == "bf16" else torch.int32,
                          device=A.device)
    nws = lib().wq_grouped_gemm_workspace_size(R, E)
    if ws is None:
        ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=A.device)
    st = status if status is not None else new_status(A.device)
    _check(lib().wq_grouped_gemm_w8a8(_ptr(A), _ptr(sa), _ptr(W), _ptr(sw), _ptr(offsets), E, R, N,
                                      K, SCHEME[scheme], ACC[acc], OUT[out_type], _ptr(out),
                                      _ptr(ws), nws, _ptr(st), _stream()), "wq_grouped_gemm_w8a8")
    return out


def grouped_gemm_w8a8_masked(A, sa, masked_m, W, sw, scheme="channel", acc="i32",
                             out_type="bf16", out=None, status=None):
    _dev(A, torch.int8, "A")
    _dev(sa, torch.float32, "sa")
    _dev(masked_m, torch.int32, "masked_m")
    _dev(W, torch.int8, "W")
    _dev(sw, torch.float32, "sw")
    E, Mmax, K = A.shape
    _, N, _ = W.shape
    if out is None:
        out = torch.empty(E, Mmax, N, dtype=torch.bfloat16 if out_type == "bf16" else torch.int32,
                          device=A.device)
    nws = lib().wq_grouped_gemm_masked_workspace_size(E, Mmax)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=A.device)
    st = status if status is not None else new_status(A.device)
    _check(lib().wq_grouped_gemm_w8a8_masked(_ptr(A), _ptr(sa), _ptr(masked_m), E, Mmax, _ptr(W),
                                             _ptr(sw), N, K, SCHEME[scheme], ACC[acc],
                                             OUT[out_type], _ptr(out), _ptr(ws), nws, _ptr(st),
                                             _stream()), "wq_grouped_gemm_w8a8_masked")
    return out


# ---------------------------------------------------------------- activation / combine
def silu_mul_quant(gu, group=0):
    _dev(gu, torch.bfloat16, "gu")
    R, I2 = gu.shape
    I = I2 // 2
    hq = torch.empty(R, I, dtype=torch.int8, device=gu.device)
    sh = torch.empty((R,) if group == 0 else (R, I // group), dtype=torch.float32, device=gu.device)
    _check(lib().wq_silu_mul_quant(_ptr(gu), R, I, group, _ptr(hq), _ptr(sh), _stream()),
           "wq_silu_mul_quant")
    return hq, sh


def moe_combine(y, pair_to_row, w, k):
    _dev(y, torch.bfloat16, "y")
    _dev(pair_to_row, torch.int32, "pair_to_row")
    _dev(w, torch.float32, "w")
    T = w.shape[0]
    H = y.shape[1]
    out = torch.empty(T, H, dtype=torch.bfloat16, device=y.device)
    _check(lib().wq_moe_combine(_ptr(y), _ptr(pair_to_row), _ptr(w), T, k, H, _ptr(out), _stream()),
           "wq_moe_combine")
    return out


# ---------------------------------------------------------------- the layer
def forward_workspace(T, H, I, E, k, scheme, device="cuda", host=False):
    f = lib().wq_moe_forward_host_workspace_size if host else lib().wq_moe_forward_workspace_size
    n = f(T, H, I, E, k, SCHEME[scheme])
    if n == 0:
        raise WQError("unsupported layer shape")
    return torch.empty(n, dtype=torch.uint8, device=device)


def moe_forward(x, logits, W13, sw13, W2, sw2, k, scheme="channel", acc="i32", out=None, ws=None,
                status=None):
    _dev(x, torch.bfloat16, "x")
    _dev(logits, torch.float32, "logits")
    _dev(W13, torch.int8, "W13")
    _dev(W2, torch.int8, "W2")
    _dev(sw13, torch.float32, "sw13")
    _dev(sw2, torch.float32, "sw2")
    T, H = x.shape
    E, N1, _ = W13.shape
    I = N1 // 2
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = forward_workspace(T, H, I, E, k, scheme, x.device)
    st = status if status is not None else new_status(x.device)
    _check(lib().wq_moe_forward(_ptr(x), _ptr(logits), _ptr(W13), _ptr(sw13), _ptr(W2), _ptr(sw2),
                                T, H, I, E, k, SCHEME[scheme], ACC[acc], _ptr(out), _ptr(ws),
                                ws.numel(), _ptr(st), _stream()), "wq_moe_forward")
    return out


def moe_forward_host(x_host, logits_host, W13, sw13, W2, sw2, k, scheme="channel", acc="i32",
                     out_host=None, ws=None, status=None):
    """Host (ideally pinned) x / logits / out; copies happen inside the call."""
    if x_host.is_cuda or logits_host.is_cuda:
        raise WQError("moe_forward_host takes host tensors")
    T, H = x_host.shape
    E, N1, _ = W13.shape
    I = N1 // 2
    if out_host is None:
        out_host = torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True)
    if ws is None:
        ws = forward_workspace(T, H, I, E, k, scheme, W13.device, host=True)
    st = status if status is not None else new_status(W13.device)
    _check(lib().wq_moe_forward_host(_ptr(x_host), _ptr(logits_host), _ptr(W13), _ptr(sw13),
                                     _ptr(W2), _ptr(sw2), T, H, I, E, k, SCHEME[scheme], ACC[acc],
                                     _ptr(out_host), _ptr(ws), ws.numel(), _ptr(st), _stream()),
           "wq_moe_forward_host")
    return out_host


def moe_forward_masked(a, sa, masked_m, W13, sw13, W2, sw2, scheme="channel", acc="i32", y=None,
                       ws=None, status=None):
    _dev(a, torch.int8, "a")
    _dev(sa, torch.float32, "sa")
    _dev(masked_m, torch.int32, "masked_m")
    E, Mmax, H = a.shape
    I = W13.shape[1] // 2
    if y is None:
        y = torch.empty(E, Mmax, H, dtype=torch.bfloat16, device=a.device)
    if ws is None:
        n = lib().wq_moe_forward_masked_workspace_size(E, Mmax, H, I, SCHEME[scheme])
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=a.device)
    st = status if status is not None else new_status(a.device)
    _check(lib().wq_moe_forward_masked(_ptr(a), _ptr(sa), _ptr(masked_m), E, Mmax, _ptr(W13),
                                       _ptr(sw13), _ptr(W2), _ptr(sw2), H, I, SCHEME[scheme],
                                       ACC[acc], _ptr(y), _ptr(ws), ws.numel(), _ptr(st),
                                       _stream()), "wq_moe_forward_masked")
    return y


# ---------------------------------------------------------------- W4A8 (int4 weights)
def quantize_weight_int4(w):
    """bf16 [N, K] -> (int4 codes two per byte uint8 [N, K/2], scales [N])."""
    _dev(w, torch.bfloat16, "w")
    N, K = w.shape
    q4 = torch.empty(N, K // 2, dtype=torch.uint8, device=w.device)
    s = torch.empty(N, dtype=torch.float32, device=w.device)
    _check(lib().wq_quantize_weight_int4(_ptr(w), N, K, _ptr(q4), _ptr(s), _stream()),
           "wq_quantize_weight_int4")
    return q4, s


def grouped_gemm_w4a8_masked(A, sa, masked_m, W4, s4, out_type="bf16", out=None, status=None):
    _dev(A, torch.int8, "A")
    _dev(sa, torch.float32, "sa")
    _dev(masked_m, torch.int32, "masked_m")
    _dev(W4, torch.uint8, "W4")
    _dev(s4, torch.float32, "s4")
    E, Mmax, K = A.shape
    N = W4.shape[1]
    if out is None:
        out = torch.empty(E, Mmax, N, dtype=torch.bfloat16 if out_type == "bf16" else torch.int32,
                          device=A.device)
    nws = lib().wq_grouped_gemm_masked_workspace_size(E, Mmax)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=A.device)
    st = status if status is not None else new_status(A.device)
    _check(lib().wq_grouped_gemm_w4a8_masked(_ptr(A), _ptr(sa), _ptr(masked_m), E, Mmax, _ptr(W4),
                                             _ptr(s4), N, K, OUT[out_type], _ptr(out), _ptr(ws),
                                             nws, _ptr(st), _stream()),
           "wq_grouped_gemm_w4a8_masked")
    return out


def moe_forward_masked_w4a8(a, sa, masked_m, W13, s13, W2, s2, y=None, ws=None, status=None):
    _dev(a, torch.int8, "a")
    _dev(sa, torch.float32, "sa")
    _dev(masked_m, torch.int32, "masked_m")
    _dev(W13, torch.uint8, "W13")
    _dev(W2, torch.uint8, "W2")
    E, Mmax, H = a.shape
    I = W13.shape[1] // 2
    if y is None:
        y = torch.empty(E, Mmax, H, dtype=torch.bfloat16, device=a.device)
    if ws is None:
        n = lib().wq_moe_forward_masked_w4a8_workspace_size(E, Mmax, H, I)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=a.device)
    st = status if status is not None else new_status(a.device)
    _check(lib().wq_moe_forward_masked_w4a8(_ptr(a), _ptr(sa), _ptr(masked_m), E, Mmax, _ptr(W13),
                                            _ptr(s13), _ptr(W2), _ptr(s2), H, I, _ptr(y), _ptr(ws),
                                            ws.numel(), _ptr(st), _stream()),
           "wq_moe_forward_masked_w4a8")
    return y


# ---------------------------------------------------------------- dense linear
def linear_workspace(T, K, N, scheme, device):
    n = lib().wq_linear_w8a8_workspace_size(T, K, N, SCHEME[scheme])
    if n == 0:
        raise WQError(f"linear shape T={T} K={K} N={N} ({scheme}) is not supported")
    return torch.empty(n, dtype=torch.uint8, device=device)


def linear_w8a8(x, W, sw, scheme="channel", acc="i32", out=None, ws=None, status=None):
    """Dense W8A8 INT8 linear: quantize x (bf16 [T, K]) and multiply by the
    int8 weights W [N, K] with their scales; bf16 [T, N]."""
    _dev(x, torch.bfloat16, "x")
    _dev(W, torch.int8, "W")
    _dev(sw, torch.float32, "sw")
    T, K = x.shape
    N = W.shape[0]
    if out is None:
        out = torch.empty(T, N, dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = linear_workspace(T, K, N, scheme, x.device)
    st = status if status is not None else new_status(x.device)
    _check(lib().wq_linear_w8a8(_ptr(x), T, K, x.stride(0), _ptr(W), _ptr(sw), N, SCHEME[scheme],
                                ACC[acc], _ptr(out), _ptr(ws), ws.numel(), _ptr(st), _stream()),
           "wq_linear_w8a8")
    return out

