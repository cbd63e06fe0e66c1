"""Host-side checks of libwq.so that need no GPU: it loads, exports every
entry point include/wq.h declares, sizes workspaces, and rejects bad
arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

from w8a8_int8_quantized_token_gb300 import binding, build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return binding.lib()


def header_names():
    txt = open(os.path.join(ROOT, "include", "wq.h")).read()
    return sorted(set(re.findall(r"WQ_API\s+[\w\s\*]*?\b(wq_\w+)\s*\(", txt)))


def test_header_declares_entry_points():
    names = header_names()
    assert len(names) >= 21
    assert set(names) == set(binding.exported_names())


def test_library_exports_every_declared_symbol(lib):
    h = ctypes.CDLL(binding.LIB_PATH)
    for n in header_names():
        assert hasattr(h, n), n


def test_status_strings(lib):
    for code in range(0, -8, -1):
        assert lib.wq_status_string(code) and lib.wq_status_string(code) != b"unknown status"
    assert lib.wq_status_string(99) == b"unknown status"


def test_launch_counter_ignores_rejected_calls(lib):
    P = ctypes.c_void_p
    fake = P(4096)
    n0 = lib.wq_kernel_launches()
    assert lib.wq_route_topk(fake, 4, 8, 9, fake, fake, None) == -1
    assert lib.wq_quantize_per_token(fake, 4, 12, 12, fake, fake, None) == -2
    assert lib.wq_kernel_launches() == n0


def test_workspace_sizes(lib):
    # forward workspace holds at least A, GU, y of the prefill shape
    T, H, I, E, k = 8192, 7168, 2048, 256, 8
    n = lib.wq_moe_forward_workspace_size(T, H, I, E, k, 0)
    R = T * k
    assert n >= R * H + R * 2 * I * 2 + R * I + R * H * 2
    assert lib.wq_moe_forward_host_workspace_size(T, H, I, E, k, 0) >= n + T * H * 4
    assert lib.wq_moe_forward_workspace_size(T, 100, I, E, k, 0) == 0  # H % 128
    assert lib.wq_moe_align_workspace_size(T, k, E) >= (R // 256) * E * 4
    assert lib.wq_grouped_gemm_workspace_size(R, E) > 0


def test_masked_workspace_holds_the_fp16_token_rows(lib):
    """The masked layer's workspace carries the fp16 copy of a GEMM input's
    rows ([E*Mmax][max(H, I)], plus int32 norms) exactly when the int8-code
    engine takes 256-token tiles on the channel scheme: more than 64 rows per
    expert buffer.  Block scheme and Mmax <= 64 go without it."""
    E, H, I = 32, 7168, 2048
    per_row = 2 * I * 2 + I + 4  # GEMM1 output, h codes, h scale
    f16_row = max(H, I) * 2 + 4
    for Mmax in (64, 65, 512):
        R = E * Mmax
        ch = lib.wq_moe_forward_masked_workspace_size(E, Mmax, H, I, 0)
        blk = lib.wq_moe_forward_masked_workspace_size(E, Mmax, H, I, 1)
        w4 = lib.wq_moe_forward_masked_w4a8_workspace_size(E, Mmax, H, I)
        assert w4 == ch
        assert blk < R * (per_row + f16_row)
        if Mmax > 64:
            assert ch >= R * (per_row + f16_row)
        else:
            assert R * per_row <= ch < R * (per_row + f16_row)


def test_invalid_arguments_rejected_on_host(lib):
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: argument checks fail first
    # k > E
    assert lib.wq_route_topk(fake, 4, 8, 9, fake, fake, None) == -1
    # E > 1024
    assert lib.wq_route_topk(fake, 4, 2000, 8, fake, fake, None) == -1
    # negative sizes
    assert lib.wq_quantize_per_token(fake, -1, 16, 16, fake, fake, None) == -1
    # ldx < K
    assert lib.wq_quantize_per_token(fake, 4, 16, 8, fake, fake, None) == -1
    # K not a multiple of 8
    assert lib.wq_quantize_per_token(fake, 4, 12, 12, fake, fake, None) == -2
    # unsupported group
    assert lib.wq_quantize_per_token_group(fake, 4, 256, 256, 100, fake, fake, None) == -2
    # bad scheme / acc / raw int32 with the block scheme
    assert lib.wq_grouped_gemm_w8a8(fake, fake, fake, fake, fake, 4, 16, 128, 128, 7, 0, 0, fake,
                                    fake, 1 << 20, None, None) == -1
    assert lib.wq_grouped_gemm_w8a8(fake, fake, fake, fake, fake, 4, 16, 128, 128, 1, 0, 1, fake,
                                    fake, 1 << 20, None, None) == -1
    # N not a multiple of 128
    assert lib.wq_grouped_gemm_w8a8(fake, fake, fake, fake, fake, 4, 16, 96, 128, 0, 0, 0, fake,
                                    fake, 1 << 20, None, None) == -2
    # workspace too small
    assert lib.wq_grouped_gemm_w8a8(fake, fake, fake, fake, fake, 4, 16, 128, 128, 0, 0, 0, fake,
                                    fake, 1, None, None) == -5
    assert lib.wq_moe_align(fake, 4, 2, 8, 1, fake, fake, fake, fake, fake, 0, None, None) == -5
    # null pointers
    assert lib.wq_moe_combine(None, fake, fake, 4, 2, 64, fake, None) == -1
    # empty problems enqueue nothing and succeed without a device
    assert lib.wq_quantize_per_token(None, 0, 16, 16, None, None, None) == 0
    assert lib.wq_grouped_gemm_w8a8(None, None, None, None, None, 4, 0, 128, 128, 0, 0, 0, None,
                                    None, 0, None, None) == 0


def test_newer_entry_points_reject_bad_arguments_on_host(lib):
    """The dense linear, the FP8 weight converter and the fp16-code entries
    check their arguments on the host, before touching a device."""
    fake = 4096  # never dereferenced: argument checks fail first
    big = 1 << 30
    # dense linear: negative T, bad scheme, K not a multiple of 128, ldx < K
    assert lib.wq_linear_w8a8(fake, -1, 128, 128, fake, fake, 256, 0, 0, fake, fake, big, None,
                              None) == -1
    assert lib.wq_linear_w8a8(fake, 4, 128, 128, fake, fake, 256, 7, 0, fake, fake, big, None,
                              None) == -1
    assert lib.wq_linear_w8a8(fake, 4, 100, 100, fake, fake, 256, 0, 0, fake, fake, big, None,
                              None) == -2
    assert lib.wq_linear_w8a8(fake, 4, 128, 64, fake, fake, 256, 0, 0, fake, fake, big, None,
                              None) == -1
    # ... a workspace smaller than its size function says; no rows is a no-op
    need = lib.wq_linear_w8a8_workspace_size(4, 128, 256, 0)
    assert need > 0 and lib.wq_linear_w8a8_workspace_size(4, 100, 256, 0) == 0
    assert lib.wq_linear_w8a8(fake, 4, 128, 128, fake, fake, 256, 0, 0, fake, fake, need - 1,
                              None, None) == -5
    assert lib.wq_linear_w8a8(None, 0, 128, 128, None, None, 256, 0, 0, None, None, 0, None,
                              None) == 0
    # FP8 weight converter: negative size, bad scheme, sizes off the 128 grid
    assert lib.wq_convert_fp8_weights(fake, fake, -1, 128, 0, fake, fake, None) == -1
    assert lib.wq_convert_fp8_weights(fake, fake, 128, 128, 5, fake, fake, None) == -1
    assert lib.wq_convert_fp8_weights(fake, fake, 100, 128, 0, fake, fake, None) == -2
    assert lib.wq_convert_fp8_weights(None, None, 0, 128, 1, None, None, None) == 0
    # SiLU-mul-quant to fp16 codes: negative rows, unsupported group, missing
    # norms for per-row scales, width not a multiple of 8
    assert lib.wq_silu_mul_quant_f16(fake, -1, 128, 0, fake, fake, fake, None) == -1
    assert lib.wq_silu_mul_quant_f16(fake, 4, 128, 100, fake, fake, fake, None) == -2
    assert lib.wq_silu_mul_quant_f16(fake, 4, 128, 0, fake, fake, None, None) == -1
    assert lib.wq_silu_mul_quant_f16(fake, 4, 12, 0, fake, fake, fake, None) == -2
    assert lib.wq_silu_mul_quant_f16(None, 0, 128, 0, None, None, None, None) == 0
    # fp16-code grouped GEMM: negative rows, missing norms (channel-wise),
    # N not a multiple of 256, workspace too small
    gemm = lambda n2, R, N, ws: lib.wq_grouped_gemm_w8a8_f16codes(
        fake, n2, fake, fake, fake, fake, 4, R, N, 128, 0, 0, 0, fake, fake, ws, None, None)
    assert gemm(fake, -1, 256, big) == -1
    assert gemm(None, 16, 256, big) == -1
    assert gemm(fake, 16, 128, big) == -2
    assert gemm(fake, 16, 256, 1) == -5
    assert gemm(None, 0, 256, 0) == 0
    # fp16 permute: no groups, rows not a multiple of 16 codes
    assert lib.wq_moe_permute_f16(fake, fake, 0, 4, 2, 128, fake, 8, fake, fake, fake, None) == -1
    assert lib.wq_moe_permute_f16(fake, fake, 1, 4, 2, 8, fake, 8, fake, fake, fake, None) == -2
    assert lib.wq_moe_permute_f16(None, None, 1, 0, 2, 128, None, 0, None, None, None, None) == 0


def test_no_device_is_reported(lib):
    # this check runs where no GPU is visible; on a GPU machine device 10**6 does not exist
    assert lib.wq_init(10 ** 6) == -3


def test_noalloc_entry_checks_arguments_before_its_scratch_limit(lib):
    """The allocation-free grouped GEMM rejects the calls the workspace entry
    rejects, with the same codes, before it compares the problem with its
    static scratch array."""
    fake = ctypes.c_void_p(4096)  # never dereferenced
    for E, R, scheme, want in ((5000, 4_000_000, 0, -1), (5000, 100, 0, -1), (256, 4_000_000, 7, -1),
                               (256, 4_000_000, 0, -2)):
        rc = lib.wq_grouped_gemm_w8a8_noalloc(fake, fake, fake, fake, fake, E, R, 4096, 7168, scheme,
                                              0, 0, fake, None, None)
        assert rc == want, (E, R, scheme, rc)
