"""The allocation-free grouped GEMM entry point (wq_grouped_gemm_w8a8_noalloc).

It serves callers that may not allocate device memory at run time; its
scratch is a static device array shared by every call.  Its results must be
those of wq_grouped_gemm_w8a8 (which takes a caller workspace) exactly, on
consecutive calls with different problems (so the second call runs on
scratch the first call left behind), and a problem too large for the array
must be refused before any work is enqueued.  Kept in the file pytest
collects last."""
import ctypes

import numpy as np
import pytest
import torch

from w8a8_int8_quantized_token_gb300 import binding as wq
from w8a8_int8_quantized_token_gb300 import build_lib

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _case(seed, counts, N, K, scheme):
    rng = np.random.default_rng(seed)
    E = len(counts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offs[-1])
    A = rng.integers(-127, 128, (R, K), dtype=np.int8)
    W = rng.integers(-60, 61, (E, N, K), dtype=np.int8)
    if scheme == "channel":
        sa, sw = rng.random(R) * 0.05, rng.random((E, N)) * 1e-3
    else:
        sa, sw = rng.random((R, K // 128)) * 0.05, rng.random((E, N // 128, K // 128)) * 1e-3
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    return t(A), t(sa.astype(np.float32)), t(W), t(sw.astype(np.float32)), t(offs)


def _noalloc(A, sa, W, sw, offs, scheme, acc, out_type, out, status):
    P = lambda x: ctypes.c_void_p(x.data_ptr())
    R, K = A.shape
    E, N, _ = W.shape
    return wq.lib().wq_grouped_gemm_w8a8_noalloc(
        P(A), P(sa), P(W), P(sw), P(offs), E, R, N, K, wq.SCHEME[scheme], wq.ACC[acc],
        wq.OUT[out_type], P(out), P(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    build_lib.build()
    wq.init(0)
    cases = [(1, [3, 0, 300, 17], 512, 1024, "channel", "i32", "bf16"),
             (2, [129, 1, 64], 256, 384, "block", "f32", "bf16"),
             (3, [40, 200], 256, 2048, "channel", "i32", "i32")]
    for seed, counts, N, K, scheme, acc, out_type in cases:
        A, sa, W, sw, offs = _case(seed, counts, N, K, scheme)
        ref = wq.grouped_gemm_w8a8(A, sa, W, sw, offs, scheme, acc, out_type)
        out = torch.zeros_like(ref)
        st = wq.new_status()
        assert _noalloc(A, sa, W, sw, offs, scheme, acc, out_type, out, st) == 0
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        if out_type == "bf16":
            assert torch.equal(out.float(), ref.float())
        else:
            assert torch.equal(out, ref)


def test_noalloc_refuses_problems_beyond_its_scratch():
    lib = wq.lib()
    fake = ctypes.c_void_p(4096)  # never dereferenced: the size check comes first
    R = 4_000_000
    assert lib.wq_grouped_gemm_workspace_size(R, 256) > 256 * 1024
    rc = lib.wq_grouped_gemm_w8a8_noalloc(fake, fake, fake, fake, fake, 256, R, 4096, 7168, 0, 0, 0,
                                          fake, None, None)
    assert rc == -2


def test_noalloc_rejects_bad_arguments_like_the_workspace_entry():
    """The same argument checks, with the same codes, come before the scratch
    limit: E > 4096 and a bad scheme are invalid arguments even when the
    problem would also be too large for the scratch array."""
    lib = wq.lib()
    fake = ctypes.c_void_p(4096)  # never dereferenced: argument checks fail first
    for E, R, scheme in ((5000, 4_000_000, 0), (5000, 100, 0), (256, 4_000_000, 7)):
        ws_rc = lib.wq_grouped_gemm_w8a8(fake, fake, fake, fake, fake, E, R, 4096, 7168, scheme, 0,
                                         0, fake, fake, 1 << 40, None, None)
        na_rc = lib.wq_grouped_gemm_w8a8_noalloc(fake, fake, fake, fake, fake, E, R, 4096, 7168,
                                                 scheme, 0, 0, fake, None, None)
        assert ws_rc == na_rc == -1, (E, R, scheme, ws_rc, na_rc)
