"""Failure path of the bounded pipeline waits, on the GPU without a fault.

Every pipeline wait in the tensor-core engines gives up after 1 s, records
WQ_ERR_TIMEOUT in the caller's status word and tears the kernel down (waits
for its own copies, frees tensor memory).  The self-test entry makes the
block engine's first wait one that nothing completes, before any copy or MMA
is issued; the test reads the status back and then runs a normal call on the
same context.
"""
import time

import numpy as np
import pytest
import torch

from oracle import wq_oracle as O
from w8a8_int8_quantized_token_gb300 import binding as wq
from wq_testutil import assert_bf16_equal, bits

DEV = torch.device("cuda:0")
WQ_ERR_TIMEOUT = -7


@pytest.fixture(scope="module", autouse=True)
def _init():
    from w8a8_int8_quantized_token_gb300 import build_lib
    build_lib.build()
    wq.init(0)


@pytest.mark.gpu
def test_wait_timeout_records_status_and_context_survives():
    rng = np.random.default_rng(3)
    E, R, N, K = 1, 16, 256, 256
    A = rng.integers(-127, 128, (R, K), dtype=np.int8)
    W = rng.integers(-127, 128, (E, N, K), dtype=np.int8)
    sa = (rng.random((R, K // 128)) * 0.05).astype(np.float32)
    sw = (rng.random((E, N // 128, K // 128)) * 1e-3).astype(np.float32)
    offs = np.array([0, R], dtype=np.int32)
    t = lambda a: torch.from_numpy(a).to(DEV)
    A16, sa_d, W_d, sw_d, offs_d = t(A).to(torch.float16), t(sa), t(W), t(sw), t(offs)
    out = torch.full((R, N), 5.0, dtype=torch.bfloat16, device=DEV)
    st = wq.new_status()
    torch.cuda.synchronize()
    t0 = time.monotonic()
    wq.selftest_wait_timeout(A16, sa_d, W_d, sw_d, offs_d, out, st)
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    assert int(st.item()) == WQ_ERR_TIMEOUT
    assert waited >= 0.9  # the wait ran to its 1 s limit
    assert bool((out == 5.0).all())  # nothing was computed or written
    # the same context runs the engine normally afterwards
    st2 = wq.new_status()
    wq.grouped_gemm_w8a8_f16codes(A16, None, sa_d, W_d, sw_d, offs_d, acc="f32", out=out,
                                  status=st2, scheme="block")
    assert int(st2.item()) == 0
    assert_bf16_equal(bits(out), O.grouped_gemm_w8a8(A, sa, W, sw, offs, "block", "f32"),
                      "block gemm after a timed-out launch")
