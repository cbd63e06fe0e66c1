"""The measurement arithmetic `bench.py` reports (no GPU): the layer's
algorithmic op count, GEMM1's algorithmic flops and bytes, the choice of
bound from the measured peaks' ridge point, the fraction, and the rule that
a captured DRAM-traffic figure is reported only for the kernel source it was
measured on."""
import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6783.8, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1707.9}


def test_layer_ops_at_prefill():
    # 2 ops per multiply-add of gate_up (2I x H) and down (H x I) over T*k pairs
    T, H, I, k = 8192, 7168, 2048, 8
    assert bench.layer_ops(T, H, I, k) == 2.0 * T * k * 3 * H * I
    assert bench.layer_ops(T, H, I, k) == pytest.approx(5.7724e12, rel=1e-4)


def test_prefill_gemm1_is_tensor_bound():
    rows, touched, H, I = 8192 * 8, 256, 7168, 2048
    r = bench.gemm1_roofline(PEAKS, "measured", 3.118, rows, touched, H, I, "channel", 2, None)
    weights = touched * 2 * I * H
    assert r["flops"] == 2.0 * rows * 2 * I * H
    assert r["algorithmic_bytes"] == (weights + touched * 2 * I * 4 + rows * H * 2 + rows * 4
                                      + rows * 2 * I * 2)
    assert r["algorithmic_bytes"] == pytest.approx(8.997e9, rel=1e-3)
    # 428 flop/B against a ridge of 1707.9 TFLOP/s / 6783.8 GB/s = 252 flop/B
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 1707.9
    assert r["achieved"] == pytest.approx(r["flops"] / 3.118e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 1707.9)
    assert r["traffic"] is None


def test_decode_gemm1_is_hbm_bound():
    rows, touched, H, I = 128 * 8, 253, 7168, 2048  # the seed-0 decode workload touches 253
    r = bench.gemm1_roofline(PEAKS, "measured", 1.165, rows, touched, H, I, "channel", 1, None)
    assert r["algorithmic_bytes"] == pytest.approx(7.448e9, rel=1e-3)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6783.8
    assert r["achieved"] == pytest.approx(r["algorithmic_bytes"] / 1.165e-3 / 1e9)


def test_block_scales_are_counted_per_block():
    rows, touched, H, I = 4096 * 8, 256, 7168, 2048
    ch = bench.gemm1_roofline(PEAKS, "m", 1.0, rows, touched, H, I, "channel", 2, None)
    bl = bench.gemm1_roofline(PEAKS, "m", 1.0, rows, touched, H, I, "block", 2, None)
    extra_w = touched * ((2 * I // 128) * (H // 128) - 2 * I) * 4
    extra_a = rows * (H // 128 - 1) * 4
    assert bl["algorithmic_bytes"] - ch["algorithmic_bytes"] == extra_w + extra_a


def test_traffic_figure_only_for_its_kernel_source(monkeypatch):
    path = os.path.join(ROOT, "w8a8_int8_quantized_token_gb300", "csrc", "wq_gemm_tc5.cu")
    digest = hashlib.sha256(open(path, "rb").read()).hexdigest()
    entry = {"kernel": "k", "file": "wq_gemm_tc5.cu", "bytes": 1.0, "how": "test"}
    monkeypatch.setitem(bench.TRAFFIC, "probe", dict(entry, sha256=digest))
    assert bench.measured_traffic("probe")["bytes"] == 1.0
    monkeypatch.setitem(bench.TRAFFIC, "probe", dict(entry, sha256="0" * 64))
    assert bench.measured_traffic("probe") is None
    assert bench.measured_traffic("no such workload") is None
