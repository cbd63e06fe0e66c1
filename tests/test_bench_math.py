"""The measurement arithmetic `bench.py` reports (no GPU): the layer's
algorithmic op count and minimal bytes, GEMM1's algorithmic flops and bytes,
the choice of the tensor peak from the clocks sampled during the timed
region, the choice of bound from the ridge point, the fractions, and the
rule that a captured DRAM-traffic figure is reported only for the kernel
source it was measured on."""
import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6783.8, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1707.9}
AT_MAX = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
CAPPED = {"sm_mhz": 1462.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}


def test_tensor_peak_follows_the_sampled_clock():
    assert bench.tensor_peak(PEAKS, AT_MAX)[0] == 1900.0      # burst: clock at its maximum
    assert bench.tensor_peak(PEAKS, CAPPED)[0] == 1707.9      # sustained: power-capped
    low = {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.tensor_peak(PEAKS, low)[0] == 1707.9
    cap_at_max = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert bench.tensor_peak(PEAKS, cap_at_max)[0] == 1707.9
    # no samples: the larger (burst) figure, so the fraction is not flattered
    assert bench.tensor_peak(PEAKS, {"sm_mhz": None, "sm_max_mhz": None})[0] == 1900.0
    assert bench.tensor_peak(PEAKS, {})[0] == 1900.0


def test_layer_ops_at_prefill():
    # 2 ops per multiply-add of gate_up (2I x H) and down (H x I) over T*k pairs
    T, H, I, k = 8192, 7168, 2048, 8
    assert bench.layer_ops(T, H, I, k) == 2.0 * T * k * 3 * H * I
    assert bench.layer_ops(T, H, I, k) == pytest.approx(5.7724e12, rel=1e-4)


def test_prefill_gemm1_is_tensor_bound():
    rows, touched, H, I = 8192 * 8, 256, 7168, 2048
    r = bench.gemm1_roofline(PEAKS, "measured", 3.118, rows, touched, H, I, "channel", 2, None,
                             AT_MAX)
    weights = touched * 2 * I * H
    assert r["flops"] == 2.0 * rows * 2 * I * H
    assert r["algorithmic_bytes"] == (weights + touched * 2 * I * 4 + rows * H * 2 + rows * 4
                                      + rows * 2 * I * 2)
    assert r["algorithmic_bytes"] == pytest.approx(8.997e9, rel=1e-3)
    # 428 flop/B against a ridge of 1900 TFLOP/s / 6783.8 GB/s = 280 flop/B; a
    # kernel timed at the maximum SM clock takes the burst peak
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 1900.0
    assert r["achieved"] == pytest.approx(r["flops"] / 3.118e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 1900.0)
    assert r["traffic"] is None
    rc = bench.gemm1_roofline(PEAKS, "measured", 3.118, rows, touched, H, I, "channel", 2, None,
                              CAPPED)
    assert rc["peak"] == 1707.9 and rc["frac"] == pytest.approx(rc["achieved"] / 1707.9)


def test_gemm2_roofline_swaps_n_and_k():
    rows, touched, H, I = 8192 * 8, 256, 7168, 2048
    r = bench.gemm_roofline(PEAKS, "measured", AT_MAX, 1.8, rows, touched, H, I, "channel", 2,
                            None, "down")
    assert r["flops"] == 2.0 * rows * H * I == pytest.approx(1.924e12, rel=1e-3)
    assert r["algorithmic_bytes"] == (touched * H * I + touched * H * 4 + rows * I * 2 + rows * 4
                                      + rows * H * 2)
    assert r["bound"] == "tensor" and r["frac"] == pytest.approx(r["flops"] / 1.8e-3 / 1e12 / 1900)


def test_layer_roofline_at_prefill():
    T, H, I, E, k = 8192, 7168, 2048, 256, 8
    nbytes = bench.layer_bytes(T, H, I, E, k, "channel", E)
    # all experts' int8 weights and channel scales, x and out in bf16, logits
    assert nbytes == E * 3 * H * I + E * (2 * I + H) * 4 + 2 * T * H * 2 + T * E * 4
    assert nbytes == pytest.approx(11.52e9, rel=2e-3)
    ops = bench.layer_ops(T, H, I, k)
    r = bench.layer_roofline(PEAKS, AT_MAX, 5.72, ops, nbytes)
    floor = max(ops / 1900e12, nbytes / 6783.8e9) * 1e3
    assert r["bound"] == "tensor" and r["floor_ms"] == pytest.approx(floor)
    assert r["frac"] == pytest.approx(floor / 5.72)
    blk = bench.layer_bytes(4096, H, I, E, k, "block", E)
    assert blk - bench.layer_bytes(4096, H, I, E, k, "channel", E) == \
        E * ((2 * I // 128) * (H // 128) + (H // 128) * (I // 128) - 2 * I - H) * 4


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
