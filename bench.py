"""Benchmark of the W8A8 INT8 fused-MoE layer (DeepSeek-V3 shape) on GB300.

One step = the whole hot path on one batch: route -> quantize -> align ->
permute -> GEMM1 (gate_up) -> SiLU-mul + re-quantize -> GEMM2 (down) ->
combine.  Weights (11.3 GB of int8) and the step's activations are resident
in HBM before the timed region.  `value` times the one-call layer
(wq_moe_forward), recorded once into a CUDA graph before the timed region
and replayed K times (every kernel of every step runs; the same steps
launched call by call are reported as eager_ms_per_step); a second timed
pass runs the same steps as
separate C-ABI calls with CUDA events between them for the per-stage times
and the rooflines; `e2e` runs the layer through wq_moe_forward_host with
pinned host activations, copies included.

  python bench.py [--steps K] [--warmup W] [--config prefill]
  python bench.py --impl reference   # the CPU oracle on a bounded sample

One GPU only: the GEMM engines share token tiles between the two CTAs of a
cluster through TMA multicast, which this build keeps to one-GPU runs, so a
launch with WORLD_SIZE > 1 (or --gpus > 1) is refused before the library is
loaded.  The reference arm (CPU only) runs on rank 0 and the other ranks
exit without work.
"""
from __future__ import annotations

import argparse
import hashlib
import ctypes
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from w8a8_int8_quantized_token_gb300 import synth  # noqa: E402

METRIC = "INT8 MoE layer TOPS and tokens/s at DeepSeek-V3 shape; % INT8 tensor peak"
SCHEME = {"channel": 0, "block": 1}
ACC = {"i32": 0, "f32": 1}


def layer_ops(T, H, I, k):
    """Algorithmic integer ops of one layer step: 2 per multiply-add of the
    two GEMMs over the T*k routed (token, expert) pairs."""
    return 2.0 * T * k * (2 * I * H + H * I)


# DRAM traffic per launch of GEMM1's main kernel (dram__bytes_read.sum +
# dram__bytes_write.sum of one ncu capture on a reduced workload with the same
# rows per expert, scaled to the full launch by the expert count).  A figure
# holds only for the kernel source it was measured on: it is reported while
# that file's SHA-256 matches, else the traffic is null.
_TC5 = {"kernel": "gemm_tc5_kernel", "file": "wq_gemm_tc5.cu",
        "sha256": "792a3b6aafe1a478f31760a40b10d4e3ee71d55eb20606dd733a170a0d73c2a6",
        "bytes": 8 * (1.078654e9 + 63.810048e6),
        "how": "ncu capture of GEMM1 at 1024 tokens / 32 experts (same 256 rows per expert), "
               "dram read+write scaled by the expert count (x 8)"}
TRAFFIC = {
    "prefill": _TC5,
    "prefill_f32": _TC5,
    "decode": {"kernel": "gemm_small_kernel", "file": "wq_gemm_small.cu",
               "sha256": "97e5d6ef521a4ed0bec73de5804f6968d9db907316f3dcdca4395170e2a3132a",
               "bytes": 8 * (941.216512e6 + 4.608e6),
               "how": "ncu capture of GEMM1 at 16 tokens / 32 experts (same 4 rows per expert), "
                      "dram read+write scaled by the expert count (x 8)"},
    "block": {"kernel": "gemm_tc6_kernel", "file": "wq_gemm_tc6.cu",
              "sha256": "05be324188f32a9e8f688e68d5af108bc705afdcf669ac468d45b2ef63f5f898",
              "bytes": 8 * (1.021679e9 + 33.830144e6),
              "how": "ncu capture of GEMM1 at 512 tokens / 32 experts (same 128 rows per expert), "
                     "dram read+write scaled by the expert count (x 8)"},
}


def measured_traffic(cfg_name):
    t = TRAFFIC.get(cfg_name)
    if t is None:
        return None
    path = os.path.join(ROOT, "w8a8_int8_quantized_token_gb300", "csrc", t["file"])
    with open(path, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != t["sha256"]:
            return None
    return t


def tensor_peak(peaks, clocks):
    """The measured bf16 dense rate that applies to kernels timed in this run.

    The peaks file holds a burst figure (cuBLAS timed alone) and a sustained
    one (a seconds-long loop under the power cap, at a lower SM clock).  A
    kernel timed inside a short step runs at the burst condition when the SM
    clock sampled during the timed region stayed at its maximum with no power
    cap; otherwise the sustained figure applies.  Without clock samples the
    burst figure (the larger, so the smaller fraction) is taken."""
    burst = peaks["bf16_tflops"]
    sus = peaks.get("bf16_tflops_sustained", burst)
    mhz, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    capped = "sw_power_cap" in clocks.get("reasons", [])
    if mhz is None or not mx:
        return burst, "burst (no clock samples)"
    if mhz >= 0.97 * mx and not capped:
        return burst, "burst (SM clock at its maximum, no power cap, during the timed region)"
    return sus, "sustained (SM clock below its maximum or power-capped during the timed region)"


def gemm_roofline(peaks, src, clocks, ms, rows, touched, N, K, scheme, code_bytes, traffic,
                  kernel, weight_bytes=1.0):
    """Roofline of one grouped GEMM launch: algorithmic flops 2*rows*N*K and
    bytes (touched experts' int8 weights and scales, the activation codes and
    scales, the bf16 output), bound by whichever of the measured bf16 dense
    rate (tcgen05 kind::f16 runs at it) and the measured HBM copy bandwidth
    the arithmetic intensity reaches first.  weight_bytes: bytes per weight
    code (1 for int8, 0.5 for int4)."""
    blk = scheme == "block"
    flops = 2.0 * rows * N * K
    nbytes = (touched * N * K * weight_bytes + touched * ((N // 128) * (K // 128) if blk else N) * 4
              + rows * K * code_bytes + rows * (K // 128 if blk else 1) * 4 + rows * N * 2)
    tf, which = tensor_peak(peaks, clocks)
    bw = peaks["hbm_gbs"]
    sec = ms / 1e3
    if flops / nbytes >= tf * 1e12 / (bw * 1e9):
        r = {"bound": "tensor", "achieved": flops / sec / 1e12, "peak": tf, "unit": "TFLOP/s",
             "peak_source": f"{src} bf16 dense, {which} (fp16 tcgen05 kind::f16 runs at the bf16 "
                            f"rate; sm_103a has no kind::i8)"}
    else:
        r = {"bound": "hbm", "achieved": nbytes / sec / 1e9, "peak": bw, "unit": "GB/s",
             "peak_source": f"{src} HBM copy bandwidth"}
    r["frac"] = r["achieved"] / r["peak"]
    r["kernel"] = kernel
    r["ms"] = ms
    r["traffic"] = traffic["bytes"] if traffic else None
    if traffic:
        r["traffic_source"] = traffic["how"]
    r["algorithmic_bytes"] = nbytes
    r["flops"] = flops
    return r


def gemm1_roofline(peaks, src, g1_ms, rows, touched, H, I, scheme, code_bytes, traffic,
                   clocks=None):
    """The gate_up GEMM (N = 2I, K = H)."""
    return gemm_roofline(peaks, src, clocks or {}, g1_ms, rows, touched, 2 * I, H, scheme,
                         code_bytes, traffic, "grouped_gemm_w8a8 gate_up (GEMM1)")


def layer_bytes(T, H, I, E_touched, k, scheme, E):
    """Minimal bytes of one layer step: the touched experts' int8 weights and
    scales, the bf16 activations in and out, the float32 router logits."""
    blk = scheme == "block"
    w = E_touched * (2 * I * H + H * I)
    sc = E_touched * (((2 * I // 128) * (H // 128) + (H // 128) * (I // 128)) if blk
                      else (2 * I + H)) * 4
    return w + sc + T * H * 2 + T * E * 4 + T * H * 2


def layer_roofline(peaks, clocks, ms, ops, nbytes):
    """The layer against its floor max(ops / tensor peak, bytes / HBM)."""
    tf, which = tensor_peak(peaks, clocks)
    bw = peaks["hbm_gbs"]
    t_ops, t_bytes = ops / (tf * 1e12), nbytes / (bw * 1e9)
    floor = max(t_ops, t_bytes)
    return {"bound": "tensor" if t_ops >= t_bytes else "hbm", "floor_ms": floor * 1e3,
            "ms": ms, "frac": floor * 1e3 / ms, "ops": ops, "bytes": nbytes,
            "tensor_peak_tflops": tf, "hbm_gbs": bw, "peak_choice": which}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def capture_graph(wq, step, dev):
    """Record one call of `step` into a CUDA graph (first use and any
    side-stream setup happen in a plain call on the capture stream first);
    returns the graph and the library kernels one replay launches."""
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        step()
    torch.cuda.current_stream().wait_stream(cs)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    n0 = wq.lib().wq_kernel_launches()
    with torch.cuda.graph(graph):
        step()
    per_step = wq.lib().wq_kernel_launches() - n0
    torch.cuda.synchronize()
    return graph, per_step


class Layer:
    """Preallocated buffers and the staged C-ABI calls of one layer step."""


    def __init__(self, wq, cfg, dev, weights):
        self.wq, self.lib, self.cfg, self.dev = wq, wq.lib(), cfg, dev
        T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
        R = T * k
        blk = cfg.scheme == "block"
        self.g1 = H // 128 if blk else 1
        self.g2 = I // 128 if blk else 1
        e = lambda *s, dt: torch.empty(*s, dtype=dt, device=dev)
        self.ids, self.w = e(R, dt=torch.int32), e(R, dt=torch.float32)
        self.q, self.s = e(T, H, dt=torch.int8), e(T * self.g1, dt=torch.float32)
        self.counts, self.offsets = e(E, dt=torch.int32), e(E + 1, dt=torch.int32)
        self.sp, self.p2r = e(R, dt=torch.int32), e(R, dt=torch.int32)
        self.aws_n = self.lib.wq_moe_align_workspace_size(T, k, E)
        self.aws = e(max(self.aws_n, 1), dt=torch.uint8)
        # the one-call layer's choice: fp16-stored codes when both GEMM widths
        # are multiples of 256 and experts hold many rows
        self.f16 = ((2 * I) % 256 == 0
                    and H % 256 == 0 and R > 64 * E)
        cdt = torch.float16 if self.f16 else torch.int8
        # the one-call layer's kernels, in its order (each token quantized
        # once and written to its k rows, as int8 or fp16 codes)
        self.stages = ["route", "align", "quant_permute", "gemm1", "silu_mul_quant", "gemm2",
                       "combine"]
        self.A, self.sa = e(R, H, dt=cdt), e(R * self.g1, dt=torch.float32)
        self.anorm, self.hnorm = e(R, dt=torch.int32), e(R, dt=torch.int32)
        self.gu = e(R, 2 * I, dt=torch.bfloat16)
        self.hq, self.sh = e(R, I, dt=cdt), e(R * self.g2, dt=torch.float32)
        self.y = e(R, H, dt=torch.bfloat16)
        self.out = e(T, H, dt=torch.bfloat16)
        self.gws_n = max(self.lib.wq_grouped_gemm_workspace_size(R, E),
                         self.lib.wq_grouped_gemm_silu_quant_workspace_size(R, E))
        self.gws = e(self.gws_n, dt=torch.uint8)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.W13, self.S13, self.W2, self.S2 = weights

    def step(self, x, logits, ev=None):
        c, L, P = self.cfg, self.lib, lambda t: ctypes.c_void_p(t.data_ptr())
        T, H, I, E, k = c.T, c.H, c.I, c.E, c.k
        R = T * k
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        sc, ac = SCHEME[c.scheme], ACC[c.acc]
        n = [0]

        def rec():
            if ev is not None:
                ev[n[0]].record()
            n[0] += 1

        def ok(rc, what):
            if rc != 0:
                raise RuntimeError(f"{what} failed: {rc}")
        rec()
        ok(L.wq_route_topk(P(logits), T, E, k, P(self.ids), P(self.w), st), "route")
        rec()
        ok(L.wq_moe_align(P(self.ids), T, k, E, 1, P(self.counts), P(self.offsets), P(self.sp),
                          P(self.p2r), P(self.aws), self.aws_n, P(self.status), st), "align")
        rec()
        group = 128 if c.scheme == "block" else 0
        if self.f16:
            ok(L.wq_quantize_permute_f16(P(x), T, H, group, P(self.p2r), k, R, P(self.A), P(self.sa),
                                         P(self.anorm), st), "quant_permute")
            rec()
            ok(L.wq_grouped_gemm_w8a8_f16codes(P(self.A), P(self.anorm), P(self.sa), P(self.W13),
                                               P(self.S13), P(self.offsets), E, R, 2 * I, H, sc, ac,
                                               0, P(self.gu), P(self.gws), self.gws_n,
                                               P(self.status), st), "gemm1")
            rec()
            ok(L.wq_silu_mul_quant_f16(P(self.gu), R, I, 128 if c.scheme == "block" else 0,
                                       P(self.hq), P(self.sh), P(self.hnorm), st), "silu_mul_quant")
            rec()
            ok(L.wq_grouped_gemm_w8a8_f16codes(P(self.hq), P(self.hnorm), P(self.sh), P(self.W2),
                                               P(self.S2), P(self.offsets), E, R, H, I, sc, ac, 0,
                                               P(self.y), P(self.gws), self.gws_n, P(self.status),
                                               st), "gemm2")
        else:
            ok(L.wq_quantize_permute(P(x), T, H, group, P(self.p2r), k, R, P(self.A), P(self.sa), st),
               "quant_permute")
            rec()
            ok(L.wq_grouped_gemm_w8a8(P(self.A), P(self.sa), P(self.W13), P(self.S13),
                                      P(self.offsets), E, R, 2 * I, H, sc, ac, 0, P(self.gu),
                                      P(self.gws), self.gws_n, P(self.status), st), "gemm1")
            rec()
            ok(L.wq_silu_mul_quant(P(self.gu), R, I, 128 if c.scheme == "block" else 0, P(self.hq),
                                   P(self.sh), st), "silu_mul_quant")
            rec()
            ok(L.wq_grouped_gemm_w8a8(P(self.hq), P(self.sh), P(self.W2), P(self.S2),
                                      P(self.offsets), E, R, H, I, sc, ac, 0, P(self.y),
                                      P(self.gws), self.gws_n, P(self.status), st), "gemm2")
        rec()
        ok(L.wq_moe_combine(P(self.y), P(self.p2r), P(self.w), T, k, H, P(self.out), st), "combine")
        rec()
        assert n[0] == len(self.stages) + 1
        return self.out


    def time_fused(self, steps):
        """Block scheme: the fused gate_up -> SiLU-and-mul -> re-quantization
        entry on the last staged step's inputs, timed against the two staged
        calls it replaces; its codes and scales must equal theirs bit for bit."""
        c, L, P = self.cfg, self.lib, lambda t: ctypes.c_void_p(t.data_ptr())
        R, I, H, E = c.T * c.k, c.I, c.H, c.E
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        hq, sh = torch.empty_like(self.hq), torch.empty_like(self.sh)

        def call():
            rc = L.wq_grouped_gemm_w8a8_silu_quant_f16codes(
                P(self.A), P(self.sa), P(self.W13), P(self.S13), P(self.offsets), E, R, I, H,
                SCHEME[c.scheme], P(hq), P(sh), P(self.gws), self.gws_n, P(self.status), st)
            if rc != 0:
                raise RuntimeError(f"fused gemm1 failed: {rc}")
        call()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            call()
        e1.record()
        torch.cuda.synchronize()
        same = bool(torch.equal(hq.view(torch.int16), self.hq.view(torch.int16))
                    and torch.equal(sh, self.sh))
        if not same:
            raise RuntimeError("fused gemm1 codes differ from the staged ones")
        return {"ms": e0.elapsed_time(e1) / steps, "bit_exact_vs_staged": same,
                "replaces": "stages gemm1 + silu_mul_quant"}


def make_weights(wq, cfg, dev):
    """Draw each expert's bf16 weights on the device and quantize them with
    the library (offline step, untimed)."""
    E, I, H = cfg.E, cfg.I, cfg.H
    W13 = torch.empty(E, 2 * I, H, dtype=torch.int8, device=dev)
    W2 = torch.empty(E, H, I, dtype=torch.int8, device=dev)
    if cfg.scheme == "block":
        S13 = torch.empty(E, 2 * I // 128, H // 128, dtype=torch.float32, device=dev)
        S2 = torch.empty(E, H // 128, I // 128, dtype=torch.float32, device=dev)
    else:
        S13 = torch.empty(E, 2 * I, dtype=torch.float32, device=dev)
        S2 = torch.empty(E, H, dtype=torch.float32, device=dev)
    for e in range(E):
        w13, w2 = synth.expert_weights(cfg, e, device=dev)
        wq.quantize_weight(w13, cfg.scheme, W13[e], S13[e])
        wq.quantize_weight(w2, cfg.scheme, W2[e], S2[e])
    torch.cuda.synchronize(dev)
    return W13, S13, W2, S2


class ExpertStack:
    """Lazy [E, ...] stack for the oracle: only the experts a sample touches
    are materialised."""

    def __init__(self, arrays: dict, shape):
        self.arrays, self.shape = arrays, shape

    def __getitem__(self, e):
        return self.arrays[e]


def oracle_sample(cfg, n_tokens, dev):
    """Prepare the CPU oracle's layer on the first n_tokens tokens of the
    workload and return a function that runs it once and returns seconds.
    Weights of the touched experts are drawn (on the device, same generator
    as the GPU run) and quantized by the oracle itself, outside the clock."""
    from oracle import wq_oracle as O
    x, lg = synth.layer_inputs(cfg, device=dev)
    x, lg = x[:n_tokens].cpu(), lg[:n_tokens].cpu()
    xb = x.view(torch.int16).numpy().view(np.uint16)
    ids, _ = O.route_topk(lg.numpy(), cfg.k)
    touched = sorted(set(ids.reshape(-1).tolist()))
    W13, S13, W2, S2 = {}, {}, {}, {}
    bitsof = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    for e in touched:
        w13, w2 = synth.expert_weights(cfg, e, device=dev)
        W13[e], S13[e], W2[e], S2[e] = O.quantize_weights(bitsof(w13), bitsof(w2), cfg.scheme)
    E, I, H = cfg.E, cfg.I, cfg.H
    args = (ExpertStack(W13, (E, 2 * I, H)), ExpertStack(S13, None),
            ExpertStack(W2, (E, H, I)), ExpertStack(S2, None))
    lgn = lg.numpy()

    def run():
        t0 = time.perf_counter()
        O.moe_forward(xb, lgn, *args, cfg.k, cfg.scheme, cfg.acc)
        return time.perf_counter() - t0
    return run, layer_ops(n_tokens, H, I, cfg.k), len(os.sched_getaffinity(0))


def workload_name(cfg):
    acc = {"i32": "int32 accumulator", "f32": "fp32 accumulator"}[cfg.acc]
    return (f"DeepSeek-V3-shape {cfg.name} MoE layer, {cfg.scheme}-wise W8A8 INT8, {acc}: "
            f"{cfg.T} tokens, hidden {cfg.H}, intermediate {cfg.I}, {cfg.E} experts top-{cfg.k}")


def run_reference(args, cfg):
    """The reference arm: the CPU oracle as it stands, on the host cores,
    each step a bounded sample (the first --cpu-tokens tokens) of the same
    workload; rank 0 only."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    n = args.cpu_tokens
    run, ops, cores = oracle_sample(cfg, n, dev)
    for _ in range(args.warmup):
        run()
    per = [run() for _ in range(args.steps)]
    dt = float(np.mean(per))
    val = ops / dt / 1e12
    sample = f"first {n} of {cfg.T} tokens of the same workload (all top-{cfg.k} experts), full layer"
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TOPS",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8", "data": "synthetic",
            "config": {"workload": workload_name(cfg), "parallelism": "replicas"},
            "tokens_per_s": n / dt,
            "cpu_baseline": {"value": val, "unit": "TOPS", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def make_weights_int4(wq, cfg, dev):
    """Each expert's bf16 weights drawn on the device and quantized to int4
    codes (two per byte) with per-channel scales by the library."""
    E, I, H = cfg.E, cfg.I, cfg.H
    W13 = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=dev)
    W2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=dev)
    S13 = torch.empty(E, 2 * I, dtype=torch.float32, device=dev)
    S2 = torch.empty(E, H, dtype=torch.float32, device=dev)
    for e in range(E):
        w13, w2 = synth.expert_weights(cfg, e, device=dev)
        W13[e], S13[e] = wq.quantize_weight_int4(w13)
        W2[e], S2[e] = wq.quantize_weight_int4(w2)
    return W13, S13, W2, S2


def run_masked(args, cfg, w4=False):
    """The masked (expert-parallel-shaped) layout: per-expert buffers
    [E, Mmax, H] of int8 codes with per-row scales and Zipf(1.2) valid counts;
    one step = wq_moe_forward_masked (GEMM1 -> SiLU-mul + re-quantize -> GEMM2
    on the valid rows), or with w4 its int4-weight form
    wq_moe_forward_masked_w4a8.  GEMM1 alone is timed in a second pass for
    the roofline figure."""
    from w8a8_int8_quantized_token_gb300 import binding as wq
    from w8a8_int8_quantized_token_gb300 import build_lib
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build_lib.build()
    wq.init(0)
    E, Mmax, H, I = cfg.E, cfg.Mmax, cfg.H, cfg.I
    weights = make_weights_int4(wq, cfg, dev) if w4 else make_weights(wq, cfg, dev)
    xm, mm = synth.masked_inputs(cfg, device=dev)
    a, sa = wq.quantize_per_token(xm.reshape(E * Mmax, H))
    a, sa = a.view(E, Mmax, H), sa.view(E, Mmax)
    mmd = torch.from_numpy(mm).to(dev)
    y = torch.empty(E, Mmax, H, dtype=torch.bfloat16, device=dev)
    n = wq.lib().wq_moe_forward_masked_workspace_size(E, Mmax, H, I, SCHEME[cfg.scheme])
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    if w4:
        step = lambda: wq.moe_forward_masked_w4a8(a, sa, mmd, *weights, y=y, ws=ws, status=st)
    else:
        step = lambda: wq.moe_forward_masked(a, sa, mmd, *weights, cfg.scheme, cfg.acc, y=y, ws=ws,
                                             status=st)
    for _ in range(args.warmup):
        step()
    # one layer call recorded into a CUDA graph (the small-segment engine's
    # second stream included), outside the timed region
    graph, per_step = capture_graph(wq, step, dev)
    for _ in range(args.warmup):
        graph.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("timed")
        e0.record()
        for _ in range(args.steps):
            graph.replay()
        e1.record()
        torch.cuda.nvtx.range_pop()
        launches = per_step * args.steps
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        eager_ms = e0.elapsed_time(e1) / args.steps
        gu = torch.empty(E, Mmax, 2 * I, dtype=torch.bfloat16, device=dev)
        if w4:
            g1 = lambda: wq.grouped_gemm_w4a8_masked(a, sa, mmd, weights[0], weights[1], out=gu,
                                                     status=st)
        else:
            g1 = lambda: wq.grouped_gemm_w8a8_masked(a, sa, mmd, weights[0], weights[1], cfg.scheme,
                                                     cfg.acc, out=gu, status=st)
        for _ in range(args.warmup):
            g1()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            g1()
        e1.record()
        torch.cuda.synchronize()
        g1_ms = e0.elapsed_time(e1) / args.steps
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    clocks = clk.summary()
    rows = int(mm.sum())
    ops = 2.0 * rows * 3 * H * I
    peaks, src = load_peaks()
    touched = int((mm > 0).sum())
    wb = 0.5 if w4 else 1.0  # bytes per weight code
    roofline = gemm_roofline(peaks, src, clocks, g1_ms, rows, touched, 2 * I, H, cfg.scheme, 1,
                             None if w4 else measured_traffic(cfg.name),
                             ("grouped_gemm_w4a8_masked" if w4 else "grouped_gemm_w8a8_masked")
                             + " gate_up (GEMM1)", weight_bytes=wb)
    # minimal bytes: touched experts' weights and scales, valid rows' codes and
    # scales in, bf16 outputs of the valid rows
    nbytes = int(touched * (3 * H * I * wb + (2 * I + H) * 4) + rows * (H + 4) + rows * H * 2)
    line = {"metric": METRIC, "value": ops / (ms / 1e3) / 1e12, "unit": "TOPS", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int4 x int8" if w4 else "int8",
            "data": "synthetic",
            "config": {"workload": f"masked-layout {'W4A8 (int4 weights)' if w4 else 'W8A8'} grouped "
                                   f"FFN: {E} local experts x {Mmax} rows, "
                                   f"hidden {H}, intermediate {I}, valid rows Zipf(1.2) = {rows}",
                       "parallelism": "single"},
            "tokens_per_s": rows / (ms / 1e3), "launch": "cuda_graph", "eager_ms_per_step": eager_ms,
            "gemm1_ms": g1_ms, "gpu_launches": launches,
            "roofline": roofline,
            "layer_roofline": layer_roofline(peaks, clocks, ms, ops, nbytes),
            "clocks": clocks}
    print(json.dumps(line), flush=True)


# dense W8A8 linear workloads ("Norm Linear"): (tokens, K, N) of DeepSeek-V3's
# dense-MLP gate_up projection (hidden 7168 -> 2 x 18432) at prefill
LINEAR = {"linear": (8192, 7168, 36864)}


def run_linear(args, name):
    """The dense W8A8 linear: quantize x per token, INT8 GEMM with its
    dequantization (wq_linear_w8a8).  One step = one call."""
    from w8a8_int8_quantized_token_gb300 import binding as wq
    from w8a8_int8_quantized_token_gb300 import build_lib
    T, K, N = LINEAR[name]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build_lib.build()
    wq.init(0)
    g = torch.Generator(device=dev).manual_seed(0)
    x = torch.randn(T, K, generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    Wq, sw = wq.quantize_weight(w, "channel")
    del w
    out = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
    ws = wq.linear_workspace(T, K, N, "channel", dev)
    st = wq.new_status(dev)
    step = lambda xx: wq.linear_w8a8(xx, Wq, sw, "channel", "i32", out=out, ws=ws, status=st)
    for _ in range(args.warmup):
        step(x)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        n0 = wq.lib().wq_kernel_launches()
        e0.record()
        for _ in range(args.steps):
            step(x)
        e1.record()
        launches = wq.lib().wq_kernel_launches() - n0
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    # end to end: the input from pinned host memory, the output back
    xh = x.cpu().pin_memory()
    outh = torch.empty(T, N, dtype=torch.bfloat16, pin_memory=True)
    xd = torch.empty_like(x)
    for _ in range(args.warmup):
        xd.copy_(xh, non_blocking=True); step(xd); outh.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(args.steps):
        xd.copy_(xh, non_blocking=True); step(xd); outh.copy_(out, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    flops = 2.0 * T * N * K
    peaks, src = load_peaks()
    clocks = clk.summary()
    tf, which = tensor_peak(peaks, clocks)
    ach = flops / (ms / 1e3) / 1e12
    line = {"metric": METRIC, "value": ach, "unit": "TOPS", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8", "data": "synthetic",
            "config": {"workload": f"dense W8A8 INT8 linear (DeepSeek-V3 dense-MLP gate_up shape), "
                                   f"channel-wise, int32 accumulator: {T} tokens, K {K}, N {N}",
                       "l2": "inputs larger than L2 (264 MB of int8 weights, 117 MB of "
                             "activations, 604 MB of output per step)",
                       "parallelism": "single"},
            "gpu_launches": launches,
            "roofline": {"bound": "tensor", "kernel": "wq_linear_w8a8 (quantize + INT8 GEMM)",
                         "achieved": ach, "peak": tf, "unit": "TFLOP/s", "frac": ach / tf,
                         "traffic": None, "flops": flops,
                         "peak_source": f"{src} bf16 dense, {which} (fp16 tcgen05 kind::f16)"},
            "e2e": {"value": flops / (e2e_ms / 1e3) / 1e12, "unit": "TOPS",
                    "h2d_bytes_per_step": T * K * 2, "d2h_bytes_per_step": T * N * 2,
                    "ms_per_step": e2e_ms},
            "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def run_convert(args):
    """Offline FP8 -> BF16 -> INT8 conversion of all 256 experts' weights of
    the DeepSeek-V3 MoE layer (W13 [256*4096, 7168] and W2 [256*7168, 2048]
    stacked, FP8 e4m3 with [128,128] block scales) to channel-wise INT8.  One
    step = both conversions.  HBM bound: each weight byte is read once (FP8)
    and written once (INT8)."""
    from w8a8_int8_quantized_token_gb300 import binding as wq
    from w8a8_int8_quantized_token_gb300 import build_lib
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build_lib.build()
    wq.init(0)
    E, H, I = 256, 7168, 2048
    mats = []
    for (N, K) in ((2 * I, H), (H, I)):
        w8 = torch.empty(E * N, K, dtype=torch.uint8, device=dev)
        s8 = torch.empty(E * N // 128, K // 128, dtype=torch.float32, device=dev)
        for e in range(E):
            a, b = synth.fp8_block_weights(N, K, seed=1_000 + e + (0 if K == H else E), device=dev)
            w8[e * N:(e + 1) * N] = a
            s8[e * N // 128:(e + 1) * N // 128] = b
        q = torch.empty(E * N, K, dtype=torch.int8, device=dev)
        s = torch.empty(E * N, dtype=torch.float32, device=dev)
        mats.append((w8, s8, q, s))
    torch.cuda.synchronize()

    def step():
        for w8, s8, q, s in mats:
            wq.convert_fp8_weights(w8, s8, "channel", q_out=q, s_out=s)
    for _ in range(args.warmup):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        n0 = wq.lib().wq_kernel_launches()
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        launches = wq.lib().wq_kernel_launches() - n0
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    nbytes = sum(w8.numel() + s8.numel() * 4 + q.numel() + s.numel() * 4 for w8, s8, q, s in mats)
    gbs = nbytes / (ms / 1e3) / 1e9
    peaks, src = load_peaks()
    line = {"metric": "FP8 -> BF16 -> INT8 weight conversion throughput", "value": gbs,
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8->int8", "data": "synthetic",
            "config": {"workload": "DeepSeek-V3 MoE layer weights, 256 experts (W13 + W2, 11.3 G "
                                   "weights), FP8 e4m3 with [128,128] scales -> channel-wise INT8",
                       "l2": "inputs larger than L2 (11.3 GB read, 11.3 GB written per step)",
                       "parallelism": "single"},
            "gpu_launches": launches,
            "roofline": {"bound": "hbm", "kernel": "convert_fp8_row_kernel", "achieved": gbs,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "traffic": None, "algorithmic_bytes": nbytes,
                         "peak_source": f"{src} HBM copy bandwidth"},
            "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def one_gpu_only(args):
    """Refuse a multi-GPU launch of our arm before the library is loaded: the
    pair GEMM engines' token loads are TMA multicasts between the two CTAs of
    a cluster, kept to one-GPU runs."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1 or args.gpus > 1:
        print(f"bench.py: refused: {max(world, args.gpus)} GPUs requested; this build runs the "
              f"layer on one GPU only (its GEMM engines use TMA multicast within a cluster, "
              f"which it keeps to one-GPU runs)", file=sys.stderr, flush=True)
        sys.exit(2)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="prefill",
                    choices=list(synth.CONFIGS) + list(LINEAR) + ["convert", "masked_w4a8"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0, help="override the token count (profiling)")
    ap.add_argument("--experts", type=int, default=0, help="override the expert count (profiling)")
    args = ap.parse_args()
    cfg = synth.CONFIGS.get(args.config)
    if cfg is not None and (args.tokens or args.experts):
        import dataclasses
        cfg = dataclasses.replace(cfg, name=cfg.name + "-reduced", T=args.tokens or cfg.T,
                                  E=args.experts or cfg.E)
    if args.impl == "reference":
        if cfg is None:
            print(json.dumps({"impl": "reference", "unavailable": "the CPU oracle arm covers the "
                              "MoE layer configurations only"}), flush=True)
            return
        run_reference(args, cfg)
        return
    one_gpu_only(args)
    if args.config in LINEAR:
        run_linear(args, args.config)
        return
    if args.config == "convert":
        run_convert(args)
        return
    if args.config == "masked_w4a8":
        run_masked(args, synth.CONFIGS["masked"], w4=True)
        return
    if cfg.masked:
        run_masked(args, cfg)
        return
    run_layer(args, cfg)


def run_layer(args, cfg):
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from w8a8_int8_quantized_token_gb300 import binding as wq
    from w8a8_int8_quantized_token_gb300 import build_lib
    build_lib.build()
    wq.init(0)

    weights = make_weights(wq, cfg, dev)
    x, logits = synth.layer_inputs(cfg, device=dev)
    layer = Layer(wq, cfg, dev, weights)
    fws = wq.forward_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.scheme, dev)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
    fst = wq.new_status(dev)
    fwd = lambda: wq.moe_forward(x, logits, *weights, cfg.k, cfg.scheme, cfg.acc, out=out, ws=fws,
                                 status=fst)

    # the staged calls reproduce the one-call layer exactly
    ref = fwd().clone()
    got = layer.step(x, logits)
    torch.cuda.synchronize()
    if not torch.equal(ref.view(torch.int16), got.view(torch.int16)):
        raise RuntimeError("staged step differs from wq_moe_forward")

    for _ in range(args.warmup):
        fwd()
        layer.step(x, logits)
    # the one-call layer recorded once into a CUDA graph, outside the timed
    # region; each timed step replays every one of its kernels
    graph, per_step = capture_graph(wq, fwd, dev)
    for _ in range(args.warmup):
        graph.replay()
    nst = len(layer.stages)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    with ClockSampler(0) as clk:
        # timed region 1: the one-call layer, K steps (the headline value)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("timed")
        start.record()
        for _ in range(args.steps):
            graph.replay()
        end.record()
        launches = per_step * args.steps
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        total_ms = start.elapsed_time(end)
        # the same steps launched one call at a time (reported beside it)
        start.record()
        for _ in range(args.steps):
            fwd()
        end.record()
        torch.cuda.synchronize()
        eager_ms = start.elapsed_time(end) / args.steps
        # timed region 2: the same steps as separate calls, events between stages
        torch.cuda.nvtx.range_push("staged")
        start.record()
        for i in range(args.steps):
            layer.step(x, logits, evs[i])
        end.record()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        staged_ms = start.elapsed_time(end) / args.steps
    stage_ms = {s: float(np.mean([evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)]))
                for j, s in enumerate(layer.stages)}
    fused = layer.time_fused(args.steps) if cfg.scheme == "block" and layer.f16 else None
    for st in (layer.status, fst):
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
    if not torch.equal(out.view(torch.int16), ref.view(torch.int16)):
        raise RuntimeError("timed steps changed the layer output")
    clocks = clk.summary()

    ms = total_ms / args.steps
    ops = layer_ops(cfg.T, cfg.H, cfg.I, cfg.k)
    tops = ops / (ms / 1e3) / 1e12
    tok_s = cfg.T / (ms / 1e3)

    # end to end: host activations in, host output back, through the one-call API
    xh, lh = x.cpu().pin_memory(), logits.cpu().pin_memory()
    outh = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, pin_memory=True)
    hws = wq.forward_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.scheme, dev, host=True)
    for _ in range(args.warmup):
        wq.moe_forward_host(xh, lh, *weights, cfg.k, cfg.scheme, cfg.acc, out_host=outh, ws=hws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        wq.moe_forward_host(xh, lh, *weights, cfg.k, cfg.scheme, cfg.acc, out_host=outh, ws=hws)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    if not torch.equal(outh.view(torch.int16), ref.cpu().view(torch.int16)):
        raise RuntimeError("host-buffer layer differs from the device one")

    peaks, src = load_peaks()
    touched = int((layer.counts > 0).sum().item())
    cb = 2 if layer.f16 else 1
    R = cfg.T * cfg.k
    roofline = gemm_roofline(peaks, src, clocks, stage_ms["gemm1"], R, touched, 2 * cfg.I, cfg.H,
                             cfg.scheme, cb, measured_traffic(cfg.name),
                             "grouped_gemm_w8a8 gate_up (GEMM1)")
    roof2 = gemm_roofline(peaks, src, clocks, stage_ms["gemm2"], R, touched, cfg.H, cfg.I,
                          cfg.scheme, cb, None, "grouped_gemm_w8a8 down (GEMM2)")
    nbytes = layer_bytes(cfg.T, cfg.H, cfg.I, touched, cfg.k, cfg.scheme, cfg.E)
    line = {"metric": METRIC, "value": tops, "unit": "TOPS", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8", "data": "synthetic",
            "config": {"workload": workload_name(cfg), "tokens": cfg.T, "hidden": cfg.H,
                       "intermediate": cfg.I, "experts": cfg.E, "top_k": cfg.k,
                       "scheme": cfg.scheme, "accumulator": cfg.acc,
                       "l2": "inputs larger than L2: 11.3 GB of int8 weights and ~2 GB of "
                             "activations are streamed every step",
                       "parallelism": "single"},
            "tokens_per_s": tok_s, "launch": "cuda_graph", "eager_ms_per_step": eager_ms,
            "stages_ms": stage_ms, "staged_ms_per_step": staged_ms,
            "fused_gemm1_silu_quant": fused,
            "gpu_launches": launches,
            "roofline": roofline,
            "roofline_gemm2": roof2,
            "layer_roofline": layer_roofline(peaks, clocks, ms, ops, nbytes),
            "e2e": {"value": ops / (e2e_ms / 1e3) / 1e12, "unit": "TOPS",
                    "h2d_bytes_per_step": cfg.T * cfg.H * 2 + cfg.T * cfg.E * 4,
                    "d2h_bytes_per_step": cfg.T * cfg.H * 2, "ms_per_step": e2e_ms},
            "clocks": clocks}
    if not args.no_cpu_baseline:
        run, sops, cores = oracle_sample(cfg, args.cpu_tokens, dev)
        # the same sample again and again until at least 10 s of CPU work
        reps, dt = 0, 0.0
        while reps == 0 or dt < 10.0:
            dt += run()
            reps += 1
        line["cpu_baseline"] = {"value": reps * sops / dt / 1e12, "unit": "TOPS", "cores": cores,
                                "kind": "oracle", "tokens_per_s": reps * args.cpu_tokens / dt,
                                "sample": f"first {args.cpu_tokens} of {cfg.T} tokens of the same "
                                          f"workload, full layer, run {reps} times ({dt:.1f} s)"}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
