"""Shared helpers of the GPU tests: conversions between torch tensors and the
oracle's numpy formats, and quantized weights produced independently by the
CUDA library and by the oracle from the same seeded bf16 weights."""
import numpy as np
import torch

from oracle import wq_oracle as O
from w8a8_int8_quantized_token_gb300 import binding as wq
from w8a8_int8_quantized_token_gb300 import synth


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def np_(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def assert_bf16_equal(got_bits, want_bits, what="output"):
    g = O.bf16_to_f32(got_bits)
    w = O.bf16_to_f32(want_bits)
    bad = ~((g == w) | (np.isnan(g) & np.isnan(w)))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {g.size} differ, e.g. at {idx.tolist()}: "
                             f"got {g[bad][:5]} want {w[bad][:5]}")


def tolerance_report(got_bits, want_bits):
    g = O.bf16_to_f32(got_bits).astype(np.float64)
    w = O.bf16_to_f32(want_bits).astype(np.float64)
    max_abs = float(np.abs(g - w).max()) if g.size else 0.0
    rel_fro = float(np.linalg.norm(g - w) / max(np.linalg.norm(w), 1e-30))
    return max_abs, rel_fro


def quantized_weights(cfg, dev, experts=None):
    """GPU-quantized weights (the library's kernels) for all experts, and the
    oracle's own quantization of the same bf16 weights for ``experts``."""
    E, I, H = cfg.E, cfg.I, cfg.H
    blk = cfg.scheme == "block"
    W13 = torch.empty(E, 2 * I, H, dtype=torch.int8, device=dev)
    W2 = torch.empty(E, H, I, dtype=torch.int8, device=dev)
    if blk:
        S13 = torch.empty(E, 2 * I // 128, H // 128, dtype=torch.float32, device=dev)
        S2 = torch.empty(E, H // 128, I // 128, dtype=torch.float32, device=dev)
    else:
        S13 = torch.empty(E, 2 * I, dtype=torch.float32, device=dev)
        S2 = torch.empty(E, H, dtype=torch.float32, device=dev)
    oracle = {}
    for e in range(E):
        w13, w2 = synth.expert_weights(cfg, e)
        wq.quantize_weight(w13.to(dev), cfg.scheme, W13[e], S13[e])
        wq.quantize_weight(w2.to(dev), cfg.scheme, W2[e], S2[e])
        if experts is None or e in experts:
            oracle[e] = O.quantize_weights(bits(w13), bits(w2), cfg.scheme)
    return (W13, S13, W2, S2), oracle


def stack_oracle(oracle, E):
    return tuple(np.stack([oracle[e][i] for e in range(E)]) for i in range(4))
