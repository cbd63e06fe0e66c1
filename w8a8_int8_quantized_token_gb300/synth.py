"""Seeded synthetic inputs for the W8A8 INT8 fused-MoE layer.

This module only draws random numbers.  It holds none of the layer's
arithmetic (no quantization, routing, GEMM, activation or combine), so both
the CUDA path and the CPU oracle can take their inputs from it without
sharing any of the method.

Recipe (the workloads of the DeepSeek-V3/R1-shaped layer that the sglang
pages "[Feature] DeepSeek V3/R1 INT8 Quantization (channel-wise)" and the
Meituan INT8 DeepSeek R1 article deploy; no dataset is used):

* activations ``x``: ``randn(T, H)`` float32; for the DeepSeek-shaped
  configurations 1% of the hidden channels (``round(0.01*H)`` columns chosen
  by ``randperm``) are multiplied by 20 to mimic outlier channels; then cast
  to bf16 (round to nearest even, torch's cast);
* router logits: ``randn(T, E)`` float32, kept in float32;
* weights, one expert at a time: ``(randn(N, K) * 0.02).to(bf16)`` for the
  gate_up matrix ``W13[e]`` (``N = 2*I`` rows, gate rows first) and then for
  the down matrix ``W2[e]`` (``N = H``, ``K = I``); every expert has its own
  generator seeded with ``seed * 1_000_003 + 1 + e`` so one expert can be
  regenerated alone (the full DeepSeek shape is 22.5 GB of bf16 weights,
  which is drawn on the device one expert at a time and never kept whole);
* masked layout: per-expert valid counts ``zipf(1.2)`` from
  ``numpy.random.default_rng(seed)``, capped at ``Mmax``.

Generators are torch's (CPU or CUDA Philox); the same seed on CPU and on the
GPU gives different numbers, so every consumer takes the tensors this module
returns rather than regenerating them elsewhere.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int            # tokens
    H: int            # hidden size (GEMM1 K, GEMM2 N)
    I: int            # moe intermediate size (GEMM1 N = 2*I, GEMM2 K)
    E: int            # routed experts
    k: int            # experts per token
    scheme: str       # "channel" | "block"
    acc: str          # "i32" | "f32"
    outliers: bool    # 1% outlier channels x20 in the activations
    seed: int = 0
    masked: bool = False
    Mmax: int = 0     # masked layout: rows per expert buffer

    @property
    def R(self) -> int:
        return self.T * self.k


CONFIGS = {
    # 16 tokens, hidden 256, intermediate 128, 8 experts, top-2
    "tiny": LayerConfig("tiny", 16, 256, 128, 8, 2, "channel", "i32", False),
    # DeepSeek-V3 shape, decode batch
    "decode": LayerConfig("decode", 128, 7168, 2048, 256, 8, "channel", "i32", True),
    # DeepSeek-V3 shape, prefill batch (int32 and fp32 accumulator)
    "prefill": LayerConfig("prefill", 8192, 7168, 2048, 256, 8, "channel", "i32", True),
    "prefill_f32": LayerConfig("prefill_f32", 8192, 7168, 2048, 256, 8, "channel", "f32", True),
    # DeepSeek-V3 shape, [128,128] block weights + per-token-group-128 acts
    "block": LayerConfig("block", 4096, 7168, 2048, 256, 8, "block", "f32", True),
    # expert-parallel-shaped masked layout: 32 local experts x 512 rows
    "masked": LayerConfig("masked", 0, 7168, 2048, 32, 1, "channel", "i32", True,
                          masked=True, Mmax=512),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def expert_seed(seed: int, e: int) -> int:
    return seed * 1_000_003 + 1 + e


def activations(T: int, H: int, outliers: bool, seed: int, device="cpu") -> torch.Tensor:
    """bf16 [T, H]: N(0,1) with optional 1% outlier channels x20."""
    g = _gen(device, seed)
    x = torch.randn(T, H, generator=g, device=device, dtype=torch.float32)
    if outliers and H > 0:
        n_out = int(round(0.01 * H))
        oc = torch.randperm(H, generator=g, device=device)[:n_out]
        x[:, oc] *= 20.0
    return x.to(torch.bfloat16)


def router_logits(T: int, E: int, seed: int, device="cpu") -> torch.Tensor:
    """float32 [T, E] N(0,1) router logits (own stream: seed + 7)."""
    g = _gen(device, seed + 7)
    return torch.randn(T, E, generator=g, device=device, dtype=torch.float32)


def expert_weights(cfg: LayerConfig, e: int, device="cpu"):
    """(W13[e] bf16 [2I, H], W2[e] bf16 [H, I]) drawn N(0, 0.02)."""
    g = _gen(device, expert_seed(cfg.seed, e))
    w13 = (torch.randn(2 * cfg.I, cfg.H, generator=g, device=device) * 0.02).to(torch.bfloat16)
    w2 = (torch.randn(cfg.H, cfg.I, generator=g, device=device) * 0.02).to(torch.bfloat16)
    return w13, w2


def masked_counts(E: int, Mmax: int, seed: int) -> np.ndarray:
    """int32 [E] valid rows per expert buffer, Zipf(s=1.2) capped at Mmax."""
    rng = np.random.default_rng(seed)
    return rng.zipf(1.2, E).clip(max=Mmax).astype(np.int32)


def layer_inputs(cfg: LayerConfig, device="cpu"):
    """Activations and router logits of one layer step (weights separate)."""
    x = activations(cfg.T, cfg.H, cfg.outliers, cfg.seed, device)
    logits = router_logits(cfg.T, cfg.E, cfg.seed, device)
    return x, logits


def masked_inputs(cfg: LayerConfig, device="cpu"):
    """bf16 activations [E, Mmax, H] (rows past the count are drawn too) and counts."""
    x = activations(cfg.E * cfg.Mmax, cfg.H, cfg.outliers, cfg.seed, device)
    return x.view(cfg.E, cfg.Mmax, cfg.H), masked_counts(cfg.E, cfg.Mmax, cfg.seed)


def small_config(name: str = "small", T=40, H=384, I=256, E=6, k=3, scheme="channel",
                 acc="i32", outliers=True, seed=1) -> LayerConfig:
    """A parity-test shape that spans several 128-row/128-col tiles with ragged tails."""
    return LayerConfig(name, T, H, I, E, k, scheme, acc, outliers, seed)


def fp8_block_weights(N: int, K: int, seed: int, device="cpu"):
    """Weights in the FP8 release format DeepSeek-V3/R1 ships: bf16 N(0, 0.02)
    draws, one float32 scale per [128, 128] block (block absmax / 448, the
    e4m3 maximum) and the e4m3 bytes of weight / scale (torch's float8 cast).
    Returns (uint8 bytes [N, K], float32 scales [N/128, K/128])."""
    g = _gen(device, seed)
    w = (torch.randn(N, K, generator=g, device=device) * 0.02).to(torch.bfloat16).float()
    blocks = w.view(N // 128, 128, K // 128, 128)
    s8 = blocks.abs().amax(dim=(1, 3)) / 448.0
    s8 = torch.where(s8 > 0, s8, torch.ones_like(s8))
    q = (blocks / s8[:, None, :, None]).view(N, K).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), s8.contiguous()

