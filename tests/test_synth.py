"""The seeded synthetic inputs (no GPU): shapes, dtypes and distributions of
the recipe the design states, the per-expert weight streams, the masked
counts at seed 0, and the configurations' sizes."""
import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
from w8a8_int8_quantized_token_gb300 import synth  # noqa: E402


def test_activations_with_outlier_channels():
    T, H = 4096, 1000
    x = synth.activations(T, H, True, seed=3)
    assert x.dtype == torch.bfloat16 and x.shape == (T, H)
    std = x.float().std(dim=0)
    big = (std > 5).nonzero().flatten()
    assert len(big) == round(0.01 * H)  # 1% of the channels
    assert torch.allclose(std[big], torch.full_like(std[big], 20.0), rtol=0.1)
    rest = torch.ones(H, dtype=torch.bool)
    rest[big] = False
    assert abs(float(std[rest].mean()) - 1.0) < 0.02 and abs(float(x.float()[:, rest].mean())) < 0.01
    assert torch.equal(x.view(torch.int16), synth.activations(T, H, True, seed=3).view(torch.int16))
    y = synth.activations(T, H, False, seed=3).float()
    assert float(y.std(dim=0).max()) < 1.2  # no outliers when not asked


def test_router_logits_are_float32_normal_on_their_own_stream():
    lg = synth.router_logits(2048, 64, seed=0)
    assert lg.dtype == torch.float32 and lg.shape == (2048, 64)
    assert abs(float(lg.mean())) < 0.02 and abs(float(lg.std()) - 1.0) < 0.02
    x = synth.activations(2048, 64, False, seed=0).float()
    assert not torch.equal(lg, x)  # not the activations' draws


def test_expert_weights_regenerate_alone():
    cfg = synth.small_config(H=256, I=128, E=4)
    w13, w2 = synth.expert_weights(cfg, 2)
    assert w13.shape == (2 * cfg.I, cfg.H) and w2.shape == (cfg.H, cfg.I)
    assert w13.dtype == torch.bfloat16 and w2.dtype == torch.bfloat16
    both = torch.cat([w13.float().flatten(), w2.float().flatten()])
    assert abs(float(both.std()) - 0.02) < 0.001
    again13, again2 = synth.expert_weights(cfg, 2)  # no other expert drawn first
    assert torch.equal(w13.view(torch.int16), again13.view(torch.int16))
    assert torch.equal(w2.view(torch.int16), again2.view(torch.int16))
    other13, _ = synth.expert_weights(cfg, 3)
    assert not torch.equal(w13, other13)


def test_masked_counts_at_seed_zero():
    c = synth.masked_counts(32, 512, 0)
    assert c.dtype == np.int32 and c.shape == (32,)
    assert int(c.sum()) == 5791 and int((c == 512).sum()) == 9
    assert int(c.min()) >= 1 and int(c.max()) <= 512


@pytest.mark.parametrize("name,shape", [
    ("tiny", (16, 256, 128, 8, 2, "channel", "i32")),
    ("decode", (128, 7168, 2048, 256, 8, "channel", "i32")),
    ("prefill", (8192, 7168, 2048, 256, 8, "channel", "i32")),
    ("prefill_f32", (8192, 7168, 2048, 256, 8, "channel", "f32")),
    ("block", (4096, 7168, 2048, 256, 8, "block", "f32")),
])
def test_configurations(name, shape):
    c = synth.CONFIGS[name]
    assert (c.T, c.H, c.I, c.E, c.k, c.scheme, c.acc) == shape
    assert c.R == c.T * c.k


def test_masked_configuration():
    c = synth.CONFIGS["masked"]
    assert c.masked and (c.E, c.Mmax, c.H, c.I) == (32, 512, 7168, 2048)
