"""The layer recorded into a CUDA graph and replayed.

Every call of the boundary is asynchronous on the caller's stream, with no
host synchronisation and no host read of device-side counts.  So a captured
step replays the same results as eager calls, bit for bit, on whatever the
input buffers hold at replay time: new activations, new routing, new masked
counts.  The masked layer's small-token engine runs on a second stream,
forked and joined through events inside the capture.
"""
import numpy as np
import pytest
import torch

from w8a8_int8_quantized_token_gb300 import binding as wq
from w8a8_int8_quantized_token_gb300 import synth
from wq_testutil import quantized_weights

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _init():
    from w8a8_int8_quantized_token_gb300 import build_lib
    build_lib.build()
    wq.init(0)


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("cfg", [
    # fp16 codes, K >= 1024: the tensor-memory-weights pair engine
    synth.small_config("graph_pair", T=300, H=1024, I=256, E=4, k=2),
    # block scheme on the block-wise pair engine
    synth.small_config("graph_block", T=300, H=512, I=256, E=4, k=2, scheme="block", acc="f32"),
    # few rows per expert: the small-token and int8-code engines
    synth.small_config("graph_int8", T=40, H=384, I=256, E=6, k=3),
], ids=lambda c: c.name)
def test_layer_graph_replay(cfg):
    (W13, S13, W2, S2), _ = quantized_weights(cfg, DEV)
    x0, lg0 = synth.layer_inputs(cfg)
    x, lg = x0.to(DEV), lg0.to(DEV)
    ws = wq.forward_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.scheme, DEV)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=DEV)
    st = wq.new_status()
    step = lambda: wq.moe_forward(x, lg, W13, S13, W2, S2, cfg.k, cfg.scheme, cfg.acc, out=out,
                                  ws=ws, status=st)
    step()  # eager warm-up (first-use setup happens outside the capture)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    # new inputs in the captured buffers, then replay
    x.copy_(synth.activations(cfg.T, cfg.H, True, 91).to(DEV))
    lg.copy_(synth.router_logits(cfg.T, cfg.E, 92).to(DEV))
    out.fill_(7.0)
    g.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want = wq.moe_forward(x.clone(), lg.clone(), W13, S13, W2, S2, cfg.k, cfg.scheme, cfg.acc)
    torch.cuda.synchronize()
    assert _same(out, want)


@pytest.mark.parametrize("w4", [False, True], ids=["int8_weights", "int4_weights"])
def test_masked_graph_replay(w4):
    """The masked layer (256-token tiles with experts of at most 16 rows: the
    small-token engine on the second stream beside the tensor-core engine),
    captured, then replayed on new counts and activations."""
    cfg = synth.small_config("graph_masked", T=0, H=256, I=128, E=4, k=1)
    E, Mmax, H, I = cfg.E, 300, cfg.H, cfg.I
    if w4:
        g_ = torch.Generator().manual_seed(17)
        W13 = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=DEV)
        W2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=DEV)
        S13 = torch.empty(E, 2 * I, device=DEV)
        S2 = torch.empty(E, H, device=DEV)
        for e in range(E):
            W13[e], S13[e] = wq.quantize_weight_int4(
                (torch.randn(2 * I, H, generator=g_) * 0.02).to(torch.bfloat16).to(DEV))
            W2[e], S2[e] = wq.quantize_weight_int4(
                (torch.randn(H, I, generator=g_) * 0.02).to(torch.bfloat16).to(DEV))
        fwd = wq.moe_forward_masked_w4a8
        ws = torch.empty(wq.lib().wq_moe_forward_masked_w4a8_workspace_size(E, Mmax, H, I),
                         dtype=torch.uint8, device=DEV)
        call = lambda a, sa, mm, y, ws_, st_: fwd(a, sa, mm, W13, S13, W2, S2, y=y, ws=ws_, status=st_)
    else:
        (W13, S13, W2, S2), _ = quantized_weights(cfg, DEV)
        ws = torch.empty(wq.lib().wq_moe_forward_masked_workspace_size(E, Mmax, H, I, 0),
                         dtype=torch.uint8, device=DEV)
        call = lambda a, sa, mm, y, ws_, st_: wq.moe_forward_masked(a, sa, mm, W13, S13, W2, S2,
                                                                    y=y, ws=ws_, status=st_)
    a, sa = wq.quantize_per_token(synth.activations(E * Mmax, H, True, 93).to(DEV))
    a, sa = a.view(E, Mmax, H).clone(), sa.view(E, Mmax).clone()
    mm = torch.tensor([300, 5, 0, 70], dtype=torch.int32, device=DEV)
    y = torch.empty(E, Mmax, H, dtype=torch.bfloat16, device=DEV)
    st = wq.new_status()
    call(a, sa, mm, y, ws, st)  # eager warm-up: creates the second stream outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(a, sa, mm, y, ws, st)
    a2, sa2 = wq.quantize_per_token(synth.activations(E * Mmax, H, True, 94).to(DEV))
    a.copy_(a2.view(E, Mmax, H))
    sa.copy_(sa2.view(E, Mmax))
    mm.copy_(torch.tensor([12, 256, 1, 300], dtype=torch.int32))
    y.fill_(7.0)
    g.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want = torch.full_like(y, 7.0)
    ws2 = torch.empty_like(ws)
    st2 = wq.new_status()
    call(a.clone(), sa.clone(), mm.clone(), want, ws2, st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    counts = mm.cpu().numpy()
    for e in range(E):
        assert _same(y[e, :counts[e]], want[e, :counts[e]])
        assert bool((y[e, counts[e]:] == 7.0).all())
