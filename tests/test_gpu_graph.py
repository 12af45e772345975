"""moe_forward inside a CUDA graph.

The DeepSeek page's CUDA-Graph paragraph ("Lower latency and higher throughput
with multi-node DeepSeek deployment") asks that a captured MoE layer read its
per-expert counts on the device rather than bake in the buffer bounds. Here one
forward pass is captured and replayed: the replay must equal eager calls bit for
bit, and after new tokens are written into the captured input buffer (so routing,
counts and offsets all change) the replay must follow them.
"""
import pytest
import torch

import mixture_experts_layer_route_gb300 as m
from moe_inputs import MoEConfig, generate

DEV = "cuda:0"

CASES = [
    MoEConfig("graph_decode", T=64, H=512, E=32, k=8, I=256),
    MoEConfig("graph_prefill", T=640, H=512, E=16, k=4, I=256, I_shared=128),
]


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_forward_replays_in_cuda_graph(cfg):
    d = generate(cfg, seed=5, device=DEV)
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                       router_bias=d["router_bias"], Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"],
                       Ws_down=d["Ws_down"])
    x_static = d["x"].clone()
    y_static = torch.empty(cfg.T, cfg.H, dtype=cfg.torch_dtype, device=DEV)
    # Eager warm-up on a side stream creates the workspace and caches the
    # library's per-device kernel attributes before capture.
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ref1 = layer(x_static).clone()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x_static, out=y_static)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y_static, ref1)

    # New tokens in the captured buffer: routing and expert loads change.
    x2 = generate(cfg.replace(T=cfg.T), seed=6, device=DEV)["x"]
    x_static.copy_(x2)
    g.replay()
    torch.cuda.synchronize()
    ref2 = layer(x2)
    torch.cuda.synchronize()
    assert not torch.equal(ref1, ref2)
    assert torch.equal(y_static, ref2)
    assert m.get_device_status(layer.workspace(cfg.T)) == m.MOE_OK
