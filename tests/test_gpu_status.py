"""Failure detection without a GPU fault: the grouped GEMM's producer is told
(a host-set test flag) to withhold its first load signal, so the MMA issuer's
bounded wait runs out after a short limit. The kernel must record
MOE_ERR_TIMEOUT in the workspace status word and return, leaving the context
usable: the next normal call succeeds and matches a run made before it."""
import pytest
import torch

import mixture_experts_layer_route_gb300 as m
from moe_inputs import MoEConfig, generate

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("tile", [m.MOE_TILE_DECODE, m.MOE_TILE_PREFILL])
def test_bounded_wait_reports_timeout_and_context_survives(tile):
    cfg = MoEConfig("s", T=96, H=256, E=8, k=2, I=128)
    d = generate(cfg, seed=3, device=DEV)
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k, tile=tile)
    ws = layer.workspace(cfg.T)
    before = layer(d["x"]).clone()
    torch.cuda.synchronize()
    assert m.get_device_status(ws) == m.MOE_OK

    pb = layer.problem(cfg.T, flags=m.MOE_FLAG_TEST_SKIP_SIGNAL, wait_limit_us=20000)
    y = torch.empty_like(before)
    m.forward(pb, d["x"], layer.W_router, None, layer.W_gate, layer.W_up, layer.W_down, None,
              None, None, y, ws)
    torch.cuda.synchronize()  # returns: the kernel gave up instead of hanging
    assert m.get_device_status(ws) == 5  # MOE_ERR_TIMEOUT

    after = layer(d["x"])  # moe_forward clears the status word when it starts
    torch.cuda.synchronize()
    assert m.get_device_status(ws) == m.MOE_OK
    assert torch.equal(after.view(torch.int16), before.view(torch.int16))


def test_sticky_status_and_reset():
    cfg = MoEConfig("s", T=32, H=128, E=4, k=2, I=64)
    ws = torch.zeros(m.workspace_size(m.make_problem(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I)),
                     dtype=torch.uint8, device=DEV)
    ws[:4].view(torch.int32).fill_(6)
    assert m.get_device_status(ws) == 6
    m.reset_device_status(ws)
    assert m.get_device_status(ws) == m.MOE_OK
