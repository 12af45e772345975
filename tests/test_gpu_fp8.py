"""Parity of the FP8 expert path (E4M3 codes with one power-of-two scale per
row) against the oracle, through the C ABI.

Bars: the row quantization (codes and scales) is bit-exact, since a code is an
integer decided in fp32 on both sides by the same exact scaling and the same
rounding rule; routing is bit-exact as in the bf16 layer; y, computed by both
sides from the same quantized operands with fp32 (GPU) or fp64 (oracle)
accumulation, is held to the layer's bound max|gpu - oracle| <= 2e-2 rms and
rel-L2 <= 5e-3 (fp32 output); the bf16 y is that fp32 y rounded to nearest.
The intermediate h (bf16, before its own quantization) is held to the stage
bound of the bf16 tests against the oracle's h before rounding.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_route_gb300 as m
from moe_inputs import MoEConfig, generate
from oracle import to_np
from test_gpu_parity import assert_bf16_is_rounded, assert_close, finish

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_rows_bitexact(oracle, dtype):
    g = torch.Generator(device=DEV).manual_seed(7)
    rows, cols = 300, 1024
    mag = 10.0 ** (torch.rand(rows, 1, device=DEV, generator=g) * 12 - 6)
    src = (torch.randn(rows, cols, device=DEV, generator=g) * mag).to(dtype)
    src[5] = 0
    src[6] = 448.0
    src[7, 3] = -1.75 * 2.0 ** -3
    q = torch.empty(rows, cols, dtype=torch.uint8, device=DEV)
    sc = torch.empty(rows, dtype=torch.float32, device=DEV)
    m.quantize_rows_e4m3(src, q, sc)
    torch.cuda.synchronize()
    rq, rsc = oracle.quantize_rows_e4m3(to_np(src))
    np.testing.assert_array_equal(sc.cpu().numpy(), rsc)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)


CASES = [
    MoEConfig("fp8_decode", T=64, H=512, E=32, k=8, I=256),
    MoEConfig("fp8_prefill_shared", T=600, H=256, E=8, k=2, I=256, I_shared=128),
    MoEConfig("fp8_zipf", T=300, H=384, E=64, k=6, I=128, zipf_s=1.1),
    MoEConfig("fp8_t1", T=1, H=128, E=4, k=4, I=128, renorm=0),
]


def _layer_and_ref(oracle, cfg, tile=m.MOE_TILE_AUTO, n_group=1, topk_group=1, seed=0):
    d = generate(cfg, seed=seed, device=DEV)
    layer = m.MoELayerFP8(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                          router_bias=d["router_bias"], Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"],
                          Ws_down=d["Ws_down"], renorm=cfg.renorm, tile=tile, n_group=n_group,
                          topk_group=topk_group)
    n = {kk: to_np(v) for kk, v in d.items()}
    ref, inter = oracle.forward_fp8(n["x"], n["W_router"], n["router_bias"], n["W_gate"],
                                    n["W_up"], n["W_down"], cfg.k, cfg.renorm, n["Ws_gate"],
                                    n["Ws_up"], n["Ws_down"], n_group, topk_group,
                                    want_intermediates=True)
    return d, n, layer, ref, inter


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_forward_fp8_vs_oracle(oracle, cfg):
    d, n, layer, ref, inter = _layer_and_ref(oracle, cfg)
    # The layer's weights: bit-exact row quantization of the bf16 matrices.
    for (q, s), name in ((layer.gate, "W_gate"), (layer.up, "W_up"), (layer.down, "W_down")):
        rq, rs = oracle.quantize_rows_e4m3(n[name])
        np.testing.assert_array_equal(q.cpu().numpy(), rq)
        np.testing.assert_array_equal(s.cpu().numpy(), rs)
    y = layer(d["x"])
    y32 = layer(d["x"], out_f32=True)
    ws = layer.workspace(cfg.T)
    finish(ws)
    T, k, I = cfg.T, cfg.k, cfg.I
    lay = m.workspace_layout(layer.problem(T))
    gids = ws[lay["topk_ids"]:lay["topk_ids"] + T * k * 4].view(torch.int32).view(T, k)
    np.testing.assert_array_equal(gids.cpu().numpy(), inter["ids"])
    gw = ws[lay["topk_w"]:lay["topk_w"] + T * k * 4].view(torch.float32).view(T, k)
    np.testing.assert_allclose(gw.cpu().numpy(), inter["w"], rtol=0, atol=1e-6)
    h = ws[lay["h"]:lay["h"] + T * k * I * 2].view(torch.bfloat16).view(T * k, I)
    # the GPU's bf16 h against the oracle's h before its bf16 rounding
    assert_close(h.float().cpu().numpy(), inter["h_f32"], "h", stage=True)
    assert_close(y32.cpu().numpy(), ref, "y")
    assert_bf16_is_rounded(y, y32)


@pytest.mark.parametrize("tile", [m.MOE_TILE_DECODE, m.MOE_TILE_MEDIUM, m.MOE_TILE_PREFILL],
                         ids=["t32", "t128", "t256"])
def test_forward_fp8_tiles_and_groups(oracle, tile):
    cfg = MoEConfig("fp8_groups", T=200, H=256, E=32, k=4, I=256, I_shared=128)
    d, n, layer, ref, inter = _layer_and_ref(oracle, cfg, tile=tile, n_group=4, topk_group=2,
                                             seed=3)
    y32 = layer(d["x"], out_f32=True)
    finish(layer.workspace(cfg.T))
    assert_close(y32.cpu().numpy(), ref, "y")


def test_forward_fp8_rejects_bad_arguments():
    cfg = MoEConfig("fp8_bad", T=8, H=128, E=4, k=2, I=192)  # I not a multiple of 128
    d = generate(cfg, seed=1, device=DEV)
    with pytest.raises(m.MoEError):
        m.MoELayerFP8(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k)(d["x"])
