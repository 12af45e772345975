"""Packed (tiled) expert weights: moe_pack_weights produces exactly the
documented tile layout, and a layer run on packed weights gives bit for bit the
output of the same layer on row-major weights (the GEMMs load the same shared-
memory blocks either way, so nothing about the arithmetic may change)."""
import pytest
import torch

import mixture_experts_layer_route_gb300 as m
from moe_inputs import MoEConfig, generate

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _tiles_reference(src):
    """The tile layout restated with torch views: tile (rb, kb) = rows
    64*rb..64*rb+63, 128-byte column piece kb, tiles in (rb, kb) order."""
    rows = src.numel() // src.shape[-1]
    b = src.reshape(rows, -1).view(torch.uint8)
    row_bytes = b.shape[1]
    return b.view(rows // 64, 64, row_bytes // 128, 128).permute(0, 2, 1, 3).contiguous()


@pytest.mark.parametrize("dtype,shape", [(torch.bfloat16, (3, 128, 256)),
                                         (torch.bfloat16, (2, 4096, 192)),
                                         (torch.float32, (2, 64, 96)),
                                         (torch.uint8, (5, 192, 384))])
def test_pack_layout(dtype, shape):
    g = torch.Generator(device=DEV).manual_seed(7)
    if dtype == torch.uint8:
        src = torch.randint(0, 256, shape, generator=g, device=DEV, dtype=torch.int32).to(torch.uint8)
    else:
        src = torch.randn(shape, generator=g, device=DEV, dtype=torch.float32).to(dtype)
    packed = m.pack_weights(src)
    torch.cuda.synchronize()
    ref = _tiles_reference(src)
    assert torch.equal(packed.view(torch.uint8).reshape(-1), ref.reshape(-1))


CASES = [
    ("decode", dict(T=64, H=512, E=16, k=4, I=256), m.MOE_TILE_AUTO),
    ("prefill_shared", dict(T=600, H=512, E=8, k=2, I=384, I_shared=256), m.MOE_TILE_AUTO),
    ("medium", dict(T=300, H=256, E=4, k=2, I=128), m.MOE_TILE_MEDIUM),
    ("decode_forced", dict(T=200, H=256, E=8, k=2, I=192, I_shared=64), m.MOE_TILE_DECODE),
    ("odd_blocks", dict(T=300, H=384, E=4, k=2, I=192), m.MOE_TILE_PREFILL),
    ("f32", dict(T=130, H=256, E=8, k=2, I=128, dtype="f32"), m.MOE_TILE_AUTO),
]


@pytest.mark.parametrize("name,shape,tile", CASES, ids=[c[0] for c in CASES])
def test_tiled_layer_bitwise_equals_row_major(name, shape, tile):
    cfg = MoEConfig(name, **shape)
    d = generate(cfg, seed=11, device=DEV, enforce_margin=False)
    kw = dict(Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"], Ws_down=d["Ws_down"], tile=tile)
    ys = []
    for tiled in (False, True):
        layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                           tiled=tiled, **kw)
        ys.append(layer(d["x"], out_f32=True))
        torch.cuda.synchronize()
        assert m.get_device_status(layer.workspace(cfg.T)) == m.MOE_OK
    assert torch.equal(ys[0], ys[1])


@pytest.mark.parametrize("shape", [dict(T=64, H=512, E=16, k=4, I=256),
                                   dict(T=520, H=512, E=8, k=2, I=256, I_shared=128)])
def test_tiled_fp8_layer_bitwise_equals_row_major(shape):
    cfg = MoEConfig("f8", **shape)
    d = generate(cfg, seed=12, device=DEV, enforce_margin=False)
    kw = dict(Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"], Ws_down=d["Ws_down"])
    ys = []
    for tiled in (False, True):
        layer = m.MoELayerFP8(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                              tiled=tiled, **kw)
        ys.append(layer(d["x"], out_f32=True))
        torch.cuda.synchronize()
        assert m.get_device_status(layer.workspace(cfg.T)) == m.MOE_OK
    assert torch.equal(ys[0], ys[1])
