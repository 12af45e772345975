"""A seeded sweep of random small layers through moe_forward and
moe_forward_fp8 against the oracle.

Each case draws T, H, E, k, I, the shared expert, dtype, tile mode, renorm,
router skew and group-limited routing from a fixed generator, so the schedule's
corners (empty and single-row experts, odd feature-block counts that fall back
to single-CTA tiles, heavy/light interleaving ratios, multi-tile experts) are
crossed with every routing form. The oracle routes the logits the forward pass
stored (ids must then match bit for bit), and y is held to the layer bound.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_route_gb300 as m
from moe_inputs import MoEConfig, generate
from oracle import to_np
from test_gpu_parity import assert_close, finish

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _draw(i):
    r = np.random.default_rng(1000 + i)
    E = int(r.choice([4, 8, 12, 16, 32, 64, 96, 128]))
    k = int(r.integers(1, min(E, 10) + 1))
    fp8 = bool(r.random() < 0.3)
    dtype = "f32" if (not fp8 and r.random() < 0.2) else "bf16"
    I = int(r.choice([128, 256, 384] if fp8 else [64, 128, 192, 256, 320]))
    Is = int(r.choice([0, 0, 128, 256] if fp8 else [0, 0, 64, 128, 192]))
    T = int(r.choice([1, 7, 33, 64, 65, 130, 300, 513]))
    H = int(r.choice([128, 256, 384, 512]))
    groups = (1, 1)
    if E % 4 == 0 and r.random() < 0.3:
        ng = 4
        tk = int(r.integers(1, ng + 1))
        if k <= tk * (E // ng):
            groups = (ng, tk)
    return dict(T=T, H=H, E=E, k=k, I=I, I_shared=Is, dtype=dtype, fp8=fp8,
                tile=int(r.choice([m.MOE_TILE_AUTO, m.MOE_TILE_AUTO, m.MOE_TILE_DECODE,
                                   m.MOE_TILE_MEDIUM, m.MOE_TILE_PREFILL])),
                renorm=int(r.random() < 0.85), zipf=float(r.choice([0.0, 0.0, 1.1])),
                groups=groups)


CASES = [_draw(i) for i in range(24)]


@pytest.mark.parametrize("c", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_random_layer_vs_oracle(oracle, c):
    cfg = MoEConfig("sweep", T=c["T"], H=c["H"], E=c["E"], k=c["k"], I=c["I"],
                    I_shared=c["I_shared"], dtype=c["dtype"], renorm=c["renorm"],
                    zipf_s=c["zipf"])
    d = generate(cfg, seed=7, device=DEV, enforce_margin=False)
    kw = dict(router_bias=d["router_bias"], Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"],
              Ws_down=d["Ws_down"], renorm=cfg.renorm, tile=c["tile"], n_group=c["groups"][0],
              topk_group=c["groups"][1])
    cls = m.MoELayerFP8 if c["fp8"] else m.MoELayer
    layer = cls(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k, **kw)
    y32 = layer(d["x"], out_f32=True)
    ws = layer.workspace(cfg.T)
    finish(ws)
    T, E, k = cfg.T, cfg.E, cfg.k
    lay = m.workspace_layout(layer.problem(T))
    logits = ws[lay["logits"]:lay["logits"] + T * E * 4].view(torch.float32).view(T, E)
    gids = ws[lay["topk_ids"]:lay["topk_ids"] + T * k * 4].view(torch.int32).view(T, k)
    rid, rw = oracle.route_grouped(logits.cpu().numpy(), k, cfg.renorm, *c["groups"])
    np.testing.assert_array_equal(gids.cpu().numpy(), rid)
    n = {kk: to_np(v) for kk, v in d.items()}
    ffn = oracle.ffn_combine_fp8 if c["fp8"] else oracle.ffn_combine
    ref = ffn(n["x"], rid, rw, n["W_gate"], n["W_up"], n["W_down"], n["Ws_gate"], n["Ws_up"],
              n["Ws_down"])
    assert_close(y32.cpu().numpy(), ref, "y", tf32=cfg.dtype == "f32")
