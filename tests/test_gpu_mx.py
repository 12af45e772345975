"""Parity of the MXFP8 expert path (E4M3 codes with one E8M0 scale per block of
32 elements along the contraction axis) against the oracle, through the C ABI.

Bars: the block quantization (codes and scale bytes) is bit-exact, since every
code is decided in fp32 on both sides by the same exact power-of-two scaling
and the same rounding rule; routing is bit-exact as in the bf16 layer. The
stored h (bf16 values of MXFP8 codes) is decided from the GPU's own fp32 h,
whose sums run in another order than the oracle's: it equals the oracle's at
all but a few positions (a code or a block scale on the other side of a
rounding boundary), and there by at most one E4M3 step (a quarter of the
value). Decode-sized batches run the E4M3-MMA kernels, which store h as MXFP8
codes with scale rows; the check reads their values. y is held to the layer's bound max|gpu - oracle| <= 2e-2 rms and
rel-L2 <= 5e-3 (fp32 output); the bf16 y is that fp32 y rounded to nearest.
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


def _extreme_rows(rows, cols, dtype, seed):
    """Rows whose 32-element blocks span 2^-60..2^60 in magnitude, with zero
    blocks, negative zeros, subnormal-range values and saturating maxima."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    mag = torch.exp2(torch.randint(-60, 61, (rows, cols // 32, 1), device=DEV, generator=g).float())
    v = torch.randn(rows, cols // 32, 32, device=DEV, generator=g) * mag
    v[0, 0] = 0.0
    v[0, 1] = -0.0
    v[1, 0, 0] = 3.75      # with 1.0 below: e = -7, 3.75 -> 448 * 2^-7
    v[1, 0, 1:] = 1.0
    v[2, 0, :4] = torch.tensor([1e-30, -1e-38, 1.0, -2e-40], device=DEV)
    return v.reshape(rows, cols).to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("cols", [64, 544, 4096])
def test_quantize_mx_bitexact(oracle, dtype, cols):
    rows = 200
    src = _extreme_rows(rows, cols, dtype, seed=cols)
    sk = m.mx_scale_cols(cols)
    q = torch.empty(rows, cols, dtype=torch.uint8, device=DEV)
    sc = torch.full((rows, sk), 0xAB, dtype=torch.uint8, device=DEV)
    m.quantize_mx(src, q, sc)
    torch.cuda.synchronize()
    rq, rs = oracle.quantize_mx(to_np(src))
    np.testing.assert_array_equal(sc.cpu().numpy(), rs)  # padding bytes are zero too
    np.testing.assert_array_equal(q.cpu().numpy(), rq)


CASES = [
    MoEConfig("mx_decode", T=64, H=512, E=32, k=8, I=256),
    MoEConfig("mx_prefill_shared", T=600, H=256, E=8, k=2, I=256, I_shared=128),
    MoEConfig("mx_zipf", T=300, H=384, E=64, k=6, I=128, zipf_s=1.1),
    MoEConfig("mx_t1", T=1, H=128, E=4, k=4, I=128, renorm=0),
    MoEConfig("mx_wide_shared", T=48, H=1024, E=16, k=4, I=640, I_shared=256),
    MoEConfig("mx_e256", T=64, H=256, E=256, k=8, I=128),
    # experts averaging 256 rows or more: 256-token tiles with K = 64 stages,
    # ragged tails, a shared expert, and a skewed routing
    MoEConfig("mx_wide_tiles_shared", T=1100, H=384, E=8, k=2, I=384, I_shared=256),
    MoEConfig("mx_wide_tiles_zipf", T=1500, H=256, E=8, k=3, I=256, zipf_s=1.2),
]


def _layer_and_ref(oracle, cfg, tile=m.MOE_TILE_AUTO, n_group=1, topk_group=1, seed=0):
    d = generate(cfg, seed=seed, device=DEV)
    layer = m.MoELayerMX(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                         router_bias=d["router_bias"], Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"],
                         Ws_down=d["Ws_down"], renorm=cfg.renorm, tile=tile, n_group=n_group,
                         topk_group=topk_group)
    n = {kk: to_np(v) for kk, v in d.items()}
    ref, inter = oracle.forward_mx(n["x"], n["W_router"], n["router_bias"], n["W_gate"],
                                   n["W_up"], n["W_down"], cfg.k, cfg.renorm, n["Ws_gate"],
                                   n["Ws_up"], n["Ws_down"], n_group, topk_group,
                                   want_intermediates=True)
    return d, n, layer, ref, inter


def stored_h(oracle, ws, off, scales_off, rows, cols):
    """The layer's stored h as values: MXFP8 codes with scale rows (decode-sized
    kernels), else bf16 values."""
    if scales_off >= 0:
        sk = m.mx_scale_cols(cols)
        q = ws[off:off + rows * cols].view(rows, cols).cpu().numpy()
        sc = ws[scales_off:scales_off + rows * sk].view(rows, sk).cpu().numpy()
        return oracle.dequantize_mx(q, sc)
    return ws[off:off + rows * cols * 2].view(torch.bfloat16).view(rows, cols).float().cpu().numpy()


def assert_mx_h(h_gpu, h_ref, what):
    """Equal but at a few positions, and there within one E4M3 step."""
    h_gpu = np.asarray(h_gpu, np.float64)
    h_ref = np.asarray(h_ref, np.float64)
    bad = h_gpu != h_ref
    assert bad.mean() <= 1e-3, (what, bad.mean())
    if bad.any():
        d = np.abs(h_gpu - h_ref)[bad]
        assert (d <= 0.26 * np.abs(h_ref)[bad] + 1e-30).all(), (what, d.max())


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_forward_mx_vs_oracle(oracle, cfg):
    d, n, layer, ref, inter = _layer_and_ref(oracle, cfg)
    # The layer's weights: bit-exact block quantization of the bf16 matrices.
    for (q, s), name, cols in ((layer.gate, "W_gate", cfg.H), (layer.up, "W_up", cfg.H),
                               (layer.down, "W_down", cfg.I)):
        rq, rs = oracle.quantize_mx(n[name])
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
    assert_mx_h(stored_h(oracle, ws, lay["h"], lay["h_scales"], T * k, I), inter["h"], "h")
    if cfg.I_shared:
        hs = stored_h(oracle, ws, lay["h_shared"], lay["h_shared_scales"], T, cfg.I_shared)
        assert_mx_h(hs, inter["hs"], "h_shared")
    assert_close(y32.cpu().numpy(), ref, "y")
    assert_bf16_is_rounded(y, y32)
    # a second call repeats the result bit for bit
    y2 = layer(d["x"], out_f32=True)
    finish(ws)
    assert torch.equal(y2.view(torch.int32), y32.view(torch.int32))


@pytest.mark.parametrize("tile", [m.MOE_TILE_DECODE, m.MOE_TILE_AUTO], ids=["t32", "t128"])
def test_forward_mx_tiles_and_groups(oracle, tile):
    cfg = MoEConfig("mx_groups", T=200, H=256, E=32, k=4, I=256, I_shared=128)
    d, n, layer, ref, inter = _layer_and_ref(oracle, cfg, tile=tile, n_group=4, topk_group=2,
                                             seed=3)
    y32 = layer(d["x"], out_f32=True)
    finish(layer.workspace(cfg.T))
    assert_close(y32.cpu().numpy(), ref, "y")


def test_forward_mx_bounded_wait_reports_timeout_and_context_survives():
    cfg = MoEConfig("mx_timeout", T=40, H=256, E=8, k=2, I=128)
    d = generate(cfg, seed=3, device=DEV)
    layer = m.MoELayerMX(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k)
    ws = layer.workspace(cfg.T)
    before = layer(d["x"]).clone()
    finish(ws)
    pb = layer.problem(cfg.T, flags=m.MOE_FLAG_TEST_SKIP_SIGNAL, wait_limit_us=20000)
    y = torch.empty_like(before)
    m.forward_mx(pb, d["x"], layer.W_router, None, *layer.gate, *layer.up, *layer.down,
                 None, None, None, None, None, None, y, ws)
    torch.cuda.synchronize()  # returns: every wait gave up instead of hanging
    assert m.get_device_status(ws) == 5  # MOE_ERR_TIMEOUT
    after = layer(d["x"])
    finish(ws)
    assert torch.equal(after.view(torch.int16), before.view(torch.int16))


def test_forward_mx_rejects_bad_arguments():
    cfg = MoEConfig("mx_bad", T=8, H=128, E=4, k=2, I=192)  # I not a multiple of 128
    d = generate(cfg, seed=1, device=DEV)
    with pytest.raises(m.MoEError):
        m.MoELayerMX(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k)(d["x"])
