"""moe_forward_single_launch: the decode-sized layer as one cooperative
persistent kernel, against the CPU oracle through the C ABI.

Bars as in test_gpu_parity: the logits within fp32 summation-order error of the
oracle's; top-k ids bit-exact and gate weights within 1e-6 of the oracle's
routing of the kernel's own fp32 logits; offsets, gather_idx and slot_pos
bit-exact; y (out_f32) within max|d| <= 2e-2 rms and rel-L2 <= 5e-3 of the
oracle, and the bf16 output its round-to-nearest-even. Beyond the oracle: two
calls give identical bits, the result agrees with the kernel chain of
moe_forward within the same bound, problems outside the path's scope are
refused on the host, a bounded wait that runs out is reported in the status
word with the context left usable, and the launch replays in a CUDA graph.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_route_gb300 as m
from moe_inputs import CONFIGS, MoEConfig, generate
from oracle import to_np
from test_gpu_fullsize import covering_tokens, oracle_rows
from test_gpu_parity import assert_bf16_is_rounded, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    MoEConfig("one_token", T=1, H=256, E=8, k=2, I=128),
    MoEConfig("small_shared_bias", T=37, H=512, E=40, k=4, I=256, I_shared=128, zipf_s=1.1),
    MoEConfig("e512_k10", T=64, H=1024, E=512, k=10, I=256, zipf_s=1.1),
    MoEConfig("e1000_k32", T=16, H=256, E=1000, k=32, I=64),
    MoEConfig("f32", T=64, H=256, E=8, k=2, I=512, dtype="f32"),
    MoEConfig("renorm0", T=48, H=512, E=64, k=6, I=128, renorm=0),
    MoEConfig("shared_odd_T", T=23, H=384, E=16, k=3, I=192, I_shared=320),
]


def _run(cfg, d, n_group=1, topk_group=1, out_f32=True, single=True):
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                       router_bias=d["router_bias"], Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"],
                       Ws_down=d["Ws_down"], renorm=cfg.renorm, n_group=n_group,
                       topk_group=topk_group)
    y = layer(d["x"], out_f32=out_f32, single_launch=single)
    ws = layer.workspace(cfg.T)
    torch.cuda.synchronize()
    st = m.get_device_status(ws)
    assert st == m.MOE_OK, m.status_string(st)
    lay = m.workspace_layout(layer.problem(cfg.T))
    T, E, k = cfg.T, cfg.E, cfg.k

    def region(off, n, dt):
        return ws[off:off + n * 4].view(dt).cpu().numpy()

    return layer, y, dict(
        logits=region(lay["logits"], T * E, torch.float32).reshape(T, E),
        ids=region(lay["topk_ids"], T * k, torch.int32).reshape(T, k),
        w=region(lay["topk_w"], T * k, torch.float32).reshape(T, k),
        offs=region(lay["expert_offsets"], E + 2, torch.int32),
        gidx=region(lay["gather_idx"], T * k, torch.int32),
        spos=region(lay["slot_pos"], T * k, torch.int32))


def _check_against_oracle(oracle, cfg, d, y, r, n_group=1, topk_group=1):
    x, Wr, b = to_np(d["x"]), to_np(d["W_router"]), to_np(d["router_bias"])
    np.testing.assert_allclose(r["logits"], oracle.router_logits(x, Wr, b), rtol=0,
                               atol=2e-5 * (cfg.H / 256) ** 0.5)
    ids, w = oracle.route_grouped(np.ascontiguousarray(r["logits"]), cfg.k, cfg.renorm, n_group,
                                  topk_group)
    np.testing.assert_array_equal(r["ids"], ids)
    np.testing.assert_allclose(r["w"], w, rtol=0, atol=1e-6)
    offs, gidx, spos = oracle.permute(r["ids"], cfg.E, 1 if cfg.I_shared else 0)
    np.testing.assert_array_equal(r["offs"], offs)
    np.testing.assert_array_equal(r["gidx"], gidx)
    np.testing.assert_array_equal(r["spos"], spos)
    n = {kk: to_np(v) for kk, v in d.items()}
    ref = oracle.ffn_combine(x, r["ids"], r["w"], n["W_gate"], n["W_up"], n["W_down"],
                             n["Ws_gate"], n["Ws_up"], n["Ws_down"])
    assert_close(y.float().cpu().numpy(), ref, f"{cfg.name} single-launch y")


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_single_launch_matches_oracle(oracle, cfg):
    d = generate(cfg, seed=17, device=DEV)
    layer, y, r = _run(cfg, d)
    _check_against_oracle(oracle, cfg, d, y, r)
    # bf16 output: the rounding of the fp32 result; and a second call repeats it
    if cfg.dtype == "bf16":
        yb = layer(d["x"], single_launch=True)
        torch.cuda.synchronize()
        assert_bf16_is_rounded(yb, y)
    y2 = layer(d["x"], out_f32=True, single_launch=True)
    torch.cuda.synchronize()
    assert torch.equal(y2.view(torch.int32), y.view(torch.int32))


@pytest.mark.parametrize("n_group,topk_group", [(8, 3), (4, 1)])
def test_single_launch_group_limited_routing(oracle, n_group, topk_group):
    cfg = MoEConfig("grouped", T=50, H=512, E=64, k=6, I=128)
    d = generate(cfg, seed=23, device=DEV)
    _, y, r = _run(cfg, d, n_group, topk_group)
    _check_against_oracle(oracle, cfg, d, y, r, n_group, topk_group)


@pytest.mark.parametrize("cfg", CASES[:4], ids=[c.name for c in CASES[:4]])
def test_single_launch_agrees_with_the_kernel_chain(cfg):
    d = generate(cfg, seed=29, device=DEV)
    _, y1, r1 = _run(cfg, d, single=True)
    _, y0, r0 = _run(cfg, d, single=False)
    np.testing.assert_array_equal(r1["ids"], r0["ids"])
    np.testing.assert_array_equal(r1["gidx"], r0["gidx"])
    assert_close(y1.cpu().numpy(), y0.cpu().numpy(), f"{cfg.name} single vs chain")


def test_single_launch_full_size_decode(oracle):
    """The Qwen3-235B-shaped decode step at full size (seed 0, as timed): all
    routing and the permutation exactly, y on every token (covering sample)."""
    cfg = CONFIGS["qwen3_235b_decode"]
    d = generate(cfg, seed=0, device=DEV)
    _, y, r = _run(cfg, d)
    ids, w = oracle.route(np.ascontiguousarray(r["logits"]), cfg.k, cfg.renorm)
    np.testing.assert_array_equal(r["ids"], ids)
    np.testing.assert_allclose(r["w"], w, rtol=0, atol=1e-6)
    offs, gidx, spos = oracle.permute(r["ids"], cfg.E, 0)
    np.testing.assert_array_equal(r["offs"], offs)
    np.testing.assert_array_equal(r["gidx"], gidx)
    toks = covering_tokens(cfg, r["offs"], r["gidx"])
    ref, ids_o = oracle_rows(oracle, cfg, d, toks)
    np.testing.assert_array_equal(r["ids"][toks], ids_o)
    assert_close(y.cpu().numpy()[toks], ref, f"full-size decode, {len(toks)} tokens")


def test_single_launch_refuses_other_problems():
    cfg = MoEConfig("big", T=65, H=256, E=8, k=2, I=128)
    d = generate(cfg, seed=1, device=DEV, enforce_margin=False)
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k)
    with pytest.raises(m.MoEError) as ei:
        layer(d["x"], single_launch=True)
    assert ei.value.code == 2  # MOE_ERR_UNSUPPORTED: 65 tokens use the tiled GEMMs


def test_single_launch_bounded_wait_reports_timeout_and_context_survives():
    cfg = MoEConfig("s", T=40, H=256, E=8, k=2, I=128)
    d = generate(cfg, seed=3, device=DEV)
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k)
    ws = layer.workspace(cfg.T)
    before = layer(d["x"], single_launch=True).clone()
    torch.cuda.synchronize()
    assert m.get_device_status(ws) == m.MOE_OK
    pb = layer.problem(cfg.T, flags=m.MOE_FLAG_TEST_SKIP_SIGNAL, wait_limit_us=20000)
    y = torch.empty_like(before)
    m.forward_single_launch(pb, d["x"], layer.W_router, None, layer.W_gate, layer.W_up,
                            layer.W_down, None, None, None, y, ws)
    torch.cuda.synchronize()  # returns: every CTA gave up instead of hanging
    assert m.get_device_status(ws) == 5  # MOE_ERR_TIMEOUT
    after = layer(d["x"], single_launch=True)
    torch.cuda.synchronize()
    assert m.get_device_status(ws) == m.MOE_OK
    assert torch.equal(after.view(torch.int16), before.view(torch.int16))


def test_single_launch_replays_in_cuda_graph():
    cfg = MoEConfig("graph_single", T=64, H=512, E=32, k=8, I=256)
    d = generate(cfg, seed=5, device=DEV)
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k)
    x_static = d["x"].clone()
    y_static = torch.empty(cfg.T, cfg.H, dtype=cfg.torch_dtype, device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ref1 = layer(x_static, single_launch=True).clone()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer(x_static, out=y_static, single_launch=True)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y_static.view(torch.int16), ref1.view(torch.int16))
    x2 = generate(cfg, seed=6, device=DEV)["x"]
    x_static.copy_(x2)
    ref2 = layer(x2, single_launch=True).clone()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y_static.view(torch.int16), ref2.view(torch.int16))
    assert m.get_device_status(layer.workspace(cfg.T)) == m.MOE_OK
