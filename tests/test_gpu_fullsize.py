"""Full-size parity on the five layer shapes, in the configuration the benchmark
times (moe_forward, automatic tile choice, seed 0).

Whole-tensor checks where the oracle is cheap: every token's top-k ids
(bit-exact) and weights (1e-6) from the oracle's routing of the GPU's own fp32
logits, and the permutation (bit-exact). Sampled checks where it is not: the
logits of 64 tokens, and the output rows of a few tokens, each recomputed by the
oracle from that token's x row and its experts' weights. Float bounds apply to
the fp32 result (out_f32); the bf16 output is checked to be its rounding.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_route_gb300 as m
from moe_inputs import CONFIGS, generate
from oracle import to_np
from test_gpu_parity import assert_bf16_is_rounded, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", params=sorted(CONFIGS))
def run(request):
    cfg = CONFIGS[request.param]
    torch.cuda.empty_cache()
    d = generate(cfg, seed=0, device=DEV)
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                       router_bias=d["router_bias"], Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"],
                       Ws_down=d["Ws_down"], renorm=cfg.renorm)
    y = layer(d["x"])
    y32 = layer(d["x"], out_f32=True)
    ws = layer.workspace(cfg.T)
    torch.cuda.synchronize()
    st = m.get_device_status(ws)
    assert st == m.MOE_OK, m.status_string(st)
    lay = m.workspace_layout(layer.problem(cfg.T))
    T, k, E = cfg.T, cfg.k, cfg.E

    def region(off, n, dt):
        return ws[off:off + n * 4].view(dt).cpu().numpy()

    out = dict(cfg=cfg, d=d, y=y32.cpu().numpy(), y_out=y, y32=y32,
               logits=region(lay["logits"], T * E, torch.float32).reshape(T, E),
               ids=region(lay["topk_ids"], T * k, torch.int32).reshape(T, k),
               w=region(lay["topk_w"], T * k, torch.float32).reshape(T, k),
               offs=region(lay["expert_offsets"], E + 2, torch.int32),
               gidx=region(lay["gather_idx"], T * k, torch.int32),
               spos=region(lay["slot_pos"], T * k, torch.int32))
    yield out
    del layer, d, y, y32, ws
    torch.cuda.empty_cache()


def test_output_is_rounded_fp32_result(run):
    """The layer's bf16 output is its fp32 result rounded to nearest, everywhere."""
    if run["cfg"].dtype == "bf16":
        assert_bf16_is_rounded(run["y_out"], run["y32"])
    else:
        assert torch.equal(run["y_out"], run["y32"])


def test_route_bitexact_all_tokens(run, oracle):
    cfg = run["cfg"]
    ids, w = oracle.route(np.ascontiguousarray(run["logits"]), cfg.k, cfg.renorm)
    np.testing.assert_array_equal(run["ids"], ids)
    np.testing.assert_allclose(run["w"], w, rtol=0, atol=1e-6)


def test_permute_bitexact_all_slots(run, oracle):
    cfg = run["cfg"]
    offs, gidx, spos = oracle.permute(run["ids"], cfg.E, 1 if cfg.I_shared else 0)
    np.testing.assert_array_equal(run["offs"], offs)
    np.testing.assert_array_equal(run["gidx"], gidx)
    np.testing.assert_array_equal(run["spos"], spos)


def test_logits_sample(run, oracle):
    cfg, d = run["cfg"], run["d"]
    rows = np.unique(np.linspace(0, cfg.T - 1, 64).astype(np.int64))
    x = to_np(d["x"][torch.from_numpy(rows).to(DEV)])
    ref = oracle.router_logits(x, to_np(d["W_router"]), to_np(d["router_bias"]))
    np.testing.assert_allclose(run["logits"][rows], ref, rtol=0,
                               atol=2e-5 * (cfg.H / 256) ** 0.5)


def test_output_sample(run, oracle):
    """Each sampled token recomputed alone by the oracle: its x row, the ids and
    weights the oracle's routing gives, and only its experts' weights."""
    cfg, d = run["cfg"], run["d"]
    n = 4 if cfg.T >= 4 else cfg.T
    toks = np.unique(np.linspace(0, cfg.T - 1, n).astype(np.int64))
    got = []
    ref = []
    for t in toks:
        lg = oracle.router_logits(to_np(d["x"][t:t + 1]), to_np(d["W_router"]),
                                  to_np(d["router_bias"]))
        ids, w = oracle.route(lg, cfg.k, cfg.renorm)
        sel = torch.from_numpy(ids[0].astype(np.int64)).to(DEV)
        local = np.arange(cfg.k, dtype=np.int32).reshape(1, cfg.k)
        y = oracle.ffn_combine(to_np(d["x"][t:t + 1]), local, w, to_np(d["W_gate"][sel]),
                               to_np(d["W_up"][sel]), to_np(d["W_down"][sel]),
                               to_np(d["Ws_gate"]), to_np(d["Ws_up"]), to_np(d["Ws_down"]))
        ref.append(y[0])
        got.append(run["y"][t])
    assert_close(np.stack(got), np.stack(ref), f"{cfg.name} sampled y")


def test_fp8_output_sample(run, oracle):
    """The E4M3-weight layer (moe_forward_fp8) at full size: sampled tokens
    recomputed alone by the oracle's FP8 experts and combine, with its routing
    and only the token's experts' weights, quantized by the oracle itself."""
    cfg, d = run["cfg"], run["d"]
    if cfg.dtype != "bf16":
        pytest.skip("E4M3 weights come with bf16 activations")
    layer = m.MoELayerFP8(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                          router_bias=d["router_bias"], Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"],
                          Ws_down=d["Ws_down"], renorm=cfg.renorm)
    y32 = layer(d["x"], out_f32=True).cpu().numpy()
    torch.cuda.synchronize()
    assert m.get_device_status(layer.workspace(cfg.T)) == m.MOE_OK
    n = 4 if cfg.T >= 4 else cfg.T
    toks = np.unique(np.linspace(0, cfg.T - 1, n).astype(np.int64))
    got, ref = [], []
    for t in toks:
        xt = to_np(d["x"][t:t + 1])
        lg = oracle.router_logits(xt, to_np(d["W_router"]), to_np(d["router_bias"]))
        ids, w = oracle.route(lg, cfg.k, cfg.renorm)
        sel = torch.from_numpy(ids[0].astype(np.int64)).to(DEV)
        local = np.arange(cfg.k, dtype=np.int32).reshape(1, cfg.k)
        y = oracle.ffn_combine_fp8(xt, local, w, to_np(d["W_gate"][sel]), to_np(d["W_up"][sel]),
                                   to_np(d["W_down"][sel]), to_np(d["Ws_gate"]),
                                   to_np(d["Ws_up"]), to_np(d["Ws_down"]))
        ref.append(y[0])
        got.append(y32[t])
    del layer
    torch.cuda.empty_cache()
    assert_close(np.stack(got), np.stack(ref), f"{cfg.name} sampled fp8 y")
