"""Full-size parity on the five layer shapes, in the configuration the benchmark
times (moe_forward, automatic tile choice, seed 0).

Whole-tensor checks where the oracle is cheap: every token's top-k ids
(bit-exact) and weights (1e-6) from the oracle's routing of the GPU's own fp32
logits, and the permutation (bit-exact). Sampled checks where it is not: the
logits of 64 tokens; the output rows of a covering sample of about 70 tokens
(spread over the batch, plus the tokens of the heaviest and the lightest
expert, of the first and the last group of the GEMMs' schedule and of the
expert with the most ragged last tile; with a shared expert every token also
reaches its group); and the intermediate h of every position of those experts
(the shared expert: its first and last tiles), elementwise. Float bounds apply
to the fp32 result (out_f32); the bf16 output is checked to be its rounding.
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

    es = 2 if cfg.dtype == "bf16" else 4
    hdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    h = ws[lay["h"]:lay["h"] + T * k * cfg.I * es].view(hdt).view(T * k, cfg.I).float()
    hs = None
    if cfg.I_shared:
        o = lay["h_shared"]
        hs = ws[o:o + T * cfg.I_shared * es].view(hdt).view(T, cfg.I_shared).float()
    out = dict(cfg=cfg, d=d, y=y32.cpu().numpy(), y_out=y, y32=y32, h=h, hs=hs,
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


# ------------------------------------------------------------ covering samples

CHUNK = 16  # experts whose weights are on the host at once


def schedule_experts(cfg, offs):
    """Experts at the extremes of the grouped GEMMs' work: the heaviest and the
    lightest non-empty expert, the first and the last group of the schedule
    (non-empty groups in four load classes, > 256, > 128, > 32 rows and the
    rest, heaviest class first, expert index order within a class), and the
    expert whose last token tile is the most ragged."""
    counts = np.diff(offs[:cfg.E + 1]).astype(np.int64)
    nz = np.nonzero(counts)[0]
    cls = np.select([counts > 256, counts > 128, counts > 32], [0, 1, 2], 3)
    order = sorted(nz, key=lambda e: (cls[e], e))
    tile = 32 if cfg.T <= 64 else 256
    tail = nz[int(np.argmin([(c % tile) or tile for c in counts[nz]]))]
    return {"heaviest": int(nz[np.argmax(counts[nz])]), "lightest": int(nz[np.argmin(counts[nz])]),
            "first": int(order[0]), "last": int(order[-1]), "ragged": int(tail)}


def covering_tokens(cfg, offs, gidx, n_even=64, per_expert=6):
    """Tokens spread over the batch plus the first and last tokens of each
    schedule-extreme expert's segment."""
    toks = set(np.linspace(0, cfg.T - 1, min(n_even, cfg.T)).astype(np.int64).tolist())
    for e in set(schedule_experts(cfg, offs).values()):
        p0, p1 = int(offs[e]), int(offs[e + 1])
        pos = list(range(p0, min(p1, p0 + per_expert))) + list(range(max(p0, p1 - per_expert), p1))
        toks |= {int(gidx[p]) // cfg.k for p in pos}
    toks |= {int(gidx[0]) // cfg.k, int(gidx[-1]) // cfg.k, cfg.T - 1}
    return np.array(sorted(toks), np.int64)


def oracle_rows(oracle, cfg, d, toks, fp8=False, mx=False):
    """The oracle's y rows of `toks`: routing from each token's own logits, then
    every (token, rank) slot through the oracle's experts + combine with k = 1
    and the slot's gate weight, CHUNK experts' weights on the host at a time;
    each token's slot rows are summed in rank order (float64), then its
    shared-expert row (weight 1) is added."""
    x = to_np(d["x"][torch.from_numpy(toks).to(DEV)])
    lg = oracle.router_logits(x, to_np(d["W_router"]), to_np(d["router_bias"]))
    ids, w = oracle.route(lg, cfg.k, cfg.renorm)
    fn = oracle.ffn_combine_mx if mx else (oracle.ffn_combine_fp8 if fp8 else oracle.ffn_combine)
    parts = np.zeros((len(toks), cfg.k, cfg.H))
    experts = np.unique(ids)
    for c0 in range(0, len(experts), CHUNK):
        ch = experts[c0:c0 + CHUNK]
        sel = torch.from_numpy(ch.astype(np.int64)).to(DEV)
        loc = np.full(cfg.E, -1, np.int64)
        loc[ch] = np.arange(len(ch))
        ti, ri = np.nonzero(np.isin(ids, ch))
        parts[ti, ri] = fn(np.ascontiguousarray(x[ti]),
                           loc[ids[ti, ri]].astype(np.int32).reshape(-1, 1),
                           np.ascontiguousarray(w[ti, ri].reshape(-1, 1)),
                           to_np(d["W_gate"][sel]), to_np(d["W_up"][sel]),
                           to_np(d["W_down"][sel]))
    y = parts[:, 0].copy()
    for r in range(1, cfg.k):
        y += parts[:, r]
    if cfg.I_shared:
        one = np.zeros((len(toks), 1), np.int32)
        y += fn(x, one, np.ones((len(toks), 1), np.float32), to_np(d["Ws_gate"])[None],
                to_np(d["Ws_up"])[None], to_np(d["Ws_down"])[None])
    return y, ids


def test_output_covering_sample(run, oracle):
    cfg, d = run["cfg"], run["d"]
    toks = covering_tokens(cfg, run["offs"], run["gidx"])
    assert len(toks) >= min(64, cfg.T)
    ref, ids = oracle_rows(oracle, cfg, d, toks)
    np.testing.assert_array_equal(run["ids"][toks], ids)
    assert_close(run["y"][toks], ref, f"{cfg.name} y on {len(toks)} covering tokens")


def test_h_of_schedule_extreme_experts(run, oracle):
    """Every position of the schedule-extreme experts (gate/up GEMM + SwiGLU
    output h, elementwise, the stage bound); with a shared expert, its first
    and last token tiles."""
    cfg, d = run["cfg"], run["d"]
    offs, gidx = run["offs"], run["gidx"]
    tf32 = cfg.dtype == "f32"
    for name, e in sorted(schedule_experts(cfg, offs).items()):
        p0, p1 = int(offs[e]), int(offs[e + 1])
        toks = gidx[p0:p1] // cfg.k
        x = to_np(d["x"][torch.from_numpy(toks.astype(np.int64)).to(DEV)])
        n = p1 - p0
        h, _ = oracle.expert_h(x, np.array([0, n, n], np.int32), np.arange(n, dtype=np.int32),
                               to_np(d["W_gate"][e:e + 1]), to_np(d["W_up"][e:e + 1]), 1)
        assert_close(run["h"][p0:p1].cpu().numpy(), h, f"{cfg.name} h of the {name} expert {e}",
                     stage=True, tf32=tf32)
    if cfg.I_shared:
        t = np.r_[0:min(64, cfg.T), max(0, cfg.T - 256):cfg.T]
        t = np.unique(t)
        x = to_np(d["x"][torch.from_numpy(t).to(DEV)])
        n = len(t)
        _, hs = oracle.expert_h(x, np.array([0, 0, n], np.int32), np.zeros(0, np.int32),
                                to_np(d["W_gate"][:1]) * 0, to_np(d["W_up"][:1]) * 0, 1,
                                to_np(d["Ws_gate"]), to_np(d["Ws_up"]))
        assert_close(run["hs"][torch.from_numpy(t).to(DEV)].cpu().numpy(), hs,
                     f"{cfg.name} shared h", stage=True, tf32=tf32)


def test_fp8_output_sample(run, oracle):
    """The E4M3-weight layer (moe_forward_fp8) at full size: a covering sample
    of tokens recomputed by the oracle's FP8 experts and combine, slot by slot,
    with only the sampled tokens' experts' weights, quantized by the oracle."""
    cfg, d = run["cfg"], run["d"]
    if cfg.dtype != "bf16":
        pytest.skip("E4M3 weights come with bf16 activations")
    layer = m.MoELayerFP8(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                          router_bias=d["router_bias"], Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"],
                          Ws_down=d["Ws_down"], renorm=cfg.renorm)
    y32 = layer(d["x"], out_f32=True).cpu().numpy()
    torch.cuda.synchronize()
    assert m.get_device_status(layer.workspace(cfg.T)) == m.MOE_OK
    del layer
    torch.cuda.empty_cache()
    toks = covering_tokens(cfg, run["offs"], run["gidx"], n_even=8, per_expert=1)
    ref, _ = oracle_rows(oracle, cfg, d, toks, fp8=True)
    assert_close(y32[toks], ref, f"{cfg.name} fp8 y on {len(toks)} covering tokens")


def test_mx_output_sample(run, oracle):
    """The MXFP8-weight layer (moe_forward_mx) at full size: a covering sample
    of tokens recomputed by the oracle's MXFP8 experts and combine, slot by
    slot, with only the sampled tokens' experts' weights, quantized by the
    oracle."""
    cfg, d = run["cfg"], run["d"]
    if cfg.dtype != "bf16":
        pytest.skip("MXFP8 weights come with bf16 activations")
    layer = m.MoELayerMX(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                         router_bias=d["router_bias"], Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"],
                         Ws_down=d["Ws_down"], renorm=cfg.renorm)
    y32 = layer(d["x"], out_f32=True).cpu().numpy()
    torch.cuda.synchronize()
    assert m.get_device_status(layer.workspace(cfg.T)) == m.MOE_OK
    del layer
    torch.cuda.empty_cache()
    toks = covering_tokens(cfg, run["offs"], run["gidx"], n_even=8, per_expert=1)
    ref, _ = oracle_rows(oracle, cfg, d, toks, mx=True)
    assert_close(y32[toks], ref, f"{cfg.name} mx y on {len(toks)} covering tokens")
