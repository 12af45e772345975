"""Parity of every CUDA stage, called through the C ABI, against the CPU
oracle on the same seeded inputs.

Bars: top-k ids, counts, offsets and the permutation are bit-exact given
identical fp32 logits; gate weights within 1e-6; the layer output y (bf16
inputs, fp32 accumulation) satisfies max|gpu - oracle| <= 2e-2 * rms(oracle)
and rel-L2 <= 5e-3. That bound is applied to y as the library computes it in
fp32 (out_f32): a bf16 y cannot be closer to the oracle than half a bf16 ulp,
2^-8 |y|, which exceeds 2e-2 rms(y) on the largest entries of heavy-tailed
outputs (a token dominated by one expert). The bf16 y is then checked to be
exactly that fp32 y rounded to nearest-even, bit for bit. The intermediate h = silu(g) * u is heavy-tailed (a product
of two near-Gaussian sums), so a bound relative to its rms does not describe
its rounding; stage outputs are held elementwise to what one rounding to the
output type allows: |gpu - oracle| <= 2^-8 |oracle| + a * rms(oracle), where
bf16 round-to-nearest is within 2^-9 relative and a = 2e-3 covers fp32
summation order and the fast exponential. fp32 inputs run on the tensor cores
as tf32, which keeps 10 mantissa bits by truncation: each product can be off by
2^-9 relative, so a sum of H of them deviates by ~2^-9 rms(sum) per element
with tails several times that, and a = 1e-2 for fp32. rel-L2 <= 5e-3 always.
"""
import os

import numpy as np
import pytest
import torch

import mixture_experts_layer_route_gb300 as m
from moe_inputs import MoEConfig, generate, generate_hidden, generate_routing
from oracle import to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
MAX_REL = 2e-2
L2_REL = 5e-3


def assert_close(got, ref, what="", stage=False, tf32=False):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    if not ref.size:
        return
    rms = float(np.sqrt(np.mean(ref ** 2)))
    d = np.abs(got - ref)
    l2 = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    log = os.environ.get("MOE_TEST_ERRLOG")
    if log and not stage:
        with open(log, "a") as f:
            test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
            f.write(f"{test}\t{what}\t{float(d.max()) / max(rms, 1e-30):.5f}\t{l2:.3e}\n")
    if stage:
        bound = 2.0 ** -8 * np.abs(ref) + (1e-2 if tf32 else 2e-3) * rms
        worst = int(np.argmax(d - bound))
        assert (d <= bound).all(), (f"{what}: |d|={d.flat[worst]:.3e} at {worst} "
                                    f"ref={ref.flat[worst]:.3e} rms={rms:.3e}")
    else:
        err = float(d.max())
        assert err <= MAX_REL * rms + 1e-12, f"{what}: max|d|={err:.3e} rms={rms:.3e}"
    assert l2 <= L2_REL, f"{what}: rel-L2={l2:.3e}"


def bf16_rne(t32):
    """fp32 tensor -> bf16 by round-to-nearest-even (torch's conversion)."""
    return t32.to(torch.bfloat16)


def assert_bf16_is_rounded(y_bf16, y_f32, what="y"):
    r = bf16_rne(y_f32)
    bad = (r.view(torch.int16) != y_bf16.view(torch.int16)).sum().item()
    assert bad == 0, f"{what}: {bad} bf16 outputs differ from RNE(fp32 output)"


def ws_for(pb):
    return torch.zeros(m.workspace_size(pb), dtype=torch.uint8, device=DEV)


def finish(ws):
    torch.cuda.synchronize()
    st = m.get_device_status(ws)
    assert st == m.MOE_OK, m.status_string(st)


# ------------------------------------------------------------------ a1 logits

@pytest.mark.parametrize("T,H,E,dtype,bias", [
    (64, 256, 8, "f32", False), (64, 4096, 128, "bf16", False), (333, 512, 40, "bf16", True),
    (1024, 4096, 512, "bf16", True), (5, 7168, 256, "bf16", False), (200, 1024, 64, "f32", True),
    # 21 tiles of the small kernel: the split count must survive slice rounding
    (448, 4096, 192, "bf16", False),
    # the 128 x 128 kernel with token and expert tails, both dtypes
    (1500, 1024, 200, "bf16", True), (1100, 512, 72, "f32", False), (8192, 4096, 128, "bf16", False),
    # tensor-core path: a 16-expert tile; four expert tiles with a tail
    (64, 512, 8, "bf16", True), (130, 1024, 1000, "bf16", False),
])
def test_router_logits(oracle, T, H, E, dtype, bias):
    cfg = MoEConfig("l", T=T, H=H, E=E, k=1, I=64, dtype=dtype, zipf_s=1.1 if bias else 0.0)
    d = generate(cfg, seed=T + E, device=DEV, enforce_margin=False)
    pb = m.make_problem(T, H, E, 1, 64, dtype=dtype)
    ws = ws_for(pb)
    logits = torch.empty(T, E, dtype=torch.float32, device=DEV)
    m.router_logits(pb, d["x"], d["W_router"], d["router_bias"], logits, ws)
    finish(ws)
    ref = oracle.router_logits(to_np(d["x"]), to_np(d["W_router"]), to_np(d["router_bias"]))
    # fp32 sums of H products in a different order: |d| ~ sqrt(H) * 2^-24 * |term|
    np.testing.assert_allclose(logits.cpu().numpy(), ref, rtol=0, atol=2e-5 * (H / 256) ** 0.5)


# ------------------------------------------------------------------ a2 route

@pytest.mark.parametrize("T,E,k,renorm,ties", [
    (64, 8, 2, 1, False), (64, 128, 8, 1, False), (1000, 512, 10, 1, False),
    (77, 256, 8, 0, False), (50, 1000, 32, 1, False), (40, 32, 32, 1, False),
    (33, 16, 1, 1, False), (300, 64, 6, 1, True), (100, 8, 8, 0, True), (7, 40, 3, 1, True),
])
def test_route_bitexact(oracle, T, E, k, renorm, ties):
    g = np.random.default_rng(T * 7 + E)
    if ties:
        logits = g.integers(-2, 3, size=(T, E)).astype(np.float32)
    else:
        logits = (2.0 * g.standard_normal((T, E))).astype(np.float32)
    lt = torch.from_numpy(logits).to(DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    m.route(lt, k, renorm, ids, w)
    torch.cuda.synchronize()
    rid, rw = oracle.route(logits, k, renorm)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=0, atol=1e-6)


@pytest.mark.parametrize("T,E,k,n_group,topk_group,renorm,ties", [
    (64, 256, 8, 8, 4, 1, False), (100, 64, 6, 8, 3, 1, True), (50, 128, 8, 4, 2, 0, False),
    (33, 512, 10, 16, 5, 1, True), (40, 32, 6, 32, 6, 1, False), (77, 12, 5, 3, 2, 1, True),
    (20, 1024, 32, 32, 8, 1, False), (64, 16, 4, 2, 2, 1, True),
])
def test_route_grouped_bitexact(oracle, T, E, k, n_group, topk_group, renorm, ties):
    """Group-limited top-k: ids bit-exact and weights within 1e-6 of the oracle
    on the same fp32 logits (ties inside and across groups when `ties`)."""
    g = np.random.default_rng(T * 11 + E + n_group)
    if ties:
        logits = g.integers(-2, 3, size=(T, E)).astype(np.float32)
    else:
        logits = (2.0 * g.standard_normal((T, E))).astype(np.float32)
    lt = torch.from_numpy(logits).to(DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    m.route_grouped(lt, k, renorm, n_group, topk_group, ids, w)
    torch.cuda.synchronize()
    rid, rw = oracle.route_grouped(logits, k, renorm, n_group, topk_group)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=0, atol=1e-6)


@pytest.mark.parametrize("T,E,k,n_group,topk_group", [
    (200, 128, 8, 1, 1), (64, 40, 5, 1, 1), (100, 256, 8, 8, 4), (50, 64, 6, 4, 2),
])
def test_route_signed_zeros_tie(oracle, T, E, k, n_group, topk_group):
    """-0 and +0 compare equal, so among zero logits the lower expert index
    wins whatever the signs; the logits mix both zeros with small integers."""
    g = np.random.default_rng(T + E + k)
    logits = g.integers(-1, 2, size=(T, E)).astype(np.float32)
    zero = g.random((T, E)) < 0.6
    logits[zero] = np.where(g.random(int(zero.sum())) < 0.5, np.float32(0.0), np.float32(-0.0))
    lt = torch.from_numpy(logits).to(DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    m.route_grouped(lt, k, 1, n_group, topk_group, ids, w)
    torch.cuda.synchronize()
    rid, rw = oracle.route_grouped(logits, k, 1, n_group, topk_group)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=0, atol=1e-6)


def test_route_grouped_rejects_bad_groups():
    lt = torch.zeros(4, 64, dtype=torch.float32, device=DEV)
    ids = torch.empty(4, 8, dtype=torch.int32, device=DEV)
    w = torch.empty(4, 8, dtype=torch.float32, device=DEV)
    for n_group, topk_group in ((6, 2), (8, 0), (8, 9), (64, 7), (16, 1)):
        with pytest.raises(m.MoEError):
            m.route_grouped(lt, 8, 1, n_group, topk_group, ids, w)


# ------------------------------------------------------------------ a3 permute

def _ids_with_counts(counts, seed):
    """k = 1 routing whose expert e receives counts[e] tokens, token order shuffled."""
    lst = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)])
    np.random.default_rng(seed).shuffle(lst)
    return lst.reshape(-1, 1)


@pytest.mark.parametrize("case", ["random", "zipf", "one_expert", "t1", "big", "shared",
                                  "e1024", "chunks_shared", "chunk_edge"])
def test_permute_bitexact(oracle, case):
    if case == "random":
        ids, _ = generate_routing(301, 16, 4, seed=1)
        E, shared = 16, 0
    elif case == "zipf":
        ids, _ = generate_routing(1024, 512, 10, seed=2, zipf_s=1.1)
        E, shared = 512, 0
    elif case == "one_expert":
        ids = np.full((500, 1), 3, np.int32)
        E, shared = 8, 0
    elif case == "t1":
        ids, _ = generate_routing(1, 8, 8, seed=3)
        E, shared = 8, 1
    elif case == "big":
        ids, _ = generate_routing(8192, 128, 8, seed=4)
        E, shared = 128, 0
    elif case == "shared":
        ids, _ = generate_routing(97, 24, 3, seed=5)
        E, shared = 24, 1
    elif case == "e1024":
        ids, _ = generate_routing(700, 1024, 12, seed=6)
        E, shared = 1024, 0
    elif case == "chunks_shared":  # several chunks of the grid-wide variant, skewed
        ids, _ = generate_routing(3001, 64, 6, seed=7, zipf_s=1.1)
        E, shared = 64, 1
    else:  # exactly two chunks (4096 slots is the single-CTA limit)
        ids, _ = generate_routing(1025, 40, 4, seed=8)
        E, shared = 40, 0
    ids = np.ascontiguousarray(np.asarray(ids, np.int32))
    T, k = ids.shape
    dids = torch.from_numpy(ids).to(DEV)
    offs = torch.empty(E + 2, dtype=torch.int32, device=DEV)
    gidx = torch.empty(T * k, dtype=torch.int32, device=DEV)
    spos = torch.empty(T * k, dtype=torch.int32, device=DEV)
    ws = ws_for(m.make_problem(T, 128, E, k, 64))
    m.permute(dids, E, shared, offs, gidx, spos, ws)
    finish(ws)
    ro, rg, rs = oracle.permute(ids, E, shared)
    np.testing.assert_array_equal(offs.cpu().numpy(), ro)
    np.testing.assert_array_equal(gidx.cpu().numpy(), rg)
    np.testing.assert_array_equal(spos.cpu().numpy(), rs)


def test_permute_out_of_range_id_sets_device_check():
    for T in (2, 3000):  # single-CTA and grid-wide variants
        ids = torch.zeros(T, 2, dtype=torch.int32, device=DEV)
        ids[:, 1] = 1
        ids[T - 1, 1] = 9
        offs = torch.empty(6, dtype=torch.int32, device=DEV)
        gidx = torch.empty(2 * T, dtype=torch.int32, device=DEV)
        spos = torch.empty(2 * T, dtype=torch.int32, device=DEV)
        ws = ws_for(m.make_problem(T, 128, 4, 2, 64))
        m.permute(ids, 4, 0, offs, gidx, spos, ws)
        torch.cuda.synchronize()
        assert m.get_device_status(ws) == 6  # MOE_ERR_DEVICE_CHECK
        m.reset_device_status(ws)
        assert m.get_device_status(ws) == m.MOE_OK


# ------------------------------------------------------------------ a4 / a5 GEMMs

# Segment lengths around the token tiles (32, 128, 256), which are also the row
# counts where the automatic choice changes tile (32|33, 128|129), and the
# 16-row MMA step.
RAGGED = [0, 1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 192, 193, 255, 256, 257,
          300, 511, 0, 4]
TILES = [m.MOE_TILE_AUTO, m.MOE_TILE_DECODE, m.MOE_TILE_MEDIUM, m.MOE_TILE_PREFILL]
TILE_IDS = ["auto", "t32", "t128", "t256"]


def _gemm_case(case, dtype):
    if case == "ragged":
        ids = _ids_with_counts(RAGGED, seed=11)
        w = np.ones(ids.shape, np.float32)
        E, H, I, Is = len(RAGGED), 256, 192, 0
    elif case == "random":
        ids, w = generate_routing(300, 16, 4, seed=12)
        ids, w = ids.numpy(), w.numpy()
        E, H, I, Is = 16, 512, 256, 0
    elif case == "shared":
        ids, w = generate_routing(150, 12, 3, seed=13)
        ids, w = ids.numpy(), w.numpy()
        E, H, I, Is = 12, 256, 128, 192
    else:  # zipf: many empty and tiny groups
        ids, w = generate_routing(257, 64, 6, seed=14, zipf_s=1.1)
        ids, w = ids.numpy(), w.numpy()
        E, H, I, Is = 64, 384, 320, 64
    T, k = ids.shape
    cfg = MoEConfig("g", T=T, H=H, E=E, k=k, I=I, I_shared=Is, dtype=dtype)
    d = generate(cfg, seed=E + T, device=DEV, enforce_margin=False)
    return cfg, d, np.ascontiguousarray(ids, dtype=np.int32), np.ascontiguousarray(w, np.float32)


@pytest.mark.parametrize("tile", TILES, ids=TILE_IDS)
@pytest.mark.parametrize("case,dtype", [("ragged", "bf16"), ("random", "bf16"),
                                        ("shared", "bf16"), ("zipf", "bf16"),
                                        ("random", "f32"), ("shared", "f32")])
def test_grouped_swiglu_gemm(oracle, case, dtype, tile):
    cfg, d, ids, _ = _gemm_case(case, dtype)
    T, k, E = cfg.T, cfg.k, cfg.E
    offs, gidx, spos = oracle.permute(ids, E, 1 if cfg.I_shared else 0)
    pb = m.make_problem(T, cfg.H, E, k, cfg.I, cfg.I_shared, dtype=dtype, tile=tile)
    ws = ws_for(pb)
    h = torch.full((T * k, cfg.I), float("nan"), dtype=cfg.torch_dtype, device=DEV)
    hs = (torch.full((T, cfg.I_shared), float("nan"), dtype=cfg.torch_dtype, device=DEV)
          if cfg.I_shared else None)
    m.grouped_swiglu_gemm(pb, d["x"], torch.from_numpy(offs).to(DEV),
                          torch.from_numpy(gidx).to(DEV), torch.from_numpy(spos).to(DEV),
                          d["W_gate"], d["W_up"], d["Ws_gate"], d["Ws_up"], h, hs, ws)
    finish(ws)
    n = {kk: to_np(v) for kk, v in d.items()}
    rh, rhs = oracle.expert_h(n["x"], offs, gidx, n["W_gate"], n["W_up"], k, n["Ws_gate"],
                              n["Ws_up"])
    assert_close(h.float().cpu().numpy(), rh, "h", stage=True, tf32=dtype == "f32")
    if cfg.I_shared:
        assert_close(hs.float().cpu().numpy(), rhs, "h_shared", stage=True,
                     tf32=dtype == "f32")


@pytest.mark.parametrize("tile", TILES, ids=TILE_IDS)
@pytest.mark.parametrize("case,dtype", [("ragged", "bf16"), ("random", "bf16"),
                                        ("shared", "bf16"), ("zipf", "bf16"),
                                        ("random", "f32"), ("shared", "f32")])
def test_down_combine(oracle, case, dtype, tile):
    cfg, d, ids, w = _gemm_case(case, dtype)
    T, k, E = cfg.T, cfg.k, cfg.E
    offs, gidx, spos = oracle.permute(ids, E, 1 if cfg.I_shared else 0)
    h = generate_hidden(T * k, cfg.I, seed=3, device=DEV, dtype=cfg.torch_dtype)
    hs = (generate_hidden(T, cfg.I_shared, seed=4, device=DEV, dtype=cfg.torch_dtype)
          if cfg.I_shared else None)
    args = (torch.from_numpy(offs).to(DEV), torch.from_numpy(gidx).to(DEV),
            torch.from_numpy(w).to(DEV), d["W_down"], d["Ws_down"])
    pb = m.make_problem(T, cfg.H, E, k, cfg.I, cfg.I_shared, dtype=dtype, tile=tile)
    pb32 = m.make_problem(T, cfg.H, E, k, cfg.I, cfg.I_shared, dtype=dtype, tile=tile,
                          out_f32=True)
    ws = ws_for(pb)
    y = torch.full((T, cfg.H), float("nan"), dtype=cfg.torch_dtype, device=DEV)
    y32 = torch.full((T, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
    m.down_combine(pb, h, hs, *args[:3], args[3], args[4], y, ws)
    m.down_combine(pb32, h, hs, *args[:3], args[3], args[4], y32, ws)
    finish(ws)
    ref = oracle.down_combine(to_np(h), offs, spos, ids, w, to_np(d["W_down"]), to_np(hs),
                              to_np(d["Ws_down"]))
    assert_close(y32.cpu().numpy(), ref, "y")
    if dtype == "bf16":
        assert_bf16_is_rounded(y, y32)
    else:
        assert torch.equal(y, y32)


# ------------------------------------------------------------------ whole layer

SMALL = [
    MoEConfig("tiny_f32", T=64, H=256, E=8, k=2, I=512, dtype="f32"),
    MoEConfig("decode_like", T=64, H=512, E=32, k=8, I=256),
    MoEConfig("prefill_like", T=1200, H=256, E=8, k=2, I=192),
    MoEConfig("zipf_like", T=300, H=384, E=128, k=10, I=128, zipf_s=1.1),
    MoEConfig("shared_like", T=257, H=256, E=16, k=4, I=128, I_shared=192),
    MoEConfig("t1", T=1, H=128, E=4, k=4, I=64, renorm=0),
    MoEConfig("f32_shared", T=100, H=256, E=6, k=3, I=128, I_shared=64, dtype="f32"),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[c.name for c in SMALL])
def test_forward_vs_oracle(oracle, cfg):
    d = generate(cfg, seed=0, device=DEV)
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                       router_bias=d["router_bias"], Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"],
                       Ws_down=d["Ws_down"], renorm=cfg.renorm)
    y = layer(d["x"])
    y32 = layer(d["x"], out_f32=True)
    ws = layer.workspace(cfg.T)
    finish(ws)
    n = {kk: to_np(v) for kk, v in d.items()}
    ref, inter = oracle.forward(n["x"], n["W_router"], n["router_bias"], n["W_gate"], n["W_up"],
                                n["W_down"], cfg.k, cfg.renorm, n["Ws_gate"], n["Ws_up"],
                                n["Ws_down"], want_intermediates=True)
    lay = m.workspace_layout(layer.problem(cfg.T))
    T, k = cfg.T, cfg.k
    gids = ws[lay["topk_ids"]:lay["topk_ids"] + T * k * 4].view(torch.int32).view(T, k)
    np.testing.assert_array_equal(gids.cpu().numpy(), inter["ids"])
    gw = ws[lay["topk_w"]:lay["topk_w"] + T * k * 4].view(torch.float32).view(T, k)
    np.testing.assert_allclose(gw.cpu().numpy(), inter["w"], rtol=0, atol=1e-6)
    assert_close(y32.cpu().numpy(), ref, "y")
    if cfg.dtype == "bf16":
        assert_bf16_is_rounded(y, y32)
    else:
        assert torch.equal(y, y32)


@pytest.mark.parametrize("T,dtype", [(300, "bf16"), (64, "bf16"), (130, "f32")])
def test_forward_grouped_routing_vs_oracle(oracle, T, dtype):
    """moe_forward with group-limited routing (8 groups, 3 kept) and a shared
    expert: the ids and weights the forward pass stored equal the oracle's
    group-limited route of the logits it stored, and y matches the oracle's
    experts and combine on those ids and weights."""
    cfg = MoEConfig("grouped", T=T, H=256, E=64, k=6, I=128, I_shared=128, dtype=dtype)
    d = generate(cfg, seed=9, device=DEV)
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                       Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"], Ws_down=d["Ws_down"],
                       n_group=8, topk_group=3)
    y32 = layer(d["x"], out_f32=True)
    ws = layer.workspace(T)
    finish(ws)
    lay = m.workspace_layout(layer.problem(T))
    E, k = cfg.E, cfg.k
    logits = ws[lay["logits"]:lay["logits"] + T * E * 4].view(torch.float32).view(T, E)
    gids = ws[lay["topk_ids"]:lay["topk_ids"] + T * k * 4].view(torch.int32).view(T, k)
    gw = ws[lay["topk_w"]:lay["topk_w"] + T * k * 4].view(torch.float32).view(T, k)
    rid, rw = oracle.route_grouped(logits.cpu().numpy(), k, 1, 8, 3)
    np.testing.assert_array_equal(gids.cpu().numpy(), rid)
    np.testing.assert_allclose(gw.cpu().numpy(), rw, rtol=0, atol=1e-6)
    assert max(len(set(r.tolist())) for r in rid // 8) <= 3  # at most topk_group groups
    n = {kk: to_np(v) for kk, v in d.items()}
    ref = oracle.ffn_combine(n["x"], rid, rw, n["W_gate"], n["W_up"], n["W_down"], n["Ws_gate"],
                             n["Ws_up"], n["Ws_down"])
    assert_close(y32.cpu().numpy(), ref, "y")


def _forward_vs_oracle(oracle, cfg, d, **layer_kw):
    """moe_forward against the oracle: the oracle routes the logits the forward
    pass stored (ids then match bit for bit, even where inputs without a
    routing margin leave near ties), and y is the oracle's experts and combine
    on those ids."""
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                       router_bias=d["router_bias"], Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"],
                       Ws_down=d["Ws_down"], renorm=cfg.renorm, **layer_kw)
    y32 = layer(d["x"], out_f32=True)
    ws = layer.workspace(cfg.T)
    finish(ws)
    T, E, k = cfg.T, cfg.E, cfg.k
    lay = m.workspace_layout(layer.problem(T))
    logits = ws[lay["logits"]:lay["logits"] + T * E * 4].view(torch.float32).view(T, E)
    gids = ws[lay["topk_ids"]:lay["topk_ids"] + T * k * 4].view(torch.int32).view(T, k)
    rid, rw = oracle.route(logits.cpu().numpy(), k, cfg.renorm)
    np.testing.assert_array_equal(gids.cpu().numpy(), rid)
    n = {kk: to_np(v) for kk, v in d.items()}
    ref = oracle.ffn_combine(n["x"], rid, rw, n["W_gate"], n["W_up"], n["W_down"], n["Ws_gate"],
                             n["Ws_up"], n["Ws_down"])
    assert_close(y32.cpu().numpy(), ref, "y")


def test_forward_most_experts_and_top32(oracle):
    """E = 1024 (the largest expert count), k = 32 (the largest top-k): most
    experts hold a handful of rows, many none."""
    cfg = MoEConfig("wide", T=256, H=256, E=1024, k=32, I=128, I_shared=128)
    _forward_vs_oracle(oracle, cfg, generate(cfg, seed=21, device=DEV))


@pytest.mark.parametrize("tile", TILES, ids=TILE_IDS)
def test_forward_one_expert_takes_every_token(oracle, tile):
    """A router bias sends every token's first choice to expert 0: one group of
    T rows (many token tiles) next to small ones."""
    cfg = MoEConfig("dominant", T=1000, H=256, E=16, k=2, I=128)
    d = generate(cfg, seed=22, device=DEV, enforce_margin=False)
    bias = torch.zeros(cfg.E, dtype=torch.float32, device=DEV)
    bias[0] = 50.0
    d["router_bias"] = bias
    _forward_vs_oracle(oracle, cfg, d, tile=tile)


def test_forward_empty_batch_touches_nothing():
    cfg = MoEConfig("empty", T=8, H=256, E=8, k=2, I=128)
    d = generate(cfg, seed=23, device=DEV)
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k)
    x0 = d["x"][:0]
    y0 = torch.full((0, cfg.H), 7.0, dtype=cfg.torch_dtype, device=DEV)
    assert layer(x0, out=y0) is y0
    torch.cuda.synchronize()


def test_forward_is_bitwise_reproducible():
    cfg = MoEConfig("r", T=300, H=256, E=16, k=4, I=128, I_shared=64)
    d = generate(cfg, seed=5, device=DEV)
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                       Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"], Ws_down=d["Ws_down"])
    y1 = layer(d["x"]).clone()
    y2 = layer(d["x"]).clone()
    finish(layer.workspace(cfg.T))
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_forward_token_permutation_equivariant():
    cfg = MoEConfig("p", T=200, H=256, E=16, k=4, I=128)
    d = generate(cfg, seed=6, device=DEV)
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k)
    perm = torch.randperm(cfg.T, generator=torch.Generator().manual_seed(1)).to(DEV)
    y = layer(d["x"])
    yp = layer(d["x"][perm].contiguous())
    finish(layer.workspace(cfg.T))
    # per-token results do not depend on the other tokens of the batch
    assert torch.equal(yp.view(torch.int16), y[perm].view(torch.int16))
