"""Pins for the CPU oracle: each test checks it against something other than
itself (a library routine, a closed form, an invariant, or brute force).

CPU only. The layer definition followed is the one stated on the pages:
"Lower latency and higher throughput with multi-node DeepSeek deployment"
(sections "MoE Router", "Expert Parallelism", "GroupGEMM"), "CuTeDSL at
Perplexity" (section "Mixture-of-Experts Dispatch/Combine", "Local") and the
Qwen3.5-397B on TPU v7x write-up (sections 4.2.2 and 6).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from moe_inputs import MoEConfig, generate
from oracle import to_np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _np_swiglu_ffn(x, Wg, Wu, Wd):
    """Dense SwiGLU FFN in float64 numpy: x [T,H], Wg/Wu [I,H], Wd [H,I]."""
    g = x @ Wg.T
    u = x @ Wu.T
    h = g / (1.0 + np.exp(-g)) * u
    return h @ Wd.T


def _small_inputs(T=9, H=32, E=6, k=3, I=16, Is=0, seed=1, zipf=0.0):
    cfg = MoEConfig("t", T=T, H=H, E=E, k=k, I=I, I_shared=Is, dtype="f32", zipf_s=zipf)
    d = generate(cfg, seed=seed)
    return cfg, {n: to_np(v) for n, v in d.items()}


# ---------------------------------------------------------------- logits (a1)

def test_logits_match_float64_matmul(oracle):
    r = _rng(0)
    x = r.standard_normal((7, 40)).astype(np.float32)
    Wr = r.standard_normal((5, 40)).astype(np.float32)
    b = r.standard_normal(5).astype(np.float32)
    ref = (x.astype(np.float64) @ Wr.astype(np.float64).T + b).astype(np.float32)
    got = oracle.router_logits(x, Wr, b)
    np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-6)
    got0 = oracle.router_logits(x, Wr, None)
    np.testing.assert_allclose(got0, (x.astype(np.float64) @ Wr.astype(np.float64).T),
                               rtol=1e-6, atol=1e-6)


# ---------------------------------------------------------------- top-k (a2)

@pytest.mark.parametrize("E,k", [(8, 2), (16, 16), (40, 7), (512, 10), (5, 1)])
def test_topk_ids_match_stable_sort(oracle, E, k):
    """Ties (many, from small integers) go to the lowest index, ids in
    descending score order: exactly a stable sort of the negated logits."""
    r = _rng(E * 31 + k)
    logits = r.integers(-3, 4, size=(50, E)).astype(np.float32)
    ids, _ = oracle.route(logits, k, renorm=1)
    ref = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    np.testing.assert_array_equal(ids, ref)


def test_topk_all_equal_logits(oracle):
    logits = np.full((4, 12), 0.25, np.float32)
    ids, w = oracle.route(logits, 5, renorm=1)
    np.testing.assert_array_equal(ids, np.tile(np.arange(5), (4, 1)))
    np.testing.assert_allclose(w, np.full((4, 5), 1 / 5), rtol=0, atol=1e-7)


def test_topk_k_equals_E_is_permutation(oracle):
    logits = _rng(3).standard_normal((6, 9)).astype(np.float32)
    ids, w = oracle.route(logits, 9, renorm=1)
    for row in ids:
        assert sorted(row.tolist()) == list(range(9))
    # renormalised over all E == the plain softmax
    from scipy.special import softmax
    ref = np.take_along_axis(softmax(logits.astype(np.float64), axis=1), ids, axis=1)
    np.testing.assert_allclose(w, ref, rtol=0, atol=1e-7)


# ---------------------------------------------------------------- weights (a2)

def test_weights_renorm_sum_to_one_and_match_softmax(oracle):
    from scipy.special import softmax
    logits = (2.0 * _rng(4).standard_normal((64, 32))).astype(np.float32)
    ids, w = oracle.route(logits, 6, renorm=1)
    np.testing.assert_allclose(w.astype(np.float64).sum(1), 1.0, atol=1e-6)
    sel = np.take_along_axis(logits.astype(np.float64), ids, axis=1)
    np.testing.assert_allclose(w, softmax(sel, axis=1), atol=1e-7, rtol=0)
    assert np.all(np.diff(sel, axis=1) <= 0)  # descending score order


def test_weights_no_renorm_is_full_softmax(oracle):
    from scipy.special import softmax
    logits = _rng(5).standard_normal((20, 16)).astype(np.float32)
    ids, w = oracle.route(logits, 4, renorm=0)
    full = softmax(logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(full, ids, axis=1), atol=1e-7, rtol=0)
    assert np.all(w.sum(1) < 1.0)


def test_weights_k1_is_exactly_one(oracle):
    logits = _rng(6).standard_normal((10, 7)).astype(np.float32)
    ids, w = oracle.route(logits, 1, renorm=1)
    assert np.all(w == 1.0)
    np.testing.assert_array_equal(ids[:, 0], np.argmax(logits, axis=1))


# ------------------------------------------- group-limited top-k (a2, DeepSeek form)

def _np_grouped_topk(logits, k, n_group, topk_group):
    """Brute force in numpy: a group's score is its largest logit; the
    topk_group best groups are kept (lower group index among equals); then a
    stable sort of the negated logits of the kept experts."""
    T, E = logits.shape
    G = E // n_group
    score = logits.reshape(T, n_group, G).max(axis=2)
    order = np.argsort(-score, axis=1, kind="stable")[:, :topk_group]
    keep = np.zeros((T, n_group), bool)
    np.put_along_axis(keep, order, True, axis=1)
    masked = np.where(np.repeat(keep, G, axis=1), logits, -np.inf)
    return np.argsort(-masked, axis=1, kind="stable")[:, :k]


@pytest.mark.parametrize("E,k,n_group,topk_group", [(16, 3, 4, 2), (64, 8, 8, 3), (256, 8, 8, 4),
                                                    (12, 5, 3, 2), (32, 6, 16, 5)])
def test_grouped_topk_matches_bruteforce(oracle, E, k, n_group, topk_group):
    """Small integer logits give ties inside groups, between group scores and
    across groups; ids and renormalised weights against the definition."""
    from scipy.special import softmax
    r = _rng(E + 7 * k + n_group)
    logits = r.integers(-3, 4, size=(64, E)).astype(np.float32)
    ids, w = oracle.route_grouped(logits, k, 1, n_group, topk_group)
    np.testing.assert_array_equal(ids, _np_grouped_topk(logits, k, n_group, topk_group))
    sel = np.take_along_axis(logits.astype(np.float64), ids, axis=1)
    np.testing.assert_allclose(w, softmax(sel, axis=1), atol=1e-7, rtol=0)


def test_grouped_topk_reduces_to_plain_topk(oracle):
    """Keeping every group, or groups of one expert with topk_group = k, is the
    plain top-k (the Mixtral case of the same router); renorm = 0 keeps the
    full softmax."""
    from scipy.special import softmax
    logits = _rng(8).standard_normal((40, 32)).astype(np.float32)
    plain = np.argsort(-logits, axis=1, kind="stable")[:, :6]
    full = softmax(logits.astype(np.float64), axis=1)
    for n_group, topk_group in ((2, 2), (8, 8), (32, 6)):
        ids, w = oracle.route_grouped(logits, 6, 0, n_group, topk_group)
        np.testing.assert_array_equal(ids, plain)
        np.testing.assert_allclose(w, np.take_along_axis(full, ids, axis=1), atol=1e-7, rtol=0)


def test_grouped_topk_stays_in_kept_groups(oracle):
    logits = (3.0 * _rng(9).standard_normal((50, 64))).astype(np.float32)
    ids, _ = oracle.route_grouped(logits, 8, 1, 8, 2)
    groups = ids // 8
    assert all(len(set(row.tolist())) <= 2 for row in groups)
    np.testing.assert_array_equal(ids[:, 0], np.argmax(logits, axis=1))


# ---------------------------------------------------------------- permute (a3)

@pytest.mark.parametrize("T,E,k,shared", [(37, 8, 2, 0), (100, 16, 4, 1), (1, 4, 4, 0),
                                          (64, 512, 10, 0), (0, 5, 2, 1)])
def test_permute_is_stable_counting_sort(oracle, T, E, k, shared):
    r = _rng(T + E + k)
    ids = np.stack([r.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if T else \
        np.zeros((0, k), np.int32)
    off, gidx, spos = oracle.permute(ids, E, has_shared=shared)
    flat = ids.reshape(-1)
    cnt = np.bincount(flat, minlength=E)
    np.testing.assert_array_equal(off[:E + 1], np.concatenate([[0], np.cumsum(cnt)]))
    assert off[E + 1] == T * k + (T if shared else 0)
    assert off[E] == T * k
    # a stable sort by expert id of the slots 0..T*k-1
    np.testing.assert_array_equal(gidx, np.argsort(flat, kind="stable"))
    # bijection and inverse
    assert sorted(gidx.tolist()) == list(range(T * k))
    np.testing.assert_array_equal(gidx[spos], np.arange(T * k))
    # segments hold one expert, tokens ascending
    for e in range(E):
        seg = gidx[off[e]:off[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg // k) > 0)


# ---------------------------------------------------------------- FFN + combine

def test_dense_bruteforce_equals_sparse(oracle):
    """Evaluate every expert on every token (numpy float64), multiply by a
    dense [T,E] gate matrix that is zero outside each token's top-k (top-k by a
    stable library sort, weights by the library softmax), and compare."""
    from scipy.special import softmax
    cfg, d = _small_inputs(T=11, H=24, E=5, k=2, I=12, seed=2)
    x, Wr = d["x"].astype(np.float64), d["W_router"].astype(np.float64)
    Wg, Wu, Wd = (d[n].astype(np.float64) for n in ("W_gate", "W_up", "W_down"))
    logits = x @ Wr.T
    top = np.argsort(-logits.astype(np.float32), axis=1, kind="stable")[:, :cfg.k]
    dense_w = np.zeros((cfg.T, cfg.E))
    sw = softmax(np.take_along_axis(logits, top, axis=1), axis=1)
    np.put_along_axis(dense_w, top, sw, axis=1)
    all_out = np.stack([_np_swiglu_ffn(x, Wg[e], Wu[e], Wd[e]) for e in range(cfg.E)], 1)
    ref = np.einsum("te,teh->th", dense_w, all_out)
    y = oracle.forward(d["x"], d["W_router"], None, d["W_gate"], d["W_up"], d["W_down"],
                       cfg.k, renorm=1)
    rel = np.abs(y - ref).max() / np.abs(ref).max()
    assert rel < 1e-5, rel


def test_k_equals_E_uniform_is_mean_of_experts(oracle):
    """W_router = 0: every logit is 0, every weight 1/E, and y is the mean of
    the E expert FFNs."""
    cfg, d = _small_inputs(T=6, H=16, E=4, k=4, I=8, seed=3)
    Wr = np.zeros_like(d["W_router"])
    y = oracle.forward(d["x"], Wr, None, d["W_gate"], d["W_up"], d["W_down"], 4, renorm=1)
    x = d["x"].astype(np.float64)
    ref = np.mean([_np_swiglu_ffn(x, d["W_gate"][e].astype(np.float64),
                                  d["W_up"][e].astype(np.float64),
                                  d["W_down"][e].astype(np.float64)) for e in range(4)], axis=0)
    np.testing.assert_allclose(y, ref, rtol=1e-5, atol=1e-6)


def test_single_expert_is_dense_swiglu_in_torch_float64(oracle):
    cfg, d = _small_inputs(T=5, H=32, E=1, k=1, I=24, seed=4)
    y = oracle.forward(d["x"], d["W_router"], None, d["W_gate"], d["W_up"], d["W_down"], 1)
    x = torch.from_numpy(d["x"]).double()
    Wg, Wu, Wd = (torch.from_numpy(d[n][0]).double() for n in ("W_gate", "W_up", "W_down"))
    ref = (torch.nn.functional.silu(x @ Wg.T) * (x @ Wu.T)) @ Wd.T
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-5, atol=1e-6)


def test_shared_expert_adds_dense_ffn(oracle):
    cfg, d = _small_inputs(T=7, H=16, E=4, k=2, I=8, Is=12, seed=5)
    args = (d["x"], d["W_router"], None, d["W_gate"], d["W_up"], d["W_down"], 2)
    y_s = oracle.forward(*args, Wsg=d["Ws_gate"], Wsu=d["Ws_up"], Wsd=d["Ws_down"])
    y_0 = oracle.forward(*args)
    shared = _np_swiglu_ffn(d["x"].astype(np.float64), d["Ws_gate"].astype(np.float64),
                            d["Ws_up"].astype(np.float64), d["Ws_down"].astype(np.float64))
    np.testing.assert_allclose(y_s - y_0, shared, rtol=1e-4, atol=1e-5)


def test_token_permutation_equivariance(oracle):
    cfg, d = _small_inputs(T=10, H=16, E=5, k=2, I=8, seed=6)
    perm = _rng(7).permutation(cfg.T)
    args = (d["W_router"], None, d["W_gate"], d["W_up"], d["W_down"], 2)
    y = oracle.forward(d["x"], *args)
    yp = oracle.forward(np.ascontiguousarray(d["x"][perm]), *args)
    np.testing.assert_array_equal(yp, y[perm])


def test_stages_compose_to_forward(oracle):
    """route -> permute -> expert_h -> down_combine equals the forward pass."""
    cfg, d = _small_inputs(T=13, H=16, E=5, k=3, I=8, Is=8, seed=8, zipf=1.1)
    y, inter = oracle.forward(d["x"], d["W_router"], d["router_bias"], d["W_gate"],
                              d["W_up"], d["W_down"], 3, Wsg=d["Ws_gate"], Wsu=d["Ws_up"],
                              Wsd=d["Ws_down"], want_intermediates=True)
    ids, w = oracle.route(oracle.router_logits(d["x"], d["W_router"], d["router_bias"]), 3)
    np.testing.assert_array_equal(ids, inter["ids"])
    off, gidx, spos = oracle.permute(ids, cfg.E, has_shared=1)
    h, hs = oracle.expert_h(d["x"], off, gidx, d["W_gate"], d["W_up"], 3, d["Ws_gate"],
                            d["Ws_up"])
    y2 = oracle.down_combine(h, off, spos, ids, w, d["W_down"], hs, d["Ws_down"])
    np.testing.assert_allclose(y2, y, rtol=1e-6, atol=1e-7)


def test_closed_form_golden(oracle):
    with open(os.path.join(GOLDEN, "closed_form_two_tokens.json")) as f:
        g = json.load(f)
    env = {"ln3": math.log(3.0), "e5": math.exp(-5.0), "log": math.log}

    def ev(a):
        if isinstance(a, list):
            return [ev(v) for v in a]
        return float(eval(a, {"__builtins__": {}}, env))

    arr = lambda n: np.ascontiguousarray(np.array(ev(g[n]), np.float32))
    y, inter = oracle.forward(arr("x"), arr("W_router"), None, arr("W_gate"), arr("W_up"),
                              arr("W_down"), g["k"], renorm=g["renorm"],
                              want_intermediates=True)
    np.testing.assert_array_equal(inter["ids"], np.array(g["expect_ids"]))
    np.testing.assert_allclose(inter["w"], np.array(ev(g["expect_w"])), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(y, np.array(ev(g["expect_y"])), rtol=2e-6, atol=1e-6)


def test_generated_inputs_keep_router_margin():
    """The seeded generator's promise: top-(k+1) adjacent logit gaps >= 1e-3."""
    from moe_inputs import MARGIN
    cfg = MoEConfig("m", T=200, H=64, E=32, k=4, I=16, zipf_s=1.1)
    d = generate(cfg, seed=0)
    lg = d["x"].double() @ d["W_router"].double().T + d["router_bias"].double()
    top = torch.topk(lg, cfg.k + 1, dim=1).values
    assert float((top[:, :-1] - top[:, 1:]).min()) >= MARGIN
