"""Pins for the oracle's FP8 expert path (CPU only).

E4M3 is the OCP 8-bit floating-point format (sign, 4 exponent bits with bias 7,
3 mantissa bits, no infinities, largest finite 448); torch's float8_e4m3fn is an
independent implementation of it and serves as the library routine for the
encoding (round to nearest, ties to even) and the decoding. The row rule (the
smallest power-of-two scale that keeps a row's largest magnitude within 448) is
checked by its defining inequalities. The FP8 layer (the composition of these
with the pinned stages of the bf16 oracle) is pinned against a second
computation of the same definition written independently here: exponents from
float64 comparisons, codes from torch's float8_e4m3fn conversion, bf16 from
torch, and a float64 dense evaluation of every expert on every token with the
gate weights masked to the top-k. Planted mistakes in the oracle's FP8
composition (quantization axis, skipped or doubled scales, a missing bf16
rounding) are shown to fail that pin.
"""
import inspect

import numpy as np
import pytest
import torch

import oracle as oracle_mod
from moe_inputs import MoEConfig, generate
from oracle import to_np


def _torch_encode(v):
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_every_code_matches_torch(oracle):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    assert np.isnan(got[[0x7F, 0xFF]]).all() and got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_encode_round_trips_and_rounds_ties_to_even(oracle):
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    vals = oracle.e4m3_decode(codes)
    np.testing.assert_array_equal(oracle.e4m3_encode(vals), codes)
    # midpoints of consecutive positive values: ties to the even mantissa
    pos = np.sort(np.unique(vals[vals > 0]).astype(np.float64))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(mids), _torch_encode(mids))
    np.testing.assert_array_equal(oracle.e4m3_encode(-mids), _torch_encode(-mids))
    assert (oracle.e4m3_encode(mids) % 2 == 0).all()


@pytest.mark.parametrize("seed", [0, 1])
def test_encode_random_values_match_torch(oracle, seed):
    r = np.random.default_rng(seed)
    lin = r.uniform(-448, 448, 20000).astype(np.float32)
    logs = (r.choice([-1, 1], 20000) * 2.0 ** r.uniform(-12, 8.8, 20000)).astype(np.float32)
    for v in (lin, logs):
        np.testing.assert_array_equal(oracle.e4m3_encode(v), _torch_encode(v))


def test_encode_saturates_beyond_448(oracle):
    v = np.array([448.0, 463.9, 464.0, 1e6, -1e6], np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(v), [0x7E, 0x7E, 0x7E, 0x7E, 0xFE])


def test_quantize_rows_follow_the_rule(oracle):
    r = np.random.default_rng(3)
    rows = [r.standard_normal(64) * 10.0 ** r.uniform(-6, 6) for _ in range(200)]
    rows += [np.zeros(64), np.full(64, 448.0), np.full(64, 1.75 * 2.0 ** -3),
             np.full(64, 1.7500001 * 2.0 ** -3), np.full(64, 3.0e-38)]
    src = np.stack(rows).astype(np.float32)
    q, sc = oracle.quantize_rows_e4m3(src)
    amax = np.abs(src).max(1).astype(np.float64)
    m, e = np.frexp(sc.astype(np.float64))
    assert (m == 0.5).all()  # every scale is a power of two
    e = e - 1
    nz = amax > 0
    assert (amax[nz] <= 448.0 * 2.0 ** e[nz]).all()
    # smallest such power of two, unless held at 2^-126
    assert ((amax[nz] > 448.0 * 2.0 ** (e[nz] - 1)) | (e[nz] == -126)).all()
    assert sc[~nz].tolist() == [1.0] and (q[~nz] == 0).all()
    # the codes are the library encoding of the scaled row
    scaled = (src.astype(np.float64) / sc[:, None].astype(np.float64)).astype(np.float32)
    np.testing.assert_array_equal(q, _torch_encode(scaled))
    # 1.75 * 2^-3 = 448 * 2^-11 exactly; a hair above needs 2^-10
    assert e[-3] == -11 and e[-2] == -10 and e[-1] == -126


def test_bf16_round_matches_torch(oracle):
    v = (np.random.default_rng(4).standard_normal(10000) * 3).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(oracle.bf16_round(v), ref)


def test_fp8_layer_is_close_to_the_unquantized_layer(oracle):
    """E4M3 keeps 3 mantissa bits: each quantized operand is within 2^-4
    relative of its value, so the layer moves by a few percent (rel-L2), and
    routing is untouched (it runs on the unquantized x)."""
    cfg = MoEConfig("q", T=40, H=256, E=8, k=2, I=128, I_shared=128, dtype="f32")
    d = {n: to_np(v) for n, v in generate(cfg, seed=2).items()}
    args = (d["x"], d["W_router"], d["router_bias"], d["W_gate"], d["W_up"], d["W_down"], cfg.k)
    sh = dict(Wsg=d["Ws_gate"], Wsu=d["Ws_up"], Wsd=d["Ws_down"])
    y8, inter8 = oracle.forward_fp8(*args, **sh, want_intermediates=True)
    y, inter = oracle.forward(*args, 1, d["Ws_gate"], d["Ws_up"], d["Ws_down"],
                              want_intermediates=True)
    np.testing.assert_array_equal(inter8["ids"], inter["ids"])
    rel = np.linalg.norm(y8 - y) / np.linalg.norm(y)
    assert 1e-3 < rel < 0.08, rel


# ---------------------------------------------------------------- independent pin

def _rows_e4m3(a):
    """Row quantization written from the definition, independently of the
    oracle: scale 2^e with e the smallest integer such that max|row| <= 448 *
    2^e (e >= -126; a zero row keeps e = 0), codes = torch float8_e4m3fn of
    row / 2^e (exact power-of-two scaling). Returns (codes, scales, values as
    float64 = decoded codes * scale)."""
    a = np.asarray(a, np.float32)
    amax = np.abs(a).max(-1).astype(np.float64)
    e = np.zeros(amax.shape, np.int64)
    nz = amax > 0
    c = np.ceil(np.log2(amax[nz] / 448.0)).astype(np.int64)
    # exact correction of the log2 candidate against the defining inequalities
    c = np.where(amax[nz] > 448.0 * np.exp2(c.astype(np.float64)), c + 1, c)
    c = np.where(amax[nz] <= 448.0 * np.exp2((c - 1).astype(np.float64)), c - 1, c)
    e[nz] = np.maximum(c, -126)
    sc = np.exp2(e.astype(np.float64))
    codes = torch.from_numpy((a.astype(np.float64) / sc[..., None]).astype(np.float32)).to(
        torch.float8_e4m3fn)
    vals = codes.to(torch.float64).numpy() * sc[..., None]
    return codes.view(torch.uint8).numpy(), sc.astype(np.float32), vals


def _bf16(a64):
    """float64 -> fp32 -> bf16 (torch's round-to-nearest-even), as float64."""
    return torch.from_numpy(np.asarray(a64, np.float64)).float().bfloat16().double().numpy()


def _route64(x, Wr, bias, k):
    """Top-k on float64 logits (stable: lower index first among equals) and
    the softmax over the chosen k, all in float64."""
    lg = x.astype(np.float64) @ Wr.astype(np.float64).T
    if bias is not None:
        lg = lg + bias.astype(np.float64)
    ids = np.argsort(-lg, axis=1, kind="stable")[:, :k].astype(np.int32)
    top = np.take_along_axis(lg, ids, 1)
    p = np.exp(top - top[:, :1])
    return ids, (p / p.sum(1, keepdims=True)).astype(np.float32)


def _fp8_layer_dense(x, ids, w, Wg, Wu, Wd, Wsg=None, Wsu=None, Wsd=None):
    """The FP8 layer's experts and combine evaluated densely in float64: every
    expert on every token, then a [T, E] gate matrix that is zero outside each
    token's top-k. Returns (y, h) with h [T, E, I] the bf16 activations."""
    T, H = x.shape
    E, I, _ = Wg.shape
    xd = _rows_e4m3(x)[2]
    Wgd = _rows_e4m3(Wg.reshape(E * I, H))[2].reshape(E, I, H)
    Wud = _rows_e4m3(Wu.reshape(E * I, H))[2].reshape(E, I, H)
    Wdd = _rows_e4m3(Wd.reshape(E * H, I))[2].reshape(E, H, I)
    g = np.einsum("th,eih->tei", xd, Wgd)
    u = np.einsum("th,eih->tei", xd, Wud)
    h = _bf16(g / (1.0 + np.exp(-g)) * u)
    hd = _rows_e4m3(h.reshape(T * E, I).astype(np.float32))[2].reshape(T, E, I)
    o = np.einsum("tei,ehi->teh", hd, Wdd)
    gate = np.zeros((T, E))
    np.put_along_axis(gate, ids.astype(np.int64), w.astype(np.float64), 1)
    y = np.einsum("te,teh->th", gate, o)
    if Wsg is not None:
        Is = Wsg.shape[0]
        gs = xd @ _rows_e4m3(Wsg)[2].T
        us = xd @ _rows_e4m3(Wsu)[2].T
        hs = _bf16(gs / (1.0 + np.exp(-gs)) * us)
        y = y + _rows_e4m3(hs.astype(np.float32))[2] @ _rows_e4m3(Wsd)[2].T
        assert Wsd.shape == (H, Is)
    return y, h


def _fp8_case(seed, shared=True, spread=False, T=40, H=256, E=8, k=2, I=128):
    """Seeded f32 layer inputs and float64 routing.

    spread: magnitudes that vary by up to 2^12 along both contraction axes,
    balanced so that every entry still matters: x column j times 2^-b_j with
    the W_gate / W_up columns j times 2^b_j (along H), and W_up row i times 2^s_i
    with the W_down column i times 2^-s_i (along I). E4M3 is a floating-point
    format, so a power-of-two scale decides a value's code only where the
    scaled value is subnormal (or saturates): with this spread, a per-row
    scale sends a row's small entries there while a per-column scale would not,
    which makes the quantization axis visible in h and y."""
    cfg = MoEConfig("q", T=T, H=H, E=E, k=k, I=I, I_shared=128 if shared else 0, dtype="f32")
    d = {n: to_np(v) for n, v in generate(cfg, seed=seed).items()}
    if spread:
        r = np.random.default_rng(seed)
        b = np.exp2(r.integers(0, 13, H)).astype(np.float32)
        d["x"] = np.ascontiguousarray(d["x"] / b)
        for n in ("W_gate", "W_up", "Ws_gate", "Ws_up"):
            if d[n] is not None:
                d[n] = np.ascontiguousarray(d[n] * b)
        for up, down in (("W_up", "W_down"), ("Ws_up", "Ws_down")):
            if d[up] is not None:
                sc = np.exp2(r.integers(0, 13, d[up].shape[-2])).astype(np.float32)
                d[up] = np.ascontiguousarray(d[up] * sc[:, None])
                d[down] = np.ascontiguousarray(d[down] / sc)
    ids, w = _route64(d["x"], d["W_router"], d["router_bias"], k)
    sh = (d["Ws_gate"], d["Ws_up"], d["Ws_down"]) if shared else (None, None, None)
    return d, ids, w, sh


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return max(float(np.abs(a - b).max()) / float(np.abs(b).max()),
               float(np.linalg.norm(a - b) / np.linalg.norm(b)))


@pytest.mark.parametrize("seed,shared,spread", [(5, True, False), (6, False, False),
                                               (9, True, True)])
def test_fp8_layer_matches_an_independent_dense_evaluation(oracle, seed, shared, spread):
    d, ids, w, sh = _fp8_case(seed, shared, spread)
    y_ref, h_ref = _fp8_layer_dense(d["x"], ids, w, d["W_gate"], d["W_up"], d["W_down"], *sh)
    y, inter = oracle.ffn_combine_fp8(d["x"], ids, w, d["W_gate"], d["W_up"], d["W_down"],
                                      *sh, want_intermediates=True)
    assert _rel(y, y_ref) <= 1e-5
    # the stored bf16 activations agree exactly at every routed position
    gidx = inter["gather_idx"]
    tok, rank = gidx // ids.shape[1], gidx % ids.shape[1]
    np.testing.assert_array_equal(inter["h"], h_ref[tok, ids[tok, rank]].astype(np.float32))
    # and the oracle's own row quantizer gives the independent codes and scales
    q, sc = oracle.quantize_rows_e4m3(inter["h"])
    q2, sc2, _ = _rows_e4m3(inter["h"])
    np.testing.assert_array_equal(q, q2)
    np.testing.assert_array_equal(sc, sc2)


def test_fp8_forward_routes_like_the_independent_router(oracle):
    d, ids, w, sh = _fp8_case(7)
    y, inter = oracle.forward_fp8(d["x"], d["W_router"], d["router_bias"], d["W_gate"],
                                  d["W_up"], d["W_down"], 2, 1, *sh, want_intermediates=True)
    np.testing.assert_array_equal(inter["ids"], ids)
    np.testing.assert_allclose(inter["w"], w, rtol=0, atol=1e-6)
    y_ref, _ = _fp8_layer_dense(d["x"], ids, w, d["W_gate"], d["W_up"], d["W_down"], *sh)
    assert _rel(y, y_ref) <= 1e-5


def test_fp8_rows_of_torch_match_the_oracle_on_extremes(oracle):
    r = np.random.default_rng(8)
    src = np.stack([r.standard_normal(32) * 10.0 ** r.uniform(-30, 30) for _ in range(300)]
                   + [np.zeros(32), np.full(32, 448.0), np.full(32, 449.0)]).astype(np.float32)
    q, sc = oracle.quantize_rows_e4m3(src)
    q2, sc2, _ = _rows_e4m3(src)
    np.testing.assert_array_equal(sc, sc2)
    np.testing.assert_array_equal(q, q2)


# Planted mistakes in a copy of the oracle's FP8 composition: each must fail the
# independent pin above (h exactly, y within 1e-5).
_T = "np.ascontiguousarray(np.swapaxes({0}, -1, -2))"
_COLS = _T.format("dq(" + _T.format("{0}") + ")")
FP8_MUTANTS = {
    "gate/up weights quantized along columns":
        ("Wgd, Wud, Wdd = dq(Wg), dq(Wu), dq(Wd)",
         "Wgd, Wud, Wdd = " + _COLS.format("Wg") + ", " + _COLS.format("Wu") + ", dq(Wd)"),
    "down weights quantized along columns":
        ("Wgd, Wud, Wdd = dq(Wg), dq(Wu), dq(Wd)",
         "Wgd, Wud, Wdd = dq(Wg), dq(Wu), " + _COLS.format("Wd")),
    "x quantized along columns": ("xd = dq(x)", "xd = " + _COLS.format("x")),
    "x not quantized": ("xd = dq(x)", "xd = x"),
    "h scale applied twice":
        ("y = self.down_combine(dq(hb),",
         "y = self.down_combine((lambda q, s: self.dequantize_rows_e4m3(q, s) * s[:, None])"
         "(*self.quantize_rows_e4m3(hb)),"),
    "h not rounded to bf16": ("hb = self.bf16_round(h)", "hb = h"),
    "h not quantized": ("y = self.down_combine(dq(hb),", "y = self.down_combine(hb,"),
    "h quantized along columns":
        ("y = self.down_combine(dq(hb),", "y = self.down_combine(" + _COLS.format("hb") + ","),
    "shared h not quantized": ("dq(hsb) if has_s else None", "hsb if has_s else None"),
    "W_down not quantized": ("Wgd, Wud, Wdd = dq(Wg), dq(Wu), dq(Wd)",
                             "Wgd, Wud, Wdd = dq(Wg), dq(Wu), Wd"),
}


def _mutant(old, new):
    src = inspect.getsource(oracle_mod.ffn_combine_fp8)
    assert src.count(old) == 1, old
    ns = dict(vars(oracle_mod))
    exec(compile(src.replace(old, new), "<fp8 mutant>", "exec"), ns)
    return ns["ffn_combine_fp8"]


def _pin_errors(fn, oracle, d, ids, w, sh, y_ref, h_ref):
    """(relative y error, fraction of routed h values that differ)."""
    y, inter = fn(oracle, d["x"], ids, w, d["W_gate"], d["W_up"], d["W_down"], *sh,
                  want_intermediates=True)
    gidx = inter["gather_idx"]
    tok, rank = gidx // ids.shape[1], gidx % ids.shape[1]
    h_bad = float(np.mean(inter["h"] != h_ref[tok, ids[tok, rank]].astype(np.float32)))
    return _rel(y, y_ref), h_bad


@pytest.mark.parametrize("name", sorted(FP8_MUTANTS))
def test_fp8_planted_mistake_is_caught(oracle, name):
    d, ids, w, sh = _fp8_case(9, spread=True)
    y_ref, h_ref = _fp8_layer_dense(d["x"], ids, w, d["W_gate"], d["W_up"], d["W_down"], *sh)
    rel, h_bad = _pin_errors(_mutant(*FP8_MUTANTS[name]), oracle, d, ids, w, sh, y_ref, h_ref)
    assert rel > 1e-3 or h_bad > 1e-3, (name, rel, h_bad)
    # the unmutated composition passes the same check
    rel0, h_bad0 = _pin_errors(oracle_mod.ffn_combine_fp8, oracle, d, ids, w, sh, y_ref, h_ref)
    assert rel0 <= 1e-5 and h_bad0 == 0.0
