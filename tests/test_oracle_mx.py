"""Pins for the oracle's MXFP8 expert path (CPU only).

The block rule is restated here from its definition with float64 arithmetic
and torch's float8_e4m3fn conversion (an independent implementation of E4M3's
round to nearest even): blocks of 32 consecutive elements along the last axis,
scale 2^e with e = floor(log2(amax)) - 8 held in [-127, 127] (e = -127 for a
block of zeros), codes of v / 2^e clamped to +-448. Closed-form cases fix the
scale byte, the saturation and the block boundaries. The MXFP8 layer (the
oracle's composition of the pinned bf16 stages with this quantization between
them) is pinned against a float64 dense evaluation of the same definition
written here, and planted mistakes in that composition (block size, block axis,
scale rule, clamping, skipped or doubled quantization, a bf16 step before h's
quantization) are shown to fail the pin.
"""
import inspect

import numpy as np
import pytest
import torch

import oracle as oracle_mod
from moe_inputs import MoEConfig, generate
from oracle import mx_scale_cols, to_np
from test_oracle_fp8 import _bf16, _rel, _route64


def _blocks_mx(a, block=32):
    """Independent MX quantization along the last axis: (codes uint8, scale
    bytes uint8 [..., cols / block], values float64 = decoded code * 2^e)."""
    a = np.asarray(a, np.float32)
    shp = a.shape
    b = a.astype(np.float64).reshape(shp[:-1] + (shp[-1] // block, block))
    amax = np.abs(b).max(-1)
    _, ex = np.frexp(amax)  # amax = m * 2^ex, m in [0.5, 1)
    e = np.where(amax > 0, np.clip(ex - 1 - 8, -127, 127), -127).astype(np.int64)
    scaled = np.clip(b / np.exp2(e.astype(np.float64))[..., None], -448.0, 448.0)
    codes = torch.from_numpy(scaled.astype(np.float32)).to(torch.float8_e4m3fn)
    vals = codes.to(torch.float64).numpy() * np.exp2(e.astype(np.float64))[..., None]
    return (codes.view(torch.uint8).numpy().reshape(shp), (e + 127).astype(np.uint8),
            vals.reshape(shp))


def _qdq(a):
    """bf16 value of each element after MX quantization (float64)."""
    return _bf16(_blocks_mx(a)[2])


def _mx_rows(r, n, cols, spread):
    """n rows of `cols` values whose 32-element blocks differ in magnitude by
    up to 2^spread, with some blocks of zeros, negative zeros and tiny values."""
    blk = r.standard_normal((n, cols // 32, 32)) * np.exp2(
        r.integers(-spread, spread + 1, (n, cols // 32, 1)))
    blk[0, 0] = 0.0
    blk[0, 1] = -0.0
    blk[1, 0, :5] = [1e-30, -1e-38, 3e-45, 0.0, -2e-40]
    return blk.reshape(n, cols).astype(np.float32)


def test_mx_scale_cols():
    assert [mx_scale_cols(c) for c in (32, 512, 544, 4096, 7168)] == [16, 16, 32, 128, 224]


@pytest.mark.parametrize("seed,spread", [(0, 3), (1, 40)])
def test_quantize_mx_matches_the_independent_rule(oracle, seed, spread):
    r = np.random.default_rng(seed)
    src = _mx_rows(r, 64, 256, spread)
    q, sc = oracle.quantize_mx(src)
    q2, sc2, vals = _blocks_mx(src)
    np.testing.assert_array_equal(q, q2)
    np.testing.assert_array_equal(sc[:, :8], sc2)
    assert (sc[:, 8:] == 0).all()  # padding of the scale rows
    np.testing.assert_array_equal(oracle.dequantize_mx(q, sc), vals.astype(np.float32))
    assert (oracle.dequantize_mx(q, sc).astype(np.float64) == vals).all()


def test_quantize_mx_closed_forms(oracle):
    src = np.zeros((6, 64), np.float32)
    src[0, :32] = 1.0              # amax 1 = 2^0: e = -8, 1.0 / 2^-8 = 256 = E4M3 2^8
    src[1, 0] = 3.75               # floor(log2 3.75) = 1: e = -7, 3.75 * 128 = 480 -> 448
    src[1, 1] = 1.0                # 128 = 2^7 exactly
    src[2, 32] = 2.0 ** -130       # fp32 subnormal amax: e held at -127
    src[3, :32] = np.arange(32)    # amax 31: e = -4, element 31 -> 496 -> 448
    src[4, 31] = 1.0               # blocks end after 32 elements:
    src[4, 32] = 1000.0            # this block's scale does not reach element 31
    src[5, 0] = -0.0
    q, sc = oracle.quantize_mx(src)
    assert sc[0, :2].tolist() == [119, 0] and (q[0, :32] == 0x78).all()
    assert sc[1, 0] == 120 and q[1, 0] == 0x7E and q[1, 1] == 0x70
    assert sc[2, 1] == 0 and q[2, 32] == 0x20  # 2^-130 * 2^127 = 2^-3: E = 4, m = 0
    assert sc[3, 0] == 123 and q[3, 31] == 0x7E and q[3, 1] == 0x58  # 1 * 16 = 2^4
    assert sc[4, :2].tolist() == [119, 128] and q[4, 31] == 0x78
    assert q[5, 0] == 0x80 and sc[5, 0] == 0  # a zero block: e = -127, sign kept
    v = oracle.dequantize_mx(q, sc)
    assert v[1, 0] == 3.5 and v[3, 31] == 28.0 and v[2, 32] == np.float32(2.0 ** -130)


def test_quantize_mx_is_blockwise(oracle):
    """Changing one block changes only that block's codes and scale."""
    r = np.random.default_rng(3)
    src = _mx_rows(r, 4, 128, 6)
    q, sc = oracle.quantize_mx(src)
    src2 = src.copy()
    src2[2, 64:96] *= 1000.0
    q2, sc2 = oracle.quantize_mx(src2)
    diff = np.argwhere(q2 != q)
    assert diff.size and (diff[:, 0] == 2).all() and (diff[:, 1] // 32 == 2).all()
    assert [tuple(i) for i in np.argwhere(sc2 != sc)] == [(2, 2)]


def test_qdq_mx_is_the_bf16_of_the_block_value(oracle):
    r = np.random.default_rng(4)
    src = _mx_rows(r, 32, 256, 60)
    np.testing.assert_array_equal(oracle.qdq_mx(src), _qdq(src).astype(np.float32))


def test_mx_layer_is_close_to_the_unquantized_layer(oracle):
    cfg = MoEConfig("q", T=40, H=256, E=8, k=2, I=128, I_shared=128, dtype="f32")
    d = {n: to_np(v) for n, v in generate(cfg, seed=2).items()}
    args = (d["x"], d["W_router"], d["router_bias"], d["W_gate"], d["W_up"], d["W_down"], cfg.k)
    ym, inter = oracle.forward_mx(*args, 1, d["Ws_gate"], d["Ws_up"], d["Ws_down"],
                                  want_intermediates=True)
    y, inter0 = oracle.forward(*args, 1, d["Ws_gate"], d["Ws_up"], d["Ws_down"],
                               want_intermediates=True)
    np.testing.assert_array_equal(inter["ids"], inter0["ids"])
    rel = np.linalg.norm(ym - y) / np.linalg.norm(y)
    assert 1e-3 < rel < 0.08, rel


# ---------------------------------------------------------------- independent pin

def _mx_layer_dense(x, ids, w, Wg, Wu, Wd, Wsg=None, Wsu=None, Wsd=None):
    """The MXFP8 layer's experts and combine evaluated densely in float64:
    every expert on every token, then a [T, E] gate matrix that is zero
    outside each token's top-k. Returns (y, h) with h [T, E, I] the quantized
    activations (bf16 values)."""
    T, H = x.shape
    E, I, _ = Wg.shape
    xm = _qdq(x)
    Wgm = _qdq(Wg.reshape(E * I, H)).reshape(E, I, H)
    Wum = _qdq(Wu.reshape(E * I, H)).reshape(E, I, H)
    Wdm = _qdq(Wd.reshape(E * H, I)).reshape(E, H, I)
    g = np.einsum("th,eih->tei", xm, Wgm)
    u = np.einsum("th,eih->tei", xm, Wum)
    h32 = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
    hm = _qdq(h32.reshape(T * E, I)).reshape(T, E, I)
    o = np.einsum("tei,ehi->teh", hm, Wdm)
    gate = np.zeros((T, E))
    np.put_along_axis(gate, ids.astype(np.int64), w.astype(np.float64), 1)
    y = np.einsum("te,teh->th", gate, o)
    if Wsg is not None:
        gs = xm @ _qdq(Wsg).T
        us = xm @ _qdq(Wsu).T
        hs = (gs / (1.0 + np.exp(-gs)) * us).astype(np.float32)
        y = y + _qdq(hs) @ _qdq(Wsd).T
    return y, hm


def _mx_case(seed, shared=True, spread=False, T=64, H=256, E=8, k=2, I=128):
    """Seeded f32 layer inputs and float64 routing.

    spread: per-block magnitudes that vary by up to 2^12 along both contraction
    axes, balanced so every block still matters: x's 32-column block j times
    2^-b_j with the matching W_gate / W_up column block times 2^b_j (along H),
    and W_up's 32-row block i times 2^s_i with W_down's matching column block
    times 2^-s_i (along I). E4M3 is a floating-point format, so a block's scale
    decides a code only where a scaled value saturates or is subnormal; with
    this spread the blocks along the contraction axis hold unrelated maxima,
    which makes the block size and axis visible in h and y."""
    cfg = MoEConfig("q", T=T, H=H, E=E, k=k, I=I, I_shared=128 if shared else 0, dtype="f32")
    d = {n: to_np(v) for n, v in generate(cfg, seed=seed).items()}
    if spread:
        r = np.random.default_rng(seed)
        b = np.repeat(np.exp2(r.integers(0, 13, H // 32)), 32).astype(np.float32)
        b *= np.exp2(r.integers(0, 4, H)).astype(np.float32)  # within-block spread too
        d["x"] = np.ascontiguousarray(d["x"] / b)
        for n in ("W_gate", "W_up", "Ws_gate", "Ws_up"):
            if d[n] is not None:
                d[n] = np.ascontiguousarray(d[n] * b)
        for up, down in (("W_up", "W_down"), ("Ws_up", "Ws_down")):
            if d[up] is not None:
                n_i = d[up].shape[-2]
                sc = np.repeat(np.exp2(r.integers(0, 13, n_i // 32)), 32).astype(np.float32)
                sc *= np.exp2(r.integers(0, 4, n_i)).astype(np.float32)
                d[up] = np.ascontiguousarray(d[up] * sc[:, None])
                d[down] = np.ascontiguousarray(d[down] / sc)
    ids, w = _route64(d["x"], d["W_router"], d["router_bias"], k)
    sh = (d["Ws_gate"], d["Ws_up"], d["Ws_down"]) if shared else (None, None, None)
    return d, ids, w, sh


@pytest.mark.parametrize("seed,shared,spread", [(5, True, False), (6, False, False),
                                               (9, True, True)])
def test_mx_layer_matches_an_independent_dense_evaluation(oracle, seed, shared, spread):
    d, ids, w, sh = _mx_case(seed, shared, spread)
    y_ref, h_ref = _mx_layer_dense(d["x"], ids, w, d["W_gate"], d["W_up"], d["W_down"], *sh)
    y, inter = oracle.ffn_combine_mx(d["x"], ids, w, d["W_gate"], d["W_up"], d["W_down"],
                                     *sh, want_intermediates=True)
    assert _rel(y, y_ref) <= 1e-5
    # the quantized activations agree exactly at every routed position (the
    # float64 dense sums round to the same fp32 h here)
    gidx = inter["gather_idx"]
    tok, rank = gidx // ids.shape[1], gidx % ids.shape[1]
    same = inter["h"] == h_ref[tok, ids[tok, rank]].astype(np.float32)
    assert same.mean() > 0.9999, same.mean()


def test_mx_forward_routes_like_the_independent_router(oracle):
    d, ids, w, sh = _mx_case(7)
    y, inter = oracle.forward_mx(d["x"], d["W_router"], d["router_bias"], d["W_gate"],
                                 d["W_up"], d["W_down"], 2, 1, *sh, want_intermediates=True)
    np.testing.assert_array_equal(inter["ids"], ids)
    np.testing.assert_allclose(inter["w"], w, rtol=0, atol=1e-6)
    y_ref, _ = _mx_layer_dense(d["x"], ids, w, d["W_gate"], d["W_up"], d["W_down"], *sh)
    assert _rel(y, y_ref) <= 1e-5


# Planted mistakes in a copy of the oracle's MX composition, or in the block
# rule it calls: each must fail the independent pin above (h, or y within 1e-5).
_SWAP = "np.ascontiguousarray(np.swapaxes({0}, -1, -2))"
_COLS = _SWAP.format("mx(" + _SWAP.format("{0}") + ")")
MX_MUTANTS = {
    "gate/up weights blocked along columns":
        ("Wgm, Wum, Wdm = mx(Wg), mx(Wu), mx(Wd)",
         "Wgm, Wum, Wdm = " + _COLS.format("Wg") + ", " + _COLS.format("Wu") + ", mx(Wd)"),
    "down weights blocked along columns":
        ("Wgm, Wum, Wdm = mx(Wg), mx(Wu), mx(Wd)",
         "Wgm, Wum, Wdm = mx(Wg), mx(Wu), " + _COLS.format("Wd")),
    "x blocked along columns": ("xm = mx(x)", "xm = " + _COLS.format("x")),
    "x not quantized": ("xm = mx(x)", "xm = x"),
    "h not quantized": ("hm = mx(h)", "hm = h"),
    "h rounded to bf16 before its quantization": ("hm = mx(h)", "hm = mx(self.bf16_round(h))"),
    "h blocked along columns": ("hm = mx(h)", "hm = " + _COLS.format("h")),
    "shared h not quantized": ("hsm = mx(hs) if has_s else None", "hsm = hs if has_s else None"),
    "W_down not quantized": ("Wgm, Wum, Wdm = mx(Wg), mx(Wu), mx(Wd)",
                             "Wgm, Wum, Wdm = mx(Wg), mx(Wu), Wd"),
    "blocks of 16": ("mx = self.qdq_mx", "mx = _blocked_qdq(16)"),
    "blocks of 64": ("mx = self.qdq_mx", "mx = _blocked_qdq(64)"),
    "scale exponent floor(log2 amax) - 7": ("mx = self.qdq_mx", "mx = _blocked_qdq(32, 7)"),
    "no clamp at 448": ("mx = self.qdq_mx", "mx = _blocked_qdq(32, 8, False)"),
    "one scale per row": ("mx = self.qdq_mx", "mx = _row_qdq"),
}


def _blocked_qdq(block, emax=8, clamp=True):
    """A wrong variant of the block rule (block size, scale exponent or clamp)."""
    def f(a):
        a = np.asarray(a, np.float32)
        shp = a.shape
        b = a.astype(np.float64).reshape(shp[:-1] + (shp[-1] // block, block))
        amax = np.abs(b).max(-1)
        _, ex = np.frexp(amax)
        e = np.where(amax > 0, np.clip(ex - 1 - emax, -127, 127), -127).astype(np.float64)
        s = b / np.exp2(e)[..., None]
        if clamp:
            s = np.clip(s, -448.0, 448.0)
        v = torch.from_numpy(s.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64)
        v = v.numpy() * np.exp2(e)[..., None]
        return np.nan_to_num(_bf16(v.reshape(shp)), nan=1e30).astype(np.float32)
    return f


def _row_qdq(a):
    a = np.asarray(a, np.float32)
    return _blocked_qdq(a.shape[-1])(a)


def _mutant(old, new):
    src = inspect.getsource(oracle_mod.ffn_combine_mx)
    assert src.count(old) == 1, old
    ns = dict(vars(oracle_mod))
    ns.update(_blocked_qdq=_blocked_qdq, _row_qdq=_row_qdq)
    exec(compile(src.replace(old, new), "<mx mutant>", "exec"), ns)
    return ns["ffn_combine_mx"]


def _pin_errors(fn, oracle, d, ids, w, sh, y_ref, h_ref):
    """(relative y error, fraction of routed h values that differ)."""
    y, inter = fn(oracle, d["x"], ids, w, d["W_gate"], d["W_up"], d["W_down"], *sh,
                  want_intermediates=True)
    gidx = inter["gather_idx"]
    tok, rank = gidx // ids.shape[1], gidx % ids.shape[1]
    h_bad = float(np.mean(inter["h"] != h_ref[tok, ids[tok, rank]].astype(np.float32)))
    return _rel(y, y_ref), h_bad


@pytest.mark.parametrize("name", sorted(MX_MUTANTS))
def test_mx_planted_mistake_is_caught(oracle, name):
    d, ids, w, sh = _mx_case(9, spread=True)
    y_ref, h_ref = _mx_layer_dense(d["x"], ids, w, d["W_gate"], d["W_up"], d["W_down"], *sh)
    rel, h_bad = _pin_errors(_mutant(*MX_MUTANTS[name]), oracle, d, ids, w, sh, y_ref, h_ref)
    assert rel > 1e-3 or h_bad > 1e-3, (name, rel, h_bad)
    # the unmutated composition passes the same check
    rel0, h_bad0 = _pin_errors(oracle_mod.ffn_combine_mx, oracle, d, ids, w, sh, y_ref, h_ref)
    assert rel0 <= 1e-5 and h_bad0 <= 1e-4
