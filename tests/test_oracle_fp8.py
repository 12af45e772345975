"""Pins for the oracle's FP8 expert path (CPU only).

E4M3 is the OCP 8-bit floating-point format (sign, 4 exponent bits with bias 7,
3 mantissa bits, no infinities, largest finite 448); torch's float8_e4m3fn is an
independent implementation of it and serves as the library routine for the
encoding (round to nearest, ties to even) and the decoding. The row rule (the
smallest power-of-two scale that keeps a row's largest magnitude within 448) is
checked by its defining inequalities. The FP8 layer is the composition of these
with the pinned stages of the bf16 oracle; its distance to the unquantized layer
is checked against what 3-bit mantissas allow.
"""
import numpy as np
import pytest
import torch

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
