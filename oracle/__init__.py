"""CPU oracle of the MoE layer forward pass (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and its
binding) never loads it. ``build()`` compiles ``moe_oracle.cpp`` with the host
compiler into ``liboracle.so`` next to this file.

All functions take and return numpy arrays (fp32 / int32, C-contiguous).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_f = ctypes.POINTER(ctypes.c_float)
_i = ctypes.POINTER(ctypes.c_int32)
_L = ctypes.c_int64


def build(force: bool = False, extra_flags=()) -> str:
    """Compile the oracle (g++ -O2 -fopenmp, IEEE semantics: no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-fopenmp", "-fPIC", "-shared",
               "-ffp-contract=off", *extra_flags, _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _declare(lib):
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_router_logits.argtypes = [_f, _f, _f, _L, _L, _L, _f]
    lib.oracle_route.argtypes = [_f, _L, _L, _L, ctypes.c_int, _i, _f]
    lib.oracle_route_grouped.argtypes = [_f, _L, _L, _L, ctypes.c_int, _L, _L, _i, _f]
    lib.oracle_permute.argtypes = [_i, _L, _L, _L, ctypes.c_int, _i, _i, _i]
    lib.oracle_expert_h.argtypes = [_f, _i, _i, _f, _f, _L, _L, _L, _L, _L, _f, _f, _f, _L, _f]
    lib.oracle_down_combine.argtypes = [_f, _i, _i, _i, _f, _f, _L, _L, _L, _L, _L, _f, _f,
                                        _L, _f]
    lib.oracle_ffn_combine.argtypes = [_f, _i, _f, _f, _f, _f, _L, _L, _L, _L, _L, _f, _f,
                                       _f, _L, _f]
    lib.oracle_moe_forward.argtypes = [_f, _f, _f, _f, _f, _f, _f, _f, _f, _L, _L, _L, _L, _L,
                                       _L, ctypes.c_int, _f, _f, _i, _f]
    _u8 = ctypes.POINTER(ctypes.c_uint8)
    lib.oracle_e4m3_decode.argtypes = [_u8, _L, _f]
    lib.oracle_e4m3_encode.argtypes = [_f, _L, _u8]
    lib.oracle_quantize_rows_e4m3.argtypes = [_f, _L, _L, _u8, _f]
    lib.oracle_bf16_round.argtypes = [_f, _L, _f]
    lib.oracle_quantize_mx.argtypes = [_f, _L, _L, _L, _u8, _u8]
    for n in ("oracle_e4m3_decode", "oracle_e4m3_encode", "oracle_quantize_rows_e4m3",
              "oracle_bf16_round", "oracle_quantize_mx"):
        getattr(lib, n).restype = None
    for n in ("oracle_router_logits", "oracle_route", "oracle_route_grouped", "oracle_permute",
              "oracle_expert_h",
              "oracle_down_combine", "oracle_ffn_combine", "oracle_moe_forward"):
        getattr(lib, n).restype = None
    return lib


def load(path: str | None = None):
    """Load (building first if needed) and return the ctypes library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        build()
        _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


class Oracle:
    """numpy-facing wrapper around one loaded oracle library."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    @staticmethod
    def _pf(a):
        if a is None:
            return None
        assert a.dtype == np.float32 and a.flags.c_contiguous, (a.dtype, a.flags)
        return a.ctypes.data_as(_f)

    @staticmethod
    def _pi(a):
        assert a.dtype == np.int32 and a.flags.c_contiguous
        return a.ctypes.data_as(_i)

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def router_logits(self, x, Wr, bias=None):
        T, H = x.shape
        E = Wr.shape[0]
        out = np.empty((T, E), np.float32)
        self.lib.oracle_router_logits(self._pf(x), self._pf(Wr), self._pf(bias), T, H, E,
                                      self._pf(out))
        return out

    def route(self, logits, k, renorm=1):
        T, E = logits.shape
        ids = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float32)
        self.lib.oracle_route(self._pf(logits), T, E, k, int(renorm), self._pi(ids),
                              self._pf(w))
        return ids, w

    def route_grouped(self, logits, k, renorm=1, n_group=1, topk_group=1):
        """Top-k limited to the best topk_group of n_group contiguous expert
        groups (group score: the group's largest logit)."""
        T, E = logits.shape
        ids = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float32)
        self.lib.oracle_route_grouped(self._pf(logits), T, E, k, int(renorm), int(n_group),
                                      int(topk_group), self._pi(ids), self._pf(w))
        return ids, w

    def permute(self, ids, E, has_shared=0):
        T, k = ids.shape
        offsets = np.empty(E + 2, np.int32)
        gather_idx = np.empty(T * k, np.int32)
        slot_pos = np.empty(T * k, np.int32)
        self.lib.oracle_permute(self._pi(np.ascontiguousarray(ids)), T, E, k, int(has_shared),
                                self._pi(offsets), self._pi(gather_idx), self._pi(slot_pos))
        return offsets, gather_idx, slot_pos

    def expert_h(self, x, offsets, gather_idx, Wg, Wu, k, Wsg=None, Wsu=None):
        T, H = x.shape
        E, I, _ = Wg.shape
        Is = 0 if Wsg is None else Wsg.shape[0]
        h = np.empty((T * k, I), np.float32)
        hs = np.empty((T, Is), np.float32) if Is else None
        self.lib.oracle_expert_h(self._pf(x), self._pi(offsets), self._pi(gather_idx),
                                 self._pf(Wg), self._pf(Wu), T, H, E, k, I, self._pf(h),
                                 self._pf(Wsg), self._pf(Wsu), Is, self._pf(hs))
        return h, hs

    def down_combine(self, h, offsets, slot_pos, ids, w, Wd, hs=None, Wsd=None):
        T, k = ids.shape
        E, H, I = Wd.shape
        Is = 0 if Wsd is None else Wsd.shape[1]
        y = np.empty((T, H), np.float32)
        self.lib.oracle_down_combine(self._pf(h), self._pi(offsets), self._pi(slot_pos),
                                     self._pi(ids), self._pf(w), self._pf(Wd), T, H, E, k, I,
                                     self._pf(hs), self._pf(Wsd), Is, self._pf(y))
        return y

    def ffn_combine(self, x, ids, w, Wg, Wu, Wd, Wsg=None, Wsu=None, Wsd=None):
        T, H = x.shape
        k = ids.shape[1]
        E, I, _ = Wg.shape
        Is = 0 if Wsg is None else Wsg.shape[0]
        y = np.empty((T, H), np.float32)
        self.lib.oracle_ffn_combine(self._pf(x), self._pi(ids), self._pf(w), self._pf(Wg),
                                    self._pf(Wu), self._pf(Wd), T, H, E, k, I, self._pf(Wsg),
                                    self._pf(Wsu), self._pf(Wsd), Is, self._pf(y))
        return y

    def forward(self, x, Wr, bias, Wg, Wu, Wd, k, renorm=1, Wsg=None, Wsu=None, Wsd=None,
                want_intermediates=False):
        T, H = x.shape
        E, I, _ = Wg.shape
        Is = 0 if Wsg is None else Wsg.shape[0]
        y = np.empty((T, H), np.float32)
        logits = np.empty((T, E), np.float32)
        ids = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float32)
        self.lib.oracle_moe_forward(self._pf(x), self._pf(Wr), self._pf(bias), self._pf(Wg),
                                    self._pf(Wu), self._pf(Wd), self._pf(Wsg), self._pf(Wsu),
                                    self._pf(Wsd), T, H, E, k, I, Is, int(renorm),
                                    self._pf(y), self._pf(logits), self._pi(ids), self._pf(w))
        if want_intermediates:
            return y, dict(logits=logits, ids=ids, w=w)
        return y


def _u8p(a):
    assert a.dtype == np.uint8 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def ffn_combine_fp8(self, x, ids, w, Wg, Wu, Wd, Wsg=None, Wsu=None, Wsd=None,
                    want_intermediates=False):
    """The experts and the combine of the FP8 layer for given routing.

    Definition (the microscaled-FP8 serving of "Hosting Qwen on Blackwell",
    with one power-of-two scale per matrix row as the block): every tensor the
    layer stores between its steps is a bf16 activation (x as given, h after
    the SwiGLU), and every FP8 GEMM quantizes its operands on entry, one scale
    per row along the contraction axis:
      - each x row (over H) and each weight row (W_gate/W_up rows over H,
        W_down rows over I) is quantized to E4M3 with its scale;
      - h = bf16(silu(g) * u), g and u exact dot products of the dequantized
        rows (rounded to fp32, then to the bf16 activation);
      - each h row (over I) is quantized like x;
      - y = sum_r w_r * (W_down[e_r] . h_r) (+ the shared expert, weight 1) on
        the dequantized values.
    """
    E = Wg.shape[0]
    k = ids.shape[1]
    has_s = Wsg is not None
    offs, gidx, spos = self.permute(np.ascontiguousarray(ids, np.int32), E,
                                    1 if has_s else 0)
    dq = lambda a: self.dequantize_rows_e4m3(*self.quantize_rows_e4m3(a))
    xd = dq(x)
    Wgd, Wud, Wdd = dq(Wg), dq(Wu), dq(Wd)
    Wsgd, Wsud, Wsdd = (dq(Wsg), dq(Wsu), dq(Wsd)) if has_s else (None, None, None)
    h, hs = self.expert_h(xd, offs, gidx, Wgd, Wud, k, Wsgd, Wsud)
    hb = self.bf16_round(h)
    hsb = self.bf16_round(hs) if has_s else None
    y = self.down_combine(dq(hb), offs, spos, np.ascontiguousarray(ids, np.int32),
                          np.ascontiguousarray(w, np.float32), Wdd,
                          dq(hsb) if has_s else None, Wsdd)
    if want_intermediates:
        return y, dict(offsets=offs, gather_idx=gidx, h=hb, hs=hsb, h_f32=h, hs_f32=hs)
    return y


def mx_scale_cols(cols):
    """Bytes of MX scales per row of `cols` elements: one per block of 32,
    padded to a multiple of 16."""
    return 16 * ((cols // 32 + 15) // 16)


def ffn_combine_mx(self, x, ids, w, Wg, Wu, Wd, Wsg=None, Wsu=None, Wsd=None,
                   want_intermediates=False):
    """The experts and the combine of the MXFP8 layer for given routing.

    Definition (MXFP8 serving of Qwen3-235B, "Hosting Qwen on Blackwell",
    quantization section: weights converted statically; the 32-element blocks
    of "CuTeDSL at Perplexity", Blackwell quantization paragraph): every
    operand of the two expert GEMMs is quantized in blocks of 32 consecutive
    elements along the contraction axis (quantize_mx):
      - x rows over H, W_gate / W_up rows over H, W_down rows over I;
      - each operand enters its GEMM as the bf16 value of code * scale (equal
        to that value unless its block's scale is below 2^-117);
      - h = silu(g) * u rounded to fp32, g and u exact dot products; each h
        row is quantized over I the same way (from fp32, no bf16 step);
      - y = sum_r w_r * (W_down[e_r] . h_r) (+ the shared expert, weight 1).
    """
    E = Wg.shape[0]
    k = ids.shape[1]
    has_s = Wsg is not None
    offs, gidx, spos = self.permute(np.ascontiguousarray(ids, np.int32), E,
                                    1 if has_s else 0)
    mx = self.qdq_mx
    xm = mx(x)
    Wgm, Wum, Wdm = mx(Wg), mx(Wu), mx(Wd)
    Wsgm, Wsum, Wsdm = (mx(Wsg), mx(Wsu), mx(Wsd)) if has_s else (None, None, None)
    h, hs = self.expert_h(xm, offs, gidx, Wgm, Wum, k, Wsgm, Wsum)
    hm = mx(h)
    hsm = mx(hs) if has_s else None
    y = self.down_combine(hm, offs, spos, np.ascontiguousarray(ids, np.int32),
                          np.ascontiguousarray(w, np.float32), Wdm, hsm, Wsdm)
    if want_intermediates:
        return y, dict(offsets=offs, gather_idx=gidx, xm=xm, h_f32=h, hs_f32=hs, h=hm, hs=hsm)
    return y


def _mx_methods():
    """MXFP8 expert path (E4M3 codes, one E8M0 scale per block of 32)."""

    def quantize_mx(self, src):
        """src [..., cols] fp32, cols a multiple of 32 -> (codes uint8
        [..., cols], scales uint8 [..., mx_scale_cols(cols)])."""
        src = np.ascontiguousarray(src, np.float32)
        cols = src.shape[-1]
        assert cols % 32 == 0, cols
        rows = src.size // cols
        sk = mx_scale_cols(cols)
        q = np.empty(src.shape, np.uint8)
        sc = np.empty(src.shape[:-1] + (sk,), np.uint8)
        self.lib.oracle_quantize_mx(self._pf(src), rows, cols, sk, _u8p(q), _u8p(sc))
        return q, sc

    def dequantize_mx(self, q, scales):
        """code * 2^(scale byte - 127), exact in fp32 for every code and scale
        quantize_mx produces from finite fp32 values."""
        q = np.ascontiguousarray(q, np.uint8)
        cols = q.shape[-1]
        e = np.asarray(scales, np.int64)[..., :cols // 32] - 127
        v = self.e4m3_decode(q).astype(np.float64).reshape(q.shape[:-1] + (cols // 32, 32))
        v = v * np.ldexp(1.0, e)[..., None]
        return np.ascontiguousarray(v.reshape(q.shape).astype(np.float32))

    def qdq_mx(self, a):
        """The bf16 value of each element after MX quantization."""
        return self.bf16_round(self.dequantize_mx(*self.quantize_mx(a)))

    def forward_mx(self, x, Wr, bias, Wg, Wu, Wd, k, renorm=1, Wsg=None, Wsu=None, Wsd=None,
                   n_group=1, topk_group=1, want_intermediates=False):
        """The layer with MXFP8 expert weights: router and routing on x as in
        forward, then ffn_combine_mx."""
        lg = self.router_logits(x, Wr, bias)
        ids, w = self.route_grouped(lg, k, renorm, n_group, topk_group)
        y, inter = self.ffn_combine_mx(x, ids, w, Wg, Wu, Wd, Wsg, Wsu, Wsd,
                                       want_intermediates=True)
        if want_intermediates:
            return y, dict(logits=lg, ids=ids, w=w, **inter)
        return y

    return dict(quantize_mx=quantize_mx, dequantize_mx=dequantize_mx, qdq_mx=qdq_mx,
                ffn_combine_mx=ffn_combine_mx, forward_mx=forward_mx)


def _fp8_methods():
    """FP8 expert path (E4M3 codes, one power-of-two scale per row): the
    quantization primitives, and the layer as a composition of the pinned
    steps above with quantization between them."""

    def e4m3_decode(self, codes):
        codes = np.ascontiguousarray(codes, np.uint8)
        out = np.empty(codes.shape, np.float32)
        self.lib.oracle_e4m3_decode(_u8p(codes), codes.size, self._pf(out))
        return out

    def e4m3_encode(self, v):
        v = np.ascontiguousarray(v, np.float32)
        out = np.empty(v.shape, np.uint8)
        self.lib.oracle_e4m3_encode(self._pf(v), v.size, _u8p(out))
        return out

    def quantize_rows_e4m3(self, src):
        """src [..., cols] fp32 -> (codes uint8 [..., cols], scales fp32 [...])."""
        src = np.ascontiguousarray(src, np.float32)
        cols = src.shape[-1]
        rows = src.size // cols
        q = np.empty(src.shape, np.uint8)
        sc = np.empty(src.shape[:-1], np.float32)
        self.lib.oracle_quantize_rows_e4m3(self._pf(src), rows, cols, _u8p(q), self._pf(sc))
        return q, sc

    def dequantize_rows_e4m3(self, q, scale):
        return self.e4m3_decode(q) * np.asarray(scale, np.float32)[..., None]

    def bf16_round(self, a):
        a = np.ascontiguousarray(a, np.float32)
        out = np.empty(a.shape, np.float32)
        self.lib.oracle_bf16_round(self._pf(a), a.size, self._pf(out))
        return out

    def forward_fp8(self, x, Wr, bias, Wg, Wu, Wd, k, renorm=1, Wsg=None, Wsu=None, Wsd=None,
                    n_group=1, topk_group=1, want_intermediates=False):
        """The layer with E4M3 expert weights: router and routing on x as in
        forward, then ffn_combine_fp8."""
        lg = self.router_logits(x, Wr, bias)
        ids, w = self.route_grouped(lg, k, renorm, n_group, topk_group)
        y, inter = self.ffn_combine_fp8(x, ids, w, Wg, Wu, Wd, Wsg, Wsu, Wsd,
                                        want_intermediates=True)
        if want_intermediates:
            return y, dict(logits=lg, ids=ids, w=w, **inter)
        return y

    return dict(e4m3_decode=e4m3_decode, e4m3_encode=e4m3_encode,
                quantize_rows_e4m3=quantize_rows_e4m3,
                dequantize_rows_e4m3=dequantize_rows_e4m3, bf16_round=bf16_round,
                ffn_combine_fp8=ffn_combine_fp8, forward_fp8=forward_fp8)


for _n, _fn in {**_fp8_methods(), **_mx_methods()}.items():
    setattr(Oracle, _n, _fn)


def to_np(t):
    """torch tensor (any device, bf16/fp32/int) -> C-contiguous numpy fp32/int32."""
    if t is None:
        return None
    import torch
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16, torch.float32, torch.float64):
        return np.ascontiguousarray(t.to(torch.float32).numpy())
    return np.ascontiguousarray(t.to(torch.int32).numpy())
