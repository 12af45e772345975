"""GB300 (sm_103a) Mixture-of-Experts FFN layer forward pass.

The compute path is libmoe.so (CUDA kernels behind a C ABI, declared in
include/moe_api.h); this package only marshals torch tensors into it:

* ``_binding``: one Python function per C entry point, same names.
* ``MoELayer``: holds the expert weights on the GPU and a workspace, and runs
  ``moe_forward`` on the current torch stream.
"""
from __future__ import annotations

import torch

from ._binding import (  # noqa: F401
    EXPORTED, MOE_DTYPE_BF16, MOE_DTYPE_E4M3, MOE_DTYPE_F32, MOE_DTYPE_MXFP8,
    MOE_FLAG_TEST_SKIP_SIGNAL, MOE_OK, MOE_TILE_AUTO, MOE_TILE_DECODE, MOE_TILE_MEDIUM,
    MOE_TILE_PREFILL, STATUS_NAMES, MoEError, MoEProblem, down_combine, down_combine_noalloc,
    forward, forward_fp8, forward_mx, forward_single_launch, get_device_status,
    grouped_swiglu_gemm, load_library, make_problem, mx_scale_cols, permute, quantize_mx,
    quantize_rows_e4m3, reset_device_status, route, route_grouped, router_logits, status_string,
    workspace_layout, workspace_size)


class MoELayer:
    """A MoE FFN layer on one GPU.

    Weights (torch CUDA tensors, contiguous, all of one dtype bf16 or fp32):
    W_router [E,H], W_gate/W_up [E,I,H], W_down [E,H,I], optional router_bias
    fp32 [E] and shared expert Ws_gate/Ws_up [Is,H], Ws_down [H,Is].
    n_group > 1 limits each token's experts to its topk_group best groups of
    E / n_group consecutive experts (moe_route_grouped).
    """

    def __init__(self, W_router, W_gate, W_up, W_down, k, router_bias=None, Ws_gate=None,
                 Ws_up=None, Ws_down=None, renorm=1, tile=MOE_TILE_AUTO, n_group=1,
                 topk_group=1):
        self.W_router, self.W_gate, self.W_up, self.W_down = W_router, W_gate, W_up, W_down
        self.router_bias = router_bias
        self.Ws_gate, self.Ws_up, self.Ws_down = Ws_gate, Ws_up, Ws_down
        self.E, self.I, self.H = W_gate.shape
        self.I_shared = 0 if Ws_gate is None else Ws_gate.shape[0]
        self.k, self.renorm, self.tile = k, renorm, tile
        self.n_group, self.topk_group = n_group, topk_group
        self.dtype = W_gate.dtype
        self._ws = {}

    def problem(self, T: int, flags: int = 0, wait_limit_us: int = 0,
                out_f32: bool = False) -> MoEProblem:
        return make_problem(T, self.H, self.E, self.k, self.I, self.I_shared, self.renorm,
                            "bf16" if self.dtype == torch.bfloat16 else "f32", self.tile, flags,
                            wait_limit_us, out_f32, self.n_group, self.topk_group)

    def workspace(self, T: int) -> torch.Tensor:
        ws = self._ws.get(T)
        if ws is None:
            n = workspace_size(self.problem(T))
            ws = torch.zeros(n, dtype=torch.uint8, device=self.W_gate.device)
            self._ws[T] = ws
        return ws

    def forward(self, x, out=None, stream=None, out_f32=False, single_launch=False):
        """y = the layer applied to x [T,H]. out_f32: return y in fp32 (the value
        before its final rounding to a bf16 layer's dtype). single_launch: run
        moe_forward_single_launch (one kernel; decode-sized batches only)."""
        T = x.shape[0]
        odt = torch.float32 if out_f32 else self.dtype
        y = out if out is not None else torch.empty((T, self.H), dtype=odt, device=x.device)
        fn = forward_single_launch if single_launch else forward
        fn(self.problem(T, out_f32=out_f32), x, self.W_router, self.router_bias,
           self.W_gate, self.W_up, self.W_down, self.Ws_gate, self.Ws_up, self.Ws_down, y,
           self.workspace(T), stream)
        return y

    __call__ = forward


def quantize_e4m3(W: torch.Tensor):
    """(codes uint8, row scales fp32) of W viewed as rows of its last dimension,
    by moe_quantize_rows_e4m3 (E4M3 with one power-of-two scale per row)."""
    rows = W.numel() // W.shape[-1]
    q = torch.empty(W.shape, dtype=torch.uint8, device=W.device)
    s = torch.empty(W.shape[:-1], dtype=torch.float32, device=W.device)
    quantize_rows_e4m3(W.reshape(rows, W.shape[-1]), q.view(rows, W.shape[-1]), s.view(rows))
    return q, s


def quantize_mx_rows(W: torch.Tensor):
    """(codes uint8, E8M0 block scales uint8) of W viewed as rows of its last
    dimension, by moe_quantize_mx (E4M3 with one power-of-two scale per block
    of 32 elements); the scales have mx_scale_cols(cols) bytes per row."""
    cols = W.shape[-1]
    rows = W.numel() // cols
    sk = mx_scale_cols(cols)
    q = torch.empty(W.shape, dtype=torch.uint8, device=W.device)
    s = torch.empty(W.shape[:-1] + (sk,), dtype=torch.uint8, device=W.device)
    quantize_mx(W.reshape(rows, cols), q.view(rows, cols), s.view(rows, sk))
    return q, s


class _QuantizedLayer:
    """A layer whose expert matrices are quantized once on the GPU from the
    same bf16 weights MoELayer takes; x, W_router and y stay bf16."""

    _dtype_name = None
    _quantize = None
    _forward = None

    def __init__(self, W_router, W_gate, W_up, W_down, k, router_bias=None, Ws_gate=None,
                 Ws_up=None, Ws_down=None, renorm=1, tile=MOE_TILE_AUTO, n_group=1,
                 topk_group=1):
        self.W_router, self.router_bias = W_router, router_bias
        self.E, self.I, self.H = W_gate.shape
        self.I_shared = 0 if Ws_gate is None else Ws_gate.shape[0]
        self.k, self.renorm, self.tile = k, renorm, tile
        self.n_group, self.topk_group = n_group, topk_group
        self.dtype = torch.bfloat16  # activations (x, y)
        q = type(self)._quantize
        self.gate, self.up, self.down = (q(W) for W in (W_gate, W_up, W_down))
        if self.I_shared:
            self.s_gate, self.s_up, self.s_down = (q(W) for W in (Ws_gate, Ws_up, Ws_down))
        else:
            self.s_gate = self.s_up = self.s_down = (None, None)
        self._ws = {}

    def problem(self, T: int, flags: int = 0, wait_limit_us: int = 0,
                out_f32: bool = False) -> MoEProblem:
        return make_problem(T, self.H, self.E, self.k, self.I, self.I_shared, self.renorm,
                            self._dtype_name, self.tile, flags, wait_limit_us, out_f32,
                            self.n_group, self.topk_group)

    def workspace(self, T: int) -> torch.Tensor:
        ws = self._ws.get(T)
        if ws is None:
            n = workspace_size(self.problem(T))
            ws = torch.zeros(n, dtype=torch.uint8, device=self.W_router.device)
            self._ws[T] = ws
        return ws

    def forward(self, x, out=None, stream=None, out_f32=False):
        T = x.shape[0]
        odt = torch.float32 if out_f32 else torch.bfloat16
        y = out if out is not None else torch.empty((T, self.H), dtype=odt, device=x.device)
        type(self)._forward(self.problem(T, out_f32=out_f32), x, self.W_router,
                            self.router_bias, *self.gate, *self.up, *self.down, *self.s_gate,
                            *self.s_up, *self.s_down, y, self.workspace(T), stream)
        return y

    __call__ = forward


class MoELayerFP8(_QuantizedLayer):
    """The layer with E4M3 expert weights, one power-of-two scale per row
    (moe_forward_fp8)."""

    _dtype_name = "e4m3"
    _quantize = staticmethod(quantize_e4m3)
    _forward = staticmethod(forward_fp8)


class MoELayerMX(_QuantizedLayer):
    """The layer with MXFP8 expert weights, one E8M0 scale per block of 32
    elements along the contraction axis (moe_forward_mx)."""

    _dtype_name = "mxfp8"
    _quantize = staticmethod(quantize_mx_rows)
    _forward = staticmethod(forward_mx)
