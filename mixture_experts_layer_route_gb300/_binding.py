"""ctypes binding of libmoe.so: the C-ABI calls under the same names, taking
torch tensors. Argument marshalling only -- every step runs in the library's
CUDA kernels. There is no fallback: if the library cannot be loaded, or a call
returns an error status, a MoEError is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT",
                6: "MOE_ERR_DEVICE_CHECK"}
MOE_DTYPE_F32, MOE_DTYPE_BF16, MOE_DTYPE_E4M3, MOE_DTYPE_MXFP8 = 0, 1, 2, 3
MOE_TILE_AUTO, MOE_TILE_DECODE, MOE_TILE_PREFILL, MOE_TILE_MEDIUM = 0, 1, 2, 3
MOE_FLAG_TEST_SKIP_SIGNAL = 0x1

# Every symbol include/moe_api.h declares.
EXPORTED = ("moe_workspace_size", "moe_router_logits", "moe_route", "moe_route_grouped",
            "moe_permute",
            "moe_grouped_swiglu_gemm", "moe_down_combine", "moe_forward",
            "moe_get_workspace_layout", "moe_get_device_status", "moe_reset_device_status",
            "moe_status_string", "moe_down_combine_noalloc", "moe_quantize_rows_e4m3",
            "moe_forward_fp8", "moe_forward_single_launch", "moe_mx_scale_cols",
            "moe_quantize_mx", "moe_forward_mx")


class MoEError(RuntimeError):
    def __init__(self, call: str, code: int):
        super().__init__(f"{call} returned {STATUS_NAMES.get(code, code)}")
        self.code = code


class MoEProblem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int64), ("E", ctypes.c_int64),
                ("k", ctypes.c_int64), ("I", ctypes.c_int64), ("I_shared", ctypes.c_int64),
                ("renorm", ctypes.c_int32), ("dtype", ctypes.c_int32), ("tile", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("wait_limit_us", ctypes.c_uint32),
                ("out_f32", ctypes.c_int32), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32)]


class MoEWorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("logits", "topk_ids", "topk_w", "expert_offsets",
                                               "gather_idx", "slot_pos", "h", "h_shared",
                                               "h_scales", "h_shared_scales")]


_lib = None
_lock = threading.Lock()
_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libmoe.so (build it with mixture_experts_layer_route_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise OSError(f"{p} is missing: build it with "
                          "`python -m mixture_experts_layer_route_gb300.build`")
        lib = ctypes.CDLL(p)
        pb = ctypes.POINTER(MoEProblem)
        sig = {
            "moe_workspace_size": [pb, ctypes.POINTER(ctypes.c_size_t)],
            "moe_router_logits": [pb, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
            "moe_route": [_P, _I64, _I64, _I64, ctypes.c_int, _P, _P, _P],
            "moe_route_grouped": [_P, _I64, _I64, _I64, ctypes.c_int, _I64, _I64, _P, _P, _P],
            "moe_permute": [_P, _I64, _I64, _I64, ctypes.c_int, _P, _P, _P, _P, ctypes.c_size_t,
                            _P],
            "moe_grouped_swiglu_gemm": [pb, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        ctypes.c_size_t, _P],
            "moe_down_combine": [pb, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
            "moe_forward": [pb, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
            "moe_forward_single_launch": [pb, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                          ctypes.c_size_t, _P],
            "moe_get_workspace_layout": [pb, ctypes.POINTER(MoEWorkspaceLayout)],
            "moe_get_device_status": [_P, _P, ctypes.POINTER(ctypes.c_int)],
            "moe_reset_device_status": [_P, _P],
            "moe_quantize_rows_e4m3": [_P, ctypes.c_int32, _I64, _I64, _P, _P, _P],
            "moe_forward_fp8": [pb, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                _P, _P, ctypes.c_size_t, _P],
            "moe_quantize_mx": [_P, ctypes.c_int32, _I64, _I64, _P, _P, _P],
            "moe_forward_mx": [pb, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                               _P, _P, ctypes.c_size_t, _P],
            "moe_down_combine_noalloc": [pb, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                         ctypes.POINTER(ctypes.c_int)],
        }
        for name, argt in sig.items():
            f = getattr(lib, name)
            f.argtypes = argt
            f.restype = ctypes.c_int
        lib.moe_mx_scale_cols.argtypes = [_I64]
        lib.moe_mx_scale_cols.restype = _I64
        lib.moe_status_string.argtypes = [ctypes.c_int]
        lib.moe_status_string.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name: str, code: int):
    if code != MOE_OK:
        raise MoEError(name, code)


def make_problem(T, H, E, k, I, I_shared=0, renorm=1, dtype="bf16", tile=MOE_TILE_AUTO,
                 flags=0, wait_limit_us=0, out_f32=False, n_group=1,
                 topk_group=1) -> MoEProblem:
    dt = (MOE_DTYPE_BF16 if dtype in ("bf16", torch.bfloat16)
          else MOE_DTYPE_E4M3 if dtype == "e4m3"
          else MOE_DTYPE_MXFP8 if dtype == "mxfp8" else MOE_DTYPE_F32)
    return MoEProblem(T, H, E, k, I, I_shared, renorm, dt, tile, flags, wait_limit_us,
                      1 if out_f32 else 0, n_group, topk_group)


def workspace_size(problem: MoEProblem) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_workspace_size", load_library().moe_workspace_size(ctypes.byref(problem),
                                                                   ctypes.byref(n)))
    return int(n.value)


def workspace_layout(problem: MoEProblem) -> dict:
    out = MoEWorkspaceLayout()
    _check("moe_get_workspace_layout",
           load_library().moe_get_workspace_layout(ctypes.byref(problem), ctypes.byref(out)))
    return {n: getattr(out, n) for n, _ in MoEWorkspaceLayout._fields_}


def router_logits(problem, x, W_router, router_bias, logits, workspace, stream=None):
    _check("moe_router_logits", load_library().moe_router_logits(
        ctypes.byref(problem), _ptr(x), _ptr(W_router), _ptr(router_bias), _ptr(logits),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def route(logits, k, renorm, topk_ids, topk_w, stream=None):
    T, E = logits.shape
    _check("moe_route", load_library().moe_route(_ptr(logits), T, E, k, int(renorm),
                                                 _ptr(topk_ids), _ptr(topk_w), _stream(stream)))


def route_grouped(logits, k, renorm, n_group, topk_group, topk_ids, topk_w, stream=None):
    T, E = logits.shape
    _check("moe_route_grouped", load_library().moe_route_grouped(
        _ptr(logits), T, E, k, int(renorm), int(n_group), int(topk_group), _ptr(topk_ids),
        _ptr(topk_w), _stream(stream)))


def permute(topk_ids, E, has_shared, expert_offsets, gather_idx, slot_pos, workspace,
            stream=None):
    T, k = topk_ids.shape
    _check("moe_permute", load_library().moe_permute(
        _ptr(topk_ids), T, E, k, int(has_shared), _ptr(expert_offsets), _ptr(gather_idx),
        _ptr(slot_pos), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def grouped_swiglu_gemm(problem, x, expert_offsets, gather_idx, slot_pos, W_gate, W_up, Ws_gate,
                        Ws_up, h, h_shared, workspace, stream=None):
    _check("moe_grouped_swiglu_gemm", load_library().moe_grouped_swiglu_gemm(
        ctypes.byref(problem), _ptr(x), _ptr(expert_offsets), _ptr(gather_idx), _ptr(slot_pos),
        _ptr(W_gate), _ptr(W_up), _ptr(Ws_gate), _ptr(Ws_up), _ptr(h), _ptr(h_shared),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def down_combine(problem, h, h_shared, expert_offsets, gather_idx, topk_w, W_down, Ws_down, y,
                 workspace, stream=None):
    _check("moe_down_combine", load_library().moe_down_combine(
        ctypes.byref(problem), _ptr(h), _ptr(h_shared), _ptr(expert_offsets), _ptr(gather_idx),
        _ptr(topk_w), _ptr(W_down), _ptr(Ws_down), _ptr(y), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def down_combine_noalloc(problem, h, h_shared, expert_offsets, gather_idx, topk_w, W_down,
                         Ws_down, y, stream=None, want_status=False):
    """moe_down_combine without a workspace (the library's static scratch).
    With want_status, waits for the stream and returns the device status."""
    st = ctypes.c_int(-1)
    _check("moe_down_combine_noalloc", load_library().moe_down_combine_noalloc(
        ctypes.byref(problem), _ptr(h), _ptr(h_shared), _ptr(expert_offsets), _ptr(gather_idx),
        _ptr(topk_w), _ptr(W_down), _ptr(Ws_down), _ptr(y), _stream(stream),
        ctypes.byref(st) if want_status else None))
    return int(st.value) if want_status else None


def quantize_rows_e4m3(src, q, scale, stream=None):
    """E4M3 codes q [rows, cols] (uint8) and power-of-two row scales (fp32) of
    src [rows, cols] (bf16 or fp32), as moe_quantize_rows_e4m3 defines them."""
    rows, cols = src.shape
    dt = MOE_DTYPE_BF16 if src.dtype == torch.bfloat16 else MOE_DTYPE_F32
    _check("moe_quantize_rows_e4m3", load_library().moe_quantize_rows_e4m3(
        _ptr(src), dt, rows, cols, _ptr(q), _ptr(scale), _stream(stream)))


def forward_fp8(problem, x, W_router, router_bias, Wq_gate, s_gate, Wq_up, s_up, Wq_down, s_down,
                Wsq_gate, ss_gate, Wsq_up, ss_up, Wsq_down, ss_down, y, workspace, stream=None):
    _check("moe_forward_fp8", load_library().moe_forward_fp8(
        ctypes.byref(problem), _ptr(x), _ptr(W_router), _ptr(router_bias), _ptr(Wq_gate),
        _ptr(s_gate), _ptr(Wq_up), _ptr(s_up), _ptr(Wq_down), _ptr(s_down), _ptr(Wsq_gate),
        _ptr(ss_gate), _ptr(Wsq_up), _ptr(ss_up), _ptr(Wsq_down), _ptr(ss_down), _ptr(y),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def mx_scale_cols(cols: int) -> int:
    """Bytes of a row of MXFP8 scales for `cols` elements (moe_mx_scale_cols)."""
    return int(load_library().moe_mx_scale_cols(int(cols)))


def quantize_mx(src, q, scales, stream=None):
    """MXFP8 codes q [rows, cols] (uint8) and E8M0 block scales
    [rows, mx_scale_cols(cols)] (uint8) of src [rows, cols] (bf16 or fp32), as
    moe_quantize_mx defines them."""
    rows, cols = src.shape
    dt = MOE_DTYPE_BF16 if src.dtype == torch.bfloat16 else MOE_DTYPE_F32
    _check("moe_quantize_mx", load_library().moe_quantize_mx(
        _ptr(src), dt, rows, cols, _ptr(q), _ptr(scales), _stream(stream)))


def forward_mx(problem, x, W_router, router_bias, Wq_gate, s_gate, Wq_up, s_up, Wq_down, s_down,
               Wsq_gate, ss_gate, Wsq_up, ss_up, Wsq_down, ss_down, y, workspace, stream=None):
    _check("moe_forward_mx", load_library().moe_forward_mx(
        ctypes.byref(problem), _ptr(x), _ptr(W_router), _ptr(router_bias), _ptr(Wq_gate),
        _ptr(s_gate), _ptr(Wq_up), _ptr(s_up), _ptr(Wq_down), _ptr(s_down), _ptr(Wsq_gate),
        _ptr(ss_gate), _ptr(Wsq_up), _ptr(ss_up), _ptr(Wsq_down), _ptr(ss_down), _ptr(y),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def forward(problem, x, W_router, router_bias, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, y,
            workspace, stream=None):
    _check("moe_forward", load_library().moe_forward(
        ctypes.byref(problem), _ptr(x), _ptr(W_router), _ptr(router_bias), _ptr(W_gate),
        _ptr(W_up), _ptr(W_down), _ptr(Ws_gate), _ptr(Ws_up), _ptr(Ws_down), _ptr(y),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def forward_single_launch(problem, x, W_router, router_bias, W_gate, W_up, W_down, Ws_gate,
                          Ws_up, Ws_down, y, workspace, stream=None):
    """moe_forward as one kernel launch (decode-sized batches); raises
    MoEError(MOE_ERR_UNSUPPORTED) for problems it does not take."""
    _check("moe_forward_single_launch", load_library().moe_forward_single_launch(
        ctypes.byref(problem), _ptr(x), _ptr(W_router), _ptr(router_bias), _ptr(W_gate),
        _ptr(W_up), _ptr(W_down), _ptr(Ws_gate), _ptr(Ws_up), _ptr(Ws_down), _ptr(y),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def get_device_status(workspace, stream=None) -> int:
    out = ctypes.c_int(-1)
    _check("moe_get_device_status", load_library().moe_get_device_status(
        _ptr(workspace), _stream(stream), ctypes.byref(out)))
    return int(out.value)


def reset_device_status(workspace, stream=None):
    _check("moe_reset_device_status",
           load_library().moe_reset_device_status(_ptr(workspace), _stream(stream)))


def status_string(code: int) -> str:
    return load_library().moe_status_string(code).decode()
