"""The C-ABI library loads, exports every symbol include/moe_api.h declares,
and rejects bad arguments on the host before touching a GPU (CPU only: no
call here reaches the CUDA runtime)."""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_route_gb300 as m
from mixture_experts_layer_route_gb300 import build as build_mod
from moe_inputs import CONFIGS

HEADER = os.path.join(os.path.dirname(__file__), "..", "include", "moe_api.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return m.load_library()


def declared_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_binding_names():
    assert sorted(m.EXPORTED) == declared_symbols()


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_library_has_no_driver_link_dependency():
    # The driver entry point is looked up at run time; the library must load on
    # a host without libcuda (this one).
    import subprocess
    out = subprocess.run(["ldd", m._binding.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


def test_status_strings(lib):
    for code, name in m.STATUS_NAMES.items():
        assert m.status_string(code) == name


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_workspace_size_of_each_config(lib, name):
    c = CONFIGS[name]
    pb = m.make_problem(c.T, c.H, c.E, c.k, c.I, c.I_shared, c.renorm, c.dtype)
    n = m.workspace_size(pb)
    KP = c.k + (1 if c.I_shared else 0)
    # at least the fp32 slot buffer and h
    assert n >= c.T * KP * c.H * 4 + c.T * c.k * c.I * c.elem_bytes
    lay = m.workspace_layout(pb)
    assert all(v % 256 == 0 for v in lay.values() if v >= 0)
    assert (lay["h_shared"] >= 0) == bool(c.I_shared)


@pytest.mark.parametrize("kw,code", [
    (dict(k=9, E=8), 1), (dict(k=0), 1), (dict(H=200), 1), (dict(I=100), 1),
    (dict(I_shared=96), 1), (dict(E=2000, k=2), 1), (dict(k=33, E=64), 1), (dict(T=-1), 1),
])
def test_invalid_problem_rejected_on_host(lib, kw, code):
    base = dict(T=64, H=256, E=8, k=2, I=128, I_shared=0)
    base.update(kw)
    pb = m.make_problem(**base)
    with pytest.raises(m.MoEError) as ei:
        m.workspace_size(pb)
    assert ei.value.code == code


def test_forward_null_pointers_rejected_on_host(lib):
    pb = m.make_problem(64, 256, 8, 2, 128)
    rc = lib.moe_forward(ctypes.byref(pb), None, None, None, None, None, None, None, None,
                         None, None, None, 0, None)
    assert rc == 1  # MOE_ERR_INVALID_ARG


def test_forward_misaligned_pointer_rejected_on_host(lib):
    pb = m.make_problem(64, 256, 8, 2, 128)
    rc = lib.moe_forward(ctypes.byref(pb), 0x1008, 0x2000, None, 0x3000, 0x4000, 0x5000, None,
                         None, None, 0x6000, 0x7000, 1 << 30, None)
    assert rc == 1


def test_forward_small_workspace_rejected_on_host(lib):
    pb = m.make_problem(64, 256, 8, 2, 128)
    rc = lib.moe_forward(ctypes.byref(pb), 0x1000, 0x2000, None, 0x3000, 0x4000, 0x5000, None,
                         None, None, 0x6000, 0x7000, 1024, None)
    assert rc == 3  # MOE_ERR_WORKSPACE


def test_shared_pointer_mismatch_rejected_on_host(lib):
    pb = m.make_problem(64, 256, 8, 2, 128, I_shared=64)
    rc = lib.moe_forward(ctypes.byref(pb), 0x1000, 0x2000, None, 0x3000, 0x4000, 0x5000, None,
                         None, None, 0x6000, 0x7000, 1 << 30, None)
    assert rc == 1


def test_route_and_permute_bad_shapes_rejected_on_host(lib):
    assert lib.moe_route(0x1000, 4, 8, 9, 1, 0x2000, 0x3000, None) == 1
    assert lib.moe_route(0x1000, 4, 8, 2, 2, 0x2000, 0x3000, None) == 1
    assert lib.moe_permute(0x1000, 4, 8, 0, 0, 0x2000, 0x3000, 0x4000, 0x5000, 4096, None) == 1
    assert lib.moe_permute(0x1000, 4, 8, 2, 0, 0x2000, 0x3000, 0x4000, 0x5000, 16, None) == 3


def test_zero_tokens_is_ok_without_launch(lib):
    pb = m.make_problem(0, 256, 8, 2, 128)
    rc = lib.moe_forward(ctypes.byref(pb), None, None, None, None, None, None, None, None, None,
                         None, None, 0, None)
    assert rc == 0


LAYOUT_CASES = [dict(T=c.T, H=c.H, E=c.E, k=c.k, I=c.I, I_shared=c.I_shared, dtype=c.dtype)
                for c in CONFIGS.values()] + [
    dict(T=64, H=4096, E=128, k=8, I=1536, I_shared=0, dtype="e4m3"),
    dict(T=4096, H=7168, E=256, k=8, I=2048, I_shared=2048, dtype="e4m3"),
    dict(T=64, H=4096, E=128, k=8, I=1536, I_shared=0, dtype="mxfp8"),
    dict(T=4096, H=7168, E=256, k=8, I=2048, I_shared=2048, dtype="mxfp8"),
    dict(T=1, H=128, E=4, k=4, I=64, I_shared=64, dtype="bf16"),
    dict(T=513, H=256, E=1024, k=32, I=128, I_shared=0, dtype="f32"),
]


@pytest.mark.parametrize("c", LAYOUT_CASES, ids=[f"{c['T']}x{c['E']}x{c['k']}-{c['dtype']}"
                                                 for c in LAYOUT_CASES])
def test_workspace_layout_regions_are_disjoint_and_inside(lib, c):
    """moe_get_workspace_layout: every intermediate lies after the status
    header, 256-byte aligned, inside moe_workspace_size(), and no two regions
    overlap (sizes from the layouts the header states)."""
    pb = m.make_problem(c["T"], c["H"], c["E"], c["k"], c["I"], c["I_shared"], 1, c["dtype"])
    size = m.workspace_size(pb)
    lay = m.workspace_layout(pb)
    T, E, k, I, Is = c["T"], c["E"], c["k"], c["I"], c["I_shared"]
    act = 4 if c["dtype"] == "f32" else 2  # h is bf16 for E4M3 layers
    sizes = dict(logits=T * E * 4, topk_ids=T * k * 4, topk_w=T * k * 4,
                 expert_offsets=(E + 2) * 4, gather_idx=T * k * 4, slot_pos=T * k * 4,
                 h=T * k * I * act, h_shared=T * Is * act)
    regions = []
    for name, nbytes in sizes.items():
        off = lay[name]
        if name == "h_shared" and not Is:
            assert off == -1
            continue
        assert off >= 256 and off % 256 == 0, name
        assert off + nbytes <= size, name
        regions.append((off, off + nbytes, name))
    regions.sort()
    for (a0, a1, an), (b0, b1, bn) in zip(regions, regions[1:]):
        assert a1 <= b0, (an, bn)


@pytest.mark.parametrize("dims", [
    dict(T=1, H=1 << 22, E=1024, k=1, I=64),   # E*H = 2^32 rows of W_down
    dict(T=1, H=128, E=1, k=1, I=1 << 31),     # I beyond int32
    dict(T=1 << 27, H=128, E=8, k=8, I=64),    # T*(k+1) beyond the index range
])
def test_noalloc_rejects_index_ranges_on_host(lib, dims):
    """moe_down_combine_noalloc applies the same int32 index limits as the
    workspace entry points (MOE_ERR_UNSUPPORTED), before its own scratch-size
    check and before any launch; the first case would fit the scratch array."""
    pb = m.make_problem(dims["T"], dims["H"], dims["E"], dims["k"], dims["I"])
    st = ctypes.c_int(-1)
    rc = lib.moe_down_combine_noalloc(ctypes.byref(pb), 0x1000, None, 0x2000, 0x3000, 0x4000,
                                      0x5000, None, 0x6000, None, ctypes.byref(st))
    assert rc == 2  # MOE_ERR_UNSUPPORTED
    assert st.value == -1  # nothing ran, nothing was written


def test_noalloc_rejects_bad_problems_like_the_workspace_call(lib):
    for kw in (dict(k=9, E=8), dict(H=200), dict(I=100), dict(T=-1)):
        base = dict(T=64, H=256, E=8, k=2, I=128)
        base.update(kw)
        pb = m.make_problem(**base)
        rc = lib.moe_down_combine_noalloc(ctypes.byref(pb), 0x1000, None, 0x2000, 0x3000,
                                          0x4000, 0x5000, None, 0x6000, None, None)
        assert rc == 1, kw
    pb = m.make_problem(64, 256, 8, 2, 128, dtype="e4m3")
    assert lib.moe_down_combine_noalloc(ctypes.byref(pb), 0x1000, None, 0x2000, 0x3000, 0x4000,
                                        0x5000, None, 0x6000, None, None) == 1


# ------------------------------------------------------------------ MXFP8 calls

def test_mx_scale_cols(lib):
    assert [lib.moe_mx_scale_cols(c) for c in (32, 512, 544, 4096, 7168)] == [16, 16, 32, 128,
                                                                              224]


def test_quantize_mx_rejects_bad_arguments_on_host(lib):
    q = lib.moe_quantize_mx
    assert q(0x1000, 1, 4, 48, 0x2000, 0x3000, None) == 1   # cols not a multiple of 32
    assert q(0x1000, 2, 4, 64, 0x2000, 0x3000, None) == 1   # E4M3 is not a source dtype
    assert q(0x1000, 1, 4, 64, 0x2008, 0x3000, None) == 1   # misaligned codes
    assert q(0x1000, 1, 4, 64, None, 0x3000, None) == 1
    assert q(None, 1, 0, 64, None, None, None) == 0         # no rows: nothing to do


@pytest.mark.parametrize("kw,code", [
    (dict(I=192), 1),               # the MXFP8 GEMMs take K in steps of 128
    (dict(I_shared=64), 1),
    (dict(H=8320), 2),              # a scale row of more than 256 bytes
    (dict(I=8320), 2),
])
def test_mx_problem_rejected_on_host(lib, kw, code):
    base = dict(T=64, H=256, E=8, k=2, I=128, I_shared=0, dtype="mxfp8")
    base.update(kw)
    with pytest.raises(m.MoEError) as ei:
        m.workspace_size(m.make_problem(**base))
    assert ei.value.code == code


def test_forward_mx_checks_dtype_and_pointers_on_host(lib):
    def call(pb, shared, ws_bytes):
        x, wr, bias = 0x1000, 0x2000, None
        routed = [0x3000 + 0x1000 * i for i in range(6)]     # codes, scales x gate/up/down
        sh = [0x20000 + 0x1000 * i for i in range(6)] if shared else [None] * 6
        return lib.moe_forward_mx(ctypes.byref(pb), x, wr, bias, *routed, *sh, 0x40000, 0x50000,
                                  ws_bytes, None)

    assert call(m.make_problem(64, 256, 8, 2, 128, dtype="bf16"), False, 1 << 30) == 1
    pb = m.make_problem(64, 256, 8, 2, 128, dtype="mxfp8")
    assert call(pb, True, 1 << 30) == 1    # shared-expert pointers without a shared expert
    assert call(pb, False, 1024) == 3      # workspace too small
    pbs = m.make_problem(64, 256, 8, 2, 128, I_shared=128, dtype="mxfp8")
    assert call(pbs, False, 1 << 30) == 1  # a shared expert without its pointers
    # the bf16 entry points refuse the MXFP8 dtype
    assert lib.moe_forward(ctypes.byref(pb), 0x1000, 0x2000, None, 0x3000, 0x4000, 0x5000, None,
                           None, None, 0x6000, 0x7000, 1 << 30, None) == 1
