"""Device-side checks of the permutation a sub-call is given (the grouped GEMMs
and the dispatch copy take expert_offsets, gather_idx and slot_pos from the
caller). Each check sits where a kernel first takes the value in (the GEMM's
schedule, a tile's per-column staging, the copy's per-row loop), so the hot
loops are untouched and the checks are always on. A bad value is reported as
MOE_ERR_DEVICE_CHECK in the status word and the access it would have made is
skipped or redirected inside the buffers; the context stays usable and the
next valid call succeeds.

Every corrupted input below reaches only a checked access: one gather_idx entry
beyond T*k in moe_down_combine (read only by the down GEMM's column staging),
decreasing expert_offsets (the schedule then runs no unit), one slot_pos entry
beyond T*k in moe_grouped_swiglu_gemm for a batch that uses the dispatch copy
(read only by the copy).
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_route_gb300 as m
from moe_inputs import MoEConfig, generate, generate_hidden, generate_routing
from oracle import Oracle, to_np
from test_gpu_parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
DEVICE_CHECK = 6


def _down_case(T=40, E=8, k=2, H=256, I=128, seed=3):
    ids, w = generate_routing(T, E, k, seed=seed)
    ids = np.ascontiguousarray(np.asarray(ids, np.int32))
    offs, gidx, spos = Oracle().permute(ids, E, 0)
    cfg = MoEConfig("d", T=T, H=H, E=E, k=k, I=I)
    d = generate(cfg, seed=seed, device=DEV, enforce_margin=False)
    h = generate_hidden(T * k, I, seed=seed + 1, device=DEV)
    pb = m.make_problem(T, H, E, k, I, out_f32=True)
    ws = torch.zeros(m.workspace_size(pb), dtype=torch.uint8, device=DEV)
    return pb, ws, d, h, ids, w, offs, gidx, spos


def _down(pb, ws, d, h, offs, gidx, w):
    y = torch.empty(pb.T, pb.H, dtype=torch.float32, device=DEV)
    m.reset_device_status(ws)
    m.down_combine(pb, h, None, torch.from_numpy(offs).to(DEV), torch.from_numpy(gidx).to(DEV),
                   w.to(DEV), d["W_down"], None, y, ws)
    torch.cuda.synchronize()
    return y, m.get_device_status(ws)


def test_gather_index_out_of_range_is_reported():
    pb, ws, d, h, ids, w, offs, gidx, spos = _down_case()
    y_ok, st = _down(pb, ws, d, h, offs, gidx, w)
    assert st == m.MOE_OK
    bad = gidx.copy()
    bad[5] = pb.T * pb.k + 7
    _, st = _down(pb, ws, d, h, offs, bad, w)
    assert st == DEVICE_CHECK
    y2, st = _down(pb, ws, d, h, offs, gidx, w)  # the context is fine
    assert st == m.MOE_OK
    assert torch.equal(y2, y_ok)
    ref = Oracle().down_combine(to_np(h), offs, spos, ids, to_np(w), to_np(d["W_down"]))
    assert_close(y2.cpu().numpy(), ref, "down_combine after a device-check failure")


def test_decreasing_offsets_are_reported():
    pb, ws, d, h, ids, w, offs, gidx, spos = _down_case(seed=4)
    bad = offs.copy()
    bad[3] = bad[2] - 1
    _, st = _down(pb, ws, d, h, bad, gidx, w)
    assert st == DEVICE_CHECK
    _, st = _down(pb, ws, d, h, offs, gidx, w)
    assert st == m.MOE_OK


def test_slot_position_out_of_range_is_reported():
    T, E, k, H, I = 96, 8, 2, 256, 128  # > 64 tokens: the dispatch copy runs
    ids, _ = generate_routing(T, E, k, seed=5)
    ids = np.ascontiguousarray(np.asarray(ids, np.int32))
    offs, gidx, spos = Oracle().permute(ids, E, 0)
    cfg = MoEConfig("g", T=T, H=H, E=E, k=k, I=I)
    d = generate(cfg, seed=5, device=DEV, enforce_margin=False)
    pb = m.make_problem(T, H, E, k, I)
    ws = torch.zeros(m.workspace_size(pb), dtype=torch.uint8, device=DEV)
    h = torch.empty(T * k, I, dtype=torch.bfloat16, device=DEV)
    dv = {n: torch.from_numpy(a).to(DEV) for n, a in (("o", offs), ("g", gidx), ("s", spos))}
    bad = spos.copy()
    bad[9] = T * k + 3
    m.grouped_swiglu_gemm(pb, d["x"], dv["o"], dv["g"], torch.from_numpy(bad).to(DEV),
                          d["W_gate"], d["W_up"], None, None, h, None, ws)
    torch.cuda.synchronize()
    assert m.get_device_status(ws) == DEVICE_CHECK
    m.reset_device_status(ws)
    m.grouped_swiglu_gemm(pb, d["x"], dv["o"], dv["g"], dv["s"], d["W_gate"], d["W_up"], None,
                          None, h, None, ws)
    torch.cuda.synchronize()
    assert m.get_device_status(ws) == m.MOE_OK
