"""moe_down_combine_noalloc: the down projection + combine for callers that
cannot allocate device memory (a host that gives the layer only its inputs and
outputs, a plugin barred from cudaMalloc, a fixed memory budget). It runs with
the library's static scratch array instead of a caller workspace.

Checked through the C ABI against the workspace entry point moe_down_combine
on the same inputs, for two calls in a row (the static array keeps the last
call's contents, so the second call must not depend on them), and against the
CPU oracle's down projection + combine on the same h and routing, with the
float tolerance the other parity tests use; plus the host-side size limit.
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_route_gb300 as m
from moe_inputs import MoEConfig, generate, generate_hidden, generate_routing
from oracle import Oracle, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed, shared):
    T, E, k, H, I = 64, 16, 4, 1024, 256
    Is = 128 if shared else 0
    ids, w = generate_routing(T, E, k, seed=seed)
    ids = np.ascontiguousarray(ids.numpy().astype(np.int32))
    offs, gidx, spos = Oracle().permute(ids, E, 1 if shared else 0)
    cfg = MoEConfig("n", T=T, H=H, E=E, k=k, I=I, I_shared=Is)
    d = generate(cfg, seed=seed, device=DEV, enforce_margin=False)
    h = generate_hidden(T * k, I, seed=seed + 1, device=DEV)
    hs = generate_hidden(T, Is, seed=seed + 2, device=DEV) if shared else None
    return cfg, d, h, hs, torch.from_numpy(offs).to(DEV), torch.from_numpy(gidx).to(DEV), \
        w.to(DEV), (ids, offs, spos)


def _within_layer_bound(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    rms = float(np.sqrt(np.mean(b ** 2)))
    return (float(np.abs(a - b).max()) <= 2e-2 * rms
            and float(np.linalg.norm(a - b) / np.linalg.norm(b)) <= 5e-3)


@pytest.mark.parametrize("shared", [False, True])
def test_noalloc_matches_workspace_entry_point_twice(shared):
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        cfg, d, h, hs, offs, gidx, w, (ids, offs_np, spos) = _case(seed, shared)
        pb = m.make_problem(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.I_shared, out_f32=True)
        ws = torch.zeros(m.workspace_size(pb), dtype=torch.uint8, device=DEV)
        y_ref = torch.empty(cfg.T, cfg.H, dtype=torch.float32, device=DEV)
        m.down_combine(pb, h, hs, offs, gidx, w, d["W_down"], d["Ws_down"], y_ref, ws)
        y = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
        st = m.down_combine_noalloc(pb, h, hs, offs, gidx, w, d["W_down"], d["Ws_down"], y,
                                    want_status=True)
        torch.cuda.synchronize()
        assert st == m.MOE_OK, m.status_string(st)
        assert m.get_device_status(ws) == m.MOE_OK
        a, b = y.cpu().numpy().astype(np.float64), y_ref.cpu().numpy().astype(np.float64)
        assert np.isfinite(a).all(), f"call {call}: non-finite output"
        assert _within_layer_bound(a, b), f"call {call}: against moe_down_combine"
        # and against the CPU oracle on the same h, routing and weights
        ref = Oracle().down_combine(to_np(h), offs_np, spos, ids, to_np(w), to_np(d["W_down"]),
                                    to_np(hs), to_np(d["Ws_down"]))
        assert _within_layer_bound(a, ref), f"call {call}: against the oracle"


def test_noalloc_bf16_output_and_no_status_request():
    cfg, d, h, hs, offs, gidx, w, _ = _case(13, False)
    pb = m.make_problem(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I)
    ws = torch.zeros(m.workspace_size(pb), dtype=torch.uint8, device=DEV)
    y_ref = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=DEV)
    y = torch.empty_like(y_ref)
    m.down_combine(pb, h, hs, offs, gidx, w, d["W_down"], d["Ws_down"], y_ref, ws)
    assert m.down_combine_noalloc(pb, h, hs, offs, gidx, w, d["W_down"], d["Ws_down"], y) is None
    torch.cuda.synchronize()
    a, b = y.float().cpu().numpy(), y_ref.float().cpu().numpy()
    rms = float(np.sqrt(np.mean(b.astype(np.float64) ** 2)))
    assert float(np.abs(a - b).max()) <= 2e-2 * rms


def test_noalloc_rejects_problems_beyond_its_scratch():
    # T * (k + 1) * H * 4 bytes = 2048 * 9 * 4096 * 4 = 288 MiB > 16 MiB
    pb = m.make_problem(2048, 4096, 16, 8, 256, I_shared=256)
    dummy = torch.empty(16, dtype=torch.int32, device=DEV)
    with pytest.raises(m.MoEError) as ei:
        m.down_combine_noalloc(pb, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy)
    assert ei.value.code == 3  # MOE_ERR_WORKSPACE
