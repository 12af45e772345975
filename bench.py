"""Benchmark of the MoE layer forward pass on GB300.

One step = the whole layer (router logits, top-k routing, permutation, grouped
gate/up GEMM with SwiGLU, down GEMM with the weighted combine) over one batch of
synthetic tokens whose weights and inputs are resident in HBM.

Default workload: the Qwen3-235B-shaped decode step (T=64, H=4096, E=128, k=8,
I=1536, bf16). The other four layer shapes are measured in the same run and
reported under "workloads" (the prefill chunk of the same layer, T=8192, also
under "prefill"): the Qwen3.5-397B-shaped Zipf-skewed layer, the
DeepSeek-V3-shaped layer with its shared expert, and the tiny fp32 layer. Each
carries its own roofline, per-stage times and a sampled parity error against
the CPU oracle. Every layer's expert weights are larger than L2 except the tiny
layer's, whose steps are timed one by one with a 512 MiB L2 flush between them.

Printed: one JSON line (rank 0). value = tokens/s of the whole job; roofline =
the dominant kernel's achieved bandwidth or FLOP rate against the measured peak;
layer_roofline = t_roof / t_measured for the whole layer with
t_roof = max(routed FLOPs / bf16 peak, touched bytes / HBM bandwidth), the bf16
peak being the burst figure (the timed regions last tens of milliseconds; the
fraction against the sustained figure is given beside it);
e2e = the same metric through MoELayer.forward with the tokens copied from
pinned host memory and the output copied back inside the timed region (on
copy streams, double-buffered, overlapping the next step's compute);
cpu_baseline = the CPU oracle on a bounded sample of the same workload;
fp8 / mxfp8 = the same workloads with the expert weights quantized (E4M3 with
a scale per row, or MXFP8 with a scale per block of 32 elements).

Multi-GPU (torchrun): each rank runs an independent replica of the layer on its
own batch (the layer has no exchange step on one GPU); the time is the max over
ranks and value counts every rank's tokens.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from moe_inputs import CONFIGS, PROFILE_CONFIGS, generate  # noqa: E402

ALL_CONFIGS = {**CONFIGS, **PROFILE_CONFIGS}

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["mixture_experts_layer_route_gb300/csrc/grouped_gemm.cuh",
                  "mixture_experts_layer_route_gb300/csrc/grouped_gemm.cu",
                  "mixture_experts_layer_route_gb300/csrc/common.cuh"]
STAGES = ["router_logits", "route", "permute", "swiglu_gemm", "down_gemm+combine"]


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def kernel_source_hash() -> str:
    """Hash of the GEMM sources' code: comments and whitespace are dropped, so
    that a comment edit does not orphan DRAM counters taken on the same code."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def traffic_for(config: str, kernel: str):
    """Per-launch DRAM bytes of `kernel` on `config` from the committed ncu
    summary, or None if absent or taken on a different kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        e = t[config][kernel]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- model

def roofline_numbers(cfg, counts):
    """Algorithmic FLOPs and bytes of the layer and of the gated GEMM, from the
    run's own per-expert counts."""
    es = cfg.elem_bytes
    T, H, E, k, I, Is = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.I_shared
    touched = int((counts > 0).sum())
    flop_layer = 2.0 * T * k * 3 * H * I + 2.0 * T * 3 * H * Is
    bytes_layer = (touched * 3 * H * I * es + (3 * H * Is * es if Is else 0)
                   + 2 * T * H * es + E * H * es)
    flop_g = 2.0 * T * k * 2 * H * I + 2.0 * T * 2 * H * Is
    bytes_g = (touched * 2 * H * I * es + (2 * H * Is * es if Is else 0) + T * H * es
               + (T * k * I + T * Is) * es)
    return dict(touched=touched, flop_layer=flop_layer, bytes_layer=bytes_layer,
                flop_gated=flop_g, bytes_gated=bytes_g)


def kernels_per_step(cfg):
    """Kernels one moe_forward launches with the automatic tile choice: router
    logits, route, permute (one kernel up to 4096 slots, else count + scatter),
    [the expert-ordered copy of the routed rows for batches of more than 64
    tokens], one launch per GEMM, combine."""
    permute = 1 if cfg.T * cfg.k <= 4096 else 2
    return 2 + permute + (1 if cfg.T > 64 else 0) + 2 + 1


def build_layer(cfg, device, seed=0):
    import mixture_experts_layer_route_gb300 as m
    d = generate(cfg, seed=seed, device=device)
    layer = m.MoELayer(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                       router_bias=d["router_bias"], Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"],
                       Ws_down=d["Ws_down"], renorm=cfg.renorm)
    return layer, d


def stage_sequence(layer, d, T, ws, lay, stream):
    """The kernels of one moe_forward call, issued through the sub-call entry
    points so that CUDA events can separate them."""
    import mixture_experts_layer_route_gb300 as m
    pb = layer.problem(T)
    E, k = layer.E, layer.k

    def buf(name, n, dt):
        o = lay[name]
        return ws[o:o + n * 4].view(dt)

    logits = buf("logits", T * E, torch.float32).view(T, E)
    ids = buf("topk_ids", T * k, torch.int32).view(T, k)
    w = buf("topk_w", T * k, torch.float32).view(T, k)
    offs = buf("expert_offsets", E + 2, torch.int32)
    gidx = buf("gather_idx", T * k, torch.int32)
    spos = buf("slot_pos", T * k, torch.int32)
    es = 2 if layer.dtype == torch.bfloat16 else 4
    h = ws[lay["h"]:lay["h"] + T * k * layer.I * es].view(layer.dtype).view(T * k, layer.I)
    hs = None
    if layer.I_shared:
        o = lay["h_shared"]
        hs = ws[o:o + T * layer.I_shared * es].view(layer.dtype).view(T, layer.I_shared)
    y = torch.empty(T, layer.H, dtype=layer.dtype, device=ws.device)
    steps = [
        lambda: m.router_logits(pb, d["x"], layer.W_router, layer.router_bias, logits, ws,
                                stream),
        lambda: m.route(logits, k, layer.renorm, ids, w, stream),
        lambda: m.permute(ids, E, 1 if layer.I_shared else 0, offs, gidx, spos, ws, stream),
        lambda: m.grouped_swiglu_gemm(pb, d["x"], offs, gidx, spos, layer.W_gate, layer.W_up,
                                      layer.Ws_gate, layer.Ws_up, h, hs, ws, stream),
        lambda: m.down_combine(pb, h, hs, offs, gidx, w, layer.W_down, layer.Ws_down, y, ws,
                               stream),
    ]
    return steps, offs


def time_forward(layer, d, steps, warmup, stream, flush=None):
    """K steps of the layer between CUDA events on `stream`. flush: a buffer
    larger than L2 written between steps, outside the timed intervals (the
    steps are then timed one by one and their durations summed)."""
    x = d["x"]
    T = x.shape[0]
    y = torch.empty(T, layer.H, dtype=layer.dtype, device=x.device)
    for _ in range(warmup):
        layer.forward(x, out=y, stream=stream)
    torch.cuda.synchronize()
    if flush is None:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for i in range(steps):
                layer.forward(x, out=y, stream=stream)
                ev[i + 1].record(stream)
        torch.cuda.synchronize()
        per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
        return ev[0].elapsed_time(ev[-1]), per
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.fill_(i & 0xFF)
            e0[i].record(stream)
            layer.forward(x, out=y, stream=stream)
            e1[i].record(stream)
    torch.cuda.synchronize()
    per = [e0[i].elapsed_time(e1[i]) for i in range(steps)]
    return sum(per), per


def time_stages(layer, d, steps, warmup, stream):
    import mixture_experts_layer_route_gb300 as m
    T = d["x"].shape[0]
    ws = layer.workspace(T)
    lay = m.workspace_layout(layer.problem(T))
    fns, offs = stage_sequence(layer, d, T, ws, lay, stream)
    for _ in range(warmup):
        for f in fns:
            f()
    torch.cuda.synchronize()
    n = len(fns)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            ev[i][0].record(stream)
            for j, f in enumerate(fns):
                f()
                ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    st = m.get_device_status(ws, stream)
    if st != m.MOE_OK:
        raise RuntimeError(f"device status {m.status_string(st)}")
    per_stage = [statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps))
                 for j in range(n)]
    counts = torch.diff(offs[:layer.E + 1]).cpu()
    return per_stage, counts


def time_e2e(layer, d, steps, warmup, stream):
    """Public API end to end: each step copies its tokens from pinned host memory
    to the device, runs the layer, and copies y back to pinned host memory. The
    copies run on their own streams, double-buffered, so that step i+1's tokens
    arrive and step i's result leaves while the next layer computes (as a
    serving loop would); every step's copies are inside the timed region."""
    x_dev = d["x"]
    T, H = x_dev.shape
    x_host = x_dev.cpu().pin_memory()
    y_host = torch.empty((T, H), dtype=layer.dtype).pin_memory()
    x_in = [torch.empty_like(x_dev) for _ in range(2)]
    y = [torch.empty_like(x_dev) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_x = [torch.cuda.Event() for _ in range(2)]   # x_in[b] filled
    ev_y = [torch.cuda.Event() for _ in range(2)]   # y[b] computed (x_in[b] read)
    ev_o = [torch.cuda.Event() for _ in range(2)]   # y[b] copied out

    def run(n):
        with torch.cuda.stream(h2d):
            x_in[0].copy_(x_host, non_blocking=True)
            ev_x[0].record(h2d)
        for i in range(n):
            b = i & 1
            stream.wait_event(ev_x[b])
            if i >= 2:
                stream.wait_event(ev_o[b])
            layer.forward(x_in[b], out=y[b], stream=stream)
            ev_y[b].record(stream)
            if i + 1 < n:
                if i >= 1:
                    h2d.wait_event(ev_y[1 - b])
                with torch.cuda.stream(h2d):
                    x_in[1 - b].copy_(x_host, non_blocking=True)
                    ev_x[1 - b].record(h2d)
            d2h.wait_event(ev_y[b])
            with torch.cuda.stream(d2h):
                y_host.copy_(y[b], non_blocking=True)
                ev_o[b].record(d2h)

    run(warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(h2d)
    run(steps)
    e1.record(d2h)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    nb = T * H * x_dev.element_size()
    return ms, nb, nb


def time_graph(layer, d, steps, warmup, stream):
    """The same forward pass captured once in a CUDA graph and replayed K times:
    identical kernels and work, without the host launch path between them."""
    x = d["x"]
    T = x.shape[0]
    y = torch.empty(T, layer.H, dtype=layer.dtype, device=x.device)
    with torch.cuda.stream(stream):
        layer.forward(x, out=y, stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        layer.forward(x, out=y)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1)


def parity_sample(cfg, layer, d, n_tokens=8):
    """The layer's fp32 output (out_f32) on n_tokens tokens spread over the
    batch, against the CPU oracle on the same tokens (router, top-k, experts,
    combine; only the experts those tokens use are copied to the host, one
    token at a time). Also checks that the routed ids agree."""
    import numpy as np

    import mixture_experts_layer_route_gb300 as m
    import oracle
    o = oracle.Oracle()
    T = cfg.T
    y = layer.forward(d["x"], out_f32=True)
    ws = layer.workspace(T)
    lay = m.workspace_layout(layer.problem(T, out_f32=True))
    ids_gpu = ws[lay["topk_ids"]:lay["topk_ids"] + T * cfg.k * 4].view(torch.int32)
    ids_gpu = ids_gpu.view(T, cfg.k).cpu().numpy()
    torch.cuda.synchronize()
    toks = sorted({int(i * T / n_tokens) for i in range(n_tokens)} | {T - 1})
    Wr, bias = oracle.to_np(d["W_router"]), oracle.to_np(d["router_bias"])
    sh = [oracle.to_np(d[n]) for n in ("Ws_gate", "Ws_up", "Ws_down")]
    max_abs, ss_d, ss_r, sq, ids_ok = 0.0, 0.0, 0.0, 0.0, True
    for t in toks:
        xt = oracle.to_np(d["x"][t:t + 1])
        ids, w = o.route(o.router_logits(xt, Wr, bias), cfg.k, cfg.renorm)
        ids_ok &= bool((ids[0] == ids_gpu[t]).all())
        sel = torch.from_numpy(ids[0].astype(np.int64)).to(d["W_gate"].device)
        ref = o.ffn_combine(xt, np.arange(cfg.k, dtype=np.int32)[None, :].copy(), w,
                            oracle.to_np(d["W_gate"][sel]), oracle.to_np(d["W_up"][sel]),
                            oracle.to_np(d["W_down"][sel]), *sh)[0].astype(np.float64)
        got = y[t].float().cpu().numpy().astype(np.float64)
        max_abs = max(max_abs, float(np.abs(got - ref).max()))
        ss_d += float(((got - ref) ** 2).sum())
        ss_r += float((ref ** 2).sum())
        sq += ref.size
    rms = (ss_r / sq) ** 0.5
    return {"tokens": len(toks), "max_abs_over_rms": max_abs / rms,
            "rel_l2": (ss_d / ss_r) ** 0.5, "ids_match": ids_ok,
            "bound": {"max_abs_over_rms": 2e-2, "rel_l2": 5e-3},
            "how": "fp32 y (out_f32) of the timed layer on tokens spread over the batch "
                   "against the CPU oracle"}


def cpu_baseline(cfg, d, budget_s=10.0, max_tokens=None):
    """The CPU oracle, as it stands, on a bounded sample of tokens of the same
    layer: tokens/s over ~budget_s seconds of oracle work."""
    import numpy as np

    import oracle
    o = oracle.Oracle()
    T = cfg.T if max_tokens is None else min(cfg.T, max_tokens)
    x = d["x"][:T]
    # Only the experts the sampled tokens use are copied to the host.
    lg = o.router_logits(oracle.to_np(x), oracle.to_np(d["W_router"]),
                         oracle.to_np(d["router_bias"]))
    ids, _ = o.route(lg, cfg.k, cfg.renorm)
    used = np.unique(ids)
    remap = np.full(cfg.E, -1, np.int64)
    remap[used] = np.arange(len(used))
    sel = torch.from_numpy(used.astype(np.int64)).to(d["W_gate"].device)
    Wr = oracle.to_np(d["W_router"])
    Wg = oracle.to_np(d["W_gate"][sel])
    Wu = oracle.to_np(d["W_up"][sel])
    Wd = oracle.to_np(d["W_down"][sel])
    sh = [oracle.to_np(d[n]) for n in ("Ws_gate", "Ws_up", "Ws_down")]
    xs = oracle.to_np(x)
    bias = oracle.to_np(d["router_bias"])
    # The oracle's own forward, restricted to the copied experts: route on the
    # full logits, then the FFN + combine on the remapped ids.
    done = 0
    t0 = time.perf_counter()
    while True:
        lg = o.router_logits(xs, Wr, bias)
        ids, w = o.route(lg, cfg.k, cfg.renorm)
        o.ffn_combine(xs, np.ascontiguousarray(remap[ids].astype(np.int32)), w, Wg, Wu, Wd,
                      *sh)
        done += T
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": done / el, "unit": "tokens/s", "cores": o.num_threads(), "kind": "oracle",
            "sample": f"{done} tokens ({T} per pass, {done // T} passes) of the {cfg.name} "
                      f"layer through the fp32 C++ oracle (router, top-k, experts, combine)",
            "seconds": el}


# ----------------------------------------------------------------- main

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()


def max_over_ranks(v, world):
    """The slowest rank's time: every rank's replica must finish before the
    job's tokens count as done."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, T, steps, ms_total):
    """Whole-job throughput of `world` independent replicas, each running
    `steps` layer passes over T tokens in ms_total (the max over ranks)."""
    return world * T * steps / (ms_total / 1e3)


L2_BYTES = 129 * 2 ** 20


def fits_l2(cfg):
    """True when the layer's weights and tokens could stay in L2 between steps."""
    w = cfg.E * 3 * cfg.H * cfg.I + 3 * cfg.H * cfg.I_shared + cfg.E * cfg.H
    return (w + 2 * cfg.T * cfg.H) * cfg.elem_bytes < 2 * L2_BYTES


def measure_config(cfg, args, world, local, with_clocks, parity_tokens=8):
    import mixture_experts_layer_route_gb300 as m
    stream = torch.cuda.Stream()
    layer, d = build_layer(cfg, "cuda", seed=args.seed)
    layer.workspace(cfg.T)
    steps = args.steps if cfg.T <= 1024 else max(3, args.steps // 8)
    flush = (torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")
             if fits_l2(cfg) else None)
    # timed region: K steps of moe_forward
    sampler = ClockSampler(local) if with_clocks else None
    barrier(world)
    if sampler:
        sampler.start()
        time.sleep(0.3)
    ms_total, per = time_forward(layer, d, steps, args.warmup, stream, flush)
    clocks = sampler.stop() if sampler else None
    barrier(world)
    ms_total = max_over_ranks(ms_total, world)
    st = m.get_device_status(layer.workspace(cfg.T), stream)
    if st != m.MOE_OK:
        raise RuntimeError(f"device status {m.status_string(st)}")
    del flush
    # per-kernel durations (same kernels, issued stage by stage between events)
    per_stage, counts = time_stages(layer, d, steps, args.warmup, stream)
    e2e_ms, h2d, d2h = time_e2e(layer, d, steps, args.warmup, stream)
    e2e_ms = max_over_ranks(e2e_ms, world)
    graph_ms = max_over_ranks(time_graph(layer, d, steps, args.warmup, stream), world)
    rl = roofline_numbers(cfg, counts.numpy())
    parity = parity_sample(cfg, layer, d, parity_tokens) if parity_tokens else None
    out = dict(cfg=cfg, steps=steps, ms_total=ms_total, per=per, per_stage=per_stage,
               counts=counts, rl=rl, clocks=clocks, e2e_ms=e2e_ms, h2d=h2d, d2h=d2h,
               graph_ms=graph_ms, parity=parity,
               l2="flushed between steps (512 MiB write, outside the timed intervals)"
               if fits_l2(cfg) else "inputs larger than L2 (expert weights), no flush",
               layer=layer, d=d)
    return out


def measure_quantized(cfg, args, world, peaks, mx=False):
    """The same workload with quantized expert weights: E4M3 with one
    power-of-two scale per row (moe_forward_fp8), or MXFP8, E4M3 with one E8M0
    scale per block of 32 (moe_forward_mx, mx=True). Weights are quantized
    once, then K timed steps of the layer. Roofline: weight bytes are one per
    element plus the scales (4 bytes per row; or the MX scale rows); the
    tensor peak is the measured bf16 burst peak, times the nominal fp8/bf16
    ratio (4.5 / 2.25 = 2) for the E4M3 MMAs (the MXFP8 GEMMs multiply bf16
    values of the codes on the bf16 MMA); the fraction against the sustained
    figure is given beside it."""
    import mixture_experts_layer_route_gb300 as m
    stream = torch.cuda.Stream()
    d = generate(cfg, seed=args.seed, device="cuda")
    cls = m.MoELayerMX if mx else m.MoELayerFP8
    layer = cls(d["W_router"], d["W_gate"], d["W_up"], d["W_down"], cfg.k,
                router_bias=d["router_bias"], Ws_gate=d["Ws_gate"], Ws_up=d["Ws_up"],
                Ws_down=d["Ws_down"], renorm=cfg.renorm)
    for n in ("W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down"):
        d[n] = None  # only the quantized copies stay resident
    torch.cuda.empty_cache()
    ws = layer.workspace(cfg.T)
    steps = args.steps if cfg.T <= 1024 else max(3, args.steps // 8)
    barrier(world)
    ms_total, per = time_forward(layer, d, steps, args.warmup, stream)
    barrier(world)
    ms_total = max_over_ranks(ms_total, world)
    st = m.get_device_status(ws, stream)
    if st != m.MOE_OK:
        raise RuntimeError(f"device status {m.status_string(st)}")
    lay = m.workspace_layout(layer.problem(cfg.T))
    offs = ws[lay["expert_offsets"]:lay["expert_offsets"] + (cfg.E + 2) * 4].view(torch.int32)
    counts = torch.diff(offs[:cfg.E + 1]).cpu().numpy()
    T, H, E, k, I, Is = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.I_shared
    touched = int((counts > 0).sum())

    def expert_bytes(i):  # one expert's gate, up and down matrices
        if mx:
            return 2 * i * (H + m.mx_scale_cols(H)) + H * (i + m.mx_scale_cols(i))
        return 3 * H * i + 4 * (2 * i + H)

    wbytes = touched * expert_bytes(I) + (expert_bytes(Is) if Is else 0)
    bytes_layer = wbytes + 2 * T * H * 2 + E * H * 2
    flop_layer = 2.0 * T * k * 3 * H * I + 2.0 * T * 3 * H * Is
    ms_step = ms_total / steps
    t_mem = bytes_layer / (peaks["hbm_gbs"] * 1e9) * 1e3
    ratio = 1.0 if mx else 2.0
    pk = ratio * peaks["bf16_tflops"]
    t_tc = flop_layer / (pk * 1e12) * 1e3
    t_roof = max(t_mem, t_tc)
    t_roof_sus = max(t_mem, flop_layer / (ratio * 1e12 * peaks["bf16_tflops_sustained"]) * 1e3)
    weights = ("MXFP8: E4M3 codes, one E8M0 scale per 32 elements (moe_forward_mx)" if mx else
               "E4M3, one power-of-two scale per row (moe_forward_fp8)")
    peak_src = ("measured bf16_tflops (burst): the MXFP8 GEMMs of batches over 64 tokens run "
                "the bf16 MMA on converted tiles (decode-sized ones the E4M3 MMA, HBM-bound)"
                if mx else "2 x measured bf16_tflops (burst; nominal fp8/bf16 ratio)")
    return {"value": world * T * steps / (ms_total / 1e3), "unit": "tokens/s",
            "ms_per_step": ms_step, "median_ms": statistics.median(per),
            "weights": weights,
            "layer_roofline": {"t_roof_ms": t_roof, "bound": "hbm" if t_mem >= t_tc else "tensor",
                               "frac": t_roof / ms_step, "frac_vs_sustained": t_roof_sus / ms_step,
                               "bytes_touched": bytes_layer,
                               "flop_routed": flop_layer, "tensor_peak_tflops": pk,
                               "tensor_peak_source": peak_src},
            "experts_touched": touched}


def measure_fp8(cfg, args, world, peaks):
    return measure_quantized(cfg, args, world, peaks, mx=False)


def measure_mx(cfg, args, world, peaks):
    return measure_quantized(cfg, args, world, peaks, mx=True)


def summarize(r, peaks, world, prefix_src):
    """Throughput, the layer's roofline fraction and the dominant kernel's
    roofline for one measured workload. The tensor peak is the measured burst
    bf16 figure (each timed region lasts tens of milliseconds); fractions
    against the sustained figure are given beside it."""
    cfg = r["cfg"]
    steps = r["steps"]
    ms_step = r["ms_total"] / steps
    value = job_tokens_per_s(world, cfg.T, steps, r["ms_total"])
    rl = r["rl"]
    st = dict(zip(STAGES, r["per_stage"]))
    g_ms = st["swiglu_gemm"]
    hbm = peaks["hbm_gbs"]
    tc, tc_sus = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    t_mem = rl["bytes_layer"] / (hbm * 1e9) * 1e3
    t_tc = rl["flop_layer"] / (tc * 1e12) * 1e3
    t_roof = max(t_mem, t_tc)
    t_roof_sus = max(t_mem, rl["flop_layer"] / (tc_sus * 1e12) * 1e3)
    bound = "hbm" if t_mem >= t_tc else "tensor"
    kname = f"grouped_gemm_kernel<{cfg.dtype},gated>"
    if bound == "hbm":
        ach = rl["bytes_gated"] / (g_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": kname, "achieved": ach,
                "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "algorithmic_bytes_per_launch": rl["bytes_gated"]}
    else:
        ach = rl["flop_gated"] / (g_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": kname, "achieved": ach,
                "peak": tc, "unit": "TFLOP/s", "frac": ach / tc, "frac_vs_sustained": ach / tc_sus,
                "algorithmic_flops_per_launch": rl["flop_gated"]}
    roof["peak_source"] = f"{prefix_src} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops, burst'})"
    roof["kernel_ms"] = g_ms
    roof["traffic"] = traffic_for(cfg.name, "swiglu_gemm")
    counts = r["counts"].numpy()
    loads = counts[counts > 0]
    return dict(
        value=value, ms_per_step=ms_step, steps=steps,
        median_ms=statistics.median(r["per"]), p10_ms=sorted(r["per"])[len(r["per"]) // 10],
        p90_ms=sorted(r["per"])[(9 * len(r["per"])) // 10],
        roofline=roof,
        layer_roofline={"t_roof_ms": t_roof, "bound": bound, "frac": t_roof / ms_step,
                        "frac_vs_sustained": t_roof_sus / ms_step,
                        "flop_routed": rl["flop_layer"], "bytes_touched": rl["bytes_layer"],
                        "experts_touched": rl["touched"]},
        stages_ms=st,
        expert_load={"touched": int(len(loads)), "empty": int((counts == 0).sum()),
                     "max": int(counts.max()), "mean": float(counts.mean()),
                     "std_over_mean": float(counts.std() / max(counts.mean(), 1e-9))},
        e2e={"value": world * cfg.T * steps / (r["e2e_ms"] / 1e3), "unit": "tokens/s",
             "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
             "ms_per_step": r["e2e_ms"] / steps},
        graph={"value": world * cfg.T * steps / (r["graph_ms"] / 1e3), "unit": "tokens/s",
               "ms_per_step": r["graph_ms"] / steps,
               "layer_roofline_frac": t_roof / (r["graph_ms"] / steps),
               "how": "the same moe_forward captured once in a CUDA graph, replayed"},
        parity=r["parity"], l2=r["l2"],
    )


WORKLOAD_ORDER = ["qwen3_235b_prefill", "qwen35_397b_zipf", "deepseek_v3", "tiny_f32"]


def workload_entry(cfg, s, fp8, mxfp8=None):
    return {"config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k,
                       "I": cfg.I, "I_shared": cfg.I_shared, "dtype": cfg.dtype,
                       "zipf_s": cfg.zipf_s, "l2": s["l2"]},
            **{k: s[k] for k in ("value", "ms_per_step", "median_ms", "roofline",
                                 "layer_roofline", "stages_ms", "expert_load", "graph", "e2e",
                                 "parity")},
            "unit": "tokens/s", "steps": s["steps"], "fp8": fp8, "mxfp8": mxfp8}


def run_native(args):
    world, rank, local = dist_setup(args)
    import mixture_experts_layer_route_gb300 as m
    from mixture_experts_layer_route_gb300 import build as b
    if rank == 0 or not os.path.exists(m._binding.LIB_PATH):
        b.build()
    barrier(world)
    peaks, src = load_peaks()
    cfg = ALL_CONFIGS[args.config]
    r = measure_config(cfg, args, world, local, with_clocks=True,
                       parity_tokens=args.parity_tokens if rank == 0 else 0)
    s = summarize(r, peaks, world, src)
    clocks = r["clocks"]
    del r
    fp8 = mxfp8 = None
    if args.fp8 and cfg.dtype == "bf16" and cfg.I % 128 == 0 and cfg.I_shared % 128 == 0:
        torch.cuda.empty_cache()
        fp8 = measure_fp8(cfg, args, world, peaks)
        torch.cuda.empty_cache()
        mxfp8 = measure_mx(cfg, args, world, peaks)
    # The other layer shapes, each measured the same way (one at a time: the
    # DeepSeek-V3-shaped layer alone holds ~23 GB of weights).
    others = {}
    names = []
    if args.prefill:
        names = WORKLOAD_ORDER if args.all_workloads else ["qwen3_235b_prefill"]
        names = [n for n in names if n != args.config]
    for name in names:
        torch.cuda.empty_cache()
        c = CONFIGS[name]
        rp = measure_config(c, args, world, local, with_clocks=False,
                            parity_tokens=args.parity_tokens if rank == 0 else 0)
        sp = summarize(rp, peaks, world, src)
        del rp
        f8 = fmx = None
        if args.fp8 and c.dtype == "bf16" and c.I % 128 == 0 and c.I_shared % 128 == 0:
            torch.cuda.empty_cache()
            f8 = measure_fp8(c, args, world, peaks)
            torch.cuda.empty_cache()
            fmx = measure_mx(c, args, world, peaks)
        others[name] = workload_entry(c, sp, f8, fmx)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        torch.cuda.empty_cache()
        layer, d = build_layer(cfg, "cuda", seed=args.seed)
        cpu = cpu_baseline(cfg, d, budget_s=args.cpu_seconds)
        del layer, d
    if rank != 0:
        return
    n_launch = kernels_per_step(cfg) * s["steps"]
    line = {
        "metric": "MoE-layer tokens/sec at 1 GB300 (decode & prefill) + % of HBM / bf16-TC roofline",
        "value": s["value"], "unit": "tokens/s", "n_gpus": world, "steps": s["steps"],
        "warmup": args.warmup, "ms_per_step": s["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if cfg.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k,
                   "I": cfg.I, "I_shared": cfg.I_shared, "renorm": cfg.renorm,
                   "seed": args.seed, "parallelism": f"replicas{world}", "l2": s["l2"]},
        "median_ms": s["median_ms"], "p10_ms": s["p10_ms"], "p90_ms": s["p90_ms"],
        "roofline": s["roofline"], "layer_roofline": s["layer_roofline"],
        "stages_ms": s["stages_ms"], "expert_load": s["expert_load"],
        "e2e": s["e2e"], "graph": s["graph"], "fp8": fp8, "mxfp8": mxfp8, "parity": s["parity"],
        "gpu_launches": n_launch,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "prefill": others.get("qwen3_235b_prefill"),
        "workloads": {k: v for k, v in others.items() if k != "qwen3_235b_prefill"},
    }
    print(json.dumps(line))


def run_reference(args):
    """The CPU oracle as the reference arm: same workload, metric and unit."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = ALL_CONFIGS[args.config]
    # Inputs only: the same seeded generator as the native arm (on the GPU when
    # there is one, for speed); nothing of the native library is loaded.
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    if dev == "cuda":
        torch.cuda.set_device(0)
    d = generate(cfg, seed=args.seed, device=dev)
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        cpu_baseline(cfg, d, budget_s=0.0, max_tokens=8)
    vals, toks, secs = [], 0, 0.0
    for _ in range(args.steps):
        r = cpu_baseline(cfg, d, budget_s=per_step)
        vals.append(r["value"])
        secs += r["seconds"]
        toks += int(r["value"] * r["seconds"] + 0.5)
    value = toks / secs
    line = {"metric": "MoE-layer tokens/sec at 1 GB300 (decode & prefill) + % of HBM / bf16-TC roofline",
            "impl": "reference", "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k,
                       "I": cfg.I, "I_shared": cfg.I_shared, "seed": args.seed},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": r["cores"],
                             "kind": "oracle", "sample": r["sample"]},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="qwen3_235b_decode", choices=sorted(ALL_CONFIGS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-prefill", dest="prefill", action="store_false",
                    help="measure the chosen workload alone (no other layer shape)")
    ap.add_argument("--no-other-workloads", dest="all_workloads", action="store_false",
                    help="besides the chosen workload, measure only the prefill chunk")
    ap.add_argument("--parity-tokens", type=int, default=8,
                    help="tokens per workload checked against the CPU oracle (0: none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", dest="fp8", action="store_false",
                    help="skip the quantized-weight measurements (E4M3 rows, MXFP8) of the "
                         "same workloads")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
