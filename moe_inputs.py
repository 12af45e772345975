"""Seeded synthetic inputs for the MoE layer forward pass.

This module is shared by the tests, the benchmark and the smoke check: it is the
only code that both the CUDA path and the CPU oracle receive data from. It draws
random tensors and rejects draws whose routing would be numerically fragile; it
produces no expected value and implements none of the layer's arithmetic beyond
that rejection test (a float64 matmul plus a sort, used only to decide whether a
row of x is redrawn).

Shapes follow the MoE layers the source pages discuss:

* "Hosting Qwen on Blackwell" (Perplexity blog): Qwen3-235B, 128 experts,
  8 routed per token (tokens-per-expert discussion of the prefill section).
* "Lower latency and higher throughput with multi-node DeepSeek deployment"
  (Perplexity blog), section "Expert Parallelism": 256 routed experts plus one
  shared expert, 8 experts per token.
* Qwen3.5-397B on TPU v7x (Chinese write-up of a Google post), sections 1.1,
  3.1 and 3.2.1: hidden 4096, 512 experts, top-10, 1024 batched tokens.

Init: x ~ N(0,1); router, gate and up weights ~ N(0, 1/H); down weights
~ N(0, 1/I), so router logits are ~ N(0,1). Rows of x whose top-(k+1) router
logits (float64, on the already-rounded inputs) have an adjacent gap below
``MARGIN`` are redrawn from a second seeded stream until none remains, so the
top-k set and its order do not depend on fp32 summation order.
"""
from __future__ import annotations

import dataclasses
import math

import torch

MARGIN = 1e-3


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int          # tokens
    H: int          # hidden size
    E: int          # routed experts
    k: int          # experts per token
    I: int          # routed expert intermediate size
    I_shared: int = 0   # shared expert intermediate size (0: no shared expert)
    dtype: str = "bf16"  # "bf16" or "f32": x, weights, h and y
    renorm: int = 1
    zipf_s: float = 0.0  # >0: per-expert router bias -s*ln(rank)

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


# The five layer shapes (names describe the layer, sizes are explicit).
CONFIGS = {
    "tiny_f32": MoEConfig("tiny_f32", T=64, H=256, E=8, k=2, I=512, dtype="f32"),
    "qwen3_235b_decode": MoEConfig("qwen3_235b_decode", T=64, H=4096, E=128, k=8, I=1536),
    "qwen3_235b_prefill": MoEConfig("qwen3_235b_prefill", T=8192, H=4096, E=128, k=8, I=1536),
    "qwen35_397b_zipf": MoEConfig("qwen35_397b_zipf", T=1024, H=4096, E=512, k=10, I=1024,
                                  zipf_s=1.1),
    "deepseek_v3": MoEConfig("deepseek_v3", T=4096, H=7168, E=256, k=8, I=2048, I_shared=2048),
}

# Reduced shapes for ncu captures: the same per-expert token counts and matrix
# sizes as the decode / prefill layers above, with fewer experts so that a
# capture holds ~1.5 GB on the device (still well above the 129 MB L2).
PROFILE_CONFIGS = {
    "qwen3_235b_prefill_e32": MoEConfig("qwen3_235b_prefill_e32", T=2048, H=4096, E=32, k=8,
                                        I=1536),
    "qwen3_235b_decode_e32": MoEConfig("qwen3_235b_decode_e32", T=16, H=4096, E=32, k=8,
                                       I=1536),
    # the prefill chunk's router shape (T=8192, H=4096, E=128) with tiny experts
    "qwen3_235b_prefill_router": MoEConfig("qwen3_235b_prefill_router", T=8192, H=4096, E=128,
                                           k=8, I=64),
}


def _randn(shape, gen, device, scale, dtype, chunk_rows=None):
    """N(0, scale^2) drawn in fp32 and rounded to dtype, chunked along dim 0."""
    out = torch.empty(shape, dtype=dtype, device=device)
    n0 = shape[0]
    step = chunk_rows or n0
    for a in range(0, n0, step):
        b = min(n0, a + step)
        t = torch.randn((b - a,) + tuple(shape[1:]), generator=gen, device=device,
                        dtype=torch.float32)
        if scale != 1.0:
            t.mul_(scale)
        out[a:b].copy_(t)
        del t
    return out


def _bad_rows(x, Wr, bias, k):
    """Rows whose top-(k+1) float64 logits have an adjacent gap < MARGIN."""
    lg = x.double() @ Wr.double().t()
    if bias is not None:
        lg += bias.double()
    kk = min(k + 1, lg.shape[1])
    top = torch.topk(lg, kk, dim=1, sorted=True).values
    if kk < 2:
        return torch.zeros(lg.shape[0], dtype=torch.bool, device=lg.device)
    gaps = top[:, :-1] - top[:, 1:]
    return (gaps < MARGIN).any(dim=1)


def generate(cfg: MoEConfig, seed: int = 0, device="cpu", enforce_margin: bool = True,
             max_redraws: int = 64):
    """Return a dict of input tensors for ``cfg`` on ``device``.

    Keys: x [T,H], W_router [E,H], router_bias [E] fp32 or None, W_gate [E,I,H],
    W_up [E,I,H], W_down [E,H,I], and Ws_gate [Is,H], Ws_up [Is,H], Ws_down [H,Is]
    (None without a shared expert). All in cfg's dtype except router_bias.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    dt = cfg.torch_dtype
    T, H, E, I = cfg.T, cfg.H, cfg.E, cfg.I
    sH, sI = 1.0 / math.sqrt(H), 1.0 / math.sqrt(I)
    x = _randn((T, H), g, dev, 1.0, dt)
    Wr = _randn((E, H), g, dev, sH, dt)
    per = max(1, (1 << 26) // max(1, I * H))  # experts per fp32 chunk (<= 256 MiB)
    Wg = _randn((E, I, H), g, dev, sH, dt, per)
    Wu = _randn((E, I, H), g, dev, sH, dt, per)
    Wd = _randn((E, H, I), g, dev, sI, dt, per)
    Ws_gate = Ws_up = Ws_down = None
    if cfg.I_shared:
        Is = cfg.I_shared
        Ws_gate = _randn((Is, H), g, dev, sH, dt)
        Ws_up = _randn((Is, H), g, dev, sH, dt)
        Ws_down = _randn((H, Is), g, dev, 1.0 / math.sqrt(Is), dt)
    bias = None
    if cfg.zipf_s > 0:
        rank = torch.randperm(E, generator=g, device=dev).to(torch.float64) + 1.0
        bias = (-cfg.zipf_s * torch.log(rank)).to(torch.float32)
    if enforce_margin and T > 0:
        g2 = torch.Generator(device=dev)
        g2.manual_seed(seed * 7919 + 1)
        for _ in range(max_redraws):
            bad = _bad_rows(x, Wr, bias, cfg.k)
            nb = int(bad.sum())
            if nb == 0:
                break
            idx = bad.nonzero().flatten()
            x[idx] = torch.randn((nb, H), generator=g2, device=dev).to(dt)
        else:
            raise RuntimeError("router margin could not be enforced")
    return dict(x=x, W_router=Wr, router_bias=bias, W_gate=Wg, W_up=Wu, W_down=Wd,
                Ws_gate=Ws_gate, Ws_up=Ws_up, Ws_down=Ws_down)


def generate_hidden(rows: int, I: int, seed: int, device="cpu", dtype=torch.bfloat16):
    """A seeded stand-in for the intermediate activations h [rows, I], used to
    test the down projection + combine stage on its own. Scale ~ the magnitude
    of silu(g)*u for unit-variance g and u."""
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return _randn((rows, I), g, torch.device(device), 0.5, dtype)


def generate_routing(T: int, E: int, k: int, seed: int, zipf_s: float = 0.0):
    """Seeded routing tables (ids [T,k] int32, distinct per row; weights [T,k]
    fp32 positive) for stage tests that bypass the router."""
    g = torch.Generator()
    g.manual_seed(seed)
    if zipf_s > 0:
        p = torch.arange(1, E + 1, dtype=torch.float64) ** (-zipf_s)
        ids = torch.stack([torch.multinomial(p, k, replacement=False, generator=g)
                           for _ in range(T)]) if T else torch.zeros(0, k, dtype=torch.int64)
    else:
        ids = torch.argsort(torch.rand(T, E, generator=g), dim=1)[:, :k]
    w = torch.rand(T, k, generator=g) + 0.05
    w = w / w.sum(dim=1, keepdim=True)
    return ids.to(torch.int32).contiguous(), w.to(torch.float32).contiguous()
