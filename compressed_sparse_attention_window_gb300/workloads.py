"""Workload shapes and the seeded synthetic input generator.

The five workloads are one layer's compressed sparse attention forward for
``m`` tokens at ``start_pos`` (shapes from the sizes DeepSeek-V4.1 Flash uses
on the reference pages: 64 heads of width 512, rope width 64, window 128, and
an indexer of 64 heads x 128).  This module only draws random numbers and
arranges them into the input tensors; it holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle can take their inputs
from it.

Input recipe (all seeded, torch CPU generator unless ``device`` says otherwise):

* bf16 activations ``q [m, nh, hd]``, ``kv [m, hd]``, ``latent [G, hd]``,
  ``q_idx [m, Hi, Di]``, prior window ring ``ring [win, hd]``, prior latent
  cache ``cache [n_c, hd]`` and indexer keys ``k_idx [n_c, Di]``: N(0, 1)
  drawn in f32, rounded to bf16 by torch.
* ``sink [nh]``: f32 N(0, 1).  ``w [m, Hi]``: f32 N(0, 1) / sqrt(Hi * Di).
* ``outliers``: 1% of the elements of every bf16 input (seeded uniform
  positions) multiplied by 20 before the bf16 rounding.
* ``repeat``: tokens repeat in blocks of 8 (kv, q, q_idx, latent rows) and the
  indexer keys repeat in blocks of 4 rows, which makes scores tie.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    m: int
    start_pos: int
    nh: int
    hd: int
    rd: int
    win: int
    ratio: int
    topk: int
    Hi: int
    Di: int
    seed: int
    structure: str = ""  # "", "outliers" or "repeat"

    @property
    def n_c(self) -> int:
        """compress_len: compressed rows that exist after this call."""
        return (self.start_pos + self.m) // self.ratio

    @property
    def G(self) -> int:
        """Latent groups this call completes (rows start_pos/ratio .. n_c-1)."""
        return self.n_c - self.start_pos // self.ratio

    @property
    def n_a(self) -> int:
        """Rows the window indices point into."""
        if self.start_pos == 0:
            return self.m
        if self.m == 1:
            return self.win
        return self.win + self.m

    @property
    def ctopk(self) -> int:
        return 0 if self.n_c == 0 else min(self.topk, self.n_c)

    @property
    def K(self) -> int:
        """Merged index row length: window indices then compressed picks."""
        return self.win + self.ctopk

    @property
    def max_pos(self) -> int:
        """Rows of the RoPE table the call can touch."""
        return self.start_pos + self.m

    @property
    def scale(self) -> float:
        """head_dim^-0.5 as an f32 value."""
        return float(torch.tensor(float(self.hd), dtype=torch.float32).pow(-0.5).item())

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


TINY_PREFILL = Workload("tiny_prefill", m=64, start_pos=0, nh=4, hd=64, rd=16, win=16, ratio=4,
                        topk=8, Hi=2, Di=32, seed=0)
DECODE = Workload("decode", m=1, start_pos=8191, nh=64, hd=512, rd=64, win=128, ratio=4,
                  topk=512, Hi=64, Di=128, seed=1)
PREFILL = Workload("prefill", m=4096, start_pos=0, nh=64, hd=512, rd=64, win=128, ratio=4,
                   topk=512, Hi=64, Di=128, seed=2, structure="outliers")
LONG_DECODE = Workload("long_decode", m=1, start_pos=131071, nh=64, hd=512, rd=64, win=128,
                       ratio=4, topk=2048, Hi=64, Di=128, seed=3)
CHUNKED = Workload("chunked_prefill", m=1024, start_pos=65536, nh=64, hd=512, rd=64, win=128,
                   ratio=128, topk=512, Hi=64, Di=128, seed=4, structure="repeat")

WORKLOADS: Dict[str, Workload] = {w.name: w for w in
                                  (TINY_PREFILL, DECODE, PREFILL, LONG_DECODE, CHUNKED)}


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def _outliers(x: torch.Tensor, g: torch.Generator) -> torch.Tensor:
    """Multiply a seeded 1% of the elements by 20 (x is f32)."""
    n = x.numel()
    k = max(1, n // 100)
    pos = torch.randint(0, n, (k,), generator=g, device=x.device)
    flat = x.reshape(-1)
    flat[pos] = flat[pos] * 20.0
    return x


def _repeat_rows(x: torch.Tensor, block: int) -> torch.Tensor:
    """Copy the first row of every block of ``block`` rows onto the others."""
    idx = (torch.arange(x.shape[0], device=x.device) // block) * block
    return x[idx].contiguous()


def make_inputs(wl: Workload, device: str = "cpu", seed: Optional[int] = None,
                cache_rows: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Seeded synthetic inputs of one workload (see the module docstring).

    ``cache_rows`` sizes the latent cache and the indexer key cache (default
    n_c, at least 1)."""
    s = wl.seed if seed is None else seed
    g = torch.Generator(device=device)
    g.manual_seed(s)
    n_c = wl.n_c
    rows = max(1, n_c if cache_rows is None else cache_rows)

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)

    raw = {
        "q": randn(wl.m, wl.nh, wl.hd),
        "kv": randn(wl.m, wl.hd),
        "latent": randn(max(wl.G, 0), wl.hd),
        "q_idx": randn(wl.m, wl.Hi, wl.Di),
        "ring": randn(wl.win, wl.hd),
        "cache": randn(rows, wl.hd),
        "k_idx": randn(rows, wl.Di),
    }
    sink = randn(wl.nh)
    w = randn(wl.m, wl.Hi) / math.sqrt(wl.Hi * wl.Di)
    if wl.structure == "outliers":
        for k in raw:
            raw[k] = _outliers(raw[k], g)
    elif wl.structure == "repeat":
        for k in ("q", "kv", "q_idx", "latent"):
            if raw[k].shape[0] > 0:
                raw[k] = _repeat_rows(raw[k], 8)
        raw["k_idx"] = _repeat_rows(raw["k_idx"], 4)
    out = {k: _bf16(v) for k, v in raw.items()}
    out["sink"] = sink
    out["w"] = w.contiguous()
    return out


# The output side of the layer (inverse RoPE, grouped wo_a, wo_b).  The pages
# give neither the model width nor the projection's rank or group count; these
# sizes are our choice: 8 groups of 4096 values (8 heads of 512), o_rank 1024,
# model width 7168.
OUT_PROJ = {"groups": 8, "o_rank": 1024, "dim": 7168}


def make_out_proj_weights(nh: int, hd: int, groups: int, o_rank: int, dim: int, seed: int = 7,
                          device: str = "cpu") -> Dict[str, torch.Tensor]:
    """Synthetic projection weights: wo_a [groups*o_rank, nh*hd/groups] and
    wo_b [dim, groups*o_rank], bf16 N(0, 1) / sqrt(fan-in)."""
    g = torch.Generator(device=device).manual_seed(seed)
    gw = nh * hd // groups
    wa = torch.randn(groups * o_rank, gw, generator=g, device=device) / math.sqrt(gw)
    wb = torch.randn(dim, groups * o_rank, generator=g, device=device) / math.sqrt(groups * o_rank)
    return {"wo_a": _bf16(wa), "wo_b": _bf16(wb)}


def bf16_bits(x: torch.Tensor):
    """A bf16 tensor's bit patterns as a numpy uint16 array (CPU copy)."""
    return x.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def from_bits(a, device: str = "cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor."""
    import numpy as np
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy())
    return t.view(torch.bfloat16).to(device)
