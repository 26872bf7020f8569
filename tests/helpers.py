"""Shared pieces of the parity tests: run the oracle and the CUDA path on the
same seeded inputs and compare.

Bars (written in the tests):
* fp4 quantiser outputs, codes and scales, window indices, ring and cache
  contents, indexer scores and top-k index sets: bit-exact.
* attention outputs: |gpu - oracle| <= 2e-2 + 1e-2 * |oracle| elementwise
  (bf16 tolerance; the oracle accumulates in f64).
"""
from __future__ import annotations

import numpy as np
import torch

from compressed_sparse_attention_window_gb300.workloads import Workload, bf16_bits, make_inputs

ATOL = 2e-2
RTOL = 1e-2


def sample_tokens(wl: Workload, n_random: int = 24, seed: int = 0):
    """Tokens the oracle evaluates one by one at full size: the ends, the
    window and ratio boundaries, and a seeded random set."""
    m = wl.m
    fixed = {0, 1, 2, 3, 4, wl.ratio - 1, wl.ratio, wl.win - 1, wl.win, wl.win + 1,
             m // 2, m - 2, m - 1}
    rng = np.random.default_rng(seed)
    rnd = set(rng.integers(0, m, n_random).tolist()) if m > 1 else set()
    return sorted(t for t in fixed | rnd if 0 <= t < m)


def oracle_forward(orc, wl: Workload, inp, tokens=None, fc=None):
    """The oracle's forward (``oracle.forward``) for workload ``wl`` on CPU
    inputs ``inp``, with the indexer, top-k and attention evaluated for
    ``tokens`` (default: all).  The workload supplies only the call's
    parameters (window, ratio, position, top-k, rope width); every row count
    the forward uses is the oracle's own."""
    b = {k: bf16_bits(inp[k]) for k in ("kv", "ring", "latent", "cache", "q_idx", "k_idx", "q")}
    return orc.forward(b["kv"], b["ring"], b["latent"], b["cache"], b["q_idx"], b["k_idx"],
                       inp["w"].numpy(), b["q"], inp["sink"].numpy(), win=wl.win, ratio=wl.ratio,
                       start_pos=wl.start_pos, topk=wl.topk, rd=wl.rd, tokens=tokens, fc=fc)


def osizes(orc, wl: Workload) -> dict:
    """The row counts (n_c, G, n_a, K, ctopk) of workload ``wl``'s call, as
    the oracle derives them."""
    return orc.step_sizes(wl.m, wl.win, wl.ratio, wl.start_pos, wl.topk)


def to_dev(inp, device="cuda"):
    return {k: v.to(device).contiguous() for k, v in inp.items()}


def assert_idx_sets_equal(gpu_idx: np.ndarray, ora_idx: np.ndarray, win: int):
    """Window part and compressed part compared as sets (with -1 counts)."""
    assert gpu_idx.shape == ora_idx.shape, (gpu_idx.shape, ora_idx.shape)
    for r in range(gpu_idx.shape[0]):
        for lo, hi in ((0, win), (win, gpu_idx.shape[1])):
            a = np.sort(gpu_idx[r, lo:hi])
            b = np.sort(ora_idx[r, lo:hi])
            assert np.array_equal(a, b), (r, lo, hi, np.setdiff1d(a, b)[:8], np.setdiff1d(b, a)[:8])


def attn_close(gpu_o: np.ndarray, ora_o: np.ndarray):
    """Returns (ok, max_abs_err, worst_ratio) for the attention tolerance."""
    g = gpu_o.astype(np.float64)
    err = np.abs(g - ora_o)
    bound = ATOL + RTOL * np.abs(ora_o)
    return bool(np.all(err <= bound)), float(err.max()), float((err / bound).max())


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return bf16_bits(t)


def bf16_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


__all__ = ["sample_tokens", "oracle_forward", "osizes", "to_dev", "assert_idx_sets_equal", "attn_close",
           "make_inputs", "bf16_to_np", "bf16_f32", "ATOL", "RTOL"]
