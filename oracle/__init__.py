"""CPU oracle for the compressed sparse attention forward (test infrastructure).

This package is TEST INFRASTRUCTURE.  It is the independent, plain and slow
definition of what the hot path computes, written in C (``ds41_oracle.c``) and
driven from Python through ctypes.  Only the test suite, the smoke check and
the CPU baseline leg of ``bench.py`` may import it; the product library never
calls it and shares no code with it.

Every function cites the page it follows (page title + function/section):

* ``metrale_model_arch/deepseek_v41_ref/compress.rs`` -- the CPU reference:
  ``to_e2m1_rne``, ``fp4_quant_e8m0_inplace``, ``fp4_quant_e4m3_inplace``,
  ``yarn_freqs_cis``, ``attention_any`` (ring update, latent branch, merge,
  ``sparse_attn`` call with ``scale = head_dim^-0.5``).
* ``metrale_model_arch/attn_v41/forward.rs`` -- ``AttnV41::forward``: the
  window ring copies, group positions, cache offset and index merge.

Parity unpinned (fixed by a reading, not by a value on the pages): the
indexer's score formula, apply_rotary's choice of dims and pairing, the YaRN
constants.

bf16 tensors travel as ``numpy.uint16`` arrays of their bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ds41_oracle.c")
_LIB = os.path.join(_HERE, "libds41_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-fopenmp"]


def build(force: bool = False) -> str:
    """Compile ``ds41_oracle.c`` into ``libds41_oracle.so`` with gcc (no fast-math,
    no FMA contraction).  Rebuilds when the source is newer than the library."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float


def _sig(lib):
    def s(name, res, *args):
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = list(args)
    s("ds41o_bf16_to_f32", _F, ctypes.c_uint16)
    s("ds41o_f32_to_bf16_rne", ctypes.c_uint16, _F)
    s("ds41o_to_e2m1_rne", _F, _F)
    s("ds41o_pow2_ceil", _F, _F)
    s("ds41o_f32_to_e4m3_rne", ctypes.c_uint8, _F)
    s("ds41o_e4m3_to_f32", _F, ctypes.c_uint8)
    s("ds41o_fp4_quant_e8m0", None, _P, _I64, _I64, _P, _P)
    s("ds41o_fp4_quant_e4m3", None, _P, _I64, _I64, _P, _P)
    s("ds41o_fp4_quant_bf16", None, _P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int)
    s("ds41o_yarn_inv_freqs", None, _I64, _I64, _F, _F, _F, _F, _P)
    s("ds41o_yarn_freqs_cis", None, _I64, _I64, _I64, _F, _F, _F, _F, _P)
    s("ds41o_apply_rotary", None, _P, _I64, _I64, _I64, _P, _P, ctypes.c_int)
    s("ds41o_rows_a_len", _I64, _I64, _I64, _I64)
    s("ds41o_window_ring_write", None, _P, _P, _P, _I64, _I64, _I64, _I64)
    s("ds41o_window_topk_idxs", None, _I64, _I64, _I64, _P)
    s("ds41o_new_groups", _I64, _I64, _I64, _I64)
    s("ds41o_compress_len", _I64, _I64, _I64, _I64)
    s("ds41o_merged_len", _I64, _I64, _I64, _I64)
    s("ds41o_attn_scale", _F, _I64)
    s("ds41o_compress_latent_write", None, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64)
    s("ds41o_visible_rows", _I64, _I64, _I64, _I64, _I64)
    s("ds41o_indexer_scores", _I64, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _P,
      _I64)
    s("ds41o_topk_merge", None, _P, _P, _P, _I64, _P, _I64, _I64, _I64, _I64, _I64, _I64)
    s("ds41o_sparse_attn", _I64, _P, _P, _I64, _P, _I64, _P, _I64, _P, _F, _P, _P, _I64, _I64,
      _P, _I64)
    s("ds41o_attn_out_proj", None, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64,
      _I64, _P, _I64)
    for n in ("ds41o_to_e2m1_rne_array", "ds41o_f32_to_bf16_array", "ds41o_f32_to_e4m3_array",
              "ds41o_e4m3_to_f32_array", "ds41o_pow2_ceil_array"):
        s(n, None, _P, _P, _I64)
    s("ds41o_num_threads", ctypes.c_int)
    s("ds41o_set_num_threads", None, ctypes.c_int)


def lib():
    """The loaded oracle library (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            _lib = ctypes.CDLL(path)
            _sig(_lib)
        return _lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


# --------------------------------------------------------------------------
# bf16 helpers (bit patterns as uint16)
# --------------------------------------------------------------------------
def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact: bf16 is the upper half word)."""
    h = _c(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


# Array versions through small C loops (used by the exhaustive pins).
def _array_fn(cname: str, in_dtype, out_dtype):
    def run(x):
        x = _c(x, in_dtype)
        out = np.empty(x.shape, out_dtype)
        getattr(lib(), cname)(_ptr(x), _ptr(out), _I64(x.size))
        return out
    run.__name__ = cname
    return run


#: compress.rs imports ``to_bf16_rne``; reading: IEEE binary32 -> bfloat16 RNE.
f32_to_bf16 = _array_fn("ds41o_f32_to_bf16_array", np.float32, np.uint16)
#: compress.rs ``to_e2m1_rne`` elementwise (f32 in, f32 out).
to_e2m1 = _array_fn("ds41o_to_e2m1_rne_array", np.float32, np.float32)
#: compress.rs imports ``f32_to_e4m3_rne``; reading: OCP E4M3, RNE, saturating.
f32_to_e4m3 = _array_fn("ds41o_f32_to_e4m3_array", np.float32, np.uint8)
#: compress.rs imports ``e4m3_to_f32``.
e4m3_to_f32 = _array_fn("ds41o_e4m3_to_f32_array", np.uint8, np.float32)
#: compress.rs imports ``pow2_ceil``; reading: smallest power of two >= x.
pow2_ceil = _array_fn("ds41o_pow2_ceil_array", np.float32, np.float32)


# --------------------------------------------------------------------------
# Quantisers
# --------------------------------------------------------------------------
def fp4_quant(x_bf16: np.ndarray, block: int, e4m3: bool):
    """compress.rs ``fp4_quant_e8m0_inplace`` (block 32) / ``fp4_quant_e4m3_inplace``
    (block 16) on bf16 rows.  Returns (y bf16 bits, codes uint8 [rows, cols/2],
    scales uint8 [rows, cols/block])."""
    x = _c(x_bf16, np.uint16)
    rows, cols = (x.shape if x.ndim == 2 else (1, x.size))
    y = np.empty((rows, cols), np.uint16)
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // block), np.uint8)
    lib().ds41o_fp4_quant_bf16(_ptr(x), _ptr(y), _ptr(codes), _ptr(scales), rows, cols, block,
                               1 if e4m3 else 0)
    return y.reshape(x.shape), codes, scales


def fp4_quant_f32(x: np.ndarray, block: int, e4m3: bool):
    """The page's in-place f32 quantisers on a flat f32 array (copy returned)."""
    y = _c(x, np.float32).copy().ravel()
    nb = y.size // block
    codes = np.zeros(y.size // 2, np.uint8)
    scales = np.zeros(nb, np.uint8)
    fn = lib().ds41o_fp4_quant_e4m3 if e4m3 else lib().ds41o_fp4_quant_e8m0
    fn(_ptr(y), y.size, block, _ptr(codes), _ptr(scales))
    return y, codes, scales


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------
YARN_DEFAULTS = dict(orig=65536, base=160000.0, factor=16.0, beta_fast=32.0, beta_slow=1.0)


def yarn_inv_freqs(dim, orig, base, factor, beta_fast, beta_slow) -> np.ndarray:
    out = np.empty(dim // 2, np.float32)
    lib().ds41o_yarn_inv_freqs(dim, orig, base, factor, beta_fast, beta_slow, _ptr(out))
    return out


def yarn_freqs_cis(dim, seqlen, orig=65536, base=160000.0, factor=16.0, beta_fast=32.0,
                   beta_slow=1.0) -> np.ndarray:
    """compress.rs ``yarn_freqs_cis``: f32 [seqlen, dim/2, 2] of (cos, sin)."""
    out = np.empty((seqlen, dim // 2, 2), np.float32)
    lib().ds41o_yarn_freqs_cis(dim, seqlen, orig, base, factor, beta_fast, beta_slow, _ptr(out))
    return out


def apply_rotary(buf: np.ndarray, rd: int, pos: Sequence[int], fc: np.ndarray,
                 inverse: bool = False) -> np.ndarray:
    """Reading of compress.rs ``apply_rotary``: rotate the last rd dims of each row."""
    b = _c(buf, np.float32).copy()
    rows, hd = b.shape
    p = _c(pos, np.int64)
    fcc = _c(fc, np.float32)
    lib().ds41o_apply_rotary(_ptr(b), rows, hd, rd, _ptr(p), _ptr(fcc), 1 if inverse else 0)
    return b


# --------------------------------------------------------------------------
# Window ring, window indices, latent write
# --------------------------------------------------------------------------
def rows_a_len(m, win, start_pos) -> int:
    return int(lib().ds41o_rows_a_len(m, win, start_pos))


def window_ring_write(kv: np.ndarray, ring: np.ndarray, win: int, start_pos: int):
    """forward.rs window-ring copies / compress.rs ring update.  Returns
    (ring after the write, rows_a)."""
    kv = _c(kv, np.uint16)
    ring2 = _c(ring, np.uint16).copy()
    m, hd = kv.shape
    n_a = rows_a_len(m, win, start_pos)
    rows_a = np.zeros((n_a, hd), np.uint16)
    lib().ds41o_window_ring_write(_ptr(kv), _ptr(ring2), _ptr(rows_a), m, hd, win, start_pos)
    return ring2, rows_a


def window_topk_idxs(win: int, m: int, start_pos: int) -> np.ndarray:
    out = np.empty((m, win), np.int32)
    lib().ds41o_window_topk_idxs(win, m, start_pos, _ptr(out))
    return out


def new_groups(m, ratio, start_pos) -> int:
    """Groups of ``ratio`` positions the call of m tokens at start_pos completes."""
    return int(lib().ds41o_new_groups(m, ratio, start_pos))


def compress_len(m, ratio, start_pos) -> int:
    """forward.rs / compress.rs ``compress_len``: compressed rows after the call."""
    return int(lib().ds41o_compress_len(m, ratio, start_pos))


def merged_len(win, topk, n_c) -> int:
    """Length of a merged index row: win window indices + min(topk, n_c) picks."""
    return int(lib().ds41o_merged_len(win, topk, n_c))


def step_sizes(m: int, win: int, ratio: int, start_pos: int, topk: int) -> dict:
    """The row counts of one call as the oracle derives them: n_c
    (compress_len), G (new groups), n_a (rows_a length, the picks' offset),
    K (merged row length) and ctopk = K - win."""
    n_c = compress_len(m, ratio, start_pos)
    K = merged_len(win, topk, n_c)
    return {"n_c": n_c, "G": new_groups(m, ratio, start_pos),
            "n_a": rows_a_len(m, win, start_pos), "K": K, "ctopk": K - win}


def compress_latent_write(latent: np.ndarray, fc: np.ndarray, cache: np.ndarray, rd: int,
                          ratio: int, start_pos: int, m: int, with_codes: bool = True):
    """forward.rs latent branch / compress.rs latent branch for a call of m
    tokens at start_pos: the oracle's own ``new_groups`` decides how many
    latent rows the call writes, and ``latent`` must hold exactly that many.
    Returns (cache after, codes [rows, hd/2], scales [rows, hd/16]) where
    codes/scales are filled only for the rows written."""
    lat = _c(latent, np.uint16)
    G = new_groups(m, ratio, start_pos)
    assert lat.ndim == 2 and lat.shape[0] == max(G, 0), (
        f"latent holds {lat.shape[0]} rows, the call completes {G} groups")
    hd = lat.shape[1]
    c2 = _c(cache, np.uint16).copy()
    rows = c2.shape[0]
    codes = np.zeros((rows, hd // 2), np.uint8) if with_codes else None
    scales = np.zeros((rows, hd // 16), np.uint8) if with_codes else None
    lib().ds41o_compress_latent_write(_ptr(lat), _ptr(_c(fc, np.float32)), _ptr(c2), _ptr(codes),
                                      _ptr(scales), G, hd, rd, ratio, start_pos)
    return c2, codes, scales


# --------------------------------------------------------------------------
# Indexer, top-k, sparse attention
# --------------------------------------------------------------------------
def visible_rows(t, start_pos, ratio, n_c) -> int:
    return int(lib().ds41o_visible_rows(t, start_pos, ratio, n_c))


def indexer_scores(q_idx: np.ndarray, k_idx: np.ndarray, w: np.ndarray, ratio: int,
                   start_pos: int, tokens: Optional[Sequence[int]] = None,
                   want_acc: bool = False):
    """Reading of the indexer (compress.rs precision header).  q_idx [m,Hi,Di] bf16,
    k_idx [n_c,Di] bf16, w [m,Hi] f32.  Returns (scores bf16 [len(tokens), n_c],
    number of inexact f32 dots), plus the f32 head sums when ``want_acc``."""
    q = _c(q_idx, np.uint16)
    k = _c(k_idx, np.uint16)
    ww = _c(w, np.float32)
    m, Hi, Di = q.shape
    n_c = k.shape[0]
    tk = _c(range(m) if tokens is None else tokens, np.int64)
    out = np.empty((tk.size, n_c), np.uint16)
    acc = np.empty((tk.size, n_c), np.float32) if want_acc else None
    bad = lib().ds41o_indexer_scores(_ptr(q), _ptr(k), _ptr(ww), _ptr(out), _ptr(acc), m, Hi, Di,
                                     n_c, ratio, start_pos, _ptr(tk), tk.size)
    if want_acc:
        return out, int(bad), acc
    return out, int(bad)


def topk_merge(scores: np.ndarray, win_idx: np.ndarray, n_c: int, win: int, ratio: int,
               start_pos: int, topk: int, offset: int,
               tokens: Optional[Sequence[int]] = None) -> np.ndarray:
    """Per-query top-k (ties to the lower row) merged after the window indices.
    scores / win_idx hold one row per entry of ``tokens``."""
    sc = _c(scores, np.uint16)
    wi = _c(win_idx, np.int32)
    tk = _c(range(sc.shape[0]) if tokens is None else tokens, np.int64)
    ctopk = 0 if n_c == 0 else min(topk, n_c)
    out = np.empty((tk.size, win + ctopk), np.int32)
    lib().ds41o_topk_merge(_ptr(sc), _ptr(wi), _ptr(out), tk.size, _ptr(tk), n_c, win, ratio,
                           start_pos, topk, offset)
    return out


def sparse_attn(q: np.ndarray, rows_a: np.ndarray, rows_b: Optional[np.ndarray],
                idx: np.ndarray, sink: np.ndarray, scale: float,
                tokens: Optional[Sequence[int]] = None):
    """Reading of ``sparse_attn`` (compress.rs): f64 attention with the sink in the
    denominator.  q [m,nh,hd] bf16; idx holds one row per entry of ``tokens``.
    Returns (o f64 [nt,nh,hd], lse f64 [nt,nh], number of out-of-range indices)."""
    qq = _c(q, np.uint16)
    m, nh, hd = qq.shape
    ra = _c(rows_a, np.uint16)
    n_a = ra.shape[0]
    if rows_b is None:
        rb = np.zeros((1, hd), np.uint16)
        n_c = 0
    else:
        rb = _c(rows_b, np.uint16)
        n_c = rb.shape[0]
    ii = _c(idx, np.int32)
    K = ii.shape[1]
    tk = _c(range(ii.shape[0]) if tokens is None else tokens, np.int64)
    o = np.empty((tk.size, nh, hd), np.float64)
    lse = np.empty((tk.size, nh), np.float64)
    bad = lib().ds41o_sparse_attn(_ptr(qq), _ptr(ra), n_a, _ptr(rb), n_c, _ptr(ii), K,
                                  _ptr(_c(sink, np.float32)), float(scale), _ptr(o), _ptr(lse),
                                  nh, hd, _ptr(tk), tk.size)
    return o, lse, int(bad)


def attn_out_proj(o: np.ndarray, fc: np.ndarray, wo_a: np.ndarray, wo_b: np.ndarray, rd: int,
                  groups: int, start_pos: int, tokens: Optional[Sequence[int]] = None):
    """Reading of the output side of ``attention_any`` (compress.rs): inverse
    RoPE of o at each token's position, the grouped wo_a projection rounded to
    bf16, then ``linear_bf16`` with wo_b.  o [m,nh,hd] bf16 bits, wo_a
    [groups*o_rank, nh*hd/groups] and wo_b [dim, groups*o_rank] bf16 bits.
    Returns (og bf16 bits [nt, groups*o_rank], out f64 [nt, dim])."""
    oo = _c(o, np.uint16)
    m, nh, hd = oo.shape
    wa = _c(wo_a, np.uint16)
    wb = _c(wo_b, np.uint16)
    gr, gw = wa.shape
    dim = wb.shape[0]
    assert nh * hd == groups * gw and gr % groups == 0 and wb.shape[1] == gr
    tk = _c(range(m) if tokens is None else tokens, np.int64)
    og = np.empty((tk.size, gr), np.uint16)
    out = np.empty((tk.size, dim), np.float64)
    lib().ds41o_attn_out_proj(_ptr(oo), _ptr(_c(fc, np.float32)), _ptr(wa), _ptr(wb), _ptr(og),
                              _ptr(out), nh, hd, rd, groups, gr // groups, dim, start_pos, _ptr(tk),
                              tk.size)
    return og, out


def attn_scale(hd: int) -> float:
    """compress.rs attention_any: ``scale = (hd as f32).powf(-0.5)``."""
    return float(lib().ds41o_attn_scale(hd))


def forward(kv, ring, latent, cache, q_idx, k_idx, w, q, sink, *, win: int, ratio: int,
            start_pos: int, topk: int, rd: int, tokens: Optional[Sequence[int]] = None,
            fc: Optional[np.ndarray] = None, timings: Optional[dict] = None) -> dict:
    """One layer's forward in the order of forward.rs AttnV41::forward and
    compress.rs attention_any: ring write + window indices, latent write,
    indexer scores + top-k + merge (only when a compressed row exists),
    sparse attention with the sink.  bf16 tensors as uint16 bit arrays: kv
    [m, hd], ring [win, hd], latent [G, hd], cache [>= n_c, hd], q_idx
    [m, Hi, Di], k_idx [>= n_c, Di], q [m, nh, hd]; w [m, Hi] and sink [nh]
    f32.  Every row count (n_c, G, n_a, K) comes from this module's own
    functions.  The indexer, top-k and attention run for ``tokens`` (default:
    all).  ``timings``, when given, accumulates seconds per stage under
    "window_ring_write", "compress_latent_write", "indexer_topk" and
    "sparse_attn_sink_fwd"."""
    import time
    m = np.asarray(kv).shape[0]
    hd = np.asarray(kv).shape[1]
    sz = step_sizes(m, win, ratio, start_pos, topk)
    n_c = sz["n_c"]
    toks = list(range(m)) if tokens is None else list(tokens)

    def tick(name, t0):
        if timings is not None:
            timings[name] = timings.get(name, 0.0) + time.perf_counter() - t0

    t0 = time.perf_counter()
    ring2, rows_a = window_ring_write(kv, ring, win, start_pos)
    win_idx = window_topk_idxs(win, m, start_pos)
    tick("window_ring_write", t0)
    if fc is None:
        fc = yarn_freqs_cis(rd, start_pos + m)
    t0 = time.perf_counter()
    cache2, codes, scales = compress_latent_write(latent, fc, cache, rd, ratio, start_pos, m)
    tick("compress_latent_write", t0)
    res = dict(ring=ring2, rows_a=rows_a, win_idx=win_idx, cache=cache2, codes=codes,
               scales=scales, tokens=toks, fc=fc, sizes=sz)
    if n_c > 0:
        t0 = time.perf_counter()
        sc, bad = indexer_scores(q_idx, _c(k_idx, np.uint16)[:n_c], w, ratio, start_pos,
                                 tokens=toks)
        assert bad == 0, f"{bad} indexer dots are not exact in f32 for these inputs"
        idx = topk_merge(sc, win_idx[toks], n_c, win, ratio, start_pos, topk, sz["n_a"],
                         tokens=toks)
        tick("indexer_topk", t0)
        res["scores"] = sc
        rows_b = cache2[:n_c]
    else:
        idx = win_idx[toks]
        rows_b = None
    assert idx.shape[1] == sz["K"]
    res["idx"] = idx
    t0 = time.perf_counter()
    o, lse, bad = sparse_attn(q, rows_a, rows_b, idx, sink, attn_scale(hd), tokens=toks)
    tick("sparse_attn_sink_fwd", t0)
    assert bad == 0
    res["o"], res["lse"] = o, lse
    return res


def num_threads() -> int:
    return int(lib().ds41o_num_threads())


def set_num_threads(n: int) -> None:
    lib().ds41o_set_num_threads(int(n))
