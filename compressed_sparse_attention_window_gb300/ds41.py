"""Thin ctypes binding of ``libds41.so`` (declared in ``include/ds41.h``).

Every function here only checks and marshals torch tensors (device, dtype,
contiguity) into the C ABI and passes the current CUDA stream; all arithmetic
runs in the library's CUDA kernels.  There is no fallback: if the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Dict, NamedTuple, Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libds41.so")

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t

ERRORS = {1: "DS41_E_ARG", 2: "DS41_E_RANGE", 3: "DS41_E_CUDA", 4: "DS41_E_INDEX",
          5: "DS41_E_WORKSPACE", 6: "DS41_E_TIMEOUT"}

#: Exported symbols of include/ds41.h and their (restype, argtypes).
SIGNATURES = {
    "ds41_last_error": (ctypes.c_char_p, []),
    "ds41_device_status": (ctypes.c_int, [_P, ctypes.c_int]),
    "ds41_fp4_quant_e8m0": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _P]),
    "ds41_fp4_quant_e4m3": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _P]),
    "ds41_yarn_freqs_cis": (ctypes.c_int, [_P, _I64, _I64, _I64, _F, _F, _F, _F, _P]),
    "ds41_rows_a_len": (_I64, [_I64, _I64, _I64]),
    "ds41_step_sizes": (ctypes.c_int, [_I64, _I64, _I64, _I64, _I64, _P]),
    "ds41_window_ring_write": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P]),
    "ds41_compress_latent_write": (ctypes.c_int, [_P, _P, _I64, _P, _I64, _P, _P, _I64, _I64, _I64,
                                                  _I64, _I64, _I64, _P]),
    "ds41_indexer_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I64, ctypes.c_int]),
    "ds41_indexer_topk": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64,
                                         _I64, _I64, _I64, _P, _SZ, _P]),
    "ds41_indexer_mxf4_workspace_bytes": (_SZ, [_I64, _I64, ctypes.c_int]),
    "ds41_indexer_topk_mxf4": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                              _I64, _I64, _I64, _I64, _I64, _P, _SZ, _P]),
    "ds41_sparse_attn_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I64]),
    "ds41_csa_forward_reuse": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _P, _F, _P, _P, _P,
                                              _P, _I64, _I64, _I64, _I64, _I64, _I64, _P, ctypes.c_size_t,
                                              _P]),
    "ds41_attn_out_proj": (ctypes.c_int, [_P, _P, _I64, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                          _I64, _I64, _I64, _I64, _P]),
    "ds41_sparse_attn_sink_fwd": (ctypes.c_int, [_P, _P, _I64, _P, _I64, _P, _I64, _P, _F, _P, _P,
                                                 _I64, _I64, _I64, _P, _SZ, _P]),
    "ds41_csa_workspace_bytes": (_SZ, [_I64] * 9),
    "ds41_csa_fp4_workspace_bytes": (_SZ, [_I64] * 7),
    "ds41_csa_forward_fp4": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _P, _P, _P, _I64, _P, _P,
                                            _P, _P, _P, _F, _P, _P, _P, _P] + [_I64] * 10
                             + [_P, _SZ, _P]),
    "ds41_csa_forward": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _P, _I64, _P, _P, _P, _P, _F,
                                        _P, _P, _P, _P] + [_I64] * 10 + [_P, _SZ, _P]),
    "ds41_csa_forward_host": (ctypes.c_int, [_P] * 6 + [_P, _P, _P, _P, _P, _P, _I64, _P, _I64, _P, _P,
                                             _P, _P, _F, _P, _P, _P, _P] + [_I64] * 10 + [_P, _SZ, _P]),
    "ds41_step_inputs_bytes": (_SZ, [_I64] * 7),
    "ds41_csa_forward_host_packed": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _P, _I64, _P, _P, _F,
                                                    _P, _P, _P, _P] + [_I64] * 10 + [_P, _SZ, _P]),
    "ds41_host_step_create": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), _P, _P, _P, _P, _P, _P, _I64,
                                             _P, _I64, _P, _P, _F, _P, _P, _P, _P] + [_I64] * 10
                              + [_P, _SZ]),
    "ds41_host_step_launch": (ctypes.c_int, [_P, _P]),
    "ds41_host_step_destroy": (ctypes.c_int, [_P]),
    "ds41_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint32, ctypes.c_int, _P, _P]),
    "ds41_sparse_attn_noalloc_capacity": (_SZ, []),
    "ds41_sparse_attn_sink_fwd_noalloc": (ctypes.c_int, [_P, _P, _I64, _P, _I64, _P, _I64, _P, _F,
                                                         _P, _P, _I64, _I64, _I64, _P]),
}


class DS41Error(RuntimeError):
    """A libds41 entry point returned an error code."""

    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed with {ERRORS.get(code, code)}: {msg}")
        self.code = code


def load(path: Optional[str] = None):
    """Load libds41.so (built by ``build.py``); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with "
                           "`python -m compressed_sparse_attention_window_gb300.build`")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _call(name: str, *args) -> None:
    lib = load()
    rc = getattr(lib, name)(*args)
    if rc != 0:
        raise DS41Error(name, rc, lib.ds41_last_error().decode(errors="replace"))


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _ptr(t: Optional[torch.Tensor], dtype=None, name: str = "") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    return t.data_ptr()


_BF = torch.bfloat16


def device_status(reset: bool = True) -> int:
    """The device status word (0 or a DS41_E_* code); synchronises."""
    v = ctypes.c_int32(0)
    _call("ds41_device_status", ctypes.addressof(v), 1 if reset else 0)
    return int(v.value)


def selftest_wait_timeout(polls: int, arrive: bool, result: torch.Tensor) -> None:
    """ds41_selftest_wait_timeout: one bounded mbarrier wait of ``polls`` polls
    that runs out (arrive False) or completes (arrive True); ``result`` is an
    int32 CUDA tensor of at least 2 elements."""
    if result.numel() < 2:
        raise ValueError("result: at least 2 int32 elements")
    _call("ds41_selftest_wait_timeout", int(polls), 1 if arrive else 0,
          _ptr(result, torch.int32, "result"), _stream())


def fp4_quant(x: torch.Tensor, e4m3: bool, want_codes: bool = False):
    """ds41_fp4_quant_e8m0 (block 32) / ds41_fp4_quant_e4m3 (block 16) on the
    rows of a 2-D bf16 tensor.  Returns y, or (y, codes, scales)."""
    rows, cols = x.shape
    block = 16 if e4m3 else 32
    y = torch.empty_like(x)
    codes = scales = None
    if want_codes:
        codes = torch.empty(rows, cols // 2, dtype=torch.uint8, device=x.device)
        scales = torch.empty(rows, cols // block, dtype=torch.uint8, device=x.device)
    fn = "ds41_fp4_quant_e4m3" if e4m3 else "ds41_fp4_quant_e8m0"
    _call(fn, _ptr(x, _BF, "x"), _ptr(y, _BF, "y"), _ptr(codes), _ptr(scales), rows, cols, _stream())
    return (y, codes, scales) if want_codes else y


def yarn_freqs_cis(dim: int, seqlen: int, original_seq_len: int = 65536, base: float = 160000.0,
                   factor: float = 16.0, beta_fast: float = 32.0, beta_slow: float = 1.0,
                   device="cuda") -> torch.Tensor:
    """ds41_yarn_freqs_cis: f32 [seqlen, dim/2, 2] of (cos, sin)."""
    out = torch.empty(seqlen, dim // 2, 2, dtype=torch.float32, device=device)
    _call("ds41_yarn_freqs_cis", _ptr(out, torch.float32, "out"), dim, seqlen, original_seq_len,
          base, factor, beta_fast, beta_slow, _stream())
    return out


def rows_a_len(m: int, win: int, start_pos: int) -> int:
    return int(load().ds41_rows_a_len(m, win, start_pos))


class StepSizes(NamedTuple):
    """Row counts of one call, from ds41_step_sizes."""
    n_a: int    # rows the window indices point into; offset of the picks
    n_c: int    # compress_len: compressed rows after the call
    G: int      # groups (latent rows) the call completes
    ctopk: int  # compressed picks per query
    K: int      # merged index row length, win + ctopk


def step_sizes(wl) -> StepSizes:
    """ds41_step_sizes for the call parameters of ``wl`` (m, start_pos, win,
    ratio, topk)."""
    a = (ctypes.c_int64 * 5)()
    _call("ds41_step_sizes", wl.m, wl.start_pos, wl.win, wl.ratio, wl.topk, ctypes.addressof(a))
    return StepSizes(*[int(v) for v in a])


def window_ring_write(kv: torch.Tensor, ring: torch.Tensor, win_idx: torch.Tensor, start_pos: int,
                      rows_a: Optional[torch.Tensor] = None) -> torch.Tensor:
    """ds41_window_ring_write: updates ``ring`` in place, fills ``win_idx``
    [m, win] and returns the rows the window indices point into (kv, the
    ring, or ``rows_a`` [win + m, hd] for a chunk past position 0)."""
    m, hd = kv.shape
    win = ring.shape[0]
    chunk = start_pos > 0 and m > 1
    if chunk and rows_a is None:
        rows_a = torch.empty(win + m, hd, dtype=kv.dtype, device=kv.device)
    n_a = ctypes.c_int64(0)
    _call("ds41_window_ring_write", _ptr(kv, _BF, "kv"), _ptr(ring, _BF, "ring"),
          _ptr(rows_a if chunk else None), _ptr(win_idx, torch.int32, "win_idx"),
          ctypes.addressof(n_a), m, hd, win, start_pos, _stream())
    if start_pos == 0:
        return kv
    if m == 1:
        return ring
    return rows_a[: n_a.value]


def compress_latent_write(latent: torch.Tensor, freqs_cis: torch.Tensor, cache: torch.Tensor,
                          rd: int, ratio: int, start_pos: int, m: int,
                          codes: Optional[torch.Tensor] = None,
                          scales: Optional[torch.Tensor] = None) -> None:
    """ds41_compress_latent_write: RoPE + bf16 + e4m3 fp4 round trip of the G
    new groups into ``cache`` rows start_pos/ratio ...; optional packed codes
    [rows, hd/2] and scale codes [rows, hd/16]."""
    G, hd = latent.shape
    _call("ds41_compress_latent_write", _ptr(latent, _BF, "latent"),
          _ptr(freqs_cis, torch.float32, "freqs_cis"), freqs_cis.shape[0],
          _ptr(cache, _BF, "cache"), cache.shape[0], _ptr(codes, torch.uint8, "codes"),
          _ptr(scales, torch.uint8, "scales"), G, hd, rd, ratio, start_pos, m, _stream())


def indexer_workspace_bytes(m, Hi, Di, n_c, scores_given) -> int:
    return int(load().ds41_indexer_workspace_bytes(m, Hi, Di, n_c, 1 if scores_given else 0))


def indexer_topk(q_idx: torch.Tensor, k_idx: torch.Tensor, w: torch.Tensor,
                 win_idx: torch.Tensor, ratio: int, start_pos: int, topk: int, offset: int,
                 idx: Optional[torch.Tensor] = None, scores: Optional[torch.Tensor] = None,
                 ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """ds41_indexer_topk: merged index rows [m, win + min(topk, n_c)] int32."""
    m, Hi, Di = q_idx.shape
    n_c = k_idx.shape[0]
    win = win_idx.shape[1]
    ctopk = min(topk, n_c)
    if idx is None:
        idx = torch.empty(m, win + ctopk, dtype=torch.int32, device=q_idx.device)
    need = indexer_workspace_bytes(m, Hi, Di, n_c, scores is not None)
    if need and (ws is None or ws.numel() < need):
        ws = torch.empty(need, dtype=torch.uint8, device=q_idx.device)
    _call("ds41_indexer_topk", _ptr(q_idx, _BF, "q_idx"), _ptr(k_idx, _BF, "k_idx"),
          _ptr(w, torch.float32, "w"), _ptr(win_idx, torch.int32, "win_idx"),
          _ptr(idx, torch.int32, "idx"), _ptr(scores, _BF, "scores"), m, Hi, Di, n_c, win, ratio,
          start_pos, topk, offset, _ptr(ws) if need else None, need, _stream())
    return idx


def indexer_topk_mxf4(q_idx: torch.Tensor, k_codes: torch.Tensor, k_scales: torch.Tensor,
                      w: torch.Tensor, win_idx: torch.Tensor, ratio: int, start_pos: int,
                      topk: int, offset: int, idx: Optional[torch.Tensor] = None,
                      scores: Optional[torch.Tensor] = None,
                      ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """ds41_indexer_topk_mxf4: the indexer top-k on a packed mxf4 key cache
    (k_codes [n_c, Di/2] and k_scales [n_c, Di/32] uint8, as
    fp4_quant(..., want_codes=True) writes them).  Returns idx."""
    m, Hi, Di = q_idx.shape
    n_c = k_codes.shape[0]
    if tuple(k_codes.shape) != (n_c, Di // 2) or tuple(k_scales.shape) != (n_c, Di // 32):
        raise ValueError(f"k_codes/k_scales: expected {(n_c, Di // 2)} / {(n_c, Di // 32)}, got "
                         f"{tuple(k_codes.shape)} / {tuple(k_scales.shape)}")
    win = win_idx.shape[1]
    ctopk = min(topk, n_c)
    if idx is None:
        idx = torch.empty(m, win + ctopk, dtype=torch.int32, device=q_idx.device)
    need = int(load().ds41_indexer_mxf4_workspace_bytes(m, n_c, 1 if scores is not None else 0))
    if need and (ws is None or ws.numel() < need):
        ws = torch.empty(need, dtype=torch.uint8, device=q_idx.device)
    _call("ds41_indexer_topk_mxf4", _ptr(q_idx, _BF, "q_idx"), _ptr(k_codes, torch.uint8, "k_codes"),
          _ptr(k_scales, torch.uint8, "k_scales"), _ptr(w, torch.float32, "w"),
          _ptr(win_idx, torch.int32, "win_idx"), _ptr(idx, torch.int32, "idx"),
          _ptr(scores, _BF, "scores"), m, Hi, Di, n_c, win, ratio, start_pos, topk, offset,
          _ptr(ws) if need else None, need, _stream())
    return idx


def _check_attn(q, rows_a, rows_b, idx, sink, o, lse) -> None:
    """Shapes and device of the attention's tensors, checked before the C call
    (the C ABI sees only pointers, so an undersized o or lse would be written
    past its end on the device)."""
    if q.dim() != 3:
        raise ValueError(f"q: expected [m, nh, hd], got {tuple(q.shape)}")
    m, nh, hd = q.shape
    dev = q.device
    if dev.type != "cuda" or dev.index != torch.cuda.current_device():
        raise ValueError(f"q is on {dev}, the current device is cuda:{torch.cuda.current_device()}: "
                         "the call runs on the current device's stream")
    for name, t in (("rows_a", rows_a), ("rows_b", rows_b), ("idx", idx), ("sink", sink),
                    ("o", o), ("lse", lse)):
        if t is not None and t.device != dev:
            raise ValueError(f"{name} is on {t.device}, q on {dev}")
    if rows_a.dim() != 2 or rows_a.shape[1] != hd:
        raise ValueError(f"rows_a: expected [n_a, {hd}], got {tuple(rows_a.shape)}")
    if rows_b is not None and (rows_b.dim() != 2 or rows_b.shape[1] != hd):
        raise ValueError(f"rows_b: expected [n_c, {hd}], got {tuple(rows_b.shape)}")
    if idx.dim() != 2 or idx.shape[0] != m:
        raise ValueError(f"idx: expected [{m}, K], got {tuple(idx.shape)}")
    if tuple(sink.shape) != (nh,):
        raise ValueError(f"sink: expected [{nh}], got {tuple(sink.shape)}")
    if o is not None and tuple(o.shape) != (m, nh, hd):
        raise ValueError(f"o: expected {(m, nh, hd)}, got {tuple(o.shape)}")
    if lse is not None and tuple(lse.shape) != (m, nh):
        raise ValueError(f"lse: expected {(m, nh)}, got {tuple(lse.shape)}")


def sparse_attn_workspace_bytes(m, nh, hd, K) -> int:
    return int(load().ds41_sparse_attn_workspace_bytes(m, nh, hd, K))


def sparse_attn_sink_fwd(q: torch.Tensor, rows_a: torch.Tensor, rows_b: Optional[torch.Tensor],
                         idx: torch.Tensor, sink: torch.Tensor, scale: float,
                         o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                         ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """ds41_sparse_attn_sink_fwd: o [m, nh, hd] bf16 (lse [m, nh] f32 if given)."""
    _check_attn(q, rows_a, rows_b, idx, sink, o, lse)
    m, nh, hd = q.shape
    K = idx.shape[1]
    n_a = rows_a.shape[0]
    n_c = 0 if rows_b is None else rows_b.shape[0]
    if o is None:
        o = torch.empty_like(q)
    need = sparse_attn_workspace_bytes(m, nh, hd, K)
    if need and (ws is None or ws.numel() < need):
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    _call("ds41_sparse_attn_sink_fwd", _ptr(q, _BF, "q"), _ptr(rows_a, _BF, "rows_a"), n_a,
          _ptr(rows_b, _BF, "rows_b"), n_c, _ptr(idx, torch.int32, "idx"), K,
          _ptr(sink, torch.float32, "sink"), float(scale), _ptr(o, _BF, "o"),
          _ptr(lse, torch.float32, "lse"), m, nh, hd, _ptr(ws) if need else None, need, _stream())
    return o


def sparse_attn_noalloc_capacity() -> int:
    """Bytes of the static scratch array behind sparse_attn_sink_fwd_noalloc."""
    return int(load().ds41_sparse_attn_noalloc_capacity())


def sparse_attn_sink_fwd_noalloc(q: torch.Tensor, rows_a: torch.Tensor,
                                 rows_b: Optional[torch.Tensor], idx: torch.Tensor,
                                 sink: torch.Tensor, scale: float, o: torch.Tensor,
                                 lse: Optional[torch.Tensor] = None) -> torch.Tensor:
    """ds41_sparse_attn_sink_fwd_noalloc: the attention for callers that cannot
    allocate device memory; the library's static scratch holds the split
    partials.  ``o`` (and ``lse``) must be provided by the caller, on the
    current device like every other tensor."""
    if o is None:
        raise ValueError("o: the caller provides the output")
    _check_attn(q, rows_a, rows_b, idx, sink, o, lse)
    m, nh, hd = q.shape
    K = idx.shape[1]
    n_c = 0 if rows_b is None else rows_b.shape[0]
    _call("ds41_sparse_attn_sink_fwd_noalloc", _ptr(q, _BF, "q"), _ptr(rows_a, _BF, "rows_a"),
          rows_a.shape[0], _ptr(rows_b, _BF, "rows_b"), n_c, _ptr(idx, torch.int32, "idx"), K,
          _ptr(sink, torch.float32, "sink"), float(scale), _ptr(o, _BF, "o"),
          _ptr(lse, torch.float32, "lse"), m, nh, hd, _stream())
    return o


def csa_forward_reuse(inp: Dict[str, torch.Tensor], wl, cache: torch.Tensor,
                      cidx: Optional[torch.Tensor],
                      out: Optional[Dict[str, torch.Tensor]] = None) -> Dict[str, torch.Tensor]:
    """ds41_csa_forward_reuse: the step of a layer that reuses the source
    layer's compressed rows ``cache`` and picks ``cidx`` [m, ctopk] (offset
    applied); q, kv, ring, sink come from ``inp``.  Returns win_idx, idx, o."""
    out = {} if out is None else out
    dev = inp["q"].device
    m, win = wl.m, wl.win
    ctopk = 0 if cidx is None else cidx.shape[1]
    if "win_idx" not in out:
        out["win_idx"] = torch.empty(m, win, dtype=torch.int32, device=dev)
    if "idx" not in out:
        out["idx"] = torch.empty(m, win + ctopk, dtype=torch.int32, device=dev)
    if "o" not in out:
        out["o"] = torch.empty_like(inp["q"])
    chunk = wl.start_pos > 0 and m > 1
    if chunk and "rows_a" not in out:
        out["rows_a"] = torch.empty(win + m, wl.hd, dtype=torch.bfloat16, device=dev)
    need = sparse_attn_workspace_bytes(m, wl.nh, wl.hd, win + ctopk)
    ws = out.get("ws_reuse")
    if need and (ws is None or ws.numel() < need):
        ws = out["ws_reuse"] = torch.empty(need, dtype=torch.uint8, device=dev)
    _call("ds41_csa_forward_reuse", _ptr(inp["q"], _BF, "q"), _ptr(inp["kv"], _BF, "kv"),
          _ptr(inp["ring"], _BF, "ring"), _ptr(out.get("rows_a") if chunk else None),
          _ptr(cache, _BF, "cache") if ctopk else None,
          _ptr(cidx, torch.int32, "cidx") if ctopk else None, ctopk,
          _ptr(inp["sink"], torch.float32, "sink"), float(wl.scale),
          _ptr(out["win_idx"], torch.int32, "win_idx"), _ptr(out["idx"], torch.int32, "idx"),
          _ptr(out["o"], _BF, "o"), _ptr(out.get("lse"), torch.float32, "lse"), m, wl.start_pos,
          wl.nh, wl.hd, win, wl.ratio, _ptr(ws) if need else None, need, _stream())
    return out


def attn_out_proj(o: torch.Tensor, freqs_cis: torch.Tensor, wo_a: torch.Tensor,
                  wo_b: torch.Tensor, rd: int, groups: int, start_pos: int,
                  og: Optional[torch.Tensor] = None,
                  out: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """ds41_attn_out_proj: o [m, nh, hd] bf16 is rotated back IN PLACE; returns
    (og [m, groups*o_rank] bf16, out [m, dim] f32)."""
    m, nh, hd = o.shape
    gr = wo_a.shape[0]
    dim = wo_b.shape[0]
    if og is None:
        og = torch.empty(m, gr, dtype=torch.bfloat16, device=o.device)
    if out is None:
        out = torch.empty(m, dim, dtype=torch.float32, device=o.device)
    _call("ds41_attn_out_proj", _ptr(o, _BF, "o"),
          _ptr(freqs_cis, torch.float32, "freqs_cis") if rd else None,
          freqs_cis.shape[0] if rd else start_pos + m, _ptr(wo_a, _BF, "wo_a"),
          _ptr(wo_b, _BF, "wo_b"), _ptr(og, _BF, "og"), _ptr(out, torch.float32, "out"), m,
          start_pos, nh, hd, rd, groups, gr // groups, dim, _stream())
    return og, out


def csa_workspace_bytes(wl) -> int:
    return int(load().ds41_csa_workspace_bytes(wl.m, wl.start_pos, wl.nh, wl.hd, wl.win, wl.ratio,
                                               wl.topk, wl.Hi, wl.Di))


def csa_forward(inp: Dict[str, torch.Tensor], wl, freqs_cis: torch.Tensor,
                out: Optional[Dict[str, torch.Tensor]] = None) -> Dict[str, torch.Tensor]:
    """ds41_csa_forward: the whole step in one call (same inputs and outputs as
    :func:`forward`)."""
    out = {} if out is None else out
    dev = inp["q"].device
    m, win = wl.m, wl.win
    sz = step_sizes(wl)
    if "win_idx" not in out:
        out["win_idx"] = torch.empty(m, win, dtype=torch.int32, device=dev)
    if "idx" not in out:
        out["idx"] = torch.empty(m, sz.K, dtype=torch.int32, device=dev)
    if "o" not in out:
        out["o"] = torch.empty_like(inp["q"])
    chunk = wl.start_pos > 0 and m > 1
    if chunk and "rows_a" not in out:
        out["rows_a"] = torch.empty(win + m, wl.hd, dtype=torch.bfloat16, device=dev)
    need = csa_workspace_bytes(wl)
    ws = out.get("ws_csa")
    if need and (ws is None or ws.numel() < need):
        ws = out["ws_csa"] = torch.empty(need, dtype=torch.uint8, device=dev)
    _call("ds41_csa_forward", _ptr(inp["q"], _BF, "q"), _ptr(inp["kv"], _BF, "kv"),
          _ptr(inp["ring"], _BF, "ring"), _ptr(out.get("rows_a") if chunk else None),
          _ptr(inp["latent"], _BF, "latent") if sz.G > 0 else None,
          _ptr(freqs_cis, torch.float32, "freqs_cis"), freqs_cis.shape[0],
          _ptr(inp["cache"], _BF, "cache"), inp["cache"].shape[0], _ptr(inp["q_idx"], _BF, "q_idx"),
          _ptr(inp["k_idx"], _BF, "k_idx"), _ptr(inp["w"], torch.float32, "w"),
          _ptr(inp["sink"], torch.float32, "sink"), float(wl.scale),
          _ptr(out["win_idx"], torch.int32, "win_idx"), _ptr(out["idx"], torch.int32, "idx"),
          _ptr(out["o"], _BF, "o"), _ptr(out.get("lse"), torch.float32, "lse"), m, wl.start_pos,
          wl.nh, wl.hd, wl.rd, win, wl.ratio, wl.topk, wl.Hi, wl.Di, _ptr(ws) if need else None,
          need, _stream())
    if sz.n_c == 0:
        out["idx"] = out["win_idx"]
    return out


def pack_keys(k_idx: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """The mxf4 form of an indexer key cache [n_c, Di] bf16: (codes [n_c, Di/2],
    scales [n_c, Di/32]) through ds41_fp4_quant_e8m0."""
    _, codes, scales = fp4_quant(k_idx, e4m3=False, want_codes=True)
    return codes, scales


def csa_fp4_workspace_bytes(wl) -> int:
    return int(load().ds41_csa_fp4_workspace_bytes(wl.m, wl.start_pos, wl.nh, wl.hd, wl.win,
                                                   wl.ratio, wl.topk))


def csa_forward_fp4(inp: Dict[str, torch.Tensor], wl, freqs_cis: torch.Tensor,
                    out: Optional[Dict[str, torch.Tensor]] = None) -> Dict[str, torch.Tensor]:
    """ds41_csa_forward_fp4: the whole step on packed fp4 caches.  ``inp`` holds
    the inputs of :func:`csa_forward` with the indexer keys as ``k_codes`` /
    ``k_scales`` (see :func:`pack_keys`) and, optionally, ``cache_codes`` /
    ``cache_scales`` for the packed latent rows."""
    out = {} if out is None else out
    dev = inp["q"].device
    m, win = wl.m, wl.win
    sz = step_sizes(wl)
    if "win_idx" not in out:
        out["win_idx"] = torch.empty(m, win, dtype=torch.int32, device=dev)
    if "idx" not in out:
        out["idx"] = torch.empty(m, sz.K, dtype=torch.int32, device=dev)
    if "o" not in out:
        out["o"] = torch.empty_like(inp["q"])
    chunk = wl.start_pos > 0 and m > 1
    if chunk and "rows_a" not in out:
        out["rows_a"] = torch.empty(win + m, wl.hd, dtype=torch.bfloat16, device=dev)
    need = csa_fp4_workspace_bytes(wl)
    ws = out.get("ws_fp4")
    if need and (ws is None or ws.numel() < need):
        ws = out["ws_fp4"] = torch.empty(need, dtype=torch.uint8, device=dev)
    cc, cs = inp.get("cache_codes"), inp.get("cache_scales")
    _call("ds41_csa_forward_fp4", _ptr(inp["q"], _BF, "q"), _ptr(inp["kv"], _BF, "kv"),
          _ptr(inp["ring"], _BF, "ring"), _ptr(out.get("rows_a") if chunk else None),
          _ptr(inp["latent"], _BF, "latent") if sz.G > 0 else None,
          _ptr(freqs_cis, torch.float32, "freqs_cis"), freqs_cis.shape[0],
          _ptr(inp["cache"], _BF, "cache"), _ptr(cc, torch.uint8, "cache_codes"),
          _ptr(cs, torch.uint8, "cache_scales"), inp["cache"].shape[0],
          _ptr(inp["q_idx"], _BF, "q_idx"), _ptr(inp["k_codes"], torch.uint8, "k_codes"),
          _ptr(inp["k_scales"], torch.uint8, "k_scales"), _ptr(inp["w"], torch.float32, "w"),
          _ptr(inp["sink"], torch.float32, "sink"), float(wl.scale),
          _ptr(out["win_idx"], torch.int32, "win_idx"), _ptr(out["idx"], torch.int32, "idx"),
          _ptr(out["o"], _BF, "o"), _ptr(out.get("lse"), torch.float32, "lse"), m, wl.start_pos,
          wl.nh, wl.hd, wl.rd, win, wl.ratio, wl.topk, wl.Hi, wl.Di, _ptr(ws) if need else None,
          need, _stream())
    if sz.n_c == 0:
        out["idx"] = out["win_idx"]
    return out


STEP_INPUTS = ("q", "kv", "latent", "q_idx", "w")


def step_input_buffers(wl, device="cpu", pinned: bool = False) -> Dict[str, torch.Tensor]:
    """Views q [m, nh, hd], kv [m, hd], latent [G, hd] (bf16), q_idx [m, Hi, Di]
    (bf16) and w [m, Hi] (f32) laid out back to back, in that order, in one
    block of ``device`` memory (page-locked when ``pinned``).  Host and device
    buffers built this way let ds41_csa_forward_host move a step's inputs in
    one copy."""
    shapes = [("q", (wl.m, wl.nh, wl.hd), _BF), ("kv", (wl.m, wl.hd), _BF),
              ("latent", (step_sizes(wl).G, wl.hd), _BF), ("q_idx", (wl.m, wl.Hi, wl.Di), _BF),
              ("w", (wl.m, wl.Hi), torch.float32)]
    sizes = [math.prod(sh) * (2 if dt == _BF else 4) for _, sh, dt in shapes]
    block = torch.empty(sum(sizes), dtype=torch.uint8, device=device)
    if pinned:
        block = block.pin_memory()
    views, off = {}, 0
    for (k, sh, dt), n in zip(shapes, sizes):
        views[k] = block[off:off + n].view(dt).view(sh)
        off += n
    return views


def _packed(bufs: Dict[str, torch.Tensor], wl) -> bool:
    """Whether the step inputs in ``bufs`` lie back to back, in STEP_INPUTS
    order, in one allocation (as step_input_buffers lays them out)."""
    prev = None
    for k in STEP_INPUTS:
        t = bufs[k]
        if t.numel() == 0:  # latent when the call completes no group: 0 bytes
            continue
        if not t.is_contiguous():
            return False
        if prev is not None:
            if (t.untyped_storage().data_ptr() != prev.untyped_storage().data_ptr()
                    or t.data_ptr() != prev.data_ptr() + prev.numel() * prev.element_size()):
                return False
        prev = t
    n = load().ds41_step_inputs_bytes(wl.m, wl.start_pos, wl.nh, wl.hd, wl.ratio, wl.Hi, wl.Di)
    q = bufs["q"]
    return prev.data_ptr() + prev.numel() * prev.element_size() - q.data_ptr() == n


class HostStep:
    """ds41_csa_forward_host prepared once for fixed buffers, as a serving loop
    runs a layer's step again and again: the step inputs q, kv, latent, q_idx,
    w come from the host tensors ``host`` (page-locked for asynchronous copies)
    into the device tensors of the same names in ``inp``, o goes back into the
    host tensor ``h_o`` (allocated page-locked when None).  The arguments are
    checked and marshalled here; each call only enqueues the copies and the
    step on the stream and returns ``h_o``, which holds the result once the
    stream has reached the copy.  When both sides hold the inputs as one block
    (step_input_buffers), the call is ds41_csa_forward_host_packed: one copy
    in instead of five.  With ``graph=True`` (packed blocks only) the call is
    recorded once into a CUDA graph by ds41_host_step_create and every call is
    one ds41_host_step_launch."""

    def __init__(self, host: Dict[str, torch.Tensor], inp: Dict[str, torch.Tensor], wl,
                 freqs_cis: torch.Tensor, out: Optional[Dict[str, torch.Tensor]] = None,
                 h_o: Optional[torch.Tensor] = None, graph: bool = False):
        out = {} if out is None else out
        dev = inp["q"].device
        m, win = wl.m, wl.win
        sz = step_sizes(wl)
        for k in STEP_INPUTS:
            if k == "latent" and sz.G <= 0:
                continue
            t, d = host[k], inp[k]
            if t.is_cuda or t.dtype != d.dtype or not t.is_contiguous() or t.shape != d.shape:
                raise ValueError(f"HostStep: host[{k!r}] must be a contiguous CPU tensor shaped "
                                 f"and typed like the device one")
        if h_o is None:
            h_o = torch.empty(tuple(inp["q"].shape), dtype=_BF).pin_memory()
        if h_o.is_cuda or h_o.dtype != _BF or tuple(h_o.shape) != tuple(inp["q"].shape):
            raise ValueError("HostStep: h_o must be a CPU bf16 tensor shaped like q")
        if "win_idx" not in out:
            out["win_idx"] = torch.empty(m, win, dtype=torch.int32, device=dev)
        if "idx" not in out:
            out["idx"] = torch.empty(m, sz.K, dtype=torch.int32, device=dev)
        if "o" not in out:
            out["o"] = torch.empty_like(inp["q"])
        chunk = wl.start_pos > 0 and m > 1
        if chunk and "rows_a" not in out:
            out["rows_a"] = torch.empty(win + m, wl.hd, dtype=torch.bfloat16, device=dev)
        need = csa_workspace_bytes(wl)
        ws = out.get("ws_csa")
        if need and (ws is None or ws.numel() < need):
            ws = out["ws_csa"] = torch.empty(need, dtype=torch.uint8, device=dev)
        g = sz.G > 0
        self.packed = _packed(host, wl) and _packed(inp, wl) and inp["q"].data_ptr() % 16 == 0
        if self.packed:
            # one block each side: ds41_csa_forward_host_packed, one copy in
            self._args = (
                host["q"].data_ptr(), inp["q"].data_ptr(), h_o.data_ptr(),
                _ptr(inp["ring"], _BF, "ring"), _ptr(out.get("rows_a") if chunk else None),
                _ptr(freqs_cis, torch.float32, "freqs_cis"), freqs_cis.shape[0],
                _ptr(inp["cache"], _BF, "cache"), inp["cache"].shape[0],
                _ptr(inp["k_idx"], _BF, "k_idx"), _ptr(inp["sink"], torch.float32, "sink"),
                float(wl.scale), _ptr(out["win_idx"], torch.int32, "win_idx"),
                _ptr(out["idx"], torch.int32, "idx"), _ptr(out["o"], _BF, "o"),
                _ptr(out.get("lse"), torch.float32, "lse"), m, wl.start_pos, wl.nh, wl.hd, wl.rd,
                win, wl.ratio, wl.topk, wl.Hi, wl.Di, _ptr(ws) if need else None, need)
            self._name = "ds41_csa_forward_host_packed"
        else:
            self._name = "ds41_csa_forward_host"
            self._args = (
                host["q"].data_ptr(), host["kv"].data_ptr(), host["latent"].data_ptr() if g else None,
                host["q_idx"].data_ptr(), host["w"].data_ptr(), h_o.data_ptr(),
                _ptr(inp["q"], _BF, "q"), _ptr(inp["kv"], _BF, "kv"),
                _ptr(inp["ring"], _BF, "ring"), _ptr(out.get("rows_a") if chunk else None),
                _ptr(inp["latent"], _BF, "latent") if g else None,
                _ptr(freqs_cis, torch.float32, "freqs_cis"), freqs_cis.shape[0],
                _ptr(inp["cache"], _BF, "cache"), inp["cache"].shape[0],
                _ptr(inp["q_idx"], _BF, "q_idx"), _ptr(inp["k_idx"], _BF, "k_idx"),
                _ptr(inp["w"], torch.float32, "w"), _ptr(inp["sink"], torch.float32, "sink"),
                float(wl.scale), _ptr(out["win_idx"], torch.int32, "win_idx"),
                _ptr(out["idx"], torch.int32, "idx"), _ptr(out["o"], _BF, "o"),
                _ptr(out.get("lse"), torch.float32, "lse"), m, wl.start_pos, wl.nh, wl.hd, wl.rd, win,
                wl.ratio, wl.topk, wl.Hi, wl.Di, _ptr(ws) if need else None, need)
        self._keep = (host, inp, out, freqs_cis)  # the buffers stay alive with the call
        self._fn = getattr(load(), self._name)
        self.h_o = h_o
        self._handle = None
        if graph:
            if not self.packed:
                raise ValueError("HostStep: graph=True needs the packed input blocks "
                                 "(step_input_buffers on both sides)")
            h = ctypes.c_void_p()
            _call("ds41_host_step_create", ctypes.byref(h), *self._args)
            self._handle = h
            self._name = "ds41_host_step_launch"
            self._fn = load().ds41_host_step_launch
            self._args = (h,)
        if sz.n_c == 0:
            out["idx"] = out["win_idx"]

    def __call__(self, stream: Optional[int] = None) -> torch.Tensor:
        rc = self._fn(*self._args, _stream() if stream is None else stream)
        if rc != 0:
            raise DS41Error(self._name, rc,
                            load().ds41_last_error().decode(errors="replace"))
        return self.h_o

    def close(self) -> None:
        """Frees the recorded graph (graph mode); launches still pending
        complete first."""
        if self._handle is not None:
            load().ds41_host_step_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def csa_forward_host(host: Dict[str, torch.Tensor], inp: Dict[str, torch.Tensor], wl,
                     freqs_cis: torch.Tensor, out: Optional[Dict[str, torch.Tensor]] = None,
                     h_o: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One ds41_csa_forward_host call (see :class:`HostStep`) on the current
    stream; returns the host tensor of o."""
    return HostStep(host, inp, wl, freqs_cis, out, h_o)()


def forward(inp: Dict[str, torch.Tensor], wl, freqs_cis: torch.Tensor,
            out: Optional[Dict[str, torch.Tensor]] = None) -> Dict[str, torch.Tensor]:
    """One layer's compressed sparse attention forward for a workload ``wl``
    (see workloads.Workload) on device tensors ``inp`` (kv, ring, latent,
    cache, q_idx, k_idx, w, q, sink): ring write + window indices, latent
    write, indexer top-k + merge, sparse attention.  ``out`` may hold
    preallocated win_idx / idx / o / rows_a / workspaces, reused across calls.
    Returns the dict of outputs."""
    out = {} if out is None else out
    dev = inp["q"].device
    m, win = wl.m, wl.win
    if "win_idx" not in out:
        out["win_idx"] = torch.empty(m, win, dtype=torch.int32, device=dev)
    rows_a = window_ring_write(inp["kv"], inp["ring"], out["win_idx"], wl.start_pos,
                               rows_a=out.get("rows_a"))
    if wl.start_pos > 0 and m > 1:
        out["rows_a"] = rows_a
    sz = step_sizes(wl)
    if sz.G > 0:
        compress_latent_write(inp["latent"], freqs_cis, inp["cache"], wl.rd, wl.ratio,
                              wl.start_pos, m)
    n_a = rows_a.shape[0]
    if sz.n_c > 0:
        idx = indexer_topk(inp["q_idx"], inp["k_idx"][: sz.n_c], inp["w"], out["win_idx"],
                           wl.ratio, wl.start_pos, wl.topk, n_a, idx=out.get("idx"),
                           ws=out.get("ws_idx"))
        rows_b = inp["cache"][: sz.n_c]
    else:
        idx = out["win_idx"]
        rows_b = None
    out["idx"] = idx
    out["o"] = sparse_attn_sink_fwd(inp["q"], rows_a, rows_b, idx, inp["sink"], wl.scale,
                                    o=out.get("o"), lse=out.get("lse"), ws=out.get("ws_attn"))
    return out
