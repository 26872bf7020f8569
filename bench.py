#!/usr/bin/env python3
"""Benchmark of one layer's compressed sparse attention forward on GB300.

One step = the whole hot path for one batch of synthetic input: window ring
write + window indices, compressed latent write, fp4 indexer scores + top-k +
merge, sparse attention with the sink.  The headline workload is single-token
decode (m=1 at start_pos 8191, 64 heads x 512, window 128, ratio 4 -> 2048
compressed rows, top-k 512, indexer 64 x 128); ``--workload`` picks another.
The same run measures the other four workloads (tiny prefill, prefill, long
decode, chunked prefill) the same way and reports them under ``configs``
(``--headline-only`` skips them).

Timing: W untimed warm-up steps, then exactly K steps between a barrier +
synchronize on both sides, CUDA events on the launching stream, the steps
replayed from CUDA graphs that each hold up to 8 consecutive steps (as a
model's forward replays its layers from one graph).  Steps rotate over
independent layer states, enough of them that the bytes one rotation's steps
touch exceed twice the L2 cache, so every step reads its window ring, latent
cache rows and indexer keys from HBM.  Each workload's entry
adds the roofline of its dominant op (timed again with events around it),
the end-to-end rate through the public API with host buffers, the number of
kernel launches in the timed region (the kernel nodes of the captured step),
the SM clocks seen during the timed region, and the CPU oracle timed per
stage, single-threaded and on all host cores, on a bounded sample.

``--impl reference`` times the CPU oracle itself on the headline workload.
Multi-GPU (torchrun): every rank runs independent replicas of the step on its
own GPU; no data-path collective; value = all ranks' tokens / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from compressed_sparse_attention_window_gb300 import ds41  # noqa: E402
from compressed_sparse_attention_window_gb300.workloads import (OUT_PROJ, WORKLOADS, make_inputs,  # noqa: E402
                                                                 make_out_proj_weights)

METRIC = "query-tokens/s of compressed sparse attn fwd (decode, prefill); % HBM/TC roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (host float)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# algorithmic work of one step (bytes / flops the method itself must move)
# ---------------------------------------------------------------------------
def attn_valid_rows(wl, split=False):
    """Valid gathered rows summed over the tokens: window positions that exist
    plus the visible compressed rows the top-k keeps (with ``split``, the two
    counts apart)."""
    win_rows = comp_rows = 0
    for t in range(wl.m):
        p = wl.start_pos + t
        vis = min(wl.n_c, (p + 1) // wl.ratio)
        win_rows += min(p + 1, wl.win)
        comp_rows += min(wl.topk, vis)
    return (win_rows, comp_rows) if split else win_rows + comp_rows


def algorithmic(wl):
    """Per-op algorithmic bytes and flops of one step: each input and output
    once, the valid gathered rows, and the causally visible indexer pairs."""
    bf, m = 2, wl.m
    rows = attn_valid_rows(wl)
    pairs = sum(min(wl.n_c, (wl.start_pos + t + 1) // wl.ratio) for t in range(wl.m))
    K = wl.K
    ops = {
        "window_ring_write": {"bytes": 2 * min(m, wl.win) * wl.hd * bf + m * wl.win * 4},
        "compress_latent_write": {"bytes": 2 * wl.G * wl.hd * bf + wl.G * (wl.rd // 2) * 8},
        "indexer_topk": {
            "bytes": (m * wl.Hi * wl.Di * bf + wl.n_c * wl.Di * bf + m * wl.Hi * 4
                      + m * wl.win * 4 + m * K * 4),
            "flops": 2 * wl.Hi * wl.Di * pairs},
        # the same on the mxf4 key cache: Di/2 code bytes + Di/32 scale bytes per row
        "indexer_topk_mxf4": {
            "bytes": (m * wl.Hi * wl.Di * bf + wl.n_c * (wl.Di // 2 + wl.Di // 32) + m * wl.Hi * 4
                      + m * wl.win * 4 + m * K * 4),
            "flops": 2 * wl.Hi * wl.Di * pairs},
        "sparse_attn_sink_fwd": {
            "bytes": rows * wl.hd * bf + 2 * m * wl.nh * wl.hd * bf + m * K * 4 + wl.nh * 4,
            "flops": 4 * wl.nh * wl.hd * rows},
    }
    # the few-token attention on the packed latent rows: hd/2 code bytes +
    # hd/16 scale bytes per gathered compressed row
    win_rows, comp_rows = attn_valid_rows(wl, split=True)
    ops["sparse_attn_sink_fwd_fp4"] = {
        "bytes": (win_rows * wl.hd * bf + comp_rows * (wl.hd // 2 + wl.hd // 16)
                  + 2 * m * wl.nh * wl.hd * bf + m * K * 4 + wl.nh * 4),
        "flops": 4 * wl.nh * wl.hd * rows}
    return ops


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


CSRC = os.path.join(ROOT, "compressed_sparse_attention_window_gb300", "csrc")
# The translation units each op's kernels (and their tensor maps) come from; a
# recorded traffic figure stands while these files and the headers they
# include are unchanged.
OP_SOURCES = {
    "window_ring_write": ["ds41_window.cu"],
    "compress_latent_write": ["ds41_window.cu"],
    "indexer_topk": ["ds41_indexer.cu", "ds41_indexer_tc.cu", "ds41_quant.cu", "ds41_tc_host.cu"],
    "indexer_topk_mxf4": ["ds41_indexer.cu", "ds41_indexer_mxf4.cu", "ds41_tc_host.cu"],
    "sparse_attn_sink_fwd": ["ds41_attn.cu", "ds41_attn_tc.cu", "ds41_tc_host.cu"],
}
_INCLUDE_RE = re.compile(r'^\s*#\s*include\s+"([^"]+)"', re.M)


def _source_closure(names):
    """The files ``names`` and every header of the CUDA sources they include,
    transitively (the public C header, declarations only, is left out)."""
    seen, todo = {}, list(names)
    while todo:
        f = todo.pop()
        if f in seen:
            continue
        path = os.path.join(CSRC, f)
        if not os.path.exists(path):
            continue
        with open(path, "rb") as fh:
            seen[f] = fh.read()
        todo.extend(_INCLUDE_RE.findall(seen[f].decode(errors="replace")))
    return seen


def csrc_digest(op=None) -> str:
    """sha256 (first 16 hex digits) over CUDA sources by sorted name: those of
    ``op``'s kernels with the headers they include, or every source when op is
    None."""
    h = hashlib.sha256()
    if op is None:
        names = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh")))
        files = {f: open(os.path.join(CSRC, f), "rb").read() for f in names}
    else:
        files = _source_closure(OP_SOURCES[op])
    for f in sorted(files):
        h.update(f.encode())
        h.update(files[f])
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, op: str):
    """DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum) per call of
    `op` on `workload`, from profiles/dram_traffic.txt, when they were taken on
    the current sources of that op's kernels (the line's digest); None
    otherwise."""
    try:
        with open(TRAFFIC_FILE) as fh:
            lines = fh.read().splitlines()
    except OSError:
        return None
    for line in lines:
        f = line.split()
        if len(f) < 6 or f[0].startswith("#") or f[0] != workload or f[1] != op:
            continue
        if op in OP_SOURCES and f[-1] == csrc_digest(op):
            return float(f[2])
    return None


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(
            p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampler
# ---------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"ds41_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait(timeout=5)
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.remove(self.path)
        # median over the samples taken under load (the top half by clock)
        load = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def build_slots(wl, n_slots, device, seed0=1000):
    """Independent layer states (inputs + outputs + workspaces) for rotation."""
    sz = ds41.step_sizes(wl)
    slots = []
    for s in range(n_slots):
        inp = make_inputs(wl, device=device, seed=seed0 + s)
        out = {"win_idx": torch.empty(wl.m, wl.win, dtype=torch.int32, device=device)}
        if wl.start_pos > 0 and wl.m > 1:
            out["rows_a"] = torch.empty(wl.win + wl.m, wl.hd, dtype=torch.bfloat16, device=device)
        if sz.n_c > 0:
            out["idx"] = torch.empty(wl.m, sz.K, dtype=torch.int32, device=device)
            nb = ds41.indexer_workspace_bytes(wl.m, wl.Hi, wl.Di, sz.n_c, False)
            if nb:
                out["ws_idx"] = torch.empty(nb, dtype=torch.uint8, device=device)
        out["o"] = torch.empty(wl.m, wl.nh, wl.hd, dtype=torch.bfloat16, device=device)
        nb = ds41.sparse_attn_workspace_bytes(wl.m, wl.nh, wl.hd, sz.K)
        if nb:
            out["ws_attn"] = torch.empty(nb, dtype=torch.uint8, device=device)
        nb = ds41.csa_workspace_bytes(wl)
        if nb:
            out["ws_csa"] = torch.empty(nb, dtype=torch.uint8, device=device)
        slots.append((inp, out))
    return slots


def slot_bytes(slot) -> int:
    inp, out = slot
    return sum(v.numel() * v.element_size() for d in (inp, out) for v in d.values())


def launches_per_step(wl) -> int:
    """Kernels one ds41_csa_forward launches for this workload, mirroring the
    library's plan (fused few-token step, or the four calls).  Used only when
    the captured graph cannot be inspected (see kernel_nodes)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sz = ds41.step_sizes(wl)
    hpad = (wl.Hi + 7) // 8 * 8
    tt = max(1, 128 // hpad)
    groups = (wl.m + tt - 1) // tt
    dec_groups = wl.m * ((wl.nh + 15) // 16)
    few_attn = dec_groups * 4 <= sms
    if sz.n_c > 0 and groups <= 4 and few_attn:
        cl = 16
        while cl > 1 and (dec_groups * cl > 2 * sms or (sz.K + cl - 1) // cl < 8):
            cl //= 2
        kseg = ((sz.n_c + cl - 1) // cl + 7) // 8 * 8
        if cl >= 4 and (sz.K + cl - 1) // cl <= 2048 and kseg <= 4096:
            return 2
        return 3
    n = 1
    if sz.G > 0:
        n += 1
    if sz.n_c > 0:
        n += 2
        if groups > 4:
            n += 1
            if wl.Hi == 64 and wl.Di == 128 and (wl.m + 3) // 4 >= sms:
                n += 1
    if few_attn:
        return n + 1
    if wl.hd == 512 and wl.nh % 64 == 0 and sz.K <= 1024 and wl.m * (wl.nh // 64) >= sms:
        return n + 1
    heads_groups = (wl.nh + 63) // 64
    chunks = (sz.K + 31) // 32
    ctas = wl.m * heads_groups
    splits = 1
    if ctas < sms:
        splits = min(chunks, (sms + ctas - 1) // ctas)
        cps = (chunks + splits - 1) // splits
        splits = (chunks + cps - 1) // cps
    return n + 1 + (1 if splits > 1 else 0)


def kernel_nodes(wl, slot, fc, stream):
    """Kernel launches of one step, counted as the kernel nodes of the step
    captured in a CUDA graph (driver API cuGraphGetNodes / cuGraphNodeGetType
    on the captured graph).  Returns (count, how)."""
    import ctypes
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)
        with torch.cuda.graph(g, stream=stream):
            ds41.csa_forward(slot[0], wl, fc, slot[1])
        raw = g.raw_cuda_graph()
        cu = ctypes.CDLL("libcuda.so.1")
        n = ctypes.c_size_t(0)
        if cu.cuGraphGetNodes(ctypes.c_void_p(raw), None, ctypes.byref(n)) != 0:
            raise RuntimeError("cuGraphGetNodes")
        nodes = (ctypes.c_void_p * max(1, n.value))()
        if cu.cuGraphGetNodes(ctypes.c_void_p(raw), nodes, ctypes.byref(n)) != 0:
            raise RuntimeError("cuGraphGetNodes")
        kinds = []
        for i in range(n.value):
            t = ctypes.c_int(-1)
            if cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) != 0:
                raise RuntimeError("cuGraphNodeGetType")
            kinds.append(t.value)
        del g
        torch.cuda.synchronize()
        return sum(1 for k in kinds if k == 0), "kernel nodes of the captured step (CU_GRAPH_NODE_TYPE_KERNEL)"
    except Exception as e:  # older torch without keep_graph / raw_cuda_graph
        return launches_per_step(wl), f"the library's launch plan mirrored on the host ({type(e).__name__})"


OPS = ["window_ring_write", "compress_latent_write", "indexer_topk", "sparse_attn_sink_fwd"]


def call_op(name, wl, inp, out, fc):
    """One call of one entry point on a layer state (outputs preallocated)."""
    sz = ds41.step_sizes(wl)
    if name == "window_ring_write":
        ds41.window_ring_write(inp["kv"], inp["ring"], out["win_idx"], wl.start_pos,
                               rows_a=out.get("rows_a"))
    elif name == "compress_latent_write":
        ds41.compress_latent_write(inp["latent"], fc, inp["cache"], wl.rd, wl.ratio,
                                   wl.start_pos, wl.m)
    elif name == "indexer_topk":
        ds41.indexer_topk(inp["q_idx"], inp["k_idx"][: sz.n_c], inp["w"], out["win_idx"],
                          wl.ratio, wl.start_pos, wl.topk, sz.n_a, idx=out["idx"],
                          ws=out.get("ws_idx"))
    else:
        if wl.start_pos == 0:
            rows_a = inp["kv"]
        elif wl.m == 1:
            rows_a = inp["ring"]
        else:
            rows_a = out["rows_a"]
        rows_b = inp["cache"][: sz.n_c] if sz.n_c > 0 else None
        idx = out["idx"] if sz.n_c > 0 else out["win_idx"]
        ds41.sparse_attn_sink_fwd(inp["q"], rows_a, rows_b, idx, inp["sink"], wl.scale,
                                  o=out["o"], ws=out.get("ws_attn"))


def time_ops(wl, slots, fc, stream, reps=5):
    """Milliseconds per call of each entry point, from CUDA graphs of one call
    per layer state replayed ``reps`` times (no host launch gaps)."""
    sz = ds41.step_sizes(wl)
    res = {}
    for name in OPS:
        if name == "compress_latent_write" and sz.G == 0:
            continue
        if name == "indexer_topk" and sz.n_c == 0:
            continue
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for inp, out in slots:
                call_op(name, wl, inp, out, fc)
        with torch.cuda.stream(stream):
            g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        res[name] = e0.elapsed_time(e1) / (reps * len(slots))
        del g
    torch.cuda.synchronize()
    return res


def time_out_proj(wl, slots, fc, stream, hbm, bf16, reps=5):
    """The output side of the layer (inverse RoPE, grouped wo_a, wo_b; not part
    of the step) on the step's attention output: milliseconds per call from a
    CUDA graph of back-to-back calls, and its roofline.  The weights (176 MiB
    at the sizes below) exceed L2, so every call streams them from HBM."""
    P = OUT_PROJ
    dev = slots[0][1]["o"].device
    w = make_out_proj_weights(wl.nh, wl.hd, P["groups"], P["o_rank"], P["dim"], device="cpu")
    wa, wb = w["wo_a"].to(dev), w["wo_b"].to(dev)
    o = slots[0][1]["o"]
    og = torch.empty(wl.m, wa.shape[0], dtype=torch.bfloat16, device=dev)
    out = torch.empty(wl.m, P["dim"], dtype=torch.float32, device=dev)

    def call():
        ds41.attn_out_proj(o, fc, wa, wb, wl.rd, P["groups"], wl.start_pos, og=og, out=out)

    with torch.cuda.stream(stream):
        call()  # warm-up outside the capture (library handle, kernel attributes)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(4):
                call()
        g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / (reps * 4)
    del g
    gr, gw = wa.shape
    flops = 2.0 * wl.m * (wl.nh * wl.hd * P["o_rank"] + gr * P["dim"])
    nbytes = 2.0 * (wa.numel() + wb.numel()) + wl.m * (2.0 * gr * 2 + 4.0 * P["dim"]
                                                        + 2.0 * wl.nh * wl.hd)
    if wl.m >= 64:
        ach = flops / (ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": bf16, "unit": "TFLOP/s",
                "frac": ach / bf16}
    else:
        ach = nbytes / (ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm}
    roof.update({"ms_per_call": ms, "flops": flops, "algorithmic_bytes": nbytes,
                 "config": f"groups {P['groups']}, o_rank {P['o_rank']}, dim {P['dim']}, "
                           "synthetic bf16 weights; inverse RoPE kernel, then a warp per weight row (m <= 16) or tcgen05 tiles"})
    return roof


def time_reuse(wl, slots, stream, reps=5):
    """The step of a layer that reuses the source layer's compressed rows and
    picks (ring write, index merge, attention; not part of the measured step):
    milliseconds per call from a CUDA graph of one call per layer state, each
    on that state's cache and the picks its own step left in idx."""
    ctopk = ds41.step_sizes(wl).ctopk
    cidx = [out["idx"][:, wl.win:].contiguous() if ctopk else None for _, out in slots]
    outs = [{} for _ in slots]
    with torch.cuda.stream(stream):
        for (inp, _), c, o in zip(slots, cidx, outs):
            ds41.csa_forward_reuse(inp, wl, inp["cache"], c, o)  # allocates outside the capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for (inp, _), c, o in zip(slots, cidx, outs):
                ds41.csa_forward_reuse(inp, wl, inp["cache"], c, o)
        g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / (reps * len(slots))
    del g
    return {"ms_per_step": ms, "query_tokens_per_s": wl.m / (ms / 1e3),
            "steps": "ring write, index merge (when the layer has compressed picks), attention"}


def dominant_roofline(wl, op_ms, args):
    """The roofline of the op that takes longest per call: algorithmic flops on
    the bf16 tensor peak for many-token attention, algorithmic bytes on HBM
    otherwise."""
    alg = algorithmic(wl)
    hbm, bf16, bf16_sus, peak_src = load_peaks()
    dom = max(op_ms, key=lambda k: op_ms[k])
    d_ms = op_ms[dom]
    if wl.m >= 256 and dom == "sparse_attn_sink_fwd":
        achieved = alg[dom]["flops"] / (d_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s",
                "frac": achieved / bf16}
    else:
        achieved = alg[dom]["bytes"] / (d_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm}
    traffic = args.traffic if (args.traffic is not None and wl.name == args.workload) \
        else recorded_traffic(wl.name, dom)
    roof.update({"kernel": dom, "ms_per_launch": d_ms, "algorithmic_bytes": alg[dom]["bytes"],
                 "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured"
                 else "fallback",
                 "traffic": traffic})
    if "flops" in alg[dom]:
        roof["algorithmic_flops"] = alg[dom]["flops"]
    return roof


def step_bytes(wl, fp4=False, packed_attn=False) -> int:
    """Algorithmic bytes one step touches (the sum of its ops' rows of
    ``algorithmic``): what has to come from HBM when the step runs L2-cold.
    ``fp4``: the indexer reads the mxf4 keys; ``packed_attn``: the attention
    gathers packed latent rows."""
    alg = algorithmic(wl)
    ops = [k for k in OPS if k in alg]
    if fp4:
        ops = [k for k in ops if k != "indexer_topk"] + ["indexer_topk_mxf4"]
    if packed_attn:
        ops = [k for k in ops if k != "sparse_attn_sink_fwd"] + ["sparse_attn_sink_fwd_fp4"]
    return sum(alg[k]["bytes"] for k in ops if k in alg)


def steps_per_graph(K: int, n_slots: int) -> int:
    """Consecutive steps (layer states) captured in one CUDA graph: the largest
    divisor of K up to 8 (and up to the number of layer states), so that
    exactly K steps are timed.  A model's forward likewise replays its layers
    from one graph; the host launch of a graph is paid once per graph."""
    for d in range(min(8, n_slots, K), 0, -1):
        if K % d == 0:
            return d
    return 1


def time_graph_steps(graphs, spg, K, W, world, dev, stream):
    """Warm-up replays covering at least W steps, then K timed steps (K / spg
    replays of graphs of spg steps each, in rotation) between a barrier +
    synchronize on both sides, events on the launching stream, clocks sampled
    meanwhile.  Returns (max-over-ranks ms, clocks)."""
    n = len(graphs)
    wr = (W + spg - 1) // spg
    with torch.cuda.stream(stream):
        for i in range(wr):
            graphs[i % n].replay()
    stream.synchronize()
    clocks = Clocks(dev.index if dev.index is not None else 0)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(K // spg):
            graphs[(wr + i) % n].replay()
        e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    ck = clocks.stop()
    return max_over_ranks(e0.elapsed_time(e1), world), ck


def capture_steps(step, slots, stream, spg=1):
    """CUDA graphs of ``step(inp, out)``, each holding spg consecutive layer
    states' steps (wrapping around), covering every layer state."""
    graphs = []
    n = len(slots)
    for j in range((n + spg - 1) // spg):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(spg):
                inp, out = slots[(j * spg + r) % n]
                step(inp, out)
        graphs.append(g)
    torch.cuda.synchronize()
    return graphs


def fp4_supported(wl) -> bool:
    return wl.Hi == 64 and wl.Di == 128


def add_fp4_caches(wl, slots):
    """The packed caches of every layer state: the indexer keys as mxf4
    (codes + e8m0 scales, from the bf16 keys through ds41_fp4_quant_e8m0), and
    the latent rows as e2m1 codes + e4m3 scales: the drawn rows go through
    ds41_fp4_quant_e4m3 (the latent write's round trip), whose values replace
    the bf16 rows, so both forms of the cache hold the same values."""
    sz = ds41.step_sizes(wl)
    for inp, _ in slots:
        inp["k_codes"], inp["k_scales"] = ds41.pack_keys(inp["k_idx"][: max(1, sz.n_c)].contiguous())
        cq, inp["cache_codes"], inp["cache_scales"] = ds41.fp4_quant(inp["cache"], e4m3=True,
                                                                     want_codes=True)
        inp["cache"].copy_(cq)
    torch.cuda.synchronize()


def time_fp4_variant(wl, slots, fc, K, W, world, dev, stream, args, latent_packed=True):
    """The step on packed fp4 caches (ds41_csa_forward_fp4; the step's own
    results bit for bit, see the tests): per-step time from graph replays over
    the same rotating layer states, the mxf4 indexer op alone, and the
    roofline of the variant's dominant op.  With ``latent_packed`` the latent
    rows are written and (few tokens) gathered packed too; without, only the
    indexer keys are packed."""
    add_fp4_caches(wl, slots)
    inps = []
    for inp, _ in slots:
        d = dict(inp)
        if not latent_packed:
            d.pop("cache_codes", None)
            d.pop("cache_scales", None)
        inps.append(d)
    outs = [dict(out) for _, out in slots]
    with torch.cuda.stream(stream):
        for inp, o in zip(inps, outs):
            ds41.csa_forward_fp4(inp, wl, fc, o)
    stream.synchronize()
    spg = steps_per_graph(K, len(slots))
    graphs = capture_steps(lambda inp, out: ds41.csa_forward_fp4(inp, wl, fc, out),
                           list(zip(inps, outs)), stream, spg)
    t_ms, ck = time_graph_steps(graphs, spg, K, W, world, dev, stream)
    del graphs
    sz = ds41.step_sizes(wl)
    op_ms = {}
    if sz.n_c > 0:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for (inp, out), o in zip(slots, outs):
                ds41.indexer_topk_mxf4(inp["q_idx"], inp["k_codes"], inp["k_scales"], inp["w"],
                                       out["win_idx"], wl.ratio, wl.start_pos, wl.topk, sz.n_a,
                                       idx=out["idx"], ws=o.get("ws_fp4"))
        with torch.cuda.stream(stream):
            g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(5):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        op_ms["indexer_topk_mxf4"] = e0.elapsed_time(e1) / (5 * len(slots))
        del g
    packed_attn = latent_packed and wl.m <= 8 and wl.hd == 512
    res = {"ms_per_step": t_ms / K, "value": wl.m * K * world / (t_ms / 1e3),
           "unit": "query-tokens/s", "steps": K, "clocks": ck, "per_op_ms": op_ms,
           "algorithmic_bytes_per_step": step_bytes(wl, fp4=True, packed_attn=packed_attn),
           "what": ("ds41_csa_forward_fp4: indexer keys as mxf4 (68 B/row), scores by "
                    "block-scaled tcgen05 MMAs; " +
                    ("latent rows written and (few tokens) gathered as e2m1 codes + e4m3 "
                     "block-16 scales (288 B/row), expanded in shared memory" if latent_packed
                     else "latent cache in bf16"))}
    if op_ms:
        alg = algorithmic(wl)["indexer_topk_mxf4"]
        hbm = load_peaks()[0]
        ms = op_ms["indexer_topk_mxf4"]
        ach = alg["bytes"] / (ms / 1e3) / 1e9
        res["roofline"] = {"kernel": "indexer_topk_mxf4", "bound": "hbm", "achieved": ach,
                           "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "ms_per_launch": ms,
                           "algorithmic_bytes": alg["bytes"], "algorithmic_flops": alg["flops"],
                           "traffic": recorded_traffic(wl.name, "indexer_topk_mxf4")}
    return res


def measure_workload(wl, K, W, world, dev, stream, args, extras=True):
    """The measurement of one workload: K timed CUDA-graph steps (max over
    ranks), the dominant op's roofline, per-op times, e2e through the host
    buffer API, the kernel launches in the timed region, clocks, the step on
    packed fp4 caches (64 x 128 indexers), and (with ``extras``) the next
    rows of the layer."""
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    fc = ds41.yarn_freqs_cis(wl.rd, wl.max_pos, device=dev)

    # Rotate over enough layer states that the bytes the steps of one
    # rotation touch exceed twice L2 (at most 256 states, 24 GB).
    one = build_slots(wl, 1, dev)
    per = slot_bytes(one[0])
    touched = step_bytes(wl, fp4=fp4_supported(wl),
                         packed_attn=fp4_supported(wl) and wl.m <= 8 and wl.hd == 512)
    n_slots = max(1, min(256, math.ceil(2.2 * l2 / touched), int(24e9 // per)))
    slots = one + (build_slots(wl, n_slots - 1, dev, seed0=2000) if n_slots > 1 else [])
    torch.cuda.synchronize()

    # eager warm-up of every slot (sets kernel attributes, status word)
    with torch.cuda.stream(stream):
        for inp, out in slots:
            ds41.csa_forward(inp, wl, fc, out)
    stream.synchronize()
    launches, launches_how = kernel_nodes(wl, slots[0], fc, stream)

    spg = steps_per_graph(K, n_slots)
    graphs = capture_steps(lambda inp, out: ds41.csa_forward(inp, wl, fc, out), slots, stream,
                           spg)
    t_max_ms, ck = time_graph_steps(graphs, spg, K, W, world, dev, stream)
    del graphs

    op_ms = time_ops(wl, slots, fc, stream)
    roof = dominant_roofline(wl, op_ms, args)
    # e2e: at most 20 steps for the big prefills (hundreds of MB of copies each)
    k_e2e = K if wl.m < 256 else min(K, 20)
    e2e = run_e2e(wl, slots, fc, stream, k_e2e, W, n_slots, world)
    res = {"value": wl.m * K * world / (t_max_ms / 1e3), "unit": "query-tokens/s",
           "steps": K, "warmup": W, "ms_per_step": t_max_ms / K,
           "workload": workload_desc(wl),
           "l2": f"inputs larger than L2: {n_slots} rotating layer states of {per / 2**20:.2f} MiB "
                 f"({n_slots * per / 2**20:.0f} MiB); one rotation's steps touch "
                 f"{n_slots * touched / 2**20:.0f} MiB (L2 {l2 / 2**20:.0f} MiB)",
           "timing": f"CUDA graphs of {spg} consecutive steps (layer states), "
                     f"{K // spg} replays, events on the launching stream",
           "roofline": roof, "per_op_ms": op_ms, "e2e": e2e,
           "gpu_launches": launches * K, "gpu_launches_per_step": launches,
           "gpu_launches_how": launches_how, "clocks": ck}
    if extras:
        hbm, bf16, _, _ = load_peaks()
        out_proj = time_out_proj(wl, slots, fc, stream, hbm, bf16) if wl.hd == 512 else None
        reuse = time_reuse(wl, slots, stream)
        res["next_rows"] = dict({"attn_out_proj": out_proj} if out_proj else {},
                                csa_forward_reuse=reuse)
    if fp4_supported(wl):
        res["variants"] = {
            "fp4_keys": time_fp4_variant(wl, slots, fc, K, W, world, dev, stream, args,
                                         latent_packed=False),
            "fp4_caches": time_fp4_variant(wl, slots, fc, K, W, world, dev, stream, args)}
    del slots, one
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_ours(args, world, rank, local):
    wl = WORKLOADS[args.workload]
    dev = torch.device("cuda", local)
    ds41.load()
    stream = torch.cuda.Stream(device=dev)
    K, W = args.steps, args.warmup
    head = measure_workload(wl, K, W, world, dev, stream, args)
    configs = {}
    if not args.headline_only:
        for name in CONFIG_ORDER:
            if name == wl.name:
                continue
            configs[name] = measure_workload(WORKLOADS[name], K, W, world, dev, stream, args)
    res = {
        "metric": METRIC, "value": head["value"], "unit": "query-tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": head["workload"],
                   "global_batch": wl.m * world, "parallelism": f"replicas{world}",
                   "l2": head["l2"],
                   "timing": head["timing"]},
        "roofline": head["roofline"],
        "per_op_ms": head["per_op_ms"],
        "next_rows": head["next_rows"],
        "variants": head.get("variants", {}),
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "gpu_launches_how": head["gpu_launches_how"],
        "clocks": head["clocks"],
    }
    if configs:
        res["configs"] = configs
    return res, wl


CONFIG_ORDER = ["tiny_prefill", "decode", "prefill", "long_decode", "chunked_prefill"]


def run_only(args, local):
    """Profiling mode: W + K eager calls of the whole step (``--only step``) or
    of one op over rotating layer states; prints the average time per call."""
    wl = WORKLOADS[args.workload]
    dev = torch.device("cuda", local)
    ds41.load()
    fc = ds41.yarn_freqs_cis(wl.rd, wl.max_pos, device=dev)
    slots = build_slots(wl, args.slots, dev)
    sz = ds41.step_sizes(wl)
    for inp, out in slots:
        ds41.forward(inp, wl, fc, out)  # fills win_idx / idx / o for the later ops
    P = OUT_PROJ
    wts = {}
    if args.only == "attn_out_proj":
        w = make_out_proj_weights(wl.nh, wl.hd, P["groups"], P["o_rank"], P["dim"])
        wts = {k: v.to(dev) for k, v in w.items()}
        for inp, out in slots:
            out["og"] = torch.empty(wl.m, wts["wo_a"].shape[0], dtype=torch.bfloat16, device=dev)
            out["proj"] = torch.empty(wl.m, P["dim"], dtype=torch.float32, device=dev)
    elif args.only == "csa_forward_reuse":
        for inp, out in slots:
            out["cidx"] = out["idx"][:, wl.win:].contiguous() if sz.ctopk else None
            out["reuse"] = {}
    elif args.only in ("indexer_topk_mxf4", "step_fp4"):
        add_fp4_caches(wl, slots)
    torch.cuda.synchronize()

    def op(i):
        inp, out = slots[i % len(slots)]
        if args.only == "step":
            ds41.csa_forward(inp, wl, fc, out)
        elif args.only in OPS:
            call_op(args.only, wl, inp, out, fc)
        elif args.only == "indexer_topk_mxf4":
            ds41.indexer_topk_mxf4(inp["q_idx"], inp["k_codes"], inp["k_scales"], inp["w"],
                                   out["win_idx"], wl.ratio, wl.start_pos, wl.topk, sz.n_a,
                                   idx=out["idx"])
        elif args.only == "step_fp4":
            ds41.csa_forward_fp4(inp, wl, fc, out)
        elif args.only == "attn_out_proj":
            ds41.attn_out_proj(out["o"], fc, wts["wo_a"], wts["wo_b"], wl.rd, P["groups"],
                               wl.start_pos, og=out["og"], out=out["proj"])
        elif args.only == "csa_forward_reuse":
            ds41.csa_forward_reuse(inp, wl, inp["cache"], out["cidx"], out["reuse"])
        else:
            raise SystemExit(f"unknown op {args.only}")

    for i in range(args.warmup):
        op(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        op(args.warmup + i)
    e1.record()
    torch.cuda.synchronize()
    print(json.dumps({"only": args.only, "workload": wl.name, "calls": args.steps,
                      "ms_per_call": e0.elapsed_time(e1) / args.steps, "slots": len(slots)}))


def run_e2e(wl, slots, fc, stream, K, W, n_slots, world=1):
    """The same metric through the C-ABI calls for host-resident step data:
    per layer state, ds41_host_step_create records once what
    ds41_csa_forward_host_packed enqueues (ds41.HostStep, graph=True), and
    every step is one ds41_host_step_launch: it copies that step's inputs from
    page-locked host memory into the device buffers (laid out back to back on
    both sides, so in one copy), runs the step and copies o back to host
    memory, on one stream; the layer states stay resident."""
    names = ds41.STEP_INPUTS
    o_host = torch.empty(slots[0][1]["o"].shape, dtype=torch.bfloat16).pin_memory()
    steps = []
    for s in range(n_slots):
        inp, out = slots[s]
        dev_in = ds41.step_input_buffers(wl, inp["q"].device)
        host_in = ds41.step_input_buffers(wl, "cpu", pinned=True)
        for k in names:
            host_in[k].copy_(inp[k].cpu())
        e_inp = dict(inp)
        e_inp.update(dev_in)
        steps.append(ds41.HostStep(host_in, e_inp, wl, fc, out, h_o=o_host, graph=True))
    h2d = sum(t.numel() * t.element_size() for t in steps[0]._keep[0].values())
    d2h = o_host.numel() * o_host.element_size()
    sid = stream.cuda_stream

    with torch.cuda.stream(stream):
        for i in range(W):
            steps[i % n_slots](sid)
    stream.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(K):
            steps[(W + i) % n_slots](sid)
        e1.record(stream)
    stream.synchronize()
    wall = time.perf_counter() - t0
    ms = max_over_ranks(max(e0.elapsed_time(e1), wall * 1e3), world)
    return {"value": wl.m * K * world / (ms / 1e3), "unit": "query-tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "how": "ds41_host_step_launch per step (the packed host step recorded once "
                   "per layer state as a CUDA graph): one pinned H2D of q/kv/latent/q_idx/w, "
                   "the step, D2H of o, one stream"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------
STAGES = ["window_ring_write", "compress_latent_write", "indexer_topk", "sparse_attn_sink_fwd"]


def _oracle_inputs(wl):
    from compressed_sparse_attention_window_gb300.workloads import bf16_bits
    inp = make_inputs(wl)
    b = {k: bf16_bits(inp[k]) for k in ("q", "kv", "latent", "q_idx", "ring", "cache", "k_idx")}
    return b, inp["sink"].numpy(), inp["w"].numpy()


def oracle_stage_rates(wl, budget_s, threads, toks_per=8, min_forwards=1, seed=0):
    """The oracle's forward (``oracle.forward``) timed stage by stage on a
    bounded sample of the workload, with ``threads`` OpenMP threads: repeated
    forwards, each running the ring and latent writes whole and the indexer +
    top-k and the attention for ``toks_per`` sampled query tokens, until
    ``budget_s`` seconds (at least ``min_forwards`` forwards).  Per stage,
    query-tokens/s = tokens the stage processed / its seconds (m per forward
    for the two writes, the sampled tokens for the other two); the whole step
    rate adds the stages' seconds per token."""
    import numpy as np

    import oracle
    b, sink, w = _oracle_inputs(wl)
    fc = oracle.yarn_freqs_cis(wl.rd, wl.max_pos)
    prev = oracle.num_threads()
    oracle.set_num_threads(threads)
    used = oracle.num_threads()
    rng = np.random.default_rng(seed)
    tp = min(wl.m, toks_per)
    timings, n, sampled = {}, 0, 0
    t0 = time.perf_counter()
    try:
        while n < min_forwards or time.perf_counter() - t0 < budget_s:
            toks = sorted(rng.choice(wl.m, tp, replace=False).tolist()) if wl.m > 1 else [0]
            oracle.forward(b["kv"], b["ring"], b["latent"], b["cache"], b["q_idx"], b["k_idx"],
                           w, b["q"], sink, win=wl.win, ratio=wl.ratio, start_pos=wl.start_pos,
                           topk=wl.topk, rd=wl.rd, tokens=toks, fc=fc, timings=timings)
            n += 1
            sampled += len(toks)
    finally:
        oracle.set_num_threads(prev)
    el = time.perf_counter() - t0
    per = {}
    sec_per_token = 0.0
    for st in STAGES:
        if st not in timings:
            continue
        tokens = n * wl.m if st in ("window_ring_write", "compress_latent_write") else sampled
        per[st] = {"seconds": timings[st], "tokens": tokens,
                   "query_tokens_per_s": tokens / timings[st] if timings[st] > 0 else None}
        sec_per_token += timings[st] / tokens
    return {"value": 1.0 / sec_per_token, "threads": used, "forwards": n,
            "sampled_tokens": sampled, "seconds": el, "per_stage": per}


def oracle_baseline(wl, budget_s):
    """cpu_baseline: the oracle as it stands, single-threaded and on all host
    cores, per stage, about ``budget_s`` seconds in all (a third single)."""
    import oracle
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    single = oracle_stage_rates(wl, budget_s / 3.0, 1, toks_per=2 if wl.m > 1 else 1)
    par = oracle_stage_rates(wl, 2.0 * budget_s / 3.0, cores)
    return {"value": par["value"], "unit": "query-tokens/s", "cores": par["threads"],
            "kind": "oracle",
            "sample": (f"{wl.name}: {par['forwards']} oracle forwards on {par['threads']} threads "
                       f"({par['sampled_tokens']} sampled query tokens through the indexer + "
                       f"top-k and the attention, the ring and latent writes whole each time, "
                       f"{par['seconds']:.1f} s), and {single['forwards']} single-threaded "
                       f"({single['sampled_tokens']} sampled tokens, {single['seconds']:.1f} s); "
                       f"value = the whole step's rate on all cores, extrapolated from the "
                       f"per-stage seconds per token"),
            "host_cores": cores,
            "per_stage": {st: {"omp": par["per_stage"][st]["query_tokens_per_s"],
                               "single": single["per_stage"][st]["query_tokens_per_s"]}
                          for st in par["per_stage"]},
            "single_thread": {"value": single["value"], "unit": "query-tokens/s"}}


def oracle_rate(wl, steps=None, budget_s=None):
    """The reference arm's measure: ``steps`` oracle forwards on all host
    cores (see oracle_stage_rates), whole-step query-tokens/s."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    r = oracle_stage_rates(wl, 0.0 if steps else (budget_s or 0.0), cores,
                           min_forwards=steps or 1)
    return {"value": r["value"], "unit": "query-tokens/s", "cores": r["threads"], "kind": "oracle",
            "seconds": r["seconds"],
            "sample": f"{r['forwards']} oracle forwards of {r['sampled_tokens'] // max(1, r['forwards'])} "
                      f"sampled query token(s) each on the {wl.name} workload ({r['seconds']:.1f} s), "
                      f"the ring and latent writes whole each time; value extrapolated from the "
                      f"per-stage seconds per token",
            "per_stage": {k: v["query_tokens_per_s"] for k, v in r["per_stage"].items()}}


def workload_desc(wl) -> str:
    """The workload's name and sizes, the same string in both arms' config."""
    return (f"{wl.name}: m={wl.m} start_pos={wl.start_pos} heads={wl.nh}x{wl.hd} rope={wl.rd} "
            f"window={wl.win} ratio={wl.ratio} compressed_rows={wl.n_c} topk={wl.topk} "
            f"indexer={wl.Hi}x{wl.Di}")


def run_reference(args, world, rank):
    if rank != 0:
        return None
    wl = WORKLOADS[args.workload]
    K, W = args.steps, args.warmup
    oracle_rate(wl, steps=W)                       # warm-up
    cb = oracle_rate(wl, steps=K)
    return {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": cb["unit"],
            "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": 1e3 * cb["seconds"] / max(1, K), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(wl), "global_batch": wl.m,
                       "parallelism": "cpu oracle, bounded sample (see cpu_baseline.sample)"},
            "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample",
                                                "per_stage")},
            "e2e": {"value": cb["value"], "unit": cb["unit"], "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=sorted(WORKLOADS))
    ap.add_argument("--headline-only", action="store_true",
                    help="measure only --workload, not the other four under 'configs'")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of CPU oracle work for the headline's cpu_baseline "
                         "(a quarter of it for each other workload)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per call of the headline's dominant op (default: "
                         "profiles/dram_traffic.txt when taken on the current sources)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None,
                    help="profiling mode: time eager calls of one op (or 'step') and exit")
    ap.add_argument("--slots", type=int, default=4, help="layer states rotated in --only mode")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    world, rank, local = dist_setup()
    if args.only:
        run_only(args, local)
        return
    if args.impl == "reference":
        res = run_reference(args, world, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
    else:
        res, wl = run_ours(args, world, rank, local)
        if rank == 0:
            if world == 1 and not args.no_cpu_baseline:
                res["cpu_baseline"] = oracle_baseline(wl, args.cpu_budget)
                for name, c in res.get("configs", {}).items():
                    c["cpu_baseline"] = oracle_baseline(WORKLOADS[name], args.cpu_budget / 4.0)
            print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
