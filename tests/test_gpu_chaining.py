"""Consecutive steps of one layer launched back to back, with no host
synchronisation between them: eagerly, as one CUDA graph, and as prepared
host-buffer steps.  The kernels of a step launch while the one before them
runs (programmatic dependent launch) and wait for it before they touch
memory; the next step's front overwrites the ring slot, the scores workspace
and (for chunks) the rows_a buffer that the previous step's attention reads.
Every step must give bit for bit what the same steps give one at a time with a
synchronisation after each.
"""
import pytest
import torch

from compressed_sparse_attention_window_gb300 import ds41
from compressed_sparse_attention_window_gb300.workloads import (CHUNKED, DECODE, TINY_PREFILL,
                                                                 make_inputs)

pytestmark = pytest.mark.gpu

STATE = ("ring", "cache", "k_idx", "sink")
PER_STEP = ("q", "kv", "latent", "q_idx", "w")
S = 6  # consecutive steps

CASES = [
    DECODE,                                     # fused front + attention selecting its rows
    DECODE.replace(start_pos=1001),             # the same, where some steps complete a group
    TINY_PREFILL.replace(m=3, start_pos=37),    # chunks of three tokens
    CHUNKED.replace(m=2, start_pos=70000),      # chunks past a heavily compressed prefix
    TINY_PREFILL,                               # 64-token chunks: the generic attention selecting its rows
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ds41.load()
    yield
    assert ds41.device_status() == 0


def _steps(wl):
    steps = [wl.replace(start_pos=wl.start_pos + i * wl.m) for i in range(S)]
    last = steps[-1]
    # the layer state sized for the last step (its cache holds every row the
    # steps write), the per-step inputs drawn with their own seeds
    state = make_inputs(last, seed=wl.seed)
    per = [make_inputs(s, seed=wl.seed + 101 + i) for i, s in enumerate(steps)]
    fc = ds41.yarn_freqs_cis(wl.rd, last.max_pos)
    return steps, state, per, fc


def _shared(steps, dev):
    """rows_a and the workspace, shared by all steps as a serving loop would."""
    sh = {}
    need = max(ds41.csa_workspace_bytes(s) for s in steps)
    if need:
        sh["ws_csa"] = torch.empty(need, dtype=torch.uint8, device=dev)
    wl = steps[0]
    if wl.start_pos > 0 and wl.m > 1:
        sh["rows_a"] = torch.empty(wl.win + wl.m, wl.hd, dtype=torch.bfloat16, device=dev)
    return sh


def _fresh_state(state):
    return {k: state[k].cuda().contiguous() for k in STATE}


def _enqueue(steps, st, per_dev, outs, fc):
    for i, wl in enumerate(steps):
        inp = dict(st)
        inp.update(per_dev[i])
        ds41.csa_forward(inp, wl, fc, outs[i])


@pytest.mark.parametrize("wl", CASES, ids=lambda w: f"{w.name}-{w.m}-{w.start_pos}")
def test_consecutive_steps_back_to_back(wl):
    steps, state, per, fc = _steps(wl)
    per_dev = [{k: p[k].cuda().contiguous() for k in PER_STEP} for p in per]

    def new_outs(sh):
        return [dict(sh) for _ in steps]

    # reference: one step at a time, synchronised after each
    st_ref = _fresh_state(state)
    outs_ref = new_outs(_shared(steps, "cuda"))
    for i, w in enumerate(steps):
        inp = dict(st_ref)
        inp.update(per_dev[i])
        ds41.csa_forward(inp, w, fc, outs_ref[i])
        torch.cuda.synchronize()
    assert ds41.device_status() == 0

    # back to back on one stream, no synchronisation until the end
    st = _fresh_state(state)
    outs = new_outs(_shared(steps, "cuda"))
    _enqueue(steps, st, per_dev, outs, fc)
    torch.cuda.synchronize()
    assert ds41.device_status() == 0
    for i in range(S):
        assert torch.equal(outs[i]["o"], outs_ref[i]["o"]), f"step {i}: o"
        assert torch.equal(outs[i]["idx"], outs_ref[i]["idx"]), f"step {i}: idx"
    assert torch.equal(st["ring"], st_ref["ring"]) and torch.equal(st["cache"], st_ref["cache"])

    # the same steps recorded as one CUDA graph and replayed from the start state
    st_g = _fresh_state(state)
    start = {k: v.clone() for k, v in st_g.items()}
    outs_g = new_outs(_shared(steps, "cuda"))
    _enqueue(steps, st_g, per_dev, outs_g, fc)  # every output allocated outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _enqueue(steps, st_g, per_dev, outs_g, fc)
    for rep in range(2):
        for k in ("ring", "cache"):
            st_g[k].copy_(start[k])
        for o in outs_g:
            o["o"].zero_()
            o["idx"].fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        assert ds41.device_status() == 0
        for i in range(S):
            assert torch.equal(outs_g[i]["o"], outs_ref[i]["o"]), f"graph {rep}, step {i}: o"
            assert torch.equal(outs_g[i]["idx"], outs_ref[i]["idx"]), f"graph {rep}, step {i}: idx"
        assert torch.equal(st_g["ring"], st_ref["ring"])
        assert torch.equal(st_g["cache"], st_ref["cache"])


@pytest.mark.parametrize("wl", [CASES[0], CASES[1], CASES[2]],
                         ids=lambda w: f"{w.name}-{w.m}-{w.start_pos}")
def test_consecutive_host_steps_back_to_back(wl):
    """Prepared host-buffer steps (one copy in, the step, the copy of o out,
    recorded as a CUDA graph) launched back to back: each step's o in host
    memory equals the synchronised device steps'."""
    steps, state, per, fc = _steps(wl)
    per_dev = [{k: p[k].cuda().contiguous() for k in PER_STEP} for p in per]
    st_ref = _fresh_state(state)
    outs_ref = [dict(_shared(steps, "cuda")) for _ in steps]
    for i, w in enumerate(steps):
        inp = dict(st_ref)
        inp.update(per_dev[i])
        ds41.csa_forward(inp, w, fc, outs_ref[i])
        torch.cuda.synchronize()

    st = _fresh_state(state)
    sh = _shared(steps, "cuda")
    calls, h_os = [], []
    for i, w in enumerate(steps):
        host = ds41.step_input_buffers(w, "cpu", pinned=True)
        dev = ds41.step_input_buffers(w, "cuda")
        for k in PER_STEP:
            host[k].copy_(per[i][k])
            dev[k].fill_(7)  # garbage until the step's copy lands
        inp = dict(st)
        inp.update(dev)
        h_o = torch.empty(tuple(dev["q"].shape), dtype=torch.bfloat16).pin_memory()
        calls.append(ds41.HostStep(host, inp, w, fc, dict(sh), h_o=h_o, graph=True))
        assert calls[-1].packed
        h_os.append(h_o)
    torch.cuda.synchronize()
    for c in calls:
        c()
    torch.cuda.synchronize()
    assert ds41.device_status() == 0
    for i in range(S):
        assert torch.equal(h_os[i], outs_ref[i]["o"].cpu()), f"host step {i}: o"
    assert torch.equal(st["ring"], st_ref["ring"]) and torch.equal(st["cache"], st_ref["cache"])
    for c in calls:
        c.close()
