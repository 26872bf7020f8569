"""The indexer on a packed mxf4 key cache (ds41_indexer_topk_mxf4): the keys
go through ds41_fp4_quant_e8m0 into e2m1 codes and e8m0 block-32 scales (the
form the compress.rs header fixes for the indexer's k), and the block-scaled
tensor-core scores must equal, bit for bit, the oracle's scores on the bf16
keys and the bf16-key entry point's scores; the top-k index sets must equal
the oracle's.  Every workload with 64 indexer heads of dim 128, few-token
(row tiles split over CTAs) and many-token (persistent CTAs over token
groups) launches, ragged groups and ragged row tiles."""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_window_gb300 import ds41
from compressed_sparse_attention_window_gb300.workloads import (CHUNKED, DECODE, LONG_DECODE,
                                                                 PREFILL, TINY_PREFILL, bf16_bits,
                                                                 make_inputs)
from helpers import assert_idx_sets_equal, osizes, sample_tokens, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ds41.load()


def _pack_keys(k_idx):
    _, codes, scales = ds41.fp4_quant(k_idx, e4m3=False, want_codes=True)
    return codes, scales


def _win_idx(orc, wl):
    return torch.from_numpy(orc.window_topk_idxs(wl.win, wl.m, wl.start_pos)).cuda()


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


CASES = [DECODE, LONG_DECODE, CHUNKED, PREFILL, DECODE.replace(start_pos=8191 + 9, topk=4000),
         LONG_DECODE.replace(structure="repeat"), DECODE.replace(m=2, start_pos=5000),
         DECODE.replace(m=3, start_pos=37, ratio=3, topk=64),
         DECODE.replace(m=5, start_pos=130, topk=16)]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: f"{w.name}-{w.m}-{w.start_pos}-{w.topk}")
def test_indexer_mxf4_matches_oracle_and_bf16_keys(orc, wl):
    inp = make_inputs(wl)
    dev = to_dev(inp)
    sz = ds41.step_sizes(wl)
    win_idx = _win_idx(orc, wl)
    k = dev["k_idx"][: sz.n_c].contiguous()
    codes, scales = _pack_keys(k)
    sc = torch.empty(wl.m, sz.n_c, dtype=torch.bfloat16, device="cuda")
    idx = ds41.indexer_topk_mxf4(dev["q_idx"], codes, scales, dev["w"], win_idx, wl.ratio,
                                 wl.start_pos, wl.topk, sz.n_a, scores=sc)
    sc_b = torch.empty_like(sc)
    idx_b = ds41.indexer_topk(dev["q_idx"], k, dev["w"], win_idx, wl.ratio, wl.start_pos,
                              wl.topk, sz.n_a, scores=sc_b)
    torch.cuda.synchronize()
    assert ds41.device_status() == 0
    assert torch.equal(sc, sc_b)
    assert torch.equal(idx, idx_b)
    osz = osizes(orc, wl)
    toks = sample_tokens(wl) if wl.m > 128 else list(range(wl.m))
    osc, bad = orc.indexer_scores(bf16_bits(inp["q_idx"]), bf16_bits(inp["k_idx"])[: osz["n_c"]],
                                  inp["w"].numpy(), wl.ratio, wl.start_pos, tokens=toks)
    assert bad == 0
    gsc = bf16_bits(sc)[toks]
    assert np.array_equal(gsc, osc), np.argwhere(gsc != osc)[:5]
    wi = orc.window_topk_idxs(wl.win, wl.m, wl.start_pos)
    oidx = orc.topk_merge(osc, wi[toks], osz["n_c"], wl.win, wl.ratio, wl.start_pos, wl.topk,
                          osz["n_a"], tokens=toks)
    assert_idx_sets_equal(idx.cpu().numpy()[toks], oidx, wl.win)


@pytest.mark.parametrize("start_pos,ratio", [(0, 8), (1000, 4), (37, 3)])
def test_indexer_mxf4_many_tokens_every_score(orc, start_pos, ratio):
    """More groups of 2 tokens than SMs: persistent CTAs over token groups,
    every score of every token against the oracle, a ragged last group (odd
    m), groups that see no row yet, a ragged last row tile; without a scores
    output the top-k reads the workspace."""
    wl = DECODE.replace(name="indexer_mxf4", m=2 * _sms() + 7, start_pos=start_pos, ratio=ratio,
                        topk=64)
    inp = make_inputs(wl, seed=start_pos + ratio)
    dev = to_dev(inp)
    sz = ds41.step_sizes(wl)
    win_idx = _win_idx(orc, wl)
    codes, scales = _pack_keys(dev["k_idx"][: sz.n_c].contiguous())
    sc = torch.empty(wl.m, sz.n_c, dtype=torch.bfloat16, device="cuda")
    idx = ds41.indexer_topk_mxf4(dev["q_idx"], codes, scales, dev["w"], win_idx, wl.ratio,
                                 wl.start_pos, wl.topk, sz.n_a, scores=sc)
    idx_ws = ds41.indexer_topk_mxf4(dev["q_idx"], codes, scales, dev["w"], win_idx, wl.ratio,
                                    wl.start_pos, wl.topk, sz.n_a)
    torch.cuda.synchronize()
    assert ds41.device_status() == 0
    assert torch.equal(idx, idx_ws)
    osz = osizes(orc, wl)
    osc, bad = orc.indexer_scores(bf16_bits(inp["q_idx"]), bf16_bits(inp["k_idx"])[: osz["n_c"]],
                                  inp["w"].numpy(), wl.ratio, wl.start_pos)
    assert bad == 0
    gsc = bf16_bits(sc)
    assert np.array_equal(gsc, osc), np.argwhere(gsc != osc)[:5]
    toks = sample_tokens(wl)
    wi = orc.window_topk_idxs(wl.win, wl.m, wl.start_pos)
    oidx = orc.topk_merge(osc[toks], wi[toks], osz["n_c"], wl.win, wl.ratio, wl.start_pos,
                          wl.topk, osz["n_a"], tokens=toks)
    assert_idx_sets_equal(idx.cpu().numpy()[toks], oidx, wl.win)


def test_indexer_mxf4_rejects_other_shapes():
    wl = TINY_PREFILL
    inp = to_dev(make_inputs(wl))
    codes, scales = _pack_keys(inp["k_idx"][:16].contiguous())
    win_idx = torch.zeros(wl.m, wl.win, dtype=torch.int32, device="cuda")
    with pytest.raises(ds41.DS41Error) as e:
        ds41.indexer_topk_mxf4(inp["q_idx"], codes, scales, inp["w"], win_idx, wl.ratio,
                               wl.start_pos, wl.topk, wl.m)
    assert e.value.code == 1


FP4_STEP = ["decode", "long_decode", "chunked_prefill", "prefill"]
FP4_EXTRA = [DECODE.replace(start_pos=8190), DECODE.replace(m=2, start_pos=5000),
             DECODE.replace(structure="repeat"), DECODE.replace(start_pos=16399, structure="repeat"),
             DECODE.replace(m=5, start_pos=4000, topk=16)]


@pytest.mark.parametrize("wl", [__import__("compressed_sparse_attention_window_gb300.workloads",
                                           fromlist=["WORKLOADS"]).WORKLOADS[n] for n in FP4_STEP]
                         + FP4_EXTRA, ids=lambda w: f"{w.name}-{w.m}-{w.start_pos}")
def test_csa_forward_fp4_matches_the_bf16_step(orc, wl):
    """The step on packed caches gives bit for bit the outputs and layer state
    of ds41_csa_forward on the bf16 caches (fused few-token front with the
    mxf4 scores kernel's step-1 CTAs and the attention gathering the packed
    latent rows, or the separate calls), its packed latent rows equal the
    oracle's codes and scales, and o matches the oracle.  The prior cache rows
    are method output: each side quantises the drawn rows with its own
    e4m3 quantiser."""
    from compressed_sparse_attention_window_gb300.workloads import from_bits
    from helpers import attn_close, oracle_forward
    inp = make_inputs(wl)
    # the oracle's prior cache: its own fp4 round trip of the drawn rows
    ocq, occ, ocs = orc.fp4_quant(bf16_bits(inp["cache"]), 16, True)
    oinp = dict(inp)
    oinp["cache"] = from_bits(ocq)
    ora_fc = orc.yarn_freqs_cis(wl.rd, max(wl.max_pos, 1))
    fc = torch.from_numpy(ora_fc).cuda()
    d1, d2 = to_dev(inp), to_dev(inp)
    cq, cc, cs = ds41.fp4_quant(d1["cache"], e4m3=True, want_codes=True)
    d1["cache"], d2["cache"] = cq.clone(), cq.clone()
    d2["cache_codes"], d2["cache_scales"] = cc, cs
    sz = ds41.step_sizes(wl)
    d2["k_codes"], d2["k_scales"] = ds41.pack_keys(d2["k_idx"][: sz.n_c].contiguous())
    out1 = ds41.csa_forward(d1, wl, fc)
    out2 = ds41.csa_forward_fp4(d2, wl, fc)
    torch.cuda.synchronize()
    assert ds41.device_status() == 0
    assert torch.equal(d1["ring"], d2["ring"]) and torch.equal(d1["cache"], d2["cache"])
    assert torch.equal(out1["win_idx"], out2["win_idx"])
    assert torch.equal(out1["idx"], out2["idx"])
    assert torch.equal(out1["o"], out2["o"])
    toks = sample_tokens(wl) if wl.m > 128 else list(range(wl.m))
    ref = oracle_forward(orc, wl, oinp, tokens=toks, fc=ora_fc)
    osz = ref["sizes"]
    first = osz["n_c"] - osz["G"]
    # the rows this call wrote: the oracle's latent codes; the rows before it:
    # the oracle's round trip of the drawn rows
    gcc, gcs = d2["cache_codes"].cpu().numpy(), d2["cache_scales"].cpu().numpy()
    assert np.array_equal(gcc[first:osz["n_c"]], ref["codes"][first:osz["n_c"]])
    assert np.array_equal(gcs[first:osz["n_c"]], ref["scales"][first:osz["n_c"]])
    assert np.array_equal(gcc[:first], occ[:first]) and np.array_equal(gcs[:first], ocs[:first])
    assert np.array_equal(bf16_bits(d2["cache"]), ref["cache"])
    assert_idx_sets_equal(out2["idx"].cpu().numpy()[toks], ref["idx"], wl.win)
    ok, err, worst = attn_close(out2["o"].float().cpu().numpy()[toks], ref["o"])
    assert ok, (wl.name, err, worst)


@pytest.mark.parametrize("name", ["decode", "long_decode"])
def test_csa_forward_fp4_graph_replay_matches_eager(name):
    from compressed_sparse_attention_window_gb300.workloads import WORKLOADS
    wl = WORKLOADS[name]
    inp = make_inputs(wl)
    fc = ds41.yarn_freqs_cis(wl.rd, max(wl.max_pos, 1))
    sz = ds41.step_sizes(wl)

    def dev():
        d = to_dev(inp)
        d["k_codes"], d["k_scales"] = ds41.pack_keys(d["k_idx"][: sz.n_c].contiguous())
        return d
    dev_e = dev()
    out_e = ds41.csa_forward_fp4(dev_e, wl, fc)
    out_g = {}
    ds41.csa_forward_fp4(dev(), wl, fc, out_g)
    dev_g = dev()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ds41.csa_forward_fp4(dev_g, wl, fc, out_g)
    for k in ("o", "idx"):
        out_g[k].fill_(0)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_e["o"], out_g["o"]) and torch.equal(out_e["idx"], out_g["idx"])
    assert torch.equal(dev_e["ring"], dev_g["ring"]) and torch.equal(dev_e["cache"], dev_g["cache"])
