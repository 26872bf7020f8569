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
