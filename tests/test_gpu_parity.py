"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: fp4 quantisers (values, codes, scales), ring / window indices /
rows_a, latent cache rows (values, codes, scales), indexer scores, top-k index
sets.  Attention: |gpu - oracle| <= 2e-2 + 1e-2 |oracle| (f64 oracle).
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_window_gb300 import ds41
from compressed_sparse_attention_window_gb300.workloads import (CHUNKED, DECODE, LONG_DECODE,
                                                                 PREFILL, TINY_PREFILL, WORKLOADS,
                                                                 OUT_PROJ, bf16_bits, from_bits,
                                                                 make_inputs,
                                                                 make_out_proj_weights)
from helpers import (assert_idx_sets_equal, attn_close, oracle_forward, osizes, sample_tokens,
                     to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ds41.load()
    yield
    assert ds41.device_status() == 0


def _special_rows(cols, block, rng):
    """Rows that hit the corners of the fp4 round trip: zero blocks, blocks at
    exactly 6*2^k, values on e2m1 midpoints, tiny and huge values, negatives."""
    rows = []
    z = np.zeros(cols, np.float32)
    rows.append(z)
    r = rng.standard_normal(cols).astype(np.float32)
    r[:block] = 0.0
    r[block: 2 * block] = -1e-30
    rows.append(r)
    e = np.zeros(cols, np.float32)
    for b in range(cols // block):
        k = (b % 20) - 10
        e[b * block] = 6.0 * 2.0 ** k
        mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -2.5, -5.0]) * 2.0 ** k
        e[b * block + 1: b * block + 1 + min(len(mids), block - 1)] = mids[: block - 1]
    rows.append(e)
    rows.append(rng.standard_normal(cols).astype(np.float32) * 1e4)
    rows.append(rng.standard_normal(cols).astype(np.float32) * 1e-6)
    return np.stack(rows)


@pytest.mark.parametrize("e4m3", [False, True])
@pytest.mark.parametrize("rows,cols", [(1, 32), (37, 128), (300, 512), (3, 4096)])
def test_fp4_quant_bit_exact(orc, e4m3, rows, cols):
    block = 16 if e4m3 else 32
    rng = np.random.default_rng(rows * 7 + cols)
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    x[rng.random(x.shape) < 0.01] *= 20
    x = np.concatenate([x, _special_rows(cols, block, rng)])
    xb = torch.from_numpy(x).to(torch.bfloat16)
    y, codes, scales = ds41.fp4_quant(xb.cuda(), e4m3, want_codes=True)
    oy, ocodes, oscales = orc.fp4_quant(bf16_bits(xb), block, e4m3)
    assert np.array_equal(bf16_bits(y), oy)
    assert np.array_equal(codes.cpu().numpy(), ocodes)
    assert np.array_equal(scales.cpu().numpy(), oscales)


def test_fp4_quant_all_bf16_values(orc):
    """Every finite bf16 bit pattern through both quantisers, each inside a
    block whose scale is fixed by a planted maximum."""
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = (allb.astype(np.uint32) << 16).view(np.float32)
    allb = allb[np.isfinite(vals)]
    for e4m3, block in ((False, 32), (True, 16)):
        per = block - 1
        n = (allb.size + per - 1) // per
        rows_per = 512 // block
        n = (n + rows_per - 1) // rows_per * rows_per
        pad = np.zeros(n * per, np.uint16)
        pad[: allb.size] = allb
        blocks = pad.reshape(n, per)
        for amax_bits in (0x3F80, 0x4300, 0x0000):  # 1.0, 128.0, none
            col0 = np.full((n, 1), amax_bits, np.uint16)
            x = np.ascontiguousarray(np.concatenate([col0, blocks], axis=1).reshape(-1, 512))
            xt = from_bits(x)
            y, codes, scales = ds41.fp4_quant(xt.cuda(), e4m3, want_codes=True)
            oy, ocodes, oscales = orc.fp4_quant(x, block, e4m3)
            assert np.array_equal(bf16_bits(y), oy)
            assert np.array_equal(codes.cpu().numpy(), ocodes)
            assert np.array_equal(scales.cpu().numpy(), oscales)


def test_yarn_table_matches_oracle(orc):
    rd, seqlen = 64, 140000
    fc_gpu = ds41.yarn_freqs_cis(rd, seqlen).cpu().numpy().astype(np.float64)
    fc_ora = orc.yarn_freqs_cis(rd, seqlen).astype(np.float64)
    f = orc.yarn_inv_freqs(rd, 65536, 160000.0, 16.0, 32.0, 1.0).astype(np.float64)
    p = np.arange(seqlen, dtype=np.float64)[:, None]
    # cos/sin of the same f32 angle agree to a few ulp; one ulp of difference in
    # a frequency moves the angle by p * ulp(f), which bounds the rest.
    ulp_f = np.spacing(f.astype(np.float32)).astype(np.float64)
    tol = 4e-7 + p * ulp_f[None, :]
    err = np.abs(fc_gpu - fc_ora).max(axis=2)
    assert np.all(err <= tol), float(err.max())
    # the frequencies themselves: identical in nearly every entry
    assert np.mean(err[:2000] <= 4e-7) == 1.0


RING_CASES = [(1, 0, 16), (16, 0, 16), (64, 0, 16), (70, 0, 16), (1, 3, 16), (1, 17, 16),
              (1, 8191, 128), (5, 40, 16), (24, 37, 16), (300, 1000, 128), (1024, 65536, 128)]


@pytest.mark.parametrize("m,sp,win", RING_CASES)
def test_window_ring_bit_exact(orc, m, sp, win):
    hd = 64
    wl = TINY_PREFILL.replace(m=m, start_pos=sp, win=win, hd=hd, rd=16)
    inp = make_inputs(wl, seed=m + sp)
    ring_d = inp["ring"].cuda()
    win_idx = torch.empty(m, win, dtype=torch.int32, device="cuda")
    rows_a = ds41.window_ring_write(inp["kv"].cuda(), ring_d, win_idx, sp)
    oring, orows = orc.window_ring_write(bf16_bits(inp["kv"]), bf16_bits(inp["ring"]), win, sp)
    assert np.array_equal(bf16_bits(ring_d), oring)
    assert np.array_equal(bf16_bits(rows_a), orows)
    assert np.array_equal(win_idx.cpu().numpy(), orc.window_topk_idxs(win, m, sp))
    assert ds41.rows_a_len(m, win, sp) == orc.rows_a_len(m, win, sp)


LATENT_CASES = [(TINY_PREFILL, None), (DECODE, None), (PREFILL, None), (LONG_DECODE, None),
                (CHUNKED, None), (TINY_PREFILL.replace(m=3, start_pos=9), None),
                (TINY_PREFILL.replace(m=1, start_pos=10), None)]


@pytest.mark.parametrize("wl", [c[0] for c in LATENT_CASES], ids=lambda w: f"{w.name}-{w.m}-{w.start_pos}")
def test_latent_write_bit_exact(orc, wl):
    inp = make_inputs(wl)
    fc = orc.yarn_freqs_cis(wl.rd, wl.max_pos)  # the table is an input of the write
    cache_d = inp["cache"].cuda()
    rows = cache_d.shape[0]
    codes = torch.zeros(rows, wl.hd // 2, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(rows, wl.hd // 16, dtype=torch.uint8, device="cuda")
    if ds41.step_sizes(wl).G > 0:
        ds41.compress_latent_write(inp["latent"].cuda(), torch.from_numpy(fc).cuda(), cache_d,
                                   wl.rd, wl.ratio, wl.start_pos, wl.m, codes, scales)
    ocache, ocodes, oscales = orc.compress_latent_write(bf16_bits(inp["latent"]), fc,
                                                        bf16_bits(inp["cache"]), wl.rd, wl.ratio,
                                                        wl.start_pos, wl.m)
    assert np.array_equal(bf16_bits(cache_d), ocache)
    osz = osizes(orc, wl)
    first = osz["n_c"] - osz["G"]
    sl = slice(first, first + osz["G"])
    assert np.array_equal(codes.cpu().numpy()[sl], ocodes[sl])
    assert np.array_equal(scales.cpu().numpy()[sl], oscales[sl])


def _gpu_indexer(wl, inp, with_scores=True):
    dev = to_dev(inp)
    win_idx = torch.from_numpy(
        np.ascontiguousarray(np.zeros((wl.m, wl.win), np.int32))).cuda()
    from oracle import window_topk_idxs
    win_idx.copy_(torch.from_numpy(window_topk_idxs(wl.win, wl.m, wl.start_pos)))
    sz = ds41.step_sizes(wl)
    scores = torch.empty(wl.m, sz.n_c, dtype=torch.bfloat16, device="cuda") if with_scores else None
    idx = ds41.indexer_topk(dev["q_idx"], dev["k_idx"][: sz.n_c], dev["w"], win_idx, wl.ratio,
                            wl.start_pos, wl.topk, sz.n_a, scores=scores)
    return idx, scores


INDEXER_CASES = [TINY_PREFILL, TINY_PREFILL.replace(topk=64), DECODE, LONG_DECODE, CHUNKED,
                 PREFILL, TINY_PREFILL.replace(m=37, start_pos=5, Hi=5, Di=64),
                 DECODE.replace(start_pos=8191 + 9, m=1, topk=4000),
                 # tied scores in long slices (the cluster top-k with keys in registers)
                 LONG_DECODE.replace(structure="repeat")]


@pytest.mark.parametrize("wl", INDEXER_CASES, ids=lambda w: f"{w.name}-{w.m}-{w.start_pos}-{w.topk}-{w.Hi}")
def test_indexer_scores_and_topk(orc, wl):
    inp = make_inputs(wl)
    idx, scores = _gpu_indexer(wl, inp)
    toks = sample_tokens(wl) if wl.m > 128 else list(range(wl.m))
    osz = osizes(orc, wl)
    sc, bad = orc.indexer_scores(bf16_bits(inp["q_idx"]), bf16_bits(inp["k_idx"])[: osz["n_c"]],
                                 inp["w"].numpy(), wl.ratio, wl.start_pos, tokens=toks)
    assert bad == 0
    gsc = bf16_bits(scores)[toks]
    assert np.array_equal(gsc, sc), np.argwhere(gsc != sc)[:5]
    win_idx = orc.window_topk_idxs(wl.win, wl.m, wl.start_pos)
    oidx = orc.topk_merge(sc, win_idx[toks], osz["n_c"], wl.win, wl.ratio, wl.start_pos, wl.topk,
                          osz["n_a"], tokens=toks)
    assert_idx_sets_equal(idx.cpu().numpy()[toks], oidx, wl.win)
    # the picks of a row come in ascending row order, -1 padding last
    g = idx.cpu().numpy()[:, wl.win:]
    for r in g[:: max(1, wl.m // 64)]:
        v = r[r >= 0]
        assert np.all(np.diff(v) > 0) and np.all(r[len(v):] == -1)


@pytest.mark.parametrize("start_pos,ratio", [(0, 8), (1000, 4), (37, 3)])
def test_indexer_many_tokens_tensor_core_path(orc, start_pos, ratio):
    """Enough tokens for a group of 4 per SM (64 heads x 128) take the tcgen05
    scores kernel: every score of every token bit-exact against the oracle,
    including a ragged last group, groups whose tokens see no row yet (their
    scores are all -inf) and a ragged last row tile; then the top-k sets."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    wl = DECODE.replace(name="indexer_tc", m=4 * sms + 3, start_pos=start_pos, ratio=ratio,
                        topk=64)
    osz = osizes(orc, wl)
    assert wl.Hi == 64 and wl.Di == 128 and osz["n_c"] > 0
    inp = make_inputs(wl, seed=start_pos + ratio)
    idx, scores = _gpu_indexer(wl, inp)
    sc, bad = orc.indexer_scores(bf16_bits(inp["q_idx"]), bf16_bits(inp["k_idx"])[: osz["n_c"]],
                                 inp["w"].numpy(), wl.ratio, wl.start_pos)
    assert bad == 0
    gsc = bf16_bits(scores)
    assert np.array_equal(gsc, sc), np.argwhere(gsc != sc)[:5]
    win_idx = orc.window_topk_idxs(wl.win, wl.m, wl.start_pos)
    toks = sample_tokens(wl)
    oidx = orc.topk_merge(sc[toks], win_idx[toks], osz["n_c"], wl.win, wl.ratio, wl.start_pos,
                          wl.topk, osz["n_a"], tokens=toks)
    assert_idx_sets_equal(idx.cpu().numpy()[toks], oidx, wl.win)


@pytest.mark.parametrize("sink_kind", ["normal", "minus_inf", "large"])
def test_sparse_attn_given_indices(orc, sink_kind):
    wl = TINY_PREFILL.replace(m=40, start_pos=0, topk=12, nh=20, hd=128)
    inp = make_inputs(wl, seed=5)
    if sink_kind == "minus_inf":
        inp["sink"][:] = -float("inf")
    elif sink_kind == "large":
        inp["sink"] *= 30
    rng = np.random.default_rng(3)
    n_a, n_c, K = 40, 17, 45
    rows_a = torch.randn(n_a, wl.hd).to(torch.bfloat16)
    rows_b = torch.randn(n_c, wl.hd).to(torch.bfloat16)
    idx = rng.integers(-1, n_a + n_c, (wl.m, K)).astype(np.int32)
    idx[3, :] = -1          # a row with no valid index
    idx[4, 1:] = -1         # a single valid index
    o = ds41.sparse_attn_sink_fwd(inp["q"].cuda(), rows_a.cuda(), rows_b.cuda(),
                                  torch.from_numpy(idx).cuda(), inp["sink"].cuda(), wl.scale)
    oo, _, bad = orc.sparse_attn(bf16_bits(inp["q"]), bf16_bits(rows_a), bf16_bits(rows_b), idx,
                                 inp["sink"].numpy(), wl.scale)
    assert bad == 0
    ok, err, worst = attn_close(o.float().cpu().numpy(), oo)
    assert ok, (err, worst)


@pytest.mark.parametrize("m,nh", [(1, 64), (2, 64), (3, 20), (12, 64), (40, 16)])
@pytest.mark.parametrize("K", [1, 31, 33, 640, 2176])
def test_sparse_attn_few_token_paths(orc, K, m, nh):
    """Few tokens take the cluster path (m * heads/16 small) or the split-K
    partials + merge (larger m); both against the oracle."""
    hd = 512
    n_a, n_c = 128, 2500
    g = torch.Generator().manual_seed(K + 7 * m)
    q = torch.randn(m, nh, hd, generator=g).to(torch.bfloat16)
    rows_a = torch.randn(n_a, hd, generator=g).to(torch.bfloat16)
    rows_b = torch.randn(n_c, hd, generator=g).to(torch.bfloat16)
    sink = torch.randn(nh, generator=g)
    rng = np.random.default_rng(K)
    idx = np.stack([rng.permutation(n_a + n_c)[:K] for _ in range(m)]).astype(np.int32)
    if K > 40:
        idx[0, 5:9] = -1
    lse = torch.empty(m, nh, device="cuda")
    o = ds41.sparse_attn_sink_fwd(q.cuda(), rows_a.cuda(), rows_b.cuda(),
                                  torch.from_numpy(idx).cuda(), sink.cuda(), hd ** -0.5, lse=lse)
    oo, olse, _ = orc.sparse_attn(bf16_bits(q), bf16_bits(rows_a), bf16_bits(rows_b), idx,
                                  sink.numpy(), np.float32(hd ** -0.5))
    ok, err, worst = attn_close(o.float().cpu().numpy(), oo)
    assert ok, (err, worst)
    assert np.allclose(lse.cpu().numpy(), olse, atol=1e-3, rtol=1e-4)


def _tc_index_rows(m, n_a, n_c, K, rng):
    """Index rows that exercise every chunk form of the many-token kernel:
    compact ranges of both sources (consecutive-row chunks with masks),
    scattered rows and sparse ranges (listed rows), repeated rows, rows with
    no or one valid index, padding with -1, and scattered rows_a beside a
    compact range of rows_b (listed chunks of the first source with
    consecutive-row chunks of the second)."""
    idx = np.full((m, K), -1, np.int32)
    for t in range(m):
        kind = t % 7
        if kind == 0:   # a window-like run of rows_a + most of a range of rows_b,
            #             the range rounded up to whole 128-row chunks (kept as
            #             consecutive-row chunks with holes in their masks)
            w = min(K // 3, n_a)
            a0 = rng.integers(0, n_a - w + 1)
            nb = min(K - w, n_c // 2)
            span = min(-(-nb // 128) * 128, n_c)
            b0 = rng.integers(0, n_c - span + 1)
            picks = b0 + rng.permutation(span)[:nb]
            row = np.concatenate([np.arange(a0, a0 + w), n_a + picks])
        elif kind == 5:  # half of a range of rows_b: listed rows (fewer chunks)
            nb = min(K, n_c // 2)
            b0 = rng.integers(0, n_c - 2 * nb + 1)
            row = n_a + b0 + rng.permutation(2 * nb)[:nb]
        elif kind == 1:  # scattered over everything
            row = rng.permutation(n_a + n_c)[:K]
        elif kind == 2:  # a compact range with repeated rows
            n = K - 3
            b0 = rng.integers(0, n_c - n + 1)
            row = n_a + b0 + rng.integers(0, n, n)
        elif kind == 6:  # scattered rows_a + a compact range of rows_b
            na = min(K // 4, n_a)
            nb = min(K - na, n_c)
            b0 = rng.integers(0, n_c - nb + 1)
            row = np.concatenate([rng.permutation(n_a)[:na], n_a + b0 + np.arange(nb)])
        elif kind == 3:  # a few valid rows among -1
            row = rng.permutation(n_a + n_c)[: max(1, K // 9)]
        else:            # rows_b only, ascending, every third row
            n = min(K, n_c // 3)
            b0 = rng.integers(0, n_c - 3 * n + 1)
            row = n_a + b0 + 3 * np.arange(n)
        row = row[:K]
        rng.shuffle(row)
        idx[t, : len(row)] = row
        if kind != 1:
            rng.shuffle(idx[t])
    idx[3, :] = -1           # no valid index at all
    idx[8, :] = -1
    idx[8, K // 2] = 5       # exactly one valid index
    return idx


@pytest.mark.parametrize("K,nh,sink_kind,sm", [(37, 64, "normal", 1.0), (640, 64, "normal", 1.0),
                                               (640, 64, "minus_inf", 1.0), (640, 128, "large", 1.0),
                                               (1000, 64, "normal", 1.0), (640, 64, "normal", -1.0),
                                               (300, 64, "normal", 0.0)])
def test_sparse_attn_many_tokens_tensor_core_path(orc, K, nh, sink_kind, sm):
    """Enough tokens for one work item per SM (hd 512, 64-head groups, K <=
    1024) take the persistent tcgen05 kernel; every token against the oracle.
    A third of the compressed rows are scaled x3 so that later chunks beat the
    running maximum by far (the rescale of O in tensor memory).  The scale is
    head_dim^-0.5 times sm: a negative scale flips which rows weigh most, and
    a zero scale weighs every selected row alike."""
    hd = 512
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    m = sms + 13
    n_a, n_c = 300, 2100
    g = torch.Generator().manual_seed(K + nh)
    q = torch.randn(m, nh, hd, generator=g).to(torch.bfloat16)
    rows_a = torch.randn(n_a, hd, generator=g).to(torch.bfloat16)
    rb = torch.randn(n_c, hd, generator=g)
    rb[::3] *= 3.0
    rows_b = rb.to(torch.bfloat16)
    sink = torch.randn(nh, generator=g)
    if sink_kind == "minus_inf":
        sink[:] = -float("inf")
    elif sink_kind == "large":
        sink *= 30
    idx = _tc_index_rows(m, n_a, n_c, K, np.random.default_rng(K * 3 + nh))
    lse = torch.empty(m, nh, device="cuda")
    scale = float(np.float32(hd ** -0.5 * sm))
    o = ds41.sparse_attn_sink_fwd(q.cuda(), rows_a.cuda(), rows_b.cuda(),
                                  torch.from_numpy(idx).cuda(), sink.cuda(), scale, lse=lse)
    oo, olse, bad = orc.sparse_attn(bf16_bits(q), bf16_bits(rows_a), bf16_bits(rows_b), idx,
                                    sink.numpy(), np.float32(scale))
    assert bad == 0
    assert ds41.device_status() == 0
    ok, err, worst = attn_close(o.float().cpu().numpy(), oo)
    assert ok, (err, worst)
    fin = np.isfinite(olse)
    assert np.array_equal(np.isfinite(lse.cpu().numpy()), fin)
    assert np.allclose(lse.cpu().numpy()[fin], olse[fin], atol=1e-3, rtol=1e-4)


def test_sparse_attn_bad_index_sets_status(orc):
    nh, hd = 4, 64
    q = torch.randn(1, nh, hd).to(torch.bfloat16).cuda()
    rows = torch.randn(8, hd).to(torch.bfloat16).cuda()
    idx = torch.tensor([[0, 1, 99, 2]], dtype=torch.int32).cuda()  # 99 is out of range
    sink = torch.zeros(nh).cuda()
    assert ds41.device_status(reset=True) == 0
    o = ds41.sparse_attn_sink_fwd(q, rows, None, idx, sink, 0.125)
    assert ds41.device_status(reset=True) == 4  # DS41_E_INDEX; the row was skipped
    ok_idx = np.array([[0, 1, -1, 2]], np.int32)
    oo, _, _ = orc.sparse_attn(bf16_bits(q), bf16_bits(rows), None, ok_idx,
                               np.zeros(nh, np.float32), 0.125)
    assert attn_close(o.float().cpu().numpy(), oo)[0]


FORWARD_CASES = ["tiny_prefill", "decode", "long_decode", "chunked_prefill", "prefill"]


@pytest.mark.parametrize("name", FORWARD_CASES)
def test_forward_end_to_end(orc, name):
    """All steps through the C ABI, launched as bench.py launches them,
    against the oracle on sampled tokens (every token for small m)."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl)
    dev = to_dev(inp)
    fc = ds41.yarn_freqs_cis(wl.rd, wl.max_pos)
    ora_fc = orc.yarn_freqs_cis(wl.rd, wl.max_pos)
    out = ds41.forward(dev, wl, torch.from_numpy(ora_fc).cuda())
    toks = sample_tokens(wl) if wl.m > 128 else list(range(wl.m))
    ref = oracle_forward(orc, wl, inp, tokens=toks, fc=ora_fc)
    assert np.array_equal(bf16_bits(dev["ring"]), ref["ring"])
    assert np.array_equal(bf16_bits(dev["cache"]), ref["cache"])
    assert_idx_sets_equal(out["idx"].cpu().numpy()[toks], ref["idx"], wl.win)
    ok, err, worst = attn_close(out["o"].float().cpu().numpy()[toks], ref["o"])
    assert ok, (name, err, worst)
    assert fc.shape == (wl.max_pos, wl.rd // 2, 2)


def test_forward_no_compressed_rows_yet(orc):
    """start_pos + m < ratio: no compressed row exists, the merged rows are the
    window rows alone."""
    wl = TINY_PREFILL.replace(m=3, start_pos=0, ratio=4)
    assert osizes(orc, wl)["n_c"] == 0 and ds41.step_sizes(wl).n_c == 0
    inp = make_inputs(wl)
    dev = to_dev(inp)
    fc = torch.from_numpy(orc.yarn_freqs_cis(wl.rd, wl.max_pos)).cuda()
    out = ds41.forward(dev, wl, fc)
    ref = oracle_forward(orc, wl, inp, fc=fc.cpu().numpy())
    assert np.array_equal(out["idx"].cpu().numpy(), ref["idx"])
    assert attn_close(out["o"].float().cpu().numpy(), ref["o"])[0]


CSA_CASES = ["tiny_prefill", "decode", "long_decode", "chunked_prefill", "prefill"]
CSA_EXTRA = [TINY_PREFILL.replace(m=1, start_pos=43), TINY_PREFILL.replace(m=3, start_pos=37),
             TINY_PREFILL.replace(m=1, start_pos=2), DECODE.replace(start_pos=8190),
             DECODE.replace(m=2, start_pos=5000), TINY_PREFILL.replace(m=2, start_pos=0),
             # tied scores: every CTA ranks all 2048 (or 546) visible rows itself ...
             DECODE.replace(structure="repeat"), CHUNKED.replace(m=1, start_pos=70000),
             # ... or, past 4096 visible rows, the cluster splits them
             DECODE.replace(start_pos=16399, structure="repeat"),
             # the generic attention selecting its own rows after the fused
             # front (one wave of CTAs): a chunk with tied scores, two head
             # groups, and past 1024 visible rows the separate top-k again
             TINY_PREFILL.replace(start_pos=200, structure="repeat"),
             TINY_PREFILL.replace(m=100, start_pos=1000),
             TINY_PREFILL.replace(m=40, nh=80, start_pos=300),
             TINY_PREFILL.replace(start_pos=5000)]


@pytest.mark.parametrize("wl", [WORKLOADS[n] for n in CSA_CASES] + CSA_EXTRA,
                         ids=lambda w: f"{w.name}-{w.m}-{w.start_pos}")
def test_csa_forward_matches_oracle_and_the_four_calls(orc, wl):
    """ds41_csa_forward (fused few-token path or the four calls) against the
    oracle, and bit-for-bit against running the four entry points."""
    inp = make_inputs(wl)
    ora_fc = orc.yarn_freqs_cis(wl.rd, max(wl.max_pos, 1))
    fc = torch.from_numpy(ora_fc).cuda()
    dev1, dev2 = to_dev(inp), to_dev(inp)
    out1 = ds41.csa_forward(dev1, wl, fc)
    out2 = ds41.forward(dev2, wl, fc)
    torch.cuda.synchronize()
    assert torch.equal(dev1["ring"], dev2["ring"]) and torch.equal(dev1["cache"], dev2["cache"])
    assert torch.equal(out1["idx"], out2["idx"])
    assert torch.equal(out1["o"], out2["o"])
    toks = sample_tokens(wl) if wl.m > 128 else list(range(wl.m))
    ref = oracle_forward(orc, wl, inp, tokens=toks, fc=ora_fc)
    assert np.array_equal(bf16_bits(dev1["ring"]), ref["ring"])
    assert np.array_equal(bf16_bits(dev1["cache"]), ref["cache"])
    assert_idx_sets_equal(out1["idx"].cpu().numpy()[toks], ref["idx"], wl.win)
    ok, err, worst = attn_close(out1["o"].float().cpu().numpy()[toks], ref["o"])
    assert ok, (wl.name, err, worst)


@pytest.mark.parametrize("name", ["decode", "long_decode", "tiny_prefill", "chunked_prefill", "prefill"])
def test_csa_forward_graph_replay_matches_eager(name):
    """The whole step captured as one CUDA graph (the form the benchmark
    replays, launches chained by programmatic dependent launch) gives bit for
    bit the outputs and the layer state of the same step run eagerly."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl)
    fc = ds41.yarn_freqs_cis(wl.rd, max(wl.max_pos, 1))
    dev_e = to_dev(inp)
    out_e = ds41.csa_forward(dev_e, wl, fc)
    out_g = {}
    ds41.csa_forward(to_dev(inp), wl, fc, out_g)  # allocates the outputs outside the capture
    dev_g = to_dev(inp)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ds41.csa_forward(dev_g, wl, fc, out_g)
    for k in ("o", "idx"):
        out_g[k].fill_(0)
    graph.replay()
    torch.cuda.synchronize()
    assert ds41.device_status() == 0
    assert torch.equal(dev_g["ring"], dev_e["ring"]) and torch.equal(dev_g["cache"], dev_e["cache"])
    assert torch.equal(out_g["idx"], out_e["idx"])
    assert torch.equal(out_g["o"], out_e["o"])


@pytest.mark.parametrize("wl", [WORKLOADS["decode"], WORKLOADS["tiny_prefill"],
                                TINY_PREFILL.replace(m=3, start_pos=37), CHUNKED.replace(m=2, start_pos=70000)],
                         ids=lambda w: f"{w.name}-{w.m}-{w.start_pos}")
@pytest.mark.parametrize("packed", [False, True])
def test_csa_forward_host_buffers(wl, packed):
    """ds41_csa_forward_host (inputs and output in page-locked host memory,
    copied on the stream; separate buffers, or one block on each side that the
    call moves in one copy) gives bit-for-bit the results of ds41_csa_forward
    on device tensors, and leaves the same layer state; a prepared call runs
    again with the same result."""
    inp = make_inputs(wl)
    fc = ds41.yarn_freqs_cis(wl.rd, max(wl.max_pos, 1))
    dev_ref = to_dev(inp)
    ref = ds41.csa_forward(dev_ref, wl, fc)
    dev = to_dev(inp)
    step = ds41.STEP_INPUTS
    if packed:
        dev.update(ds41.step_input_buffers(wl, "cuda"))
        host = ds41.step_input_buffers(wl, "cpu", pinned=True)
        for k in step:
            host[k].copy_(inp[k])
    else:
        host = {k: inp[k].contiguous().pin_memory() for k in step}
    for k in step:  # the device buffers start as garbage: the call must fill them
        dev[k].fill_(7)
    out = {}
    h_o = ds41.csa_forward_host(host, dev, wl, fc, out)
    torch.cuda.synchronize()
    assert torch.equal(h_o, ref["o"].cpu())
    assert torch.equal(out["idx"], ref["idx"])
    assert torch.equal(dev["ring"], dev_ref["ring"]) and torch.equal(dev["cache"], dev_ref["cache"])
    # a prepared call, run twice from the same starting layer state
    start = to_dev(inp)
    again = ds41.HostStep(host, dev, wl, fc, out, h_o=h_o)
    assert again.packed == packed  # one block each side: the packed entry point
    for _ in range(2):
        h_o.zero_()
        dev["ring"].copy_(start["ring"])
        dev["cache"].copy_(start["cache"])
        again()
        torch.cuda.synchronize()
        assert torch.equal(h_o, ref["o"].cpu())
    if packed:
        # the same call recorded once into a CUDA graph (ds41_host_step_create),
        # launched twice from the same starting state: the same bits
        rec = ds41.HostStep(host, dev, wl, fc, out, h_o=h_o, graph=True)
        for _ in range(2):
            h_o.zero_()
            dev["ring"].copy_(start["ring"])
            dev["cache"].copy_(start["cache"])
            rec()
            torch.cuda.synchronize()
            assert torch.equal(h_o, ref["o"].cpu())
            assert torch.equal(out["idx"], ref["idx"])
            assert torch.equal(dev["ring"], dev_ref["ring"])
            assert torch.equal(dev["cache"], dev_ref["cache"])
        rec.close()


@pytest.mark.parametrize("wl", [WORKLOADS["decode"], WORKLOADS["tiny_prefill"]],
                         ids=lambda w: w.name)
@pytest.mark.parametrize("packed", [False, True])
def test_csa_forward_host_pageable(wl, packed):
    """Pageable host buffers (not page-locked, so not mapped for the device)
    go through the copy engines rather than the copy kernel, and give the
    same bits as the device-tensor step."""
    inp = make_inputs(wl)
    fc = ds41.yarn_freqs_cis(wl.rd, max(wl.max_pos, 1))
    dev_ref = to_dev(inp)
    ref = ds41.csa_forward(dev_ref, wl, fc)
    dev = to_dev(inp)
    step = ds41.STEP_INPUTS
    if packed:
        dev.update(ds41.step_input_buffers(wl, "cuda"))
        host = ds41.step_input_buffers(wl, "cpu", pinned=False)
        for k in step:
            host[k].copy_(inp[k])
    else:
        host = {k: inp[k].contiguous().clone() for k in step}
    assert not any(host[k].is_pinned() for k in step)
    h_o = torch.empty(tuple(inp["q"].shape), dtype=torch.bfloat16)  # pageable too
    out = {}
    got = ds41.csa_forward_host(host, dev, wl, fc, out, h_o=h_o)
    torch.cuda.synchronize()
    assert torch.equal(got, ref["o"].cpu())
    assert torch.equal(out["idx"], ref["idx"])
    assert torch.equal(dev["ring"], dev_ref["ring"]) and torch.equal(dev["cache"], dev_ref["cache"])


# --------------------------------------------------------------------------
# The output side of the layer: inverse RoPE, grouped wo_a, wo_b
# --------------------------------------------------------------------------
def _out_proj_check(orc, o_bits, fc, wa, wb, og, out, rd, groups, start_pos, toks):
    """og against the oracle's f64-summed og.  Here the rotated dims of o are
    rounded to bf16 (the tensor-core operand; the oracle keeps them f32, as
    the pages do), which moves each product by at most 2^-9 of its size (a
    rotated value is at most the norm of its pair, so allow 2^-8), and og's
    own bf16 rounding can then land one step apart (2^-7 relative):
      |og - og_ref| <= 2^-8 * sum_i |o_i| |w_i| + 2^-7 |og_ref|.
    out within 1e-2 of its rms plus 1e-2 relative (bf16 operands)."""
    rog, rout = orc.attn_out_proj(o_bits, fc, bf16_bits(wa), bf16_bits(wb), rd=rd, groups=groups,
                                  start_pos=start_pos, tokens=toks)
    gog = og.float().cpu().numpy()[toks].astype(np.float64)
    fog = (rog.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    m, nh, hd = o_bits.shape
    ao = np.abs((o_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    ao = ao.reshape(m, groups, -1)[toks]
    aw = np.abs(wa.float().numpy().astype(np.float64))
    o_rank = aw.shape[0] // groups
    S = np.concatenate([ao[:, g] @ aw[g * o_rank:(g + 1) * o_rank].T for g in range(groups)], 1)
    assert np.all(np.abs(gog - fog) <= 2.0 ** -8 * S + 2.0 ** -7 * np.abs(fog))
    gout = out.cpu().numpy()[toks].astype(np.float64)
    rms = np.sqrt(np.mean(rout ** 2))
    err = np.abs(gout - rout)
    assert np.all(err <= 1e-2 * rms + 1e-2 * np.abs(rout)), (err.max(), rms)


@pytest.mark.parametrize("m,nh,hd,rd,groups,o_rank,dim,start_pos",
                         [(3, 4, 64, 16, 2, 32, 48, 5), (37, 8, 128, 32, 4, 64, 200, 0),
                          (1, 64, 512, 64, 8, 1024, 7168, 8191),
                          (5, 64, 512, 64, 8, 1024, 7168, 100),
                          (40, 16, 512, 64, 4, 256, 1024, 7),
                          (100, 8, 256, 32, 2, 128, 256, 9),
                          (130, 8, 512, 64, 2, 128, 384, 3)])
def test_attn_out_proj_matches_oracle(orc, m, nh, hd, rd, groups, o_rank, dim, start_pos):
    """ds41_attn_out_proj against the oracle, every token, from a small case
    to one decode token at the full sizes: the few-token kernel (a warp per
    weight row, tokens in chunks of 1, 2, 4 or 8), the tensor-core kernel with
    token tiles of 64, 128 and 256 (ragged last tile), and the few-token
    kernel for more tokens when the row groups are not whole 128-row tiles."""
    g = torch.Generator().manual_seed(m + nh + dim)
    o = torch.randn(m, nh, hd, generator=g).to(torch.bfloat16)
    wts = make_out_proj_weights(nh, hd, groups, o_rank, dim, seed=m)
    fc = ds41.yarn_freqs_cis(rd, start_pos + m) if rd else torch.zeros(1, 1, 2).cuda()
    o_bits = bf16_bits(o)
    od = o.cuda()
    og, out = ds41.attn_out_proj(od, fc, wts["wo_a"].cuda(), wts["wo_b"].cuda(), rd, groups,
                                 start_pos)
    torch.cuda.synchronize()
    _out_proj_check(orc, o_bits, fc.cpu().numpy(), wts["wo_a"], wts["wo_b"], og, out, rd, groups,
                    start_pos, list(range(m)))
    # only the rotary dims of o changed
    od_f = bf16_bits(od.cpu()).reshape(m, nh, hd)
    assert np.array_equal(od_f[:, :, : hd - rd], o_bits.reshape(m, nh, hd)[:, :, : hd - rd])


@pytest.mark.parametrize("name", ["prefill", "chunked_prefill"])
def test_attn_out_proj_full_size_sampled(orc, name):
    """The attention output of a many-token workload through the output side
    at the full sizes, checked on sampled tokens."""
    wl = WORKLOADS[name]
    P = OUT_PROJ
    inp = make_inputs(wl)
    dev = to_dev(inp)
    fc = ds41.yarn_freqs_cis(wl.rd, wl.max_pos)
    o = ds41.csa_forward(dev, wl, fc)["o"]
    o_bits = bf16_bits(o)
    wts = make_out_proj_weights(wl.nh, wl.hd, P["groups"], P["o_rank"], P["dim"])
    og, out = ds41.attn_out_proj(o, fc, wts["wo_a"].cuda(), wts["wo_b"].cuda(), wl.rd, P["groups"],
                                 wl.start_pos)
    torch.cuda.synchronize()
    assert ds41.device_status() == 0
    toks = sample_tokens(wl)[:8]
    _out_proj_check(orc, o_bits, fc.cpu().numpy(), wts["wo_a"], wts["wo_b"], og, out, wl.rd,
                    P["groups"], wl.start_pos, toks)


# --------------------------------------------------------------------------
# A layer that reuses the source layer's compressed rows and picks
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["decode", "long_decode", "tiny_prefill", "chunked_prefill",
                                  "prefill"])
def test_csa_forward_reuse(orc, name):
    """ds41_csa_forward_reuse for a second layer (its own q, kv, ring, sink)
    on the first layer's compressed rows and picks: bit for bit the ring
    write, the merge and the attention called separately, and the oracle's
    attention over the oracle's own window indices and picks of the first
    layer."""
    wl = WORKLOADS[name]
    fc = ds41.yarn_freqs_cis(wl.rd, max(wl.max_pos, 1))
    src = make_inputs(wl)
    dev_s = to_dev(src)
    out_s = ds41.csa_forward(dev_s, wl, fc)
    sz = ds41.step_sizes(wl)
    ctopk = sz.ctopk
    cidx = out_s["idx"][:, wl.win:].contiguous() if ctopk else None
    cache = dev_s["cache"]
    lay = make_inputs(wl, seed=4242)
    dev_r = to_dev(lay)
    out_r = ds41.csa_forward_reuse(dev_r, wl, cache, cidx)
    # the same through the separate entry points
    dev_c = to_dev(lay)
    chunk = wl.start_pos > 0 and wl.m > 1
    rows_a = torch.empty(wl.win + wl.m, wl.hd, dtype=torch.bfloat16, device="cuda") if chunk else None
    win_idx = torch.empty(wl.m, wl.win, dtype=torch.int32, device="cuda")
    ds41.window_ring_write(dev_c["kv"], dev_c["ring"], win_idx, wl.start_pos, rows_a=rows_a)
    ra = dev_c["kv"] if wl.start_pos == 0 else (dev_c["ring"] if wl.m == 1 else rows_a)
    idx = torch.cat([win_idx, cidx], 1) if ctopk else win_idx
    o_c = ds41.sparse_attn_sink_fwd(dev_c["q"], ra, cache[: sz.n_c] if ctopk else None, idx,
                                    dev_c["sink"], wl.scale)
    torch.cuda.synchronize()
    assert ds41.device_status() == 0
    assert torch.equal(dev_r["ring"], dev_c["ring"])
    assert torch.equal(out_r["win_idx"], win_idx)
    if ctopk:
        assert torch.equal(out_r["idx"], idx)
    assert torch.equal(out_r["o"], o_c)
    # the oracle: this layer's rows_a and window indices, the first layer's picks
    toks = sample_tokens(wl) if wl.m > 128 else list(range(wl.m))
    ref_s = oracle_forward(orc, wl, src, tokens=toks, fc=fc.cpu().numpy())
    _, rows_a_o = orc.window_ring_write(bf16_bits(lay["kv"]), bf16_bits(lay["ring"]), wl.win,
                                        wl.start_pos)
    win_o = orc.window_topk_idxs(wl.win, wl.m, wl.start_pos)[toks]
    on_c = ref_s["sizes"]["n_c"]
    idx_o = np.concatenate([win_o, ref_s["idx"][:, wl.win:]], 1) if on_c else win_o
    o_ref, _, bad = orc.sparse_attn(bf16_bits(lay["q"]), rows_a_o,
                                    ref_s["cache"][:on_c] if on_c else None, idx_o,
                                    lay["sink"].numpy(), orc.attn_scale(wl.hd), tokens=toks)
    assert bad == 0
    ok, err, worst = attn_close(out_r["o"].float().cpu().numpy()[toks], o_ref)
    assert ok, (name, err, worst)
