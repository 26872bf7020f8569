"""The algorithmic work bench.py divides by (the roofline numerators), pinned
to closed forms worked out by hand, and the guard that reports recorded DRAM
traffic only for the kernel sources it was measured on."""
import bench
from compressed_sparse_attention_window_gb300.workloads import WORKLOADS


def test_prefill_valid_rows_closed_form():
    """Prefill (m = 4096 at 0, window 128, ratio 4, top-k 512): token t sees
    min(t + 1, 128) window rows and min(512, (t + 1) // 4) compressed rows.
    Window: 1 + .. + 128 + (4096 - 128) * 128 = 8256 + 507904 = 516160.
    Compressed: n = t + 1 below 2048 gives each q = 0 .. 511 four times,
    4 * (511 * 512 / 2) = 523264; n = 2048 .. 4096 gives 2049 * 512 = 1049088.
    Total 2088512 rows; attention flops 4 * 64 * 512 * rows = 273.7 G."""
    wl = WORKLOADS["prefill"]
    assert bench.attn_valid_rows(wl) == 516160 + 523264 + 1049088 == 2088512
    alg = bench.algorithmic(wl)
    assert alg["sparse_attn_sink_fwd"]["flops"] == 4 * 64 * 512 * 2088512
    assert round(alg["sparse_attn_sink_fwd"]["flops"] / 1e9, 1) == 273.7


def test_chunked_and_decode_valid_rows():
    """Chunked prefill (m = 1024 at 65536, ratio 128): every token has a full
    window of 128 and at least 65537 // 128 = 512 visible rows, so the top-512
    keeps 512: 1024 * 640 = 655360 rows (85.9 GFLOP).  Decode at 8191 sees 128
    window rows and 8192 // 4 = 2048 compressed rows, keeps 512: 640 rows."""
    ch = WORKLOADS["chunked_prefill"]
    assert bench.attn_valid_rows(ch) == 1024 * 640
    assert round(bench.algorithmic(ch)["sparse_attn_sink_fwd"]["flops"] / 1e9, 1) == 85.9
    assert bench.attn_valid_rows(WORKLOADS["decode"]) == 640
    assert bench.attn_valid_rows(WORKLOADS["long_decode"]) == 128 + 2048


def test_indexer_pairs_closed_form():
    """Prefill indexer flops: 2 * 64 * 128 per causally visible (query, row)
    pair; token t sees min(1024, n // 4) rows, n = t + 1.  n = 1 .. 2047 gives
    q = 0 .. 511 four times (523264), n = 2048 .. 4095 gives q = 512 .. 1023
    four times (4 * (512 + 1023) * 512 / 2 = 1571840), and n = 4096 gives
    1024: 2096128 pairs."""
    alg = bench.algorithmic(WORKLOADS["prefill"])
    assert alg["indexer_topk"]["flops"] == 2 * 64 * 128 * 2096128


def test_recorded_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    """A traffic line gives its number only while the digest at its end
    matches the current sources of that op's kernels."""
    cur = bench.csrc_digest("sparse_attn_sink_fwd")
    assert cur != bench.csrc_digest("indexer_topk_mxf4")
    table = tmp_path / "t.txt"
    table.write_text("# workload op bytes time kernels digest\n"
                     f"prefill sparse_attn_sink_fwd 5e8 600.0 k {cur}\n"
                     "prefill indexer_topk 1e8 90.0 k 0000000000000000\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(table))
    assert bench.recorded_traffic("prefill", "sparse_attn_sink_fwd") == 5e8
    assert bench.recorded_traffic("prefill", "indexer_topk") is None
    assert bench.recorded_traffic("prefill", "no_such_op") is None
    assert bench.recorded_traffic("decode", "sparse_attn_sink_fwd") is None


def test_committed_traffic_table_parses():
    """Every line of the committed table names a known op and carries bytes,
    a time and a 16-digit digest."""
    for line in open(bench.TRAFFIC_FILE).read().splitlines():
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        assert f[1] in bench.OP_SOURCES, line
        float(f[2]), float(f[3])
        assert len(f[-1]) == 16, line


def test_packed_cache_bytes_closed_form():
    """Decode on packed caches: the attention gathers 128 window rows of
    1024 B and 512 compressed rows of 256 code bytes + 32 scale bytes, plus q
    and o (2 x 64 x 512 x 2 B), 640 indices and 64 sinks:
    131072 + 147456 + 131072 + 2560 + 256 = 412416 B (789248 B on the bf16
    cache).  The mxf4 indexer reads 2048 key rows of 64 + 4 B instead of 256 B:
    16384 (q) + 139264 + 256 (w) + 512 (window indices) + 2560 (idx)."""
    alg = bench.algorithmic(WORKLOADS["decode"])
    assert alg["sparse_attn_sink_fwd"]["bytes"] == 789248
    assert alg["sparse_attn_sink_fwd_fp4"]["bytes"] == 412416
    assert alg["indexer_topk_mxf4"]["bytes"] == 16384 + 2048 * 68 + 256 + 512 + 2560
