"""The C ABI library: it builds for sm_103a, loads, exports every entry point
include/ds41.h declares, and rejects bad arguments on the host before any
device work (no GPU needed for these)."""
import ctypes
import os
import re

import pytest

from compressed_sparse_attention_window_gb300 import build as ds41_build
from compressed_sparse_attention_window_gb300 import ds41

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ds41.h")


@pytest.fixture(scope="module")
def lib():
    ds41_build.build()
    return ds41.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ds41_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = _declared()
    for n in ("ds41_fp4_quant_e8m0", "ds41_fp4_quant_e4m3", "ds41_window_ring_write",
              "ds41_compress_latent_write", "ds41_indexer_topk", "ds41_sparse_attn_sink_fwd"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(_declared()) == set(ds41.SIGNATURES), "binding signatures out of date"


def test_rows_a_len(lib):
    assert lib.ds41_rows_a_len(64, 16, 0) == 64
    assert lib.ds41_rows_a_len(1, 128, 8191) == 128
    assert lib.ds41_rows_a_len(1024, 128, 65536) == 1152


def test_step_sizes(lib):
    """ds41_step_sizes on the five workloads' call parameters, against the row
    counts worked out by hand: n_a, n_c, G, ctopk, K."""
    from compressed_sparse_attention_window_gb300.workloads import WORKLOADS
    want = {"tiny_prefill": (64, 16, 16, 8, 24), "decode": (128, 2048, 1, 512, 640),
            "prefill": (4096, 1024, 1024, 512, 640), "long_decode": (128, 32768, 1, 2048, 2176),
            "chunked_prefill": (1152, 520, 8, 512, 640)}
    for name, w in want.items():
        assert tuple(ds41.step_sizes(WORKLOADS[name])) == w, name
    out = (ctypes.c_int64 * 5)()
    assert lib.ds41_step_sizes(3, 0, 16, 4, 8, ctypes.addressof(out)) == 0
    assert tuple(out) == (3, 0, 0, 0, 16)  # no compressed row yet: no picks
    assert lib.ds41_step_sizes(0, 0, 16, 4, 8, ctypes.addressof(out)) == 2
    assert lib.ds41_step_sizes(3, 0, 16, 0, 8, ctypes.addressof(out)) == 1
    assert lib.ds41_step_sizes(3, 0, 16, 4, 8, None) == 1


def test_selftest_checks_arguments(lib):
    assert lib.ds41_selftest_wait_timeout(100, 0, None, None) == 1
    assert lib.ds41_selftest_wait_timeout(0, 0, FAKE, None) == 1


def _err(lib):
    return lib.ds41_last_error().decode()


FAKE = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first


def test_host_argument_checks(lib):
    # the forward's own limits: at least one token
    assert lib.ds41_window_ring_write(FAKE, FAKE, None, FAKE, None, 0, 64, 16, 0, None) == 2
    assert "m=0" in _err(lib)
    # a chunk past position 0 needs rows_a
    assert lib.ds41_window_ring_write(FAKE, FAKE, None, FAKE, None, 4, 64, 16, 8, None) == 1
    # hd not a multiple of 8
    assert lib.ds41_window_ring_write(FAKE, FAKE, None, FAKE, None, 4, 60, 16, 0, None) == 1
    # misaligned pointer
    bad = ctypes.c_void_p((1 << 20) + 2)
    assert lib.ds41_fp4_quant_e8m0(bad, FAKE, None, None, 1, 32, None) == 1
    # cols not a multiple of the block
    assert lib.ds41_fp4_quant_e8m0(FAKE, FAKE, None, None, 1, 48, None) == 1
    assert lib.ds41_fp4_quant_e4m3(FAKE, FAKE, None, None, 1, 24, None) == 1
    # wrong group count for the latent write
    assert lib.ds41_compress_latent_write(FAKE, FAKE, 100, FAKE, 100, None, None, 3, 64, 16, 4,
                                          0, 8, None) == 1
    # cache too small
    assert lib.ds41_compress_latent_write(FAKE, FAKE, 100, FAKE, 1, None, None, 2, 64, 16, 4, 0,
                                          8, None) == 2
    # indexer: unsupported Di, topk < 1
    assert lib.ds41_indexer_topk(FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 2, 48, 4, 16, 4, 0, 8, 16,
                                 None, 0, None) == 1
    assert lib.ds41_indexer_topk(FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 2, 32, 4, 16, 4, 0, 0, 16,
                                 None, 0, None) == 2
    # attention: unsupported head dim, no tokens
    assert lib.ds41_sparse_attn_sink_fwd(FAKE, FAKE, 4, None, 0, FAKE, 4, FAKE,
                                         ctypes.c_float(0.1), FAKE, None, 1, 4, 96, None, 0,
                                         None) == 1
    assert lib.ds41_sparse_attn_sink_fwd(FAKE, FAKE, 4, None, 0, FAKE, 4, FAKE,
                                         ctypes.c_float(0.1), FAKE, None, 0, 4, 64, None, 0,
                                         None) == 2


def test_workspace_sizes_are_host_only(lib):
    # the indexer needs scratch for its scores unless the caller takes them
    assert lib.ds41_indexer_workspace_bytes(4096, 64, 128, 1024, 0) >= 4096 * 1024 * 2
    assert lib.ds41_indexer_workspace_bytes(1, 64, 128, 2048, 1) == 0


def test_host_buffer_entry_points_check_arguments(lib):
    """ds41_csa_forward_host[_packed] reject bad sizes and missing buffers on
    the host, before any copy is enqueued."""
    # sizes of the decode workload: m=1, start_pos=8191, 64x512 heads, ratio 4,
    # indexer 64x128: q 64 KiB + kv 1 KiB + one latent row 1 KiB + q_idx 16 KiB + w 256 B
    assert lib.ds41_step_inputs_bytes(1, 8191, 64, 512, 4, 64, 128) == 65536 + 1024 + 1024 + 16384 + 256
    # no group completes: no latent bytes
    assert lib.ds41_step_inputs_bytes(1, 8192, 64, 512, 4, 64, 128) == 65536 + 1024 + 16384 + 256
    assert lib.ds41_step_inputs_bytes(0, 0, 64, 512, 4, 64, 128) == 0
    f = ctypes.c_float(0.04)
    sizes = (8191, 64, 512, 64, 128, 4, 512, 64, 128)  # start_pos nh hd rd win ratio topk Hi Di

    def host_call(h_latent, m):
        # h_q h_kv h_latent h_q_idx h_w h_o | q kv ring rows_a latent freqs_cis max_pos cache
        # cache_rows q_idx k_idx w sink scale win_idx idx o lse | m, sizes | ws ws_bytes stream
        return lib.ds41_csa_forward_host(FAKE, FAKE, h_latent, FAKE, FAKE, FAKE,
                                         FAKE, FAKE, FAKE, None, FAKE, FAKE, 1 << 20, FAKE, 1 << 20,
                                         FAKE, FAKE, FAKE, FAKE, f, FAKE, FAKE, FAKE, None,
                                         m, *sizes, None, 0, None)

    # per-buffer form: a completed group needs h_latent
    assert host_call(None, 1) == 1 and "null pointer" in _err(lib)
    assert host_call(FAKE, 0) == 1  # no token
    # packed form: no host block
    rc = lib.ds41_csa_forward_host_packed(None, FAKE, FAKE, FAKE, None, FAKE, 1 << 20, FAKE, 1 << 20,
                                          FAKE, FAKE, f, FAKE, FAKE, FAKE, None,
                                          1, *sizes, None, 0, None)
    assert rc == 1 and "null pointer" in _err(lib)


def test_host_step_checks_arguments(lib):
    """ds41_host_step_create rejects a missing handle slot, sizes and buffers
    on the host (leaving the handle NULL); launching a NULL handle is an
    argument error and destroying one a no-op."""
    f = ctypes.c_float(0.04)
    sizes = (8191, 64, 512, 64, 128, 4, 512, 64, 128)  # start_pos nh hd rd win ratio topk Hi Di
    h = ctypes.c_void_p(0x1234)

    def create(out, h_in, m):
        # out | h_in d_in h_o ring rows_a freqs_cis max_pos cache cache_rows k_idx sink scale
        # win_idx idx o lse | m, sizes | ws ws_bytes
        return lib.ds41_host_step_create(out, h_in, FAKE, FAKE, FAKE, None, FAKE, 1 << 20, FAKE,
                                         1 << 20, FAKE, FAKE, f, FAKE, FAKE, FAKE, None, m, *sizes,
                                         None, 0)

    assert create(None, FAKE, 1) == 1 and "out is NULL" in _err(lib)
    assert create(ctypes.byref(h), None, 1) == 1 and "null pointer" in _err(lib)
    assert h.value is None
    h = ctypes.c_void_p(0x1234)
    assert create(ctypes.byref(h), FAKE, 0) == 1 and h.value is None  # no token
    assert lib.ds41_host_step_launch(None, None) == 1 and "NULL" in _err(lib)
    assert lib.ds41_host_step_destroy(None) == 0


def test_attn_out_proj_checks_arguments(lib):
    """ds41_attn_out_proj rejects bad sizes and pointers on the host, before
    anything is enqueued (no GPU needed)."""
    def call(o=FAKE, fc=FAKE, max_pos=100, m=2, start_pos=0, nh=4, hd=64, rd=16, groups=2,
             o_rank=32, dim=48, og=FAKE):
        return lib.ds41_attn_out_proj(o, fc, max_pos, FAKE, FAKE, og, FAKE, m, start_pos, nh, hd,
                                      rd, groups, o_rank, dim, None)
    assert call(m=0) == 2                      # no token
    assert call(start_pos=99) == 2             # positions past freqs_cis
    assert call(o=None) == 1 and "non-null" in _err(lib)
    assert call(og=None) == 1
    assert call(rd=15) == 1                    # odd rotary width
    assert call(groups=3) == 1                 # 256 values do not split into 3 groups
    assert call(dim=50) == 1                   # dim % 4
    assert call(fc=None) == 1                  # a rotation needs the table


def test_csa_forward_reuse_checks_arguments(lib):
    """ds41_csa_forward_reuse checks the ring write's and the attention's
    arguments before it enqueues anything (no GPU needed; the workspace size
    depends on the device and is not checked here)."""
    f = ctypes.c_float(0.04)

    def call(q=FAKE, cidx=FAKE, ctopk=512, hd=512, m=1, start_pos=8191, ratio=4, ws=FAKE,
             ws_bytes=1 << 30):
        # q kv ring rows_a cache cidx ctopk sink scale win_idx idx o lse | m start_pos nh hd win
        # ratio | ws ws_bytes stream
        return lib.ds41_csa_forward_reuse(q, FAKE, FAKE, None, FAKE, cidx, ctopk, FAKE, f, FAKE,
                                          FAKE, FAKE, None, m, start_pos, 64, hd, 128, ratio, ws,
                                          ws_bytes, None)
    assert call(m=0) == 2
    assert call(ctopk=4096) == 1               # more picks than compressed rows
    assert call(cidx=None) == 1                # picks required when ctopk > 0
    assert call(hd=96) == 1                    # the attention's head width
    assert call(q=None) == 1
