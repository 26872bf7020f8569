"""The attention entry point that allocates nothing.

Some callers cannot allocate device memory: serving runtimes that reserve all
of it at start-up and forbid allocation afterwards, and plugin hosts that
hand a kernel only its input and output buffers.
ds41_sparse_attn_sink_fwd_noalloc gives them the split attention with its
partials in the library's static scratch array.  These tests call it
through the C ABI on two calls in a row (the second call finds the first
call's partials still in the shared array) and check that it returns
exactly what the workspace entry point returns (both run the same kernels on
the same plan), and, once, what the oracle returns within the attention
tolerance of the parity tests.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_window_gb300 import ds41
from compressed_sparse_attention_window_gb300.workloads import bf16_bits
from helpers import attn_close

pytestmark = pytest.mark.gpu


def _case(seed, m, nh, hd, n_a, n_c, K):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(m, nh, hd, generator=g).to(torch.bfloat16).cuda()
    rows_a = torch.randn(n_a, hd, generator=g).to(torch.bfloat16).cuda()
    rows_b = torch.randn(n_c, hd, generator=g).to(torch.bfloat16).cuda()
    sink = torch.randn(nh, generator=g).cuda()
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(n_a + n_c)[:K] for _ in range(m)]).astype(np.int32)
    idx[:, -3:] = -1
    return q, rows_a, rows_b, torch.from_numpy(idx).cuda(), sink


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ds41.load()


def _fitting(shapes):
    """The shapes whose split partials fit the static array on this GPU (the
    plan depends on its SM count)."""
    cap = ds41.sparse_attn_noalloc_capacity()
    return [s for s in shapes
            if 0 < ds41.sparse_attn_workspace_bytes(s[0], s[1], s[2], s[5]) <= cap]


def test_noalloc_matches_workspace_entry_point_twice(orc):
    # token counts between the cluster path and full prefill take the split
    # path, whose partials live in the static scratch
    cands = [(10, 64, 512, 128, 2048, 640), (40, 16, 512, 128, 32768, 2176),
             (6, 64, 512, 128, 4096, 640), (24, 32, 256, 128, 1024, 300)]
    shapes = _fitting(cands)
    if len(shapes) < 2:
        pytest.skip("fewer than two split-path shapes fit the static scratch on this GPU")
    for call, (m, nh, hd, n_a, n_c, K) in enumerate(shapes[:2]):
        q, ra, rb, idx, sink = _case(100 + call, m, nh, hd, n_a, n_c, K)
        scale = hd ** -0.5
        ref_lse = torch.empty(m, nh, device="cuda")
        ref = ds41.sparse_attn_sink_fwd(q, ra, rb, idx, sink, scale, lse=ref_lse)
        o = torch.empty_like(q)
        lse = torch.empty(m, nh, device="cuda")
        ds41.sparse_attn_sink_fwd_noalloc(q, ra, rb, idx, sink, scale, o, lse=lse)
        torch.cuda.synchronize()
        assert torch.equal(o, ref), call
        assert torch.equal(lse, ref_lse), call
        if call == 0:
            oo, olse, bad = orc.sparse_attn(bf16_bits(q), bf16_bits(ra), bf16_bits(rb),
                                            idx.cpu().numpy(), sink.cpu().numpy(),
                                            np.float32(scale))
            assert bad == 0
            ok, err, worst = attn_close(o.float().cpu().numpy(), oo)
            assert ok, (err, worst)
            assert np.allclose(lse.cpu().numpy(), olse, atol=1e-3, rtol=1e-4)
    assert ds41.device_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    cap = ds41.sparse_attn_noalloc_capacity()
    m, nh, hd, K = None, 64, 512, 2176
    for mm in (12, 16, 24, 32):
        if ds41.sparse_attn_workspace_bytes(mm, nh, hd, K) > cap:
            m = mm
            break
    if m is None:
        pytest.skip("no split-path shape here needs more than the static scratch")
    q, ra, rb, idx, sink = _case(7, m, nh, hd, 128, 4096, K)
    o = torch.zeros_like(q)
    with pytest.raises(ds41.DS41Error) as e:
        ds41.sparse_attn_sink_fwd_noalloc(q, ra, rb, idx, sink, hd ** -0.5, o)
    assert e.value.code == 5  # DS41_E_WORKSPACE, nothing enqueued
    torch.cuda.synchronize()
    assert torch.count_nonzero(o).item() == 0


def test_noalloc_checks_output_shapes():
    q, ra, rb, idx, sink = _case(9, 10, 64, 512, 128, 2048, 640)
    with pytest.raises(ValueError):
        ds41.sparse_attn_sink_fwd_noalloc(q, ra, rb, idx, sink, 512 ** -0.5, torch.empty_like(q[:5]))
    with pytest.raises(ValueError):
        ds41.sparse_attn_sink_fwd_noalloc(q, ra, rb, idx, sink, 512 ** -0.5, torch.empty_like(q),
                                          lse=torch.empty(10, 32, device="cuda"))
