"""The attention entry point that allocates nothing.

Some callers cannot allocate device memory (serving runtimes that reserve all
of it at start-up, plugin hosts that provide only input and output buffers).
ds41_sparse_attn_sink_fwd_noalloc gives them the split attention with its
partials in the library's static scratch array.  These tests call it through
the C ABI and check that it returns what the workspace entry point returns,
within the attention tolerance of the parity tests, on two calls in a row
(the second call finds the first call's partials still in the shared array).
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_window_gb300 import ds41

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 1e-2


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


def test_noalloc_matches_workspace_entry_point_twice():
    # token counts between the cluster path and full prefill take the split
    # path, whose partials live in the static scratch
    shapes = [(10, 64, 512, 128, 2048, 640), (40, 16, 512, 128, 32768, 2176)]
    for call, (m, nh, hd, n_a, n_c, K) in enumerate(shapes):
        assert ds41.sparse_attn_workspace_bytes(m, nh, hd, K) > 0
        q, ra, rb, idx, sink = _case(100 + call, m, nh, hd, n_a, n_c, K)
        scale = hd ** -0.5
        ref_lse = torch.empty(m, nh, device="cuda")
        ref = ds41.sparse_attn_sink_fwd(q, ra, rb, idx, sink, scale, lse=ref_lse)
        o = torch.empty_like(q)
        lse = torch.empty(m, nh, device="cuda")
        ds41.sparse_attn_sink_fwd_noalloc(q, ra, rb, idx, sink, scale, o, lse=lse)
        torch.cuda.synchronize()
        a = o.float().cpu().numpy()
        b = ref.float().cpu().numpy()
        assert np.all(np.abs(a - b) <= ATOL + RTOL * np.abs(b)), call
        assert np.allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), atol=1e-3, rtol=1e-4)
    assert ds41.device_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    m, nh, hd, K = 12, 64, 512, 2176
    need = ds41.sparse_attn_workspace_bytes(m, nh, hd, K)
    assert need > ds41.sparse_attn_noalloc_capacity()
    q, ra, rb, idx, sink = _case(7, m, nh, hd, 128, 4096, K)
    o = torch.zeros_like(q)
    with pytest.raises(ds41.DS41Error) as e:
        ds41.sparse_attn_sink_fwd_noalloc(q, ra, rb, idx, sink, hd ** -0.5, o)
    assert e.value.code == 5  # DS41_E_WORKSPACE, nothing enqueued
    torch.cuda.synchronize()
    assert torch.count_nonzero(o).item() == 0
