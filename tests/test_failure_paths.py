"""The failure path of the bounded device-side waits, on the GPU, without a
GPU fault: a kernel that holds tensor memory waits on an mbarrier that nobody
arrives on, with a short poll bound.  It must give up, raise DS41_E_TIMEOUT in
the device status word, free its tensor memory and return; the device stays
usable, and a step run afterwards still matches the oracle."""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_window_gb300 import ds41
from compressed_sparse_attention_window_gb300.workloads import TINY_PREFILL, bf16_bits, make_inputs
from helpers import assert_idx_sets_equal, attn_close, oracle_forward, to_dev

pytestmark = pytest.mark.gpu

DS41_E_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ds41.load()


def test_wait_that_nobody_completes_gives_up(orc):
    assert ds41.device_status(reset=True) == 0
    res = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    ds41.selftest_wait_timeout(1000, False, res)
    torch.cuda.synchronize()  # the kernel returned
    done, abort_seen = res[:2].tolist()
    assert done == 0 and abort_seen == 1
    assert ds41.device_status(reset=True) == DS41_E_TIMEOUT
    assert ds41.device_status(reset=True) == 0
    # the same wait completes when its arrival comes
    ds41.selftest_wait_timeout(1000, True, res)
    torch.cuda.synchronize()
    assert res[:2].tolist() == [1, 0]
    assert ds41.device_status(reset=True) == 0
    # the device is still usable: a whole step, against the oracle
    wl = TINY_PREFILL
    inp = make_inputs(wl, seed=11)
    dev = to_dev(inp)
    ora_fc = orc.yarn_freqs_cis(wl.rd, wl.max_pos)
    out = ds41.csa_forward(dev, wl, torch.from_numpy(ora_fc).cuda())
    torch.cuda.synchronize()
    ref = oracle_forward(orc, wl, inp, fc=ora_fc)
    assert np.array_equal(bf16_bits(dev["ring"]), ref["ring"])
    assert_idx_sets_equal(out["idx"].cpu().numpy(), ref["idx"], wl.win)
    assert attn_close(out["o"].float().cpu().numpy(), ref["o"])[0]
    assert ds41.device_status(reset=True) == 0


def test_wait_timeout_checks_its_arguments():
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(ds41.DS41Error):
        ds41.selftest_wait_timeout(0, False, res)
    with pytest.raises(ds41.DS41Error):
        ds41.selftest_wait_timeout(1 << 23, False, res)
