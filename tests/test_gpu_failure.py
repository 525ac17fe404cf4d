"""Failure detection without a GPU fault: every wait inside the fused kernel is
bounded in time and reports through a device status word instead of hanging.
The self-test kernel waits on an mbarrier that nothing ever arrives on; the
wait must run out, set the status and return, and the context must stay usable.
"""
import pytest
import torch

from chunked_gated_delta_gdr_gb300 import api
from chunked_gated_delta_gdr_gb300.inputs import make_workload
from gdr_testlib import assert_ht_close, assert_o_close, covered_tokens, oracle_heads, run_gpu

pytestmark = pytest.mark.gpu

WAIT_SELFTEST = 0x7001


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_gdr_gb300 import build
    build.build()
    if torch.cuda.get_device_capability() != (10, 3):
        pytest.skip("needs sm_103 (GB300)")


def test_bounded_wait_runs_out_and_reports():
    api.clear_device_status()
    assert api.device_status() == 0
    api.wait_selftest(2000)
    assert api.device_status() == WAIT_SELFTEST
    api.clear_device_status()
    assert api.device_status() == 0
    # the context is still healthy: a forward runs and matches the oracle
    w = make_workload("after_timeout", 81, [200, 0, 77], 2, 4, 128, with_h0=True)
    o, ht = run_gpu(w, "fused")
    o_ref, ht_ref = oracle_heads(w, range(w.H))
    assert_o_close(o, o_ref, covered_tokens(w.cu_seqlens, w.T))
    assert_ht_close(ht, ht_ref)
    assert api.device_status() == 0


def test_wait_selftest_rejects_bad_limits():
    with pytest.raises(api.nat.GdrError):
        api.wait_selftest(0)
    with pytest.raises(api.nat.GdrError):
        api.wait_selftest(2_000_000)
