"""gdr_chunk_out_noalloc: the output stage for callers that cannot allocate
device memory (engines with a fixed memory plan, custom-call hosts that own
every buffer).  Its chunk tables live in a static device array inside libgdr
instead of a caller workspace.  This file is collected last on purpose: if it
fails, a run that stops at the first failure has already run everything else.
"""
import ctypes

import pytest
import torch

from chunked_gated_delta_gdr_gb300 import _native as nat
from chunked_gated_delta_gdr_gb300 import api
from chunked_gated_delta_gdr_gb300.inputs import make_workload
from gdr_testlib import O_ATOL, O_COS, assert_o_close, covered_tokens, oracle_heads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_gdr_gb300 import build
    build.build()
    if torch.cuda.get_device_capability() != (10, 3):
        pytest.skip("needs sm_103 (GB300)")


def _stage_inputs(w):
    wd = w.to("cuda")
    wgt, u, gc = api.chunk_prep(wd.k, wd.v, wd.g, wd.beta, wd.cu_seqlens)
    h, vn, _ = api.state_scan(wd.k, wgt, u, gc, wd.h0, wd.cu_seqlens, False)
    return wd, h, vn, gc


def _close(a, b):
    a, b = a.float(), b.float()
    err = (a - b).abs().max().item()
    cos = (a * b).sum().item() / max((a.norm() * b.norm()).item(), 1e-30)
    assert err <= O_ATOL, err
    assert cos >= O_COS, cos


def test_noalloc_matches_workspace_entry_point_twice():
    cases = [make_workload("na1", 301, [130, 0, 64, 7], 2, 4, 128, with_h0=True),
             make_workload("na2", 302, [1, 200, 0, 0, 65], 1, 2, 64, with_h0=False)]
    for w in cases:  # two calls in a row, different shapes: no state kept between calls
        wd, h, vn, gc = _stage_inputs(w)
        ref = api.chunk_out(wd.q, wd.k, vn, h, gc, w.scale, wd.cu_seqlens)
        got = api.chunk_out_noalloc(wd.q, wd.k, vn, h, gc, w.scale, wd.cu_seqlens)
        torch.cuda.synchronize()
        _close(got, ref)
        # and directly against the fp64 token recurrence, so that a fault shared by both
        # output-stage entry points cannot hide behind their agreement
        o_ref, _ = oracle_heads(w, range(w.H), want_ht=False)
        assert_o_close(got, o_ref, covered_tokens(w.cu_seqlens, w.T))
    # and the same problem twice more in a row on the shared static array
    w = cases[0]
    wd, h, vn, gc = _stage_inputs(w)
    ref = api.chunk_out(wd.q, wd.k, vn, h, gc, w.scale, wd.cu_seqlens)
    for _ in range(2):
        got = api.chunk_out_noalloc(wd.q, wd.k, vn, h, gc, w.scale, wd.cu_seqlens)
        _close(got, ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = nat.lib()
    buf = torch.zeros(1024, dtype=torch.int32, device="cuda")  # never read: the call must fail first
    T, H, D, n_seq = 1 << 28, 1, 64, 1
    cap = lib.gdr_chunk_count_bound(T, n_seq)
    keep = []

    def desc(shape, dtype):
        shp = (ctypes.c_int64 * 4)(*(list(shape) + [0] * (4 - len(shape))))
        d = nat.GdrTensor(ctypes.c_void_p(buf.data_ptr()), dtype, len(shape), shp, None)
        keep.append(d)
        return ctypes.byref(d)

    rc = lib.gdr_chunk_out_noalloc(desc([T, 1, D], nat.GDR_BF16), desc([T, 1, D], nat.GDR_BF16),
                                   desc([T, H, D], nat.GDR_BF16), desc([cap, H, D, D], nat.GDR_BF16),
                                   desc([T, H], nat.GDR_F32), ctypes.c_float(1.0),
                                   ctypes.c_void_p(buf.data_ptr()), n_seq,
                                   desc([T, H, D], nat.GDR_BF16), None)
    assert rc == -13
    assert "static scratch" in lib.gdr_status_string(rc).decode()
