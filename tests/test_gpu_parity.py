"""GPU parity: libgdr (through its C ABI) against the fp64 oracle.

Covers both execution paths on small ragged inputs (several chunks, partial
last chunks, grouped heads, initial/final states), every stage's
intermediates against the chunkwise form, the device chunk enumeration (exact),
ghost segments (bit-exact, "Findings from integrating FlashQLA's Blackwell GDN
kernels into a JAX trainer", section 2: up to 120 appended ghosts), the
fresh-cu_seqlens loop of section 1, run-to-run bit identity, host buffers,
empty inputs, and the five named workloads at full size on sampled heads.
"""
import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_gdr_gb300 import api
from chunked_gated_delta_gdr_gb300.inputs import WORKLOADS, make_named, make_workload
from gdr_testlib import (assert_ht_close, assert_o_close, chunk_enumeration, covered_tokens,
                         oracle_heads, run_gpu)

pytestmark = pytest.mark.gpu

PATHS = ["staged", "fused"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_gated_delta_gdr_gb300 import build
    build.build()
    cap = torch.cuda.get_device_capability()
    if cap != (10, 3):
        pytest.skip(f"needs sm_103 (GB300), found {cap}")


def _fused_ok():
    w = make_workload("probe", 1, [64], 1, 1, 64)
    try:
        run_gpu(w, path="fused")
        return True
    except api.nat.GdrError as e:
        if e.status == -9:
            return False
        raise


def _skip_unsupported(path):
    if path == "fused" and not _fused_ok():
        pytest.skip("fused path not available for this build")


SMALL = [
    ("d64_ragged_gqa", 11, [1, 63, 64, 65, 200, 0, 130], 2, 4, 64, True),
    ("d128_ragged", 12, [150, 0, 0, 64, 257, 3], 2, 2, 128, True),
    ("d128_gqa_noh0", 13, [129, 500, 7], 1, 4, 128, False),
    ("d64_many_short", 14, [5, 17, 0, 33, 1, 2, 64, 0, 63, 90], 4, 4, 64, True),
]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_against_oracle(case, path):
    _skip_unsupported(path)
    name, seed, lens, Hk, H, D, with_h0 = case
    w = make_workload(name, seed, lens, Hk, H, D, with_h0=with_h0, want_ht=True)
    o, ht = run_gpu(w, path)
    o_ref, ht_ref = oracle_heads(w, range(w.H))
    mask = covered_tokens(w.cu_seqlens, w.T)
    assert_o_close(o, o_ref, mask)
    assert_ht_close(ht, ht_ref)


@pytest.mark.parametrize("path", PATHS)
def test_tiny_workload(path):
    _skip_unsupported(path)
    w = make_named("tiny")
    o, ht = run_gpu(w, path)
    o_ref, ht_ref = oracle_heads(w, range(w.H))
    assert_o_close(o, o_ref, covered_tokens(w.cu_seqlens, w.T))
    assert_ht_close(ht, ht_ref)


def test_stage_intermediates_against_chunked_form():
    w = make_workload("stages", 21, [100, 0, 64, 37], 2, 4, 64, with_h0=True)
    wd = w.to("cuda")
    wgt, u, gc = api.chunk_prep(wd.k, wd.v, wd.g, wd.beta, wd.cu_seqlens)
    h, vn, ht = api.state_scan(wd.k, wgt, u, gc, wd.h0, wd.cu_seqlens, True)
    o = api.chunk_out(wd.q, wd.k, vn, h, gc, w.scale, wd.cu_seqlens)
    o_ref, ht_ref, inter = oracle.chunked_wy(w.q, w.k, w.v, w.g, w.beta, w.scale, w.h0,
                                             w.cu_seqlens, intermediates=True)
    segs, chunks = chunk_enumeration(w.cu_seqlens, w.T)
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    W, U, G, Hh, VN = f(wgt), f(u), f(gc), f(h), f(vn)
    for cid, (n, s, ln, _) in enumerate(chunks):
        for hh in range(w.H):
            ref = inter[(n, hh, s)]
            np.testing.assert_allclose(G[s:s + ln, hh], ref["G"], rtol=1e-5, atol=1e-5)
            for got, key in ((W[s:s + ln, hh], "W"), (U[s:s + ln, hh], "U"),
                             (Hh[cid, hh], "h"), (VN[s:s + ln, hh], "v_new")):
                scale = max(np.abs(ref[key]).max(), 1e-6)
                err = np.abs(got - ref[key]).max() / scale
                assert err < 2e-2, (key, cid, hh, err)
    assert_o_close(o, o_ref, covered_tokens(w.cu_seqlens, w.T))
    assert_ht_close(ht, ht_ref)


def test_chunk_index_exact():
    g = torch.Generator().manual_seed(5)
    cases = [[0], [0, 0, 0], [0, 64], [0, 1, 65, 65, 129, 300], [0, 100, 50, 400, 9999],
             [5, 70, -3, 200], list(range(0, 64 * 40, 37))]
    for _ in range(20):
        lens = torch.randint(0, 300, (int(torch.randint(1, 3000, (1,), generator=g)),),
                             generator=g)
        lens[torch.rand(lens.shape, generator=g) < 0.3] = 0
        cases.append([0] + torch.cumsum(lens, 0).tolist())
    for cu in cases:
        T = max(max(cu), 0) if len(cu) > 1 else 10
        T = min(T, 5000) if cu[-1] == 9999 else T
        cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
        seg, chunks, n = api.chunk_index(cu_d, T)
        segs_ref, chunks_ref = chunk_enumeration(cu, T)
        assert int(n.item()) == len(chunks_ref)
        assert seg.cpu().tolist() == [list(s) for s in segs_ref]
        got = chunks.cpu().tolist()[:len(chunks_ref)]
        assert got == [list(c) for c in chunks_ref]


def test_fresh_cu_seqlens_loop():
    """A new cu_seqlens every iteration, allocated at recycled addresses: the
    device chunk grid must always match the enumeration of the current array."""
    g = torch.Generator().manual_seed(7)
    for i in range(300):
        lens = torch.randint(1, 512, (8,), generator=g)
        cu = torch.cat([torch.zeros(1, dtype=torch.int32),
                        torch.cumsum(lens, 0).to(torch.int32)]).cuda()
        T = int(cu[-1])
        _, chunks, n = api.chunk_index(cu, T)
        _, ref = chunk_enumeration(cu.cpu(), T)
        assert int(n.item()) == len(ref), i
        assert chunks.cpu().tolist()[:len(ref)] == [list(c) for c in ref], i
        del cu, chunks, n


@pytest.mark.parametrize("path", PATHS)
def test_ghost_segments_bit_exact(path):
    _skip_unsupported(path)
    lens = [300, 64, 1, 129]
    w = make_workload("ghost", 31, lens, 2, 4, 128, with_h0=True)
    o, ht = run_gpu(w, path)
    for extra in (1, 16, 120):
        lens2 = lens + [0] * extra
        w2 = make_workload("ghost2", 31, lens2, 2, 4, 128, with_h0=False)
        h0 = torch.zeros(len(lens2), 4, 128, 128)
        h0[:len(lens)] = w.h0
        h0[len(lens):] = 0.5
        w2.q, w2.k, w2.v, w2.g, w2.beta, w2.h0 = w.q, w.k, w.v, w.g, w.beta, h0
        o2, ht2 = run_gpu(w2, path)
        assert torch.equal(o, o2), extra
        assert torch.equal(ht, ht2[:len(lens)]), extra
        assert torch.equal(ht2[len(lens):].cpu(), h0[len(lens):]), extra
    # ghosts interleaved between real segments
    lens3 = [0, 300, 0, 0, 64, 1, 0, 129, 0]
    w3 = make_workload("ghost3", 31, lens3, 2, 4, 128, with_h0=False)
    h0 = torch.zeros(len(lens3), 4, 128, 128)
    real = [1, 4, 5, 7]
    for i, n in enumerate(real):
        h0[n] = w.h0[i]
    w3.q, w3.k, w3.v, w3.g, w3.beta, w3.h0 = w.q, w.k, w.v, w.g, w.beta, h0
    o3, ht3 = run_gpu(w3, path)
    assert torch.equal(o, o3)
    for i, n in enumerate(real):
        assert torch.equal(ht[i], ht3[n])


@pytest.mark.parametrize("path", PATHS)
def test_run_to_run_bit_identity(path):
    _skip_unsupported(path)
    w = make_workload("det", 41, [700, 33, 0, 1000], 2, 4, 128, with_h0=True)
    o0, ht0 = run_gpu(w, path)
    for _ in range(10):
        o, ht = run_gpu(w, path)
        assert torch.equal(o, o0)
        assert torch.equal(ht, ht0)


def test_paths_agree():
    if not _fused_ok():
        pytest.skip("fused path not available for this build")
    w = make_workload("agree", 51, [333, 64, 0, 1029], 2, 4, 128, with_h0=True)
    oa, ha = run_gpu(w, "staged")
    ob, hb = run_gpu(w, "fused")
    assert (oa.float() - ob.float()).abs().max().item() <= 8e-3
    assert ((ha - hb).abs().max() / ha.abs().max()).item() <= 2e-2


def test_host_buffers_match_device():
    w = make_workload("host", 61, [200, 57], 2, 2, 64, with_h0=True)
    o_d, ht_d = run_gpu(w)
    pin = lambda t: None if t is None else t.pin_memory()
    o_h, ht_h = api.chunk_fwd(pin(w.q), pin(w.k), pin(w.v), pin(w.g), pin(w.beta),
                              scale=w.scale, initial_state=pin(w.h0),
                              cu_seqlens=w.cu_seqlens, output_final_state=True)
    assert o_h.device.type == "cpu"
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(ht_h, ht_d.cpu())


def test_alloc_entry_point_matches():
    w = make_workload("alloc", 62, [200, 0, 57], 2, 2, 64, with_h0=True)
    o_d, ht_d = run_gpu(w)
    wd = w.to("cuda")
    o2, ht2 = api.chunk_fwd_alloc(wd.q, wd.k, wd.v, wd.g, wd.beta, w.scale, wd.h0,
                                  wd.cu_seqlens, True)
    assert torch.equal(o2, o_d) and torch.equal(ht2, ht_d)


@pytest.mark.parametrize("path", PATHS)
def test_empty_and_uncovered(path):
    _skip_unsupported(path)
    # T = 0 with three ghost segments: ht = h0
    w = make_workload("empty", 71, [0, 0, 0], 1, 2, 64, with_h0=True)
    o, ht = run_gpu(w, path)
    assert o.numel() == 0
    assert torch.equal(ht.cpu(), w.h0)
    # n_seq = 0: nothing happens
    w0 = make_workload("none", 72, [], 1, 2, 64)
    o0, ht0 = run_gpu(w0, path)
    assert o0.numel() == 0 and ht0.numel() == 0
    # tokens outside every segment keep their previous contents
    w = make_workload("uncov", 73, [100, 40], 1, 2, 64)
    wd = w.to("cuda")
    cu = torch.tensor([0, 60, 60, 100], dtype=torch.int32, device="cuda")
    out = torch.full((w.T, 2, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    api.chunk_fwd(wd.q, wd.k, wd.v, wd.g, wd.beta, scale=w.scale, cu_seqlens=cu, out=out,
                  path=path)
    assert (out[100:] == 7.0).all()
    assert not (out[:100] == 7.0).all()


def test_check_cu_seqlens():
    cu = torch.tensor([0, 10, 5, 20, 30], dtype=torch.int32, device="cuda")
    assert api.check_cu_seqlens(cu, 25) == (2, 2)
    cu = torch.tensor([0, 10, 20], dtype=torch.int32, device="cuda")
    assert api.check_cu_seqlens(cu, 25) == (0, -1)


# ---------------------------------------------------------------- full-size workloads

SAMPLED_HEADS = {"tiny": None, "fixed_b4_t4096_h16": [0, 9, 15],
                 "packed_64k_h32": [0, 13, 31], "long_t20468_h32": [3, 30],
                 "gqa_packed_128k_h16x32": [0, 1, 17, 30]}


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name", WORKLOADS)
def test_named_workload_full_size(name, path):
    _skip_unsupported(path)
    w = make_named(name)
    o, ht = run_gpu(w, path)
    heads = SAMPLED_HEADS[name] or list(range(w.H))
    o_ref, ht_ref = oracle_heads(w, heads)
    mask = covered_tokens(w.cu_seqlens, w.T)
    assert_o_close(o[:, heads], o_ref, mask)
    if w.want_ht:
        assert_ht_close(ht[:, heads], ht_ref)
    assert api.device_status() == 0, "a bounded wait ran out"


def test_unaligned_inputs_take_the_staged_element_loads():
    # q, k, v at an odd element offset (rows not 16-byte aligned): the fused path cannot
    # take them, AUTO runs the staged kernels with element loads, and the result is
    # bit-identical to the staged path's vector loads on aligned copies (and the fused
    # path refuses such inputs)
    w = make_workload("unaligned", 81, [150, 0, 77], 2, 4, 64, with_h0=True)
    wd = w.to("cuda")

    def shifted(t):
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
        view = buf[1:].view(t.shape)
        view.copy_(t)
        return view

    q, k, v = shifted(wd.q), shifted(wd.k), shifted(wd.v)
    assert q.data_ptr() % 16 != 0
    kw = dict(scale=w.scale, initial_state=wd.h0, cu_seqlens=wd.cu_seqlens,
              output_final_state=True)
    o1, ht1 = api.chunk_fwd(q, k, v, wd.g, wd.beta, path="auto", **kw)
    o2, ht2 = api.chunk_fwd(wd.q, wd.k, wd.v, wd.g, wd.beta, path="staged", **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(ht1, ht2)
    with pytest.raises(api.nat.GdrError):
        api.chunk_fwd(q, k, v, wd.g, wd.beta, path="fused", **kw)


@pytest.mark.parametrize("parts", [2, 3, 4])
def test_pipelined_host_forward_matches_device(parts):
    # host tensors cut into runs of whole segments, one stream each (copy in, forward,
    # copy out): bit-identical to one device call, ht included
    lens = [700, 0, 1300, 64, 1, 900, 0, 2048, 333, 1000, 0]
    w = make_workload("pipelined", 77, lens, 4, 8, 64, with_h0=True)
    assert api.split_pieces(w.T, w.n_seq, w.H) == 1
    o_d, ht_d = run_gpu(w)
    pin = lambda t: None if t is None else t.pin_memory()
    o_h, ht_h = api._chunk_fwd_host_pipelined(pin(w.q), pin(w.k), pin(w.v), pin(w.g),
                                              pin(w.beta), w.scale, pin(w.h0), w.cu_seqlens,
                                              True, "auto", None, None, parts=parts,
                                              min_tokens=0)
    mask = torch.from_numpy(covered_tokens(w.cu_seqlens, w.T))
    assert torch.equal(o_h[mask], o_d.cpu()[mask]) and torch.equal(ht_h, ht_d.cpu())


@pytest.mark.parametrize("path", ["fused", "staged"])
def test_gate_rows_with_a_padded_token_stride(path):
    # g and beta as views whose rows are H + 1 elements apart (the innermost stride is 1,
    # as the boundary requires): the same values as contiguous tensors, so the outputs
    # must be bit-identical, and they match the oracle
    _skip_unsupported(path)
    w = make_workload("gate_vec", 83, [300, 0, 77, 1], 2, 8, 64, with_h0=True)
    wd = w.to("cuda")
    kw = dict(scale=w.scale, initial_state=wd.h0, cu_seqlens=wd.cu_seqlens,
              output_final_state=True, path=path)
    o1, ht1 = api.chunk_fwd(wd.q, wd.k, wd.v, wd.g, wd.beta, **kw)
    g2 = torch.zeros(w.T, w.H + 1, dtype=torch.float32, device="cuda")[:, :w.H]
    b2 = torch.zeros(w.T, w.H + 1, dtype=torch.bfloat16, device="cuda")[:, :w.H]
    g2.copy_(wd.g)
    b2.copy_(wd.beta)
    assert g2.stride(0) == w.H + 1 and b2.stride(0) == w.H + 1
    o2, ht2 = api.chunk_fwd(wd.q, wd.k, wd.v, g2, b2, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(ht1, ht2)
    o_ref, ht_ref = oracle_heads(w, range(w.H))
    assert_o_close(o1, o_ref, covered_tokens(w.cu_seqlens, w.T))
    assert_ht_close(ht1, ht_ref)
