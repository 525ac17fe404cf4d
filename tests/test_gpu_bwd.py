"""GPU parity of the backward (``gdr_chunk_bwd``) against the fp64 oracle's backward.

The pages describe FlashQLA's GDN kernels as a training backend with a bit-reproducible
backward that tolerates length-0 segments ("Findings from integrating FlashQLA's
Blackwell GDN kernels into a JAX trainer", intro and section 2), and state no gradient
tolerance.  The tolerance here follows from the arithmetic: the backward recomputes the
forward's chunk states S_0, V', W and U rounded to bf16 as the forward stores them,
and each gradient is a chain of a few products of such operands (about five roundings
of 2^-9 relative each) with fp32 accumulation, so every gradient tensor is compared by
max |delta| / max |ref| <= 2e-2 (about 2x that bound) and cosine >= 0.9995 over covered
tokens.  dh0 uses the same bound.  Results must be bit-identical from run to run.
"""
import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_gdr_gb300 import api
from chunked_gated_delta_gdr_gb300.inputs import make_named, make_workload
from gdr_testlib import covered_tokens

pytestmark = pytest.mark.gpu

REL = 2e-2
COS = 0.9995

# lengths (zeros allowed), Hk, H, d, with h0 and dht
CASES = {
    "d64_ragged_gqa": ([150, 0, 64, 1, 200], 2, 4, 64, True),
    "d128_h0": ([300, 129], 1, 2, 128, True),
    "d128_no_state": ([256], 2, 2, 128, False),
}


def _upstream(w, seed, with_dht):
    gen = torch.Generator().manual_seed(seed)
    do = (0.1 * torch.randn(w.T, w.H, w.dv, generator=gen)).to(torch.bfloat16)
    dht = (0.1 * torch.randn(w.n_seq, w.H, w.dk, w.dv, generator=gen)) if with_dht else None
    return do, dht


def _run_bwd(w, do, dht):
    wd = w.to("cuda")
    out = api.chunk_bwd(wd.q, wd.k, wd.v, wd.g, wd.beta, do.cuda(), scale=w.scale,
                        initial_state=wd.h0, cu_seqlens=wd.cu_seqlens,
                        dht=None if dht is None else dht.cuda(), want_dh0=True)
    torch.cuda.synchronize()
    return out


def _oracle_bwd(w, do, dht, heads=None):
    if heads is None:
        return oracle.recurrent_bwd(w.q, w.k, w.v, w.g, w.beta, w.scale, w.h0, w.cu_seqlens, do,
                                    dht)
    # a subset of value heads (whole query/key groups)
    group = w.H // w.Hk
    hk = sorted({h // group for h in heads})
    hv = [hh for g_ in hk for hh in range(g_ * group, (g_ + 1) * group)]
    sel = lambda t, idx: t[:, idx].contiguous()
    h0 = None if w.h0 is None else w.h0[:, hv].contiguous()
    return oracle.recurrent_bwd(sel(w.q, hk), sel(w.k, hk), sel(w.v, hv), sel(w.g, hv),
                                sel(w.beta, hv), w.scale, h0, w.cu_seqlens, sel(do, hv),
                                None if dht is None else dht[:, hv].contiguous()), hk, hv


def _close(name, got, ref, mask=None):
    a = got.float().cpu().numpy().astype(np.float64)
    b = np.asarray(ref, dtype=np.float64)
    if mask is not None:
        a, b = a[mask], b[mask]
    scale = max(float(np.abs(b).max()), 1e-30)
    rel = float(np.abs(a - b).max()) / scale
    cos = float((a * b).sum() / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))
    assert rel <= REL, f"{name}: max|delta|/max|ref| {rel:.3e} > {REL}"
    assert cos >= COS, f"{name}: cosine {cos:.6f} < {COS}"
    return rel, cos


NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_against_oracle(case):
    lens, Hk, H, d, state = CASES[case]
    w = make_workload(case, 23, lens, Hk, H, d, with_h0=state)
    do, dht = _upstream(w, 24, state)
    got = _run_bwd(w, do, dht)
    ref = oracle.recurrent_bwd(w.q, w.k, w.v, w.g, w.beta, w.scale, w.h0, w.cu_seqlens, do, dht)
    mask = covered_tokens(w.cu_seqlens, w.T)
    for name, a, b in zip(NAMES, got, ref):
        _close(name, a, b, None if name == "dh0" else mask)
    # tokens outside every segment: none here; empty segments hand dht back as dh0
    for n, (s, e) in enumerate(zip(w.cu_seqlens[:-1].tolist(), w.cu_seqlens[1:].tolist())):
        if s == e:
            want = torch.zeros_like(got[5][n]) if dht is None else dht[n].cuda()
            assert torch.equal(got[5][n], want)


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_bit_identical_run_to_run(case):
    lens, Hk, H, d, state = CASES[case]
    w = make_workload(case, 23, lens, Hk, H, d, with_h0=state)
    do, dht = _upstream(w, 24, state)
    a = _run_bwd(w, do, dht)
    b = _run_bwd(w, do, dht)
    for name, x, y in zip(NAMES, a, b):
        assert torch.equal(x, y), name


def test_backward_ghost_segments_change_nothing():
    # trailing length-0 segments (as a static-shape caller pads cu_seqlens) leave every
    # gradient of the real tokens bit-identical
    w = make_workload("ghosts", 31, [200, 77], 1, 2, 64, with_h0=True)
    do, dht = _upstream(w, 32, True)
    a = _run_bwd(w, do, dht)
    w2 = make_workload("ghosts", 31, [200, 77, 0, 0, 0], 1, 2, 64, with_h0=True)
    w2.q, w2.k, w2.v, w2.g, w2.beta = w.q, w.k, w.v, w.g, w.beta
    w2.h0 = torch.cat([w.h0, torch.randn(3, 2, 64, 64)])
    dht2 = torch.cat([dht, torch.randn(3, 2, 64, 64)])
    b = _run_bwd(w2, do, dht2)
    for name, x, y in zip(NAMES[:5], a[:5], b[:5]):
        assert torch.equal(x, y), name
    assert torch.equal(a[5], b[5][:2])
    assert torch.equal(b[5][2:], dht2[2:].cuda())


def test_autograd_wrapper_matches_chunk_bwd():
    w = make_workload("autograd", 41, [130, 70], 1, 2, 64, with_h0=True)
    do, dht = _upstream(w, 42, True)
    wd = w.to("cuda")
    leaves = [t.clone().requires_grad_(True) for t in (wd.q, wd.k, wd.v, wd.g, wd.beta, wd.h0)]
    o, ht = api.chunk_gated_delta_rule(*leaves[:5], scale=w.scale, initial_state=leaves[5],
                                       output_final_state=True, cu_seqlens=wd.cu_seqlens)
    ((o.float() * do.cuda().float()).sum() + (ht * dht.cuda()).sum()).backward()
    ref = _run_bwd(w, do, dht)
    for leaf, r, name in zip(leaves, ref, NAMES):
        assert torch.equal(leaf.grad, r.to(leaf.dtype)), name


@pytest.mark.slow
def test_backward_full_size_packed_sampled_heads():
    # the packed 64k-token workload (H = 32, d = 128, 16 trailing ghosts), value heads 0
    # and 31 against the oracle
    w = make_named("packed_64k_h32")
    do, dht = _upstream(w, 51, False)
    got = _run_bwd(w, do, dht)
    (ref, hk, hv) = _oracle_bwd(w, do, dht, heads=[0, 31])
    mask = covered_tokens(w.cu_seqlens, w.T)
    _close("dq", got[0][:, hk], ref[0], mask)
    _close("dk", got[1][:, hk], ref[1], mask)
    for name, i in (("dv", 2), ("dg", 3), ("dbeta", 4)):
        _close(name, got[i][:, hv], ref[i], mask)
    _close("dh0", got[5][:, hv], ref[5])


def test_backward_many_units_per_block():
    # more (segment, head) units than the GPU has SMs, so that every block of the fused
    # recompute crosses unit boundaries (where a unit's last W is read at the end of the
    # unit): no bounded wait may run out, and the gradients match the oracle
    rng = np.random.default_rng(7)
    lens = [int(x) for x in rng.integers(1, 260, size=160)] + [0, 0]
    w = make_workload("many_units", 81, lens, 1, 2, 64, with_h0=True)
    do, dht = _upstream(w, 82, True)
    api.clear_device_status()
    got = _run_bwd(w, do, dht)
    assert api.device_status() == 0
    ref = oracle.recurrent_bwd(w.q, w.k, w.v, w.g, w.beta, w.scale, w.h0, w.cu_seqlens, do, dht)
    mask = covered_tokens(w.cu_seqlens, w.T)
    for name, a, b in zip(NAMES, got, ref):
        _close(name, a, b, None if name == "dh0" else mask)


def test_backward_unaligned_views_take_the_scalar_loads():
    # q, k, v and dout as views whose rows are not 16-byte aligned (an odd element
    # offset into a larger buffer): the kernels fall back to element loads, and the
    # intra-chunk dV' step to its warp-tile kernel (the aligned call runs it on the tensor
    # cores with P in bf16), so the gradients agree with the aligned call within the
    # backward tolerance and with the oracle
    w = make_workload("unaligned", 61, [130, 0, 70], 1, 2, 64, with_h0=True)
    do, dht = _upstream(w, 62, True)
    ref = _run_bwd(w, do, dht)
    wd = w.to("cuda")

    def shifted(t):
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
        view = buf[1:].view(t.shape)
        view.copy_(t)
        return view

    q, k, v, dof = shifted(wd.q), shifted(wd.k), shifted(wd.v), shifted(do.cuda())
    assert q.data_ptr() % 16 != 0
    got = api.chunk_bwd(q, k, v, wd.g, wd.beta, dof, scale=w.scale, initial_state=wd.h0,
                        cu_seqlens=wd.cu_seqlens, dht=dht.cuda(), want_dh0=True)
    torch.cuda.synchronize()
    for name, a, b in zip(NAMES, got, ref):
        scale = max(b.abs().max().item(), 1e-30)
        assert (a - b).abs().max().item() <= REL * scale, name
    ref64 = oracle.recurrent_bwd(w.q, w.k, w.v, w.g, w.beta, w.scale, w.h0, w.cu_seqlens, do, dht)
    mask = covered_tokens(w.cu_seqlens, w.T)
    for name, a, b in zip(NAMES, got, ref64):
        _close(name, a, b, None if name == "dh0" else mask)


def test_backward_only_empty_segments():
    # every segment empty: no chunk runs, dh0 is dht, every other gradient is zero
    w = make_workload("empty", 71, [0, 0, 0], 1, 2, 64, with_h0=True)
    gen = torch.Generator().manual_seed(72)
    T = 8  # tokens that no segment covers
    q = torch.randn(T, 1, 64, generator=gen).to(torch.bfloat16).cuda()
    v = torch.randn(T, 2, 64, generator=gen).to(torch.bfloat16).cuda()
    g = -torch.rand(T, 2, generator=gen).cuda()
    beta = torch.rand(T, 2, generator=gen).to(torch.bfloat16).cuda()
    do = torch.randn(T, 2, 64, generator=gen).to(torch.bfloat16).cuda()
    dht = torch.randn(3, 2, 64, 64, generator=gen).cuda()
    cu = torch.tensor([0, 0, 0, 0], dtype=torch.int32, device="cuda")
    dq, dk, dv, dg, db, dh0 = api.chunk_bwd(q, q, v, g, beta, do, initial_state=w.h0.cuda(),
                                            cu_seqlens=cu, dht=dht, want_dh0=True)
    torch.cuda.synchronize()
    for t in (dq, dk, dv, dg, db):
        assert not t.any()
    assert torch.equal(dh0, dht)


def test_more_segments_than_a_grid_dimension_holds():
    # 70000 segments (a grid's y and z extents stop at 65535): a few real ones among
    # empty ones; both forward paths and the backward against the oracle
    lens = [0] * 70000
    for i, L in ((3, 90), (40000, 64), (69998, 7)):
        lens[i] = L
    w = make_workload("many_segments", 91, lens, 1, 2, 64, with_h0=False)
    o_ref, ht_ref = oracle.recurrent(w.q, w.k, w.v, w.g, w.beta, w.scale, None, w.cu_seqlens)
    wd = w.to("cuda")
    mask = covered_tokens(w.cu_seqlens, w.T)
    for path in ("staged", "fused"):
        o, ht = api.chunk_fwd(wd.q, wd.k, wd.v, wd.g, wd.beta, scale=w.scale,
                              cu_seqlens=wd.cu_seqlens, output_final_state=True, path=path)
        torch.cuda.synchronize()
        err = float(np.abs(o.float().cpu().numpy()[mask] - o_ref[mask]).max())
        assert err <= 4e-3, (path, err)
        rel = float(np.abs(ht.cpu().numpy() - ht_ref).max() / np.abs(ht_ref).max())
        assert rel <= 1e-2, (path, rel)
    do, dht = _upstream(w, 92, False)
    got = _run_bwd(w, do, dht)
    ref = oracle.recurrent_bwd(w.q, w.k, w.v, w.g, w.beta, w.scale, None, w.cu_seqlens, do, None)
    for name, a, b in zip(NAMES[:5], got[:5], ref[:5]):
        _close(name, a, b, mask)


@pytest.mark.parametrize("parts", [2, 4])
def test_pipelined_host_backward_matches_device(parts):
    # host tensors cut into runs of whole segments, one stream each: the gradients equal
    # one device call's bit for bit, and tokens outside every segment get zeros
    lens = [0, 500, 64, 0, 1200, 1, 700, 0]
    w = make_workload("pipelined_bwd", 95, lens, 2, 4, 64, with_h0=True)
    do, dht = _upstream(w, 96, True)
    ref = _run_bwd(w, do, dht)
    pin = lambda t: None if t is None else t.pin_memory()
    # a few uncovered tokens after the last segment
    extra = 5
    padt = lambda t: torch.cat([t, torch.zeros((extra,) + tuple(t.shape[1:]), dtype=t.dtype)])
    got = api._chunk_bwd_host_pipelined(
        pin(padt(w.q)), pin(padt(w.k)), pin(padt(w.v)), pin(padt(w.g)), pin(padt(w.beta)),
        pin(padt(do)), w.scale, pin(w.h0), w.cu_seqlens, pin(dht), True, None, parts=parts,
        min_tokens=0)
    for name, a, b in zip(NAMES, got, ref):
        if name == "dh0":
            assert torch.equal(a, b.cpu()), name
        else:
            assert torch.equal(a[:w.T], b.cpu()), name
            assert not a[w.T:].any(), name


def test_backward_strong_decays_stay_finite():
    """Decays of about e^-6 per token: within a chunk the cumulative gate spans several
    hundred, so e^{G_i - G_j} is only finite as a ratio with j < i, and a partial chunk's
    padded rows sit far above its real ones.  Every gradient must stay finite and match
    the oracle."""
    w = make_workload("strong_decay", 97, [150, 37, 64], 1, 2, 64, with_h0=True)
    gen = torch.Generator().manual_seed(98)
    w.g = -6.0 + 0.5 * torch.randn(w.T, w.H, generator=gen)
    do, dht = _upstream(w, 99, True)
    ref = oracle.recurrent_bwd(w.q, w.k, w.v, w.g, w.beta, w.scale, w.h0, w.cu_seqlens, do, dht)
    got = _run_bwd(w, do, dht)
    mask = covered_tokens(w.cu_seqlens, w.T)
    for name, a, b in zip(NAMES, got, ref):
        assert torch.isfinite(a).all(), name
        _close(name, a, b, None if name == "dh0" else mask)
