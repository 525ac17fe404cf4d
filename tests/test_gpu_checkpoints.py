"""GPU parity of the state checkpoints (``gdr_chunk_fwd_ckpt``) against the fp64 oracle.

Checkpoint m of segment n is the state after the segment's first m * N tokens (N the
checkpoint interval); the FlashInfer KDA prefill keeps such checkpoints for prefix caching
("feat(cake_kda): add paired recurrent training for SM100a and SM103a", kept inference
surface).  Checkpoints are compared with the state tolerance (max |delta| / max |ref|), the
offsets exactly, and o and ht must be bit-identical to a plain forward on the same path.
"""
import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_gdr_gb300 import api
from chunked_gated_delta_gdr_gb300.inputs import make_named, make_workload
from gdr_testlib import assert_ht_close, assert_o_close, covered_tokens, run_gpu

pytestmark = pytest.mark.gpu


def _oracle_ckpt(w, heads, every):
    group = w.H // w.Hk
    hk = [h // group for h in heads]
    sel = lambda t, idx: t[:, idx].contiguous()
    h0 = None if w.h0 is None else w.h0[:, heads].contiguous()
    return oracle.recurrent_checkpoints(sel(w.q, hk), sel(w.k, hk), sel(w.v, heads),
                                        sel(w.g, heads), sel(w.beta, heads), w.scale, h0,
                                        w.cu_seqlens, every)


def _run_ckpt(w, every, path):
    wd = w.to("cuda")
    out = api.chunk_fwd_checkpoints(wd.q, wd.k, wd.v, wd.g, wd.beta, every, scale=w.scale,
                                    initial_state=wd.h0, cu_seqlens=wd.cu_seqlens,
                                    output_final_state=True, path=path)
    torch.cuda.synchronize()
    return out


# lengths (zeros allowed), Hk, H, d, interval
CASES = {
    "d64_ragged_every64": ([150, 0, 128, 200, 64, 5, 256], 2, 4, 64, 64),
    "d128_every128": ([700, 0, 129, 512, 1], 2, 4, 128, 128),
    "d128_every192_gqa": ([1000, 383, 384], 1, 4, 128, 192),
}


@pytest.mark.parametrize("path", ["staged", "fused"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_checkpoints_against_oracle(case, path):
    lens, Hk, H, d, every = CASES[case]
    w = make_workload(case, 17, lens, Hk, H, d, with_h0=True)
    o, ht, ck, starts = _run_ckpt(w, every, path)
    o_ref, ht_ref, ck_ref, off_ref = _oracle_ckpt(w, range(H), every)
    assert starts.cpu().numpy().tolist() == off_ref.tolist()
    n = int(off_ref[-1])
    assert ck.shape[0] >= n
    assert_ht_close(ck[:n], ck_ref)
    assert_o_close(o, o_ref, covered_tokens(w.cu_seqlens, w.T))
    assert_ht_close(ht, ht_ref)
    # the checkpoints add reads only: o and ht are those of the plain forward
    o2, ht2 = run_gpu(w, path=path)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(ht, ht2)


def test_no_checkpoint_rows_for_short_segments():
    w = make_workload("short", 5, [63, 0, 1], 1, 2, 64, with_h0=True)
    o, ht, ck, starts = _run_ckpt(w, 64, "fused")
    assert starts.cpu().tolist() == [0, 0, 0, 0]
    assert ck.shape[0] == 1  # floor(64 / 64) rows allocated, none written


@pytest.mark.slow
def test_checkpoints_full_size_long_sequence():
    # the single 20468-token segment at H = 32, d = 128 with h0: checkpoints every 4096
    # tokens (4 of them), value heads 0 and 31 against the oracle
    w = make_named("long_t20468_h32")
    o, ht, ck, starts = _run_ckpt(w, 4096, "fused")
    heads = [0, 31]
    _, ht_ref, ck_ref, off_ref = _oracle_ckpt(w, heads, 4096)
    assert starts.cpu().tolist() == off_ref.tolist() == [0, 4]
    assert_ht_close(ck[:4, heads], ck_ref)
    assert_ht_close(ht[:, heads], ht_ref)
