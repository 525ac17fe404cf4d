"""GPU parity of the fused path's sequence split against the fp64 oracle.

When the (segment, head) pairs are too few to fill the GPU, GDR_PATH_FUSED cuts long
segments into pieces that run on different SMs and joins them through the affine state
map of each piece, S_out = M S_in + R (FlashQLA splits one sequence over CTAs with
`seq_split_idx`, "Findings from integrating FlashQLA's sm_100 GDN kernels ...",
section 2; the context-parallel final_correction of "feat(cake_kda): add paired
recurrent training for SM100a and SM103a" joins pieces the same way).  The pieces change
only where the state is rounded, so o and ht meet the same tolerances as the unsplit
path, and the result stays bit-identical from run to run.
"""
import pytest
import torch

from chunked_gated_delta_gdr_gb300 import api
from chunked_gated_delta_gdr_gb300.inputs import make_named, make_workload
from gdr_testlib import assert_ht_close, assert_o_close, covered_tokens, oracle_heads, run_gpu

pytestmark = pytest.mark.gpu

# lengths (zeros allowed), Hk, H, d, with h0
CASES = {
    # one segment of 141 chunks: 8 pieces of 17-18 chunks, ragged tail
    "one_long_d128_h0": ([9000], 2, 4, 128, True),
    # 79 chunks -> 4 pieces, 11 and 33 -> whole, a 1-token segment, an empty one
    "mixed_d64_h0": ([5000, 0, 700, 2100, 1], 1, 2, 64, True),
    # 48 full chunks -> 3 pieces of 16, zero initial state
    "exact_d128": ([64 * 48], 1, 2, 128, False),
    # 32 heads: the first piece weighs two of the others (94 chunks -> 37, 19, 19, 19)
    "lead2_h32_d64": ([6000], 8, 32, 64, True),
}


def _workload(case):
    lens, Hk, H, d, h0 = CASES[case]
    return make_workload(case, 29, lens, Hk, H, d, with_h0=h0)


@pytest.mark.parametrize("case", sorted(CASES))
def test_split_against_oracle(case):
    w = _workload(case)
    assert api.split_pieces(w.T, w.n_seq, w.H) > 1, "the case must exercise the split"
    o, ht = run_gpu(w, path="fused")
    torch.cuda.synchronize()
    o_ref, ht_ref = oracle_heads(w, range(w.H))
    assert_o_close(o, o_ref, covered_tokens(w.cu_seqlens, w.T))
    assert_ht_close(ht, ht_ref)


@pytest.mark.parametrize("case", sorted(CASES))
def test_split_deterministic_and_close_to_whole(case):
    w = _workload(case)
    o1, ht1 = run_gpu(w, path="fused")
    o2, ht2 = run_gpu(w, path="fused")
    ow, htw = run_gpu(w, path="fused_whole")
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(ht1, ht2)
    mask = torch.from_numpy(covered_tokens(w.cu_seqlens, w.T)).to(o1.device)
    assert (o1[mask].float() - ow[mask].float()).abs().max().item() <= 4e-3
    scale = htw.abs().max().item()
    assert (ht1 - htw).abs().max().item() <= 1e-2 * scale


def test_split_workspace_covers_the_pieces():
    w = _workload("one_long_d128_h0")
    whole = api.workspace_bytes(w.T, w.n_seq, w.H, w.dk, w.dv, "fused_whole")
    split = api.workspace_bytes(w.T, w.n_seq, w.H, w.dk, w.dv, "fused")
    P = api.split_pieces(w.T, w.n_seq, w.H)
    # initial states, R and M of every piece: 3 x P x n_seq x H states of d x d fp32
    assert split - whole >= 3 * P * w.n_seq * w.H * w.dk * w.dv * 4


@pytest.mark.slow
def test_split_full_size_long_sequence():
    # the single 20468-token segment at H = 32, d = 128 with h0: value heads 0 and 31
    w = make_named("long_t20468_h32")
    assert api.split_pieces(w.T, w.n_seq, w.H) > 1
    o, ht = run_gpu(w, path="fused")
    torch.cuda.synchronize()
    heads = [0, 31]
    o_ref, ht_ref = oracle_heads(w, heads, n_threads=2)
    assert_o_close(o[:, heads], o_ref, covered_tokens(w.cu_seqlens, w.T))
    assert_ht_close(ht[:, heads], ht_ref)
