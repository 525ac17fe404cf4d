"""The bench's algorithmic counts (the numerators of its roofline fractions), on the CPU,
against the per-workload figures worked out by hand when the measurement was planned:
bytes = T (4 d Hk + 4 d H + 6 H) + N H d^2 4 (h0 + ht) and FLOPs = 2 (5 c^2 d + 3 c d^2)
per chunk of c tokens and value head."""
import pytest

import bench
from chunked_gated_delta_gdr_gb300.inputs import make_named

# name: (bytes, relative precision of the stated figure, FLOPs, its precision)
STATED = {
    "tiny": (297_984, 0, 3.36e7, 5e-3),
    "fixed_b4_t4096_h16": (274.2e6, 5e-4, 4.72e10, 5e-3),
    "packed_64k_h32": (2.160e9, 5e-4, 3.78e11, 5e-3),
    "long_t20468_h32": (678.8e6, 5e-4, 1.18e11, 5e-3),
}


@pytest.mark.parametrize("name", sorted(STATED))
def test_counts_match_the_stated_figures(name):
    w = make_named(name)
    b, bp, f, fp = STATED[name]
    assert bench.algorithmic_bytes(w) == pytest.approx(b, rel=bp, abs=0)
    assert bench.algorithmic_flops(w) == pytest.approx(f, rel=fp)


def test_grouped_heads_workload_with_states():
    # 3.246 GB of tensors plus 4.19 MB of h0 and ht per segment (16 key heads, 32 value
    # heads, d = 128)
    w = make_named("gqa_packed_128k_h16x32")
    assert bench.algorithmic_bytes(w) == pytest.approx(3.246e9 + w.n_seq * 4.194e6, rel=5e-4)
    assert bench.algorithmic_flops(w) == pytest.approx(7.56e11, rel=5e-3)


def test_partial_chunks_count_their_own_length():
    # a 65-token segment is one full chunk and one chunk of a single token
    w = make_named("tiny")
    d = w.dk
    per_head = lambda c: 2 * (5 * c * c * d + 3 * c * d * d)
    assert bench.algorithmic_flops(w) == w.H * 4 * per_head(64)  # 256 tokens
    w.cu_seqlens[-1] = 65
    assert bench.algorithmic_flops(w) == w.H * (per_head(64) + per_head(1))
