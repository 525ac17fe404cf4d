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


def test_traffic_record_from_an_ncu_log(tmp_path):
    # two captured launches of k_fused and one of another kernel, in the CSV layout of
    # `ncu --csv --log-file`; the record averages the fused launches, stamps the sha256
    # of the kernel sources computed here, and scales by algorithmic bytes
    hdr = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
           '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
           '"Metric Value"')

    def row(i, kern, metric, unit, val):
        return (f'"{i}","1","python3","h","{kern}","1","7","(352, 1, 1)","(152, 1, 1)","0",'
                f'"10.3","Command line profiler metrics","{metric}","{unit}","{val}"')

    fused = "void unnamed>::k_fused<0>(CUtensorMap_st, unnamed>::Params)"
    lines = ["==PROF== Connected", hdr,
             row(0, fused, "dram__bytes_read.sum", "byte", "400"),
             row(0, fused, "dram__bytes_write.sum", "byte", "100"),
             row(1, "k_worklist", "dram__bytes_read.sum", "byte", "7"),
             row(2, fused, "dram__bytes_read.sum", "Kbyte", "0.6"),
             row(2, fused, "dram__bytes_write.sum", "byte", "100")]
    csv_path = tmp_path / "log.csv"
    csv_path.write_text("\n".join(lines) + "\n")
    out = tmp_path / "rec.json"
    assert bench.record_traffic(str(csv_path), "packed_16k_h32", str(out), "cmd") == 0
    import json
    rec = json.loads(out.read_text())
    assert rec["launches"] == 2
    assert rec["dram_bytes_per_launch"] == pytest.approx((400 + 100 + 600 + 100) / 2)
    assert rec["source_sha256"] == bench.kernel_sha()
    f = rec["scaled"]["packed_64k_h32"]["factor"]
    assert f == pytest.approx(bench.algorithmic_bytes(make_named("packed_64k_h32")) /
                              bench.algorithmic_bytes(make_named("packed_16k_h32")))
    # the bench reads it only while the sources hash the same
    bench_rec, bench.TRAFFIC_RECORD = bench.TRAFFIC_RECORD, str(out)
    try:
        assert bench.read_traffic(bench.kernel_sha(), "packed_64k_h32") == pytest.approx(600 * f)
        assert bench.read_traffic("0" * 16, "packed_64k_h32") is None
    finally:
        bench.TRAFFIC_RECORD = bench_rec
