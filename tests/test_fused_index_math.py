"""Index arithmetic of the fused kernel's operand-tile loop, checked on the CPU.

The prep warpgroup writes Tm diag(beta) and -Tm diag(beta e^G) over the lower
triangle's 8-column groups only (the groups above are cleared once at kernel start).
Thread `pid` (0..127) takes the row pair (q, 63 - q), q = pid >> 2, which holds
q/8 + 1 + (63 - q)/8 + 1 = 9 groups, and of those the groups gi = pid & 3, +4, +8.
These tests restate that mapping from ``role_prep`` in ``csrc/gdr_fused.cu`` and check
the properties the kernel relies on: every group on or below the diagonal written by
exactly one thread, none above it, at most three per thread, and the kept columns of a
group (u <= row - c0) exactly those on or below the diagonal.
"""
from collections import Counter


def groups_of(pid):
    """(row, first column) of each 8-column group thread `pid` writes, in loop order."""
    q = pid >> 2
    nq = (q >> 3) + 1
    out = []
    for gi in range(pid & 3, 9, 4):
        ri = q if gi < nq else 63 - q
        c0 = 8 * (gi if gi < nq else gi - nq)
        out.append((ri, c0))
    return out


def test_every_lower_group_exactly_once():
    seen = Counter(g for pid in range(128) for g in groups_of(pid))
    want = {(r, 8 * c) for r in range(64) for c in range(r // 8 + 1)}
    assert set(seen) == want
    assert all(n == 1 for n in seen.values())
    assert len(want) == 288


def test_no_group_above_the_diagonal():
    for pid in range(128):
        for ri, c0 in groups_of(pid):
            assert c0 <= ri, (pid, ri, c0)


def test_at_most_three_groups_per_thread():
    counts = [len(groups_of(pid)) for pid in range(128)]
    assert max(counts) == 3 and min(counts) == 2
    # the four threads of a row pair share its nine groups
    for q in range(32):
        assert sum(counts[4 * q + s] for s in range(4)) == 9


def test_kept_columns_are_on_or_below_the_diagonal():
    for pid in range(128):
        for ri, c0 in groups_of(pid):
            lim = ri - c0
            kept = [c0 + u for u in range(8) if u <= lim]
            assert kept == [c for c in range(c0, c0 + 8) if c <= ri]
