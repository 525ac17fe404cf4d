"""Host logic of the pinned-host-buffer path, on the CPU: the reading of cu_seqlens and
the cut of the packed segments into runs that the binding gives separate streams."""
import random

import pytest

from chunked_gated_delta_gdr_gb300 import api


def test_segment_bounds_clamp_and_running_maximum():
    # out-of-range values clamp to [0, T]; a value below its predecessor is raised to it
    assert api._segment_bounds([-5, 10, 7, 300, 250, 1000], 400) == [0, 10, 10, 300, 300, 400]
    assert api._segment_bounds([0], 0) == [0]


def check_groups(bounds, parts, groups):
    n = len(bounds) - 1
    total = bounds[-1] - bounds[0]
    assert len(groups) <= max(parts, 1)
    if total == 0:
        assert groups == []
        return
    # consecutive runs of whole segments covering every segment once, none empty
    assert groups[0][0] == 0 and groups[-1][1] == n
    for (a0, a1), (b0, b1) in zip(groups, groups[1:]):
        assert a1 == b0
    for n0, n1 in groups:
        assert n0 < n1 and bounds[n1] > bounds[n0]


@pytest.mark.parametrize("seed", range(40))
def test_segment_groups_cover_every_segment_once(seed):
    rnd = random.Random(seed)
    n = rnd.randint(1, 30)
    lens = [rnd.choice([0, 0, 1, 63, 64, 65, rnd.randint(1, 5000)]) for _ in range(n)]
    start = rnd.choice([0, 0, 17])
    cu = [start]
    for x in lens:
        cu.append(cu[-1] + x)
    bounds = api._segment_bounds(cu, cu[-1] + rnd.choice([0, 9]))
    for parts in range(1, 7):
        check_groups(bounds, parts, api._segment_groups(bounds, parts))


def test_segment_groups_balance_equal_segments():
    bounds = [64 * i for i in range(17)]  # 16 segments of 64 tokens
    groups = api._segment_groups(bounds, 4)
    assert groups == [(0, 4), (4, 8), (8, 12), (12, 16)]


def test_segment_groups_keep_a_long_segment_whole():
    bounds = [0, 10, 10000, 10010, 10020]
    groups = api._segment_groups(bounds, 4)
    check_groups(bounds, 4, groups)
    assert any(n0 <= 1 < n1 for n0, n1 in groups)  # segment 1 lies in one run
    assert len(groups) < 4  # the long segment leaves too few tokens for four runs
