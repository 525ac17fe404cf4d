"""The fused path's sequence-split planner (``gdr_split_plan``), host code, on the CPU.

The planner picks the number of pieces P and the first piece's weight a that minimise
the two passes of the split, measured in units of the whole segment.  These tests check
its choice against an independent event-driven list schedule of the same passes: pass A
runs each (segment, head)'s first piece (length a) and, for every middle piece, the
offset R and the transition M of its affine state map (length 1 each); pass B runs the
P - 1 later pieces (length 1).  On each pass the SMs take the units in that order as
they come free.
"""
import heapq

import pytest

from chunked_gated_delta_gdr_gb300 import api

MAX_PIECES = 8
LEADS = (1, 2, 3)


def list_schedule(lengths, sms):
    """Makespan of jobs taken in order by whichever of `sms` machines frees first."""
    free = [0] * sms
    heapq.heapify(free)
    end = 0
    for length in lengths:
        t = heapq.heappop(free) + length
        end = max(end, t)
        heapq.heappush(free, t)
    return end


def split_cost(units, sms, pieces, lead):
    """Pass A + pass B of a split into `pieces`, over the whole segment's length."""
    pass_a = [lead] * units + [1] * (units * 2 * (pieces - 2))
    pass_b = [1] * (units * (pieces - 1))
    return (list_schedule(pass_a, sms) + list_schedule(pass_b, sms)) / (lead + pieces - 1)


def best_plan(units, sms):
    """The cheapest (pieces, lead); ties to fewer pieces, then the lighter first piece;
    no split unless a plan beats the whole segment (cost 1) and 3 units per SM fit."""
    if units <= 0 or sms <= 0 or 3 * units > sms:
        return 1, 1
    best, best_cost = (1, 1), 1.0
    for pieces in range(3, MAX_PIECES + 1):
        for lead in LEADS:
            c = split_cost(units, sms, pieces, lead)
            if c < best_cost - 1e-9:
                best, best_cost = (pieces, lead), c
    return best


def test_long_sequence_plan():
    """One sequence of 32 value heads on 152 SMs (the long single-sequence workload):
    five pieces, the first twice as long.  Pass A: the 32 first pieces take 2 time units
    while 120 SMs run the 192 R and M units in 2; pass B: 128 later pieces in 1; so half
    the whole segment's time."""
    assert api.split_plan(32, 152) == (5, 2)
    assert split_cost(32, 152, 5, 2) == pytest.approx(3 / 6)


@pytest.mark.parametrize("units,sms", [(0, 152), (-3, 152), (5, 0), (51, 152), (200, 152)])
def test_no_split(units, sms):
    assert api.split_plan(units, sms) == (1, 1)


@pytest.mark.parametrize("sms", [16, 76, 132, 148, 152])
def test_plan_matches_list_schedule(sms):
    for units in range(1, sms // 3 + 1):
        assert api.split_plan(units, sms) == best_plan(units, sms), (units, sms)


def test_planted_cost_mistakes_are_seen():
    """The simulation separates plans that a wrong pass-A count would confuse: with the
    R and M units left out of pass A, more pieces would always look cheaper."""
    units, sms = 32, 152
    chosen = api.split_plan(units, sms)
    wrong = min(((p, a) for p in range(3, MAX_PIECES + 1) for a in LEADS),
                key=lambda pa: (list_schedule([pa[1]] * units, sms)
                                + list_schedule([1] * (units * (pa[0] - 1)), sms))
                / (pa[1] + pa[0] - 1))
    assert chosen != wrong
