"""Pins of the counting-barrier simulation: exactly R-1 arrivals land in
every slot of every round ("comm: lift the GIN scale-out ceiling by making
the rail barrier a counting barrier", section "Fix"), a missing arrival
makes the waiters of that round give up with one arrival missing (its
section "Cost" describes the timeout message as the count of missing
arrivals), and the 64-bit rolling comparison survives wrap-around (NCCL
Device API GIN article, section on signals and counters)."""

import pytest

from oracle import barrier


def test_rolling_compare():
    assert barrier.rolling_reached(5, 5)
    assert barrier.rolling_reached(6, 5)
    assert not barrier.rolling_reached(4, 5)
    top = (1 << 64) - 1
    assert barrier.rolling_reached(2, top)          # wrapped past the target
    assert not barrier.rolling_reached(top, 2)
    # counters keep 56 bits (GIN article): the compare looks at those only
    top56 = (1 << 56) - 1
    assert barrier.rolling_reached(1, top56, bits=56)
    assert not barrier.rolling_reached(top56, 1, bits=56)
    assert barrier.rolling_reached((1 << 60) + 7, 7, bits=56)   # bits above 56 ignored


def test_barrier_round_counts():
    assert barrier.barrier_rounds(4) == 5           # 2(R-1) rounds, 5 gaps
    assert barrier.barrier_rounds(4, phases=1) == 2
    assert barrier.barrier_rounds(2) == 1
    assert barrier.barrier_rounds(1) == 0


@pytest.mark.parametrize("R,G", [(2, 1), (3, 2), (4, 1), (8, 2)])
def test_exactly_r_minus_1_arrivals_per_slot(R, G):
    T = barrier.barrier_rounds(R)
    sim = barrier.CountingBarrierSim(R, G, T)
    for epoch in (1, 2, 3):
        assert sim.run_call(epoch) == []
        for g in range(G):
            for t in range(T):
                for w in range(R):
                    assert sim.slots[g][t][w] == epoch * (R - 1)
                    assert sim.slots[g][t][w] == barrier.expected_slot_value(R, epoch)
                    assert sim.shadows[g][t][w] == sim.slots[g][t][w]


def test_skipped_arrival_times_out_with_one_missing():
    R, G = 4, 2
    T = barrier.barrier_rounds(R)
    sim = barrier.CountingBarrierSim(R, G, T)
    fails = sim.run_call(1, timeout_s=0.2, skip=(2, 1, 3))
    at_round = [f for f in fails if f["round"] == 3 and f["channel"] == 1]
    assert sorted(f["rank"] for f in at_round) == [0, 1, 3]
    assert all(f["missing"] == 1 and f["expected"] == R - 1 for f in at_round)
    # the other channel is untouched
    assert all(f["channel"] == 1 for f in fails)
