"""Counting barrier between ring rounds, simulated with host threads (test
infrastructure only).

"comm: lift the GIN scale-out ceiling by making the rail barrier a counting
barrier", section "Fix": a barrier only has to count arrivals, so every peer
adds 1 to one signal of the waiter, and the waiter moves its shadow forward
by (number of ranks - 1) and polls that one signal until it is reached.  The
same page, section "Scoped to the rail team, deliberately", warns that one
anonymous counter reused across rounds lets a peer that is a round ahead
stand in for a late one; the reading taken here is one signal per (channel,
barrier round, waiter), so a count can only come from the round it belongs
to.  The NCCL Device API GIN article (section on signals and counters) gives
the signal as a 64-bit value compared in a rolling way, so that x < x + 1
survives wrap-around.

The simulation: R x G threads (rank r of channel g), each running the
barrier rounds of one call.  Every waiter keeps a shadow per slot and moves
it forward by R-1 before it polls.  After a call with sequence number
``epoch`` (1 for the first call on a fresh slot array) every slot and every
shadow must hold ``epoch * (R - 1)``.  A rank told to skip one arrival makes exactly that
waiter of that round give up after the time limit with one arrival missing.
"""

import threading
import time

__all__ = ["rolling_reached", "CountingBarrierSim", "expected_slot_value", "barrier_rounds"]

_MASK64 = (1 << 64) - 1


def rolling_reached(observed, target, bits=64):
    """True when ``observed`` has reached ``target`` in rolling order on the
    low ``bits`` bits: the difference observed - target, taken modulo
    2^bits, lies in the lower half (signals compare 64 bits, counters 56)."""
    mask = (1 << bits) - 1
    d = (observed - target) & mask
    return d < (1 << (bits - 1))


def barrier_rounds(R, phases=2):
    """Barriers one call needs: one between each pair of consecutive rounds.
    AllReduce has 2(R-1) rounds (phases=2), ReduceScatter or AllGather alone
    R-1 (phases=1)."""
    rounds = phases * (R - 1)
    return max(rounds - 1, 0)


def expected_slot_value(R, epoch):
    """What every slot holds after ``epoch`` complete calls: each of the R-1
    peers of a waiter adds 1 once per call."""
    return (epoch * (R - 1)) & _MASK64


class CountingBarrierSim:
    """Signal slots indexed [channel][barrier round][waiter rank], and one
    shadow per slot, owned by its waiter."""

    def __init__(self, R, G, T):
        self.R, self.G, self.T = R, G, T
        self.slots = [[[0] * R for _ in range(T)] for _ in range(G)]
        self.shadows = [[[0] * R for _ in range(T)] for _ in range(G)]
        self._lock = threading.Lock()

    def arrive(self, g, t, r):
        """Rank r of channel g has finished round t: add 1 to the slot of
        every peer (SignalAdd 1, never Inc)."""
        with self._lock:
            for p in range(self.R):
                if p != r:
                    self.slots[g][t][p] = (self.slots[g][t][p] + 1) & _MASK64

    def wait(self, g, t, r, epoch, timeout_s):
        """Move rank r's shadow of this slot forward by R-1 (the arrivals it
        expects), then poll its slot until it meets the shadow.  Returns
        (ok, observed, target).  ``epoch`` is the call's sequence number; on
        a fresh slot array the shadow then equals epoch*(R-1)."""
        self.shadows[g][t][r] = (self.shadows[g][t][r] + self.R - 1) & _MASK64
        target = self.shadows[g][t][r]
        deadline = time.monotonic() + timeout_s
        while True:
            with self._lock:
                observed = self.slots[g][t][r]
            if rolling_reached(observed, target):
                return True, observed, target
            if time.monotonic() > deadline:
                return False, observed, target
            time.sleep(0.0002)

    def run_call(self, epoch, timeout_s=5.0, skip=None):
        """One call: every (rank, channel) thread runs T rounds of
        arrive-then-wait.  ``skip=(r, g, t)`` makes that rank not arrive in
        that round.  A waiter that gives up stops.  Returns the list of
        failures as dicts {rank, channel, round, observed, expected, missing}."""
        failures = []
        flock = threading.Lock()

        def body(r, g):
            for t in range(self.T):
                if skip != (r, g, t):
                    self.arrive(g, t, r)
                ok, observed, target = self.wait(g, t, r, epoch, timeout_s)
                if not ok:
                    with flock:
                        failures.append(dict(rank=r, channel=g, round=t, observed=observed,
                                             expected=target,
                                             missing=(target - observed) & _MASK64))
                    return

        threads = [threading.Thread(target=body, args=(r, g))
                   for g in range(self.G) for r in range(self.R)]
        for th in threads:
            th.start()
        for th in threads:
            th.join()
        return failures
