"""The signal layer on the device (the GIN article's signals and shadows:
SignalAdd, readSignal and waitSignal on the low `bits` bits, resetSignal,
increaseSignalShadow / waitSignalMeetShadow), through the C ABI.

The barrier and the flags compare every signal with its waiter's shadow in
rolling order, so seeding both with values just below 2^56 and narrowing the
comparison to 56 bits (RA_OPT_SIGNAL_BITS) runs the protocol across the wrap
of a 56-bit counter; the oracle's ``barrier.rolling_reached(..., bits=56)``
is the pin for what the device decides there.  Results stay bitwise the
oracle's ring."""

import numpy as np
import pytest

from oracle import barrier, elementops, ring
from ring_allreduce_gb300 import inputs
from rahelpers import DeviceRanks, assert_bitwise_equal

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

B56 = 1 << 56
M56 = B56 - 1


@pytest.fixture(scope="module")
def ra():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_gb300 import build
    build.build()
    from ring_allreduce_gb300 import binding
    return binding


def _case(R, n, seed):
    x = inputs.generate(R, n, "f32", "normal", seed)
    return x, DeviceRanks(R, n, np.float32, host=x), DeviceRanks(R, n, np.float32), \
        ring.ring_allreduce(x, elementops.get_op("f32", "sum"))


def _check(out, want, what):
    got = out.host()
    for r in range(len(want)):
        assert_bitwise_equal(got[r], want[r], f"{what} rank {r}")


@pytest.mark.parametrize("R,G", [(4, 2), (8, 3)])
def test_counting_barrier_across_a_56_bit_wrap(ra, R, G):
    """Signals seeded 3 counts below 2^56 with garbage above bit 55, shadows
    seeded with the same low 56 bits and zero above: with 56-bit rolling
    comparisons every barrier round still waits for exactly R-1 arrivals,
    the calls stay bitwise correct, and readSignal (56 bits) returns the
    wrapped counts.  The high byte would make a 64-bit comparison pass at
    once, so this is the 56-bit path only."""
    n = R * 6000 + 5
    x, inp, out, want = _case(R, n, 31 + R)
    start = B56 - 3
    with ra.RingAllReduce(R, n, "f32", "sum", variant="persistent") as h:
        h.set_option(ra.Option.CTAS, G)
        h.allreduce(inp.views, out.views)            # lays the slots out for this shape
        assert h.device_status()[0] == ra.Status.OK
        h.seed_signals((0x5A << 56) | start, start)
        h.set_option(ra.Option.SIGNAL_BITS, 56)
        for k in range(1, 4):
            h.allreduce(inp.views, out.views)
            status, err = h.device_status()
            assert status == ra.Status.OK, err.as_dict()
            slots = h.read_signals()[0]
            shadows = h.read_shadows()
            exp = (start + k * (R - 1)) & M56
            assert all(v == exp for v in slots), (k, slots[:8])
            assert all((v & M56) == exp for v in shadows), (k, shadows[:8])
            # the device's verdict matches the pin: each signal has met its shadow
            assert all(barrier.rolling_reached(s, sh & M56, bits=56) for s, sh in zip(slots, shadows))
    _check(out, want, f"counting R={R} across 2^56")


def test_counting_barrier_timeout_across_a_56_bit_wrap(ra):
    """Seeded so that a barrier round's target is 2^56 (0 in 56 bits) and,
    with one arrival withheld, the signal stops at 2^56 - 1: a plain
    comparison of the low bits would call that reached; the rolling one must
    not.  The waiter gives up (RA_ERR_TIMEOUT) reporting observed 2^56 - 1
    and expected 0 in 56 bits, which the oracle's rolling_reached agrees is
    one short; resetSignal then clears the slots and the next call is
    correct."""
    R, n = 4, 4 * 4096
    x, inp, out, want = _case(R, n, 77)
    start = B56 - (R - 1)
    with ra.RingAllReduce(R, n, "f32", "sum", variant="persistent") as h:
        h.set_option(ra.Option.TIMEOUT_NS, 20_000_000)
        h.allreduce(inp.views, out.views)
        assert h.device_status()[0] == ra.Status.OK
        h.seed_signals(start, start)
        h.set_option(ra.Option.SIGNAL_BITS, 56)
        last = barrier.barrier_rounds(R) - 1
        h.set_option(ra.Option.SKIP_ARRIVAL, (2 << 16) | last)
        h.allreduce(inp.views, out.views)
        status, err = h.device_status()
        assert status == ra.Status.ERR_TIMEOUT
        assert err.code == 1 and err.round == last and err.rank != 2
        assert (err.observed, err.expected) == (M56, 0), err.as_dict()
        assert not barrier.rolling_reached(err.observed, err.expected, bits=56)
        assert barrier.rolling_reached((err.observed + 1) & M56, err.expected, bits=56)
        assert err.observed >= err.expected   # where a non-rolling compare would have let it pass
        assert "(1 missing)" in ra.ra_last_error()
        # the status call reset every signal (resetSignal): a fresh count
        h.set_option(ra.Option.SKIP_ARRIVAL, -1)
        h.allreduce(inp.views, out.views)
        assert h.device_status()[0] == ra.Status.OK
        slots = h.read_signals()[0]
        assert all(v == R - 1 for v in slots), slots[:8]
    _check(out, want, "after the wrap timeout")


@pytest.mark.parametrize("slices,window", [(1, 1), (3, 1), (4, 2)])
def test_pipelined_flags_and_shadows_across_a_56_bit_wrap(ra, slices, window):
    """The pipelined flags are signals too (SignalAdd of 1 per finished
    round) and each waiter keeps a shadow of its predecessor's flag
    (increaseSignalShadow by 1 per round, waitSignalMeetShadow): seeded just
    below 2^56 with garbage above bit 55 and compared on 56 bits, every call
    stays correct and after k calls every flag reads k * rounds past the
    seed, as does every shadow."""
    R, n = 5, 5 * 7000 + 3
    x, inp, out, want = _case(R, n, 55 + slices)
    rounds = 2 * (R - 1)
    start = B56 - 5
    with ra.RingAllReduce(R, n, "f32", "sum", variant="pipelined") as h:
        h.set_option(ra.Option.CTAS, 2)
        h.set_option(ra.Option.SLICES, slices)
        h.set_option(ra.Option.WINDOW, window)
        h.allreduce(inp.views, out.views)
        assert h.device_status()[0] == ra.Status.OK
        flags = h.read_signals()[0]
        assert flags == h.read_shadows() and all(v == rounds for v in flags)
        h.seed_signals((0xC3 << 56) | start, start)
        h.set_option(ra.Option.SIGNAL_BITS, 56)
        for k in range(1, 3):
            h.allreduce(inp.views, out.views)
            status, err = h.device_status()
            assert status == ra.Status.OK, err.as_dict()
            flags = h.read_signals()[0]
            shadows = h.read_shadows()
            exp = (start + k * rounds) & M56
            assert len(flags) == 2 * R * slices
            assert all(v == exp for v in flags), (k, flags[:8])
            assert all((v & M56) == exp for v in shadows), (k, shadows[:8])
    _check(out, want, f"pipelined slices={slices} window={window} across 2^56")


def test_read_signals_returns_the_low_bits(ra):
    """readSignal(bits): the same slots read with 64 and with 20 bits."""
    R, n = 4, 4 * 5000
    x, inp, out, want = _case(R, n, 12)
    with ra.RingAllReduce(R, n, "f32", "sum", variant="persistent") as h:
        h.allreduce(inp.views, out.views)
        v = (0x12345 << 40) | ((1 << 20) - 2)   # two counts below a 20-bit wrap
        h.seed_signals(v, v)
        full = h.read_signals()[0]
        h.set_option(ra.Option.SIGNAL_BITS, 20)
        low = h.read_signals()[0]
        assert all(s == v for s in full) and all(s == (v & ((1 << 20) - 1)) for s in low)
        # a 20-bit call from there: the counts roll over 2^20 and stay right
        h.allreduce(inp.views, out.views)
        assert h.device_status()[0] == ra.Status.OK
        low = h.read_signals()[0]
        assert all(s == ((v + R - 1) & ((1 << 20) - 1)) for s in low)
    _check(out, want, "20-bit signals")


def test_signal_bits_option_range(ra):
    with ra.RingAllReduce(4, 1024, "f32", "sum") as h:
        assert h.get_option(ra.Option.SIGNAL_BITS) == 64
        for bad in (0, 15, 65):
            with pytest.raises(ra.RAError) as e:
                h.set_option(ra.Option.SIGNAL_BITS, bad)
            assert e.value.status == ra.Status.ERR_INVALID
        h.set_option(ra.Option.SIGNAL_BITS, 56)
        assert h.get_option(ra.Option.SIGNAL_BITS) == 56
