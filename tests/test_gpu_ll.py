"""The pipelined variant with flag-in-data messages (RA_PROTOCOL_LL through
an inbox in device memory, RA_PROTOCOL_LL_CLUSTER through the successor's
shared memory in a thread-block cluster) against the oracle, bitwise,
through the C ABI: every dtype and op, the three collectives, in place,
launch shapes, calls that follow one another, the restart of the inbox's
flags before they would wrap, a withheld message that must time out rather
than be taken from an earlier call's words, CUDA graph replay of the cluster
form, and the limits of both."""

import numpy as np
import pytest

from oracle import elementops, ring
from ring_allreduce_gb300 import inputs
from rahelpers import DeviceRanks, assert_bitwise_equal

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

DTYPE_OPS = [("f32", "sum"), ("f32", "max"), ("bf16", "sum"), ("bf16", "max"),
             ("i32", "sum"), ("i32", "max"), ("f16", "sum"), ("f16", "max"),
             ("f64", "sum"), ("f64", "max"), ("i64", "sum"), ("i64", "max")]
# (R, n): degenerate, n < R, ragged tails, chunks of one CTA and of several
SHAPES = [(2, 1), (3, 2), (4, 4096), (5, 1001), (8, 1024), (8, 8 * 1024 + 13), (13, 7777), (16, 2**14 + 3),
          (32, 4097), (8, 2**16 + 5)]


@pytest.fixture(scope="module")
def ra():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_gb300 import build
    build.build()
    from ring_allreduce_gb300 import binding
    return binding


def _dist(dtype):
    return {"f32": "normal", "bf16": "grad", "i32": "int20", "f16": "grad", "f64": "normal", "i64": "int40"}[dtype]


def _run(ra, h, kind, inp, out):
    if kind == "allreduce":
        h.allreduce(inp.views, out.views)
    elif kind == "reduce_scatter":
        h.reduce_scatter(inp.views, out.views)
    else:
        h.all_gather(inp.views)


PROTOCOLS = ["LL", "LL_CLUSTER"]


def _shapes(protocol):
    # the cluster form holds a channel's R ranks in one cluster: R <= 16
    return [(R, n) for R, n in SHAPES if protocol == "LL" or R <= 16]


def run_ll(ra, x, dtype, op, kind="allreduce", inplace=False, ctas=0, protocol="LL"):
    R, n = len(x), len(x[0])
    st = inputs.storage_dtype(dtype)
    inp = DeviceRanks(R, n, st, host=x)
    out = inp if inplace else DeviceRanks(R, n, st)
    with ra.RingAllReduce(R, n, dtype, op, variant="pipelined") as h:
        h.set_option(ra.Option.PROTOCOL, ra.Protocol[protocol])
        if ctas:
            h.set_option(ra.Option.CTAS, ctas)
        _run(ra, h, kind, inp, out)
        status, err = h.device_status()
        assert status == ra.Status.OK, err.as_dict()
    torch.cuda.synchronize()
    assert inp.guards_intact(), "write outside an input buffer"
    assert out.guards_intact(), "write outside an output buffer"
    return out.host()


def _owned(R, n, got, want, what):
    plan = ring.chunk_plan(R, n)
    for r in range(R):
        off, L = plan[ring.owned_chunk(R, r)]
        assert_bitwise_equal(got[r][off:off + L], want[r][off:off + L], f"{what} rank {r}")


@pytest.mark.parametrize("protocol", PROTOCOLS)
@pytest.mark.parametrize("dtype,op", DTYPE_OPS)
def test_ll_allreduce_matches_oracle(ra, protocol, dtype, op):
    o = elementops.get_op(dtype, op)
    for i, (R, n) in enumerate(_shapes(protocol)):
        x = inputs.generate(R, n, dtype, _dist(dtype), seed=700 + i)
        want = ring.ring_allreduce(x, o)
        got = run_ll(ra, x, dtype, op, protocol=protocol)
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], f"{protocol} {dtype}/{op} R={R} n={n} rank {r}")


@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("bf16", "sum"), ("i32", "max"), ("f16", "sum"),
                                      ("f64", "sum"), ("i64", "max")])
@pytest.mark.parametrize("protocol", PROTOCOLS)
def test_ll_reduce_scatter_owned_chunk(ra, protocol, dtype, op):
    o = elementops.get_op(dtype, op)
    for i, (R, n) in enumerate(_shapes(protocol)):
        x = inputs.generate(R, n, dtype, _dist(dtype), seed=800 + i)
        _owned(R, n, run_ll(ra, x, dtype, op, kind="reduce_scatter", protocol=protocol),
               ring.ring_reduce_scatter(x, o), f"{protocol} RS {dtype} R={R} n={n}")


@pytest.mark.parametrize("protocol", PROTOCOLS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16", "f64", "i64"])
def test_ll_all_gather_from_reduce_scatter_layout(ra, protocol, dtype):
    """Only chunk (r+1) of buf[r] matters; the junk elsewhere is overwritten."""
    o = elementops.get_op(dtype, "sum")
    for i, (R, n) in enumerate(_shapes(protocol)):
        x = inputs.generate(R, n, dtype, _dist(dtype), seed=900 + i)
        rs = ring.ring_reduce_scatter(x, o)
        junk = inputs.generate(R, n, dtype, _dist(dtype), seed=999)
        plan = ring.chunk_plan(R, n)
        buf = []
        for r in range(R):
            b = junk[r].copy()
            off, L = plan[ring.owned_chunk(R, r)]
            b[off:off + L] = rs[r][off:off + L]
            buf.append(b)
        want = ring.ring_all_gather(buf, o)
        got = run_ll(ra, buf, dtype, "sum", kind="all_gather", inplace=True, protocol=protocol)
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], f"{protocol} AG {dtype} R={R} n={n} rank {r}")


@pytest.mark.parametrize("protocol", PROTOCOLS)
@pytest.mark.parametrize("kind", ["allreduce", "reduce_scatter"])
def test_ll_in_place(ra, protocol, kind):
    o = elementops.get_op("f32", "sum")
    for i, (R, n) in enumerate(_shapes(protocol)):
        x = inputs.generate(R, n, "f32", "normal", seed=1000 + i)
        got = run_ll(ra, x, "f32", "sum", kind=kind, inplace=True, protocol=protocol)
        if kind == "allreduce":
            want = ring.ring_allreduce(x, o)
            for r in range(R):
                assert_bitwise_equal(got[r], want[r], f"LL in place R={R} n={n}")
        else:
            _owned(R, n, got, ring.ring_reduce_scatter(x, o), f"LL RS in place R={R} n={n}")


@pytest.mark.parametrize("protocol", PROTOCOLS)
@pytest.mark.parametrize("R,n,ctas", [(8, 1000, 1), (8, 8 * 1024 + 13, 3), (4, 4096, 64), (5, 5 * 4 * 256, 1)])
def test_ll_launch_shapes(ra, protocol, R, n, ctas):
    """Channels given: one CTA carries up to 4 positions per thread (n = 1000
    and 5120 at one channel); 64 channels leave most threads without a
    position."""
    x = inputs.generate(R, n, "bf16", "grad", seed=11 + ctas)
    want = ring.ring_allreduce(x, elementops.get_op("bf16", "sum"))
    got = run_ll(ra, x, "bf16", "sum", ctas=ctas, protocol=protocol)
    for r in range(R):
        assert_bitwise_equal(got[r], want[r], f"LL ctas={ctas} R={R} n={n} rank {r}")


@pytest.mark.parametrize("protocol", PROTOCOLS)
def test_ll_too_few_channels_is_unsupported(ra, protocol):
    # chunks of 4101 elements: more than 4 channels of 256 threads carry at
    # 4 positions per thread (4096)
    R, n = 8, 8 * 4101
    with ra.RingAllReduce(R, n, "f32", "sum", variant="pipelined") as h:
        h.set_option(ra.Option.PROTOCOL, ra.Protocol[protocol])
        h.set_option(ra.Option.CTAS, 4)
        inp, out = DeviceRanks(R, n, np.float32), DeviceRanks(R, n, np.float32)
        with pytest.raises(ra.RAError) as e:
            h.allreduce(inp.views, out.views)
        assert e.value.status == ra.Status.ERR_UNSUPPORTED


@pytest.mark.parametrize("protocol", PROTOCOLS)
def test_ll_calls_in_a_row_and_mixed_collectives(ra, protocol):
    """One handle: AllReduce, ReduceScatter, AllGather and AllReduce again on
    other inputs.  LL: one inbox whose flags are new with every call, so no
    word an earlier call left behind is taken for this call's message (the
    flag moves on by each call's rounds).  LL_CLUSTER: rows zeroed by every
    launch."""
    R, n = 6, 6 * 777 + 5
    o = elementops.get_op("f32", "sum")
    with ra.RingAllReduce(R, n, "f32", "sum", variant="pipelined") as h:
        h.set_option(ra.Option.PROTOCOL, ra.Protocol[protocol])
        flag0 = h.get_option(ra.Option.LL_FLAG)
        assert flag0 == 1
        for seed, kind in enumerate(["allreduce", "allreduce", "reduce_scatter", "all_gather", "allreduce"]):
            x = inputs.generate(R, n, "f32", "normal", seed=40 + seed)
            inp, out = DeviceRanks(R, n, np.float32, host=x), DeviceRanks(R, n, np.float32)
            _run(ra, h, kind, inp, out)
            status, err = h.device_status()
            assert status == ra.Status.OK, err.as_dict()
            if kind == "allreduce":
                want, got = ring.ring_allreduce(x, o), out.host()
                for r in range(R):
                    assert_bitwise_equal(got[r], want[r], f"call {seed} rank {r}")
            elif kind == "reduce_scatter":
                _owned(R, n, out.host(), ring.ring_reduce_scatter(x, o), f"call {seed}")
            else:
                want, got = ring.ring_all_gather(x, o), inp.host()
                for r in range(R):
                    assert_bitwise_equal(got[r], want[r], f"AG call {seed} rank {r}")
        rounds = 2 * (R - 1)
        moved = 3 * rounds + 2 * (R - 1) if protocol == "LL" else 0
        assert h.get_option(ra.Option.LL_FLAG) == flag0 + moved


def test_ll_flags_restart_before_they_wrap(ra):
    """A call whose flags would pass 2^32 - 1 zeroes the inbox and starts
    again at 1; the call whose last message carries 2^32 - 3 (and leaves
    2^32 - 1 for the next) does not."""
    R, n = 4, 4 * 1500 + 3
    rounds = 2 * (R - 1)
    o = elementops.get_op("i32", "sum")
    with ra.RingAllReduce(R, n, "i32", "sum", variant="pipelined") as h:
        h.set_option(ra.Option.PROTOCOL, ra.Protocol.LL)
        for bad in (0, 2**32):
            with pytest.raises(ra.RAError):
                h.set_option(ra.Option.LL_FLAG, bad)
        x = inputs.generate(R, n, "i32", "int20", seed=3)
        inp, out = DeviceRanks(R, n, np.int32, host=x), DeviceRanks(R, n, np.int32)
        want = ring.ring_allreduce(x, o)
        h.allreduce(inp.views, out.views)           # fills the inbox with low flags
        start = 2**32 - 1 - rounds                  # messages carry start .. 2^32 - 3
        h.set_option(ra.Option.LL_FLAG, start)
        for expect_after in (2**32 - 1, 1 + rounds, 1 + 2 * rounds):
            out = DeviceRanks(R, n, np.int32)
            h.allreduce(inp.views, out.views)
            status, err = h.device_status()
            assert status == ra.Status.OK, err.as_dict()
            assert h.get_option(ra.Option.LL_FLAG) == expect_after
            got = out.host()
            for r in range(R):
                assert_bitwise_equal(got[r], want[r], f"flag {expect_after} rank {r}")


@pytest.mark.parametrize("protocol", PROTOCOLS)
def test_ll_withheld_message_times_out(ra, protocol):
    """After a good call, a rank that sends nothing from the next-to-last
    round on leaves exactly its successor waiting in the last round.  LL:
    on a word that holds the previous call's message, whose flag is the
    awaited one less the call's rounds.  LL_CLUSTER: on a word the launch
    zeroed (flag 0; message m carries m + 1).  The next call is correct."""
    R, n = 4, 4 * 4096
    rounds = 2 * (R - 1)
    x = inputs.generate(R, n, "f32", "normal", 8)
    want = ring.ring_allreduce(x, elementops.get_op("f32", "sum"))
    inp = DeviceRanks(R, n, np.float32, host=x)
    out = DeviceRanks(R, n, np.float32)
    with ra.RingAllReduce(R, n, "f32", "sum", variant="pipelined") as h:
        h.set_option(ra.Option.PROTOCOL, ra.Protocol[protocol])
        h.set_option(ra.Option.TIMEOUT_NS, 20_000_000)
        h.allreduce(inp.views, out.views)
        assert h.device_status()[0] == ra.Status.OK
        h.set_option(ra.Option.SKIP_ARRIVAL, (2 << 16) | (rounds - 2))
        h.allreduce(inp.views, out.views)
        status, err = h.device_status()
        assert status == ra.Status.ERR_TIMEOUT
        assert err.code == 5 and err.rank == 3 and err.peer == 2 and err.round == rounds - 1, err.as_dict()
        if protocol == "LL":
            assert err.expected == 1 + rounds + (rounds - 2)
            assert err.observed == err.expected - rounds
        else:
            assert (err.observed, err.expected) == (0, rounds - 1)
        assert "LL message" in ra.ra_last_error()
        h.set_option(ra.Option.SKIP_ARRIVAL, -1)
        out = DeviceRanks(R, n, np.float32)
        h.allreduce(inp.views, out.views)
        assert h.device_status()[0] == ra.Status.OK
    got = out.host()
    for r in range(R):
        assert_bitwise_equal(got[r], want[r])


def test_ll_inbox_limit(ra):
    """(2R-3) x R x C words of 8 bytes at most 64 MiB: R = 32 with 2^22
    elements per rank needs more and is refused before any launch."""
    R, n = 32, 2**22
    with ra.RingAllReduce(R, n, "f32", "sum", variant="pipelined") as h:
        h.set_option(ra.Option.PROTOCOL, ra.Protocol.LL)
        inp = DeviceRanks(R, n, np.float32)
        with pytest.raises(ra.RAError) as e:
            h.allreduce(inp.views, inp.views)
        assert e.value.status == ra.Status.ERR_UNSUPPORTED
        assert "inbox" in ra.ra_last_error()


def test_ll_cluster_limits(ra):
    """R above 16 cannot form one cluster; rows above 200 KiB per CTA (here
    29 rows x 4 positions x 256 threads x 16 bytes at R = 16 with 8-byte
    elements and one channel) do not fit: both refused before any launch."""
    for R, n, dtype, ctas in ((17, 17 * 64, "f32", 0), (16, 16 * 1024, "f64", 1)):
        with ra.RingAllReduce(R, n, dtype, "sum", variant="pipelined") as h:
            h.set_option(ra.Option.PROTOCOL, ra.Protocol.LL_CLUSTER)
            if ctas:
                h.set_option(ra.Option.CTAS, ctas)
            st = inputs.storage_dtype(dtype)
            inp, out = DeviceRanks(R, n, st), DeviceRanks(R, n, st)
            with pytest.raises(ra.RAError) as e:
                h.allreduce(inp.views, out.views)
            assert e.value.status == ra.Status.ERR_UNSUPPORTED, (R, n)


def test_ll_cluster_replays_from_a_caller_graph(ra):
    """The cluster form keeps nothing between calls, so a caller's CUDA graph
    may capture it and replay it on new data."""
    R, n = 8, 8 * 999 + 7
    o = elementops.get_op("bf16", "sum")
    inp = DeviceRanks(R, n, np.uint16, host=inputs.generate(R, n, "bf16", "grad", 1))
    out = DeviceRanks(R, n, np.uint16)
    with ra.RingAllReduce(R, n, "bf16", "sum", variant="pipelined") as h:
        h.set_option(ra.Option.PROTOCOL, ra.Protocol.LL_CLUSTER)
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            h.allreduce(inp.views, out.views, side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            h.allreduce(inp.views, out.views, side)
        for seed in (7, 8, 9):
            x = inputs.generate(R, n, "bf16", "grad", seed)
            inp.big.copy_(DeviceRanks(R, n, np.uint16, host=x).big)
            g.replay()
            torch.cuda.synchronize()
            want, got = ring.ring_allreduce(x, o), out.host()
            for r in range(R):
                assert_bitwise_equal(got[r], want[r], f"replay seed {seed} rank {r}")
        assert h.device_status()[0] == ra.Status.OK


def test_protocol_option_values(ra):
    with ra.RingAllReduce(4, 1024, "f32", "sum") as h:
        assert h.get_option(ra.Option.PROTOCOL) == ra.Protocol.SIMPLE
        with pytest.raises(ra.RAError) as e:
            h.set_option(ra.Option.PROTOCOL, 3)
        assert e.value.status == ra.Status.ERR_INVALID
        h.set_option(ra.Option.PROTOCOL, ra.Protocol.LL)
        assert h.get_option(ra.Option.PROTOCOL) == ra.Protocol.LL


@pytest.mark.parametrize("protocol,R,n", [("LL", 8, 8 * 58000 + 3), ("LL_CLUSTER", 8, 2**20 + 3),
                                          ("LL_CLUSTER", 16, 16 * 40000 + 1)])
def test_ll_largest_default_shapes(ra, protocol, R, n):
    """LL near its co-residency limit (chunks of 58001 elements: four positions
    per thread over some 57 channels of one cooperative launch) and
    LL_CLUSTER with hundreds of independent clusters running in waves: both
    bitwise the oracle's ring."""
    x = inputs.generate(R, n, "f32", "normal", seed=R + n % 97)
    want = ring.ring_allreduce(x, elementops.get_op("f32", "sum"))
    got = run_ll(ra, x, "f32", "sum", protocol=protocol)
    for r in range(R):
        assert_bitwise_equal(got[r], want[r], f"{protocol} R={R} n={n} rank {r}")
