"""Parity of the CUDA library with the oracle, element by element and
bitwise (the fold order is fixed, so the tolerance is 0 ulp), through the
C ABI, for every variant, dtype and op, on seeded inputs; plus guard bands
around every buffer, in-place calls, the barrier's arrival count, the
timeout path and argument checks on a real device."""

import numpy as np
import pytest

from oracle import barrier, elementops, ring
from ring_allreduce_gb300 import inputs
from rahelpers import DeviceBuffers, DeviceRanks, assert_bitwise_equal

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

VARIANTS = ["direct", "ring", "persistent", "pipelined", "local"]
DTYPE_OPS = [("f32", "sum"), ("f32", "max"), ("bf16", "sum"), ("bf16", "max"),
             ("i32", "sum"), ("i32", "max"), ("f16", "sum"), ("f16", "max"),
             ("f64", "sum"), ("f64", "max"), ("i64", "sum"), ("i64", "max")]
# (R, n): degenerate, n < R, ragged, several tiles per chunk with a ragged tail
SHAPES = [(2, 1), (3, 2), (4, 4096), (5, 1001), (8, 8 * 1024 + 13), (2, 2**20 + 7),
          (8, 2**20 + 7), (13, 77777), (16, 2**16 + 3), (32, 2**16 + 1)]


@pytest.fixture(scope="module")
def ra():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_gb300 import build
    build.build()
    from ring_allreduce_gb300 import binding
    return binding


def _dist(dtype):
    return {"f32": "normal", "bf16": "grad", "i32": "int20", "f16": "grad", "f64": "normal", "i64": "int40"}[dtype]


def run_gpu(ra, x, dtype, op, variant, kind="allreduce", inplace=False, ctas=0, repeat=1, options=()):
    R, n = len(x), len(x[0])
    st = inputs.storage_dtype(dtype)
    inp = DeviceRanks(R, n, st, host=x)
    out = inp if inplace else DeviceRanks(R, n, st)
    with ra.RingAllReduce(R, n, dtype, op, variant=variant) as h:
        if ctas:
            h.set_option(ra.Option.CTAS, ctas)
        for key, value in options:
            h.set_option(key, value)
        for _ in range(repeat):
            if kind == "allreduce":
                h.allreduce(inp.views, out.views)
            elif kind == "reduce_scatter":
                h.reduce_scatter(inp.views, out.views)
            else:
                h.all_gather(inp.views)
        status, err = h.device_status()
        assert status == ra.Status.OK, err.as_dict()
    torch.cuda.synchronize()
    assert inp.guards_intact(), "write outside an input buffer"
    assert out.guards_intact(), "write outside an output buffer"
    return out.host()


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype,op", DTYPE_OPS)
def test_allreduce_matches_oracle(ra, variant, dtype, op):
    o = elementops.get_op(dtype, op)
    for i, (R, n) in enumerate(SHAPES):
        x = inputs.generate(R, n, dtype, _dist(dtype), seed=100 + i)
        want = ring.ring_allreduce(x, o)
        got = run_gpu(ra, x, dtype, op, variant)
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], f"{variant} {dtype}/{op} R={R} n={n} rank {r}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("bf16", "sum"), ("i32", "max"), ("f16", "sum"),
                                      ("f64", "sum"), ("i64", "max")])
def test_reduce_scatter_owned_chunk(ra, variant, dtype, op):
    o = elementops.get_op(dtype, op)
    for i, (R, n) in enumerate(SHAPES):
        x = inputs.generate(R, n, dtype, _dist(dtype), seed=200 + i)
        want = ring.ring_reduce_scatter(x, o)
        got = run_gpu(ra, x, dtype, op, variant, kind="reduce_scatter")
        plan = ring.chunk_plan(R, n)
        for r in range(R):
            off, L = plan[ring.owned_chunk(R, r)]
            assert_bitwise_equal(got[r][off:off + L], want[r][off:off + L], f"{variant} R={R} n={n} rank {r}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16", "f64", "i64"])
def test_all_gather_from_reduce_scatter_layout(ra, variant, dtype):
    """AllGather takes the layout ReduceScatter leaves: only chunk (r+1) of
    buf[r] matters; the other chunks hold junk that must be overwritten."""
    o = elementops.get_op(dtype, "sum")
    for i, (R, n) in enumerate(SHAPES):
        x = inputs.generate(R, n, dtype, _dist(dtype), seed=300 + i)
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
        got = run_gpu(ra, buf, dtype, "sum", variant, kind="all_gather", inplace=True)
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], f"{variant} R={R} n={n} rank {r}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("kind", ["allreduce", "reduce_scatter"])
def test_in_place(ra, variant, kind):
    o = elementops.get_op("f32", "sum")
    for i, (R, n) in enumerate(SHAPES):
        x = inputs.generate(R, n, "f32", "normal", seed=400 + i)
        got = run_gpu(ra, x, "f32", "sum", variant, kind=kind, inplace=True)
        if kind == "allreduce":
            want = ring.ring_allreduce(x, o)
            for r in range(R):
                assert_bitwise_equal(got[r], want[r], f"{variant} R={R} n={n}")
        else:
            want = ring.ring_reduce_scatter(x, o)
            plan = ring.chunk_plan(R, n)
            for r in range(R):
                off, L = plan[ring.owned_chunk(R, r)]
                assert_bitwise_equal(got[r][off:off + L], want[r][off:off + L], f"{variant} R={R} n={n}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("ctas", [1, 3, 64])
def test_launch_shapes(ra, variant, ctas):
    """Odd CTA counts still cover every element exactly once."""
    o = elementops.get_op("bf16", "sum")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for R, n in ((8, 2**20 + 7), (3, 100003)):
        x = inputs.generate(R, n, "bf16", "grad", seed=ctas)
        if variant in ("persistent", "pipelined") and R * ctas > sms:
            # more channels than can be co-resident: refused on the host
            with pytest.raises(ra.RAError) as e:
                run_gpu(ra, x, "bf16", "sum", variant, ctas=4 * sms)
            assert e.value.status == ra.Status.ERR_UNSUPPORTED
            continue
        want = ring.ring_allreduce(x, o)
        got = run_gpu(ra, x, "bf16", "sum", variant, ctas=ctas)
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], f"{variant} ctas={ctas} R={R}")


def test_single_rank_and_empty(ra):
    x = inputs.generate(1, 1000, "f32", "normal", 5)
    for v in VARIANTS:
        got = run_gpu(ra, x, "f32", "sum", v)
        assert_bitwise_equal(got[0], x[0])
    for v in VARIANTS:
        got = run_gpu(ra, [np.zeros(0, np.float32)] * 4, "f32", "sum", v)
        assert all(len(g) == 0 for g in got)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype,big", [("f32", 2.0**24), ("bf16", 256.0), ("f16", 2048.0), ("f64", 2.0**53)])
def test_ring_start_rank_pin_on_gpu(ra, variant, dtype, big):
    """Chunk k holds big, 1, 1, -big on ranks k..k+3: the ring's fold from
    rank k gives 0, any other start gives 2."""
    R, per = 4, 1000
    vals = [np.zeros(R * per, dtype=np.float32) for _ in range(R)]
    pattern = [big, 1.0, 1.0, -big]
    for k in range(R):
        for j in range(R):
            vals[(k + j) % R][k * per:(k + 1) * per] = pattern[j]
    if dtype == "bf16":
        x = [torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16) for v in vals]
    elif dtype == "f16":
        x = [torch.from_numpy(v).to(torch.float16).numpy() for v in vals]
    elif dtype == "f64":
        x = [v.astype(np.float64) for v in vals]
    else:
        x = vals
    got = run_gpu(ra, x, dtype, "sum", variant)
    for r in range(R):
        g = elementops.bf16_bits_to_f32(got[r]) if dtype == "bf16" else got[r]
        assert (g == 0).all()


@pytest.mark.parametrize("R,G", [(2, 1), (4, 3), (8, 5), (32, 2)])
def test_barrier_exactly_r_minus_1_arrivals(ra, R, G):
    """After k persistent calls every signal slot holds k (R-1): each of the
    R-1 peers arrived exactly once per round and call."""
    n = R * 5000 + 3
    x = inputs.generate(R, n, "f32", "normal", 7)
    inp = DeviceRanks(R, n, np.float32, host=x)
    out = DeviceRanks(R, n, np.float32)
    want = ring.ring_allreduce(x, elementops.get_op("f32", "sum"))
    with ra.RingAllReduce(R, n, "f32", "sum", variant="persistent") as h:
        h.set_option(ra.Option.CTAS, G)
        for k in range(1, 4):
            h.allreduce(inp.views, out.views)
            slots, ch, rounds, calls = h.read_signals()
            assert (ch, rounds, calls) == (G, barrier.barrier_rounds(R), k)
            assert len(slots) == G * rounds * R
            exp = barrier.expected_slot_value(R, k)
            assert all(v == exp for v in slots), slots
            shadows = h.read_shadows()
            assert len(shadows) == len(slots) and all(v == exp for v in shadows), shadows
        status, _ = h.device_status()
        assert status == ra.Status.OK
    got = out.host()
    for r in range(R):
        assert_bitwise_equal(got[r], want[r])


@pytest.mark.parametrize("kind", ["counting", "per_peer", "cluster"])
@pytest.mark.parametrize("passes", [2, 3, 8])
def test_persistent_passes(ra, kind, passes):
    """The persistent variant with its channel slices cut into passes (each
    through every round, with barrier rounds of its own): bitwise the
    oracle's on aligned and ragged plans, two calls in a row; the counting
    barrier's slots then hold k (R-1) in every (channel, pass, round), and
    the per-peer barrier stays at one pass."""
    o = elementops.get_op("bf16", "sum")
    opts = [(ra.Option.SLICES, passes)]
    if kind != "counting":
        opts.append((ra.Option.BARRIER, ra.Barrier.PER_PEER if kind == "per_peer" else ra.Barrier.CLUSTER))
    for R, n in ((8, 2**20 + 7), (3, 100003), (16, 2**16 + 3), (4, 2**22 + 5)):
        x = inputs.generate(R, n, "bf16", "grad", seed=passes + R)
        want = ring.ring_allreduce(x, o)
        got = run_gpu(ra, x, "bf16", "sum", "persistent", options=opts, repeat=2)
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], f"{kind} passes={passes} R={R}")
    if kind == "cluster":
        return
    R, G = 5, 3
    n = R * 9000 + 1
    x = inputs.generate(R, n, "f32", "normal", 11)
    inp, out = DeviceRanks(R, n, np.float32, host=x), DeviceRanks(R, n, np.float32)
    with ra.RingAllReduce(R, n, "f32", "sum", variant="persistent") as h:
        h.set_option(ra.Option.CTAS, G)
        for key, value in opts:
            h.set_option(key, value)
        J = passes if kind == "counting" else 1
        for k in range(1, 3):
            h.allreduce(inp.views, out.views)
            slots, ch, rounds, calls = h.read_signals()
            assert (ch, rounds, calls) == (G, J * barrier.barrier_rounds(R), k)
            if kind == "counting":
                assert len(slots) == G * rounds * R
                assert all(v == barrier.expected_slot_value(R, k) for v in slots), slots
                assert h.read_shadows() == slots
        assert h.device_status()[0] == ra.Status.OK
    want = ring.ring_allreduce(x, elementops.get_op("f32", "sum"))
    got = out.host()
    for r in range(R):
        assert_bitwise_equal(got[r], want[r], f"{kind} passes={passes} arrivals run")


@pytest.mark.parametrize("passes", [2, 3, 8])
@pytest.mark.parametrize("kind", ["allreduce", "reduce_scatter", "all_gather"])
def test_ring_passes(ra, passes, kind):
    """The ring variant with its chunks taken through the rounds in passes
    (each pass launches every round on one part of every chunk): bitwise the
    oracle's for every collective, on aligned and ragged plans (bf16 chunk
    starts off 16 bytes), graph captured on the first call and replayed on
    the second."""
    o = elementops.get_op("bf16", "sum")
    for R, n in ((8, 2**20 + 7), (3, 100003), (16, 2**16 + 3), (4, 2**22 + 5)):
        x = inputs.generate(R, n, "bf16", "grad", seed=passes + 3 * R)
        if kind == "all_gather":
            x = ring.ring_reduce_scatter(x, o)
            want = ring.ring_allreduce(inputs.generate(R, n, "bf16", "grad", seed=passes + 3 * R), o)
        elif kind == "reduce_scatter":
            want = ring.ring_reduce_scatter(x, o)
        else:
            want = ring.ring_allreduce(x, o)
        got = run_gpu(ra, x, "bf16", "sum", "ring", kind=kind, inplace=(kind == "all_gather"),
                      options=[(ra.Option.SLICES, passes)], repeat=2)
        for r in range(R):
            if kind == "reduce_scatter":
                off, L = ring.chunk_plan(R, n)[ring.owned_chunk(R, r)]
                assert_bitwise_equal(got[r][off:off + L], want[r][off:off + L], f"{kind} passes={passes} R={R}")
            else:
                assert_bitwise_equal(got[r], want[r], f"{kind} passes={passes} R={R}")


def test_barrier_timeout_reports_missing_arrival(ra):
    """A rank that withholds its arrival makes its peers' waits run out:
    the call reports RA_ERR_TIMEOUT with one arrival missing, nothing
    faults, and the handle works again afterwards."""
    R, n = 4, 4 * 4096
    x = inputs.generate(R, n, "f32", "normal", 8)
    inp = DeviceRanks(R, n, np.float32, host=x)
    out = DeviceRanks(R, n, np.float32)
    with ra.RingAllReduce(R, n, "f32", "sum", variant="persistent") as h:
        h.set_option(ra.Option.TIMEOUT_NS, 20_000_000)   # 20 ms
        # rank 2 withholds its arrival at the last barrier (round 4 of 5), so
        # it finishes while its three peers wait for it
        last = barrier.barrier_rounds(R) - 1
        h.set_option(ra.Option.SKIP_ARRIVAL, (2 << 16) | last)
        h.allreduce(inp.views, out.views)
        status, err = h.device_status()
        assert status == ra.Status.ERR_TIMEOUT
        assert err.code == 1 and err.round == last and err.rank != 2
        assert err.expected - err.observed == 1
        assert "missing" in ra.ra_last_error()
        # recovers: failure injection off, next call is correct
        h.set_option(ra.Option.SKIP_ARRIVAL, -1)
        h.set_option(ra.Option.TIMEOUT_NS, 1_000_000_000)
        h.allreduce(inp.views, out.views)
        status, err = h.device_status()
        assert status == ra.Status.OK
    want = ring.ring_allreduce(x, elementops.get_op("f32", "sum"))
    got = out.host()
    for r in range(R):
        assert_bitwise_equal(got[r], want[r])


def test_argument_checks_on_device(ra):
    R, n = 4, 1024
    inp = DeviceRanks(R, n, np.float32, host=inputs.generate(R, n, "f32", "normal", 1))
    out = DeviceRanks(R, n, np.float32)
    h = ra.RingAllReduce(R, n, "f32", "sum")
    try:
        bad = [p + 4 for p in out.ptrs()]                     # misaligned
        with pytest.raises(ra.RAError) as e:
            h.allreduce(inp.ptrs(), bad)
        assert e.value.status == ra.Status.ERR_INVALID
        ov = out.ptrs()
        ov[1] = ov[0] + 256                                   # outputs overlap
        with pytest.raises(ra.RAError) as e:
            h.allreduce(inp.ptrs(), ov)
        assert e.value.status == ra.Status.ERR_INVALID
        cpu = [torch.zeros(n, dtype=torch.float32) for _ in range(R)]   # host memory
        with pytest.raises(ra.RAError) as e:
            h.allreduce(inp.ptrs(), cpu)
        assert e.value.status == ra.Status.ERR_INVALID
        with pytest.raises(ra.RAError) as e:
            h.allreduce(inp.ptrs(), [0] * R)
        assert e.value.status == ra.Status.ERR_INVALID
        mixed = out.ptrs()
        mixed[2] = inp.ptrs()[1]                              # out[2] is another rank's input
        with pytest.raises(ra.RAError) as e:
            h.allreduce(inp.ptrs(), mixed)
        assert e.value.status == ra.Status.ERR_INVALID
        # option values outside their ranges are refused and change nothing
        for key, value in ((ra.Option.SLICES, -1), (ra.Option.SLICES, 65), (ra.Option.WINDOW, -1),
                           (ra.Option.WINDOW, 65), (ra.Option.VARIANT, 99), (ra.Option.BARRIER, 7),
                           (ra.Option.TIMEOUT_NS, 10), (ra.Option.TIMEOUT_NS, 60_000_000_001),
                           (ra.Option.CTAS, -2), (ra.Option.GATHER, 3),
                           (ra.Option.HOST_WINDOWS, 9)):
            before = h.get_option(key)
            with pytest.raises(ra.RAError) as e:
                h.set_option(key, value)
            assert e.value.status == ra.Status.ERR_INVALID, (key, value)
            assert h.get_option(key) == before, key
        with pytest.raises(ra.RAError) as e:
            h.set_option(999, 1)
        assert e.value.status == ra.Status.ERR_INVALID
        # nothing was enqueued: the device is fine and a good call works
        h.allreduce(inp.ptrs(), out.ptrs())
        assert h.device_status()[0] == ra.Status.OK
    finally:
        h.close()


@pytest.mark.parametrize("kind", ["allreduce", "reduce_scatter", "all_gather"])
def test_ring_graph_replay_and_rebuild(ra, kind):
    """The ring variant replays its captured graph on repeated calls with the
    same buffers (reading the data they hold now), captures a new one when
    the buffers change, and gives the same bits with graphs switched off."""
    R, n = 8, 2**18 + 5
    o = elementops.get_op("f32", "sum")
    plan = ring.chunk_plan(R, n)
    bufs = [DeviceRanks(R, n, np.float32) for _ in range(2)]
    outs = [DeviceRanks(R, n, np.float32) for _ in range(2)]
    with ra.RingAllReduce(R, n, "f32", "sum", variant="ring") as h:
        for step, (b, out, graphs) in enumerate([(0, 0, 1), (0, 0, 1), (1, 1, 1), (0, 1, 1), (1, 0, 0)]):
            if step == 4:
                h.set_option(ra.Option.GRAPHS, graphs)
            x = inputs.generate(R, n, "f32", "normal", seed=50 + step)
            if kind == "all_gather":
                rs = ring.ring_reduce_scatter(x, o, fill=np.float32(0))
                want = ring.ring_all_gather(rs, o)
                src = DeviceRanks(R, n, np.float32, host=rs)
                outs[out].big.copy_(src.big)
                h.all_gather(outs[out].views)
            else:
                bufs[b].big.copy_(DeviceRanks(R, n, np.float32, host=x).big)
                if kind == "allreduce":
                    want = ring.ring_allreduce(x, o)
                    h.allreduce(bufs[b].views, outs[out].views)
                else:
                    want = ring.ring_reduce_scatter(x, o)
                    h.reduce_scatter(bufs[b].views, outs[out].views)
            assert h.device_status()[0] == ra.Status.OK
            got = outs[out].host()
            for r in range(R):
                if kind == "reduce_scatter":
                    off, L = plan[ring.owned_chunk(R, r)]
                    assert_bitwise_equal(got[r][off:off + L], want[r][off:off + L], f"step {step}")
                else:
                    assert_bitwise_equal(got[r], want[r], f"step {step} rank {r}")
            assert outs[out].guards_intact()


@pytest.mark.parametrize("variant,options", [("direct", ()), ("ring", ()), ("persistent", ()),
                                             ("persistent", (("BARRIER", "CLUSTER"),)), ("local", ())])
def test_calls_inside_a_caller_graph(ra, variant, options):
    """A caller may capture ra_allreduce into its own CUDA graph (after one
    call on the same buffers outside it) and replay it on new data, several
    times: the counting barrier keeps its waiters' shadows in device memory,
    so every replay moves them on."""
    R, n = 4, 100003
    o = elementops.get_op("f32", "sum")
    inp = DeviceRanks(R, n, np.float32, host=inputs.generate(R, n, "f32", "normal", 1))
    out = DeviceRanks(R, n, np.float32)
    h = ra.RingAllReduce(R, n, "f32", "sum", variant=variant)
    for key, value in options:
        h.set_option(ra.Option[key], ra.Barrier[value])
    try:
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            h.allreduce(inp.views, out.views, side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            h.allreduce(inp.views, out.views, side)
        for seed in (7, 8, 9):
            x = inputs.generate(R, n, "f32", "normal", seed)
            inp.big.copy_(DeviceRanks(R, n, np.float32, host=x).big)
            g.replay()
            torch.cuda.synchronize()
            want = ring.ring_allreduce(x, o)
            got = out.host()
            for r in range(R):
                assert_bitwise_equal(got[r], want[r], f"{variant} seed {seed}")
        assert h.device_status()[0] == ra.Status.OK
    finally:
        h.close()



@pytest.mark.parametrize("variant,key,value", [("pipelined", None, None), ("pipelined", "PROTOCOL", "LL"),
                                               ("persistent", "BARRIER", "PER_PEER")])
def test_host_state_launches_replay_from_graphs(ra, variant, key, value):
    """The per-peer barrier's epoch, the pipelined flags' shadow start and the
    LL flag base are handed to each launch by the host, and every CTA keeps
    its own copy in device memory.  A call captured into a CUDA graph -- and
    every call after it -- takes them from there: one call from the host,
    three replays on new data and one more call from the host are all
    bitwise the oracle's, and the signals count all five calls."""
    R, n = 4, 4 * 3001
    o = elementops.get_op("f32", "sum")
    inp = DeviceRanks(R, n, np.float32, host=inputs.generate(R, n, "f32", "normal", 2))
    out = DeviceRanks(R, n, np.float32)
    with ra.RingAllReduce(R, n, "f32", "sum", variant=variant) as h:
        if key:
            h.set_option(ra.Option[key], (ra.Protocol if key == "PROTOCOL" else ra.Barrier)[value])
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            h.allreduce(inp.views, out.views, side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            h.allreduce(inp.views, out.views, side)
        for seed in (7, 8, 9, 10):
            x = inputs.generate(R, n, "f32", "normal", seed)
            inp.big.copy_(DeviceRanks(R, n, np.float32, host=x).big)
            if seed < 10:
                g.replay()
            else:
                h.allreduce(inp.views, out.views)   # from the host again, after the replays
            torch.cuda.synchronize()
            status, err = h.device_status()
            assert status == ra.Status.OK, (seed, err.as_dict())
            want, got = ring.ring_allreduce(x, o), out.host()
            for r in range(R):
                assert_bitwise_equal(got[r], want[r], f"{variant} {value} seed {seed} rank {r}")
        if key != "PROTOCOL":
            calls = 5
            slots = h.read_signals()[0]
            assert slots
            if variant == "pipelined":
                # every flag: 5 calls x 2(R-1) finished rounds
                assert all(v == calls * 2 * (R - 1) for v in slots), slots[:8]
            else:
                # per-peer slots [channel][round][waiter][peer]: each peer added 1 per call;
                # a waiter's own column is never written
                for i, v in enumerate(slots):
                    assert v == (0 if (i // R) % R == i % R else calls), (i, v)


def test_replayed_ll_calls_stop_before_their_flags_wrap(ra):
    """An LL call from the host whose last message carries 2^32 - 3 leaves
    2^32 - 1 as the next base; a replayed call cannot start the flags again
    (it cannot zero the inbox), so it does nothing and reports code 6; the
    status call zeroes the inbox and the next call is correct."""
    R, n = 4, 4 * 1500 + 3
    rounds = 2 * (R - 1)
    o = elementops.get_op("i32", "sum")
    x = inputs.generate(R, n, "i32", "int20", seed=3)
    inp, out = DeviceRanks(R, n, np.int32, host=x), DeviceRanks(R, n, np.int32)
    want = ring.ring_allreduce(x, o)
    with ra.RingAllReduce(R, n, "i32", "sum", variant="pipelined") as h:
        h.set_option(ra.Option.PROTOCOL, ra.Protocol.LL)
        h.set_option(ra.Option.LL_FLAG, 2**32 - 1 - rounds)
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            h.allreduce(inp.views, out.views, side)
        torch.cuda.synchronize()
        assert h.device_status()[0] == ra.Status.OK
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            h.allreduce(inp.views, out.views, side)
        g.replay()
        torch.cuda.synchronize()
        status, err = h.device_status()
        assert status == ra.Status.ERR_TIMEOUT and err.code == 6, err.as_dict()
        assert err.observed == 2**32 - 1
        assert "exhausted" in ra.ra_last_error()
        out2 = DeviceRanks(R, n, np.int32)
        h.allreduce(inp.views, out2.views)
        assert h.device_status()[0] == ra.Status.OK
        got = out2.host()
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], f"after the reset rank {r}")


@pytest.mark.parametrize("dtype,op", DTYPE_OPS)
def test_per_peer_barrier_matches_oracle(ra, dtype, op):
    o = elementops.get_op(dtype, op)
    for i, (R, n) in enumerate(SHAPES):
        x = inputs.generate(R, n, dtype, _dist(dtype), seed=600 + i)
        want = ring.ring_allreduce(x, o)
        got = run_gpu(ra, x, dtype, op, "persistent", options=[(ra.Option.BARRIER, ra.Barrier.PER_PEER)])
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], f"per-peer {dtype}/{op} R={R} n={n} rank {r}")


@pytest.mark.parametrize("slices,window", [(0, 0), (1, 0), (2, 0), (7, 0), (64, 0), (7, 3), (5, 2), (64, 64),
                                           (8, 64)])
def test_pipelined_sub_slices(ra, slices, window):
    """Sub-slice counts and windows (every round over a window of sub-slices
    before the next window; a last window shorter than the others; one window
    over all of them, the round-by-round order)."""
    o = elementops.get_op("bf16", "sum")
    for R, n in ((8, 2**20 + 7), (3, 100003), (16, 2**16 + 3), (4, 2**22 + 5)):
        x = inputs.generate(R, n, "bf16", "grad", seed=slices + 100 * window)
        want = ring.ring_allreduce(x, o)
        got = run_gpu(ra, x, "bf16", "sum", "pipelined",
                      options=[(ra.Option.SLICES, slices), (ra.Option.WINDOW, window)], repeat=2)
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], f"slices={slices} window={window} R={R}")


@pytest.mark.parametrize("R,G", [(2, 1), (5, 3), (8, 4)])
def test_per_peer_slots_and_pipelined_flags(ra, R, G):
    """Per-peer barrier: after k calls every (waiter, peer) slot holds k and
    a waiter's own slot 0.  Pipelined: every (channel, rank, sub-slice) flag
    holds k * rounds."""
    n = R * 7000 + 3
    x = inputs.generate(R, n, "f32", "normal", 9)
    inp = DeviceRanks(R, n, np.float32, host=x)
    want = ring.ring_allreduce(x, elementops.get_op("f32", "sum"))
    for variant in ("persistent", "pipelined"):
        out = DeviceRanks(R, n, np.float32)
        with ra.RingAllReduce(R, n, "f32", "sum", variant=variant) as h:
            h.set_option(ra.Option.CTAS, G)
            if variant == "persistent":
                h.set_option(ra.Option.BARRIER, ra.Barrier.PER_PEER)
            else:
                h.set_option(ra.Option.SLICES, 3)
            for k in range(1, 4):
                h.allreduce(inp.views, out.views)
                slots, ch, rounds, calls = h.read_signals()
                assert (ch, calls) == (G, k)
                if variant == "persistent":
                    assert rounds == barrier.barrier_rounds(R) and len(slots) == G * rounds * R * R
                    for idx, v in enumerate(slots):
                        waiter, peer = (idx // R) % R, idx % R
                        assert v == (0 if waiter == peer else k), (idx, v)
                else:
                    assert rounds == 2 * (R - 1) and len(slots) == G * R * 3
                    assert all(v == k * rounds for v in slots), slots
            assert h.device_status()[0] == ra.Status.OK
        got = out.host()
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], variant)


def test_per_peer_timeout_names_the_missing_peer(ra):
    R, n = 4, 4 * 4096
    x = inputs.generate(R, n, "f32", "normal", 8)
    inp = DeviceRanks(R, n, np.float32, host=x)
    out = DeviceRanks(R, n, np.float32)
    with ra.RingAllReduce(R, n, "f32", "sum", variant="persistent") as h:
        h.set_option(ra.Option.BARRIER, ra.Barrier.PER_PEER)
        h.set_option(ra.Option.TIMEOUT_NS, 20_000_000)
        last = barrier.barrier_rounds(R) - 1
        h.set_option(ra.Option.SKIP_ARRIVAL, (2 << 16) | last)
        h.allreduce(inp.views, out.views)
        status, err = h.device_status()
        assert status == ra.Status.ERR_TIMEOUT
        assert err.code == 3 and err.round == last and err.rank != 2
        assert err.peer == 2, "a per-peer slot names the rank that did not arrive"
        assert err.expected - err.observed == 1
        h.set_option(ra.Option.SKIP_ARRIVAL, -1)
        h.allreduce(inp.views, out.views)
        assert h.device_status()[0] == ra.Status.OK
    want = ring.ring_allreduce(x, elementops.get_op("f32", "sum"))
    got = out.host()
    for r in range(R):
        assert_bitwise_equal(got[r], want[r])


def test_pipelined_timeout_names_the_predecessor(ra):
    """A rank that stops publishing progress from the next-to-last round on
    leaves exactly its successor waiting in the last round."""
    R, n = 4, 4 * 4096
    x = inputs.generate(R, n, "f32", "normal", 8)
    inp = DeviceRanks(R, n, np.float32, host=x)
    out = DeviceRanks(R, n, np.float32)
    rounds = 2 * (R - 1)
    with ra.RingAllReduce(R, n, "f32", "sum", variant="pipelined") as h:
        h.set_option(ra.Option.TIMEOUT_NS, 20_000_000)
        h.set_option(ra.Option.SKIP_ARRIVAL, (2 << 16) | (rounds - 2))
        h.allreduce(inp.views, out.views)
        status, err = h.device_status()
        assert status == ra.Status.ERR_TIMEOUT
        assert err.code == 4 and err.rank == 3 and err.peer == 2 and err.round == rounds - 1
        assert err.expected - err.observed == 1
        h.set_option(ra.Option.SKIP_ARRIVAL, -1)
        h.allreduce(inp.views, out.views)
        assert h.device_status()[0] == ra.Status.OK
    want = ring.ring_allreduce(x, elementops.get_op("f32", "sum"))
    got = out.host()
    for r in range(R):
        assert_bitwise_equal(got[r], want[r])



@pytest.mark.parametrize("dtype,op", DTYPE_OPS)
def test_compact_reduce_scatter_and_all_gather(ra, dtype, op):
    """Compact outputs / inputs (rank r: chunk (r+1) mod R only), on plans
    whose chunk starts are 16-byte aligned (direct kernel, shifted pointers)
    and on ragged ones (element-wide kernel), every element compared."""
    o = elementops.get_op(dtype, op)
    st = inputs.storage_dtype(dtype)
    for i, (R, n) in enumerate(SHAPES + [(4, 4096 + 8), (6, 6 * 64 * 1024)]):
        x = inputs.generate(R, n, dtype, _dist(dtype), seed=700 + i)
        lengths = [ring.chunk_plan(R, n)[ring.owned_chunk(R, r)][1] for r in range(R)]
        want_rs = ring.ring_reduce_scatter_compact(x, o)
        want_ag = ring.ring_all_gather_compact(want_rs, n, o)
        inp = DeviceRanks(R, n, st, host=x)
        cmp = DeviceBuffers(lengths, st)
        full = DeviceRanks(R, n, st)
        with ra.RingAllReduce(R, n, dtype, op) as h:
            h.reduce_scatter_compact(inp.ptrs(), cmp.ptrs())
            h.all_gather_compact(cmp.ptrs(), full.ptrs())
            assert h.device_status()[0] == ra.Status.OK
        assert inp.guards_intact() and cmp.guards_intact() and full.guards_intact()
        got_rs, got_ag = cmp.host(), full.host()
        for r in range(R):
            assert_bitwise_equal(got_rs[r], want_rs[r], f"RS {dtype}/{op} R={R} n={n} rank {r}")
            assert_bitwise_equal(got_ag[r], want_ag[r], f"AG {dtype}/{op} R={R} n={n} rank {r}")



def test_prepared_calls_match_oracle(ra):
    """RingAllReduce.prepare marshals once; repeated calls read the buffers'
    current contents."""
    R, n = 8, 2**16 + 5
    o = elementops.get_op("f32", "sum")
    inp = DeviceRanks(R, n, np.float32)
    out = DeviceRanks(R, n, np.float32)
    for variant in VARIANTS:
        with ra.RingAllReduce(R, n, "f32", "sum", variant=variant) as h:
            call = h.prepare("allreduce", inp.views, out.views)
            for seed in (1, 2):
                x = inputs.generate(R, n, "f32", "normal", seed)
                inp.big.copy_(DeviceRanks(R, n, np.float32, host=x).big)
                call()
                assert h.device_status()[0] == ra.Status.OK
                want = ring.ring_allreduce(x, o)
                got = out.host()
                for r in range(R):
                    assert_bitwise_equal(got[r], want[r], f"{variant} seed {seed}")
            with pytest.raises(ValueError):
                h.prepare("allreduce", inp.views[:3], out.views)


@pytest.mark.parametrize("gather", [1, 2])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f64"])
def test_all_gather_kernels(ra, gather, dtype):
    """Both AllGather kernels of the direct variant (16-byte vectors; TMA
    broadcast through shared memory), in place and compact, bitwise."""
    o = elementops.get_op(dtype, "sum")
    st = inputs.storage_dtype(dtype)
    for i, (R, n) in enumerate(SHAPES + [(8, 8 * 40000), (4, 4 * 16384 * 3 + 8)]):
        x = inputs.generate(R, n, dtype, _dist(dtype), seed=800 + i)
        rs = ring.ring_reduce_scatter(x, o, fill=np.zeros(1, st)[0])
        want = ring.ring_all_gather(rs, o)
        got = run_gpu(ra, rs, dtype, "sum", "direct", kind="all_gather", inplace=True,
                      options=[(ra.Option.GATHER, gather)])
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], f"gather={gather} {dtype} R={R} n={n} rank {r}")
        chunks = ring.ring_reduce_scatter_compact(x, o)
        lengths = [len(c) for c in chunks]
        cmp = DeviceBuffers(lengths, st, host=chunks)
        full = DeviceRanks(R, n, st)
        with ra.RingAllReduce(R, n, dtype, "sum") as h:
            h.set_option(ra.Option.GATHER, gather)
            h.all_gather_compact(cmp.ptrs(), full.ptrs())
            assert h.device_status()[0] == ra.Status.OK
        assert cmp.guards_intact() and full.guards_intact()
        got = full.host()
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], f"compact gather={gather} {dtype} R={R} n={n} rank {r}")



@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("bf16", "sum"), ("i32", "max"), ("f64", "sum")])
def test_cluster_barrier_matches_oracle(ra, dtype, op):
    """Persistent variant with each channel's R CTAs in one thread-block
    cluster (hardware cluster barrier between rounds); R <= 16."""
    o = elementops.get_op(dtype, op)
    for i, (R, n) in enumerate(SHAPES):
        x = inputs.generate(R, n, dtype, _dist(dtype), seed=900 + i)
        opts = [(ra.Option.BARRIER, ra.Barrier.CLUSTER)]
        if R > 16:
            with pytest.raises(ra.RAError) as e:
                run_gpu(ra, x, dtype, op, "persistent", options=opts)
            assert e.value.status == ra.Status.ERR_UNSUPPORTED
            continue
        for kind in ("allreduce", "reduce_scatter"):
            got = run_gpu(ra, x, dtype, op, "persistent", kind=kind, options=opts)
            if kind == "allreduce":
                want = ring.ring_allreduce(x, o)
                for r in range(R):
                    assert_bitwise_equal(got[r], want[r], f"cluster {dtype}/{op} R={R} n={n} rank {r}")
            else:
                want = ring.ring_reduce_scatter(x, o)
                plan = ring.chunk_plan(R, n)
                for r in range(R):
                    off, L = plan[ring.owned_chunk(R, r)]
                    assert_bitwise_equal(got[r][off:off + L], want[r][off:off + L], f"cluster RS R={R} n={n}")
