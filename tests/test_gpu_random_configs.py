"""Seeded random configurations through every entry point: variant, dtype and
op, R from 1 to 32, n from 0 to a few hundred thousand (ragged, tiny, n < R),
in place or not, and the collective (AllReduce, ReduceScatter, AllGather,
AllReduce of host buffers).  Each one is compared bitwise with the oracle on
its own seeded inputs; the configuration list itself comes from a fixed seed,
so a failure names a configuration that can be rerun alone."""

import numpy as np
import pytest

from oracle import elementops, ring
from ring_allreduce_gb300 import inputs
from rahelpers import DeviceRanks, assert_bitwise_equal

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

VARIANTS = ["direct", "ring", "persistent", "pipelined", "local"]
DTYPE_OPS = [("f32", "sum"), ("f32", "max"), ("bf16", "sum"), ("bf16", "max"),
             ("i32", "sum"), ("i32", "max"), ("f16", "sum"), ("f16", "max"),
             ("f64", "sum"), ("f64", "max"), ("i64", "sum"), ("i64", "max")]
KINDS = ["allreduce", "reduce_scatter", "all_gather", "allreduce_host"]
DIST = {"f32": "normal", "bf16": "grad", "i32": "int20", "f16": "grad", "f64": "normal", "i64": "int40"}


def _configs(count=200, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        R = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 11, 16, 23, 32]))
        n = int(rng.choice([0, 1, 2, R - 1, R, 3 * R + 1, int(rng.integers(1, 5000)),
                            int(rng.integers(5000, 300000))]))
        n = max(n, 0)
        dtype, op = DTYPE_OPS[int(rng.integers(len(DTYPE_OPS)))]
        variant = VARIANTS[int(rng.integers(len(VARIANTS)))]
        kind = KINDS[int(rng.integers(len(KINDS)))]
        inplace = bool(rng.integers(2)) and kind in ("allreduce", "reduce_scatter")
        out.append((i, R, n, dtype, op, variant, kind, inplace))
    return out


@pytest.fixture(scope="module")
def ra():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_gb300 import build
    build.build()
    from ring_allreduce_gb300 import binding
    return binding


def _ll_configs(count=80, seed=20261203):
    """The pipelined variant's flag-in-data protocols: LL (R up to 32) and
    LL_CLUSTER (R up to 16), n within their limits (the LL inbox, the
    cluster's shared memory), every collective but host buffers."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        protocol = ["LL", "LL_CLUSTER"][int(rng.integers(2))]
        Rs = [2, 3, 4, 5, 7, 8, 11, 16] + ([23, 32] if protocol == "LL" else [])
        R = int(rng.choice(Rs))
        n = int(rng.choice([1, 2, R - 1, R, 3 * R + 1, int(rng.integers(1, 5000)), int(rng.integers(5000, 60000))]))
        n = max(n, 1)
        dtype, op = DTYPE_OPS[int(rng.integers(len(DTYPE_OPS)))]
        kind = KINDS[int(rng.integers(3))]
        inplace = bool(rng.integers(2)) and kind in ("allreduce", "reduce_scatter")
        out.append((1000 + i, R, n, dtype, op, "pipelined-" + protocol, kind, inplace))
    return out


@pytest.mark.parametrize("cfg", _configs(), ids=lambda c: "-".join(str(v) for v in c))
def test_random_configuration(ra, cfg):
    _run_configuration(ra, cfg)


@pytest.mark.parametrize("cfg", _ll_configs(), ids=lambda c: "-".join(str(v) for v in c))
def test_random_ll_configuration(ra, cfg):
    _run_configuration(ra, cfg)


def _run_configuration(ra, cfg):
    i, R, n, dtype, op, variant, kind, inplace = cfg
    o = elementops.get_op(dtype, op)
    x = inputs.generate(R, n, dtype, DIST[dtype], seed=7000 + i)
    st = inputs.storage_dtype(dtype)
    plan = ring.chunk_plan(R, n)
    variant, _, protocol = variant.partition("-")
    with ra.RingAllReduce(R, n, dtype, op, variant=variant) as h:
        if protocol:
            h.set_option(ra.Option.PROTOCOL, ra.Protocol[protocol])
        if kind == "allreduce_host":
            ins = [torch.from_numpy(v.view(f"i{v.dtype.itemsize}").copy()).pin_memory() for v in x]
            outs = [torch.zeros_like(t).pin_memory() for t in ins]
            h.allreduce_host(ins, outs)
            torch.cuda.synchronize()
            got = [t.numpy().view(st) for t in outs]
            want = ring.ring_allreduce(x, o)
            for r in range(R):
                assert_bitwise_equal(got[r], want[r], f"cfg {cfg} rank {r}")
            return
        if kind == "all_gather":
            # the layout ReduceScatter leaves, with junk around each owned chunk
            rs = ring.ring_reduce_scatter(x, o)
            junk = inputs.generate(R, n, dtype, DIST[dtype], seed=8000 + i)
            buf = []
            for r in range(R):
                b = junk[r].copy()
                off, L = plan[ring.owned_chunk(R, r)]
                b[off:off + L] = rs[r][off:off + L]
                buf.append(b)
            dev = DeviceRanks(R, n, st, host=buf)
            h.all_gather(dev.views)
            status, err = h.device_status()
            assert status == ra.Status.OK, err.as_dict()
            torch.cuda.synchronize()
            assert dev.guards_intact()
            got, want = dev.host(), ring.ring_all_gather(buf, o)
            for r in range(R):
                assert_bitwise_equal(got[r], want[r], f"cfg {cfg} rank {r}")
            return
        inp = DeviceRanks(R, n, st, host=x)
        out = inp if inplace else DeviceRanks(R, n, st)
        if kind == "allreduce":
            h.allreduce(inp.views, out.views)
        else:
            h.reduce_scatter(inp.views, out.views)
        status, err = h.device_status()
        assert status == ra.Status.OK, err.as_dict()
        torch.cuda.synchronize()
        assert inp.guards_intact() and out.guards_intact()
        got = out.host()
        if kind == "allreduce":
            want = ring.ring_allreduce(x, o)
            for r in range(R):
                assert_bitwise_equal(got[r], want[r], f"cfg {cfg} rank {r}")
        else:
            want = ring.ring_reduce_scatter(x, o)
            for r in range(R):
                off, L = plan[ring.owned_chunk(R, r)]
                assert_bitwise_equal(got[r][off:off + L], want[r][off:off + L], f"cfg {cfg} rank {r}")
