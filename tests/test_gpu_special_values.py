"""IEEE edge cases on the GPU: signed zeros, subnormals, the smallest normal,
rounding ties, overflow to infinity, infinities and NaN in the rank inputs,
for every floating-point dtype, both ops and every variant, through the C ABI,
compared element by element with the oracle.

Every result that is a number (infinities included) must match the oracle
bitwise: the fold order is the ring's and each hop is one correctly rounded
operation, with no flush of subnormals.  Where the oracle's sum is NaN the
GPU's must be NaN too; its bits are not compared, because IEEE 754 leaves the
payload of a NaN produced by an addition to the implementation.  MAX moves
inputs only (the incoming partial is kept unless the local value is
strictly greater), so its results, NaN included, are compared bitwise.

Shapes: an aligned chunk plan, and two ragged ones whose chunk starts are
off 16 bytes for every element width (element-wide head and tail paths)."""

import numpy as np
import pytest

from oracle import elementops, ring
from ring_allreduce_gb300 import inputs
from rahelpers import DeviceBuffers, DeviceRanks, assert_bitwise_equal

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

# the pipelined variant also with its flag-in-data protocols, whose words
# split 8-byte elements into two 32-bit halves
VARIANTS = ["direct", "ring", "persistent", "pipelined", "local", "pipelined-LL", "pipelined-LL_CLUSTER"]


def _handle(ra, R, n, dtype, op, variant):
    v, _, protocol = variant.partition("-")
    h = ra.RingAllReduce(R, n, dtype, op, variant=v)
    if protocol:
        h.set_option(ra.Option.PROTOCOL, ra.Protocol[protocol])
    return h
FLOAT_DTYPES = ["f32", "bf16", "f16", "f64"]
SHAPES = [(8, 8192), (5, 4099), (3, 65539)]


@pytest.fixture(scope="module")
def ra():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_gb300 import build
    build.build()
    from ring_allreduce_gb300 import binding
    return binding


def _as_float(a, dtype):
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return a


def assert_matches(got, want, dtype, op, what):
    got, want = np.ascontiguousarray(got), np.ascontiguousarray(want)
    if op == "max":
        assert_bitwise_equal(got, want, what)
        return
    gf, wf = _as_float(got, dtype), _as_float(want, dtype)
    nan_w, nan_g = np.isnan(wf), np.isnan(gf)
    bad = np.nonzero(nan_w != nan_g)[0]
    assert len(bad) == 0, f"{what}: NaN where the oracle has none, or the reverse, at {bad[:8].tolist()}"
    keep = ~nan_w
    assert_bitwise_equal(got[keep], want[keep], what)


def _inputs(R, n, dtype, seed):
    x = inputs.generate(R, n, dtype, "special", seed)
    # the draw must reach what this test is about
    f = np.concatenate([_as_float(v, dtype) for v in x]).astype(np.float64)
    tiny = np.finfo(np.float32 if dtype in ("f32", "bf16") else
                    (np.float16 if dtype == "f16" else np.float64)).tiny
    assert np.isnan(f).any() and np.isinf(f).any() and (f == 0).any()
    assert ((f != 0) & (np.abs(f) < tiny)).any(), "no subnormal drawn"
    return x


def _oracle(fn, x, op):
    with np.errstate(all="ignore"):   # inf - inf and overflow are part of the test
        return fn(x, op)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("op", ["sum", "max"])
@pytest.mark.parametrize("dtype", FLOAT_DTYPES)
def test_allreduce_special_values(ra, dtype, op, variant):
    for si, (R, n) in enumerate(SHAPES):
        x = _inputs(R, n, dtype, 100 + si)
        want = _oracle(ring.ring_allreduce, x, elementops.get_op(dtype, op))
        st = inputs.storage_dtype(dtype)
        inp, out = DeviceRanks(R, n, st, host=x), DeviceRanks(R, n, st)
        with _handle(ra, R, n, dtype, op, variant) as h:
            h.allreduce(inp.views, out.views)
            status, err = h.device_status()
            assert status == ra.Status.OK, err.as_dict()
        torch.cuda.synchronize()
        assert inp.guards_intact() and out.guards_intact()
        got = out.host()
        for r in range(R):
            assert_matches(got[r], want[r], dtype, op, f"{variant} {dtype} {op} R={R} n={n} rank {r}")
        # the special values must not all have vanished into NaN
        wf = _as_float(want[0], dtype)
        assert np.isfinite(wf).mean() > 0.2


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype", FLOAT_DTYPES)
def test_reduce_scatter_special_values(ra, dtype, variant):
    op = "sum"
    R, n = 5, 4099
    x = _inputs(R, n, dtype, 200)
    want = _oracle(ring.ring_reduce_scatter, x, elementops.get_op(dtype, op))
    st = inputs.storage_dtype(dtype)
    inp, out = DeviceRanks(R, n, st, host=x), DeviceRanks(R, n, st)
    with _handle(ra, R, n, dtype, op, variant) as h:
        h.reduce_scatter(inp.views, out.views)
        assert h.device_status()[0] == ra.Status.OK
    got = out.host()
    plan = ring.chunk_plan(R, n)
    for r in range(R):
        off, L = plan[ring.owned_chunk(R, r)]
        assert_matches(got[r][off:off + L], want[r][off:off + L], dtype, op, f"{variant} {dtype} rank {r}")


@pytest.mark.parametrize("dtype", FLOAT_DTYPES)
def test_compact_reduce_scatter_special_values(ra, dtype):
    op = "sum"
    for R, n in SHAPES:
        x = _inputs(R, n, dtype, 300 + R)
        want = _oracle(ring.ring_reduce_scatter, x, elementops.get_op(dtype, op))
        st = inputs.storage_dtype(dtype)
        inp = DeviceRanks(R, n, st, host=x)
        plan = ring.chunk_plan(R, n)
        owned = [plan[ring.owned_chunk(R, r)] for r in range(R)]
        cmp = DeviceBuffers([L for _, L in owned], st)
        with ra.RingAllReduce(R, n, dtype, op) as h:
            h.reduce_scatter_compact(inp.views, cmp.views)
            assert h.device_status()[0] == ra.Status.OK
        torch.cuda.synchronize()
        assert cmp.guards_intact()
        got = cmp.host()
        for r, (off, L) in enumerate(owned):
            assert_matches(got[r], want[r][off:off + L], dtype, op, f"compact {dtype} R={R} rank {r}")
