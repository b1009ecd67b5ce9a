"""The named workloads at their full sizes, every element compared bitwise
with the oracle (tolerance 0 ulp), in the launch configuration bench.py
times (default options), for every variant:

  r4_small   R=4,  n=4096 fp32, integers in [-8, 8]: ReduceScatter then
             AllGather, and the placement GPU0:S1, GPU1:S2, GPU2:S3, GPU3:S0
  r8_f32     R=8,  n=2^24 fp32 N(0,1)
  r8_bf16    R=8,  n=2^26+3 bf16 (ragged last chunk), bf16 rounding per hop
  r16_i32    R=16, n=2^24 int32, sum and max
  sweep      R=8 fp32 for n = 2^10 .. 2^26, and R in {2,4,16,32} at 2^24
"""

import numpy as np
import pytest

from oracle import elementops, ring
from ring_allreduce_gb300 import inputs
from rahelpers import DeviceRanks, assert_bitwise_equal

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")

VARIANTS = ["direct", "ring", "persistent", "pipelined", "local"]
# the pipelined variant's flag-in-data protocols, for the small calls they are for
SMALL_VARIANTS = VARIANTS + ["pipelined-LL", "pipelined-LL_CLUSTER"]


def _handle(ra, R, n, dtype, op, variant):
    v, _, protocol = variant.partition("-")
    h = ra.RingAllReduce(R, n, dtype, op, variant=v)
    if protocol:
        h.set_option(ra.Option.PROTOCOL, ra.Protocol[protocol])
    return h


@pytest.fixture(scope="module")
def ra():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_gb300 import build
    build.build()
    from ring_allreduce_gb300 import binding
    return binding


def _check_allreduce(ra, x, dtype, op, variants, want=None):
    R, n = len(x), len(x[0])
    want = want if want is not None else ring.ring_allreduce(x, elementops.get_op(dtype, op))
    st = inputs.storage_dtype(dtype)
    inp = DeviceRanks(R, n, st, host=x)
    for v in variants:
        out = DeviceRanks(R, n, st)
        with _handle(ra, R, n, dtype, op, v) as h:
            h.allreduce(inp.views, out.views)
            status, err = h.device_status()
            assert status == ra.Status.OK, err.as_dict()
        assert inp.guards_intact() and out.guards_intact()
        got = out.host()
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], f"{v} {dtype}/{op} R={R} n={n} rank {r}")
        del out
    del inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", SMALL_VARIANTS)
def test_r4_small_placement_and_allgather(ra, variant):
    x = inputs.workload_inputs("r4_small")
    op = elementops.get_op("f32", "sum")
    R, n = 4, 4096
    S = ring.ring_allreduce(x, op)[0]
    inp = DeviceRanks(R, n, np.float32, host=x)
    out = DeviceRanks(R, n, np.float32)
    with _handle(ra, R, n, "f32", "sum", variant) as h:
        h.reduce_scatter(inp.views, out.views)
        assert h.device_status()[0] == ra.Status.OK
        rs = out.host()
        # GPU0 holds S1, GPU1 S2, GPU2 S3, GPU3 S0 (chunks of 1024 elements)
        for r, k in enumerate([1, 2, 3, 0]):
            assert h.owned_chunk(r) == (k * 1024, 1024)
            assert_bitwise_equal(rs[r][k * 1024:(k + 1) * 1024], S[k * 1024:(k + 1) * 1024], f"GPU{r} S{k}")
        h.all_gather(out.views)
        assert h.device_status()[0] == ra.Status.OK
    ag = out.host()
    for r in range(R):
        assert_bitwise_equal(ag[r], S, f"rank {r}")
    assert out.guards_intact()


def test_r8_f32(ra):
    x = inputs.workload_inputs("r8_f32")
    _check_allreduce(ra, x, "f32", "sum", VARIANTS)


def test_r8_bf16_ragged(ra):
    x = inputs.workload_inputs("r8_bf16")
    plan = ring.chunk_plan(8, 2**26 + 3)
    assert plan[7][1] == 8388604
    _check_allreduce(ra, x, "bf16", "sum", VARIANTS)


@pytest.mark.parametrize("op", ["sum", "max"])
def test_r16_i32(ra, op):
    x = inputs.workload_inputs("r16_i32")
    _check_allreduce(ra, x, "i32", op, VARIANTS)


@pytest.mark.parametrize("n", inputs.SWEEP_N)
def test_sweep_r8_f32(ra, n):
    x = inputs.generate(8, n, "f32", "normal", inputs.SWEEP_SEED)
    _check_allreduce(ra, x, "f32", "sum", SMALL_VARIANTS if n <= 2**18 else VARIANTS)


@pytest.mark.parametrize("R", [R for R in inputs.SWEEP_R if R != 8])
def test_sweep_ranks_f32(ra, R):
    x = inputs.generate(R, 2**24, "f32", "normal", inputs.SWEEP_SEED)
    _check_allreduce(ra, x, "f32", "sum", VARIANTS)
