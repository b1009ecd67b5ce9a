"""Sizes past 32-bit element indices, and handles used concurrently.

n = 2^31 + 3 int32 elements per rank (8 GiB per buffer, ragged chunks that
straddle the 2^31 boundary): too large for the CPU oracle, so the inputs are
built on the device from a closed form, x_0[i] = i mod 1000 and x_1[i] = 7,
whose sum S[i] = (i mod 1000) + 7 and maximum are known exactly; outputs are
compared with them on the device (torch only verifies here).  Every
variant, in place and not."""

import numpy as np
import pytest

from oracle import elementops, ring
from ring_allreduce_gb300 import inputs
from rahelpers import DeviceRanks, assert_bitwise_equal

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

VARIANTS = ["direct", "ring", "persistent", "pipelined", "local"]


@pytest.fixture(scope="module")
def ra():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_gb300 import build
    build.build()
    from ring_allreduce_gb300 import binding
    return binding


@pytest.mark.slow
def test_past_int32_indices(ra):
    R, n = 2, 2**31 + 3
    free, _ = torch.cuda.mem_get_info()
    if free < 8 * n * 4 + (4 << 30):
        pytest.skip("needs about 70 GiB of free device memory")
    idx = torch.arange(n, device="cuda", dtype=torch.int64)
    x0 = (idx % 1000).to(torch.int32)
    del idx
    x1 = torch.full((n,), 7, device="cuda", dtype=torch.int32)
    want_sum = x0 + 7
    want_max = torch.maximum(x0, x1)
    out = [torch.empty(n, device="cuda", dtype=torch.int32) for _ in range(R)]
    for variant in VARIANTS:
        for op, want in (("sum", want_sum), ("max", want_max)):
            with ra.RingAllReduce(R, n, "i32", op, variant=variant) as h:
                for o in out:
                    o.fill_(-1)
                h.allreduce([x0, x1], out)
                assert h.device_status()[0] == ra.Status.OK
                for r in range(R):
                    assert torch.equal(out[r], want), f"{variant} {op} rank {r}"
    # in place, sum: the inputs become the result
    with ra.RingAllReduce(R, n, "i32", "sum") as h:
        h.allreduce([x0, x1], [x0, x1])
        assert h.device_status()[0] == ra.Status.OK
        assert torch.equal(x0, want_sum) and torch.equal(x1, want_sum)


def test_two_handles_on_two_streams(ra):
    """Handles keep no shared state: two collectives on two streams at once
    (a direct and a persistent one) both give the oracle's bits."""
    R, n = 8, 2**20 + 7
    o = elementops.get_op("f32", "sum")
    xa = inputs.generate(R, n, "f32", "normal", 31)
    xb = inputs.generate(R, n, "f32", "normal", 32)
    ia, ib = DeviceRanks(R, n, np.float32, host=xa), DeviceRanks(R, n, np.float32, host=xb)
    oa, ob = DeviceRanks(R, n, np.float32), DeviceRanks(R, n, np.float32)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with ra.RingAllReduce(R, n, "f32", "sum", variant="direct") as ha, \
            ra.RingAllReduce(R, n, "f32", "sum", variant="pipelined") as hb:
        for _ in range(5):
            ha.allreduce(ia.views, oa.views, sa)
            hb.allreduce(ib.views, ob.views, sb)
        assert ha.device_status(sa)[0] == ra.Status.OK
        assert hb.device_status(sb)[0] == ra.Status.OK
    wa, wb = ring.ring_allreduce(xa, o), ring.ring_allreduce(xb, o)
    ga, gb = oa.host(), ob.host()
    for r in range(R):
        assert_bitwise_equal(ga[r], wa[r], f"stream a rank {r}")
        assert_bitwise_equal(gb[r], wb[r], f"stream b rank {r}")
