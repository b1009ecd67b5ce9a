"""ra_allreduce_noalloc: the AllReduce for callers that may not allocate
device memory -- code whose device memory belongs to another allocator (a
framework's caching allocator, a host that gives plug-ins a fixed budget)
and may not call cudaMalloc, and code that cannot take cudaFree's
device-wide synchronisation.  It takes its scratch (barrier signal slots and
error record) from a fixed array inside the library instead of from
ra_create.

Checked here through the C ABI: two calls in a row give, bitwise, what the
oracle's ring simulation gives on the same inputs, and what the handle-based
ra_allreduce gives (the tolerance of every parity test here is 0 ulp), leave
the guard bands around every buffer alone, and the second call does not
change the device's free memory.  One case is large enough that the array's
size, not the GPU, limits the channel count (R = 32: 8 channels), so the
signals and shadows at the array's far end are used.  This file is collected
last, so a stop at the first failure has run everything else.
"""

import ctypes

import numpy as np
import pytest

from oracle import elementops, ring
from ring_allreduce_gb300 import inputs
from rahelpers import DeviceRanks, assert_bitwise_equal

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

CASES = [  # (R, n, dtype, op): ragged n, several channels, three dtypes
    (8, 2**20 + 7, "f32", "sum"),
    (5, 300001, "bf16", "sum"),
    (16, 2**18 + 3, "i32", "max"),
    (32, 2**22 + 5, "f32", "sum"),   # 8 channels: the array's size is the limit
]


@pytest.fixture(scope="module")
def ra():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_gb300 import build
    build.build()
    from ring_allreduce_gb300 import binding
    return binding


def _ptrs(ranks):
    arr = (ctypes.c_void_p * ranks.R)()
    for r, p in enumerate(ranks.ptrs()):
        arr[r] = p
    return arr


@pytest.mark.parametrize("R,n,dtype,op", CASES)
def test_noalloc_matches_allreduce_two_calls_in_a_row(ra, R, n, dtype, op):
    dist = {"f32": "normal", "bf16": "grad", "i32": "int20"}[dtype]
    x = inputs.generate(R, n, dtype, dist, seed=2024 + R)
    st = inputs.storage_dtype(dtype)
    inp = DeviceRanks(R, n, st, host=x)

    # the oracle's ring, and the existing entry point through a handle
    want = ring.ring_allreduce(x, elementops.get_op(dtype, op))
    ref_out = DeviceRanks(R, n, st)
    with ra.RingAllReduce(R, n, dtype, op) as h:
        h.allreduce(inp.views, ref_out.views)
        status, err = h.device_status()
        assert status == ra.Status.OK, err.as_dict()
    handle = ref_out.host()

    outs = [DeviceRanks(R, n, st) for _ in range(2)]   # allocated before either call
    lib = ra.load_library()
    dt = int(ra.DType[dtype.upper()])
    o = int(ra.Op[op.upper()])
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    for call, out in enumerate(outs):
        free_before = torch.cuda.mem_get_info()[0]
        rc = lib.ra_allreduce_noalloc(R, n, dt, o, _ptrs(inp), _ptrs(out), stream)
        assert rc == ra.Status.OK, ra.ra_last_error()
        torch.cuda.synchronize()
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free_before, "second call changed free device memory"
        assert inp.guards_intact() and out.guards_intact(), f"call {call}: write outside a buffer"
        got = out.host()
        for r in range(R):
            assert_bitwise_equal(got[r], want[r], f"call {call} {dtype}/{op} R={R} n={n} rank {r} vs the oracle")
            assert_bitwise_equal(got[r], handle[r], f"call {call} {dtype}/{op} R={R} n={n} rank {r} vs ra_allreduce")


def test_noalloc_rejects_bad_arguments(ra):
    lib = ra.load_library()
    inp = DeviceRanks(4, 1024, np.float32)
    out = DeviceRanks(4, 1024, np.float32)
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.ra_allreduce_noalloc(1, 1024, 0, 0, _ptrs(inp), _ptrs(out), stream) == ra.Status.ERR_INVALID
    assert lib.ra_allreduce_noalloc(33, 1024, 0, 0, _ptrs(inp), _ptrs(out), stream) == ra.Status.ERR_INVALID
    assert lib.ra_allreduce_noalloc(4, 1024, 9, 0, _ptrs(inp), _ptrs(out), stream) == ra.Status.ERR_INVALID
    bad = _ptrs(out)
    bad[1] = bad[0]
    assert lib.ra_allreduce_noalloc(4, 1024, 0, 0, _ptrs(inp), bad, stream) == ra.Status.ERR_INVALID
    assert "overlap" in ra.ra_last_error()
    # more than 2^40 elements: rejected before n * element size is formed
    assert lib.ra_allreduce_noalloc(4, 2**40 + 1, 0, 0, _ptrs(inp), _ptrs(out), stream) == ra.Status.ERR_INVALID
    assert "2^40" in ra.ra_last_error()
    # host memory (a numpy array) and an address CUDA does not know: rejected on
    # the host, nothing is launched
    host = np.zeros(4 * 1024 + 16, dtype=np.float32)
    base = (host.ctypes.data + 15) // 16 * 16
    bad = _ptrs(out)
    bad[2] = base
    assert lib.ra_allreduce_noalloc(4, 1024, 0, 0, _ptrs(inp), bad, stream) == ra.Status.ERR_INVALID
    assert "out[2]" in ra.ra_last_error()
    bad = _ptrs(inp)
    bad[3] = 0x10000   # 16-byte aligned, never allocated
    assert lib.ra_allreduce_noalloc(4, 1024, 0, 0, bad, _ptrs(out), stream) == ra.Status.ERR_INVALID
    assert "in[3]" in ra.ra_last_error()
    torch.cuda.synchronize()
    assert inp.guards_intact() and out.guards_intact()
