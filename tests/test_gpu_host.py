"""ra_allreduce_host: AllReduce of R buffers in host memory through the
library's device copies, window by window (copy in, fold, copy out on three
streams).  Results are compared bitwise with the oracle, for every dtype and
op, on page-locked and pageable buffers, in place, across window boundaries
(up to the 8-window case with a ragged last window), and for calls issued
back to back on one handle, whose windows overlap."""

import numpy as np
import pytest

from oracle import elementops, ring
from ring_allreduce_gb300 import inputs
from rahelpers import assert_bitwise_equal

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

DTYPE_OPS = [("f32", "sum"), ("f32", "max"), ("bf16", "sum"), ("bf16", "max"),
             ("i32", "sum"), ("i32", "max"), ("f16", "sum"), ("f16", "max"),
             ("f64", "sum"), ("f64", "max"), ("i64", "sum"), ("i64", "max")]
# (R, n): degenerate, ragged, one window by default; the window boundaries are
# exercised with RA_OPT_HOST_WINDOWS below
SHAPES = [(2, 1), (3, 1001), (8, 8 * 1024 + 13), (13, 77777), (4, 2**21 + 5), (2, 2**22 + 3)]


@pytest.fixture(scope="module")
def ra():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_gb300 import build
    build.build()
    from ring_allreduce_gb300 import binding
    return binding


def _dist(dtype):
    return {"f32": "normal", "bf16": "grad", "i32": "int20", "f16": "grad", "f64": "normal", "i64": "int40"}[dtype]


def _pinned(arr):
    """A page-locked torch CPU tensor holding the bytes of a numpy array."""
    ints = arr.view(f"i{arr.dtype.itemsize}")
    return torch.from_numpy(ints.copy()).pin_memory()


def _host(t, like):
    return t.numpy().view(like.dtype)


@pytest.mark.parametrize("dtype,op", DTYPE_OPS)
def test_host_buffers_match_oracle(ra, dtype, op):
    o = elementops.get_op(dtype, op)
    for i, (R, n) in enumerate(SHAPES):
        if dtype not in ("f32", "bf16") and n > 2**20:
            continue   # the windowed cases once per element width class
        x = inputs.generate(R, n, dtype, _dist(dtype), seed=500 + i)
        want = ring.ring_allreduce(x, o)
        ins = [_pinned(v) for v in x]
        outs = [_pinned(np.zeros_like(v)) for v in x]
        stream = torch.cuda.Stream()
        with ra.RingAllReduce(R, n, dtype, op) as h:
            h.allreduce_host(ins, outs, stream)
            stream.synchronize()
            assert h.device_status()[0] == ra.Status.OK
        for r in range(R):
            assert_bitwise_equal(_host(outs[r], x[r]), want[r], f"{dtype}/{op} R={R} n={n} rank {r}")
            assert_bitwise_equal(_host(ins[r], x[r]), x[r], "inputs untouched")


def test_host_pageable_and_in_place(ra):
    o = elementops.get_op("bf16", "sum")
    R, n = 8, 2**20 + 3
    x = inputs.generate(R, n, "bf16", "grad", seed=510)
    want = ring.ring_allreduce(x, o)
    ins = [v.copy() for v in x]                       # plain numpy: pageable memory
    outs = [np.empty_like(v) for v in x]
    with ra.RingAllReduce(R, n, "bf16", "sum") as h:
        h.allreduce_host(ins, outs)
        torch.cuda.synchronize()
        for r in range(R):
            assert_bitwise_equal(outs[r], want[r], f"pageable rank {r}")
        h.allreduce_host(ins, ins)                    # in place
        torch.cuda.synchronize()
    for r in range(R):
        assert_bitwise_equal(ins[r], want[r], f"in place rank {r}")


@pytest.mark.parametrize("windows", [0, 2, 5, 8])
def test_host_windows_ragged(ra, windows):
    """32 MiB per rank in 1 (default), 2, 5 and 8 windows on 2 MiB
    boundaries, the last window short, chunk boundaries inside windows
    (R = 3 does not divide the window size)."""
    o = elementops.get_op("f32", "sum")
    R, n = 3, 2**23 + 5
    x = inputs.generate(R, n, "f32", "normal", seed=520)
    want = ring.ring_allreduce(x, o)
    ins = [_pinned(v) for v in x]
    outs = [_pinned(np.zeros_like(v)) for v in x]
    with ra.RingAllReduce(R, n, "f32", "sum") as h:
        h.set_option(ra.Option.HOST_WINDOWS, windows)
        h.allreduce_host(ins, outs)
        torch.cuda.synchronize()
    for r in range(R):
        assert_bitwise_equal(_host(outs[r], x[r]), want[r], f"windows={windows} rank {r}")


def test_host_calls_back_to_back(ra):
    """Three calls on one handle with no synchronisation between them: each
    call's windows wait only for the previous call's use of the same
    window of the device copies, and every result is the oracle's."""
    o = elementops.get_op("f32", "sum")
    R, n = 4, 2**22 + 7
    xs = [inputs.generate(R, n, "f32", "normal", seed=530 + k) for k in range(3)]
    wants = [ring.ring_allreduce(x, o) for x in xs]
    ins = [[_pinned(v) for v in x] for x in xs]
    outs = [[_pinned(np.zeros_like(v)) for v in x] for x in xs]
    stream = torch.cuda.Stream()
    with ra.RingAllReduce(R, n, "f32", "sum") as h:
        for k in range(3):
            h.allreduce_host(ins[k], outs[k], stream)
        stream.synchronize()
        assert h.device_status()[0] == ra.Status.OK
    for k in range(3):
        for r in range(R):
            assert_bitwise_equal(_host(outs[k][r], xs[k][r]), wants[k][r], f"call {k} rank {r}")


def test_host_rejects_device_memory(ra):
    R, n = 2, 1000
    dev = [torch.zeros(n, device="cuda") for _ in range(R)]
    host = [torch.zeros(n).pin_memory() for _ in range(R)]
    with ra.RingAllReduce(R, n, "f32", "sum") as h:
        with pytest.raises(ValueError):
            h.allreduce_host(dev, host)
        with pytest.raises(ra.RAError) as e:   # raw addresses reach the C side
            ra.ra_allreduce_host(h.h, [t.data_ptr() for t in dev], [t.data_ptr() for t in host])
        assert e.value.status == ra.Status.ERR_INVALID
        with pytest.raises(ra.RAError) as e:   # outputs overlapping each other
            ra.ra_allreduce_host(h.h, [t.data_ptr() for t in host], [host[0].data_ptr(), host[0].data_ptr() + 4])
        assert e.value.status == ra.Status.ERR_INVALID


def test_host_strided_and_scattered_buffers(ra):
    """Rows of one page-locked allocation, in order and in reverse order,
    with 1, 3 and 8 windows: only each row's n elements are written."""
    o = elementops.get_op("f32", "sum")
    R, n = 5, 3 * 2**20 + 1
    x = inputs.generate(R, n, "f32", "normal", seed=540)
    want = ring.ring_allreduce(x, o)
    pad = n + 37                                     # row stride, not a multiple of 16 bytes
    big_in = torch.zeros((R, pad), dtype=torch.int32).pin_memory()
    for r in range(R):
        big_in[r, :n] = torch.from_numpy(x[r].view(np.int32))
    for windows in (1, 3, 8):
        for order in (list(range(R)), list(reversed(range(R)))):
            big_out = torch.zeros((R, pad), dtype=torch.int32).pin_memory()
            ins = [big_in[r, :n] for r in order]
            outs = [big_out[r, :n] for r in order]
            with ra.RingAllReduce(R, n, "f32", "sum") as h:
                h.set_option(ra.Option.HOST_WINDOWS, windows)
                h.allreduce_host(ins, outs)
                torch.cuda.synchronize()
            wanted = ring.ring_allreduce([x[r] for r in order], o)
            for i, r in enumerate(order):
                assert_bitwise_equal(big_out[r, :n].numpy().view(np.float32), wanted[i],
                                     f"windows={windows} order={order[:2]} rank {i}")
                assert not big_out[r, n:].any(), "row padding written"
    del want


def test_host_calls_on_two_streams(ra):
    """Calls alternating between two streams overlap; the windows of the
    handle's device copies still pass from call to call in order, so every
    result is the oracle's."""
    o = elementops.get_op("bf16", "sum")
    R, n = 8, 2**21 + 3
    xs = [inputs.generate(R, n, "bf16", "grad", seed=550 + k) for k in range(4)]
    wants = [ring.ring_allreduce(x, o) for x in xs]
    ins = [[_pinned(v) for v in x] for x in xs]
    outs = [[_pinned(np.zeros_like(v)) for v in x] for x in xs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    with ra.RingAllReduce(R, n, "bf16", "sum") as h:
        for k in range(4):
            h.allreduce_host(ins[k], outs[k], streams[k % 2])
        torch.cuda.synchronize()
    for k in range(4):
        for r in range(R):
            assert_bitwise_equal(_host(outs[k][r], xs[k][r]), wants[k][r], f"call {k} rank {r}")


def test_host_window_count_changes_between_calls(ra):
    """Calls with 2, 8, 3 and 8 windows issued back to back on two streams,
    no synchronisation between them: a call whose windows differ from the
    last call's waits for every earlier use of the device copies."""
    o = elementops.get_op("f32", "sum")
    R, n = 4, 2**22 + 9
    xs = [inputs.generate(R, n, "f32", "normal", seed=560 + k) for k in range(4)]
    wants = [ring.ring_allreduce(x, o) for x in xs]
    ins = [[_pinned(v) for v in x] for x in xs]
    outs = [[_pinned(np.zeros_like(v)) for v in x] for x in xs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    with ra.RingAllReduce(R, n, "f32", "sum") as h:
        for k, windows in enumerate((2, 8, 3, 8)):
            h.set_option(ra.Option.HOST_WINDOWS, windows)
            h.allreduce_host(ins[k], outs[k], streams[k % 2])
        torch.cuda.synchronize()
    for k in range(4):
        for r in range(R):
            assert_bitwise_equal(_host(outs[k][r], xs[k][r]), wants[k][r], f"call {k} rank {r}")
