"""Child process of test_gpu_debug_bounds.py: loads the bounds-checked
library (RA_GB300_DEBUG_BOUNDS=1 must be set before the binding is imported),
drives every entry point, variant, barrier and AllGather kernel over small
ragged shapes, checks the results against the oracle, and prints one JSON
line: the checks' report after the clean calls, and after a call whose
buffers were registered 16 bytes short (the checks must see that one).  It
also runs the bounded waits of the kernels fed by TMA bulk copies to their
limit: a copy the checks skip never arrives, so the wait on it runs out and
reports (error code 2), and the next call on the handle is correct again."""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import torch  # noqa: E402

from oracle import elementops, ring  # noqa: E402
from ring_allreduce_gb300 import inputs  # noqa: E402
from rahelpers import DeviceRanks  # noqa: E402

assert os.environ.get("RA_GB300_DEBUG_BOUNDS") == "1"
from ring_allreduce_gb300 import binding as ra  # noqa: E402

assert ra.library_path().endswith("libra_gb300_debug.so"), ra.library_path()
DIST = {"f32": "normal", "bf16": "grad", "i32": "int20", "f16": "grad", "f64": "normal", "i64": "int40"}
mismatches = []


def check(tag, got, want):
    if not np.array_equal(np.ascontiguousarray(got).view(np.uint8), np.ascontiguousarray(want).view(np.uint8)):
        mismatches.append(tag)


def run(R, n, dtype, op, variant, kind, options=()):
    o = elementops.get_op(dtype, op)
    st = inputs.storage_dtype(dtype)
    x = inputs.generate(R, n, dtype, DIST[dtype], seed=R * 1000 + n)
    plan = ring.chunk_plan(R, n)
    tag = f"{variant} {kind} {dtype}/{op} R={R} n={n} {options}"
    with ra.RingAllReduce(R, n, dtype, op, variant=variant) as h:
        for key, value in options:
            h.set_option(key, value)
        if kind == "host":
            ins = [v.copy() for v in x]
            outs = [np.zeros_like(v) for v in x]
            h.allreduce_host(ins, outs)
            torch.cuda.synchronize()
            want = ring.ring_allreduce(x, o)
            for r in range(R):
                check(tag, outs[r], want[r])
            return
        if kind in ("rs_compact", "ag_compact"):
            inp = DeviceRanks(R, n, st, host=x)
            lens = [h.owned_chunk(r)[1] for r in range(R)]
            comp = [torch.zeros(max(L, 1), dtype=inp.big.dtype, device="cuda") for L in lens]
            h.reduce_scatter_compact(inp.views, comp)
            full = DeviceRanks(R, n, st)
            h.all_gather_compact(comp, full.views)
            torch.cuda.synchronize()
            want = ring.ring_allreduce(x, o)
            got = full.host()
            for r in range(R):
                check(tag, got[r], want[r])
            return
        inp = DeviceRanks(R, n, st, host=x)
        out = DeviceRanks(R, n, st)
        if kind == "allreduce":
            h.allreduce(inp.views, out.views)
            want = ring.ring_allreduce(x, o)
            torch.cuda.synchronize()
            got = out.host()
            for r in range(R):
                check(tag, got[r], want[r])
        elif kind == "reduce_scatter":
            h.reduce_scatter(inp.views, out.views)
            want = ring.ring_reduce_scatter(x, o)
            torch.cuda.synchronize()
            got = out.host()
            for r in range(R):
                off, L = plan[ring.owned_chunk(R, r)]
                check(tag, got[r][off:off + L], want[r][off:off + L])
        else:
            rs = ring.ring_reduce_scatter(x, o)
            buf = []
            for r in range(R):
                b = np.zeros_like(x[r])
                off, L = plan[ring.owned_chunk(R, r)]
                b[off:off + L] = rs[r][off:off + L]
                buf.append(b)
            dev = DeviceRanks(R, n, st, host=buf)
            h.all_gather(dev.views)
            want = ring.ring_all_gather(buf, o)
            torch.cuda.synchronize()
            got = dev.host()
            for r in range(R):
                check(tag, got[r], want[r])
        status, err = h.device_status()
        if status != ra.Status.OK:
            mismatches.append(f"{tag}: {status.name} {err.as_dict()}")


def main():
    torch.cuda.set_device(0)
    ra.ra_debug_bounds_report(reset=True)
    shapes = [(2, 1), (3, 1001), (8, 8 * 1024 + 13), (5, 70001), (16, 2**16 + 3), (32, 4099)]
    calls = 0
    for R, n in shapes:
        for variant in ("direct", "ring", "persistent", "pipelined", "local"):
            for kind in ("allreduce", "reduce_scatter", "all_gather"):
                run(R, n, "bf16", "sum", variant, kind)
                calls += 1
        for dtype, op in (("f32", "max"), ("f64", "sum"), ("i64", "max"), ("i32", "sum")):
            run(R, n, dtype, op, "direct", "allreduce")
            run(R, n, dtype, op, "local", "allreduce")
            calls += 2
        run(R, n, "bf16", "sum", "direct", "rs_compact")
        run(R, n, "f32", "sum", "direct", "host")
        run(R, n, "f32", "sum", "direct", "all_gather", options=[(ra.Option.GATHER, 2)])
        run(R, n, "f32", "sum", "persistent", "allreduce", options=[(ra.Option.BARRIER, ra.Barrier.PER_PEER)])
        if R <= 16:
            run(R, n, "f32", "sum", "persistent", "allreduce", options=[(ra.Option.BARRIER, ra.Barrier.CLUSTER)])
        run(R, n, "f32", "sum", "pipelined", "allreduce", options=[(ra.Option.SLICES, 3)])
        run(R, n, "bf16", "sum", "pipelined", "allreduce", options=[(ra.Option.SLICES, 5), (ra.Option.WINDOW, 2)])
        # flag-in-data messages: the inbox rows and the positions past a ragged chunk's end
        for kind in ("allreduce", "reduce_scatter", "all_gather"):
            run(R, n, "bf16", "sum", "pipelined", kind, options=[(ra.Option.PROTOCOL, ra.Protocol.LL)])
        run(R, n, "f64", "sum", "pipelined", "allreduce", options=[(ra.Option.PROTOCOL, ra.Protocol.LL)])
        calls += 4
        if R <= 16:
            for kind in ("allreduce", "reduce_scatter", "all_gather"):
                run(R, n, "bf16", "sum", "pipelined", kind, options=[(ra.Option.PROTOCOL, ra.Protocol.LL_CLUSTER)])
            run(R, n, "f64", "sum", "pipelined", "allreduce", options=[(ra.Option.PROTOCOL, ra.Protocol.LL_CLUSTER)])
            calls += 4
        # passes: every round on one part of every chunk (slice) before the next part
        for kind in ("allreduce", "reduce_scatter", "all_gather"):
            run(R, n, "bf16", "sum", "ring", kind, options=[(ra.Option.SLICES, 3)])
            run(R, n, "bf16", "sum", "persistent", kind, options=[(ra.Option.SLICES, 3)])
        if R <= 16:
            run(R, n, "f32", "sum", "persistent", "allreduce",
                options=[(ra.Option.SLICES, 2), (ra.Option.BARRIER, ra.Barrier.CLUSTER)])
        calls += 13 if R <= 16 else 12
    # the allocation-free entry point
    R, n = 4, 10007
    x = inputs.generate(R, n, "f32", "normal", seed=5)
    inp, out = DeviceRanks(R, n, np.float32, host=x), DeviceRanks(R, n, np.float32)
    ra.ra_allreduce_noalloc(R, n, ra.DType.F32, ra.Op.SUM, inp.views, out.views)
    torch.cuda.synchronize()
    want = ring.ring_allreduce(x, elementops.get_op("f32", "sum"))
    got = out.host()
    for r in range(R):
        check("noalloc", got[r], want[r])
    calls += 1
    clean_count, clean_first = ra.ra_debug_bounds_report(reset=True)

    # the control: buffers registered 16 bytes short; the kernel's accesses to
    # their last 16 bytes must be reported (and skipped)
    R, n = 4, 4096
    x = inputs.generate(R, n, "f32", "normal", seed=6)
    inp, out = DeviceRanks(R, n, np.float32, host=x), DeviceRanks(R, n, np.float32)
    with ra.RingAllReduce(R, n, "f32", "sum", variant="direct") as h:
        h.set_option(ra.Option.DEBUG_SHRINK, 16)
        h.allreduce(inp.views, out.views)
        torch.cuda.synchronize()
    ends = [v.data_ptr() + n * 4 for v in inp.views + out.views]
    shrunk_count, shrunk_first = ra.ra_debug_bounds_report(reset=True)

    # bounded waits run out: the local kernel (AllReduce; one copying warp at
    # R = 8, four at R = 16) and the ring variant's AllGather rounds wait on
    # bulk copies that the checks skip
    timeouts = {}
    for variant, kind, R in (("local", "allreduce", 8), ("local", "allreduce", 16), ("ring", "all_gather", 8)):
        n = R * 4096
        x = inputs.generate(R, n, "f32", "normal", seed=7)
        o = elementops.get_op("f32", "sum")
        with ra.RingAllReduce(R, n, "f32", "sum", variant=variant) as h:
            h.set_option(ra.Option.TIMEOUT_NS, 50_000_000)
            h.set_option(ra.Option.DEBUG_SHRINK, 16)
            bufs = DeviceRanks(R, n, np.float32, host=x)
            outs = DeviceRanks(R, n, np.float32)
            if kind == "allreduce":
                h.allreduce(bufs.views, outs.views)
            else:
                h.all_gather(bufs.views)
            status, err = h.device_status()
            first = {"status": status.name, "code": int(err.code)}
            # the handle is usable again, with the checks back to the full buffers
            h.set_option(ra.Option.DEBUG_SHRINK, 0)
            bufs = DeviceRanks(R, n, np.float32, host=x)
            outs = DeviceRanks(R, n, np.float32)
            if kind == "allreduce":
                h.allreduce(bufs.views, outs.views)
                want = ring.ring_allreduce(x, o)
            else:
                h.all_gather(bufs.views)
                want = ring.ring_all_gather(x, o)
            status2, _ = h.device_status()
            torch.cuda.synchronize()
            got = outs.host() if kind == "allreduce" else bufs.host()
            first["after"] = status2.name
            first["after_equal"] = all(np.array_equal(got[r].view(np.uint32), want[r].view(np.uint32))
                                       for r in range(R))
        timeouts[f"{variant} R={R}"] = first
    ra.ra_debug_bounds_report(reset=True)
    print(json.dumps({
        "timeouts": timeouts,
        "calls": calls,
        "mismatches": mismatches[:10],
        "clean": {"count": clean_count, "first": clean_first},
        "shrunk": {"count": shrunk_count, "first": shrunk_first,
                   "first_in_a_cut_tail": any(e - 16 <= shrunk_first < e for e in ends)},
    }))


if __name__ == "__main__":
    main()
