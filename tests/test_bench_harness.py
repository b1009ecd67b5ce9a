"""The multi-GPU path of bench.py is N independent replicas; its host logic
(max of the per-rank times, sum of the per-rank work) is checked here with
two gloo processes on CPU."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    d = bench._init_pg(world)
    t, u = bench.aggregate(0.5 + rank, 100.0 * (rank + 1), d)
    q.put((rank, t, u))
    d.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for _, t, u in res:
        assert t == pytest.approx(1.5)     # slowest rank
        assert u == pytest.approx(300.0)   # all ranks' work


def test_aggregate_single_process_is_identity():
    import bench
    assert bench.aggregate(0.25, 7.0, None) == (0.25, 7.0)


@pytest.mark.parametrize("R,n,dtype,threads", [
    (4, 4096, "f32", 3),          # divisible
    (8, 1000003, "f32", 16),      # ragged: a short last chunk
    (5, 13, "bf16", 4),           # tiny chunks, more threads than a range holds
    (7, 30, "i32", 2),            # trailing chunks short and empty (C = 5: 6 chunks hold 30)
    (6, 0, "f32", 4),             # nothing to do
    (3, 20011, "f64", 5),
])
def test_threaded_cpu_baseline_is_the_oracle_bit_for_bit(R, n, dtype, threads):
    """bench.py's multi-core CPU figure runs the oracle on element ranges in
    parallel; every output must carry the bits of one oracle call on the
    whole input (the fold order of an element depends on its chunk only)."""
    import numpy as np
    import bench
    from oracle import elementops, ring
    from ring_allreduce_gb300 import inputs
    dist = {"f32": "normal", "bf16": "grad", "i32": "int20", "f64": "normal"}[dtype]
    x = inputs.generate(R, n, dtype, dist, seed=77 + R)
    op = elementops.get_op(dtype, "sum")
    want = ring.ring_allreduce(x, op)
    got = bench.oracle_threaded_allreduce(x, op, threads)
    for r in range(R):
        assert np.ascontiguousarray(got[r]).view(np.uint8).tobytes() == \
            np.ascontiguousarray(want[r]).view(np.uint8).tobytes(), f"rank {r}"


def test_threaded_cpu_baseline_catches_a_wrong_start_rank():
    """The split must keep each element in its own chunk: folding a range as
    if it sat in the next chunk (a start rank one off) changes the bits of
    the ring-start pattern (2^24, 1, 1, -2^24 gives 0 only from rank k)."""
    import numpy as np
    import bench
    from oracle import elementops, ring
    R, n = 4, 16
    x = [np.zeros(n, np.float32) for _ in range(R)]
    for k in range(R):   # chunk k (4 elements): x_k = 2^24, x_{k+1} = 1, x_{k+2} = 1, x_{k+3} = -2^24
        for j, v in enumerate((2.0**24, 1.0, 1.0, -2.0**24)):
            x[(k + j) % R][4 * k:4 * k + 4] = v
    op = elementops.get_op("f32", "sum")
    got = bench.oracle_threaded_allreduce(x, op, 3)
    assert all(np.all(got[r] == 0.0) for r in range(R))
    assert np.all(ring.ring_allreduce(x, op)[0] == 0.0)
    rotated = [x[(r + 1) % R] for r in range(R)]   # every element's fold starts one rank later
    assert np.all(bench.oracle_threaded_allreduce(rotated, op, 3)[0] == 2.0)


class _FakeNvml:
    """Stands in for libnvidia-ml: an SM clock and a clock-event reason mask
    that a test sets, read through the same calls and pointers."""

    def __init__(self, mhz, mask, max_mhz=2070):
        self.mhz, self.mask, self.max_mhz = mhz, mask, max_mhz

    def nvmlInit_v2(self):
        return 0

    def nvmlDeviceGetHandleByUUID(self, uuid, handle):
        assert uuid.startswith(b"GPU-")
        handle._obj.value = 1
        return 0

    def nvmlDeviceGetMaxClockInfo(self, h, kind, out):
        out._obj.value = self.max_mhz
        return 0

    def nvmlDeviceGetClockInfo(self, h, kind, out):
        assert kind == 1   # SM clock
        out._obj.value = self.mhz
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, h, out):
        out._obj.value = self.mask
        return 0


def test_nvml_clock_sampler_reads_clocks_and_reasons():
    import time
    import bench
    fake = _FakeNvml(1980, 0x4 | 0x1)   # power cap, plus an idle bit that is not reported
    s = bench.NvmlClockSampler("GPU-0000", lib=fake).start()
    assert s is not None
    s.begin()
    time.sleep(0.03)
    s.end()
    r = s.stop()
    assert r["sm_mhz"] == 1980 and r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"]
    assert r["samples"] >= 3          # about one per millisecond
    fake2 = _FakeNvml(2070, 0x8 | 0x40)
    s = bench.NvmlClockSampler("GPU-0000", lib=fake2).start()
    s.begin()
    time.sleep(0.01)
    s.end()
    assert s.stop()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_nvml_clock_sampler_without_nvml_falls_back():
    import bench
    class NoInit(_FakeNvml):
        def nvmlInit_v2(self):
            return 9
    assert bench.NvmlClockSampler("GPU-0000", lib=NoInit(0, 0)).start() is None


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _reference_arm(env_extra, *args):
    import subprocess
    import sys
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_the_contract_line():
    """The reference arm (the oracle on the host cores, no GPU) prints one
    JSON line with the contract's keys, on the config it actually ran."""
    import json
    res = _reference_arm({}, "--workload", "r4_small", "--steps", "3", "--warmup", "3")
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["R"] == 4 and d["config"]["n_per_rank"] == 4096   # the whole small workload ran
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert "n=4096" in d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_prints_nothing_on_other_ranks():
    res = _reference_arm({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"},
                         "--gpus", "2", "--workload", "r4_small", "--steps", "1", "--warmup", "3")
    assert res.returncode == 0, res.stderr[-2000:]
    assert not [l for l in res.stdout.splitlines() if l.startswith("{")], res.stdout


def test_config_says_how_timing_stands_to_the_l2():
    """Inputs larger than L2 need no flush between steps; a call that fits in
    L2 is said to be timed back to back, a latency figure."""
    import argparse
    import bench
    args = argparse.Namespace(workload="r8_f32", n=None, variant="auto", protocol="simple")
    big = bench.workload_config(args, 8, 2**24, "sum", 4, 1)["l2"]
    assert big.startswith("inputs larger than L2: 512 MiB of inputs")
    args = argparse.Namespace(workload="r4_small", n=None, variant="auto", protocol="simple")
    small = bench.workload_config(args, 4, 4096, "sum", 4, 1)["l2"]
    assert small.startswith("inputs in L2 (64 KiB of inputs") and "latency" in small


def test_roofline_traffic_only_from_a_summary_of_the_current_kernel(monkeypatch):
    """`roofline.traffic` is the committed ncu summary's DRAM bytes per launch,
    scaled by the units a launch processes, while the summary names the
    direct kernel's current source hash; null once the kernel has changed."""
    import bench
    from ring_allreduce_gb300 import build
    t, path = bench.profile_traffic("r8_f32", 2**24)
    assert path.endswith("direct_kernel_r8_f32.md")
    assert t is not None and 0.9 * 2**30 < t < 1.2 * 2**30    # about the compulsory 1 GiB
    t2, _ = bench.profile_traffic("r8_f32", 2**25)
    assert t2 == 2 * t
    real = build.kernel_source_hash
    monkeypatch.setattr(build, "kernel_source_hash", lambda k=None: "0" * 16 if k == "direct" else real(k))
    assert bench.profile_traffic("r8_f32", 2**24)[0] is None
