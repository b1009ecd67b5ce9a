#!/usr/bin/env python3
"""Benchmark of the ring AllReduce library on synthetic rank buffers.

One step is one ra_allreduce call over R rank buffers resident in HBM: the
chunk plan, every ReduceScatter and AllGather round of the ring (done by the
selected variant; the default carries every element's ring fold out in one
launch).  Prints one JSON line.

  value     algbw = n * bytes_per_element / time per step (the per-rank
            payload over time, the usual AllReduce convention), summed over
            replicas when run on several GPUs (each GPU runs its own R-rank
            ring: the collective does not span GPUs)
  busbw     algbw * 2(R-1)/R: what every rank of a real ring sends, section
            13 of the ring page ("Why AllReduce = ReduceScatter + AllGather --
            NCCL Ring AllReduce"), 2N(k-1)/k per rank
  roofline  the dominant kernel's compulsory HBM bytes (read every input
            once, write every output once: 2 R n b) over its CUDA-event
            launch time, against the measured device copy bandwidth

--impl reference times the CPU oracle instead (host cores, bounded sample
of the same workload).  --sweep prints one line per size / rank count of the
sweep workloads (not the headline).
"""

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ring allreduce algbw GB/s and % of GB300 HBM roofline (R ranks on 1 GPU)"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 10**6   # GB300's L2

WORKLOAD_TEXT = {
    "r8_f32": "ring allreduce, R=8 ranks x n=2^24 fp32 per rank (64 MiB/rank), N(0,1), sum, seed 1",
    "r8_bf16": "ring allreduce, R=8 ranks x n=2^26+3 bf16 per rank (ragged), grad-like N(0,1e-3) with 1% x100, "
               "sum with bf16 rounding per hop, seed 2",
    "r16_i32": "ring allreduce, R=16 ranks x n=2^24 int32 per rank, uniform [-2^20,2^20], sum, seed 3",
    "r4_small": "ring allreduce, R=4 ranks x n=4096 fp32 per rank, integers in [-8,8], sum, seed 0",
}


# ------------------------------------------------------------------ helpers

def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _init_pg(ws):
    if ws <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    # the harness only needs a barrier and a max over ranks: gloo on the host
    dist.init_process_group("gloo")
    return dist


def aggregate(local_seconds, local_units, dist):
    """Max of the per-rank times and sum of the per-rank work over the
    process group (identity without one)."""
    if dist is None:
        return local_seconds, local_units
    import torch
    t = torch.tensor([local_seconds], dtype=torch.float64)
    u = torch.tensor([local_units], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def build_info(torch):
    """What the numbers were taken on: kernel source hashes, toolkit,
    driver, device (a copy of the sources need not carry its git history)."""
    from ring_allreduce_gb300 import build
    info = {"sources": {k: build.kernel_source_hash(k) for k in build.KERNEL_SOURCES},
            "torch": torch.__version__}
    try:
        out = subprocess.run(["nvcc", "--version"], capture_output=True, text=True, timeout=20).stdout
        info["nvcc"] = out.strip().splitlines()[-1]
    except Exception:
        info["nvcc"] = None
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version,name", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.strip().splitlines()[0]
        info["driver"], info["gpu"] = [x.strip() for x in out.split(",", 1)]
    except Exception:
        info["driver"] = info["gpu"] = None
    return info


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(workload, units_full):
    """Traffic per launch of the direct kernel from the committed ncu
    summary, scaled to the full workload, or None when the summary was
    taken on other kernel sources."""
    from ring_allreduce_gb300 import build
    path = os.path.join(ROOT, "profiles", f"direct_kernel_{workload}.md")
    if not os.path.exists(path):
        return None, None
    text = open(path).read()
    m_hash = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*(\d+)", text)
    m_units = re.search(r"units_per_launch:\s*(\d+)", text)
    if not (m_hash and m_bytes and m_units):
        return None, path
    if m_hash.group(1) != build.kernel_source_hash("direct"):
        return None, path
    return int(m_bytes.group(1)) * units_full / int(m_units.group(1)), path


class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (the driver's
    libnvidia-ml, by ctypes; read-only queries) about every millisecond on a
    thread, so that even a timed region of a few milliseconds holds several
    samples.  Same interface and result as ClockSampler; start() returns
    None where NVML cannot be loaded or the GPU not found."""

    SM = 1   # NVML_CLOCK_SM
    # clock-event reason bits of NVML's public API
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, gpu_uuid, period_s=0.001, lib=None):
        self.uuid = gpu_uuid
        self.period = period_s
        self.lib = lib
        self.rows = []
        self.t_begin = self.t_end = None
        self._stop = threading.Event()

    def _open(self):
        import ctypes
        lib = self.lib or ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) != 0:
            return False
        self._read_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(h, self.SM, ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        self.h, self.ctypes, self.nvml = h, ctypes, lib
        return True

    def start(self):
        try:
            if not self._open():
                return None
        except (OSError, AttributeError):
            return None
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()
        return self

    def sample_now(self):
        c, m = self.ctypes.c_uint(0), self.ctypes.c_ulonglong(0)
        ok = self.nvml.nvmlDeviceGetClockInfo(self.h, self.SM, self.ctypes.byref(c)) == 0
        ok = ok and self._read_reasons(self.h, self.ctypes.byref(m)) == 0
        if ok:
            self.rows.append((time.monotonic(), float(c.value), int(m.value)))

    def _read(self):
        while not self._stop.is_set():
            self.sample_now()
            time.sleep(self.period)

    def begin(self):
        self.t_begin = time.monotonic()

    def end(self):
        self.t_end = time.monotonic()

    def stop(self):
        self._stop.set()
        self.th.join(timeout=2)
        inside = [r for r in self.rows if self.t_begin <= r[0] <= self.t_end]
        if not inside:
            return None
        reasons = sorted({name for r in inside for bit, name in self.REASONS.items() if r[2] & bit})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(inside),
                "note": "NVML samples inside the timed region (a thread about every millisecond, and the "
                        "timing thread itself while the device runs the enqueued steps)"}


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while a region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_ms=50):
        self.idx = gpu_index
        self.period = period_ms
        self.lines = []
        self.proc = None
        self.t_begin = self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def begin(self):
        self.t_begin = time.monotonic()

    def end(self):
        self.t_end = time.monotonic()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((t, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t_begin <= r[0] <= self.t_end + 0.05]
        note = "samples inside the timed region"
        if not inside:
            mid = (self.t_begin + self.t_end) / 2
            inside = sorted(rows, key=lambda r: abs(r[0] - mid))[:2]
            note = "timed region shorter than the sampling period: nearest samples"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "note": note}


# ------------------------------------------------------------- GPU arm

def _device_ranks(torch, R, n, np_dtype, host=None):
    """R rank buffers as rows of one device tensor; rows padded so every
    rank's base is 16-byte aligned."""
    import numpy as np
    tdt = {np.dtype(np.float32): torch.float32, np.dtype(np.uint16): torch.int16,
           np.dtype(np.int32): torch.int32, np.dtype(np.float16): torch.float16,
           np.dtype(np.float64): torch.float64, np.dtype(np.int64): torch.int64}[np.dtype(np_dtype)]
    stride = ((n + 63) // 64) * 64
    big = torch.empty((R, stride), dtype=tdt, device="cuda")
    if host is not None:
        for r in range(R):
            a = host[r].view(np.int16) if np.dtype(np_dtype) == np.uint16 else host[r]
            big[r, :n].copy_(torch.from_numpy(a))
    return big, [big[r, :n] for r in range(R)]


def _time_variant(torch, ra, h, ins, outs, steps, warmup, per_launch=True, queued=False):
    """CUDA-event times of `steps` calls after `warmup` (total ms, per-call
    ms).  queued: a spin kernel holds the stream while the host enqueues
    every timed call, so the device runs them back to back and the per-call
    times are device time -- without it a call shorter than the host's own
    cost of issuing it (a few microseconds from Python) measures the host."""
    stream = torch.cuda.current_stream()
    call = h.prepare("allreduce", ins, outs, stream)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)] \
        if per_launch else []
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if queued:
        torch.cuda._sleep(int(1e6 + 40000 * steps))   # ~20 us of SM cycles per call to enqueue
    t0.record(stream)
    for i in range(steps):
        if per_launch:
            ev[i][0].record(stream)
        call()
        if per_launch:
            ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    total_ms = t0.elapsed_time(t1)
    launch_ms = [a.elapsed_time(b) for a, b in ev] if per_launch else []
    return total_ms, launch_ms


def run_gpu_arm(args):
    import numpy as np
    import torch

    from ring_allreduce_gb300 import build, inputs
    build.build()
    from ring_allreduce_gb300 import binding as ra

    ws, rank, local = _dist_env()
    dist = _init_pg(ws)
    torch.cuda.set_device(local)
    w = dict(inputs.WORKLOADS[args.workload])
    R = w["R"]
    n = args.n or w["n"]
    dtype = w["dtype"]
    op = args.op or w["ops"][0]
    if op not in w["ops"]:
        raise SystemExit(f"workload {args.workload} runs ops {w['ops']}, not {op}")
    b = inputs.itemsize(dtype)
    st_dtype = inputs.storage_dtype(dtype)

    host = inputs.generate(R, n, dtype, w["dist"], w["seed"])
    big_in, ins = _device_ranks(torch, R, n, st_dtype, host)
    big_out, outs = _device_ranks(torch, R, n, st_dtype)
    h = ra.RingAllReduce(R, n, dtype, op, variant=args.variant)
    if args.protocol != "simple":
        h.set_option(ra.Option.PROTOCOL, ra.Protocol[args.protocol.upper()])
    variant_name = args.variant

    # ---- timed region: K steps, barrier + synchronize on both sides
    gpu_id = str(local)
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    clocks = None
    if rank == 0 and not args.no_clocks:
        clocks = NvmlClockSampler(gpu_id).start() or ClockSampler(gpu_id).start()
    stream = torch.cuda.current_stream()
    call = h.prepare("allreduce", ins, outs, stream)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.begin()
    t0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    t1.record(stream)
    if clocks and hasattr(clocks, "sample_now"):
        # the device is still running the enqueued steps: sample from this
        # thread until it is done (a sampling thread may not get the
        # interpreter in a region of a few milliseconds)
        while not t1.query():
            clocks.sample_now()
            time.sleep(0.0005)
    torch.cuda.synchronize()
    if clocks:
        clocks.end()
    if dist:
        dist.barrier()
    total_s = t0.elapsed_time(t1) / 1e3
    launch_ms = [a.elapsed_time(bb) for a, bb in ev]
    clk = clocks.stop() if clocks else None
    st_code, err = h.device_status()
    if st_code != ra.Status.OK:
        raise RuntimeError(f"device status {st_code.name}: {err.as_dict()}")

    t_step, total_units = aggregate(total_s / args.steps, float(n * b), dist)
    algbw = total_units / t_step / 1e9
    busbw = algbw * 2 * (R - 1) / R if R > 1 else algbw

    # dominant kernel: the one launch per step of the direct variant
    compulsory = 2 * R * n * b
    ring_bytes = 5 * (R - 1) * n * b
    launch_avg_s = statistics.mean(launch_ms) / 1e3
    peak, peak_kind = measured_peaks()
    achieved = compulsory / launch_avg_s / 1e9
    traffic, prof_path = profile_traffic(args.workload, n) if args.n is None else (None, None)

    result = {
        "metric": METRIC,
        "value": round(algbw, 3),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_step * 1e3, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype,
        "data": "synthetic",
        "config": workload_config(args, R, n, op, b, ws),
        "busbw": round(busbw, 3),
        "hbm_frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
        "roofline": {
            "bound": "hbm",
            "kernel": "ra::direct_kernel" if variant_name in ("auto", "direct") else f"{variant_name} step",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s",
            "bytes_per_launch": compulsory,
            "bytes_model": "compulsory 2*R*n*b (each input read once, each output written once)",
            "launch_ms_avg": round(launch_avg_s * 1e3, 6),
            # the same bytes over the whole step (ms_per_step, back to back:
            # includes the drain of the previous launch's writes from L2)
            "achieved_step": round(compulsory / t_step / 1e9, 1),
            "frac_step": round(compulsory / t_step / 1e9 / peak, 4),
            "traffic": traffic,
            "traffic_source": os.path.relpath(prof_path, ROOT) if prof_path else None,
        },
        "gpu_launches": args.steps * (2 * (R - 1) * ring_passes(n * b) if variant_name == "ring" else 1),
    }
    if clk is not None:
        result["clocks"] = clk
    if rank == 0:
        result["build"] = build_info(torch)

    # ---- other variants, same workload (fewer steps)
    if not args.no_variants and rank == 0:
        var = {}
        for v in ("direct", "ring", "persistent", "pipelined", "local"):
            hv = ra.RingAllReduce(R, n, dtype, op, variant=v)
            steps_v = max(5, min(args.steps, 100))
            total_ms, lm = _time_variant(torch, ra, hv, ins, outs, steps_v, max(3, args.warmup // 4 or 3))
            assert hv.device_status()[0] == ra.Status.OK
            hv.close()
            t = statistics.mean(lm) / 1e3
            by = compulsory if v in ("direct", "local") else ring_bytes
            var[v] = {"algbw": round(n * b / t / 1e9, 3),
                      "us_per_call": round(t * 1e6, 2),
                      "frac_compulsory": round(compulsory / t / 1e9 / peak, 4),
                      "frac_own_bytes": round(by / t / 1e9 / peak, 4),
                      "own_bytes": by}
        result["variants"] = var

    # ---- end to end through the public API, host buffers
    if not args.no_e2e:
        e2e = run_e2e(torch, ra, h, big_in, big_out, R, n, max(4, min(args.steps, 50)), dist)
        result["e2e"] = e2e

    # ---- CPU baseline: the oracle on a bounded sample, rank 0 at N = 1
    if rank == 0 and ws == 1 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_seconds, op_name=op)

    h.close()
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist:
        dist.destroy_process_group()


def ring_passes(round_bytes):
    """Passes the ring variant takes its chunks through the rounds in (the
    library's default: the fewest that keep n b / J within 32 MiB, at most
    8); each pass launches all 2(R-1) round kernels."""
    return max(1, min(8, -(-round_bytes // (32 << 20))))


def l2_statement(in_bytes):
    """How a step's timing stands to the L2: inputs larger than it (each step
    reads them from DRAM, no flush needed), or a call small enough to live
    in it, timed back to back as the latency figure it is."""
    if in_bytes > L2_BYTES:
        return (f"inputs larger than L2: {in_bytes / 2**20:.0f} MiB of inputs, "
                f"{in_bytes / 2**20:.0f} MiB of outputs per step, no flush")
    return (f"inputs in L2 ({in_bytes / 2**10:.0f} KiB of inputs, as much of outputs): calls timed "
            f"back to back without a flush, a latency figure rather than a bandwidth one")


def workload_config(args, R, n, op, b, ws):
    """The `config` of a bench line: the workload, identical for the GPU arm
    and the reference arm (which times the oracle on a sample of it)."""
    return {
        "workload": WORKLOAD_TEXT.get(args.workload, args.workload).replace(", sum,", f", {op},") if args.n is None
        else f"{args.workload} with n={n}",
        "R": R, "n_per_rank": n, "op": op, "variant": args.variant,
        **({"protocol": args.protocol} if args.protocol != "simple" else {}),
        "l2": l2_statement(R * n * b),
        "parallelism": f"replicas x{ws} (each GPU runs its own {R}-rank ring)",
    }


def run_e2e(torch, ra, h, big_in, big_out, R, n, steps, dist):
    """Algbw end to end through the C entry point for host buffers,
    ra_allreduce_host: every step hands it the R page-locked host inputs and
    R page-locked host outputs; the library copies each window of the inputs
    in, folds it, and copies it out while the next window comes in, and
    consecutive steps overlap the same way.  Every transfer of every step is
    inside the timed region."""
    import numpy as np
    pin_in = torch.empty(big_in.shape, dtype=big_in.dtype, pin_memory=True)
    pin_in.copy_(big_in)
    pin_out = torch.zeros(big_out.shape, dtype=big_out.dtype, pin_memory=True)
    ins = [pin_in[r, :n] for r in range(R)]
    outs = [pin_out[r, :n] for r in range(R)]
    # two streams, alternated: a call waits for everything before it on its
    # stream, so step k+1's uploads overlap step k's downloads only when the
    # two are on different streams
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    # untimed warm-up calls, copies included: the first transfers into and out
    # of each pinned buffer are slower than the rest
    for k in range(4):
        h.allreduce_host(ins, outs, streams[k % 2])
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(streams[0])
    streams[1].wait_event(e0)
    for k in range(steps):
        h.allreduce_host(ins, outs, streams[k % 2])
    streams[0].wait_stream(streams[1])
    e1.record(streams[0])
    torch.cuda.synchronize()
    b = big_in.element_size()
    te, units = aggregate(e0.elapsed_time(e1) / 1e3 / steps, float(n * b), dist)
    for r in (0, R - 1):
        if not np.array_equal(pin_out[r, :n].numpy().view(np.uint8), big_out[r, :n].cpu().numpy().view(np.uint8)):
            raise RuntimeError("e2e read-back differs from the device result")
    floor_s = link_floor(torch, pin_in, pin_out, big_in, big_out, steps)
    return {"value": round(units / te / 1e9, 3), "unit": "GB/s",
            "h2d_bytes_per_step": R * n * b, "d2h_bytes_per_step": R * n * b,
            "steps": steps, "ms_per_step": round(te * 1e3, 4),
            "link_floor_ms": round(floor_s * 1e3, 4),
            "frac_of_link_floor": round(floor_s / te, 4),
            "note": "every step: ra_allreduce_host on R page-locked host inputs and R page-locked host "
                    "outputs (all R inputs copied in, all R outputs copied back by the library, window "
                    "by window); steps alternate between two streams so that one step's uploads overlap "
                    "the previous step's downloads. link_floor_ms: the same bytes as bare copies in the "
                    "same run, all uploads on one stream and all downloads on another, one copy per "
                    "direction and step (no fold): the host link's own time for a step"}


def link_floor(torch, pin_in, pin_out, dev_in, dev_out, steps):
    """Seconds per step of the host link alone: one upload of all R input
    rows and one download of all R output rows per step, uploads and
    downloads on two streams so they run at once."""
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    scratch = torch.empty_like(dev_in)
    for _ in range(2):
        with torch.cuda.stream(up):
            scratch.copy_(pin_in, non_blocking=True)
        with torch.cuda.stream(down):
            pin_out.copy_(dev_out, non_blocking=True)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(up)
    down.wait_event(e0)
    for _ in range(steps):
        with torch.cuda.stream(up):
            scratch.copy_(pin_in, non_blocking=True)
        with torch.cuda.stream(down):
            pin_out.copy_(dev_out, non_blocking=True)
    up.wait_stream(down)
    e1.record(up)
    torch.cuda.synchronize()
    del scratch
    return e0.elapsed_time(e1) / 1e3 / steps


# ------------------------------------------------------------- CPU oracle

def _oracle_step_seconds(workload, n_sample, op_name=None):
    from oracle import elementops, ring
    from ring_allreduce_gb300 import inputs
    w = inputs.WORKLOADS[workload]
    x = inputs.generate(w["R"], n_sample, w["dtype"], w["dist"], w["seed"])
    op = elementops.get_op(w["dtype"], op_name or w["ops"][0])
    t = time.perf_counter()
    ring.ring_allreduce(x, op)
    return time.perf_counter() - t, x, op


def host_cores():
    """Cores this process may run on (its CPU affinity)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_threaded_allreduce(x, op, threads):
    """The oracle's ring AllReduce, as it stands, run on `threads` element
    ranges at once (host threads; numpy releases the interpreter lock inside
    its array operations).

    Element i of chunk k is folded in the ring order that starts at rank k,
    whatever the other elements do, so the elements [k C + a, k C + b) of
    every chunk k form an AllReduce of their own: stacked chunk after chunk
    (a rank vector of R (b - a) elements, whose chunk plan is again one piece
    per chunk) and run through the oracle, they come out with the bits the
    whole call gives them.  A short last chunk is padded with zeros to the
    range; the padded places fold among themselves and are dropped.  Returns
    the R outputs; the CPU tests check them bitwise against the oracle."""
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor

    from oracle import ring
    R, n = len(x), len(x[0])
    plan = ring.chunk_plan(R, n)
    C = max(L for _, L in plan) if n else 0
    out = [np.empty_like(np.asarray(v)) for v in x]
    if n == 0:
        return out
    threads = max(1, min(threads, C))
    cuts = [C * t // threads for t in range(threads + 1)]

    def piece(t):
        a, b = cuts[t], cuts[t + 1]
        w = b - a
        if w <= 0:
            return
        sub = []
        for r in range(R):
            v = np.zeros(R * w, dtype=x[r].dtype)
            for k, (o, L) in enumerate(plan):
                hi = min(b, L)
                if hi > a:
                    v[k * w:k * w + hi - a] = x[r][o + a:o + hi]
            sub.append(v)
        res = ring.ring_allreduce(sub, op)
        for r in range(R):
            for k, (o, L) in enumerate(plan):
                hi = min(b, L)
                if hi > a:
                    out[r][o + a:o + hi] = res[r][k * w:k * w + hi - a]

    with ThreadPoolExecutor(max_workers=threads) as pool:
        list(pool.map(piece, range(threads)))
    return out


def _timed_calls(fn, budget_s):
    fn()   # warm-up call, not timed
    times = []
    t_start = time.perf_counter()
    while (time.perf_counter() - t_start < budget_s and len(times) < 1000) or len(times) < 2:
        t = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t)
    return times


def cpu_baseline(workload, budget_s=15.0, n_sample=None, op_name=None):
    """Time the oracle, as it stands, on R ranks of a sample of the
    workload, on one thread (value) and split over element ranges on every
    core this process may use (`threaded`); values are algbw on the sample."""
    from oracle import ring
    from ring_allreduce_gb300 import inputs
    w = inputs.WORKLOADS[workload]
    b = inputs.itemsize(w["dtype"])
    n_sample = n_sample or w["n"]
    _, x, op = _oracle_step_seconds(workload, n_sample, op_name)
    cores = host_cores()
    times = _timed_calls(lambda: ring.ring_allreduce(x, op), budget_s * 2 / 3)
    times_mt = _timed_calls(lambda: oracle_threaded_allreduce(x, op, cores), budget_s / 3)
    t_mean, t_mt = statistics.mean(times), statistics.mean(times_mt)
    what = 'the full workload' if n_sample == w['n'] else 'same recipe and seed as the workload'
    return {"value": round(n_sample * b / t_mean / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"R={w['R']} ranks x n={n_sample} per rank ({what}), "
                      f"{len(times)} oracle calls, {sum(times):.1f} s; numpy, one thread",
            "ms_per_call": round(t_mean * 1e3, 3),
            "host_cores": cores,
            "threaded": {"value": round(n_sample * b / t_mt / 1e9, 6), "unit": "GB/s", "cores": cores,
                         "kind": "oracle split over element ranges, one host thread per core",
                         "sample": f"the same inputs, {len(times_mt)} calls, {sum(times_mt):.1f} s",
                         "ms_per_call": round(t_mt * 1e3, 3)}}


def run_reference_arm(args):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return
    from ring_allreduce_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    b = inputs.itemsize(w["dtype"])
    n_full = args.n or w["n"]
    # the whole workload when warm-up + K steps of it take at most three
    # minutes (25 calls of the R = 8 x 2^24 fp32 headline: ~4 s), else the
    # largest power-of-two sample that does, named in `config`
    budget = 180.0 / max(1, args.steps + args.warmup)
    t_full, x, op = _oracle_step_seconds(args.workload, n_full, args.op)
    n_sample = n_full
    if t_full > budget:
        n_sample = 2**12
        while n_sample * 2 < n_full:
            t, _, _ = _oracle_step_seconds(args.workload, n_sample * 2)
            if t > budget:
                break
            n_sample *= 2
        _, x, op = _oracle_step_seconds(args.workload, n_sample, args.op)
    from oracle import ring
    for _ in range(args.warmup):
        ring.ring_allreduce(x, op)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        ring.ring_allreduce(x, op)
        times.append(time.perf_counter() - t)
    t_step = statistics.mean(times)
    value = n_sample * b / t_step / 1e9
    what = "the full workload" if n_sample == n_full else "a sample: same recipe and seed as the workload"
    sample = f"R={w['R']} ranks x n={n_sample} per rank ({what}) per step; numpy oracle, one thread"
    cfg_args = argparse.Namespace(**vars(args))
    if n_sample != n_full:
        cfg_args.n = n_sample
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w["dtype"],
        "data": "synthetic",
        "config": workload_config(cfg_args, w["R"], n_sample, args.op or w["ops"][0], b, ws),
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
                         "host_cores": host_cores()},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------ sweep

SWEEP_VARIANTS = [
    ("direct", "direct", lambda ra: []),
    ("ring", "ring", lambda ra: []),
    ("persistent", "persistent", lambda ra: []),
    ("persistent_per_peer", "persistent", lambda ra: [(ra.Option.BARRIER, ra.Barrier.PER_PEER)]),
    ("persistent_cluster", "persistent", lambda ra: [(ra.Option.BARRIER, ra.Barrier.CLUSTER)]),
    ("pipelined", "pipelined", lambda ra: []),
    ("pipelined_ll", "pipelined", lambda ra: [(ra.Option.PROTOCOL, ra.Protocol.LL)]),
    ("pipelined_ll_cluster", "pipelined", lambda ra: [(ra.Option.PROTOCOL, ra.Protocol.LL_CLUSTER)]),
    ("local", "local", lambda ra: []),
]


def run_barriers(args):
    """Barrier cost, counting vs per-peer, as the rank count grows: the
    persistent variant on a tiny buffer (R x 256 fp32 elements, one channel),
    so each call is one cooperative launch plus 2R-3 barrier rounds; the
    pipelined variant on the same buffer for comparison.  One JSON line per R."""
    import torch
    from ring_allreduce_gb300 import build, inputs
    build.build()
    from ring_allreduce_gb300 import binding as ra
    for R in (2, 3, 4, 6, 8, 12, 16, 24, 32):
        n = 256 * R
        host = inputs.generate(R, n, "f32", "normal", inputs.SWEEP_SEED)
        _, ins = _device_ranks(torch, R, n, inputs.storage_dtype("f32"), host)
        _, outs = _device_ranks(torch, R, n, inputs.storage_dtype("f32"))
        line = {"barriers": "persistent, one channel", "R": R, "n_per_rank": n, "barrier_rounds": 2 * R - 3}
        for name, v, opts in (("counting", "persistent", []),
                              ("per_peer", "persistent", [(ra.Option.BARRIER, ra.Barrier.PER_PEER)]),
                              ("cluster", "persistent", [(ra.Option.BARRIER, ra.Barrier.CLUSTER)]),
                              ("pipelined", "pipelined", []),
                              ("pipelined_ll", "pipelined", [(ra.Option.PROTOCOL, ra.Protocol.LL)]),
                              ("pipelined_ll_cluster", "pipelined",
                               [(ra.Option.PROTOCOL, ra.Protocol.LL_CLUSTER)])):
            if name in ("cluster", "pipelined_ll_cluster") and R > 16:
                line[name] = None
                continue
            h = ra.RingAllReduce(R, n, "f32", "sum", variant=v)
            h.set_option(ra.Option.CTAS, 1)
            for key, value in opts:
                h.set_option(key, value)
            _, lm = _time_variant(torch, ra, h, ins, outs, 500, 20)
            _, lq = _time_variant(torch, ra, h, ins, outs, 300, 5, queued=True)
            assert h.device_status()[0] == ra.Status.OK
            h.close()
            line[name] = {"us_per_call": round(statistics.median(lm) * 1e3, 2),
                          "device_us": round(statistics.median(lq) * 1e3, 2)}
        print(json.dumps(line), flush=True)


def run_extras(args):
    """The collectives and dtypes beyond the headline workload, direct
    kernel, one JSON line each: AllReduce for every dtype (R = 8, n = 2^24),
    and ReduceScatter / AllGather with full and compact buffers, on an
    aligned plan (2^24 fp32) and a ragged one (2^26+3 bf16).  frac is the
    fraction of the measured copy bandwidth on the call's compulsory bytes."""
    import torch
    from ring_allreduce_gb300 import build, inputs
    build.build()
    from ring_allreduce_gb300 import binding as ra
    peak, _ = measured_peaks()
    R = 8

    def timed(fn, steps=50):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps / 1e3

    dists = {"f32": "normal", "bf16": "grad", "i32": "int20", "f16": "grad", "f64": "normal", "i64": "int40"}
    for dt in ("f32", "bf16", "i32", "f16", "f64", "i64"):
        n = 2**24
        b = inputs.itemsize(dt)
        host = inputs.generate(R, n, dt, dists[dt], 1)
        _, ins = _device_ranks(torch, R, n, inputs.storage_dtype(dt), host)
        _, outs = _device_ranks(torch, R, n, inputs.storage_dtype(dt))
        for op in ("sum", "max"):
            h = ra.RingAllReduce(R, n, dt, op)
            t = timed(lambda: h.allreduce(ins, outs))
            assert h.device_status()[0] == ra.Status.OK
            h.close()
            byts = 2 * R * n * b
            print(json.dumps({"extra": "allreduce", "dtype": dt, "op": op, "R": R, "n_per_rank": n,
                              "us": round(t * 1e6, 2), "algbw": round(n * b / t / 1e9, 2),
                              "frac": round(byts / t / 1e9 / peak, 4)}), flush=True)
        del ins, outs
        torch.cuda.empty_cache()
    for dt, n in (("f32", 2**24), ("bf16", 2**26 + 3), ("i32", 2**24)):
        b = inputs.itemsize(dt)
        st = inputs.storage_dtype(dt)
        host = inputs.generate(R, n, dt, dists[dt], 1)
        _, ins = _device_ranks(torch, R, n, st, host)
        full_big, full = _device_ranks(torch, R, n, st)
        h = ra.RingAllReduce(R, n, dt, "sum")
        lens = [h.owned_chunk(r)[1] for r in range(R)]
        cmp = [torch.empty(((L + 63) // 64) * 64, dtype=full_big.dtype, device="cuda")[:L] for L in lens]
        def gather_tma():
            hg.all_gather(full)

        hg = ra.RingAllReduce(R, n, dt, "sum")
        hg.set_option(ra.Option.GATHER, 2)
        cases = [
            ("reduce_scatter", lambda: h.reduce_scatter(ins, full), (R + 1) * n * b),
            ("all_gather", lambda: h.all_gather(full), R * n * b),
            ("all_gather_tma_broadcast", gather_tma, R * n * b),
            ("reduce_scatter_compact", lambda: h.reduce_scatter_compact(ins, cmp), (R + 1) * n * b),
            ("all_gather_compact", lambda: h.all_gather_compact(cmp, full), (R + 1) * n * b),
        ]
        for name, fn, byts in cases:
            t = timed(fn)
            print(json.dumps({"extra": name, "dtype": dt, "R": R, "n_per_rank": n,
                              "aligned_chunks": (-(-n // R) * b) % 16 == 0,
                              "us": round(t * 1e6, 2), "frac": round(byts / t / 1e9 / peak, 4),
                              "bytes": byts}), flush=True)
        assert h.device_status()[0] == ra.Status.OK
        assert hg.device_status()[0] == ra.Status.OK
        h.close()
        hg.close()
        del ins, full, full_big, cmp
        torch.cuda.empty_cache()


def run_l2(args):
    """Copy bandwidth through L2: a device copy (torch) of one buffer into
    another, both small enough to stay in the 129 MB L2, replayed 64 times
    from a CUDA graph so that launches do not count; bytes = read + write.
    The last line is a copy far larger than L2 (DRAM).  One JSON line per
    size: what a plain copy reaches when its data never leaves L2 -- the
    scale for the L2 traffic of the variants that pass their partials
    through memory."""
    import torch
    peak, _ = measured_peaks()
    for mib in (4, 8, 16, 24, 32, 48, 1024):
        nbytes = mib << 20
        src = torch.ones(nbytes // 4, dtype=torch.float32, device="cuda")
        dst = torch.empty_like(src)
        copies = 64 if mib <= 64 else 4
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            for _ in range(3):
                dst.copy_(src)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for _ in range(copies):
                dst.copy_(src)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        times = []
        for _ in range(7):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) / 1e3 / copies)
        t = statistics.median(times)
        print(json.dumps({"l2_copy_mib": mib, "us_per_copy": round(t * 1e6, 2),
                          "tb_per_s": round(2 * nbytes / t / 1e12, 2),
                          "of_measured_hbm": round(2 * nbytes / t / 1e9 / peak, 3)}), flush=True)
        del src, dst, g
        torch.cuda.empty_cache()


def run_sweep(args):
    """Latency/bandwidth sweep (R=8 fp32 sum over n, and R over 2..32 at
    n=2^24), every variant; one JSON line per point on stdout."""
    import torch
    from ring_allreduce_gb300 import build, inputs
    build.build()
    from ring_allreduce_gb300 import binding as ra
    peak, _ = measured_peaks()
    points = [(8, n) for n in inputs.SWEEP_N] + [(R, 2**24) for R in inputs.SWEEP_R if R != 8]
    for R, n in points:
        host = inputs.generate(R, n, "f32", "normal", inputs.SWEEP_SEED)
        _, ins = _device_ranks(torch, R, n, inputs.storage_dtype("f32"), host)
        _, outs = _device_ranks(torch, R, n, inputs.storage_dtype("f32"))
        line = {"sweep": "r8_f32_n" if R == 8 else "f32_R", "R": R, "n_per_rank": n}
        for name, v, opts in SWEEP_VARIANTS:
            if name in ("persistent_cluster", "pipelined_ll_cluster") and R > 16:
                line[name] = None
                continue
            h = ra.RingAllReduce(R, n, "f32", "sum", variant=v)
            for key, value in opts(ra):
                h.set_option(key, value)
            steps = 200 if n <= 2**20 else 30
            try:
                _, lm = _time_variant(torch, ra, h, ins, outs, steps, 10)
            except ra.RAError as e:
                # flag-in-data messages are for small chunks: above its inbox
                # limit the call is refused before any launch
                assert e.status == ra.Status.ERR_UNSUPPORTED, e
                h.close()
                line[name] = None
                continue
            assert h.device_status()[0] == ra.Status.OK
            h.close()
            t = statistics.median(lm) / 1e3
            line[name] = {"us": round(t * 1e6, 2), "algbw": round(n * 4 / t / 1e9, 2),
                       "busbw": round(n * 4 / t / 1e9 * 2 * (R - 1) / R, 2),
                       "frac_compulsory": round(2 * R * n * 4 / t / 1e9 / peak, 4)}
            if n <= 2**20:
                # small calls: also their device time, issued back to back
                h = ra.RingAllReduce(R, n, "f32", "sum", variant=v)
                for key, value in opts(ra):
                    h.set_option(key, value)
                _, lq = _time_variant(torch, ra, h, ins, outs, 200, 5, queued=True)
                assert h.device_status()[0] == ra.Status.OK
                h.close()
                line[name]["device_us"] = round(statistics.median(lq) * 1e3, 2)
        # reference, not a variant: a plain device copy (torch) of the same
        # R n b bytes read and written, timed the same way -- what a copy
        # reaches at this size
        src, dst = ins[0].new_empty(R * n), outs[0].new_empty(R * n)
        src.copy_(torch.cat(ins))
        steps = 200 if n <= 2**20 else 30
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for _ in range(10):
            dst.copy_(src)
        torch.cuda.synchronize()
        for a, bb in ev:
            a.record()
            dst.copy_(src)
            bb.record()
        torch.cuda.synchronize()
        t = statistics.median([a.elapsed_time(bb) for a, bb in ev]) / 1e3
        line["copy_same_bytes"] = {"us": round(t * 1e6, 2),
                                   "frac_compulsory": round(2 * R * n * 4 / t / 1e9 / peak, 4)}
        if n <= 2**20:
            torch.cuda._sleep(int(1e6 + 40000 * steps))
            for a, bb in ev:
                a.record()
                dst.copy_(src)
                bb.record()
            torch.cuda.synchronize()
            line["copy_same_bytes"]["device_us"] = round(
                statistics.median([a.elapsed_time(bb) for a, bb in ev]) * 1e3, 2)
        print(json.dumps(line), flush=True)
        del ins, outs, src, dst
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="r8_f32", choices=["r8_f32", "r8_bf16", "r16_i32", "r4_small"])
    ap.add_argument("--op", default=None, choices=["sum", "max"],
                    help="reduction of the workload (default: its first; r16_i32 runs sum and max)")
    ap.add_argument("--n", type=int, default=None, help="override n per rank (profiling of a smaller case)")
    ap.add_argument("--variant", default="auto", choices=["auto", "direct", "ring", "persistent", "pipelined", "local"])
    ap.add_argument("--protocol", default="simple", choices=["simple", "ll", "ll_cluster"],
                    help="message protocol of the pipelined variant")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--l2", action="store_true",
                    help="copy bandwidth through L2: a device copy over buffers that stay in L2, by size")
    ap.add_argument("--barriers", action="store_true", help="barrier cost vs R, counting vs per-peer")
    ap.add_argument("--extras", action="store_true", help="other dtypes and collectives (direct kernel)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws != args.gpus and ws > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={ws}")
    if args.impl == "reference":
        run_reference_arm(args)
    elif args.sweep:
        run_sweep(args)
    elif args.l2:
        run_l2(args)
    elif args.barriers:
        run_barriers(args)
    elif args.extras:
        run_extras(args)
    else:
        run_gpu_arm(args)


if __name__ == "__main__":
    main()
