"""Build the CUDA library libra_gb300.so in-tree, for sm_103a only.

``python -m ring_allreduce_gb300.build`` (or ``build()``) compiles every
translation unit under ``csrc/`` with nvcc in parallel into ``_build/`` and
links ``libra_gb300.so`` next to this file.  Nothing is rebuilt when the
library is newer than every source and header and the flags are unchanged.
Set RA_PTXAS_VERBOSE=1 to print ptxas register / spill / shared-memory use.
``build(debug=True)`` builds ``libra_gb300_debug.so`` from the same sources
with -DRA_DEBUG_BOUNDS (into ``_build_debug/``): every global access of every
kernel is checked against the byte ranges registered for the call, and
violations are counted and skipped (``ra_debug_bounds_report``).
"""

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libra_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
DEBUG_BUILD_DIR = os.path.join(HERE, "_build_debug")
DEBUG_LIB_PATH = os.path.join(HERE, "libra_gb300_debug.so")

SOURCES = ["ra_host.cpp", "ra_direct.cu", "ra_round.cu", "ra_persistent.cu", "ra_pipelined.cu", "ra_compact.cu",
           "ra_bcast.cu", "ra_static.cu", "ra_local.cu", "ra_ll.cu"]
# (source, object stem, preprocessor definitions): ra_direct_inst.cu is
# compiled once per dtype so its instantiations build in parallel
DTYPES = ["RA_F32", "RA_BF16", "RA_I32", "RA_F16", "RA_F64", "RA_I64"]
UNITS = ([(src, os.path.splitext(src)[0], {}) for src in SOURCES] +
         [("ra_direct_inst.cu", "ra_direct_" + dt[3:].lower(), {"RA_INST_DTYPE": dt}) for dt in DTYPES])
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# IEEE arithmetic throughout: no fast-math, no flush to zero, no contraction.
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "-ftz=false",
         "-prec-div=true", "-prec-sqrt=true", "-fmad=false"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libra_gb300.so")
    return cand


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "ra.h"))
    files.append(os.path.abspath(__file__))
    return sorted(f for f in files if os.path.isfile(f))


# The files each kernel's device code is built from.
KERNEL_SOURCES = {
    "direct": ["ra_direct.cu", "ra_direct.cuh", "ra_direct_inst.cu", "ra_device.cuh", "ra_internal.h"],
    "round": ["ra_round.cu", "ra_device.cuh", "ra_internal.h"],
    "persistent": ["ra_persistent.cu", "ra_signal.cuh", "ra_device.cuh", "ra_internal.h"],
    "pipelined": ["ra_pipelined.cu", "ra_signal.cuh", "ra_device.cuh", "ra_internal.h"],
    "compact": ["ra_compact.cu", "ra_device.cuh", "ra_internal.h"],
    "bcast": ["ra_bcast.cu", "ra_device.cuh", "ra_internal.h"],
    "local": ["ra_local.cu", "ra_device.cuh", "ra_internal.h"],
    "ll": ["ra_ll.cu", "ra_ll.h", "ra_device.cuh", "ra_internal.h"],
}


def kernel_source_hash(kernel=None):
    """Short hash of the sources of one kernel (``KERNEL_SOURCES``), or of
    every CUDA / C++ source and the public header when ``kernel`` is None.
    A profile summary taken on another hash describes a different kernel."""
    h = hashlib.sha256()
    files = KERNEL_SOURCES[kernel] if kernel else sorted(os.listdir(CSRC))
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    if kernel is None:
        with open(os.path.join(INCLUDE, "ra.h"), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _stamp(extra):
    h = hashlib.sha256(" ".join(ARCH + FLAGS + extra).encode())
    for f in _inputs():
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def build(force=False, verbose=None, jobs=None, debug=False):
    """Compile and link the library (the bounds-checked one with debug=True);
    returns its path."""
    verbose = os.environ.get("RA_PTXAS_VERBOSE") == "1" if verbose is None else verbose
    extra = (["-Xptxas", "-v"] if verbose else []) + (["-DRA_DEBUG_BOUNDS"] if debug else [])
    build_dir, lib_path = (DEBUG_BUILD_DIR, DEBUG_LIB_PATH) if debug else (BUILD_DIR, LIB_PATH)
    stamp = _stamp(extra)
    stamp_file = os.path.join(build_dir, "stamp")
    if not force and os.path.exists(lib_path) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(unit):
        src, stem, defs = unit
        obj = os.path.join(build_dir, stem + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, *[f"-D{k}={v}" for k, v in defs.items()],
               "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        return stem, obj, res

    with ThreadPoolExecutor(max_workers=jobs or min(len(UNITS), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, UNITS))
    failed = [(s, r) for s, _, r in results if r.returncode != 0]
    for s, _, r in results:
        if verbose or r.returncode != 0:
            sys.stderr.write(f"--- {s}\n{r.stdout}{r.stderr}")
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(s for s, _ in failed))
    objs = [o for _, o, _ in results]
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError(f"link of {os.path.basename(lib_path)} failed")
    os.replace(tmp, lib_path)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
