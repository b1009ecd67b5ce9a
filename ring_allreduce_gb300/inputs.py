"""Seeded synthetic rank inputs for the ring AllReduce workloads.

The test suite hands the same bytes to the CPU oracle and to the CUDA
library, and ``bench.py`` uploads them to the GPU.  This module holds none of
the method's arithmetic: it only draws random numbers (numpy PCG64, one
generator per workload, ranks drawn one after another r = 0..R-1) and casts
them to the storage format.  The cast to bf16 goes through torch's
float32 -> bfloat16 conversion.

Workloads (gradient-shaped buffers, no dataset involved):

=========  ===  =========  =====  ==========================================  ====  ====
name        R   n / rank   dtype  values                                       op    seed
=========  ===  =========  =====  ==========================================  ====  ====
r4_small    4   4096       f32    uniform integers in [-8, 8]                  sum   0
r8_f32      8   2^24       f32    i.i.d. N(0, 1)                               sum   1
r8_bf16     8   2^26+3     bf16   N(0, 1e-3) (sigma), 1 % of entries x100      sum   2
r16_i32    16   2^24       i32    uniform integers in [-2^20, 2^20]            sum,  3
                                                                               max
sweep       8   2^10..2^26 f32    N(0, 1), generator re-seeded for each size   sum   4
sweep_R   2..32 2^24       f32    N(0, 1)                                      sum   4
=========  ===  =========  =====  ==========================================  ====  ====
"""

import numpy as np

__all__ = ["WORKLOADS", "DISTS", "generate", "workload_inputs", "storage_dtype", "itemsize"]

# dtype name -> numpy storage dtype (bf16 is held as its 16-bit pattern)
_STORAGE = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32, "f16": np.float16, "f64": np.float64,
            "i64": np.int64}
_ITEMSIZE = {"f32": 4, "bf16": 2, "i32": 4, "f16": 2, "f64": 8, "i64": 8}

WORKLOADS = {
    "r4_small": dict(R=4, n=4096, dtype="f32", ops=("sum",), dist="int8", seed=0),
    "r8_f32": dict(R=8, n=2**24, dtype="f32", ops=("sum",), dist="normal", seed=1),
    "r8_bf16": dict(R=8, n=2**26 + 3, dtype="bf16", ops=("sum",), dist="grad", seed=2),
    "r16_i32": dict(R=16, n=2**24, dtype="i32", ops=("sum", "max"), dist="int20", seed=3),
}

SWEEP_N = [2**e for e in range(10, 27, 2)]
SWEEP_R = [2, 4, 8, 16, 32]
SWEEP_SEED = 4


def storage_dtype(dtype):
    return _STORAGE[dtype]


def itemsize(dtype):
    return _ITEMSIZE[dtype]


def _to_bf16_bits(v32):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _to_f16(v32):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32))
    return t.to(torch.float16).numpy().copy()


def _draw(rng, n, dist, dtype):
    if dist == "int8":
        v = rng.integers(-8, 8, endpoint=True, size=n).astype(np.float64)
    elif dist == "normal":
        if dtype == "f32":
            return rng.standard_normal(n, dtype=np.float32)
        v = rng.standard_normal(n)
    elif dist == "grad":
        v = rng.normal(0.0, 1e-3, size=n)
        mask = rng.random(n) < 0.01
        v[mask] *= 100.0
    elif dist == "int20":
        if dtype in ("i32", "i64"):
            return rng.integers(-2**20, 2**20, endpoint=True, size=n, dtype=_STORAGE[dtype])
        v = rng.integers(-2**20, 2**20, endpoint=True, size=n).astype(np.float64)
    elif dist == "int40":
        if dtype == "i64":
            return rng.integers(-2**40, 2**40, endpoint=True, size=n, dtype=np.int64)
        v = rng.integers(-2**40, 2**40, endpoint=True, size=n).astype(np.float64)
    elif dist == "uniform":
        v = rng.uniform(-1.0, 1.0, size=n)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    if dtype == "f32":
        return v.astype(np.float32)
    if dtype == "bf16":
        return _to_bf16_bits(v.astype(np.float32))
    if dtype == "i32":
        return np.clip(np.rint(v), -2**31, 2**31 - 1).astype(np.int32)
    if dtype == "f16":
        return _to_f16(v.astype(np.float32))
    if dtype == "f64":
        return v.astype(np.float64)
    if dtype == "i64":
        return np.rint(v).astype(np.int64)
    raise ValueError(f"unknown dtype {dtype!r}")


DISTS = ("int8", "normal", "grad", "int20", "int40", "uniform")


def generate(R, n, dtype, dist, seed):
    """R rank inputs of n elements each, drawn rank after rank from
    ``numpy.random.default_rng(seed)``.  Returns a list of numpy arrays in
    the storage dtype (float32, uint16 bf16 patterns, int32, float16,
    float64 or int64)."""
    rng = np.random.default_rng(seed)
    return [_draw(rng, n, dist, dtype) for _ in range(R)]


def workload_inputs(name, n=None, R=None):
    """Inputs of a named workload; ``n`` / ``R`` override its size (the
    recipe, seed and dtype stay the same)."""
    w = WORKLOADS[name]
    return generate(R if R is not None else w["R"], n if n is not None else w["n"],
                    w["dtype"], w["dist"], w["seed"])
