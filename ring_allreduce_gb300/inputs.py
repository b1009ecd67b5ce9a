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

The ``special`` distribution (floating-point dtypes, edge-case tests only) mixes
IEEE special values into the draws: signed zeros, the smallest and largest
subnormals, the smallest normal, +-1 and 1 + ulp, half an ulp of 1 and a quarter
(so that sums hit rounding ties), half the largest finite value and the largest
finite value (so that sums overflow), infinities and a quiet NaN, and values of
random sign and significand spread over the whole exponent range.
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


# significand bits (hidden bit included) and exponent range of the float
# formats, for the ``special`` draws
_FLOAT_FORMAT = {"f32": (24, -126, 127), "bf16": (8, -126, 127), "f16": (11, -14, 15), "f64": (53, -1022, 1023)}


def _special_bits16(rng, n):
    """bf16 bit patterns of the ``special`` distribution."""
    table = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x807F, 0x0080, 0x8080,
                      0x3F80, 0xBF80, 0x3F81, 0xBF81, 0x3B80, 0xBB80, 0x3B00, 0x3B00 | 0x8000,
                      0x7F7F, 0xFF7F, 0x7EFF, 0xFEFF], dtype=np.uint16)
    kind = rng.random(n)
    pick = table[rng.integers(0, len(table), size=n)]
    p, emin, emax = _FLOAT_FORMAT["bf16"]
    wide = np.ldexp(rng.uniform(1.0, 2.0, size=n) * rng.choice([-1.0, 1.0], size=n),
                    rng.integers(emin, emax, endpoint=True, size=n)).astype(np.float32)
    spread = _to_bf16_bits(wide)
    out = np.where(kind < 0.45, spread, pick)
    out = np.where((kind >= 0.90) & (kind < 0.94), np.uint16(0x7F80), out)
    out = np.where((kind >= 0.94) & (kind < 0.98), np.uint16(0xFF80), out)
    out = np.where(kind >= 0.98, np.uint16(0x7FC0), out)
    return out.astype(np.uint16)


def _special_float(rng, n, dtype):
    """f32 / f16 / f64 values of the ``special`` distribution."""
    ft = {"f32": np.float32, "f16": np.float16, "f64": np.float64}[dtype]
    fi = np.finfo(ft)
    p, emin, emax = _FLOAT_FORMAT[dtype]
    sub_max = ft(fi.smallest_normal) - ft(fi.smallest_subnormal)
    one = ft(1.0)
    table = np.array([0.0, -0.0, fi.smallest_subnormal, -fi.smallest_subnormal, sub_max, -sub_max,
                      fi.smallest_normal, -fi.smallest_normal, 1.0, -1.0, one + fi.eps, -(one + fi.eps),
                      np.ldexp(1.0, -p), -np.ldexp(1.0, -p), np.ldexp(1.0, -p - 1), -np.ldexp(1.0, -p - 1),
                      fi.max, -fi.max, ft(fi.max) / ft(2), -(ft(fi.max) / ft(2))], dtype=ft)
    kind = rng.random(n)
    pick = table[rng.integers(0, len(table), size=n)]
    with np.errstate(over="ignore"):
        spread = np.ldexp(rng.uniform(1.0, 2.0, size=n) * rng.choice([-1.0, 1.0], size=n),
                          rng.integers(emin, emax, endpoint=True, size=n)).astype(ft)
    out = np.where(kind < 0.45, spread, pick)
    out = np.where((kind >= 0.90) & (kind < 0.94), ft(np.inf), out)
    out = np.where((kind >= 0.94) & (kind < 0.98), ft(-np.inf), out)
    out = np.where(kind >= 0.98, ft(np.nan), out)
    return out.astype(ft)


def _draw(rng, n, dist, dtype):
    if dist == "special":
        if dtype == "bf16":
            return _special_bits16(rng, n)
        if dtype in ("f32", "f16", "f64"):
            return _special_float(rng, n, dtype)
        raise ValueError("the special distribution is for floating-point dtypes")
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


DISTS = ("int8", "normal", "grad", "int20", "int40", "uniform", "special")


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
