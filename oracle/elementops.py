"""The reduction applied at each ring hop (test infrastructure only).

"Why AllReduce = ReduceScatter + AllGather -- NCCL Ring AllReduce", section 5
(rounds 1-3) and section 7: a rank that receives a partial result adds its
own chunk to it, ``new_partial = partial_sum + local_chunk``.  Section 1
names SUM as the reduction; MAX is the second operation this library
offers.  Each operation below is ``combine(incoming, local)`` applied
elementwise, with ``incoming`` the partial that arrived from the ring
predecessor and ``local`` the receiving rank's own input.

Precision (the page fixes the order of the additions, not the number
format; the readings below are the plain ones):

* fp32 SUM: one IEEE binary32 addition, round-to-nearest-even, no fused
  operation, no flush of subnormals (numpy float32 arithmetic).
* bf16 SUM: the partial is stored in bf16 at every hop, as a ring that
  ships bf16 messages would store it.  Both operands are widened to binary32
  exactly, added in binary32 and the sum is rounded to bf16 with
  round-to-nearest-even.  binary32 carries 24 significand bits, at least
  2*8+2, so this double rounding gives the correctly rounded bf16 sum.
* fp16 SUM: as bf16: both operands widened exactly to binary32, one
  binary32 addition, rounded to the nearest fp16, ties to even (24 >= 2*11+2,
  so this double rounding is the correctly rounded fp16 sum).
* fp64 SUM: one IEEE binary64 addition.
* int32 / int64 SUM: two's-complement wrap-around.
* MAX (every dtype): ``local if local > incoming else incoming``; on a tie,
  or when the comparison is false (NaN), the incoming partial is kept.

bf16 values are held as their 16-bit patterns in ``numpy.uint16`` arrays;
fp16 values in ``numpy.float16`` arrays.
"""

import numpy as np

__all__ = ["OPS", "get_op", "bf16_bits_to_f32", "f32_to_bf16_bits_rne", "Sym"]


def bf16_bits_to_f32(bits):
    """Widen bf16 bit patterns (uint16) to float32 exactly: bf16 is the top
    half of a binary32 word, so shifting the pattern left by 16 is exact."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16_bits_rne(values):
    """Round float32 values to bf16 bit patterns, round-to-nearest-even.

    A binary32 word ``b`` keeps its top 16 bits.  The 16 bits dropped are
    compared with half an ulp (0x8000): above rounds up, below rounds down,
    exactly half rounds to the neighbour whose last kept bit is 0.  Adding
    0x7FFF plus the last kept bit and truncating does exactly that, and a
    carry out of the significand moves into the exponent (the largest finite
    values round to infinity, as they must).  NaN keeps its sign and top
    bits and is made quiet.
    """
    f = np.ascontiguousarray(values, dtype=np.float32)
    b = f.view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    rounded = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    is_nan = (b & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    quiet = (b >> np.uint32(16)) | np.uint32(0x0040)
    return np.where(is_nan, quiet, rounded).astype(np.uint16)


class _Op:
    name = ""
    storage = None      # numpy dtype the values are stored in
    itemsize = 0        # bytes per element on the wire

    def combine(self, incoming, local):  # pragma: no cover - interface
        raise NotImplementedError


class F32Sum(_Op):
    name, storage, itemsize = "f32_sum", np.float32, 4

    def combine(self, incoming, local):
        return np.add(incoming, local, dtype=np.float32)


class F32Max(_Op):
    name, storage, itemsize = "f32_max", np.float32, 4

    def combine(self, incoming, local):
        return np.where(local > incoming, local, incoming).astype(np.float32)


class BF16Sum(_Op):
    name, storage, itemsize = "bf16_sum", np.uint16, 2

    def combine(self, incoming, local):
        s = np.add(bf16_bits_to_f32(incoming), bf16_bits_to_f32(local), dtype=np.float32)
        return f32_to_bf16_bits_rne(s)


class BF16Max(_Op):
    name, storage, itemsize = "bf16_max", np.uint16, 2

    def combine(self, incoming, local):
        take_local = bf16_bits_to_f32(local) > bf16_bits_to_f32(incoming)
        return np.where(take_local, local, incoming).astype(np.uint16)


class I32Sum(_Op):
    name, storage, itemsize = "i32_sum", np.int32, 4

    def combine(self, incoming, local):
        wide = np.asarray(incoming, dtype=np.int64) + np.asarray(local, dtype=np.int64)
        # two's-complement wrap to 32 bits
        return ((wide + 2**31) % 2**32 - 2**31).astype(np.int32)


class I32Max(_Op):
    name, storage, itemsize = "i32_max", np.int32, 4

    def combine(self, incoming, local):
        return np.where(local > incoming, local, incoming).astype(np.int32)


class F16Sum(_Op):
    name, storage, itemsize = "f16_sum", np.float16, 2

    def combine(self, incoming, local):
        wide = np.add(np.asarray(incoming, dtype=np.float16).astype(np.float32),
                      np.asarray(local, dtype=np.float16).astype(np.float32), dtype=np.float32)
        with np.errstate(over="ignore"):      # a sum beyond fp16's range rounds to infinity
            return wide.astype(np.float16)


class F16Max(_Op):
    name, storage, itemsize = "f16_max", np.float16, 2

    def combine(self, incoming, local):
        take_local = np.asarray(local, np.float16).astype(np.float32) > np.asarray(incoming, np.float16).astype(np.float32)
        return np.where(take_local, local, incoming).astype(np.float16)


class F64Sum(_Op):
    name, storage, itemsize = "f64_sum", np.float64, 8

    def combine(self, incoming, local):
        return np.add(incoming, local, dtype=np.float64)


class F64Max(_Op):
    name, storage, itemsize = "f64_max", np.float64, 8

    def combine(self, incoming, local):
        return np.where(local > incoming, local, incoming).astype(np.float64)


class I64Sum(_Op):
    name, storage, itemsize = "i64_sum", np.int64, 8

    def combine(self, incoming, local):
        # unsigned addition wraps modulo 2^64; reinterpreted as two's complement
        u = np.add(np.asarray(incoming, np.int64).view(np.uint64), np.asarray(local, np.int64).view(np.uint64),
                   dtype=np.uint64)
        return u.view(np.int64)


class I64Max(_Op):
    name, storage, itemsize = "i64_max", np.int64, 8

    def combine(self, incoming, local):
        return np.where(local > incoming, local, incoming).astype(np.int64)


class Sym(_Op):
    """Symbolic elements for the page's worked example.

    Each value is a tuple of term names; the reduction appends the local
    terms to the incoming ones, so a result records every contribution in
    the order the ring folded it (``("b1", "c1", "d1", "a1")`` is
    ``((b1 + c1) + d1) + a1``).  Values live in numpy object arrays.
    """

    name, storage, itemsize = "sym", object, 1

    def combine(self, incoming, local):
        out = np.empty(len(incoming), dtype=object)
        for i in range(len(incoming)):
            out[i] = tuple(incoming[i]) + tuple(local[i])
        return out


OPS = {
    ("f32", "sum"): F32Sum(),
    ("f32", "max"): F32Max(),
    ("bf16", "sum"): BF16Sum(),
    ("bf16", "max"): BF16Max(),
    ("i32", "sum"): I32Sum(),
    ("i32", "max"): I32Max(),
    ("f16", "sum"): F16Sum(),
    ("f16", "max"): F16Max(),
    ("f64", "sum"): F64Sum(),
    ("f64", "max"): F64Max(),
    ("i64", "sum"): I64Sum(),
    ("i64", "max"): I64Max(),
}


def get_op(dtype, op):
    """Return the reduction for ``dtype`` in {"f32", "bf16", "i32", "f16",
    "f64", "i64"} and ``op`` in {"sum", "max"}."""
    try:
        return OPS[(dtype, op)]
    except KeyError:
        raise ValueError(f"unsupported dtype/op {dtype}/{op}") from None
