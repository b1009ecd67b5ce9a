"""Numeric pins of the oracle: every check compares it with something that
does not come from the oracle itself (closed forms, folds through other
arithmetic -- numpy float32 scalars, torch's bfloat16, Python integers --,
error bounds of recursive summation, and values the ring page fixes)."""

import math

import numpy as np
import pytest
import torch

from oracle import elementops, ring
from ring_allreduce_gb300 import inputs

DTYPE_OPS = [("f32", "sum"), ("f32", "max"), ("bf16", "sum"), ("bf16", "max"),
             ("i32", "sum"), ("i32", "max"), ("f16", "sum"), ("f16", "max"),
             ("f64", "sum"), ("f64", "max"), ("i64", "sum"), ("i64", "max")]
DIST = {"f32": "normal", "bf16": "normal", "i32": "int20", "f16": "normal", "f64": "normal", "i64": "int40"}


# ---------------------------------------------------------------- chunk plan

def test_chunk_plan_workloads():
    """C = ceil(n/R); the ragged bf16 workload (n = 2^26+3, R = 8) has
    C = 8,388,609 and a last chunk of 8,388,604."""
    plan = ring.chunk_plan(8, 2**26 + 3)
    assert plan[0] == (0, 8388609)
    assert plan[7] == (7 * 8388609, 8388604)
    assert ring.chunk_plan(4, 4096) == [(0, 1024), (1024, 1024), (2048, 1024), (3072, 1024)]
    assert all(L == 2**20 for _, L in ring.chunk_plan(16, 2**24))


@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 8, 16, 32])
def test_chunk_plan_partitions(R):
    for n in list(range(0, 3 * R + 3)) + [1000, 1001, 2**20 + 7]:
        plan = ring.chunk_plan(R, n)
        assert len(plan) == R
        pos = 0
        for off, L in plan:
            assert off == pos and L >= 0
            pos += L
        assert pos == n
        C = -(-n // R)
        assert all(L <= C for _, L in plan)
        # only the tail is short: lengths never increase
        assert all(plan[k][1] >= plan[k + 1][1] for k in range(R - 1))


def test_chunk_plan_small_n_has_empty_trailing_chunks():
    assert ring.chunk_plan(4, 2) == [(0, 1), (1, 1), (2, 0), (2, 0)]
    assert ring.chunk_plan(4, 5) == [(0, 2), (2, 2), (4, 1), (5, 0)]
    assert ring.chunk_plan(3, 0) == [(0, 0), (0, 0), (0, 0)]


# ---------------------------------------------------------- bf16 rounding

def _torch_bf16_bits(f32):
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_rounding_matches_torch_on_random_patterns():
    rng = np.random.default_rng(123)
    bits = rng.integers(0, 2**32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    np.testing.assert_array_equal(elementops.f32_to_bf16_bits_rne(f), _torch_bf16_bits(f))


def test_bf16_rounding_hand_cases():
    cases = [
        (1.0, 0x3F80),
        (1.0 + 2.0**-8, 0x3F80),          # exactly half an ulp above 1: tie, even is 1.0
        (1.0 + 3 * 2.0**-8, 0x3F82),      # tie between 0x3F81 (odd) and 0x3F82 (even)
        (1.0 + 2.0**-8 + 2.0**-20, 0x3F81),   # just above the tie rounds up
        (-1.0 - 2.0**-8, 0xBF80),
        (float(np.finfo(np.float32).max), 0x7F80),   # rounds to +inf
        (2.0**-149, 0x0000),              # smallest subnormal: below half of bf16's smallest
        (2.0**-133, 0x0001),              # bf16's smallest subnormal
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (float("inf"), 0x7F80),
    ]
    f = np.array([c[0] for c in cases], dtype=np.float32)
    got = elementops.f32_to_bf16_bits_rne(f)
    assert [int(g) for g in got] == [c[1] for c in cases]
    nan = elementops.f32_to_bf16_bits_rne(np.array([np.nan], dtype=np.float32))
    assert math.isnan(float(elementops.bf16_bits_to_f32(nan)[0]))


def test_bf16_widen_is_exact():
    bits = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    f = elementops.bf16_bits_to_f32(bits)
    finite = np.isfinite(f)
    back = elementops.f32_to_bf16_bits_rne(f[finite])
    np.testing.assert_array_equal(back, bits[finite])
    np.testing.assert_array_equal(f[finite], torch.from_numpy(bits[finite].view(np.int16))
                                  .view(torch.bfloat16).float().numpy())


def test_bf16_sum_matches_torch_bfloat16_add():
    rng = np.random.default_rng(7)
    a = inputs.generate(1, 200_000, "bf16", "grad", 11)[0]
    b = inputs.generate(1, 200_000, "bf16", "normal", 12)[0]
    # also sums of values of very different magnitude
    c = _torch_bf16_bits((rng.standard_normal(50_000) * 2.0 ** rng.integers(-30, 30, 50_000)))
    d = _torch_bf16_bits(rng.standard_normal(50_000))
    for x, y in ((a, b), (c, d), (b, a)):
        tx = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
        ty = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16)
        want = (tx + ty).view(torch.int16).numpy().view(np.uint16)
        got = elementops.get_op("bf16", "sum").combine(x, y)
        np.testing.assert_array_equal(got, want)


# -------------------------------------------------- brute force, tiny sizes

def _brute_allreduce(x, dtype, op):
    """Direct fold of each element in ring order, through arithmetic the
    oracle does not use: numpy float32 scalars, torch bfloat16 scalars,
    Python integers with an explicit 32-bit wrap."""
    R = len(x)
    n = len(x[0])
    C = -(-n // R) if n else 0
    res = []
    for i in range(n):
        k = i // C
        order = [(k + j) % R for j in range(R)]
        if dtype == "f32":
            acc = np.float32(x[order[0]][i])
            for q in order[1:]:
                v = np.float32(x[q][i])
                acc = (acc + v) if op == "sum" else (v if v > acc else acc)
            res.append(acc)
        elif dtype == "bf16":
            def t(q):
                return torch.tensor([int(np.int16(x[q][i].view(np.int16)))],
                                    dtype=torch.int16).view(torch.bfloat16)
            acc = t(order[0])
            for q in order[1:]:
                v = t(q)
                if op == "sum":
                    acc = acc + v
                else:
                    acc = v if bool(v.float() > acc.float()) else acc
            res.append(np.uint16(int(acc.view(torch.int16)) & 0xFFFF))
        elif dtype == "f16":
            acc = torch.tensor(float(x[order[0]][i]), dtype=torch.float16)
            for q in order[1:]:
                v = torch.tensor(float(x[q][i]), dtype=torch.float16)
                acc = (acc + v) if op == "sum" else (v if bool(v > acc) else acc)
            res.append(np.float16(acc.item()))
        elif dtype == "f64":
            acc = float(x[order[0]][i])            # Python floats are IEEE binary64
            for q in order[1:]:
                v = float(x[q][i])
                acc = (acc + v) if op == "sum" else (v if v > acc else acc)
            res.append(np.float64(acc))
        else:
            bits = 32 if dtype == "i32" else 64
            acc = int(x[order[0]][i])
            for q in order[1:]:
                v = int(x[q][i])
                if op == "sum":
                    acc = (acc + v + 2**(bits - 1)) % 2**bits - 2**(bits - 1)
                else:
                    acc = v if v > acc else acc
            res.append(acc)
    return np.array(res, dtype=inputs.storage_dtype(dtype))


@pytest.mark.parametrize("dtype,op", DTYPE_OPS)
def test_brute_force_tiny(dtype, op):
    for R in range(2, 7):
        for n in range(0, 3 * R + 3):
            x = inputs.generate(R, n, dtype, DIST[dtype], seed=1000 * R + n)
            if dtype in ("i32", "i64") and n:
                x[0][0] = 2**(31 if dtype == "i32" else 63) - 1     # force a wrap in the sum
                x[1][0] = 5
            got = ring.ring_allreduce(x, elementops.get_op(dtype, op))
            want = _brute_allreduce(x, dtype, op)
            for r in range(R):
                np.testing.assert_array_equal(got[r].view(np.uint8), want.view(np.uint8))


# ------------------------------------------------------------ closed forms

@pytest.mark.parametrize("R", [2, 3, 4, 8, 16])
def test_closed_form_int_pattern(R):
    """x_r[i] = r*1000 + i  =>  S[i] = 1000 R(R-1)/2 + R i  (after the
    identifiable rank/element pattern of the GIN AlltoAll example)."""
    n = 5 * R + 3
    x = [np.arange(n, dtype=np.int32) + np.int32(1000 * r) for r in range(R)]
    out = ring.ring_allreduce(x, elementops.get_op("i32", "sum"))
    want = 1000 * R * (R - 1) // 2 + R * np.arange(n)
    for r in range(R):
        np.testing.assert_array_equal(out[r], want)


@pytest.mark.parametrize("R", [2, 5, 17, 30])
def test_closed_form_each_rank_once(R):
    """x_r = 2^r: the sum 2^R - 1 has bit r set exactly when rank r was
    counted, and only once; MAX gives 2^(R-1)."""
    n = 3 * R + 1
    x = [np.full(n, 1 << r, dtype=np.int32) for r in range(R)]
    s = ring.ring_allreduce(x, elementops.get_op("i32", "sum"))
    m = ring.ring_allreduce(x, elementops.get_op("i32", "max"))
    for r in range(R):
        assert (s[r] == (1 << R) - 1).all()
        assert (m[r] == 1 << (R - 1)).all()
    if R <= 24:
        xf = [v.astype(np.float32) for v in x]
        sf = ring.ring_allreduce(xf, elementops.get_op("f32", "sum"))
        assert (sf[0] == np.float32((1 << R) - 1)).all()


# ------------------------------------------------------ order sensitivity

@pytest.mark.parametrize("dtype,big", [("f32", 2.0**24), ("bf16", 256.0), ("f16", 2048.0), ("f64", 2.0**53)])
def test_ring_start_rank_and_order(dtype, big):
    """Chunk k holds big, 1, 1, -big on ranks k, k+1, k+2, k+3.  Folding
    from rank k gives ((big + 1) + 1) - big = 0 (each +1 is a tie that rounds
    to even); folding from any other rank gives 2.  The result therefore
    shows which rank a chunk's fold started at."""
    R, per = 4, 3
    n = R * per
    pattern = [big, 1.0, 1.0, -big]
    vals = [np.zeros(n, dtype=np.float32) for _ in range(R)]
    for k in range(R):
        for j in range(R):
            vals[(k + j) % R][k * per:(k + 1) * per] = pattern[j]
    if dtype == "bf16":
        x = [_torch_bf16_bits(v) for v in vals]
    elif dtype == "f16":
        x = [torch.from_numpy(v).to(torch.float16).numpy() for v in vals]
    elif dtype == "f64":
        x = [v.astype(np.float64) for v in vals]
    else:
        x = vals
    out = ring.ring_allreduce(x, elementops.get_op(dtype, "sum"))
    res = elementops.bf16_bits_to_f32(out[0]) if dtype == "bf16" else out[0]
    assert (res == 0).all()
    # the other starting ranks give 2 (checked with numpy f32 scalars, torch
    # bf16 / f16, Python binary64 floats)
    for start in range(1, R):
        order = [pattern[(start + j) % R] for j in range(R)]
        if dtype == "f32":
            acc = np.float32(order[0])
            for v in order[1:]:
                acc = acc + np.float32(v)
            assert acc == 2
        elif dtype == "f64":
            acc = order[0]
            for v in order[1:]:
                acc = acc + v
            assert acc == 2
        else:
            tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
            acc = torch.tensor(order[0], dtype=tdt)
            for v in order[1:]:
                acc = acc + torch.tensor(v, dtype=tdt)
            assert float(acc) == 2


# -------------------------------------------------------------- error bound

@pytest.mark.parametrize("R", [2, 8, 32])
def test_fp32_error_within_recursive_summation_bound(R):
    """|ring - exact| <= gamma_{R-1} * sum |x_r| with gamma_m = m u / (1 - m u),
    u = 2^-24 (recursive summation, any order)."""
    n = 4099
    x = inputs.generate(R, n, "f32", "normal", 77)
    out = ring.ring_allreduce(x, elementops.get_op("f32", "sum"))[0].astype(np.float64)
    u = 2.0**-24
    g = (R - 1) * u / (1 - (R - 1) * u)
    stacked = np.stack([v.astype(np.float64) for v in x])
    exact = np.array([math.fsum(stacked[:, i]) for i in range(n)])
    bound = g * np.abs(stacked).sum(axis=0)
    assert (np.abs(out - exact) <= bound).all()
    # and it is not simply the fp64 sum rounded once: the order shows
    assert (out != exact.astype(np.float32)).any() or R == 2


# ----------------------------------------------------- structural invariants

@pytest.mark.parametrize("dtype,op", DTYPE_OPS)
def test_allreduce_equals_reducescatter_then_allgather(dtype, op):
    for R, n in ((2, 9), (3, 10), (4, 4096), (5, 1001), (8, 8 * 257 + 3)):
        x = inputs.generate(R, n, dtype, "grad" if dtype in ("bf16", "f16") else DIST[dtype], R * n)
        o = elementops.get_op(dtype, op)
        ar = ring.ring_allreduce(x, o)
        rs = ring.ring_reduce_scatter(x, o)
        ag = ring.ring_all_gather(rs, o)
        for r in range(R):
            np.testing.assert_array_equal(ar[r], ag[r])
            np.testing.assert_array_equal(ar[r], ar[0])
        plan = ring.chunk_plan(R, n)
        for r in range(R):
            off, L = plan[ring.owned_chunk(R, r)]
            np.testing.assert_array_equal(rs[r][off:off + L], ar[0][off:off + L])


def test_reduce_scatter_leaves_other_chunks_alone():
    x = inputs.generate(4, 40, "f32", "normal", 3)
    rs = ring.ring_reduce_scatter(x, elementops.get_op("f32", "sum"), fill=np.float32(-7))
    plan = ring.chunk_plan(4, 40)
    for r in range(4):
        for k in range(4):
            off, L = plan[k]
            if k != ring.owned_chunk(4, r):
                assert (rs[r][off:off + L] == -7).all()


@pytest.mark.parametrize("R", [2, 3, 4, 8, 16])
def test_volume_per_rank(R):
    """Section 13 of the ring page: each rank sends (k-1) N/k in each phase,
    2N(k-1)/k in all; with a ragged n every chunk still crosses R-1 links in
    each phase, so all ranks together send 2(R-1) n elements."""
    n = 64 * R
    x = inputs.generate(R, n, "f32", "normal", 5)
    stats = {}
    ring.ring_allreduce(x, elementops.get_op("f32", "sum"), stats=stats)
    N = n * 4
    for r in range(R):
        assert stats["bytes_sent"][r] * R == 2 * N * (R - 1)
    n2 = 64 * R + 5
    x2 = inputs.generate(R, n2, "bf16", "grad", 5)
    ring.ring_allreduce(x2, elementops.get_op("bf16", "sum"), stats=stats)
    assert sum(stats["bytes_sent"]) == 2 * (R - 1) * n2 * 2
    stats_rs, stats_ag = {}, {}
    rs = ring.ring_reduce_scatter(x, elementops.get_op("f32", "sum"), stats=stats_rs)
    ring.ring_all_gather(rs, elementops.get_op("f32", "sum"), stats=stats_ag)
    for r in range(R):
        assert stats_rs["bytes_sent"][r] * R == N * (R - 1)
        assert stats_ag["bytes_sent"][r] * R == N * (R - 1)


def test_single_rank_is_a_copy():
    x = inputs.generate(1, 17, "f32", "normal", 9)
    out = ring.ring_allreduce(x, elementops.get_op("f32", "sum"))
    np.testing.assert_array_equal(out[0], x[0])


def test_workload_recipe_shapes():
    x = inputs.workload_inputs("r4_small")
    assert len(x) == 4 and all(v.dtype == np.float32 and len(v) == 4096 for v in x)
    assert all(((v >= -8) & (v <= 8) & (v == np.round(v))).all() for v in x)
    g = inputs.generate(2, 100_000, "bf16", "grad", 2)
    f = elementops.bf16_bits_to_f32(g[0])
    assert 5e-4 < np.std(f[np.abs(f) < 0.01]) < 2e-3
    assert 0.004 < np.mean(np.abs(f) > 0.02) < 0.02


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_max_tie_keeps_incoming(dtype):
    """MAX keeps the incoming partial unless the local value is strictly
    greater, so +0 and -0 meeting keep whichever arrived first.  Ranks 0,1
    hold (+0, -0) on chunk 0 and (-0, +0) on chunk 1 (R = 2, chunk k starts at
    rank k)."""
    pos, neg = np.float32(0.0), np.float32(-0.0)
    a = np.array([pos, pos, neg, neg], dtype=np.float32)   # rank 0
    b = np.array([neg, neg, pos, pos], dtype=np.float32)   # rank 1
    x = [a, b]
    if dtype == "bf16":
        x = [_torch_bf16_bits(v) for v in x]
    out = ring.ring_allreduce(x, elementops.get_op(dtype, "max"))
    bits = out[0].view(np.uint32 if dtype == "f32" else np.uint16)
    sign = np.uint32(0x80000000) if dtype == "f32" else np.uint16(0x8000)
    # chunk 0 starts at rank 0 (+0 first), chunk 1 at rank 1 (+0 first)
    assert ((bits & sign) == 0).all()



def test_f16_rounding_matches_torch():
    """float32 -> float16 round-to-nearest-even (numpy's conversion, which the
    oracle's fp16 hop uses) equals torch's conversion on random patterns."""
    rng = np.random.default_rng(321)
    bits = rng.integers(0, 2**32, size=500_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    with np.errstate(over="ignore"):      # values beyond fp16's range round to infinity
        a = f.astype(np.float16)
    b = torch.from_numpy(f).to(torch.float16).numpy()
    np.testing.assert_array_equal(a.view(np.uint16), b.view(np.uint16))


def test_f16_sum_matches_torch_float16_add():
    rng = np.random.default_rng(5)
    x = torch.from_numpy((rng.standard_normal(200_000) * 2.0 ** rng.integers(-14, 14, 200_000))
                         .astype(np.float32)).to(torch.float16)
    y = torch.from_numpy(rng.standard_normal(200_000).astype(np.float32)).to(torch.float16)
    want = (x + y).numpy()
    got = elementops.get_op("f16", "sum").combine(x.numpy(), y.numpy())
    np.testing.assert_array_equal(got.view(np.uint16), want.view(np.uint16))


@pytest.mark.parametrize("R", [2, 9, 62])
def test_closed_form_int64(R):
    """x_r = 2^r for 64-bit ranks: the sum 2^R - 1 counts every rank once;
    x_r[i] = r * 10^12 + i gives 10^12 R(R-1)/2 + R i."""
    n = 2 * R + 3
    x = [np.full(n, 1 << r, dtype=np.int64) for r in range(R)]
    s = ring.ring_allreduce(x, elementops.get_op("i64", "sum"))
    assert all((v == (1 << R) - 1).all() for v in s)
    y = [np.arange(n, dtype=np.int64) + np.int64(10**12 * r) for r in range(R)]
    t = ring.ring_allreduce(y, elementops.get_op("i64", "sum"))
    assert all((v == 10**12 * R * (R - 1) // 2 + R * np.arange(n)).all() for v in t)


# IEEE 754 facts for one addition a + b, written as bit patterns by hand:
# (a, b, a + b).  Ties go to the even neighbour, the overflow threshold is the
# largest finite value plus half its ulp, subnormals are exact, -0 + -0 = -0,
# +0 + -0 = +0, inf - inf is NaN (any NaN).
_NAN = None
_IEEE_SUMS = {
    "f32": [
        (0x7F800000, 0xFF800000, _NAN),          # inf + -inf
        (0x7F7FFFFF, 0x7F7FFFFF, 0x7F800000),    # max + max overflows
        (0xFF7FFFFF, 0xFF7FFFFF, 0xFF800000),
        (0x7F7FFFFF, 0x73000000, 0x7F800000),    # max + 2^103 (half its ulp): tie, odd max -> inf
        (0x7F7FFFFF, 0x72FFFFFF, 0x7F7FFFFF),    # just below the threshold stays max
        (0x80000000, 0x80000000, 0x80000000),    # -0 + -0
        (0x00000000, 0x80000000, 0x00000000),    # +0 + -0
        (0x80000000, 0x00000000, 0x00000000),
        (0x00000001, 0x00000001, 0x00000002),    # subnormals add exactly
        (0x00800000, 0x80000001, 0x007FFFFF),    # smallest normal - smallest subnormal
        (0x3F800000, 0x33800000, 0x3F800000),    # 1 + 2^-24: tie to even -> 1
        (0x3F800001, 0x33800000, 0x3F800002),    # (1 + 2^-23) + 2^-24: tie to even -> up
        (0x7FC00000, 0x3F800000, _NAN),          # NaN + 1
        (0x7F800000, 0x3F800000, 0x7F800000),    # inf + 1
    ],
    "bf16": [
        (0x7F80, 0xFF80, _NAN),
        (0x7F7F, 0x7F7F, 0x7F80),
        (0xFF7F, 0xFF7F, 0xFF80),
        (0x8000, 0x8000, 0x8000),
        (0x0000, 0x8000, 0x0000),
        (0x0001, 0x0001, 0x0002),
        (0x0080, 0x8001, 0x007F),
        (0x3F80, 0x3B80, 0x3F80),                # 1 + 2^-8: tie to even -> 1
        (0x3F81, 0x3B80, 0x3F82),                # (1 + 2^-7) + 2^-8: tie to even -> up
        (0x3F80, 0x3B81, 0x3F81),                # just above the tie rounds up
        (0x7FC0, 0x3F80, _NAN),
        (0x7F80, 0x3F80, 0x7F80),
    ],
    "f16": [
        (0x7C00, 0xFC00, _NAN),
        (0x7BFF, 0x7BFF, 0x7C00),
        (0x7BFF, 0x4C00, 0x7C00),                # 65504 + 16 = 65520: tie, odd max -> inf
        (0x7BFF, 0x4BFF, 0x7BFF),                # 65504 + 15.99: stays 65504
        (0x8000, 0x8000, 0x8000),
        (0x0000, 0x8000, 0x0000),
        (0x0001, 0x0001, 0x0002),
        (0x0400, 0x8001, 0x03FF),
        (0x3C00, 0x1000, 0x3C00),                # 1 + 2^-11: tie to even -> 1
        (0x3C01, 0x1000, 0x3C02),
        (0x7E00, 0x3C00, _NAN),
        (0x7C00, 0x3C00, 0x7C00),
    ],
    "f64": [
        (0x7FF0000000000000, 0xFFF0000000000000, _NAN),
        (0x7FEFFFFFFFFFFFFF, 0x7FEFFFFFFFFFFFFF, 0x7FF0000000000000),
        (0x8000000000000000, 0x8000000000000000, 0x8000000000000000),
        (0x0000000000000000, 0x8000000000000000, 0x0000000000000000),
        (0x0000000000000001, 0x0000000000000001, 0x0000000000000002),
        (0x0010000000000000, 0x8000000000000001, 0x000FFFFFFFFFFFFF),
        (0x3FF0000000000000, 0x3CA0000000000000, 0x3FF0000000000000),   # 1 + 2^-53
        (0x3FF0000000000001, 0x3CA0000000000000, 0x3FF0000000000002),
        (0x7FF8000000000000, 0x3FF0000000000000, _NAN),
        (0x7FF0000000000000, 0x3FF0000000000000, 0x7FF0000000000000),
    ],
}
_BITS = {"f32": (np.uint32, np.float32), "bf16": (np.uint16, np.uint16), "f16": (np.uint16, np.float16),
         "f64": (np.uint64, np.float64)}


def _bits_is_nan(dtype, bits):
    u = int(bits)
    if dtype == "f32":
        return (u & 0x7FFFFFFF) > 0x7F800000
    if dtype == "bf16":
        return (u & 0x7FFF) > 0x7F80
    if dtype == "f16":
        return (u & 0x7FFF) > 0x7C00
    return (u & 0x7FFFFFFFFFFFFFFF) > 0x7FF0000000000000


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "f64"])
def test_ieee_special_sums(dtype):
    """Each case as a two-rank ring over one element (chunk 0 holds it and
    starts at rank 0, so S = x_0 (+) x_1 with x_0 incoming): the oracle's
    result is the IEEE result written above, in every rank's output."""
    ubits, store = _BITS[dtype]
    op = elementops.get_op(dtype, "sum")
    for a, b, want in _IEEE_SUMS[dtype]:
        x = [np.array([a], dtype=ubits).view(store), np.array([b], dtype=ubits).view(store)]
        with np.errstate(all="ignore"):
            out = ring.ring_allreduce(x, op)
        for r in range(2):
            got = out[r].view(ubits)[0]
            if want is _NAN:
                assert _bits_is_nan(dtype, got), (dtype, hex(a), hex(b), hex(int(got)))
            else:
                assert int(got) == want, (dtype, hex(a), hex(b), hex(int(got)), hex(want))
