"""The seeded input generators that both the oracle and the kernels take
their inputs from: deterministic, rank after rank from one numpy PCG64
stream, and each named workload drawn to its stated recipe (values,
storage type, seed).  No GPU needed."""

import numpy as np
import pytest

from oracle import elementops
from ring_allreduce_gb300 import inputs


def test_same_seed_same_inputs_and_ranks_drawn_in_order():
    a = inputs.generate(3, 1000, "f32", "normal", 5)
    b = inputs.generate(3, 1000, "f32", "normal", 5)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    # ranks are consecutive draws of one stream: rank 1 of R=3 is rank 1 of R=2
    c = inputs.generate(2, 1000, "f32", "normal", 5)
    np.testing.assert_array_equal(a[1], c[1])
    assert not np.array_equal(a[0], a[1])
    assert not np.array_equal(a[0], inputs.generate(1, 1000, "f32", "normal", 6)[0])


@pytest.mark.parametrize("name,storage", [("r4_small", np.float32), ("r8_f32", np.float32),
                                          ("r8_bf16", np.uint16), ("r16_i32", np.int32)])
def test_workload_recipes(name, storage):
    w = inputs.WORKLOADS[name]
    n = 200_000
    x = inputs.generate(2, n, w["dtype"], w["dist"], w["seed"])
    assert all(r.dtype == storage and r.shape == (n,) for r in x)
    np.testing.assert_array_equal(x[0], inputs.workload_inputs(name, n=n, R=2)[0])
    if w["dist"] == "int8":        # integers in [-8, 8]
        v = np.concatenate(x)
        assert np.array_equal(v, np.rint(v)) and v.min() == -8 and v.max() == 8
    elif w["dist"] == "normal":    # N(0, 1)
        v = np.concatenate(x).astype(np.float64)
        assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01
    elif w["dist"] == "grad":      # N(0, 1e-3), 1 % of the values x 100 (bf16 patterns)
        v = np.abs(elementops.bf16_bits_to_f32(np.concatenate(x)).astype(np.float64))
        big = v > 0.02             # beyond 20 sigma of N(0, 1e-3): the scaled ones, nearly all of them
        assert 0.007 < big.mean() < 0.011
        assert 0.66e-3 < np.median(v[~big]) < 0.69e-3   # median of |N(0, 1e-3)|: 0.674e-3
    elif w["dist"] == "int20":     # integers in [-2^20, 2^20]
        v = np.concatenate(x)
        assert v.min() >= -2**20 and v.max() <= 2**20 and v.min() < -2**19 and v.max() > 2**19
    assert w["seed"] == {"r4_small": 0, "r8_f32": 1, "r8_bf16": 2, "r16_i32": 3}[name]
