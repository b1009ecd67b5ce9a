"""The oracle's per-hop addition against the GPU's own adders.

The oracle adds bf16 and fp16 by widening both operands to binary32 exactly,
adding there and rounding the sum to nearest-even in the narrow format; fp32
and fp64 are single IEEE additions.  Here the same operand pairs are added by
PyTorch's CUDA elementwise kernels (not this library's kernels), on the GPU's
own arithmetic and format conversions, and the two must agree bit for bit for
every result that is a number.  Where the oracle's sum is NaN the GPU's must
be NaN too (IEEE 754 leaves a produced NaN's payload open).

Operands: the "special" draw (signed zeros, subnormals, the smallest normal,
rounding ties, overflow, infinities, NaN), normal values, and pairs of very
different magnitude, so that every rounding path of the narrow formats is
exercised."""

import numpy as np
import pytest

from oracle import elementops
from ring_allreduce_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

N = 1 << 18

_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "f64": torch.float64}
_BITS = {"f32": torch.int32, "bf16": torch.int16, "f16": torch.int16, "f64": torch.int64}


def _as_float(bits, dtype):
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return bits


def _pairs(dtype):
    x = inputs.generate(2, N, dtype, "special", 41)
    yield x[0], x[1]
    z = inputs.generate(2, N, dtype, "normal", 42)
    yield z[0], z[1]
    yield x[0], z[1]
    # very different magnitudes: every amount of alignment shift
    rng = np.random.default_rng(43)
    scale = 2.0 ** rng.integers(-40, 40, N)
    big = (rng.standard_normal(N) * scale).astype(np.float32)
    t = torch.from_numpy(big).to(_TORCH[dtype])
    bits = t.view(_BITS[dtype]).numpy()
    st = inputs.storage_dtype(dtype)
    yield bits.view(st), z[0]


def _gpu_add(a, b, dtype):
    ta = torch.from_numpy(np.ascontiguousarray(a).view(_np_bits(dtype))).cuda().view(_TORCH[dtype])
    tb = torch.from_numpy(np.ascontiguousarray(b).view(_np_bits(dtype))).cuda().view(_TORCH[dtype])
    s = (ta + tb).view(_BITS[dtype]).cpu().numpy()
    return s.view(inputs.storage_dtype(dtype))


def _np_bits(dtype):
    return {"f32": np.int32, "bf16": np.int16, "f16": np.int16, "f64": np.int64}[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32", "f64"])
def test_oracle_sum_matches_gpu_native_add(dtype):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    op = elementops.get_op(dtype, "sum")
    for a, b in _pairs(dtype):
        with np.errstate(all="ignore"):
            want = np.ascontiguousarray(op.combine(a, b))
        got = _gpu_add(a, b, dtype)
        wf, gf = _as_float(want, dtype), _as_float(got, dtype)
        nan_w, nan_g = np.isnan(wf), np.isnan(gf)
        bad = np.nonzero(nan_w != nan_g)[0]
        assert len(bad) == 0, f"{dtype}: NaN on one side only at {bad[:8].tolist()}"
        keep = ~nan_w
        diff = np.nonzero(want[keep].view(_np_bits(dtype)) != got[keep].view(_np_bits(dtype)))[0]
        assert len(diff) == 0, (f"{dtype}: {len(diff)} sums differ from the GPU's, first at "
                                f"{np.nonzero(keep)[0][diff[:4]].tolist()}")
