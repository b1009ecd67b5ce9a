"""Shared helpers of the test suite: rank buffers on the device with guard
bands, uploads of the seeded inputs, and comparisons with the oracle."""

import numpy as np

GUARD = 64          # elements of guard band before and after every rank buffer
SENTINEL = 0x5A     # byte value the guard bands and untouched outputs hold

_TORCH_DT = None


def torch_dtype(np_dtype):
    import torch
    return {np.dtype(np.float32): torch.float32, np.dtype(np.uint16): torch.int16,
            np.dtype(np.int32): torch.int32, np.dtype(np.float16): torch.float16,
            np.dtype(np.float64): torch.float64, np.dtype(np.int64): torch.int64}[np.dtype(np_dtype)]


def _stride(n):
    # row length in elements: guard + data + guard, rounded to 64 elements,
    # so every row (and every data start) stays 16-byte aligned
    return ((GUARD + n + GUARD + 63) // 64) * 64


class DeviceRanks:
    """R rank buffers of n elements inside one device tensor, each with a
    guard band on both sides filled with SENTINEL bytes."""

    def __init__(self, R, n, np_dtype, host=None):
        import torch
        self.R, self.n, self.np_dtype = R, n, np.dtype(np_dtype)
        self.stride = _stride(n)
        tdt = torch_dtype(np_dtype)
        self.big = torch.empty((R, self.stride), dtype=tdt, device="cuda")
        self.big.view(torch.uint8).fill_(SENTINEL)
        if host is not None:
            arr = np.ascontiguousarray(np.stack(host)).view(self.np_dtype)
            if self.np_dtype == np.uint16:
                arr = arr.view(np.int16)
            self.big[:, GUARD:GUARD + n] = torch.from_numpy(arr).to("cuda")
        self.views = [self.big[r, GUARD:GUARD + n] for r in range(R)]

    def ptrs(self):
        return [v.data_ptr() for v in self.views]

    def host(self):
        """The R buffers as numpy arrays of the storage dtype."""
        a = self.big[:, GUARD:GUARD + self.n].cpu().numpy()
        return [a[r].view(self.np_dtype) for r in range(self.R)]

    def guards_intact(self):
        import torch
        g = self.big.view(torch.uint8).view(self.R, -1)
        item = self.np_dtype.itemsize
        lo = g[:, :GUARD * item]
        hi = g[:, (GUARD + self.n) * item:]
        return bool((lo == SENTINEL).all()) and bool((hi == SENTINEL).all())


def assert_bitwise_equal(got, want, what=""):
    got = np.ascontiguousarray(got)
    want = np.ascontiguousarray(want)
    assert got.shape == want.shape, what
    gb, wb = got.view(np.uint8), want.view(np.uint8)
    if not np.array_equal(gb, wb):
        item = got.dtype.itemsize
        bad = np.nonzero((gb != wb).reshape(-1, item).any(axis=1))[0]
        raise AssertionError(f"{what}: {len(bad)} elements differ, first at {bad[:8].tolist()}: "
                             f"got {got[bad[:4]].tolist()} want {want[bad[:4]].tolist()}")


class DeviceBuffers:
    """Separately allocated device buffers of per-rank lengths (compact
    chunks), each with guard bands on both sides."""

    def __init__(self, lengths, np_dtype, host=None):
        import torch
        self.np_dtype = np.dtype(np_dtype)
        self.lengths = list(lengths)
        tdt = torch_dtype(np_dtype)
        self.bigs = []
        self.views = []
        for r, L in enumerate(self.lengths):
            big = torch.empty(GUARD + L + GUARD, dtype=tdt, device="cuda")
            big.view(torch.uint8).fill_(SENTINEL)
            if host is not None and L:
                arr = np.ascontiguousarray(host[r]).view(self.np_dtype)
                if self.np_dtype == np.uint16:
                    arr = arr.view(np.int16)
                big[GUARD:GUARD + L] = torch.from_numpy(arr).to("cuda")
            self.bigs.append(big)
            self.views.append(big[GUARD:GUARD + L])

    def ptrs(self):
        return [self.bigs[r].data_ptr() + GUARD * self.np_dtype.itemsize for r in range(len(self.bigs))]

    def host(self):
        return [self.bigs[r][GUARD:GUARD + L].cpu().numpy().view(self.np_dtype) for r, L in enumerate(self.lengths)]

    def guards_intact(self):
        import torch
        item = self.np_dtype.itemsize
        for big, L in zip(self.bigs, self.lengths):
            g = big.view(torch.uint8)
            if not bool((g[:GUARD * item] == SENTINEL).all()) or not bool((g[(GUARD + L) * item:] == SENTINEL).all()):
                return False
        return True
