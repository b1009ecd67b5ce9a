"""Thin Python binding of libra_gb300.so (include/ra.h) over ctypes.

Argument marshalling only: rank buffers are torch CUDA tensors (or raw
device addresses), their addresses go into C pointer arrays, the stream is a
torch stream (or a raw cudaStream_t).  Every step of the collective runs in
the library's kernels.  Importing this module loads the library and raises
ImportError when it has not been built -- there is no fallback.
"""

import ctypes
import enum
import os

from . import build as _build

__all__ = [
    "Status", "DType", "Op", "Variant", "Barrier", "Protocol", "Option", "DeviceError", "RAError",
    "load_library", "library_path", "ra_create", "ra_destroy", "ra_reduce_scatter",
    "ra_all_gather", "ra_allreduce", "ra_allreduce_host", "ra_reduce_scatter_compact", "ra_all_gather_compact", "ra_chunk_plan", "ra_owned_chunk", "ra_set_option",
    "ra_get_option", "ra_get_device_status", "ra_read_signals", "ra_read_shadows", "ra_seed_signals",
    "ra_allreduce_noalloc",
    "ra_debug_bounds_report",
    "ra_last_error",
    "ra_status_string", "RingAllReduce", "PreparedCall", "EXPORTED",
]


class Status(enum.IntEnum):
    OK = 0
    ERR_INVALID = 1
    ERR_CUDA = 2
    ERR_OOM = 3
    ERR_UNSUPPORTED = 4
    ERR_TIMEOUT = 5


class DType(enum.IntEnum):
    F32 = 0
    BF16 = 1
    I32 = 2
    F16 = 3
    F64 = 4
    I64 = 5


class Op(enum.IntEnum):
    SUM = 0
    MAX = 1


class Variant(enum.IntEnum):
    AUTO = 0
    DIRECT = 1
    RING = 2
    PERSISTENT = 3
    PIPELINED = 4
    LOCAL = 5


class Barrier(enum.IntEnum):
    COUNTING = 0
    PER_PEER = 1
    CLUSTER = 2


class Protocol(enum.IntEnum):
    SIMPLE = 0
    LL = 1
    LL_CLUSTER = 2


class Option(enum.IntEnum):
    VARIANT = 1
    TIMEOUT_NS = 2
    CTAS = 3
    CHECK_POINTERS = 4
    SKIP_ARRIVAL = 5
    GRAPHS = 6
    BARRIER = 7
    SLICES = 8
    GATHER = 9
    HOST_WINDOWS = 10
    DEBUG_SHRINK = 11
    WINDOW = 12
    SIGNAL_BITS = 14
    PROTOCOL = 15
    LL_FLAG = 16


class DeviceError(ctypes.Structure):
    _fields_ = [("code", ctypes.c_uint32), ("round", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("channel", ctypes.c_int32), ("peer", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("observed", ctypes.c_uint64), ("expected", ctypes.c_uint64)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class RAError(RuntimeError):
    def __init__(self, status, message):
        self.status = Status(status)
        super().__init__(f"{self.status.name}: {message}")


_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_ST = ctypes.c_int
# name -> (restype, argtypes); every function include/ra.h declares
EXPORTED = {
    "ra_create": (_ST, [ctypes.c_int, _SZ, ctypes.c_int, ctypes.c_int, ctypes.POINTER(_P)]),
    "ra_destroy": (_ST, [_P]),
    "ra_reduce_scatter": (_ST, [_P, ctypes.POINTER(_P), ctypes.POINTER(_P), _P]),
    "ra_all_gather": (_ST, [_P, ctypes.POINTER(_P), _P]),
    "ra_allreduce": (_ST, [_P, ctypes.POINTER(_P), ctypes.POINTER(_P), _P]),
    "ra_allreduce_host": (_ST, [_P, ctypes.POINTER(_P), ctypes.POINTER(_P), _P]),
    "ra_reduce_scatter_compact": (_ST, [_P, ctypes.POINTER(_P), ctypes.POINTER(_P), _P]),
    "ra_all_gather_compact": (_ST, [_P, ctypes.POINTER(_P), ctypes.POINTER(_P), _P]),
    "ra_chunk_plan": (_ST, [ctypes.c_int, _SZ, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "ra_owned_chunk": (_ST, [_P, ctypes.c_int, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "ra_set_option": (_ST, [_P, ctypes.c_int, ctypes.c_longlong]),
    "ra_get_option": (_ST, [_P, ctypes.c_int, ctypes.POINTER(ctypes.c_longlong)]),
    "ra_get_device_status": (_ST, [_P, _P, ctypes.POINTER(DeviceError)]),
    "ra_read_signals": (_ST, [_P, ctypes.POINTER(ctypes.c_uint64), _SZ, ctypes.POINTER(_SZ),
                              ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                              ctypes.POINTER(ctypes.c_longlong)]),
    "ra_allreduce_noalloc": (_ST, [ctypes.c_int, _SZ, ctypes.c_int, ctypes.c_int, ctypes.POINTER(_P),
                                   ctypes.POINTER(_P), _P]),
    "ra_read_shadows": (_ST, [_P, ctypes.POINTER(ctypes.c_uint64), _SZ, ctypes.POINTER(_SZ)]),
    "ra_seed_signals": (_ST, [_P, ctypes.c_uint64, ctypes.c_uint64]),
    "ra_debug_bounds_report": (_ST, [ctypes.POINTER(ctypes.c_ulonglong), ctypes.POINTER(ctypes.c_ulonglong),
                                     ctypes.c_int]),
    "ra_last_error": (ctypes.c_char_p, []),
    "ra_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}

_LIB = None


def library_path():
    """The library to load: the bounds-checked debug build when the
    environment sets RA_GB300_DEBUG_BOUNDS=1 (build it with
    build.build(debug=True)), else the release build."""
    if os.environ.get("RA_GB300_DEBUG_BOUNDS") == "1":
        return _build.DEBUG_LIB_PATH
    return _build.LIB_PATH


def load_library(path=None):
    """Load libra_gb300.so once and declare its C signatures."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or library_path()
    if not os.path.exists(path):
        raise ImportError(f"libra_gb300.so is not built ({path}); run "
                          "`python -m ring_allreduce_gb300.build` (or __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in EXPORTED.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


_lib = load_library()


def ra_last_error():
    return _lib.ra_last_error().decode()


def ra_status_string(status):
    return _lib.ra_status_string(int(status)).decode()


def _check(status):
    if status != Status.OK:
        raise RAError(status, ra_last_error())


def _addr(x):
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return x.ctypes.data   # a numpy array (host buffers of ra_allreduce_host)


def _ptr_array(bufs):
    arr = (_P * len(bufs))()
    for i, b in enumerate(bufs):
        arr[i] = _addr(b)
    return arr


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def ra_create(R, n, dtype, op):
    h = _P()
    _check(_lib.ra_create(int(R), int(n), int(dtype), int(op), ctypes.byref(h)))
    return h


def ra_destroy(h):
    _check(_lib.ra_destroy(h))


def ra_allreduce(h, ins, outs, stream=None):
    _check(_lib.ra_allreduce(h, _ptr_array(ins), _ptr_array(outs), _stream(stream)))


def ra_debug_bounds_report(reset=True):
    """Bounds-checked builds only: (accesses outside the registered ranges
    since the last reset, address of the first); RAError UNSUPPORTED in
    release builds."""
    count, first = ctypes.c_ulonglong(), ctypes.c_ulonglong()
    _check(_lib.ra_debug_bounds_report(ctypes.byref(count), ctypes.byref(first), 1 if reset else 0))
    return count.value, first.value


def ra_allreduce_host(h, ins, outs, stream=None):
    """ins, outs: R host buffers (CPU torch tensors, numpy arrays or
    addresses); page-locked ones let the copies overlap."""
    _check(_lib.ra_allreduce_host(h, _ptr_array(ins), _ptr_array(outs), _stream(stream)))


def ra_reduce_scatter(h, ins, outs, stream=None):
    _check(_lib.ra_reduce_scatter(h, _ptr_array(ins), _ptr_array(outs), _stream(stream)))


def ra_all_gather(h, bufs, stream=None):
    _check(_lib.ra_all_gather(h, _ptr_array(bufs), _stream(stream)))


def ra_allreduce_noalloc(R, n, dtype, op, ins, outs, stream=None):
    """AllReduce with the library's fixed scratch array: no handle, no
    device allocation (for callers that may not allocate device memory)."""
    if len(ins) != R or len(outs) != R:
        raise ValueError(f"expected {R} rank buffers")
    _check(_lib.ra_allreduce_noalloc(int(R), int(n), int(dtype), int(op), _ptr_array(ins),
                                     _ptr_array(outs), _stream(stream)))


def ra_reduce_scatter_compact(h, ins, outs, stream=None):
    _check(_lib.ra_reduce_scatter_compact(h, _ptr_array(ins), _ptr_array(outs), _stream(stream)))


def ra_all_gather_compact(h, ins, outs, stream=None):
    _check(_lib.ra_all_gather_compact(h, _ptr_array(ins), _ptr_array(outs), _stream(stream)))


def ra_chunk_plan(R, n):
    off = (_SZ * max(R, 1))()
    ln = (_SZ * max(R, 1))()
    _check(_lib.ra_chunk_plan(int(R), int(n), off, ln))
    return [(off[k], ln[k]) for k in range(R)]


def ra_owned_chunk(h, r):
    off, ln = _SZ(), _SZ()
    _check(_lib.ra_owned_chunk(h, int(r), ctypes.byref(off), ctypes.byref(ln)))
    return off.value, ln.value


def ra_set_option(h, key, value):
    _check(_lib.ra_set_option(h, int(key), int(value)))


def ra_get_option(h, key):
    v = ctypes.c_longlong()
    _check(_lib.ra_get_option(h, int(key), ctypes.byref(v)))
    return v.value


def ra_get_device_status(h, stream=None):
    """Synchronise the stream and return (status, DeviceError); does not
    raise on RA_ERR_TIMEOUT, which it reports."""
    err = DeviceError()
    st = _lib.ra_get_device_status(h, _stream(stream), ctypes.byref(err))
    if st not in (Status.OK, Status.ERR_TIMEOUT):
        _check(st)
    return Status(st), err


def ra_read_signals(h):
    """Signal array of the last persistent or pipelined call (its kind and
    scheme), flat, plus (channels, rounds, calls); the layouts are those of
    ra_read_signals in ra.h."""
    count, ch, rd, calls = _SZ(), ctypes.c_int(), ctypes.c_int(), ctypes.c_longlong()
    _check(_lib.ra_read_signals(h, None, 0, ctypes.byref(count), ctypes.byref(ch), ctypes.byref(rd),
                                ctypes.byref(calls)))
    buf = (ctypes.c_uint64 * max(count.value, 1))()
    _check(_lib.ra_read_signals(h, buf, count.value, ctypes.byref(count), ctypes.byref(ch),
                                ctypes.byref(rd), ctypes.byref(calls)))
    return list(buf)[:count.value], ch.value, rd.value, calls.value


def ra_seed_signals(h, signal_value, shadow_value):
    """Set the counting-barrier and pipelined-flag signals to one value and
    their shadows to another (wrap-around tests)."""
    _check(_lib.ra_seed_signals(h, ctypes.c_uint64(int(signal_value)), ctypes.c_uint64(int(shadow_value))))


def ra_read_shadows(h):
    """The waiters' shadows of the last counting-barrier or pipelined call, flat."""
    count = _SZ()
    _check(_lib.ra_read_shadows(h, None, 0, ctypes.byref(count)))
    buf = (ctypes.c_uint64 * max(count.value, 1))()
    _check(_lib.ra_read_shadows(h, buf, count.value, ctypes.byref(count)))
    return list(buf)[:count.value]


_DTYPES = {"f32": DType.F32, "bf16": DType.BF16, "i32": DType.I32, "f16": DType.F16, "f64": DType.F64,
           "i64": DType.I64}
_OPS = {"sum": Op.SUM, "max": Op.MAX}


class RingAllReduce:
    """A handle for R ranks of n elements; buffers are passed per call."""

    def __init__(self, R, n, dtype="f32", op="sum", variant=None):
        self.R, self.n = int(R), int(n)
        self.dtype = _DTYPES[dtype] if isinstance(dtype, str) else DType(dtype)
        self.op = _OPS[op] if isinstance(op, str) else Op(op)
        self.itemsize = {DType.F32: 4, DType.BF16: 2, DType.I32: 4, DType.F16: 2, DType.F64: 8,
                         DType.I64: 8}[self.dtype]
        self.h = ra_create(self.R, self.n, self.dtype, self.op)
        if variant is not None:
            self.set_option(Option.VARIANT, Variant[variant.upper()] if isinstance(variant, str) else variant)

    def _ranks(self, *lists):
        # the C side reads exactly R pointers from each array
        for lst in lists:
            if len(lst) != self.R:
                raise ValueError(f"expected {self.R} rank buffers, got {len(lst)}")

    def allreduce(self, ins, outs, stream=None):
        self._ranks(ins, outs)
        ra_allreduce(self.h, ins, outs, stream)

    def allreduce_host(self, ins, outs, stream=None):
        """AllReduce of R host buffers through the library's device copies
        (ra_allreduce_host): asynchronous on `stream`."""
        self._ranks(ins, outs)
        for b in list(ins) + list(outs):
            if isinstance(b, int):
                continue
            size = b.numel() * b.element_size() if hasattr(b, "numel") else b.nbytes
            if size < self.n * self.itemsize:
                raise ValueError(f"host buffer of {size} bytes, need {self.n * self.itemsize}")
            if hasattr(b, "is_cuda") and b.is_cuda:
                raise ValueError("allreduce_host takes host buffers; use allreduce for device tensors")
        ra_allreduce_host(self.h, ins, outs, stream)

    def reduce_scatter(self, ins, outs, stream=None):
        self._ranks(ins, outs)
        ra_reduce_scatter(self.h, ins, outs, stream)

    def all_gather(self, bufs, stream=None):
        self._ranks(bufs)
        ra_all_gather(self.h, bufs, stream)

    def reduce_scatter_compact(self, ins, outs, stream=None):
        """outs[r]: rank r's chunk only (length from owned_chunk(r))."""
        self._ranks(ins, outs)
        ra_reduce_scatter_compact(self.h, ins, outs, stream)

    def all_gather_compact(self, ins, outs, stream=None):
        """ins[r]: rank r's chunk only; outs[r]: all n elements."""
        self._ranks(ins, outs)
        ra_all_gather_compact(self.h, ins, outs, stream)

    def prepare(self, kind, ins, outs=None, stream=None):
        """Marshal the buffers and stream once and return a callable that
        runs the collective on them: for repeated calls on the same buffers
        (a training loop's gradient buckets), where rebuilding the pointer
        arrays each call would cost more than a small collective itself.
        kind: "allreduce", "reduce_scatter", "all_gather" (ins only),
        "reduce_scatter_compact" or "all_gather_compact"."""
        return PreparedCall(self, kind, ins, outs, stream)

    def owned_chunk(self, r):
        return ra_owned_chunk(self.h, r)

    def set_option(self, key, value):
        ra_set_option(self.h, key, value)

    def get_option(self, key):
        return ra_get_option(self.h, key)

    def device_status(self, stream=None):
        return ra_get_device_status(self.h, stream)

    def read_signals(self):
        return ra_read_signals(self.h)

    def read_shadows(self):
        return ra_read_shadows(self.h)

    def seed_signals(self, signal_value, shadow_value):
        ra_seed_signals(self.h, signal_value, shadow_value)

    def close(self):
        if self.h:
            ra_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class PreparedCall:
    """A collective with its arguments marshalled once (see
    RingAllReduce.prepare).  The buffers must stay alive and in place."""

    def __init__(self, owner, kind, ins, outs, stream):
        two = {"allreduce": _lib.ra_allreduce, "reduce_scatter": _lib.ra_reduce_scatter,
               "reduce_scatter_compact": _lib.ra_reduce_scatter_compact,
               "all_gather_compact": _lib.ra_all_gather_compact}
        if kind == "all_gather":
            owner._ranks(ins)
            self._fn = _lib.ra_all_gather
            self._args = (owner.h, _ptr_array(ins), _stream(stream))
        elif kind in two:
            owner._ranks(ins, outs)
            self._fn = two[kind]
            self._args = (owner.h, _ptr_array(ins), _ptr_array(outs), _stream(stream))
        else:
            raise ValueError(f"unknown collective {kind!r}")
        self._owner = owner      # keeps the handle alive

    def __call__(self):
        st = self._fn(*self._args)
        if st != Status.OK:
            raise RAError(st, ra_last_error())
