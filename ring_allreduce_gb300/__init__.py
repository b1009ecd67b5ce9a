"""Ring AllReduce for R ranks held as R buffers in one GB300's HBM.

The compute path is the CUDA library ``libra_gb300.so`` (``include/ra.h``);
this package is its thin Python binding (ctypes marshalling, torch for device
memory and streams).  The binding is loaded on first use of one of its names,
so ``ring_allreduce_gb300.inputs`` can be imported on a machine where the
library has not been built.  Using the binding without the built library
raises ImportError: there is no CPU fallback.
"""

_BINDING_NAMES = {
    "ra_create", "ra_destroy", "ra_reduce_scatter", "ra_all_gather", "ra_allreduce",
    "ra_reduce_scatter_compact", "ra_all_gather_compact",
    "ra_chunk_plan", "ra_owned_chunk", "ra_set_option", "ra_get_option",
    "ra_get_device_status", "ra_read_signals", "ra_read_shadows", "ra_allreduce_noalloc", "ra_last_error", "ra_status_string",
    "RingAllReduce", "PreparedCall", "RAError", "Status", "DType", "Op", "Variant", "Barrier", "Option",
    "DeviceError", "load_library", "library_path",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")
