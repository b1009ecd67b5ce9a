"""The C-ABI library loads and exports every function include/ra.h
declares, and its host-only logic (chunk plan, argument checks, status
names) behaves as documented.  Runs without a GPU: no compute call is made."""

import ctypes
import os
import re

import pytest

from conftest import ROOT
from oracle import ring

HEADER = os.path.join(ROOT, "include", "ra.h")


@pytest.fixture(scope="session")
def lib():
    from ring_allreduce_gb300 import build
    build.build()
    from ring_allreduce_gb300 import binding
    return binding


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(ra_\w+)\s*\(", text, flags=re.M))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("ra_create", "ra_reduce_scatter", "ra_all_gather", "ra_allreduce", "ra_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.library_path())
    names = _declared()
    assert names, "no declarations parsed"
    for n in sorted(names):
        assert hasattr(so, n), f"{n} declared in ra.h but not exported"
    assert set(lib.EXPORTED) == names


def test_chunk_plan_matches_oracle(lib):
    for R in (1, 2, 3, 4, 5, 8, 16, 32):
        for n in list(range(0, 2 * R + 3)) + [4096, 2**24, 2**26 + 3, 10**9 + 7]:
            assert lib.ra_chunk_plan(R, n) == ring.chunk_plan(R, n)


def test_chunk_plan_rejects_bad_R(lib):
    off = (ctypes.c_size_t * 64)()
    ln = (ctypes.c_size_t * 64)()
    for R in (0, -1, 33):
        assert lib._lib.ra_chunk_plan(R, 10, off, ln) == lib.Status.ERR_INVALID
    assert lib._lib.ra_chunk_plan(4, 10, None, ln) == lib.Status.ERR_INVALID


def test_create_rejects_invalid_arguments(lib):
    for args in ((0, 16, 0, 0), (33, 16, 0, 0), (4, 16, 7, 0), (4, 16, 0, 5), (4, 2**41, 0, 0)):
        h = ctypes.c_void_p()
        st = lib._lib.ra_create(*args, ctypes.byref(h))
        assert st == lib.Status.ERR_INVALID, args
        assert not h.value
        assert lib.ra_last_error()
    assert lib._lib.ra_create(4, 16, 0, 0, None) == lib.Status.ERR_INVALID


def test_create_without_device_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = lib._lib.ra_create(4, 4096, 0, 0, ctypes.byref(h))
    assert st == lib.Status.ERR_CUDA
    assert "cuda" in lib.ra_last_error().lower()


def test_null_handle_calls_are_rejected(lib):
    arr = (ctypes.c_void_p * 2)()
    assert lib._lib.ra_allreduce(None, arr, arr, None) == lib.Status.ERR_INVALID
    assert lib._lib.ra_reduce_scatter(None, arr, arr, None) == lib.Status.ERR_INVALID
    assert lib._lib.ra_all_gather(None, arr, None) == lib.Status.ERR_INVALID
    assert lib._lib.ra_set_option(None, 1, 0) == lib.Status.ERR_INVALID
    assert lib._lib.ra_destroy(None) == lib.Status.OK


def test_status_strings(lib):
    for s in lib.Status:
        assert lib.ra_status_string(s) == "RA_" + s.name


def _header_enum(prefix):
    """{NAME: value} of the enumerators of ra.h that start with `prefix`."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return {m.group(1): int(m.group(2)) for m in re.finditer(rf"\b{prefix}(\w+)\s*=\s*(\d+)", text)}


@pytest.mark.parametrize("prefix,cls", [("RA_OPT_", "Option"), ("RA_VARIANT_", "Variant"),
                                        ("RA_BARRIER_", "Barrier"), ("RA_PROTOCOL_", "Protocol")])
def test_binding_enums_match_the_header(lib, prefix, cls):
    want = _header_enum(prefix)
    assert want, prefix
    got = {e.name: int(e) for e in getattr(lib, cls)}
    assert got == want
