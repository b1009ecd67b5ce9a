"""The boundary from C: include/ra.h compiles as strict C99 (no GPU
needed), and a C program that uses only ra.h, libra_gb300.so and the CUDA
runtime runs every variant on a GPU and checks itself against closed forms
(tests/c/ra_c_example.c)."""

import os
import shutil
import subprocess

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "tests", "c", "ra_c_example.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _cc():
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    return cc


def test_header_is_strict_c99(tmp_path):
    """ra.h alone, pedantic C99: no C++ and no CUDA types in the ABI."""
    tu = tmp_path / "only_header.c"
    tu.write_text('#include "ra.h"\nint main(void) { ra_status s = RA_OK; return (int)s; }\n')
    cmd = [_cc(), "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-c", str(tu),
           "-I", os.path.join(ROOT, "include"), "-o", str(tmp_path / "h.o")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


def test_example_compiles_as_c99(tmp_path):
    cmd = [_cc(), "-std=c99", "-Wall", "-Wextra", "-Werror", "-c", SRC,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-o", str(tmp_path / "ex.o")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


@pytest.mark.gpu
def test_c_program_runs_every_variant(tmp_path):
    from ring_allreduce_gb300 import build
    lib = build.build()
    exe = tmp_path / "ra_c_example"
    libdir = os.path.dirname(lib)
    cmd = [_cc(), "-std=c99", "-O2", SRC, "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), "-L", libdir, "-lra_gb300",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{libdir}",
           f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-o", str(exe)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "c example: ok" in run.stdout
