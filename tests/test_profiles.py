"""The committed profile summaries describe the kernels in the tree.

Every summary under profiles/ names the kernel sources it was measured on,
as a 16-hex-digit hash of each kernel's source files
(`build.kernel_source_hash`).  A summary citing a hash the sources no longer
have describes a different kernel, so every cited hash must be the current
one.  No GPU needed."""

import glob
import os
import re

import pytest

from ring_allreduce_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def _cited(text, fname):
    """(kernel, hash) pairs a summary cites: "<kernel> <hash>" in a sources
    line, or "source_hash <hash> (<kernel> kernel sources ...)"; a bare
    "source_hash: <hash>" belongs to the kernel the file is named after."""
    out = []
    for m in re.finditer(r"\b([a-z]+) ([0-9a-f]{16})\b", text):
        if m.group(1) in build.KERNEL_SOURCES:
            out.append((m.group(1), m.group(2)))
    for m in re.finditer(r"source_hash:?\s+([0-9a-f]{16})(?:\s+\((\w+) kernel sources)?", text):
        out.append((m.group(2) or fname.split("_kernel")[0], m.group(1)))
    return out


def test_there_are_profiles():
    assert len(PROFILES) >= 10


@pytest.mark.parametrize("path", PROFILES, ids=[os.path.basename(p) for p in PROFILES])
def test_profile_cites_current_sources(path):
    with open(path, encoding="utf-8") as fh:
        text = fh.read()
    cited = _cited(text, os.path.basename(path))
    assert cited, f"{os.path.basename(path)} names no kernel source hash"
    for kernel, h in cited:
        assert kernel in build.KERNEL_SOURCES, f"{os.path.basename(path)}: unknown kernel {kernel!r}"
        assert h == build.kernel_source_hash(kernel), (
            f"{os.path.basename(path)} was measured on {kernel} sources {h}; "
            f"they are now {build.kernel_source_hash(kernel)}")


def _doc_citations():
    """Every profiles/<name> a top-level document cites (globs included)."""
    out = set()
    for doc in ("DESIGN.md", "README.md", "BASELINE.md"):
        path = os.path.join(ROOT, doc)
        if os.path.exists(path):
            with open(path, encoding="utf-8") as fh:
                out.update(re.findall(r"profiles/[A-Za-z0-9_*.]+", fh.read()))
    return sorted(c.rstrip(".") for c in out)


@pytest.mark.parametrize("cited", _doc_citations())
def test_cited_profiles_exist(cited):
    assert glob.glob(os.path.join(ROOT, cited)), f"{cited} is cited but no such summary is committed"


@pytest.mark.parametrize("path", PROFILES, ids=[os.path.basename(p) for p in PROFILES])
def test_profile_states_its_command(path):
    """Each summary gives the command that produced its figures."""
    with open(path, encoding="utf-8") as fh:
        text = fh.read()
    assert re.search(r"^Commands?\b", text, re.M), f"{os.path.basename(path)} states no command"
    assert "python " in text, f"{os.path.basename(path)} names no command line"
