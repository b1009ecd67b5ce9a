"""The bounds-checked build (libra_gb300_debug.so, -DRA_DEBUG_BOUNDS) stands
in for a memory checker: every global access of every kernel is checked
against the byte ranges of the call's buffers and of the handle's device
memory, and an access outside them is counted and skipped instead of
faulting.  A child process drives every entry point, variant, barrier and
AllGather kernel through it; there must be no such access, every result must
be the oracle's, and a call whose buffers are registered 16 bytes short must
be caught, at an address in one of the cut tails.  With buffers registered
short, the bulk copies the checks skip never arrive: the local kernel's and
the TMA AllGather round's bounded waits then run out, report RA_ERR_TIMEOUT
with code 2, and the handle's next call is correct."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
HERE = os.path.dirname(os.path.abspath(__file__))


def test_bounds_checked_build_sees_no_stray_access():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, RA_GB300_DEBUG_BOUNDS="1")
    res = subprocess.run([sys.executable, os.path.join(HERE, "bounds_check_driver.py")], env=env,
                         capture_output=True, text=True, timeout=1200)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    out = json.loads(res.stdout.strip().splitlines()[-1])
    assert out["calls"] > 100
    assert out["mismatches"] == [], out["mismatches"]
    assert out["clean"]["count"] == 0, out["clean"]
    assert out["shrunk"]["count"] > 0, out["shrunk"]
    assert out["shrunk"]["first_in_a_cut_tail"], out["shrunk"]
    for variant, t in out["timeouts"].items():
        assert t["status"] == "ERR_TIMEOUT" and t["code"] == 2, (variant, t)
        assert t["after"] == "OK" and t["after_equal"], (variant, t)
