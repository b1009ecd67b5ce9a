"""Pins the oracle to the 4-GPU worked example printed on "Why AllReduce =
ReduceScatter + AllGather -- NCCL Ring AllReduce" (sections 2, 5, 6 and 8),
transcribed in tests/golden/ring_r4_worked_example.txt, and extends the same
symbolic check to other ring sizes."""

import os

import numpy as np
import pytest

from oracle import elementops, ring

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ring_r4_worked_example.txt")
LETTERS = "abcdefghijklmnopqrstuvwxyz"


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _terms(s):
    return tuple(s.split("+"))


def _sym_inputs(R, per_chunk=1):
    """Rank r holds chunks named <letter r><chunk k>; each chunk has
    ``per_chunk`` elements carrying the same name plus an element suffix
    when per_chunk > 1."""
    n = R * per_chunk
    x = []
    for r in range(R):
        a = np.empty(n, dtype=object)
        for k in range(R):
            for e in range(per_chunk):
                name = f"{LETTERS[r]}{k}" if per_chunk == 1 else f"{LETTERS[r]}{k}.{e}"
                a[k * per_chunk + e] = (name,)
        x.append(a)
    return x


def _run_r4():
    x = _sym_inputs(4)
    log, trace = [], [[] for _ in range(4)]
    out = ring.ring_allreduce(x, elementops.Sym(), trace=trace, log=log)
    return x, out, log, trace


def test_reduce_scatter_sends_and_partials_match_page():
    _, _, log, _ = _run_r4()
    sends = {(e[1], e[3], e[4]): e[6][0] for e in log if e[0] == "rs" and e[2] == "send"}
    holds = {(e[1], e[3]): e[5][0] for e in log if e[0] == "rs" and e[2] == "reduce"}
    checked = 0
    for row in _golden():
        if row[0] == "rs_send":
            s, src, dst, payload = int(row[1]), int(row[2]), int(row[3]), row[4]
            assert sends[(s, src, dst)] == _terms(payload), row
            checked += 1
        elif row[0] == "rs_hold":
            s, gpu, payload = int(row[1]), int(row[2]), row[3]
            assert holds[(s, gpu)] == _terms(payload), row
            checked += 1
    assert checked == 20


def test_reduce_scatter_placement_matches_page():
    """GPU0:S1, GPU1:S2, GPU2:S3, GPU3:S0, each S_k holding every rank's
    chunk k exactly once."""
    x = _sym_inputs(4)
    rs = ring.ring_reduce_scatter(x, elementops.Sym())
    finals = [r for r in _golden() if r[0] == "rs_final"]
    assert len(finals) == 4
    for row in finals:
        gpu, sname, terms = int(row[1]), row[2], _terms(row[3])
        k = int(sname[1:])
        assert ring.owned_chunk(4, gpu) == k
        got = rs[gpu][k]
        assert sorted(got) == sorted(terms)
        assert len(got) == len(set(got)) == 4


def test_allgather_sends_and_holdings_match_page():
    _, out, log, _ = _run_r4()
    S = {}
    for r in range(4):
        k = ring.owned_chunk(4, r)
        S[f"S{k}"] = next(e[5][0] for e in log if e[0] == "rs" and e[2] == "reduce"
                          and e[1] == 3 and e[3] == r)
    ag_sends = {(e[1], e[3], e[4]): e[6][0] for e in log if e[0] == "ag" and e[2] == "send"}
    copies = [(e[1], e[3], e[4]) for e in log if e[0] == "ag" and e[2] == "copy"]
    n_checked = 0
    for row in _golden():
        if row[0] == "ag_send":
            s, src, dst, sname = int(row[1]), int(row[2]), int(row[3]), row[4]
            assert ag_sends[(s, src, dst)] == S[sname], row
            n_checked += 1
        elif row[0] == "ag_holds":
            s, gpu, names = int(row[1]), int(row[2]), row[3:]
            held = {ring.owned_chunk(4, gpu)} | {c for (rr, g, c) in copies if rr <= s and g == gpu}
            assert held == {int(nm[1:]) for nm in names}, row
            n_checked += 1
    assert n_checked == 13
    for r in range(4):
        for k in range(4):
            assert out[r][k] == S[f"S{k}"]


def test_primitive_sequence_matches_page_k4():
    _, _, _, trace = _run_r4()
    row = next(r for r in _golden() if r[0] == "primitives")
    assert int(row[1]) == 4
    for r in range(4):
        assert trace[r] == row[2:]


@pytest.mark.parametrize("R", [2, 3, 4, 5, 7, 8])
def test_primitive_sequence_general_k(R):
    """Section 8 of the ring page: step 0 send, steps 1..k-2 recvReduceSend,
    step k-1 recvReduceCopySend, steps k..2k-3 recvCopySend, step 2k-2
    recv; 2k-1 steps in all (section 10)."""
    x = _sym_inputs(R)
    trace = [[] for _ in range(R)]
    ring.ring_allreduce(x, elementops.Sym(), trace=trace)
    want = (["send"] + ["recvReduceSend"] * (R - 2) + ["recvReduceCopySend"]
            + ["recvCopySend"] * (R - 2) + ["recv"])
    for r in range(R):
        assert trace[r] == want
        assert len(trace[r]) == 2 * R - 1


@pytest.mark.parametrize("R", [2, 3, 4, 5, 6, 7])
@pytest.mark.parametrize("per_chunk", [1, 3])
def test_fold_order_is_ring_order_from_rank_k(R, per_chunk):
    """Every S_k folds x_k, x_{k+1}, ..., x_{k-1} in that order (the ring
    page's section 5: chunk k starts at rank k and each rank on the way adds
    its own chunk), every rank exactly once, and every rank ends with the same
    R values."""
    x = _sym_inputs(R, per_chunk)
    out = ring.ring_allreduce(x, elementops.Sym())
    for k in range(R):
        for e in range(per_chunk):
            i = k * per_chunk + e
            suffix = "" if per_chunk == 1 else f".{e}"
            want = tuple(f"{LETTERS[(k + j) % R]}{k}{suffix}" for j in range(R))
            for r in range(R):
                assert out[r][i] == want


def test_reduce_scatter_then_allgather_is_allreduce_symbolic():
    for R in range(1, 7):
        x = _sym_inputs(R, 2)
        op = elementops.Sym()
        ar = ring.ring_allreduce(x, op)
        ag = ring.ring_all_gather(ring.ring_reduce_scatter(x, op), op)
        for r in range(R):
            assert list(ar[r]) == list(ag[r])


def test_compact_forms_follow_the_placement():
    """Compact ReduceScatter keeps exactly rank r's S_{(r+1) mod R}; compact
    AllGather of those chunks gives every rank [S0 .. S_{R-1}]."""
    x = _sym_inputs(4, 2)
    op = elementops.Sym()
    rs = ring.ring_reduce_scatter_compact(x, op)
    ar = ring.ring_allreduce(x, op)
    for r, k in enumerate([1, 2, 3, 0]):
        assert list(rs[r]) == list(ar[0][2 * k:2 * k + 2])
    ag = ring.ring_all_gather_compact(rs, 8, op)
    for r in range(4):
        assert list(ag[r]) == list(ar[0])
