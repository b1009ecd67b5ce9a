"""Ring ReduceScatter, AllGather and AllReduce, simulated rank by rank
(test infrastructure only).

Follows "Why AllReduce = ReduceScatter + AllGather -- NCCL Ring AllReduce":

* section 4: the ring GPU0 -> GPU1 -> ... -> GPU(R-1) -> GPU0; every rank
  receives from its predecessor r-1 and sends to its successor r+1 (mod R).
* section 5 (Ring ReduceScatter): in round 1 every rank r sends its own
  chunk r at the same time; each receiver adds its own copy of that chunk;
  in every later round the partial just made is passed on and the receiver
  adds its own chunk again.  After R-1 rounds rank r holds the complete
  S_{(r+1) mod R} (for R=4: GPU0 S1, GPU1 S2, GPU2 S3, GPU3 S0; also the
  placement drawn in section 2).
* section 6 (Ring AllGather): the complete chunks travel on along the same
  ring for R-1 more rounds; a receiver copies, it does not reduce.
* section 8 (the primitive sequence of Table V of "Demystifying NCCL" as the
  page restates it): send, recvReduceSend x (k-2), recvReduceCopySend,
  recvCopySend x (k-2), recv.  Each rank's steps are recorded under those
  names, built from what the step did (receive / reduce / copy to the output
  / send), not written out from the table.
* section 12: the N elements are cut into k chunks of about N/k each.
* section 13: every rank sends one chunk per round, (k-1) N/k in each phase.

Readings where the page leaves a choice (each restated in the design notes):

* the page's "about N/k" becomes C = ceil(n/R) and chunk k = [kC, min((k+1)C, n));
  the last chunks are the short ones and may be empty;
* ``(+)`` is applied as ``incoming (+) local`` (section 7: partial_sum +
  local_chunk; section 5 writes "a0 + b0" at the receiver of a0);
* in round 1 rank r sends chunk r (section 5, round 1), which fixes every
  later round and the placement S_k on rank k-1.

The simulation moves whole chunks with numpy; each rank's message is an
explicit copy, so no rank ever reads another rank's state except through a
message that was sent to it.
"""

import numpy as np

__all__ = [
    "chunk_plan", "owned_chunk", "ring_reduce_scatter", "ring_all_gather",
    "ring_allreduce", "primitive_name", "ring_reduce_scatter_compact",
    "ring_all_gather_compact",
]


def chunk_plan(R, n):
    """Split n elements into R chunks (section 12 of the ring page).

    Returns a list of (offset, length) for k = 0..R-1 with C = ceil(n/R) and
    chunk k = [k*C, min((k+1)*C, n)), clipped to n.  Chunks past the end are
    empty (length 0) and still take part in the ring as empty messages.
    """
    if R < 1:
        raise ValueError("R must be >= 1")
    if n < 0:
        raise ValueError("n must be >= 0")
    C = -(-n // R)
    plan = []
    for k in range(R):
        lo = min(k * C, n)
        hi = min((k + 1) * C, n)
        plan.append((lo, hi - lo))
    return plan


def owned_chunk(R, r):
    """Index of the chunk rank r holds complete after ReduceScatter: the
    ring page's placement GPU0:S1, GPU1:S2, GPU2:S3, GPU3:S0, i.e. (r+1) mod R."""
    return (r + 1) % R


def primitive_name(recv, reduce, copy_out, send):
    """Name of one primitive step from what it does, in NCCL's naming as
    the ring page (section 9) describes it: a receive may reduce, may copy
    the finished value into the rank's output while also passing it on, and
    may send.  A final receive with no send lands in the output by itself
    ("recv"); the first step of a rank only sends ("send")."""
    if not recv:
        return "send" if send else ""
    name = "recv"
    if reduce:
        name += "Reduce"
    if copy_out and (reduce or send):
        name += "Copy"
    if send:
        name += "Send"
    return name


class _Wire:
    """The messages in flight in one round: what each rank sent, and the
    bytes each rank has sent so far."""

    def __init__(self, R, itemsize):
        self.R = R
        self.itemsize = itemsize
        self.sent = [None] * R
        self.bytes_sent = [0] * R

    def send(self, r, payload):
        self.sent[r] = np.array(payload, copy=True)
        self.bytes_sent[r] += len(payload) * self.itemsize

    def deliver(self, r):
        """What rank r receives this round: its predecessor's message."""
        return self.sent[(r - 1) % self.R]


def _new_output(x, fill):
    out = np.empty_like(x)
    if fill is not None:
        out[...] = fill
    return out


def _reduce_scatter_rounds(x, op, wire, trace, log, out, fuse_first_allgather_send):
    """ReduceScatter: step 0 plus R-1 rounds.  Returns each rank's last
    message (its complete chunk, which AllGather sends on)."""
    R = len(x)
    n = len(x[0])
    plan = chunk_plan(R, n)

    def sl(c):
        o, L = plan[c]
        return slice(o, o + L)

    # step 0: every rank sends its own chunk r at the same time (round 1 of section 5)
    for r in range(R):
        wire.send(r, x[r][sl(r)])
        trace[r].append(primitive_name(False, False, False, True))
        if log is not None:
            log.append(("rs", 1, "send", r, (r + 1) % R, r, tuple(wire.sent[r])))
    last = [None] * R
    for s in range(1, R):
        received = [wire.deliver(r) for r in range(R)]
        final = s == R - 1
        for r in range(R):
            c = (r - s) % R
            partial = op.combine(received[r], x[r][sl(c)])
            if final:
                out[r][sl(c)] = partial          # the complete S_c, kept by rank r
            last[r] = partial
            sends_on = (not final) or fuse_first_allgather_send
            trace[r].append(primitive_name(True, True, final, sends_on))
            if log is not None:
                log.append(("rs", s, "reduce", r, c, tuple(partial)))
        if not final:
            for r in range(R):
                wire.send(r, last[r])
                if log is not None:
                    c = (r - s) % R
                    log.append(("rs", s + 1, "send", r, (r + 1) % R, c, tuple(last[r])))
    return last


def _all_gather_rounds(R, plan, first_msgs, op, wire, trace, log, out, first_send_traced):
    """AllGather: every rank starts by sending its complete chunk (r+1) mod R,
    then R-1 rounds of receive + copy (+ send), section 6."""

    def sl(c):
        o, L = plan[c]
        return slice(o, o + L)

    for r in range(R):
        wire.send(r, first_msgs[r])
        if not first_send_traced:
            trace[r].append(primitive_name(False, False, False, True))
        if log is not None:
            log.append(("ag", 1, "send", r, (r + 1) % R, owned_chunk(R, r), tuple(wire.sent[r])))
    for s in range(1, R):
        received = [wire.deliver(r) for r in range(R)]
        last_round = s == R - 1
        for r in range(R):
            c = (r + 1 - s) % R
            out[r][sl(c)] = received[r]
            trace[r].append(primitive_name(True, False, True, not last_round))
            if log is not None:
                log.append(("ag", s, "copy", r, c, tuple(received[r])))
        if not last_round:
            for r in range(R):
                wire.send(r, received[r])
                if log is not None:
                    c = (r + 1 - s) % R
                    log.append(("ag", s + 1, "send", r, (r + 1) % R, c, tuple(received[r])))


def _check_inputs(x, op):
    R = len(x)
    if R < 1:
        raise ValueError("need at least one rank")
    n = len(x[0])
    for r in range(R):
        if len(x[r]) != n:
            raise ValueError("every rank must hold n elements")
    return R, n


def ring_reduce_scatter(x, op, fill=None, trace=None, log=None, stats=None):
    """Ring ReduceScatter of the R rank inputs ``x`` (section 5).

    Returns R arrays of length n.  In array r only chunk (r+1) mod R is
    defined: it holds S_{(r+1) mod R}.  The other entries are left at
    ``fill`` (uninitialised when fill is None).  ``trace`` (list of R lists)
    receives each rank's primitive steps; ``stats`` (dict) receives the bytes
    each rank sent; ``log`` receives (phase, round, event, ...) records.
    """
    R, n = _check_inputs(x, op)
    x = [np.asarray(v) for v in x]
    trace = trace if trace is not None else [[] for _ in range(R)]
    wire = _Wire(R, op.itemsize)
    out = [_new_output(x[r], fill) for r in range(R)]
    if R == 1:
        out[0][...] = x[0]
    else:
        _reduce_scatter_rounds(x, op, wire, trace, log, out, fuse_first_allgather_send=False)
    if stats is not None:
        stats["bytes_sent"] = list(wire.bytes_sent)
    return out


def ring_all_gather(buf, op, trace=None, log=None, stats=None):
    """Ring AllGather (section 6) of the ReduceScatter result ``buf``:
    rank r contributes its chunk (r+1) mod R; returns R full arrays."""
    R, n = _check_inputs(buf, op)
    plan = chunk_plan(R, n)
    trace = trace if trace is not None else [[] for _ in range(R)]
    wire = _Wire(R, op.itemsize)
    out = [np.array(np.asarray(b), copy=True) for b in buf]
    if R > 1:
        first = []
        for r in range(R):
            o, L = plan[owned_chunk(R, r)]
            first.append(out[r][o:o + L])
        _all_gather_rounds(R, plan, first, op, wire, trace, log, out, first_send_traced=False)
    if stats is not None:
        stats["bytes_sent"] = list(wire.bytes_sent)
    return out


def ring_allreduce(x, op, trace=None, log=None, stats=None):
    """Ring AllReduce as one sequence of primitives (sections 4-8).

    ReduceScatter rounds, then AllGather rounds, with the boundary step fused
    as the page's section 9 describes recvReduceCopySend: the last reduction
    of a chunk writes the complete value into the rank's output and the same
    message is the first AllGather send.  Returns the R outputs.
    """
    R, n = _check_inputs(x, op)
    x = [np.asarray(v) for v in x]
    plan = chunk_plan(R, n)
    trace = trace if trace is not None else [[] for _ in range(R)]
    wire = _Wire(R, op.itemsize)
    out = [_new_output(x[r], None) for r in range(R)]
    if R == 1:
        out[0][...] = x[0]
    else:
        complete = _reduce_scatter_rounds(x, op, wire, trace, log, out, fuse_first_allgather_send=True)
        _all_gather_rounds(R, plan, complete, op, wire, trace, log, out, first_send_traced=True)
    if stats is not None:
        stats["bytes_sent"] = list(wire.bytes_sent)
    return out


def ring_reduce_scatter_compact(x, op):
    """ReduceScatter where each rank keeps only the chunk it owns, (r+1) mod R
    (the placement of section 2 and 5): returns R arrays, rank r's of length
    L_{(r+1) mod R}, cut from ``ring_reduce_scatter``."""
    R, n = _check_inputs(x, op)
    full = ring_reduce_scatter(x, op)
    plan = chunk_plan(R, n)
    out = []
    for r in range(R):
        off, L = plan[owned_chunk(R, r)]
        out.append(np.array(full[r][off:off + L], copy=True))
    return out


def ring_all_gather_compact(chunks, n, op):
    """AllGather from compact inputs: rank r brings chunk (r+1) mod R
    (``chunks[r]``); the chunks are placed where ReduceScatter leaves them and
    ``ring_all_gather`` runs on that layout.  Returns R arrays of n."""
    R = len(chunks)
    plan = chunk_plan(R, n)
    dtype = np.asarray(chunks[0]).dtype if R else np.float32
    buf = []
    for r in range(R):
        b = np.zeros(n, dtype=dtype)
        off, L = plan[owned_chunk(R, r)]
        if len(chunks[r]) != L:
            raise ValueError(f"rank {r} brings {len(chunks[r])} elements, its chunk has {L}")
        b[off:off + L] = chunks[r]
        buf.append(b)
    return ring_all_gather(buf, op)
