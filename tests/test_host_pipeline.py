"""A CPU model of lamp_attn_fwd_host's copy / compute pipeline (the enqueue
sequence of lamp_host.cu) under CUDA stream and event semantics: work on
one stream runs in order, one operation after the other; an event record
completes once the work enqueued before it on its stream has; a stream wait
binds, when it is enqueued, to the event's latest record (none: no wait).
Operations take time (a start and an end), so a buffer that is rewritten
while another operation still reads it is caught.  Checked for any number
of chunks, slots and compute streams: a chunk's copy in never overwrites
inputs that an earlier chunk's computation still reads, a computation finds
its own chunk's inputs and never overwrites outputs the read-back of an
earlier chunk still reads, the read-back finds its own chunk's outputs, and
the caller's stream ends after all of it."""
import random

import pytest


class Sim:
    def __init__(self, seed):
        self.rng = random.Random(seed)
        self.streams = {}     # name -> list of ops (in enqueue order)
        self.records = {}     # event -> list of record ops
        self.buf = {}         # buffer -> (chunk, version)
        self.done_ops = set()

    def op(self, stream, kind, **kw):
        o = dict(kind=kind, stream=stream, started=False, ended=False, **kw)
        self.streams.setdefault(stream, []).append(o)
        return o

    def record(self, ev, stream):
        o = self.op(stream, "record", ev=ev)
        self.records.setdefault(ev, []).append(o)

    def wait(self, stream, ev):
        recs = self.records.get(ev)
        self.op(stream, "wait", dep=recs[-1] if recs else None)

    def _ready(self, o):
        q = self.streams[o["stream"]]
        i = q.index(o)
        if i > 0 and not q[i - 1]["ended"]:
            return False
        return o["kind"] != "wait" or o["dep"] is None or o["dep"]["ended"]

    def run(self):
        steps = 0
        while True:
            steps += 1
            assert steps < 200000, "no progress"
            cand = []
            for q in self.streams.values():
                for o in q:
                    if not o["ended"]:
                        if o["started"] or self._ready(o):
                            cand.append(o)
                        break
            if not cand:
                assert all(o["ended"] for q in self.streams.values() for o in q), "deadlock"
                return
            o = self.rng.choice(cand)
            if not o["started"]:
                o["started"] = True
                self._start(o)
                if o["kind"] in ("record", "wait"):
                    o["ended"] = True
            else:
                self._end(o)
                o["ended"] = True

    # buffers written at the start of an operation get a new version; reads
    # check the chunk at the start and that no write came in before the end
    def _start(self, o):
        o["seen"] = {b: self.buf.get(b) for b in o.get("reads", ())}
        for b, want in zip(o.get("reads", ()), o.get("want", ())):
            assert self.buf.get(b, (None,))[0] == want, f"{o['kind']} of chunk {o['chunk']} reads {b} of another chunk"
        for b in o.get("writes", ()):
            self.buf[b] = (o["chunk"], self.buf.get(b, (None, 0))[1] + 1)

    def _end(self, o):
        for b in o.get("reads", ()):
            assert self.buf.get(b) == o["seen"][b], f"{b} rewritten while {o['kind']} of chunk {o['chunk']} read it"
        for b in o.get("writes", ()):
            assert self.buf[b][0] == o["chunk"], f"{b} written by two operations at once"


def host_call(seed, nchunks, nslots, ncomp):
    """The enqueue sequence of lamp_attn_fwd_host, chunk by chunk."""
    s = Sim(seed)
    sc = "comp0"
    comp = [sc] + [f"comp{i}" for i in range(1, ncomp)]
    s.op(sc, "caller work before the call")
    s.record("start", sc)
    for st in ["h2d", "d2h"] + comp[1:]:
        s.wait(st, "start")
    for c in range(nchunks):
        slot = c % nslots
        reuse = c >= nslots
        e_in, e_done, e_out = f"in{slot}", f"done{slot}", f"out{slot}"
        inp, outb = f"inputs{slot}", f"outputs{slot}"
        if reuse:
            s.wait("h2d", e_done)
        s.op("h2d", "copy in", chunk=c, writes=(inp,))
        s.record(e_in, "h2d")
        cst = comp[c % ncomp]
        s.wait(cst, e_in)
        if reuse:
            s.wait(cst, e_out)
        s.op(cst, "compute", chunk=c, reads=(inp,), want=(c,), writes=(outb, f"workspace{slot}"))
        s.record(e_done, cst)
        s.wait("d2h", e_done)
        s.op("d2h", "read back", chunk=c, reads=(outb,), want=(c,))
        s.record(e_out, "d2h")
    s.record("join_d2h", "d2h")
    s.wait(sc, "join_d2h")
    s.record("join_h2d", "h2d")
    s.wait(sc, "join_h2d")
    for i, st in enumerate(comp[1:]):
        s.record(f"join{i}", st)
        s.wait(sc, f"join{i}")
    last = s.op(sc, "caller sees the results")
    s.run()
    # every read-back ended before the caller's stream went on
    for o in s.streams["d2h"]:
        assert o["ended"]
    assert last["ended"]


@pytest.mark.parametrize("nchunks,nslots,ncomp", [(1, 1, 4), (8, 8, 4), (8, 2, 4), (8, 2, 2), (16, 16, 4),
                                                  (16, 3, 4), (16, 2, 1), (5, 2, 4), (32, 7, 4)])
def test_host_pipeline_random_completion_orders(nchunks, nslots, ncomp):
    for seed in range(40):
        host_call(seed * 31 + nchunks, nchunks, nslots, ncomp)


def test_model_catches_a_missing_wait():
    """Without the copy stream's wait for the slot's previous computation,
    some completion order overwrites inputs still being read."""
    failures = 0
    for seed in range(200):
        try:
            _host_call_without_done_wait(seed, 8, 2, 4)
        except AssertionError:
            failures += 1
    assert failures > 0


def _host_call_without_done_wait(seed, nchunks, nslots, ncomp):
    s = Sim(seed)
    comp = ["comp0"] + [f"comp{i}" for i in range(1, ncomp)]
    for c in range(nchunks):
        slot = c % nslots
        reuse = c >= nslots
        inp, outb = f"inputs{slot}", f"outputs{slot}"
        s.op("h2d", "copy in", chunk=c, writes=(inp,))  # (no wait for the slot's previous computation)
        s.record(f"in{slot}", "h2d")
        cst = comp[c % ncomp]
        s.wait(cst, f"in{slot}")
        if reuse:
            s.wait(cst, f"out{slot}")
        s.op(cst, "compute", chunk=c, reads=(inp,), want=(c,), writes=(outb,))
        s.record(f"done{slot}", cst)
        s.wait("d2h", f"done{slot}")
        s.op("d2h", "read back", chunk=c, reads=(outb,), want=(c,))
        s.record(f"out{slot}", "d2h")
    s.run()
