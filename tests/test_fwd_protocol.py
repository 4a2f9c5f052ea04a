"""CPU models of the fused attention kernel's protocol (lamp_fwd.cu) under
random interleavings: the two-stage path (d <= 128, one or two query tiles
per CTA), the one-stage path (d = 256; below) and the detector-only tau
sweep (below).  For the two-stage path:  The TMA producer, each tile's MMA-issuing thread and each
tile's softmax (one actor per tile: its warps meet at the step's tile
barrier anyway) run the kernel's loops with its phase / parity formulas
against mbarriers with the hardware's semantics, while copies and MMAs
complete asynchronously (each issuing thread's MMAs and commits in issue
order).  The sub-block flags of every step are random inputs; each tile
has its own key range (causal rows see fewer keys in the first tile).

Checked: an MMA reads the stage that holds its key, and a stage is refilled
only after every tile's MMAs on its previous key are done (the softmax's
exact re-derivations read K8 there too, until the step's decision); QK8
rewrites the S8 buffer only after the softmax has read the previous step's
logits; the softmax finds its own step's 16-bit products in the S16 buffer
whenever the step has a flag (speculative products of unflagged steps
included in its phase count), P.V reads its own step's P, the decision
byte is read before the next step of that parity rewrites it, the
recompute counters follow from the flags, and every run finishes."""
import random

import pytest

NS = 2  # K/V stages


class Bar:
    def __init__(self, count=1):
        self.count, self.pending, self.tx, self.phase = count, count, 0, 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self):
        assert self.pending > 0
        self.pending -= 1
        self._maybe_complete()

    def expect_tx(self, n):
        self.tx += n
        self.arrive()

    def complete_tx(self, n):
        self.tx -= n
        self._maybe_complete()

    def passed(self, parity):
        return (self.phase & 1) != parity


def run(seed, ranges, flags, drop=None):
    """ranges[t] = (JLO, JHI) key tiles of query tile t; flags[t][i]: step i
    of tile t has a flagged sub-block.  ``drop`` takes one wait out of the
    model (to show the checks catch it)."""
    rng = random.Random(seed)
    NT = len(ranges)
    J0 = min(r[0] for r in ranges)
    J1 = max(r[1] for r in ranges)
    stage_of = lambda j: (j - J0) % NS  # noqa: E731
    KV_FULL = [Bar() for _ in range(NS)]
    KV_EMPTY = [[Bar() for _ in range(NT)] for _ in range(NS)]
    S_FULL, S16_FULL, DEC, P_FULL, PV_DONE = ([Bar() for _ in range(NT)] for _ in range(5))
    stage = [None] * NS                   # key held by each stage
    S8 = [None] * NT                      # step whose QK8 completed into the tile's S8 buffer
    S16 = [None] * NT
    P = [None] * NT                       # step whose P the softmax stored
    s8_read = [-1] * NT                   # last step whose S8 the softmax has read
    s16_read = [-1] * NT                  # last step whose S16 the softmax has read (flagged steps)
    ANY = [[None, None] for _ in range(NT)]  # (step, flag) published before DEC
    open_reads = {}                       # key -> MMA ops on it not yet completed
    mma_q = [[] for _ in range(NT)]       # per MMA thread: ops in issue order
    copies = []                           # producer copies in issue order: (stage, key)
    issued16 = [0] * NT
    counts = [[0, 0, 0] for _ in range(NT)]  # recompute used, ahead and unused, after the decision

    def producer():
        rel = 0
        for j in range(J0, J1):
            s, u = stage_of(j), (j - J0) // NS
            if u >= 1:
                jr = j - NS
                for t in range(NT):
                    # every tile with keys releases each key up to its last,
                    # those before its first one unused ("skip": only the
                    # keys it uses, the form that let a late-starting
                    # tile's parity wait pass a phase early)
                    used = ranges[t][0] <= jr < ranges[t][1] if drop == "skip" else \
                        (ranges[t][1] > ranges[t][0] and jr < ranges[t][1])
                    if not used:
                        continue
                    bit = 1 << (2 * t + s)
                    while drop != "kv_empty" and not KV_EMPTY[s][t].passed(1 if rel & bit else 0):
                        yield
                    rel ^= bit
                assert open_reads.get(jr, 0) == 0, "stage refilled while MMAs still read its key"
            KV_FULL[s].expect_tx(1)
            copies.append((s, j))
            yield

    def mma(t):
        jlo, jhi = ranges[t]
        n = jhi - jlo
        if n <= 0:
            return

        def issue(kind, i=None, bar=None):
            if kind in ("qk8", "qk16", "pv"):
                open_reads[jlo + i] = open_reads.get(jlo + i, 0) + 1
            mma_q[t].append((kind, i, bar))

        def any_of(i):
            step, f = ANY[t][i & 1]
            assert step == i, "decision byte rewritten before it was read"
            return f

        if drop != "skip":
            for j in range(J0, jlo):  # keys before the tile's first one: land, then handed back unused
                while not KV_FULL[stage_of(j)].passed(((j - J0) // NS) & 1):
                    yield
                KV_EMPTY[stage_of(j)][t].arrive()
                yield
        spec = True
        for i in range(n):
            j = jlo + i
            if i > 0:
                while not DEC[t].passed((i - 1) & 1):
                    yield
            while not KV_FULL[stage_of(j)].passed(((j - J0) // NS) & 1):
                yield
            issue("qk8", i)
            issue("commit", bar=S_FULL[t])
            if i > 0:
                prev = any_of(i - 1)
                counts[t][0] += prev
                counts[t][1] += spec and not prev
                counts[t][2] += prev and not spec
                if prev and not spec:
                    issue("qk16", i - 1)
                    issue("commit", bar=S16_FULL[t])
                    issued16[t] += 1
                spec = prev
                while not P_FULL[t].passed((i - 1) & 1):
                    yield
                issue("pv", i - 1)
                issue("commit", bar=PV_DONE[t])
                issue("commit", bar=KV_EMPTY[stage_of(j - 1)][t])
            if spec:
                issue("qk16", i)
                issue("commit", bar=S16_FULL[t])
                issued16[t] += 1
            yield
        while not DEC[t].passed((n - 1) & 1):
            yield
        last = any_of(n - 1)
        counts[t][0] += last
        counts[t][1] += spec and not last
        counts[t][2] += last and not spec
        if last and not spec:
            issue("qk16", n - 1)
            issue("commit", bar=S16_FULL[t])
            issued16[t] += 1
        while not P_FULL[t].passed((n - 1) & 1):
            yield
        issue("pv", n - 1)
        issue("commit", bar=PV_DONE[t])
        issue("commit", bar=KV_EMPTY[stage_of(jhi - 1)][t])

    def softmax(t):
        jlo, jhi = ranges[t]
        n16, prev_any = 0, True
        for jj in range(jhi - jlo):
            while not S_FULL[t].passed(jj & 1):
                yield
            assert S8[t] == jj, "S8 of another step"
            assert stage[stage_of(jlo + jj)] == jlo + jj, "K8 of the step's key gone before its decision"
            s8_read[t] = jj
            yield  # guard, maximum, detector, tile barrier
            any_ = flags[t][jj]
            ANY[t][jj & 1] = (jj, any_)
            DEC[t].arrive()
            yield  # P8
            if jj > 0:
                while drop != "pv_done" and not PV_DONE[t].passed((jj - 1) & 1):
                    yield
            if any_:
                while not S16_FULL[t].passed(n16 & 1):
                    yield
                assert S16[t] == jj, "S16 of another step"
                s16_read[t] = jj
            n16 += 1 if (any_ or prev_any) else 0
            prev_any = any_
            yield  # P16
            assert P[t] is None or P[t] == jj - 1
            assert jj == 0 or pv_done_steps[t] >= jj - 1, "P rewritten before its P.V is done"
            P[t] = jj
            P_FULL[t].arrive()
            yield
        assert n16 == issued16[t], "the softmax counts other S16 phases than the MMA thread issued"

    pv_done_steps = [-1] * NT

    def complete_mma(t):
        kind, i, bar = mma_q[t].pop(0)
        jlo = ranges[t][0]
        if kind == "commit":
            bar.arrive()
            return
        assert stage[stage_of(jlo + i)] == jlo + i, f"{kind} on a stage that no longer holds its key"
        open_reads[jlo + i] -= 1
        if kind == "qk8":
            assert s8_read[t] == i - 1, "QK8 rewrote S8 before the softmax read it"
            S8[t] = i
        elif kind == "qk16":
            # the previous products in the buffer were consumed or never needed
            S16[t] = i
        else:
            assert P[t] == i, "P.V of another step's P"
            pv_done_steps[t] = i

    actors = [producer()] + [mma(t) for t in range(NT)] + [softmax(t) for t in range(NT)]
    live = list(actors)
    steps = 0
    while live or copies or any(mma_q):
        steps += 1
        assert steps < 300000, "no progress"
        choices = [("actor", x) for x in live]
        if copies:
            choices.append(("copy", None))
        for t in range(NT):
            if mma_q[t]:
                choices.append(("mma", t))
        kind, x = rng.choice(choices)
        if kind == "actor":
            try:
                next(x)
            except StopIteration:
                live.remove(x)
        elif kind == "copy":
            s, j = copies.pop(0)
            stage[s] = j
            KV_FULL[s].complete_tx(1)
        else:
            complete_mma(x)
    for t in range(NT):
        f = flags[t][: ranges[t][1] - ranges[t][0]]
        ahead = [True] + f[:-1]
        assert counts[t][0] == sum(f)
        assert counts[t][1] == sum(a and not b for a, b in zip(ahead, f))
        assert counts[t][2] == sum(b and not a for a, b in zip(ahead, f))
    return steps


def _case(rng, density):
    # causal-like: both tiles from key 0, the second two keys longer; or
    # sliding-like: later starts
    n0 = rng.randint(1, 7)
    if rng.random() < 0.5:
        ranges = [(0, n0), (0, n0 + 2)]
    else:
        a = rng.randint(0, 3)
        ranges = [(a, a + n0), (a + rng.randint(0, 2), a + n0 + 2)]
    flags = [[rng.random() < density for _ in range(r[1] - r[0])] for r in ranges]
    return ranges, flags


@pytest.mark.parametrize("density", [0.0, 0.15, 0.5, 0.85, 1.0])
def test_fwd_protocol_random_interleavings(density):
    rng = random.Random(int(density * 100) + 17)
    for k in range(120):
        ranges, flags = _case(rng, density)
        run(rng.randrange(1 << 30), ranges, flags)
        # one query tile per CTA (the optional modes at d = 128)
        run(rng.randrange(1 << 30), ranges[:1], flags[:1])


@pytest.mark.parametrize("drop", ["kv_empty", "pv_done", "skip"])
def test_model_catches_a_missing_wait(drop):
    """The checks are not vacuous: with the producer's stage-release wait or
    the softmax's P.V-done wait taken out of the model, some interleaving
    refills a stage still in use or rewrites P before its P.V; and without
    the late-starting tile's waits and releases of the keys before its
    first one ("skip"), its first QK8 can pass the stage's parity wait a
    phase early and read a stage that does not yet hold its key."""
    rng = random.Random(5)
    failures = 0
    for k in range(300):
        ranges, flags = _case(rng, 0.5)
        try:
            run(rng.randrange(1 << 30), ranges, flags, drop=drop)
        except AssertionError:
            failures += 1
    assert failures > 0


# ---------------------------------------------------------------------------
# The one-stage path (d = 256, one query tile per CTA): K8 in two slots by
# key parity, K16 and V in their own parts of the stage with their own
# barriers, two S16 buffers (one barrier each); the producer loads K16(j),
# K8(j + 1), V(j) in that order; the MMA thread issues QK8(i), then step
# i - 1's late QK16 or its K16 release, step i's speculative QK16, then
# P.V(i - 1).

def run_one_stage(seed, n, flags, drop=None):
    rng = random.Random(seed)
    K8_FULL, K8_EMPTY = [Bar(), Bar()], [Bar(), Bar()]
    K16_FULL, K16_EMPTY, V_FULL, V_EMPTY = Bar(), Bar(), Bar(), Bar()
    S_FULL, DEC, P_FULL, PV_DONE = Bar(), Bar(), Bar(), Bar()
    S16_FULL = [Bar(), Bar()]
    k8 = [None, None]                 # key in each K8 slot
    k16 = [None]
    vv = [None]
    S8, S16, P = [None], [None, None], [None]
    s8_read = [-1]
    ANY = [None, None]
    reads = {"k8": {}, "k16": {}, "v": {}}
    mq = []                           # MMA ops and commits in issue order
    copies = []                       # (part, slot, key) in issue order
    issued16 = [0, 0]
    pv_done = [-1]

    def producer():
        def load_k8(u):
            K8_FULL[u & 1].expect_tx(1)
            copies.append(("k8", u & 1, u))

        if n > 0:
            load_k8(0)
        for u in range(n):
            if u >= 1:
                while not K16_EMPTY.passed((u - 1) & 1):
                    yield
                assert reads["k16"].get(u - 1, 0) == 0
            K16_FULL.expect_tx(1)
            copies.append(("k16", 0, u))
            yield
            if u + 1 < n:
                v = u + 1  # its slot held key v - 2
                if v >= 2:
                    while drop != "k8_empty" and not K8_EMPTY[v & 1].passed(((v - 2) >> 1) & 1):
                        yield
                    assert reads["k8"].get(v - 2, 0) == 0, "K8 slot refilled while still read"
                load_k8(v)
                yield
            if u >= 1:
                while not V_EMPTY.passed((u - 1) & 1):
                    yield
                assert reads["v"].get(u - 1, 0) == 0
            V_FULL.expect_tx(1)
            copies.append(("v", 0, u))
            yield

    def issue(kind, i=None, bar=None):
        for part in {"qk8": ("k8",), "qk16": ("k16",), "pv": ("v",)}.get(kind, ()):
            reads[part][i] = reads[part].get(i, 0) + 1
        mq.append((kind, i, bar))

    def mma():
        if n <= 0:
            return
        counts = [0, 0, 0]

        def qk16(i):
            issue("qk16", i)
            issue("commit", bar=S16_FULL[i & 1])
            issue("commit", bar=K16_EMPTY)
            issued16[i & 1] += 1

        def decided(i):
            while not K16_FULL.passed(i & 1):
                yield
            step, f = ANY[i & 1]
            assert step == i
            if f:
                qk16(i)
            else:
                K16_EMPTY.arrive()

        spec = True
        for i in range(n):
            ph = i & 1
            if i > 0:
                while not DEC.passed((i - 1) & 1):
                    yield
                K8_EMPTY[(i - 1) & 1].arrive()  # K8 slot of key i - 1
            while not K8_FULL[i & 1].passed((i >> 1) & 1):
                yield
            issue("qk8", i)
            issue("commit", bar=S_FULL)
            if i > 0:
                step, prev = ANY[(i - 1) & 1]
                assert step == i - 1
                if not spec:
                    yield from decided(i - 1)
                spec = prev
            if spec:
                while not K16_FULL.passed(ph):
                    yield
                qk16(i)
            if i > 0:
                while not P_FULL.passed((i - 1) & 1):
                    yield
                while not V_FULL.passed(ph ^ 1):
                    yield
                issue("pv", i - 1)
                issue("commit", bar=PV_DONE)
                issue("commit", bar=V_EMPTY)
            yield
        while not DEC.passed((n - 1) & 1):
            yield
        if not spec:
            yield from decided(n - 1)
        while not P_FULL.passed((n - 1) & 1):
            yield
        while not V_FULL.passed((n - 1) & 1):
            yield
        issue("pv", n - 1)
        issue("commit", bar=PV_DONE)

    def softmax():
        n16, prev_any = [0, 0], True
        for jj in range(n):
            while not S_FULL.passed(jj & 1):
                yield
            assert S8[0] == jj
            assert k8[jj & 1] == jj, "K8 of the step's key gone before its decision"
            s8_read[0] = jj
            yield
            any_ = flags[jj]
            ANY[jj & 1] = (jj, any_)
            DEC.arrive()
            yield
            if jj > 0:
                while not PV_DONE.passed((jj - 1) & 1):
                    yield
            b = jj & 1
            if any_:
                while not S16_FULL[b].passed(n16[b] & 1):
                    yield
                assert S16[b] == jj, "S16 of another step"
            n16[b] += 1 if (any_ or prev_any) else 0
            prev_any = any_
            yield
            assert jj == 0 or pv_done[0] >= jj - 1
            P[0] = jj
            P_FULL.arrive()
            yield
        assert n16 == issued16

    def complete_mma():
        kind, i, bar = mq.pop(0)
        if kind == "commit":
            bar.arrive()
            return
        if kind == "qk8":
            assert k8[i & 1] == i and s8_read[0] == i - 1
            reads["k8"][i] -= 1
            S8[0] = i
        elif kind == "qk16":
            assert k16[0] == i
            reads["k16"][i] -= 1
            S16[i & 1] = i
        else:
            assert vv[0] == i and P[0] == i
            reads["v"][i] -= 1
            pv_done[0] = i

    live = [producer(), mma(), softmax()]
    steps = 0
    while live or copies or mq:
        steps += 1
        assert steps < 300000, "no progress"
        choices = [("actor", x) for x in live] + ([("copy", None)] if copies else []) + \
            ([("mma", None)] if mq else [])
        kind, x = rng.choice(choices)
        if kind == "actor":
            try:
                next(x)
            except StopIteration:
                live.remove(x)
        elif kind == "copy":
            part, slot, key = copies.pop(0)
            if part == "k8":
                k8[slot] = key
                K8_FULL[slot].complete_tx(1)
            elif part == "k16":
                k16[0] = key
                K16_FULL.complete_tx(1)
            else:
                vv[0] = key
                V_FULL.complete_tx(1)
        else:
            complete_mma()


@pytest.mark.parametrize("density", [0.0, 0.15, 0.5, 0.85, 1.0])
def test_one_stage_protocol_random_interleavings(density):
    rng = random.Random(int(density * 100) + 29)
    for k in range(150):
        n = rng.randint(1, 9)
        run_one_stage(rng.randrange(1 << 30), n, [rng.random() < density for _ in range(n)])


def test_one_stage_model_catches_a_missing_wait():
    rng = random.Random(3)
    failures = 0
    for k in range(300):
        n = rng.randint(3, 9)
        try:
            run_one_stage(rng.randrange(1 << 30), n, [rng.random() < 0.5 for _ in range(n)], drop="k8_empty")
        except AssertionError:
            failures += 1
    assert failures > 0


# ---------------------------------------------------------------------------
# The detector-only tau-sweep pass on the two-stage path: QK8 only, a key's
# stage handed back once the softmax has published its step (its exact
# re-derivations read K8 until then), a late-starting tile's earlier keys
# handed back unused.

def run_sweep(seed, ranges, drop=None):
    rng = random.Random(seed)
    NT = len(ranges)
    J0 = min(r[0] for r in ranges)
    J1 = max(r[1] for r in ranges)
    stage_of = lambda j: (j - J0) % NS  # noqa: E731
    KV_FULL = [Bar() for _ in range(NS)]
    KV_EMPTY = [[Bar() for _ in range(NT)] for _ in range(NS)]
    S_FULL, DEC = [Bar() for _ in range(NT)], [Bar() for _ in range(NT)]
    stage = [None] * NS
    S8 = [None] * NT
    in_use = {}  # key -> tiles that have not released it
    mq = [[] for _ in range(NT)]
    copies = []

    def producer():
        rel = 0
        for j in range(J0, J1):
            s, u = stage_of(j), (j - J0) // NS
            if u >= 1:
                jr = j - NS
                for t in range(NT):
                    used = ranges[t][0] <= jr < ranges[t][1] if drop == "skip" else \
                        (ranges[t][1] > ranges[t][0] and jr < ranges[t][1])
                    if not used:
                        continue
                    bit = 1 << (2 * t + s)
                    while not KV_EMPTY[s][t].passed(1 if rel & bit else 0):
                        yield
                    rel ^= bit
                assert not in_use.get(jr), "stage refilled while a tile still reads its key"
            KV_FULL[s].expect_tx(1)
            copies.append((s, j))
            yield

    def mma(t):
        jlo, jhi = ranges[t]
        n = jhi - jlo
        if n <= 0:
            return
        if drop != "skip":
            for j in range(J0, jlo):
                while not KV_FULL[stage_of(j)].passed(((j - J0) // NS) & 1):
                    yield
                KV_EMPTY[stage_of(j)][t].arrive()
                yield
        for i in range(n):
            j = jlo + i
            if i > 0:
                while not DEC[t].passed((i - 1) & 1):
                    yield
                in_use[j - 1].discard(t)
                KV_EMPTY[stage_of(j - 1)][t].arrive()
            while not KV_FULL[stage_of(j)].passed(((j - J0) // NS) & 1):
                yield
            in_use.setdefault(j, set()).add(t)
            mq[t].append(("qk8", i))
            mq[t].append(("commit", S_FULL[t]))
            yield
        while not DEC[t].passed((n - 1) & 1):
            yield
        in_use[jhi - 1].discard(t)
        KV_EMPTY[stage_of(jhi - 1)][t].arrive()

    def softmax(t):
        jlo, jhi = ranges[t]
        for jj in range(jhi - jlo):
            while not S_FULL[t].passed(jj & 1):
                yield
            assert S8[t] == jj
            assert stage[stage_of(jlo + jj)] == jlo + jj, "K8 of the step's key gone before its decision"
            yield
            DEC[t].arrive()
            yield

    def complete(t):
        kind, x = mq[t].pop(0)
        if kind == "commit":
            x.arrive()
            return
        j = ranges[t][0] + x
        assert stage[stage_of(j)] == j, "QK8 on a stage that does not hold its key"
        S8[t] = x

    live = [producer()] + [mma(t) for t in range(NT)] + [softmax(t) for t in range(NT)]
    steps = 0
    while live or copies or any(mq):
        steps += 1
        assert steps < 300000, "no progress"
        choices = [("actor", x) for x in live] + ([("copy", None)] if copies else []) + \
            [("mma", t) for t in range(NT) if mq[t]]
        kind, x = rng.choice(choices)
        if kind == "actor":
            try:
                next(x)
            except StopIteration:
                live.remove(x)
        elif kind == "copy":
            s, j = copies.pop(0)
            stage[s] = j
            KV_FULL[s].complete_tx(1)
        else:
            complete(x)


def test_sweep_protocol_random_interleavings():
    rng = random.Random(41)
    for k in range(300):
        ranges, _ = _case(rng, 0.0)
        run_sweep(rng.randrange(1 << 30), ranges)


def test_sweep_model_catches_the_early_parity_pass():
    rng = random.Random(43)
    failures = 0
    for k in range(300):
        ranges, _ = _case(rng, 0.0)
        try:
            run_sweep(rng.randrange(1 << 30), ranges, drop="skip")
        except AssertionError:
            failures += 1
    assert failures > 0
