"""A CPU model of the QKV projection kernel's barrier protocol (the CTA
pair of lamp_qkv.cu) under random interleavings: both CTAs' TMA producers,
the first CTA's MMA thread and the eight epilogue warps run the kernel's
loops with its phase / parity formulas, against mbarriers with the
hardware's semantics (arrival count, transaction bytes that may arrive
before they are expected, completion when both reach zero, a parity wait
that passes once the phase of that parity has completed), while copies and
MMA commits complete asynchronously, in issue order per source.  Checked:
a stage is refilled only after the MMAs that read it are done, an MMA reads
a stage only after both CTAs' copies into it landed, an accumulator is
rewritten only after both CTAs' epilogues read it, an epilogue reads only a
finished accumulator, and every run finishes (a lag of two phases on a
parity wait would hang and is caught as a deadlock)."""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.tx, self.phase = count, count, 0, 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self):
        assert self.pending > 0
        self.pending -= 1
        self._maybe_complete()

    def expect_tx(self, n):  # arrive.expect_tx
        self.tx += n
        self.arrive()

    def complete_tx(self, n):
        self.tx -= n
        self._maybe_complete()

    def passed(self, parity):  # try_wait.parity
        return (self.phase & 1) != parity


def run(seed, ntiles, nkb, nst=6, stage_bytes=32, drop=None):
    """One random interleaving; ``drop`` takes one wait out of the model
    ("acce": the MMA's wait for the accumulator's release, "empty": the
    producers' wait for a stage's release) to show that the checks catch it."""
    rng = random.Random(seed)
    full = [Bar(1) for _ in range(nst)]                      # first CTA's: its producer + both CTAs' bytes
    empty = [[Bar(1) for _ in range(nst)] for _ in range(2)]  # per CTA: the pair's MMA commit (multicast)
    accf = [[Bar(1) for _ in range(2)] for _ in range(2)]     # per CTA and accumulator
    acce = [Bar(8) for _ in range(2)]                          # first CTA's: one lane of each epilogue warp
    landed = [[None] * nst for _ in range(2)]                  # K block held by each CTA's stage
    mma_done = [-1]                                            # last K block whose MMAs completed
    acc_tile = [None, None]                                    # tile whose MMAs completed in each accumulator
    reads_left = {}                                            # tile -> epilogue warps still to read it
    inflight_copy = [[], []]                                   # per CTA: (stage, K block), in issue order
    inflight_commit = []                                       # ("empty", s, it) / ("accf", a, lt) in issue order

    def producer(r):
        it = 0
        for tile in range(ntiles):
            for kb in range(nkb):
                s, u = it % nst, it // nst
                if u > 0 and drop != "empty":
                    while not empty[r][s].passed((u - 1) & 1):
                        yield
                # refill only after the MMAs that read the previous K block of this stage
                assert mma_done[0] >= it - nst
                if r == 0:
                    full[s].expect_tx(2 * stage_bytes)
                inflight_copy[r].append((s, it))
                it += 1
                yield

    def mma():
        it = 0
        for lt in range(ntiles):
            a = lt & 1
            if lt >= 2:
                while drop != "acce" and not acce[a].passed(((lt >> 1) - 1) & 1):
                    yield
                assert reads_left.get(lt - 2, 0) == 0  # both epilogues read tile lt - 2
            for kb in range(nkb):
                s, u = it % nst, it // nst
                while not full[s].passed(u & 1):
                    yield
                assert landed[0][s] == it and landed[1][s] == it
                inflight_commit.append(("empty", s, it))
                it += 1
                yield
            inflight_commit.append(("accf", a, lt))
            yield

    def epilogue(r, w):
        for lt in range(ntiles):
            a = lt & 1
            while not accf[r][a].passed((lt >> 1) & 1):
                yield
            assert acc_tile[a] == lt  # the accumulator holds this tile's finished sums
            yield  # the TMEM loads
            reads_left[lt] -= 1
            acce[a].arrive()
            yield

    for lt in range(ntiles):
        reads_left[lt] = 8
    actors = [producer(0), producer(1), mma()] + [epilogue(r, w) for r in range(2) for w in range(4)]
    live = list(actors)
    steps = 0
    while live or inflight_copy[0] or inflight_copy[1] or inflight_commit:
        steps += 1
        assert steps < 200000, "no progress"
        choices = [("actor", x) for x in live]
        for r in range(2):
            if inflight_copy[r]:
                choices.append(("copy", r))
        if inflight_commit:
            choices.append(("commit", None))
        kind, x = rng.choice(choices)
        if kind == "actor":
            try:
                next(x)
            except StopIteration:
                live.remove(x)
        elif kind == "copy":
            s, it = inflight_copy[x].pop(0)
            landed[x][s] = it
            full[s].complete_tx(stage_bytes)
        else:
            what, i, n = inflight_commit.pop(0)
            if what == "empty":
                mma_done[0] = n
                for r in range(2):
                    empty[r][i].arrive()
            else:
                acc_tile[i] = n
                for r in range(2):
                    accf[r][i].arrive()
    assert all(v == 0 for v in reads_left.values())
    return steps


@pytest.mark.parametrize("ntiles,nkb", [(1, 1), (2, 3), (5, 3), (7, 1), (4, 13), (9, 6)])
def test_pair_protocol_random_interleavings(ntiles, nkb):
    for seed in range(60):
        run(seed * 7919 + ntiles * 31 + nkb, ntiles, nkb)


@pytest.mark.parametrize("drop", ["acce", "empty"])
def test_model_catches_a_missing_wait(drop):
    """The checks are not vacuous: with one of the kernel's waits taken out
    of the model, some interleaving refills a stage the MMAs still read or
    rewrites an accumulator an epilogue has not read (or a barrier's
    arrivals run past its phase)."""
    failures = 0
    for seed in range(200):
        try:
            run(seed, 6, 3, drop=drop)
        except AssertionError:
            failures += 1
    assert failures > 0
