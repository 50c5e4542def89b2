"""A model of the staged kernel's row protocol, run under random interleavings on the CPU.

The kernel's producer (one thread a CTA) and its consumer groups share a ring of
`stages` shared-memory slots through two mbarriers a slot (full: the producer's arrive
plus the bytes of the row's copies; empty: the group's release). Rows enter the ring at
a fixed stride (with a row counter, only each CTA's first `static` rows: a ring-full or
more), then in runs of `run` rows claimed by atomic adds;
after the last row each group gets an end marker (row -1), and the last CTA to finish
claiming zeroes the counter pair. This file restates those steps as coroutines, with
the mbarrier's phase / parity rule (a wait on parity P returns once the phase of parity
P has completed; a fresh barrier counts the phase before its first as complete), copies
that land at arbitrary later times, and CTAs and groups interleaved at random. It checks
the protocol, not the CUDA code: every row processed exactly once, no deadlock, every
copy landed before its CTA exits, the counter pair zero at the end. Three planted
mistakes must each be caught, so that the model is not vacuous."""
import random

import pytest


class Bar:
    """An mbarrier: `count` arrivals and all expected bytes complete a phase."""

    def __init__(self, count):
        self.count, self.pending, self.tx, self.completed = count, count, 0, 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.completed += 1
            self.pending = self.count

    def arrive(self):
        assert self.pending > 0, "arrival beyond the barrier's count"
        self.pending -= 1
        self._maybe_complete()

    def arrive_expect_tx(self, copies):
        self.tx += copies
        self.arrive()

    def complete_tx(self):
        assert self.tx > 0
        self.tx -= 1
        self._maybe_complete()

    def done(self, parity):
        return (self.completed & 1) != parity


class Deadlock(Exception):
    pass


def simulate(tokens, grid, stages, groups, claimed, run, residual, rng, mutant=None, static=None):
    static = stages if static is None else static
    counter = [0, 0]  # next claim, CTAs done
    processed = []
    landing = []      # barriers with a copy in flight, one entry per copy
    actors = []

    def cta(b):
        full = [Bar(1) for _ in range(stages)]
        empty = [Bar(1) for _ in range(stages)]  # one arrival a group (the kernel: one a warp)
        slot_row = [None] * stages
        n_static = (tokens - b + grid - 1) // grid if tokens > b else 0
        if claimed and n_static > static:
            n_static = static
        first = min(n_static, stages)
        copies = 2 if residual else 1

        def issue(row, slot):
            slot_row[slot] = row
            full[slot].arrive_expect_tx(copies)
            landing.extend([full[slot]] * copies)

        for k in range(first):  # before the weight row, no slot to wait for
            issue(b + k * grid, k)

        def producer():
            st = {"k": first, "slot": first % stages, "phase": (first // stages) & 1}

            def put(row):
                if st["k"] >= stages and mutant != "no_empty_wait":
                    bar, par = empty[st["slot"]], st["phase"] ^ 1
                    yield lambda: bar.done(par)
                if row >= 0:
                    issue(row, st["slot"])
                else:
                    slot_row[st["slot"]] = -1
                    full[st["slot"]].arrive()
                st["k"] += 1
                st["slot"] += 1
                if st["slot"] == stages:
                    st["slot"], st["phase"] = 0, st["phase"] ^ 1

            for i in range(first, n_static):
                yield from put(b + i * grid)
            if claimed:
                r0 = grid * (stages if mutant == "r0_from_stages" else static)
                c0 = counter[0]
                counter[0] += run
                yield None
                c1 = counter[0]
                counter[0] += run
                yield None
                while r0 + c0 < tokens:
                    for row in range(r0 + c0, min(r0 + c0 + run, tokens)):
                        yield from put(row)
                    c0 = c1
                    if r0 + c0 >= tokens:
                        break
                    c1 = counter[0]
                    counter[0] += run
                    yield None
                counter[1] += 1
                if counter[1] == grid and mutant != "no_reset":
                    counter[0] = counter[1] = 0
                yield None
            for _ in range(groups - (1 if mutant == "one_marker_short" else 0)):
                yield from put(-1)
            k = st["k"]
            for j in range(max(k - stages, 0), k):
                bar, par = full[j % stages], (j // stages) & 1
                yield lambda: bar.done(par)
            # every copy into this CTA's ring has landed
            assert not any(any(x is f for f in full) for x in landing), "a CTA exited with a copy in flight"

        def consumer(g):
            slot, phase = g, 0
            while True:
                bar, par = full[slot], phase
                yield lambda: bar.done(par)
                row = slot_row[slot]
                if row < 0:
                    return
                processed.append(row)
                yield None
                empty[slot].arrive()
                slot += groups
                if slot >= stages:
                    slot, phase = slot - stages, phase ^ 1

        return [producer()] + [consumer(g) for g in range(groups)]

    for b in range(grid):
        for gen in cta(b):
            actors.append([gen, None, False])  # generator, its wait, started
    live = actors
    steps = 0
    while live or landing:
        runnable = [a for a in live if not a[2] or a[1] is None or a[1]()]
        n_choices = len(runnable) + (1 if landing else 0)
        if n_choices == 0:
            raise Deadlock(f"{len(live)} actors blocked, no copy in flight")
        pick = rng.randrange(n_choices)
        if pick == len(runnable):
            landing.pop(rng.randrange(len(landing))).complete_tx()
        else:
            a = runnable[pick]
            try:
                a[1] = a[0].send(None)
                a[2] = True
            except StopIteration:
                live = [x for x in live if x is not a]
        steps += 1
        assert steps < 200000, "runaway simulation"
    return processed, counter


def shapes(n, seed):
    rng = random.Random(seed)
    for _ in range(n):
        stages = rng.choice([2, 3, 4, 6, 8])
        groups = rng.choice([g for g in range(1, stages + 1) if stages % g == 0])
        yield (rng.randint(1, 120), rng.randint(1, 5), stages, groups, rng.random() < 0.7,
               rng.choice([1, 2, 3, 7]), rng.random() < 0.5, rng.randrange(1 << 30))


@pytest.mark.parametrize("tokens,grid,stages,groups,claimed,run,residual,seed", list(shapes(160, 2024)))
def test_every_row_once_no_deadlock_counter_zero(tokens, grid, stages, groups, claimed, run, residual, seed):
    processed, counter = simulate(tokens, grid, stages, groups, claimed, run, residual, random.Random(seed))
    assert sorted(processed) == list(range(tokens))
    assert counter == [0, 0]


def static_shapes(n, seed):
    rng = random.Random(seed)
    for _ in range(n):
        stages = rng.choice([2, 4, 6, 10])
        groups = rng.choice([g for g in range(1, stages + 1) if stages % g == 0])
        tokens, grid = rng.randint(1, 160), rng.randint(1, 5)
        per = tokens // grid
        yield (tokens, grid, stages, groups, rng.choice([1, 2, 3]), rng.random() < 0.5,
               max(stages, per - (per + 3) // 4) + rng.choice([0, 0, 1, 5]), rng.randrange(1 << 30))


@pytest.mark.parametrize("tokens,grid,stages,groups,run,residual,static,seed", list(static_shapes(80, 77)))
def test_claims_after_a_longer_fixed_stride(tokens, grid, stages, groups, run, residual, static, seed):
    """Each CTA's first `static` rows at the fixed stride (a ring-full or more; up to its
    whole share), then claimed runs from row grid * static."""
    processed, counter = simulate(tokens, grid, stages, groups, True, run, residual, random.Random(seed),
                                  static=static)
    assert sorted(processed) == list(range(tokens))
    assert counter == [0, 0]


@pytest.mark.parametrize("seed", range(12))
def test_many_interleavings_of_one_shape(seed):
    """Claims crossing the last row, more groups than rows per CTA, two copies a row."""
    processed, counter = simulate(47, 4, 6, 3, True, 3, True, random.Random(seed))
    assert sorted(processed) == list(range(47))
    assert counter == [0, 0]


def test_planted_mistakes_are_caught():
    rng = random.Random(5)
    # claims counted from the first ring-full while the fixed stride ran longer: rows twice
    processed, _ = simulate(120, 3, 4, 2, True, 3, False, rng, mutant="r0_from_stages", static=30)
    assert sorted(processed) != list(range(120))
    # one end marker short: a group waits forever
    with pytest.raises(Deadlock):
        simulate(40, 3, 4, 2, True, 2, False, rng, mutant="one_marker_short")
    # no reset: the next launch given the pair would skip rows
    _, counter = simulate(40, 3, 4, 2, True, 2, False, rng, mutant="no_reset")
    assert counter != [0, 0]
    # no wait for a free slot: a row overwrites one not yet consumed, somewhere in 20 tries
    caught = 0
    for s in range(20):
        try:
            processed, _ = simulate(60, 2, 2, 1, True, 1, False, random.Random(s), mutant="no_empty_wait")
            caught += sorted(processed) != list(range(60))
        except (AssertionError, Deadlock):
            caught += 1
    assert caught > 0
