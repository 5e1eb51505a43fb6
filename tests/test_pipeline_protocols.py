"""Host-side models of the tensor-core kernels' mbarrier protocols.

Each kernel is a set of roles (a producer, MMA issuers, epilogues, ...) that
hand buffers to one another through mbarriers.  A waiter names the phase it
wants only by its parity (one bit), so a waiter two phases ahead of a barrier
passes early and one two phases behind waits forever.  These models replay every role's
waits and arrivals, in the order the kernels issue them, under random
interleavings, and fail on a deadlock, on a wait satisfied by any phase but
the one it wants, or on a role touching a buffer that holds another chunk.
They model the protocols as written in the kernel sources (kept in step by
hand); they do not run the kernels.

Covered:
  * the summary kernel's stage rings and accumulators: with two MMA-issuing
    warps each unit goes through its issuer's own ring of stages and unit it
    accumulates in TMEM slot it % 4, each issuer alternating two (safe); one
    ring shared by
    both issuers lets an issuer that skips the other's units wait on a stage
    two phases ahead and read it early (the negative control: the form that
    faulted a backward run on the Wan shape -- the split-precision layout's
    three stages, three chunks per unit);
  * the causal output kernel: three token stages, two state buffers, units
    taken in pairs whose chunks alternate, the MMA warp issuing whichever of
    a chunk's two MMA groups is ready.
"""

from __future__ import annotations

import random

import pytest


class Bar:
    """An mbarrier: `count` arrivals complete a phase."""

    def __init__(self, count: int):
        self.count, self.pend, self.ph = count, count, 0

    def arrive(self, n: int = 1):
        self.pend -= n
        assert self.pend >= 0, "more arrivals than the barrier's count"
        if self.pend == 0:
            self.ph += 1
            self.pend = self.count

    def done(self, q: int) -> bool:
        """What a parity wait for phase q (0-based; -1 = the phase before the
        first) sees: complete whenever the number of completed phases differs
        from q by an odd number.  That answer is right only when exactly q + 1
        phases have completed; fails when the waiter is two phases ahead (it
        would pass early) or two phases behind (it would wait forever)."""
        passes = (self.ph - q) % 2 == 1
        if passes:
            assert self.ph == q + 1, ("parity wait passes on the wrong phase", q, self.ph)
        else:
            assert self.ph <= q, ("parity wait two phases behind", q, self.ph)
        return passes


def schedule(roles, rnd, limit=20000):
    """Run generator roles in random order; a role yields while it waits."""
    live = list(range(len(roles)))
    idle = 0
    while live:
        r = rnd.choice(live)
        try:
            progressed = next(roles[r])
        except StopIteration:
            live.remove(r)
            idle = 0
            continue
        idle = 0 if progressed else idle + 1
        if idle > limit:
            raise AssertionError("deadlock")


def wait(bar: Bar, q: int):
    while not bar.done(q):
        yield False


# --------------------------------------------------------------- summary kernel
def summary_protocol(units: int, cpp: int, nstages: int, nissuers: int, shared_ring: bool, seed: int,
                     nacc: int = 4):
    rnd = random.Random(seed)
    full = [Bar(1) for _ in range(nstages)]
    kready = [Bar(1) for _ in range(nstages)]
    empty = [Bar(1) for _ in range(nstages)]
    # unit it accumulates in TMEM slot it % nacc (each issuer alternates its own slots)
    accfull = [Bar(1) for _ in range(nacc)]
    accempty = [Bar(1) for _ in range(nacc)]
    content = [None] * nstages

    def ring(it):
        if shared_ring or nissuers == 1:
            return list(range(nstages))
        j = it % nissuers
        return list(range(j, nstages, nissuers))

    def walk():
        ctr = {}
        for it in range(units):
            r = tuple(ring(it))
            for c in range(cpp):
                k = ctr.get(r, 0)
                ctr[r] = k + 1
                yield it, c, r[k % len(r)], k // len(r)

    def producer():
        for it, c, s, k in walk():
            yield from wait(empty[s], k - 1)
            content[s] = (it, c)
            full[s].arrive()
            yield True

    def phi():
        for it, c, s, k in walk():
            yield from wait(full[s], k)
            assert content[s] == (it, c), "phi read another chunk"
            kready[s].arrive()
            yield True

    def issuer(j):
        uses = [0] * nacc
        for it, c, s, k in walk():
            if it % nissuers != j:
                continue
            acc = it % nacc
            if c == 0:
                yield from wait(accempty[acc], uses[acc] - 1)
            yield from wait(kready[s], k)
            assert content[s] == (it, c), "MMA read another chunk"
            empty[s].arrive()
            if c == cpp - 1:
                accfull[acc].arrive()
                uses[acc] += 1
            yield True

    def epilogue():
        for it in range(units):
            acc = it % nacc
            yield from wait(accfull[acc], it // nacc)
            accempty[acc].arrive()
            yield True

    schedule([producer(), phi(), epilogue()] + [issuer(j) for j in range(nissuers)], rnd)


@pytest.mark.parametrize("nacc", [2, 4])
@pytest.mark.parametrize("nstages,nissuers", [(6, 2), (5, 2), (4, 2), (3, 1), (5, 1)])
def test_summary_stage_rings_are_safe(nstages, nissuers, nacc):
    for units in (1, 2, 3, 5, 8, 11):
        for cpp in (1, 2, 3, 4):
            for seed in range(25):
                summary_protocol(units, cpp, nstages, nissuers, shared_ring=False, seed=seed, nacc=nacc)


@pytest.mark.parametrize("nstages,cpp", [(3, 3), (4, 4)])
def test_summary_shared_ring_with_two_issuers_reads_a_stage_early(nstages, cpp):
    failures = 0
    for seed in range(40):
        try:
            summary_protocol(8, cpp, nstages, 2, shared_ring=True, seed=seed)
        except AssertionError:
            failures += 1
    assert failures > 0


# ------------------------------------------------------- causal output kernel
def causal_protocol(units: int, nck: int, seed: int):
    rnd = random.Random(seed)
    NS = 3
    tfull = [Bar(1) for _ in range(NS)]
    pready = [Bar(4) for _ in range(NS)]
    tempty = [Bar(1) for _ in range(NS)]
    stfull = [Bar(1) for _ in range(2)]
    stfree = [Bar(1) for _ in range(2)]
    stupd = [Bar(2) for _ in range(2)]
    afull = [Bar(1) for _ in range(2)]
    afree = [Bar(4) for _ in range(2)]
    sfull, sfree, ptready, ptfree, ufree = Bar(1), Bar(4), Bar(4), Bar(1), Bar(2)
    chunks = []
    n = 0
    for k0 in range(0, units, 2):
        sides = [0, 1] if k0 + 1 < units else [0]
        for c in range(nck):
            for side in sides:
                chunks.append((n, k0 + side, c))
                n += 1

    def producer():
        for n, k, c in chunks:
            s = n % NS
            yield from wait(tempty[s], n // NS - 1)
            tfull[s].arrive()
            yield True

    def records():
        for k in range(units):
            x = k & 1
            yield from wait(stfree[x], (k >> 1) - 1)
            stfull[x].arrive()
            yield True

    def mma():
        nupd, nu, q, i = [0, 0], 0, [], 0
        while i < len(chunks) or q:
            opts = []
            if q:
                pn, ps, pmore = q[0]
                if ptready.done(pn) and (not pmore or nu == 0 or ufree.done(nu - 1)):
                    opts.append("sg")
            if i < len(chunks) and len(q) < 2:
                n, k, c = chunks[i]
                s, x, acc = n % NS, k & 1, n & 1
                ok = stfull[x].done(k >> 1) if c == 0 else stupd[x].done(nupd[x])
                if ok and pready[s].done(n // NS) and afree[acc].done((n >> 1) - 1) and sfree.done(n - 1):
                    opts.append("as")
            if not opts:
                yield False
                continue
            if rnd.choice(opts) == "sg":
                pn, ps, pmore = q.pop(0)
                nu += pmore
                tempty[ps].arrive()
                ptfree.arrive()
                afull[pn & 1].arrive()
            else:
                n, k, c = chunks[i]
                x = k & 1
                if c > 0:
                    nupd[x] += 1
                sfull.arrive()
                if c + 1 == nck:
                    stfree[x].arrive()
                q.append((n, n % NS, c + 1 < nck))
                i += 1
            yield True

    def phi():
        for n, k, c in chunks:
            s = n % NS
            yield from wait(tfull[s], n // NS)
            pready[s].arrive(4)
            yield True

    def scores():
        for n, k, c in chunks:
            yield from wait(sfull, n)
            yield from wait(ptfree, n - 1)
            sfree.arrive(4)
            ptready.arrive(4)
            yield True

    def outputs():
        for n, k, c in chunks:
            acc, x, upd = n & 1, k & 1, c + 1 < nck
            if upd and c == 0:
                yield from wait(stfull[x], k >> 1)
            yield from wait(afull[acc], n >> 1)
            if upd:
                ufree.arrive(2)
                stupd[x].arrive(2)
            afree[acc].arrive(4)
            yield True

    schedule([producer(), records(), mma(), phi(), scores(), outputs()], rnd)


@pytest.mark.parametrize("nck", [1, 2, 3, 4])
def test_causal_protocol_is_safe(nck):
    for units in (1, 2, 3, 4, 7):
        for seed in range(25):
            causal_protocol(units, nck, seed)
