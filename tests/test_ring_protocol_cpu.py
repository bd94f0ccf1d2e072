"""A model of the copy rings of the CUDA-core kernel that runs both products in one
launch (gemv.cu, kMode 3), checked on the CPU under random interleavings.

The model follows the kernel's bookkeeping: a weight ring of 10 two-step chunks, an
activation ring of 3 eight-step chunks (the down product's steps padded to a fresh
chunk), two reduction slots, per-(tile, down step) counters for the intermediate's
step rows, and the agents' programs as the kernel runs them: the multiply warps
(one agent per step phase), three weight-paced producers, the fourth producer that
copies the down product's activation rows, the epilogue, and the other CTAs'
contributions to the counters. Barriers are modelled like `mbarrier`: a phase
completes when its arrivals and bytes are in, and a parity wait passes when the
barrier's current phase has the other parity. A wait that passes on the wrong phase
(two uses of a slot apart) and a deadlock are both failures. The negative control
runs the fourth producer as first written (interleaving gate/up chunks, parity
waits unpaced by weight copies) and expects the model to catch it."""
import random

import pytest

NWS, NB, BS, WC = 10, 3, 8, 2  # weight slots, activation slots, steps a chunk


class Alias(Exception):
    pass


class Deadlock(Exception):
    pass


class Bar:
    def __init__(self, count):
        self.count, self.pend, self.tx, self.done = count, count, 0, 0

    def arrive(self, n=1):
        self.pend -= n
        assert self.pend >= 0, "more arrivals than the phase expects"
        self._complete()

    def expect(self, nbytes):
        self.tx += nbytes
        self.arrive()

    def land(self, nbytes):
        self.tx -= nbytes
        assert self.tx >= 0, "more bytes than expected"
        self._complete()

    def _complete(self):
        if self.pend == 0 and self.tx == 0:
            self.done += 1
            self.pend = self.count

    def passes(self, parity):
        return (self.done & 1) != parity


def segments(R, KBn, begin, end, ph):
    """A CTA's share [begin, end) of a product as (phase, steps, tile, row tile) in
    the kernel's unit order: the unit the share starts inside, the one it ends
    inside, then the whole units."""
    if end <= begin:
        return []
    segs = []
    for u in range(begin // KBn, (end - 1) // KBn + 1):
        segs.append((u, max(begin, u * KBn), min(end, (u + 1) * KBn)))
    first, last = segs[0], segs[-1]
    p0 = first[1] > first[0] * KBn or first[2] < (first[0] + 1) * KBn
    p1 = len(segs) > 1 and last[2] < (last[0] + 1) * KBn
    order = ([first] if p0 else []) + ([last] if p1 else [])
    order += [sg for sg in segs if not ((sg is first and p0) or (sg is last and p1))]
    return [(ph, e - s, u // R, u % R, s - u * KBn) for (u, s, e) in order]


def simulate(units_a, units_b, seed, paced_copier=True):
    rnd = random.Random(seed)
    n1 = sum(u[1] for u in units_a)
    n_it = n1 + sum(u[1] for u in units_b)
    n_chunks = (n_it + 1) // 2
    nbA = (n1 + BS - 1) // BS
    pad = nbA * BS - n1 if n_it > n1 else 0
    n_bch = (n_it + pad + BS - 1) // BS
    WF = [Bar(1) for _ in range(NWS)]
    WE = [Bar(4 * WC) for _ in range(NWS)]
    BF = [Bar(1) for _ in range(NB)]
    BE = [Bar(4 * BS) for _ in range(NB)]
    RF = [Bar(16) for _ in range(2)]
    RE = [Bar(4) for _ in range(2)]
    ready, inflight, wslot, bslot = {}, [], {}, {}
    phase_a_done = [0]
    steps = []  # per step: (product, tile, down step)
    for (ph, ns, ti, rt, kb0) in units_a + units_b:
        steps += [(ph, ti, kb0 + k) for k in range(ns)]

    def chunk(nb):
        it0 = nb * BS if nb < nbA else nb * BS - pad
        return it0, min(it0 + BS, n1 if nb < nbA else n_it)

    def wait(bar, parity, target):
        while not bar.passes(parity):
            yield False
        if bar.done < target:
            raise Alias(f"parity wait passed at phase {bar.done}, wanted {target}")

    def issue_w(c):
        WF[c % NWS].expect(1)
        wslot[c % NWS] = c
        inflight.append(WF[c % NWS])

    def issue_b(nb):
        s = nb % NB
        it0, it1 = chunk(nb)
        BF[s].expect(1)
        bslot[s] = nb
        inflight.append(BF[s])
        if pad > 0 and nb == nbA - 1:  # the short gate/up chunk's missing reader arrivals
            BE[s].arrive(4 * (BS - (it1 - it0)))

    def counters_ready(nc):
        it0, it1 = chunk(nc)
        for it in range(it0, it1):
            ph, ti, kb = steps[it]
            if ph == 1:
                while ready.get((ti, kb), 0) < 2:
                    yield False

    def producer(q):
        # weight chunks round the first three producers; gate/up activation chunks
        # round the same three (as first written: round all four)
        kB = 3 if paced_copier else 4
        copier = q == 3
        nb = n_bch if (copier and paced_copier) else q
        nw = n_chunks if copier else q
        while nw < NWS:
            nw += 3
        while nb < nbA or nw < n_chunks:
            if nb < nbA and (nw >= n_chunks or nb * BS <= nw * WC):
                yield from wait(BE[nb % NB], ((nb // NB) & 1) ^ 1, nb // NB)
                issue_b(nb)
                nb += kB
            else:
                yield from wait(WE[nw % NWS], ((nw // NWS) & 1) ^ 1, nw // NWS)
                issue_w(nw)
                nw += 3
            yield True
        if copier and nbA < n_bch:
            if paced_copier:
                while phase_a_done[0] < 4:  # (4 agents stand for the 16 warps)
                    yield False
            for nc in range(nbA, n_bch):
                yield from counters_ready(nc)
                if nc >= NB:
                    yield from wait(BE[nc % NB], ((nc // NB) & 1) ^ 1, nc // NB)
                issue_b(nc)
                yield True

    def multiply(p):
        ru, base, signalled = 0, 0, False
        for (ph, ns, ti, rt, kb0) in units_a + units_b:
            if ph == 1 and not signalled:
                phase_a_done[0] += 1
                signalled = True
            for it in range(base, base + ns):
                if it % 4 != p:
                    continue
                c = it // WC
                yield from wait(WF[c % NWS], (c // NWS) & 1, c // NWS + 1)
                assert wslot[c % NWS] == c
                cb = (it + (pad if it >= n1 else 0)) // BS
                yield from wait(BF[cb % NB], (cb // NB) & 1, cb // NB + 1)
                assert bslot[cb % NB] == cb
                yield True
                WE[c % NWS].arrive(4)
                BE[cb % NB].arrive(4)
            base += ns
            yield from wait(RE[ru & 1], ((ru >> 1) & 1) ^ 1, ru >> 1)
            RF[ru & 1].arrive(4)
            ru += 1
            yield True
        if not signalled:
            phase_a_done[0] += 1

    def epilogue():
        for ru, (ph, ns, ti, rt, kb0) in enumerate(units_a + units_b):
            yield from wait(RF[ru & 1], (ru >> 1) & 1, (ru >> 1) + 1)
            yield True
            if ph == 0:
                ready[(ti, rt >> 1)] = ready.get((ti, rt >> 1), 0) + 1
            RE[ru & 1].arrive(4)

    def other_ctas():
        local = {}
        for (ph, ns, ti, rt, kb0) in units_a:
            local[(ti, rt >> 1)] = local.get((ti, rt >> 1), 0) + 1
        for key in sorted({(ti, kb) for (ph, ti, kb) in steps if ph == 1}):
            for _ in range(2 - min(2, local.get(key, 0))):
                for _ in range(rnd.randrange(30)):
                    yield False
                ready[key] = ready.get(key, 0) + 1
                yield True

    for c in range(min(NWS, n_chunks)):  # the multiply warps' first weight copies
        issue_w(c)
    live = [producer(q) for q in range(4)] + [multiply(p) for p in range(4)] + [epilogue(), other_ctas()]
    idle = 0
    while live or inflight:
        if inflight and (not live or rnd.random() < 0.3):
            inflight.pop(rnd.randrange(len(inflight))).land(1)
            idle = 0
            continue
        agent = rnd.choice(live)
        try:
            idle = 0 if next(agent) else idle + 1
        except StopIteration:
            live.remove(agent)
            idle = 0
        if idle > 20000:
            if inflight:
                inflight.pop(0).land(1)
                idle = 0
            else:
                raise Deadlock()


def shares(ntiles, dims, G, c):
    RA, KA, RB, KB = dims
    totA, totB = ntiles * RA * KA, ntiles * RB * KB
    ua = segments(RA, KA, -(-c * totA // G), -(-(c + 1) * totA // G), 0)
    ub = segments(RB, KB, -(-c * totB // G), -(-(c + 1) * totB // G), 1)
    return ua, ub


SMALL = (4, 4, 4, 2)       # E=16-style test shape: 2N/128, K/128, K/128, N/128
FULL = (32, 56, 56, 16)    # the full-size layer


@pytest.mark.parametrize("ntiles,dims,G,c", [
    (4, SMALL, 1, 0), (8, SMALL, 1, 0), (4, SMALL, 3, 1), (4, SMALL, 152, 0), (4, SMALL, 152, 151),
    (1, FULL, 1, 0), (8, FULL, 3, 0), (8, FULL, 7, 3), (8, FULL, 152, 0), (8, FULL, 152, 76), (2, FULL, 2, 1),
])
def test_one_launch_rings_never_alias_or_deadlock(ntiles, dims, G, c):
    ua, ub = shares(ntiles, dims, G, c)
    for seed in range(3):
        simulate(ua, ub, seed)


def test_model_catches_the_unpaced_copier():
    # the fourth producer as first written: it also takes every fourth gate/up
    # chunk and issues no weight copies, so its parity waits can run two uses of a
    # slot ahead of the readers (the kernel faulted this way on one CTA)
    ua, ub = shares(4, SMALL, 1, 0)
    with pytest.raises(Alias):
        for seed in range(6):
            simulate(ua, ub, seed, paced_copier=False)
