"""CPU model of the mbarrier protocol of the streaming row-window kernel
(ts::wcsr_ts_kernel in csrc/wcsr.cu): preparing warps fill item slots, gathering
warps fill stage rings, MMA issuers consume stages and commit them back
(asynchronously, in issue order), epilogue warps drain accumulators.  Every role
is a sequence of parity waits and arrivals, run under random interleavings.

The model checks two things the kernel relies on: no interleaving deadlocks, and
every MMA reads the fill of its own step (a parity wait cannot tell fill k from
fill k + 2, so a party that can run two phases ahead reads stale data).  It
shows why the kernel keeps one stage ring per issuer with a single filling warp
per stage: with a ring shared by two issuers, or with two filling warps per
stage, the model finds stale reads or deadlocks."""
import random

import pytest

SLOTS, GATHER, EPI, PREP = 8, 8, 4, 8


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):  # the phase with this parity has completed
        return (self.phase & 1) != parity


def run(nks, issuers, stages, per_issuer_rings, seed):
    """Returns (deadlocked, stale_reads) for one interleaving of the protocol."""
    rnd = random.Random(seed)
    rings = issuers if per_issuer_rings else 1
    ring = stages // rings
    acc = 2 * issuers
    item_full = [Bar(1) for _ in range(SLOTS)]
    item_empty = [Bar(GATHER + issuers + EPI) for _ in range(SLOTS)]
    stage_full = [[Bar(1) for _ in range(ring)] for _ in range(rings)]
    stage_empty = [[Bar(1) for _ in range(ring)] for _ in range(rings)]
    content = [[None] * ring for _ in range(rings)]
    acc_full = [Bar(1) for _ in range(acc)]
    acc_empty = [Bar(EPI) for _ in range(acc)]
    recs = [None] * SLOTS
    pending = []  # asynchronous commits: (issuer, barrier), delivered in issue order per issuer
    stale = []
    n = len(nks)

    def prep(w):
        for ic in range(w, n, PREP):
            yield item_empty[ic % SLOTS], ((ic // SLOTS) & 1) ^ 1
            recs[ic % SLOTS] = nks[ic]
            item_full[ic % SLOTS].arrive()

    def gather(g):
        t = [0] * rings  # steps of earlier items, per ring
        for ic in range(n):
            yield item_full[ic % SLOTS], (ic // SLOTS) & 1
            nk, r = recs[ic % SLOTS], (ic % issuers if per_issuer_rings else 0)
            for k in range((g - t[r] % GATHER + GATHER) % GATHER, nk, GATHER):
                step = t[r] + k
                yield stage_empty[r][step % ring], ((step // ring) & 1) ^ 1
                content[r][step % ring] = (ic, k)
                stage_full[r][step % ring].arrive()
            t[r] += nk
            item_empty[ic % SLOTS].arrive()

    def issuer(j):
        t = 0  # this issuer's steps through its ring (shared ring: all steps)
        for ic in range(n):
            yield item_full[ic % SLOTS], (ic // SLOTS) & 1
            nk = recs[ic % SLOTS]
            r = j if per_issuer_rings else 0
            if ic % issuers != j:
                if not per_issuer_rings:
                    t += nk
                item_empty[ic % SLOTS].arrive()
                continue
            b = ic % acc
            yield acc_empty[b], ((ic // acc) & 1) ^ 1
            for k in range(nk):
                step = t + k
                yield stage_full[r][step % ring], (step // ring) & 1
                if content[r][step % ring] != (ic, k):
                    stale.append((ic, k))
                pending.append((j, stage_empty[r][step % ring]))
            t += nk
            pending.append((j, acc_full[b]))
            item_empty[ic % SLOTS].arrive()

    def epilogue(_):
        for ic in range(n):
            yield item_full[ic % SLOTS], (ic // SLOTS) & 1
            yield acc_full[ic % acc], (ic // acc) & 1
            acc_empty[ic % acc].arrive()
            item_empty[ic % SLOTS].arrive()

    roles = ([prep(w) for w in range(PREP)] + [gather(g) for g in range(GATHER)] +
             [issuer(j) for j in range(issuers)] + [epilogue(e) for e in range(EPI)])
    waits = [next(r, None) for r in roles]
    while True:
        ready = [i for i, w in enumerate(waits) if w is not None and w[0].done(w[1])]
        heads = {}
        for idx, (j, _) in enumerate(pending):
            heads.setdefault(j, idx)
        choices = [("role", i) for i in ready] + [("commit", idx) for idx in heads.values()]
        if not choices:
            return any(w is not None for w in waits), stale
        kind, x = rnd.choice(choices)
        if kind == "commit":
            pending.pop(x)[1].arrive()
        else:
            waits[x] = next(roles[x], None)


def _sequences(count):
    r = random.Random(7)
    for seed in range(count):
        yield seed, [r.choice([0, 1, 2, 3, 5, 8, 16, 31, 32]) for _ in range(r.randint(1, 40))]


@pytest.mark.parametrize("issuers,stages", [(1, 16), (2, 16)])
def test_per_issuer_rings_neither_deadlock_nor_read_stale_stages(issuers, stages):
    """The kernel's layout: 16 stages, one ring per issuer, ring length a multiple of
    the eight gathering warps (so each stage has a single filling warp)."""
    for seed, nks in _sequences(150):
        deadlocked, stale = run(nks, issuers, stages, True, seed)
        assert not deadlocked and not stale, (seed, nks)


def test_a_ring_shared_by_two_issuers_fails():
    """Two issuers skipping each other's steps on one ring: an issuer can pass a
    stage's parity wait two fills early."""
    bad = sum(any(run(nks, 2, 16, False, seed)) for seed, nks in _sequences(60))
    assert bad > 0


def test_two_filling_warps_per_stage_fail():
    """Four issuers with 4-stage rings: stage s is filled by gathering warps s and
    s + 4, which can run two fills apart."""
    bad = sum(any(run(nks, 4, 16, True, seed)) for seed, nks in _sequences(60))
    assert bad > 0
