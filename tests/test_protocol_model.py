"""A model check of two synchronization protocols of the expert kernel, on the CPU.

Each protocol is played out over many random interleavings with the semantics of an mbarrier
parity wait: a barrier counts its completed phases k, and a wait for the phase of parity P
passes while k % 2 != P.  Such a wait is exact only while the barrier is at most one phase
behind the waiter, which is what each protocol has to guarantee.  The checks assert that no
wait passes on the wrong phase in the configurations the kernel uses, and that the model does
find the failure when the safeguard is taken away, so that it is able to see one.

1. The ring of shared-memory slots with two MMA issuers.  The producer copies blocks 0, 1, ...
   into slot b % S after the slot's previous block was consumed (its `empty` barrier); the
   down blocks come in units that alternate between two issuers, each consuming its own blocks
   in order after the slot's `full` barrier.  An issuer skips the other's blocks, so it can
   reach block b while the copy of block b - S is not even issued; the slot's full barrier is
   then a whole phase behind and the parity wait passes at once.  The kernel's safeguard: the
   producer records in shared memory which block it copies into each slot, and an issuer waits
   for its block's record before the parity wait.

2. The ring of h entries.  Runs 0, 1, ... are formed by W_r of the H h-former warps (a leader
   and the next W_r - 1), each of which first waits for the entry's release by the run R
   entries before (`h_empty`), and consumed in order (`h_full`); releases complete in run
   order.  A warp's wait is exact once run r - 2R is released.  Any H consecutive runs give
   every warp a part, so with R >= H a warp's own last wait tells it so.  With R < H the
   kernel keeps a shared count of the runs seen released and waits for it first; waiting for
   every run's entry in order, also for the runs a warp skips, can deadlock (a skipping warp
   falls two phases behind an entry that other warps keep releasing).

3. The down accumulators with two issuers: units alternate between the issuers and cycle
   through B accumulators; the epilogue reads them in order.
"""
import numpy as np
import pytest


class Barrier:
    """Phase counting of an mbarrier: `count` arrivals complete a phase."""

    def __init__(self, count=1):
        self.count, self.k, self.arrived = count, 0, 0

    def passes(self, parity):
        return self.k % 2 != parity

    def arrive(self, n=1):
        self.arrived += n
        assert self.arrived <= self.count
        if self.arrived == self.count:
            self.k += 1
            self.arrived = 0


def ring_run(rng, S, units, records, slow_issuer):
    """One random interleaving of the two-issuer ring.  Returns the first violation (a block
    consumed from a slot that does not hold it), or None."""
    owner = []
    for u, size in enumerate(units):
        owner += [u % 2] * size
    B = len(owner)
    full = [Barrier() for _ in range(S)]
    empty = [Barrier() for _ in range(S)]
    content = [None] * S       # block in each slot once its copy landed
    rec = [-1] * S             # the producer's record of the block copied into each slot
    prod = 0                   # next block the producer copies
    landing, committing = [], []   # copies in flight, MMAs in flight (slot, block)
    mine = [[b for b in range(B) if owner[b] == i] for i in range(2)]
    pos = [0, 0]               # next block of each issuer
    while True:
        acts = []
        if prod < B and empty[prod % S].passes(((prod // S) & 1) ^ 1):
            acts.append("produce")
        if landing:
            acts.append("land")
        if committing:
            acts.append("commit")
        for i in (0, 1):
            if pos[i] < len(mine[i]):
                b = mine[i][pos[i]]
                s = b % S
                if (not records or rec[s] == b) and full[s].passes((b // S) & 1):
                    acts += [("consume", i)] * (1 if i == slow_issuer else 3)
        if not acts:
            assert prod == B and all(p == len(m) for p, m in zip(pos, mine))
            return None
        a = acts[rng.integers(len(acts))]
        if a == "produce":
            s = prod % S
            rec[s] = prod
            landing.append((s, prod))
            prod += 1
        elif a == "land":
            s, b = landing.pop(rng.integers(len(landing)))
            content[s] = b
            full[s].arrive()
        elif a == "commit":
            s, b = committing.pop(rng.integers(len(committing)))
            empty[s].arrive()
        else:
            i = a[1]
            b = mine[i][pos[i]]
            s = b % S
            if content[s] != b:
                return (b, content[s])
            content[s] = None
            committing.append((s, b))
            pos[i] += 1


def ring_violations(records, trials=300, seed=1):
    rng = np.random.default_rng(seed)
    bad = 0
    for t in range(trials):
        S = int(rng.choice([6, 7, 8]))           # ring slots of the kernel's forms
        units = list(rng.integers(1, 5, size=int(rng.integers(6, 24))))   # units of 1-4 blocks
        if ring_run(rng, S, units, records, slow_issuer=t % 2) is not None:
            bad += 1
    return bad


def test_two_issuer_ring_is_exact_with_slot_records():
    assert ring_violations(records=True) == 0


def test_two_issuer_ring_without_records_fails_in_the_model():
    """The hazard that faulted the first two-issuer kernel: found in the model."""
    assert ring_violations(records=False) > 0


def hring_run(rng, R, H, widths, rotate, in_order, seen=False):
    """One random interleaving of the h ring.  Returns the first violation: a warp that passed
    an entry's release wait before the run R entries before was consumed, or a consumer that
    passed h_full before all of a run's arrivals; None if there is none."""
    n = len(widths)
    h_full = [Barrier(H) for _ in range(R)]
    h_empty = [Barrier(1) for _ in range(R)]
    consumed = [False] * n
    arrivals = [0] * n
    # the part of each warp in each run: its index from the leader, or None
    part = [[None] * n for _ in range(H)]
    lead = 0
    for r, W in enumerate(widths):
        leader = lead % H if rotate else r % H
        for w in range(H):
            k = (w - leader) % H
            part[w][r] = k if k < W else None
        lead += W
    pos = [0] * H       # next run each warp looks at
    hseen = 0           # seen mode: runs below this are known released (shared word)
    waited = [False] * H   # the warp passed the entry's wait for its current run
    cons = 0            # next run the consumer takes
    releasing = []      # consumed runs whose release is in flight, oldest first
    while True:
        acts = []
        for w in range(H):
            r = pos[w]
            if r >= n:
                continue
            e, ph = r % R, ((r // R) & 1) ^ 1
            if part[w][r] is None and (seen or not in_order):
                acts.append(("skip", w))
            elif not waited[w]:
                # seen mode: the parity wait only once run r - 2R is known released
                if (not seen or r < 2 * R or hseen >= r - 2 * R + 1) and h_empty[e].passes(ph):
                    acts.append(("wait", w))
            else:
                acts.append(("form", w))
        if cons < n and h_full[cons % R].passes((cons // R) & 1):
            acts.append(("consume", None))
        if releasing:
            acts.append(("release", None))
        if not acts:
            return None if cons == n else ("deadlock", cons)
        kind, w = acts[rng.integers(len(acts))]
        if kind == "skip":
            pos[w] += 1
        elif kind == "wait":
            r = pos[w]
            if r >= R and not consumed[r - R]:
                return ("entry reused early", w, r)
            waited[w] = True
            if seen and r >= R:
                hseen = max(hseen, r - R + 1)
        elif kind == "form":
            r = pos[w]
            waited[w] = False
            pos[w] += 1
            k = part[w][r]
            if k is None:        # a warp outside the run that waited in order
                continue
            W = widths[r]
            cnt = H - W + 1 if k == 0 else 1
            arrivals[r] += cnt
            h_full[r % R].arrive(cnt)
        elif kind == "consume":
            if arrivals[cons] != H:
                return ("consumed before formed", cons)
            consumed[cons] = True
            releasing.append(cons)
            cons += 1
        else:
            # releases complete in run order: every party (each issuer's commit, which covers
            # all its earlier MMAs, and each epilogue warp) arrives for the runs in order
            r = releasing.pop(0)
            h_empty[r % R].arrive()


def hring_violations(R, H, rotate, in_order, trials=300, seed=2, wmax=None, seen=False):
    rng = np.random.default_rng(seed)
    bad = 0
    for _ in range(trials):
        widths = list(rng.integers(1, (wmax or H) + 1, size=int(rng.integers(4, 30))))
        if hring_run(rng, R, H, widths, rotate, in_order, seen) is not None:
            bad += 1
    return bad


@pytest.mark.parametrize("rotate", [True, False])
def test_h_ring_with_as_many_entries_as_warps_is_exact(rotate):
    """R = H = 4 (the 16- and 32-token forms with 2-block units), leaders rotating by the
    warps each run takes or, as before, run r led by warp r mod 4."""
    assert hring_violations(4, 4, rotate, in_order=False) == 0


def test_h_ring_with_fewer_entries_uses_the_released_count():
    """R = 2 < H = 4 (the 64-token forms and the 32-token one with 4-block units): exact and
    deadlock-free with the shared count of released runs; with no safeguard the model finds
    the early pass the first 2-entry kernel faulted on, and with in-order waits on every
    run's entry it finds a deadlock."""
    for rotate in (True, False):
        assert hring_violations(2, 4, rotate, in_order=False, seen=True, trials=500) == 0
    assert hring_violations(2, 4, rotate=True, in_order=False) > 0
    assert hring_violations(2, 4, rotate=True, in_order=True) > 0


@pytest.mark.parametrize("R,H", [(1, 4), (3, 4), (4, 5), (2, 5)])
def test_h_ring_released_count_is_exact_for_any_ring(R, H):
    assert hring_violations(R, H, rotate=True, in_order=False, seen=True) == 0


def dacc_run(rng, B, units):
    """One random interleaving of the down accumulators with two issuers: unit u goes to issuer
    u % 2 and to accumulator u % B; an issuer waits for its accumulator's release by the unit B
    before (`dacc_empty`), fills it and commits `dacc_full`; the epilogue takes the units in
    order.  Returns the first violation (the epilogue reading an accumulator that does not hold
    its unit, or an issuer overwriting one the epilogue has not read), or None."""
    full = [Barrier() for _ in range(B)]
    empty = [Barrier() for _ in range(B)]
    content = [None] * B
    read = [False] * units
    mine = [[u for u in range(units) if u % 2 == i] for i in range(2)]
    pos = [0, 0]
    epi = 0
    filling = []        # MMAs in flight: (accumulator, unit)
    while True:
        acts = []
        for i in (0, 1):
            if pos[i] < len(mine[i]):
                u = mine[i][pos[i]]
                if empty[u % B].passes(((u // B) & 1) ^ 1):
                    acts.append(("issue", i))
        if filling:
            acts.append(("complete", None))
        if epi < units and full[epi % B].passes((epi // B) & 1):
            acts.append(("read", None))
        if not acts:
            return None if epi == units else ("deadlock", epi)
        kind, i = acts[rng.integers(len(acts))]
        if kind == "issue":
            u = mine[i][pos[i]]
            if u >= B and not read[u - B]:
                return ("overwrite", u)
            filling.append((u % B, u))
            pos[i] += 1
        elif kind == "complete":
            b, u = filling.pop(rng.integers(len(filling)))
            content[b] = u
            full[b].arrive()
        else:
            b = epi % B
            if content[b] != epi:
                return ("read", epi, content[b])
            read[epi] = True
            empty[b].arrive()
            epi += 1


def test_down_accumulators_with_two_issuers():
    """With an even number of accumulators (8 or 6 in the kernel, which requires an even count)
    each belongs to one issuer, whose waits on it follow each other phase by phase.  Odd counts
    from 3 are exact as well (an issuer's unit between two uses of an accumulator waits on
    another one, whose release by the in-order epilogue implies the earlier release), but a
    single accumulator shared by both issuers is not: the model finds an issuer overwriting a
    unit the epilogue has not read."""
    rng = np.random.default_rng(3)
    for B in (6, 8, 3, 5):
        assert all(dacc_run(rng, B, int(rng.integers(4, 60))) is None for _ in range(300))
    assert any(dacc_run(rng, 1, int(rng.integers(4, 30))) is not None for _ in range(300))
