"""Model check of the band kernel's K/V ring protocol (CPU only).

The band kernel streams a CTA's key/value tiles through a ring of NSLOT shared-memory
slots: fill 2j is K_j, fill 2j+1 is V_j (j counts the CTA's key tiles over all its units).
Each slot has a "full" mbarrier (completed when its copy lands) and an "empty" mbarrier
(completed when its tiles' last reader is done); an mbarrier wait names only the parity
of the phase it waits for.  This test drives the protocol's agents in random orders:
  * the producer warp, which issues fills once their slot is free;
  * the tensor-memory copies (TMA), which land in any order after issue;
  * the MMA-issuing thread, in the order the kernel issues S and P V;
  * the release arrivals (commits, or softmax warpgroup B).
At every wait that succeeds it checks that the barrier has completed exactly the phase
the waiter counts (one more would alias on parity), that the parity function the kernel
uses gives that phase's parity, and that the run ends without deadlock.  Every MMA
checks that the tiles it reads have landed and are still in their slots, and every
fill checks that its slot's previous tile has been read by all its readers.

Five build flavours are covered:
  two query tiles    paired fills + key releases from softmax B   (no global positions)
  two query tiles    one barrier per fill + key releases          (globals, short bands)
  two query tiles    one barrier per fill + a release per fill    (globals, long bands)
  one query tile     paired fills + value releases                (no global positions)
  one query tile     one barrier per fill + value releases        (globals)
A model of the protocol, not of the kernel's code: the parity functions below restate the
kernel's arithmetic so that a change to the ordering has to be reflected here as well."""
import copy
import random

import pytest


# -- phase ordinals (how many earlier completions a slot's barrier has had) --------------
def key_ord(p, ns):
    """ordinal of key fill p's release when only key fills release (odd ring: a slot
    alternates key and value fills; even ring: a slot holds key fills only)"""
    s, i = p % ns, p // ns
    return (i - (s & 1)) // 2 if ns % 2 else i


def val_ord(p, ns):
    """ordinal of value fill p's release when only value fills release (odd ring)"""
    s, i = p % ns, p // ns
    return (i - ((1 + s) & 1)) // 2


def own_ord(q, ns):
    """ordinal of owner fill q's full-barrier completion with paired fills: owners are the
    key fills (and the CTA's last value fill, which has none after it)"""
    s, i = q % ns, q // ns
    if ns % 2:
        return (i - (s & 1) + 1) // 2
    return i if s % 2 == 0 else 0


# -- the kernel's parity functions -----------------------------------------------------
def kpar(p, ns):
    sl, i = p % ns, p // ns
    return ((i - (sl & 1)) // 2 if ns % 2 == 1 else i) & 1


def vpar(p, ns):
    sl, i = p % ns, p // ns
    return ((i - ((1 + sl) & 1)) // 2) & 1


def fpar(q, ns):
    sl, i = q % ns, q // ns
    n = (i - (sl & 1) + 1) // 2 if ns % 2 == 1 else (i if sl % 2 == 0 else 0)
    return n & 1


class Barrier:
    def __init__(self):
        self.done = 0

    def check_wait(self, n, parity):
        """True once phase n has completed; asserts it is the newest completed phase and
        that the waiter's parity names it"""
        if self.done <= n:
            return False
        assert self.done == n + 1, f"phase aliasing: waiting for {n}, {self.done} done"
        assert parity == (n & 1), f"parity {parity} for phase {n}"
        return True


class Ring:
    def __init__(self, units, ns, nqt, paired, release, rng):
        assert release in ("key", "value", "all")
        assert not (release == "value" and ns % 2 == 0)
        self.units, self.ns, self.nqt, self.paired, self.release, self.rng = units, ns, nqt, paired, release, rng
        self.tiles = sum(units)
        self.nfill = 2 * self.tiles
        self.full = [Barrier() for _ in range(ns)]
        self.empty = [Barrier() for _ in range(ns)]
        self.inflight = []      # copies issued, not landed: (fill, owner fill of its barrier)
        self.arm = {}           # owner fill -> copies still to land on its barrier
        self.g = 0              # next fill to issue (paired: next owner step)
        self.releases = []      # pending release arrivals, in issue order: fill
        self.landed = set()     # fills whose copy has landed
        self.occupant = {}      # slot -> last fill issued into it
        self.reads = {}         # fill -> MMAs that have read it
        self.readers = 2 if nqt == 2 else 1  # S_A, S_B (or P V_A, P V_B); one S or P V
        self.ops = self._mma_ops()
        self.i = 0

    # ---- the orders the kernel issues its MMAs in
    def _mma_ops(self):
        ops, J = [], 0
        for n in self.units:
            if self.nqt == 2:
                ops += [("S", J, "A"), ("S", J, "B")]
                if self.release in ("key", "all"):
                    ops.append(("rel", 2 * J))
                for j in range(n):
                    jg = J + j
                    ops.append(("PV", jg, "A"))
                    if j + 1 < n:
                        ops.append(("S", jg + 1, "A"))
                    ops.append(("PV", jg, "B"))
                    if self.release == "all":
                        ops.append(("rel", 2 * jg + 1))
                    if j + 1 < n:
                        ops.append(("S", jg + 1, "B"))
                        if self.release in ("key", "all"):
                            ops.append(("rel", 2 * jg + 2))
            else:
                ops.append(("S", J, "A"))
                for j in range(n):
                    jg = J + j
                    if j + 1 < n:
                        ops.append(("S", jg + 1, "A"))
                    ops.append(("PV", jg, "last" if j + 1 == n else "mid"))
                    ops.append(("rel", 2 * jg + 1))
            J += n
        return ops

    def owner(self, p):
        if not self.paired or p % 2 == 0:
            return p
        return p + 1 if p + 1 < self.nfill else p

    # ---- full-barrier waits on the MMA side, as the kernel makes them
    def wait_full(self, p):
        ns = self.ns
        if self.paired:
            q = self.owner(p)
            return self.full[q % ns].check_wait(own_ord(q, ns), fpar(q, ns))
        return self.full[p % ns].check_wait(p // ns, (p // ns) & 1)

    def mma_needs(self, op):
        kind, jg, who = op
        if kind == "S":
            if not self.paired:
                return [] if (self.nqt == 2 and who == "B") else [2 * jg]
            if self.nqt == 2:
                return [2 * jg] if (who == "A" and jg == 0) else []
            return [2 * jg]
        if kind == "PV":
            if not self.paired:
                return [2 * jg + 1] if who in ("A", "mid", "last") else []
            if self.nqt == 2:
                return [2 * jg + 1] if who == "A" else []
            return [2 * jg + 1] if who == "last" else []
        return []

    def issue(self, p):
        prev = self.occupant.get(p % self.ns)
        if prev is not None:
            assert self.reads.get(prev, 0) == self.readers, f"fill {p} overwrites {prev} before it is read"
        self.occupant[p % self.ns] = p

    # ---- producer side: is fill p's slot free?
    def slot_free(self, p):
        ns = self.ns
        if p < ns:
            return True
        prev = p - ns
        if self.release == "all":
            return self.empty[p % ns].check_wait(prev // ns, ((p // ns) - 1) & 1)
        if self.release == "key":
            kp = prev + 1 if prev & 1 else prev
            return self.empty[kp % ns].check_wait(key_ord(kp, ns), kpar(kp, ns))
        vp = prev if prev & 1 else prev + 1
        return self.empty[vp % ns].check_wait(val_ord(vp, ns), vpar(vp, ns))

    def producer_step(self):
        ns = self.ns
        if not self.paired:
            p = self.g
            if p >= self.nfill or not self.slot_free(p):
                return False
            self.issue(p)
            self.arm[p] = 1
            self.inflight.append((p, p))
            self.g += 1
            return True
        if self.g == 0:
            if self.nfill == 0:
                return False
            self.issue(0)
            self.arm[0] = 1
            self.inflight.append((0, 0))
            self.g = 1
            return True
        pv = self.g
        if pv >= self.nfill:
            return False
        own = self.owner(pv)
        if not (self.slot_free(pv) and (own == pv or self.slot_free(own))):
            return False
        self.issue(pv)
        if own != pv:
            self.issue(own)
        self.arm[own] = 2 if own != pv else 1
        self.inflight += [(pv, own)] + ([(own, own)] if own != pv else [])
        self.g = own + 1
        return True

    def land_one(self):
        if not self.inflight:
            return False
        k = self.rng.randrange(len(self.inflight))
        p, own = self.inflight.pop(k)
        self.landed.add(p)
        self.arm[own] -= 1
        if self.arm[own] == 0:
            bar = self.full[own % self.ns]
            expect = own_ord(own, self.ns) if self.paired else own // self.ns
            assert bar.done == expect, f"fill {own}: barrier at {bar.done}, expected {expect}"
            bar.done += 1
        return True

    def release_one(self):
        if not self.releases:
            return False
        p = self.releases.pop(0)
        ns = self.ns
        expect = {"all": p // ns, "key": key_ord(p, ns), "value": val_ord(p, ns)}[self.release]
        assert self.empty[p % ns].done == expect, f"release of {p}"
        self.empty[p % ns].done += 1
        return True

    def mma_step(self):
        if self.i >= len(self.ops):
            return False
        op = self.ops[self.i]
        if op[0] == "rel":
            self.releases.append(op[1])
        elif not all(self.wait_full(p) for p in self.mma_needs(op)):
            return False
        else:
            p = 2 * op[1] + (1 if op[0] == "PV" else 0)  # the K or V tile this MMA reads
            assert p in self.landed, f"{op} reads fill {p} before it lands"
            assert self.occupant.get(p % self.ns) == p, f"{op} reads fill {p} after its slot was refilled"
            self.reads[p] = self.reads.get(p, 0) + 1
        self.i += 1
        return True

    def run(self, drain_checks=0.0, drain_back=None):
        """drain_checks: probability, per scheduling round, of checking the exit-path drain
        as if the producer stopped there (drain_back: how many fills back it looks)."""
        agents = [self.producer_step, self.land_one, self.release_one, self.mma_step]
        while self.i < len(self.ops) or self.g < self.nfill or self.inflight or self.releases:
            if drain_checks and self.rng.random() < drain_checks:
                self.check_drain(drain_back)
            order = agents[:]
            self.rng.shuffle(order)
            if not any(a() for a in order):
                raise AssertionError(f"deadlock: units={self.units} ns={self.ns} g={self.g} op={self.ops[self.i]}")
        assert all(v == 0 for v in self.arm.values())

    # ---- exit path: the producer stops after issuing fills 0 .. g-1
    def drain_set(self, back):
        """The barriers the kernel's producer drains: owners among fills g-back .. g-1
        (paired: key fills and the CTA's last fill), each with the parity of that fill."""
        lo = max(0, self.g - back)
        if self.paired:
            return [q for q in range(lo, self.g) if q % 2 == 0 or q + 1 == self.nfill]
        return list(range(lo, self.g))

    def check_drain(self, back=None):
        """Every copy still in flight must be covered by the drain, and once they have all
        landed each drain wait must name the newest completed phase of its barrier (an
        older one would alias on parity and wait until its time limit)."""
        ns = self.ns
        back = ns if back is None else back
        d = self.drain_set(back)
        missing = {own for _, own in self.inflight} - set(d)
        assert not missing, f"copies on barriers of fills {sorted(missing)} in flight, not drained (g={self.g})"
        sim = copy.deepcopy(self)
        while sim.land_one():
            pass
        for q in d:
            if sim.paired:
                ok = sim.full[q % ns].check_wait(own_ord(q, ns), fpar(q, ns))
            else:
                ok = sim.full[q % ns].check_wait(q // ns, (q // ns) & 1)
            assert ok, f"drain of fill {q} names a phase that never completes"


FLAVOURS = [
    # (query tiles, paired fills, releases, ring sizes)
    (2, True, "key", (3, 4, 5, 6, 12)),
    (2, False, "key", (3, 4, 5, 6, 12)),
    (2, False, "all", (3, 4, 5, 6, 12)),
    (2, True, "all", (3, 4, 5, 6, 12)),
    (1, True, "value", (3, 5, 7)),
    (1, False, "value", (3, 5, 7)),
]


@pytest.mark.parametrize("nqt,paired,release,rings", FLAVOURS)
def test_ring_protocol(nqt, paired, release, rings):
    rng = random.Random(1234 + 10 * nqt + (1 if paired else 0))
    mixes = [[1], [2], [1, 1], [1, 1, 1], [33, 33], [6, 7, 5], [18, 18]]
    mixes += [[rng.randint(1, 40) for _ in range(rng.randint(1, 5))] for _ in range(150)]
    for ns in rings:
        for units in mixes:
            Ring(units, ns, nqt, paired, release, rng).run()


def test_parity_functions_match_ordinals():
    for ns in (3, 4, 5, 6, 7, 12):
        for p in range(0, 40 * ns, 2):
            assert kpar(p, ns) == key_ord(p, ns) & 1
            assert fpar(p, ns) == own_ord(p, ns) & 1
        if ns % 2:
            for p in range(1, 40 * ns, 2):
                assert vpar(p, ns) == val_ord(p, ns) & 1


def test_model_catches_a_wrong_parity():
    """the model itself must reject a protocol error: an owner ordinal off by one"""
    global own_ord
    saved = own_ord
    try:
        own_ord = lambda q, ns: saved(q, ns) + (1 if q >= ns else 0)  # noqa: E731
        with pytest.raises(AssertionError):
            Ring([6, 7, 5], 5, 2, True, "key", random.Random(0)).run()
    finally:
        own_ord = saved


def test_model_catches_an_early_release():
    """and a data race: releasing K_{j+1}'s slot before P V_B(j), the last reader of V_j
    (which shares the key release in that build), lets the producer overwrite V_j"""
    class Early(Ring):
        def _mma_ops(self):
            out = []
            for op in super()._mma_ops():
                pvb = ("PV", op[1] // 2 - 1, "B")
                if op[0] == "rel" and pvb in out:
                    out.insert(out.index(pvb), op)  # ahead of P V_B(j)
                else:
                    out.append(op)
            return out

    caught = 0
    for seed in range(40):
        try:
            Early([12, 9, 14], 5, 2, True, "key", random.Random(seed)).run()
        except AssertionError as e:
            assert "overwrites" in str(e), e
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("nqt,paired,release,rings", FLAVOURS)
def test_drain_after_a_stop(nqt, paired, release, rings):
    """The exit path of the producer (a bounded wait gave up elsewhere, or a planted stop):
    at random points of random runs, the fills g-NSLOT .. g-1 hold every copy in flight,
    one per slot, and draining them names each barrier's newest phase."""
    rng = random.Random(4321 + 10 * nqt + (1 if paired else 0))
    mixes = [[1], [2, 3], [6, 7, 5], [18, 18]] + [[rng.randint(1, 30) for _ in range(rng.randint(1, 4))]
                                                    for _ in range(25)]
    for ns in rings:
        for units in mixes:
            Ring(units, ns, nqt, paired, release, rng).run(drain_checks=0.05)


def test_model_catches_a_drain_window_one_fill_too_long():
    """Looking NSLOT + 1 fills back, an even ring drains two key fills of one slot: the
    older one's parity names a phase that has been overtaken (a false drain timeout)."""
    caught = 0
    for seed in range(20):
        try:
            Ring([18, 18], 12, 2, True, "key", random.Random(seed)).run(drain_checks=0.2, drain_back=13)
        except AssertionError as e:
            assert "aliasing" in str(e) or "never completes" in str(e), e
            caught += 1
    assert caught > 0
