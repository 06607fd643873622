"""Models of the attention kernels' hand-off protocols between their MMA issuers and their
element-wise (softmax) warps, run under random schedules to look for races.

Test infrastructure: it restates, in Python, the order of waits, products, commits and counter
updates of the tensor-core dQ and dK/dV kernels (csrc/attn_bwd_tc.cu) and of the forward
kernel (csrc/attn_tc.cu, one ring step) and checks the data those steps hand over.  Nothing here runs the kernels; item boundaries, epilogues and the K/V rings
are left out.

What is modelled:
- three 128-column tensor-memory slots in rotation (tile g: S in slot s(g), dP in slot d(g) =
  s(g - 1), S(g) overwriting the slot of dS(g - 2));
- each element-wise warp owns its own lanes of every slot: a product writes all lanes, a warp
  reads and writes its own, the dQ product reads all;
- an issuer's products run in its own order; products of two issuers interleave freely;
- `tcgen05.commit`: an arrival once every earlier product of that issuer has run;
- mbarrier waits with the hardware's parity test (a wait for completion k passes when the
  number of completed phases differs from k in parity - so it also passes two phases late);
- counters the warps add to (release) and issuers wait on (acquire).
A check fails when a warp or a product reads a slot whose lanes do not hold what it expects
(overwritten early or not yet written), or when the schedule deadlocks.
"""
import random


class Barrier:
    def __init__(self):
        self.done = 0  # completed phases

    def passes(self, k):
        """A parity wait for completion number k (0-based)."""
        return (self.done & 1) != (k & 1)


class Violation(Exception):
    pass


def s_slot(g):
    return (0, 2, 1)[g % 3]


def d_slot(g):
    return (1, 0, 2)[g % 3]


class Model:
    """variant: 'split' (warp 1: S and dP; warp 2: dQ) or 'rearranged' (warp 1: S and dQ;
    warp 2: dP); ds_by_parity / read_by_parity: the dS-stored (S-read) counts kept apart by
    tile parity instead of summed."""

    def __init__(self, variant, ds_by_parity, read_by_parity=False, warps=4, tiles=10, seed=0, slow=None):
        self.variant, self.nw, self.T = variant, warps, tiles
        self.ds_by_parity, self.read_by_parity = ds_by_parity, read_by_parity
        self.rng = random.Random(seed)
        self.slow = slow  # actor name scheduled rarely, to open lags
        self.tags = [[None] * warps for _ in range(3)]
        self.p0 = [0, 0]   # S read (by parity, or summed in [0])
        self.p1 = [0, 0]   # dS stored
        self.s_issued = 0
        self.bar = {n: Barrier() for n in ("s0", "s1", "d0", "d1", "q0", "q1")}
        self.fifo = {"w1": [], "w2": []}
        self.actors = {}

    # ---- counters
    def _add(self, ctr, by_parity, g):
        ctr[(g & 1) if by_parity else 0] += 1

    def _reached(self, ctr, by_parity, g):
        """Every warp has counted tile g (as far as the count can tell)."""
        if by_parity:
            return ctr[g & 1] >= self.nw * ((g >> 1) + 1)
        return ctr[0] >= self.nw * (g + 1)

    # ---- products
    def _write(self, slot, tag):
        self.tags[slot] = [tag] * self.nw

    def _read_all(self, slot, tag, what):
        if any(t != tag for t in self.tags[slot]):
            raise Violation(f"{what}: slot {slot} holds {self.tags[slot]}, expected {tag}")

    def _read_own(self, slot, w, tag, what):
        if self.tags[slot][w] != tag:
            raise Violation(f"{what}: warp {w} finds {self.tags[slot][w]} in slot {slot}, expected {tag}")

    # ---- programs (generators yielding a wait predicate, or None for one step)
    def w1_split(self):
        for g in range(self.T):
            if g >= 2:
                k = (g - 2) >> 1
                yield lambda g=g, k=k: self.bar[f"q{g & 1}"].passes(k)
            self.fifo["w1"].append(("mma", lambda g=g: self._write(s_slot(g), ("S", g))))
            yield None
            if g > 0:
                yield lambda g=g: self._reached(self.p0, self.read_by_parity, g - 1)
            self.fifo["w1"].append(("mma", lambda g=g: self._write(d_slot(g), ("dP", g))))
            self.fifo["w1"].append(("commit", "s0"))
            yield None

    def w2_split(self):
        for g in range(self.T):
            yield lambda g=g: self._reached(self.p1, self.ds_by_parity, g)
            self.fifo["w2"].append(("mma", lambda g=g: self._read_all(d_slot(g), ("dS", g), f"dQ({g})")))
            self.fifo["w2"].append(("commit", f"q{g & 1}"))
            yield None

    def w1_rearranged(self):
        for g in range(self.T + 1):
            if g < self.T:
                self.fifo["w1"].append(("mma", lambda g=g: self._write(s_slot(g), ("S", g))))
                self.fifo["w1"].append(("commit", f"s{g & 1}"))
                yield None
                self.s_issued += 1
                yield None
            if g >= 1:  # dQ(g - 1) once every warp stored its dS
                yield lambda g=g: self._reached(self.p1, self.ds_by_parity, g - 1)
                self.fifo["w1"].append(("mma", lambda g=g: self._read_all(d_slot(g - 1), ("dS", g - 1),
                                                                           f"dQ({g - 1})")))
                yield None

    def w2_rearranged(self):
        for g in range(self.T):
            if g > 0:
                yield lambda g=g: self._reached(self.p0, self.read_by_parity, g - 1)
            yield lambda g=g: self.s_issued >= g + 1
            self.fifo["w2"].append(("mma", lambda g=g: self._write(d_slot(g), ("dP", g))))
            self.fifo["w2"].append(("commit", f"d{g & 1}"))
            yield None

    def ew(self, w):
        for g in range(self.T):
            if self.variant == "split":
                yield lambda g=g: self.bar["s0"].passes(g)  # S(g) and dP(g)
            else:
                yield lambda g=g: self.bar[f"s{g & 1}"].passes(g >> 1)
            self._read_own(s_slot(g), w, ("S", g), f"warp {w} S({g})")
            yield None
            self._add(self.p0, self.read_by_parity, g)
            yield None
            if self.variant != "split":
                yield lambda g=g: self.bar[f"d{g & 1}"].passes(g >> 1)
            self._read_own(d_slot(g), w, ("dP", g), f"warp {w} dP({g})")
            yield None
            self.tags[d_slot(g)][w] = ("dS", g)
            yield None
            self._add(self.p1, self.ds_by_parity, g)
            yield None

    def pipe(self, who):
        while True:
            if not self.fifo[who]:
                yield lambda: bool(self.fifo[who]) or self._issuer_done(who)
                if not self.fifo[who]:
                    return
            kind, x = self.fifo[who].pop(0)
            if kind == "mma":
                x()
            else:
                self.bar[x].done += 1
            yield None

    def _issuer_done(self, who):
        return self.actors.get(who) is None

    def run(self):
        if self.variant == "split":
            self.actors["w1"], self.actors["w2"] = self.w1_split(), self.w2_split()
        else:
            self.actors["w1"], self.actors["w2"] = self.w1_rearranged(), self.w2_rearranged()
        for w in range(self.nw):
            self.actors[f"ew{w}"] = self.ew(w)
        self.actors["pipe1"], self.actors["pipe2"] = self.pipe("w1"), self.pipe("w2")
        return self._schedule()

    def _schedule(self):
        """Runs the actors to the end, one step of a random ready actor at a time."""
        waiting = {n: None for n in self.actors}
        while any(a is not None for a in self.actors.values()):
            ready = [n for n, a in self.actors.items() if a is not None and (waiting[n] is None or waiting[n]())]
            if not ready:
                raise Violation("deadlock: " + ", ".join(n for n, a in self.actors.items() if a is not None))
            if self.slow in ready and len(ready) > 1 and self.rng.random() < 0.9:
                ready.remove(self.slow)
            name = self.rng.choice(ready)
            try:
                waiting[name] = next(self.actors[name])
            except StopIteration:
                self.actors[name] = None
                waiting[name] = None
        return True


def find_violation(variant, ds_by_parity, read_by_parity=False, runs=300, tiles=10, warps=4):
    """The first violation over `runs` random schedules (half of them with one slow warp), or None."""
    for seed in range(runs):
        slow = "ew0" if seed % 2 else None
        try:
            Model(variant, ds_by_parity, read_by_parity, warps=warps, tiles=tiles, seed=seed, slow=slow).run()
        except Violation as e:
            return f"seed {seed}: {e}"
    return None


class DkdvModel(Model):
    """The dK/dV kernel's protocol: one issuer; slot 0 holds S^T(t) and then the P^T(t) the
    warps write over it (read by dV(t)), slot 1 dP^T(t) and then dS^T(t) (read by dK(t)).
    Product order dV(t), S^T(t + 1), dK(t), dP^T(t + 1); swap_order=True puts S^T(t + 1)
    before dV(t) (a planted mistake: it overwrites P^T(t) before dV(t) reads it)."""

    def __init__(self, swap_order=False, warps=4, tiles=10, seed=0, slow=None):
        super().__init__("dkdv", ds_by_parity=False, warps=warps, tiles=tiles, seed=seed, slow=slow)
        self.tags = [[None] * warps for _ in range(2)]
        self.swap = swap_order

    def issuer(self):
        f = self.fifo["w1"]
        f.append(("mma", lambda: self._write(0, ("S", 0))))
        f.append(("commit", "s0"))
        f.append(("mma", lambda: self._write(1, ("dP", 0))))
        f.append(("commit", "s1"))
        yield None
        for t in range(self.T):
            nxt = t + 1 < self.T
            if self.swap and nxt:
                f.append(("mma", lambda t=t: self._write(0, ("S", t + 1))))
                f.append(("commit", "s0"))
            yield lambda t=t: self._reached(self.p0, False, t)
            f.append(("mma", lambda t=t: self._read_all(0, ("P", t), f"dV({t})")))
            if nxt and not self.swap:
                f.append(("mma", lambda t=t: self._write(0, ("S", t + 1))))
                f.append(("commit", "s0"))
            yield None
            yield lambda t=t: self._reached(self.p1, False, t)
            f.append(("mma", lambda t=t: self._read_all(1, ("dS", t), f"dK({t})")))
            if nxt:
                f.append(("mma", lambda t=t: self._write(1, ("dP", t + 1))))
                f.append(("commit", "s1"))
            yield None

    def ew(self, w):
        for t in range(self.T):
            yield lambda t=t: self.bar["s0"].passes(t)
            self._read_own(0, w, ("S", t), f"warp {w} S^T({t})")
            yield None
            self.tags[0][w] = ("P", t)
            yield None
            self._add(self.p0, False, t)
            yield lambda t=t: self.bar["s1"].passes(t)
            self._read_own(1, w, ("dP", t), f"warp {w} dP^T({t})")
            yield None
            self.tags[1][w] = ("dS", t)
            yield None
            self._add(self.p1, False, t)
            yield None

    def run(self):
        self.actors["w1"] = self.issuer()
        for w in range(self.nw):
            self.actors[f"ew{w}"] = self.ew(w)
        self.actors["pipe1"] = self.pipe("w1")
        return self._schedule()


def find_violation_dkdv(swap_order=False, runs=300, tiles=10, warps=4):
    """As find_violation, for the dK/dV kernel's protocol."""
    for seed in range(runs):
        try:
            DkdvModel(swap_order, warps=warps, tiles=tiles, seed=seed, slow="ew0" if seed % 2 else None).run()
        except Violation as e:
            return f"seed {seed}: {e}"
    return None


class ForwardModel(Model):
    """The forward kernel's protocol for one item (kernel mode 0): two halves of query rows,
    each with an S slot (P written over it) and an O accumulator in tensor memory; a ring of
    two shared-memory stages, stage 0 = K_0 and stage s + 1 = (V_s, K_s+1), refilled by the
    producer once the MMA thread releases them; half 0 sits out tile 0 and takes its S signal
    from the stage release, half 1 from its own barrier; the softmax warps count P stored per
    half and may rescale O (read and write it) before they do.  pv_late=True issues each
    half's next QK^T before its P V (a planted mistake: it overwrites P before P V reads it)."""

    def __init__(self, pv_late=False, warps=2, tiles=10, seed=0, slow=None):
        super().__init__("fwd", ds_by_parity=False, warps=warps, tiles=tiles, seed=seed, slow=slow)
        self.S = [[None] * warps for _ in range(2)]   # per half, per warp's lanes
        self.O = [[None] * warps for _ in range(2)]
        self.stage = [None, None]                     # shared-memory slot -> stage it holds
        self.pc = [0, 0]
        self.bar = {n: Barrier() for n in ("full0", "full1", "empty0", "empty1", "s1", "o0", "o1")}
        self.pv_late = pv_late

    def part(self, h, t):
        return h == 1 or t >= 1

    def producer(self):
        for s in range(self.T + 1):
            if s >= 2:
                yield lambda s=s: self.bar[f"empty{s % 2}"].passes((s - 2) // 2)
            self.stage[s % 2] = s
            yield None
            self.bar[f"full{s % 2}"].done += 1
            yield None

    def _stage_holds(self, s, what):
        if self.stage[s % 2] != s:
            raise Violation(f"{what}: stage slot {s % 2} holds stage {self.stage[s % 2]}, expected {s}")

    def _qk(self, h, t, s):
        def run():
            self._stage_holds(s, f"QK_{h}({t})")
            self.S[h] = [("S", t)] * self.nw
        return run

    def _pv(self, h, t, s):
        def run():
            self._stage_holds(s, f"PV_{h}({t})")
            if any(x != ("P", t) for x in self.S[h]):
                raise Violation(f"PV_{h}({t}): S slot of half {h} holds {self.S[h]}")
            prev = ("O", t - 1) if t > (0 if h == 1 else 1) else None
            if any(x != prev for x in self.O[h]):
                raise Violation(f"PV_{h}({t}): O of half {h} holds {self.O[h]}, expected {prev}")
            self.O[h] = [("O", t)] * self.nw
        return run

    def mma(self):
        f = self.fifo["w1"]
        yield lambda: self.bar["full0"].passes(0)
        f.append(("mma", self._qk(1, 0, 0)))     # half 0 sits out tile 0
        f.append(("commit", "s1"))
        f.append(("commit", "empty0"))
        yield None
        for t in range(self.T):
            s = t + 1  # stage (V_t, K_t+1)
            yield lambda s=s: self.bar[f"full{s % 2}"].passes(s // 2)
            for h in (1, 0):
                nxt = t + 1 < self.T
                if self.pv_late and nxt:
                    f.append(("mma", self._qk(h, t + 1, s)))
                if self.part(h, t):
                    self.pc[h] += 1
                    yield lambda h=h, k=self.pc[h]: self.p1[h] >= self.nw * k
                    f.append(("mma", self._pv(h, t, s)))
                    if t == self.T - 1:
                        f.append(("commit", f"o{h}"))
                if nxt and not self.pv_late:
                    f.append(("mma", self._qk(h, t + 1, s)))
                if nxt and h == 1:
                    f.append(("commit", "s1"))
                yield None
            f.append(("commit", f"empty{s % 2}"))
            yield None

    def softmax(self, h, w):
        scnt = 0
        for t in range(self.T):
            if not self.part(h, t):
                continue
            if h == 0:
                yield lambda t=t: self.bar[f"empty{t % 2}"].passes(t // 2)  # release of the stage of QK_0(t)
            else:
                yield lambda k=scnt: self.bar["s1"].passes(k)
                scnt += 1
            if self.S[h][w] != ("S", t):
                raise Violation(f"half {h} warp {w} S({t}): finds {self.S[h][w]}")
            yield None
            first = t == (0 if h == 1 else 1)
            if not first:  # an O rescale reads and writes the accumulator
                if self.O[h][w] != ("O", t - 1):
                    raise Violation(f"half {h} warp {w} rescale at tile {t}: O holds {self.O[h][w]}")
                yield None
            self.S[h][w] = ("P", t)
            yield None
            self.p1[h] += 1
            yield None
        yield lambda: self.bar[f"o{h}"].passes(0)
        if self.O[h][w] != ("O", self.T - 1):
            raise Violation(f"half {h} warp {w} epilogue: O holds {self.O[h][w]}")
        yield None

    def run(self):
        self.actors["prod"] = self.producer()
        self.actors["w1"] = self.mma()
        for h in (0, 1):
            for w in range(self.nw):
                self.actors[f"sm{h}{w}"] = self.softmax(h, w)
        self.actors["pipe1"] = self.pipe("w1")
        return self._schedule()


def find_violation_fwd(pv_late=False, runs=300, tiles=10, warps=2):
    """As find_violation, for the forward kernel's protocol (one item)."""
    for seed in range(runs):
        try:
            ForwardModel(pv_late, warps=warps, tiles=tiles, seed=seed, slow="sm00" if seed % 2 else None).run()
        except Violation as e:
            return f"seed {seed}: {e}"
    return None
