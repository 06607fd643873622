"""Models of the attention kernels' hand-off protocols between their MMA issuers and their
element-wise (softmax) warps, run under random schedules to look for races.

Test infrastructure: it restates, in Python, the order of waits, products, commits and counter
updates of the tensor-core dQ and dK/dV kernels (csrc/attn_bwd_tc.cu) and of the forward
kernel (csrc/attn_tc.cu) and checks the data those steps hand over.  Nothing here runs the
kernels.  The dQ and dK/dV models run one item or a sequence of items (each item's
accumulators are read by the warps' epilogue before the next item's first products overwrite
them; the shared-memory rings are left out, their waits being taken one per completion); the
forward model runs sequences of items with its producer, its stage ring and the Q reloads,
since one of its waits skips phases.

What is modelled:
- the backward kernels' three 128-column tensor-memory slots in rotation (tile g: S in slot
  s(g), dP in slot d(g) = s(g - 1), S(g) overwriting the slot of dS(g - 2)); the forward
  kernel's S/P slot and O accumulator per half of the item's rows;
- each element-wise warp owns its own lanes of every slot: a product writes all lanes, a warp
  reads and writes its own, the dQ product reads all;
- an issuer's products run in its own order; products of two issuers interleave freely;
- `tcgen05.commit`: an arrival once every earlier product of that issuer has run;
- mbarrier waits with the hardware's parity test: a wait for completion k (0-based) passes
  when the number of completed phases differs from k in parity, so it passes one phase early
  (k - 1 completed) and not at all two phases late (k + 2 completed);
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

    def __init__(self, variant, ds_by_parity, read_by_parity=False, warps=4, tiles=10, seed=0, slow=None,
                 items=None, late_epilogue=False):
        items = items if items is not None else [tiles]
        self.variant, self.nw, self.T = variant, warps, sum(items)
        # the dQ kernel's items: tile g belongs to item item_of[g] as its t_of[g]-th tile; each
        # item's dQ products accumulate into one tensor-memory accumulator (the first of an
        # item overwrites it), read by the warps' epilogue once the item's last dQ completes
        self.items = items
        self.item_of = [i for i, n in enumerate(items) for _ in range(n)]
        self.t_of = [t for n in items for t in range(n)]
        self.DQ = [None] * warps
        # planted mistake: a warp reads an item's dQ only after storing the next item's first dS
        self.late_epilogue = late_epilogue
        self.ds_by_parity, self.read_by_parity = ds_by_parity, read_by_parity
        self.rng = random.Random(seed)
        self.slow = slow  # actor name scheduled rarely, to open lags
        self.tags = [[None] * warps for _ in range(3)]
        self.p0 = [0, 0]   # S read (by parity, or summed in [0])
        self.p1 = [0, 0]   # dS stored
        self.s_issued = 0
        self.bar = {n: Barrier() for n in ("s0", "s1", "d0", "d1", "q0", "q1", "o")}
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

    def _dq(self, g):
        """dQ(g): reads every warp's dS(g); accumulates into the item's dQ (the first
        product of an item overwrites the accumulator)."""
        def run():
            self._read_all(d_slot(g), ("dS", g), f"dQ({g})")
            i, t = self.item_of[g], self.t_of[g]
            if t > 0 and any(x != ("dQ", i, g - 1) for x in self.DQ):
                raise Violation(f"dQ({g}): accumulator holds {self.DQ}, expected {('dQ', i, g - 1)}")
            self.DQ = [("dQ", i, g)] * self.nw
        return run

    def _dq_ready(self, g):
        return self._reached(self.p1, self.ds_by_parity, g)

    def _item_last(self, g):
        return self.t_of[g] == self.items[self.item_of[g]] - 1

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
            yield lambda g=g: self._dq_ready(g)
            self.fifo["w2"].append(("mma", self._dq(g)))
            self.fifo["w2"].append(("commit", f"q{g & 1}"))
            if self._item_last(g):
                self.fifo["w2"].append(("commit", "o"))
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
                yield lambda g=g: self._dq_ready(g - 1)
                self.fifo["w1"].append(("mma", self._dq(g - 1)))
                if self._item_last(g - 1):
                    self.fifo["w1"].append(("commit", "o"))
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
            # epilogue: the item's dQ, once its last product completed
            if self.late_epilogue:
                if self.t_of[g] == 0 and g > 0:
                    yield from self._epilogue(w, g - 1)
                if g == self.T - 1:
                    yield from self._epilogue(w, g)
            elif self._item_last(g):
                yield from self._epilogue(w, g)

    def _epilogue(self, w, g):
        i = self.item_of[g]
        yield lambda i=i: self.bar["o"].passes(i)
        if self.DQ[w] != ("dQ", i, g):
            raise Violation(f"warp {w} epilogue of item {i}: dQ accumulator holds {self.DQ[w]}")
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


def find_violation(variant, ds_by_parity, read_by_parity=False, runs=300, tiles=10, warps=4, items=False,
                   late_epilogue=False):
    """The first violation over `runs` random schedules (half of them with one slow warp), or None.
    items=True: each schedule runs a random sequence of items of 1 to 4 tiles (else one item)."""
    for seed in range(runs):
        slow = "ew0" if seed % 2 else None
        its = None
        if items:
            rng = random.Random(2000 + seed)
            its = [rng.randint(1, 4) for _ in range(rng.randint(2, 4))]
        try:
            Model(variant, ds_by_parity, read_by_parity, warps=warps, tiles=tiles, seed=seed, slow=slow,
                  items=its, late_epilogue=late_epilogue).run()
        except Violation as e:
            return f"seed {seed}: {e}"
    return None


class DkdvModel(Model):
    """The dK/dV kernel's protocol: one issuer; slot 0 holds S^T(t) and then the P^T(t) the
    warps write over it (read by dV(t)), slot 1 dP^T(t) and then dS^T(t) (read by dK(t)).
    Product order dV(t), S^T(t + 1), dK(t), dP^T(t + 1); swap_order=True puts S^T(t + 1)
    before dV(t) (a planted mistake: it overwrites P^T(t) before dV(t) reads it).  Over a
    run of items, an item starts with S^T and dP^T of its first tile, its first dV and dK
    overwrite the accumulators and the warps read them in their epilogue once the item's
    last dK completed; late_epilogue=True moves that read after the next item's first P^T
    (a planted mistake)."""

    def __init__(self, swap_order=False, warps=4, tiles=10, seed=0, slow=None, items=None, late_epilogue=False):
        super().__init__("dkdv", ds_by_parity=False, warps=warps, tiles=tiles, seed=seed, slow=slow,
                         items=items, late_epilogue=late_epilogue)
        self.tags = [[None] * warps for _ in range(2)]
        self.swap = swap_order
        self.acc = {"dV": [None] * warps, "dK": [None] * warps}

    def _acc(self, name, slot, want, g):
        """dV(g) or dK(g): reads every warp's lanes of the slot, accumulates into the item's
        accumulator (the item's first product overwrites it)."""
        def run():
            self._read_all(slot, (want, g), f"{name}({g})")
            i, t = self.item_of[g], self.t_of[g]
            if t > 0 and any(x != (name, i, g - 1) for x in self.acc[name]):
                raise Violation(f"{name}({g}): accumulator holds {self.acc[name]}, expected {(name, i, g - 1)}")
            self.acc[name] = [(name, i, g)] * self.nw
        return run

    def issuer(self):
        f = self.fifo["w1"]
        for g in range(self.T):
            if self.t_of[g] == 0:  # the item's first tile
                f.append(("mma", lambda g=g: self._write(0, ("S", g))))
                f.append(("commit", "s0"))
                f.append(("mma", lambda g=g: self._write(1, ("dP", g))))
                f.append(("commit", "s1"))
                yield None
            nxt = not self._item_last(g)
            if self.swap and nxt:
                f.append(("mma", lambda g=g: self._write(0, ("S", g + 1))))
                f.append(("commit", "s0"))
            yield lambda g=g: self._reached(self.p0, False, g)
            f.append(("mma", self._acc("dV", 0, "P", g)))
            if nxt and not self.swap:
                f.append(("mma", lambda g=g: self._write(0, ("S", g + 1))))
                f.append(("commit", "s0"))
            yield None
            yield lambda g=g: self._reached(self.p1, False, g)
            f.append(("mma", self._acc("dK", 1, "dS", g)))
            if not nxt:
                f.append(("commit", "o"))
            if nxt:
                f.append(("mma", lambda g=g: self._write(1, ("dP", g + 1))))
                f.append(("commit", "s1"))
            yield None

    def ew(self, w):
        for g in range(self.T):
            yield lambda g=g: self.bar["s0"].passes(g)
            self._read_own(0, w, ("S", g), f"warp {w} S^T({g})")
            yield None
            self.tags[0][w] = ("P", g)
            yield None
            self._add(self.p0, False, g)
            if self.late_epilogue and self.t_of[g] == 0 and g > 0:
                yield from self._epilogue_kv(w, g - 1)
            yield lambda g=g: self.bar["s1"].passes(g)
            self._read_own(1, w, ("dP", g), f"warp {w} dP^T({g})")
            yield None
            self.tags[1][w] = ("dS", g)
            yield None
            self._add(self.p1, False, g)
            yield None
            if self._item_last(g) and (not self.late_epilogue or g == self.T - 1):
                yield from self._epilogue_kv(w, g)

    def _epilogue_kv(self, w, g):
        i = self.item_of[g]
        yield lambda i=i: self.bar["o"].passes(i)
        for name in ("dV", "dK"):
            if self.acc[name][w] != (name, i, g):
                raise Violation(f"warp {w} epilogue of item {i}: {name} accumulator holds {self.acc[name][w]}")
        yield None

    def run(self):
        self.actors["w1"] = self.issuer()
        for w in range(self.nw):
            self.actors[f"ew{w}"] = self.ew(w)
        self.actors["pipe1"] = self.pipe("w1")
        return self._schedule()


def find_violation_dkdv(swap_order=False, runs=300, tiles=10, warps=4, items=False, late_epilogue=False):
    """As find_violation, for the dK/dV kernel's protocol."""
    for seed in range(runs):
        its = None
        if items:
            rng = random.Random(3000 + seed)
            its = [rng.randint(1, 4) for _ in range(rng.randint(2, 4))]
        try:
            DkdvModel(swap_order, warps=warps, tiles=tiles, seed=seed, slow="ew0" if seed % 2 else None,
                      items=its, late_epilogue=late_epilogue).run()
        except Violation as e:
            return f"seed {seed}: {e}"
    return None


class ForwardModel(Model):
    """The forward kernel's protocol over a run of items (tests/protocol_model.py's forward
    part; csrc/attn_tc.cu).  Each item has two halves of query rows; half h has an S slot
    (P written over it), an O accumulator and a Q buffer.  Stages run on across items: an
    item's stage 0 holds K_0, stage t + 1 holds (V_t, K_t+1); a ring of `nstage` stage
    buffers is refilled by the producer once the MMA thread releases a stage, and the
    producer reloads Q_h once the MMA thread has issued the item's last Q_h K^T.

    items: (nmax, skips, has1) per item: its tile count, the tiles half 0 sits out, whether
    half 1 has rows.  last_half: the half (0) whose softmax learns of its next S from the
    release of the stage that computed it, or None (both halves signalled by their own
    barrier, the fused contiguous / zigzag ring).  o_after_release: the last half's O-ready
    commit goes after the release of the item's last stage (else before it, at its P V).
    pv_late: the next Q K^T before P V (a planted mistake: it overwrites P before it is read)."""

    def __init__(self, items, last_half=0, o_after_release=True, pv_late=False, nstage=2, warps=2,
                 seed=0, slow=None):
        super().__init__("fwd", ds_by_parity=False, warps=warps, tiles=0, seed=seed, slow=slow)
        self.items = items
        self.lh = last_half
        self.o_after = o_after_release
        self.pv_late = pv_late
        self.ns = nstage
        self.S = [[None] * warps for _ in range(2)]  # per half, per warp's lanes
        self.O = [[None] * warps for _ in range(2)]
        self.Q = [None, None]
        self.buf = [None] * nstage                   # stage buffer -> the stage it holds
        self.pcount = [0, 0]                         # P tiles published, summed over the warps
        names = ["s0", "s1", "o0", "o1", "q_full0", "q_full1", "q_empty0", "q_empty1"]
        names += [f"full{i}" for i in range(nstage)] + [f"empty{i}" for i in range(nstage)]
        self.bar = {n: Barrier() for n in names}
        self.fifo = {"w1": []}
        order = (1, 0) if last_half == 0 else (0, 1)
        self.order = order

    # ---- item shape
    def part(self, i, h, t):
        nmax, skips, has1 = self.items[i]
        return has1 if h else t not in skips

    def last(self, i, h):
        nmax = self.items[i][0]
        return max(t for t in range(nmax) if self.part(i, h, t))

    def has(self, i, h):
        return any(self.part(i, h, t) for t in range(self.items[i][0]))

    def sbase(self, i):
        return sum(1 + n for n, _, _ in self.items[:i])

    # ---- products
    def _qk(self, i, h, t, gs):
        def run():
            if self.buf[gs % self.ns] != gs:
                raise Violation(f"QK_{h}({i},{t}): buffer {gs % self.ns} holds stage {self.buf[gs % self.ns]}, not {gs}")
            if self.Q[h] != i:
                raise Violation(f"QK_{h}({i},{t}): Q_{h} holds item {self.Q[h]}")
            self.S[h] = [("S", i, t)] * self.nw
        return run

    def _pv(self, i, h, t, gs, prev):
        def run():
            if self.buf[gs % self.ns] != gs:
                raise Violation(f"PV_{h}({i},{t}): buffer {gs % self.ns} holds stage {self.buf[gs % self.ns]}, not {gs}")
            if any(x != ("P", i, t) for x in self.S[h]):
                raise Violation(f"PV_{h}({i},{t}): S slot of half {h} holds {self.S[h]}")
            want = None if prev is None else ("O", i, prev)
            if prev is not None and any(x != want for x in self.O[h]):
                raise Violation(f"PV_{h}({i},{t}): O of half {h} holds {self.O[h]}, expected {want}")
            self.O[h] = [("O", i, t)] * self.nw
        return run

    # ---- programs
    def producer(self):
        gs, qn = 0, [0, 0]
        for i, (nmax, _, _) in enumerate(self.items):
            for st in range(-1, nmax):
                if gs >= self.ns:
                    yield lambda gs=gs: self.bar[f"empty{gs % self.ns}"].passes(gs // self.ns - 1)
                self.buf[gs % self.ns] = gs
                yield None
                self.bar[f"full{gs % self.ns}"].done += 1
                yield None
                if st == -1:  # Q of the item, once its previous user has issued its last Q K^T
                    for h in (0, 1):
                        if not self.has(i, h):
                            continue
                        if qn[h] >= 1:
                            yield lambda h=h, k=qn[h] - 1: self.bar[f"q_empty{h}"].passes(k)
                        self.Q[h] = i
                        yield None
                        self.bar[f"q_full{h}"].done += 1
                        qn[h] += 1
                        yield None
                gs += 1

    def mma(self):
        f = self.fifo["w1"]
        gs, qn, pc = 0, [0, 0], [0, 0]
        for i, (nmax, _, _) in enumerate(self.items):
            for h in (0, 1):
                if self.has(i, h):
                    yield lambda h=h, k=qn[h]: self.bar[f"q_full{h}"].passes(k)
                    qn[h] += 1
            yield lambda gs=gs: self.bar[f"full{gs % self.ns}"].passes(gs // self.ns)
            for h in (0, 1):
                if self.part(i, h, 0):
                    f.append(("mma", self._qk(i, h, 0, gs)))
                    if h != self.lh:
                        f.append(("commit", f"s{h}"))
                    if self.last(i, h) == 0:
                        f.append(("commit", f"q_empty{h}"))
            f.append(("commit", f"empty{gs % self.ns}"))
            gs += 1
            yield None
            prev = [None, None]
            for t in range(nmax):
                yield lambda gs=gs: self.bar[f"full{gs % self.ns}"].passes(gs // self.ns)
                o_due = False
                for h in self.order:
                    nxt = t + 1 < nmax and self.part(i, h, t + 1)
                    if self.pv_late and nxt:
                        f.append(("mma", self._qk(i, h, t + 1, gs)))
                    if self.part(i, h, t):
                        pc[h] += 1
                        yield lambda h=h, k=pc[h]: self.pcount[h] >= self.nw * k
                        f.append(("mma", self._pv(i, h, t, gs, prev[h])))
                        prev[h] = t
                        if t == self.last(i, h):
                            if h == self.lh and self.o_after:
                                o_due = True
                            else:
                                f.append(("commit", f"o{h}"))
                    if nxt and not self.pv_late:
                        f.append(("mma", self._qk(i, h, t + 1, gs)))
                    if nxt:
                        if h != self.lh:
                            f.append(("commit", f"s{h}"))
                        if t + 1 == self.last(i, h):
                            f.append(("commit", f"q_empty{h}"))
                    yield None
                f.append(("commit", f"empty{gs % self.ns}"))
                if o_due:
                    f.append(("commit", f"o{self.lh}"))
                gs += 1
                yield None

    def softmax(self, h, w):
        scnt = ocnt = 0
        for i, (nmax, _, _) in enumerate(self.items):
            sb = self.sbase(i)
            if not self.has(i, h):
                continue
            prev = None
            for t in range(nmax):
                if not self.part(i, h, t):
                    continue
                if h == self.lh:
                    gs = sb + t
                    yield lambda gs=gs: self.bar[f"empty{gs % self.ns}"].passes(gs // self.ns)
                else:
                    yield lambda k=scnt: self.bar[f"s{h}"].passes(k)
                    scnt += 1
                if self.S[h][w] != ("S", i, t):
                    raise Violation(f"half {h} warp {w} S({i},{t}): finds {self.S[h][w]}")
                yield None
                if prev is not None:  # a rescale reads and writes the accumulator
                    if self.O[h][w] != ("O", i, prev):
                        raise Violation(f"half {h} warp {w} rescale at ({i},{t}): O holds {self.O[h][w]}")
                    yield None
                self.S[h][w] = ("P", i, t)
                yield None
                self.pcount[h] += 1
                prev = t
                yield None
            yield lambda k=ocnt: self.bar[f"o{h}"].passes(k)
            ocnt += 1
            if self.O[h][w] != ("O", i, prev):
                raise Violation(f"half {h} warp {w} epilogue of item {i}: O holds {self.O[h][w]}")
            yield None

    def run(self):
        self.actors["prod"] = self.producer()
        self.actors["w1"] = self.mma()
        for h in (0, 1):
            for w in range(self.nw):
                self.actors[f"sm{h}{w}"] = self.softmax(h, w)
        self.actors["pipe1"] = self.pipe("w1")
        return self._schedule()


def random_items(rng, mode, n=4):
    """Item shapes of a kernel mode: 'single' (one ring step or the single pass: half 0 may
    sit out the first tile), 'fused' (contiguous / zigzag ring: half 0 may sit out the last
    tile of the first step) or 'striped' (half 0 sits out the first tile of every step)."""
    items = []
    for _ in range(n):
        has1 = rng.random() < 0.8
        if mode == "striped":
            T, R = rng.randint(2, 3), rng.randint(1, 3)
            items.append((R * T, set(range(0, R * T, T)) if has1 else set(), has1))
            continue
        t0 = rng.randint(1, 4)
        nmax = t0 + (rng.randint(0, 3) if mode == "fused" else 0)
        skip = set()
        if has1 and t0 >= 2 and rng.random() < 0.7:
            skip = {0} if mode == "single" else {t0 - 1}
        items.append((nmax, skip, has1))
    return items


def find_violation_fwd(mode="single", o_after_release=True, pv_late=False, runs=300, nstage=2, warps=2):
    """As find_violation, for the forward kernel's protocol over random runs of items."""
    for seed in range(runs):
        rng = random.Random(1000 + seed)
        items = random_items(rng, mode)
        slow = ("pipe1", "sm00", None)[seed % 3]
        try:
            ForwardModel(items, last_half=None if mode == "fused" else 0, o_after_release=o_after_release,
                         pv_late=pv_late, nstage=nstage, warps=warps, seed=seed, slow=slow).run()
        except Violation as e:
            return f"seed {seed} items {items}: {e}"
    return None
