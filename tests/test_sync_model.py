"""Executable models of the kernels' synchronisation (host only, no GPU).

attn_fwd_short_kernel (csrc/attn_fwd.cu) runs six roles per CTA that meet only through
mbarriers: the TMA producer, the S-GEMM issuer, the PV-GEMM issuer, the two softmax halves and
the merge/epilogue warpgroup (`Model`); attn_fwd_kernel runs four (the producer with its K/V
ring, one MMA thread, two softmax warpgroups; `MainModel`); attn_bwd_kernel (csrc/attn_bwd.cu)
runs four (the producer, one MMA thread, two P/dS warpgroups, warpgroup 1 also draining dQ
through TMA reductions and writing dK, dV; `BwdModel`).  Each model restates every role
as a sequence of barrier waits,
arrivals and asynchronous completions (TMA loads, tcgen05 commits), in the kernel's order, and
runs it under many random schedules and unit lengths.  It checks:

* no deadlock;
* no phase overrun: an mbarrier wait is a parity wait, so a waiter that falls two phases
  behind would match the wrong phase; every wait must find the barrier at most one phase
  past the one it wants;
* every buffer hazard the barriers exist for: a tensor-core or TMA access (S, P, O in tensor
  memory; Q, K, V tiles; the per-unit statistics) never meets a buffer holding the wrong step's
  or unit's data.

Planted mistakes (the statistics buffer reused without the epilogue's release; a ring slot
refilled without its release; dS stored while the dQ reductions still read the region) must
be caught.
The model mirrors the protocol, not the arithmetic; a change to the kernel's barriers must be
made here too.
"""
import random

import pytest


class Deadlock(Exception):
    pass


class Violation(Exception):
    pass


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.done += 1


class Model:
    """One CTA's run of the short-query kernel's protocol over `units` (key tiles per unit)."""

    def __init__(self, units, rng, release_stats=True):
        self.units, self.rng, self.release_stats = units, rng, release_stats
        B = Barrier
        self.b = {}
        for i in range(2):
            for n, c in (("KFull", 1), ("VFull", 1), ("QFull", 1), ("QEmpty", 1), ("SFull", 1),
                         ("PFull", 2), ("PVDone", 1), ("Stats", 2), ("StatsFree", 1)):
                self.b[(n, i)] = B("%s[%d]" % (n, i), c)
        self.b[("OFull", 0)] = B("OFull", 1)
        self.b[("OEmpty", 0)] = B("OEmpty", 1)
        # buffer contents: what each holds (None = free/undefined)
        self.q_buf = [None, None]          # unit whose Q tile is in query buffer i
        self.k_slot = [None, None]         # step whose K tile is in step slot i
        self.v_slot = [None, None]
        self.s_buf = [None, None]          # ("S", g) or ("P", g) in S buffer i
        self.o_owner = None                # unit accumulating in O (None: read out, free)
        self.o_steps = 0
        self.stats = [None, None]          # (unit, half, read by the epilogue) in buffer i
        self.pending = []                  # asynchronous completions: (time, seq, fn)
        self.now = 0
        self.seq = 0
        self.last_done = {}                # per issuing thread: last completion time

    # --- primitives --------------------------------------------------------------------
    def later(self, fn, channel=None, lo=1, hi=30):
        """Complete `fn` after a random delay; operations of one `channel` (one issuing
        thread's tcgen05 work) complete in issue order, TMA loads in any order."""
        self.seq += 1
        t = self.now + self.rng.randint(lo, hi)
        if channel is not None:
            t = max(t, self.last_done.get(channel, 0) + 1)
            self.last_done[channel] = t
        self.pending.append((t, self.seq, fn))

    def wait(self, key, phase):
        """Generator step: block until phase `phase` of barrier `key` has completed."""
        bar = self.b[key]
        while True:
            if bar.done > phase + 1:
                raise Violation("phase overrun on %s: waiting for phase %d, %d completed"
                                % (bar.name, phase, bar.done))
            if bar.done == phase + 1:
                return
            yield ("wait", bar.name, phase)

    def check(self, cond, what):
        if not cond:
            raise Violation(what)

    # --- roles -------------------------------------------------------------------------
    def producer(self):
        g = 0
        for u, nk in enumerate(self.units):
            qb = u & 1
            if u >= 2:
                yield from self.wait(("QEmpty", qb), (u >> 1) - 1)
            self.check(self.q_buf[qb] in (None, u - 2), "Q buffer %d overwritten early" % qb)

            def load_q(qb=qb, u=u):
                self.q_buf[qb] = u
                self.b[("QFull", qb)].arrive()
            self.later(load_q)
            for jj in range(nk):
                ss = g & 1
                if g >= 2:
                    yield from self.wait(("SFull", ss), (g - 2) >> 1)      # S_{g-2} read K
                self.check(self.k_slot[ss] in (None, g - 2), "K slot overwritten early")

                def load_k(ss=ss, g=g):
                    self.k_slot[ss] = g
                    self.b[("KFull", ss)].arrive()
                self.later(load_k)
                if g >= 2:
                    yield from self.wait(("PVDone", ss), (g - 2) >> 1)     # PV_{g-2} read V
                self.check(self.v_slot[ss] in (None, g - 2), "V slot overwritten early")

                def load_v(ss=ss, g=g):
                    self.v_slot[ss] = g
                    self.b[("VFull", ss)].arrive()
                self.later(load_v)
                g += 1
                yield ("step",)

    def s_issuer(self):
        g = 0
        for u, nk in enumerate(self.units):
            qb = u & 1
            yield from self.wait(("QFull", qb), u >> 1)
            for jj in range(nk):
                sb = g & 1
                yield from self.wait(("KFull", sb), g >> 1)
                if g >= 2:
                    yield from self.wait(("PVDone", sb), (g >> 1) - 1)

                def run_s(sb=sb, g=g, u=u, qb=qb, last=(jj + 1 == nk)):
                    self.check(self.q_buf[qb] == u, "S GEMM read the wrong Q tile")
                    self.check(self.k_slot[sb] == g, "S GEMM read the wrong K tile")
                    self.check(self.s_buf[sb] in (None, ("P", g - 2)), "S overwrote P before its PV")
                    self.s_buf[sb] = ("S", g)
                    self.b[("SFull", sb)].arrive()
                    if last:
                        self.b[("QEmpty", qb)].arrive()
                self.later(run_s, channel="s")
                g += 1
                yield ("step",)

    def pv_issuer(self):
        g = 0
        for u, nk in enumerate(self.units):
            for jj in range(nk):
                sb = g & 1
                yield from self.wait(("VFull", sb), g >> 1)
                if jj == 0 and u > 0:
                    yield from self.wait(("OEmpty", 0), u - 1)
                yield from self.wait(("PFull", sb), g >> 1)

                def run_pv(sb=sb, g=g, u=u, first=(jj == 0), last=(jj + 1 == nk)):
                    self.check(self.s_buf[sb] == ("P", g), "PV GEMM read the wrong P")
                    self.check(self.v_slot[sb] == g, "PV GEMM read the wrong V tile")
                    if first:
                        self.check(self.o_owner is None, "PV overwrote O before the epilogue read it")
                        self.o_owner, self.o_steps = u, 0
                    self.check(self.o_owner == u, "PV accumulated into another unit's O")
                    self.o_steps += 1
                    self.b[("PVDone", sb)].arrive()
                    if last:
                        self.b[("OFull", 0)].arrive()
                self.later(run_pv, channel="pv")
                g += 1
                yield ("step",)

    def softmax(self, h):
        g = 0
        for u, nk in enumerate(self.units):
            for jj in range(nk):
                sb = g & 1
                yield from self.wait(("SFull", sb), g >> 1)
                self.check(self.s_buf[sb] in (("S", g), ("P", g)), "softmax read the wrong S")
                yield ("step",)
                # lazy rescale of O (rare in the kernel, random here): needs PV_{g-1} done
                if jj > 0 and self.rng.random() < 0.2:
                    yield from self.wait(("PVDone", (g - 1) & 1), (g - 1) >> 1)
                    self.check(self.o_owner == u and self.o_steps == jj, "rescale met O mid-update")
                self.s_buf[sb] = ("P", g)      # both halves write their P columns
                self.b[("PFull", sb)].arrive()
                g += 1
            if u >= 2 and self.release_stats:
                yield from self.wait(("StatsFree", u & 1), (u >> 1) - 1)
            prev = self.stats[u & 1]
            self.check(prev is None or prev[0] in (u - 2, u), "statistics of unit %d overwritten unread"
                       % (prev[0] if prev else -1))
            if prev is not None and prev[0] == u - 2 and not prev[2]:
                raise Violation("statistics of unit %d overwritten before the epilogue read them" % (u - 2))
            self.stats[u & 1] = (u, h, False)
            self.b[("Stats", u & 1)].arrive()
            yield ("step",)

    def epilogue(self):
        for u, nk in enumerate(self.units):
            yield from self.wait(("OFull", 0), u)
            yield from self.wait(("Stats", u & 1), u >> 1)
            st = self.stats[u & 1]
            self.check(st is not None and st[0] == u, "epilogue read another unit's statistics")
            self.stats[u & 1] = (u, st[1], True)
            if self.release_stats:
                self.b[("StatsFree", u & 1)].arrive()
            yield ("step",)
            self.check(self.o_owner == u and self.o_steps == nk, "epilogue read an unfinished O")
            self.o_owner = None
            self.b[("OEmpty", 0)].arrive()
            yield ("step",)

    # --- scheduler ---------------------------------------------------------------------
    def run(self, max_events=200000):
        roles = {"producer": self.producer(), "s": self.s_issuer(), "pv": self.pv_issuer(),
                 "sm0": self.softmax(0), "sm1": self.softmax(1), "epi": self.epilogue()}
        self._schedule(roles, max_events)

    def _schedule(self, roles, max_events):
        """Advance a random runnable role, or complete the earliest asynchronous operation
        (always when every role is blocked, sometimes otherwise); no role runnable and nothing
        in flight is a deadlock."""
        blocked = {}
        for _ in range(max_events):
            live = [r for r in roles if roles[r] is not None]
            if not live and not self.pending:
                return
            cand = live[:]
            self.rng.shuffle(cand)
            progressed = False
            for r in cand:
                try:
                    ev = next(roles[r])
                except StopIteration:
                    roles[r] = None
                    progressed = True
                    break
                if ev[0] != "wait" or blocked.get(r) != ev:
                    blocked[r] = ev if ev[0] == "wait" else None
                    progressed = True
                    break
            if not progressed or self.rng.random() < 0.3:
                if not self.pending:
                    if not progressed:
                        raise Deadlock("deadlock: " + ", ".join("%s waits %s" % (r, blocked.get(r))
                                                                   for r in live))
                    continue
                self.pending.sort()
                t, _, fn = self.pending.pop(0)
                self.now = max(self.now, t)
                fn()
                blocked.clear()
        raise Deadlock("no completion within the event budget")


UNIT_PATTERNS = [[1], [3], [1, 1, 1, 1, 1, 1], [2, 1, 3, 1, 1, 2], [4, 4, 4], [1, 5, 1, 1, 2, 1, 1]]


@pytest.mark.parametrize("units", UNIT_PATTERNS, ids=lambda u: "-".join(map(str, u)))
def test_protocol_under_random_schedules(units):
    for seed in range(150):
        Model(units, random.Random(seed * 7919 + len(units))).run()


def test_random_unit_lengths():
    rng = random.Random(12345)
    for _ in range(200):
        units = [rng.randint(1, 4) for _ in range(rng.randint(1, 9))]
        Model(units, random.Random(rng.random())).run()


def test_planted_missing_statistics_release_is_caught():
    # without the epilogue's release of the statistics buffer, units of one key tile let the
    # softmax overwrite a unit's statistics before the epilogue read them (or overrun the
    # statistics barrier): some schedule must expose it
    found = False
    for seed in range(400):
        try:
            Model([1] * 8, random.Random(seed), release_stats=False).run()
        except (Violation, Deadlock):
            found = True
            break
    assert found


class MainModel(Model):
    """attn_fwd_kernel's protocol: one CTA, units of two query tiles, a K,V,K,V ring of
    `stages` slots with full/empty barriers, one MMA thread issuing S_t(j+1) right after
    PV_t(j) (in order), and two softmax warpgroups that each run their tile's epilogue.
    Units in `dead1` have no query in their second tile (a decoding step's rows all sit in
    the first): that tile's softmax warps keep every wait and arrival but read no S, store
    no P and read no O; the GEMMs still run on whatever the tile holds ("X": released by the
    softmax without a P).  `dead_arrives=False` plants the mistake of skipping the arrival."""

    def __init__(self, units, rng, stages=4, wait_empty=True, dead1=frozenset(), dead_arrives=True):
        self.units, self.rng, self.S, self.wait_empty = units, rng, stages, wait_empty
        self.dead1, self.dead_arrives = dead1, dead_arrives
        self.b = {}
        for i in range(stages):
            self.b[("Full", i)] = Barrier("Full[%d]" % i, 1)
            self.b[("Empty", i)] = Barrier("Empty[%d]" % i, 1)
        for t in range(2):
            for n in ("SFull", "PFull", "OFull"):
                self.b[(n, t)] = Barrier("%s[%d]" % (n, t), 1)
        self.b[("QFull", 0)] = Barrier("QFull", 1)
        self.b[("QEmpty", 0)] = Barrier("QEmpty", 1)
        self.ring = [None] * stages            # ring position held by each slot
        self.q = None                          # unit whose Q tiles are loaded
        self.s_buf = [None, None]              # ("S", step) / ("P", step) per tile
        self.o = [None, None]                  # (unit, steps accumulated) per tile
        self.pending, self.now, self.seq, self.last_done = [], 0, 0, {}

    def producer(self):
        pos = 0
        for u, nk in enumerate(self.units):
            if u > 0:
                yield from self.wait(("QEmpty", 0), u - 1)

            def load_q(u=u):
                self.q = u
                self.b[("QFull", 0)].arrive()
            self.later(load_q)
            for _ in range(nk):
                for _kv in range(2):
                    slot = pos % self.S
                    if pos >= self.S and self.wait_empty:
                        yield from self.wait(("Empty", slot), pos // self.S - 1)
                    self.check(self.ring[slot] in (None, pos - self.S), "ring slot overwritten early")

                    def load(slot=slot, pos=pos):
                        self.ring[slot] = pos
                        self.b[("Full", slot)].arrive()
                    self.later(load)
                    pos += 1
                yield ("step",)

    def mma(self):
        pos = 0
        g = 0                                  # steps consumed (same count for both tiles)
        for u, nk in enumerate(self.units):
            yield from self.wait(("QFull", 0), u)
            kslot = pos % self.S
            yield from self.wait(("Full", kslot), pos // self.S)
            for t in range(2):
                self.later(self._s(t, u, g, kslot, pos), channel="mma")
            self.later(self._commit(("Empty", kslot)), channel="mma")
            if nk == 1:
                self.later(self._commit(("QEmpty", 0)), channel="mma")
            pos += 1
            for jj in range(nk):
                vpos = pos
                vslot = vpos % self.S
                more = jj + 1 < nk
                yield from self.wait(("Full", vslot), vpos // self.S)
                kpos = vpos + 1
                kslot = kpos % self.S
                for t in range(2):
                    yield from self.wait(("PFull", t), g)
                    self.later(self._pv(t, u, g, jj, vslot, vpos), channel="mma")
                    if not more:
                        self.later(self._commit(("OFull", t)), channel="mma")
                    if t == 1:
                        self.later(self._commit(("Empty", vslot)), channel="mma")
                    if more:
                        if t == 0:
                            yield from self.wait(("Full", kslot), kpos // self.S)
                        self.later(self._s(t, u, g + 1, kslot, kpos), channel="mma")
                        if t == 1:
                            self.later(self._commit(("Empty", kslot)), channel="mma")
                            if jj + 2 == nk:
                                self.later(self._commit(("QEmpty", 0)), channel="mma")
                g += 1
                pos += 2 if more else 1
                yield ("step",)

    def _commit(self, key):
        return lambda: self.b[key].arrive()

    def _s(self, t, u, g, kslot, kpos):
        def run():
            self.check(self.q == u, "S GEMM read another unit's Q")
            self.check(self.ring[kslot] == kpos, "S GEMM read the wrong K")
            self.check(self.s_buf[t] in (None, ("P", g - 1), ("X", g - 1)), "S overwrote P before its PV")
            self.s_buf[t] = ("S", g)
            self.b[("SFull", t)].arrive()
        return run

    def _pv(self, t, u, g, jj, vslot, vpos):
        def run():
            released = "X" if (t == 1 and u in self.dead1) else "P"
            self.check(self.s_buf[t] == (released, g), "PV read the wrong P")
            self.check(self.ring[vslot] == vpos, "PV read the wrong V")
            if jj == 0:
                self.check(self.o[t] is None, "PV overwrote O before the epilogue read it")
                self.o[t] = (u, 0)
            self.check(self.o[t] == (u, jj), "PV accumulated out of order")
            self.o[t] = (u, jj + 1)
        return run

    def softmax(self, t):
        g = 0
        for u, nk in enumerate(self.units):
            dead = t == 1 and u in self.dead1
            for jj in range(nk):
                yield from self.wait(("SFull", t), g)
                if not dead:
                    self.check(self.s_buf[t] == ("S", g), "softmax read the wrong S")
                    if jj > 0 and self.rng.random() < 0.2:
                        # lazy rescale reads O_t: S_t(g) completing implies PV_t(g-1) did (in order)
                        self.check(self.o[t] == (u, jj), "rescale met O mid-update")
                yield ("step",)
                self.s_buf[t] = ("X", g) if dead else ("P", g)
                if not dead or self.dead_arrives:
                    self.b[("PFull", t)].arrive()
                g += 1
            yield from self.wait(("OFull", t), u)
            if not dead:
                self.check(self.o[t] == (u, nk), "epilogue read an unfinished O")
            yield ("step",)
            self.o[t] = None                   # read out (or, dead, passed over); the next unit's first PV may write

    def run(self, max_events=200000):
        roles = {"producer": self.producer(), "mma": self.mma(), "sm0": self.softmax(0),
                 "sm1": self.softmax(1)}
        self._schedule(roles, max_events)




@pytest.mark.parametrize("stages", [4, 8])
@pytest.mark.parametrize("units", UNIT_PATTERNS, ids=lambda u: "-".join(map(str, u)))
def test_main_kernel_protocol(units, stages):
    for seed in range(100):
        MainModel(units, random.Random(seed * 104729 + stages), stages).run()


@pytest.mark.parametrize("units", UNIT_PATTERNS, ids=lambda u: "-".join(map(str, u)))
def test_main_kernel_protocol_with_dead_second_tiles(units):
    # decoding blocks: some units' second query tile holds no query
    for seed in range(60):
        rng = random.Random(seed * 7919 + len(units))
        dead1 = frozenset(u for u in range(len(units)) if rng.random() < 0.5)
        MainModel(units, rng, 4, dead1=dead1).run()


def test_main_kernel_dead_tile_without_arrival_is_caught():
    # dead softmax warps that skip the P-ready arrival leave the MMA thread waiting
    with pytest.raises(Deadlock):
        MainModel([3, 2], random.Random(1), 4, dead1=frozenset({0}), dead_arrives=False).run()


def test_main_kernel_planted_missing_release_is_caught():
    # a producer that refills a ring slot without waiting for its release must be caught
    found = False
    for seed in range(300):
        try:
            MainModel([3, 2, 4], random.Random(seed), 4, wait_empty=False).run()
        except (Violation, Deadlock):
            found = True
            break
    assert found


class BwdModel(Model):
    """attn_bwd_kernel's protocol: units (b, K/V head, key tile) of `nsteps` query steps each
    (0 for a causal key tile no query sees), a TMA producer (K and V per unit, a two-stage Q/dO
    ring, the step's row statistics), one MMA thread, and two P/dS warpgroups; each warpgroup
    also reads its half of dQ's columns out and stages them in the step's own Q/dO stage (free
    once the step's GEMMs are done), and warpgroup 1 writes dK, dV.  The producer issues a
    stage's dQ reductions just before refilling it and waits for them to have read it."""

    def __init__(self, units, rng, wait_reduce_reads=True, read_barrier=True, box_free_wait=True,
                 rounds=2):
        # wait_reduce_reads=False plants a mistake: the producer refills a stage without waiting
        # for the reductions issued from it to have read it; read_barrier=False another: a
        # warpgroup stores P^T and dS^T without waiting for the other to have loaded S^T, dP^T
        self.units, self.rng, self.wait_reduce_reads = units, rng, wait_reduce_reads
        self.read_barrier = read_barrier
        # box_free_wait=False plants a third: a warpgroup restages its half of the dS region for
        # the next 64 columns of dV/dK without waiting for the previous box store to have read it
        self.box_free_wait, self.rounds = box_free_wait, rounds
        self.b = {}
        for n, c in (("KV", 1), ("KVEmpty", 1), ("Stats", 1), ("SFull", 1), ("DPFull", 1),
                     ("PFull", 2), ("Read", 2), ("DQFull", 1), ("DQEmpty", 2), ("DKVFull", 1),
                     ("DKVEmpty", 2)):
            self.b[(n, 0)] = Barrier(n, c)
        for i in range(2):
            self.b[("BoxFree", i)] = Barrier("BoxFree[%d]" % i, 1)
        for i in range(2):
            self.b[("QFull", i)] = Barrier("QFull[%d]" % i, 1)
            self.b[("QEmpty", i)] = Barrier("QEmpty[%d]" % i, 1)
            self.b[("Staged", i)] = Barrier("Staged[%d]" % i, 2)
        self.kv = None                   # unit whose K, V are in shared memory
        self.qdo = [None, None]          # step whose Q, dO are in each ring stage
        self.stats = None                # step whose statistics are loaded
        self.t_sp = None                 # TMEM columns 0-127: ("S", s) or ("P", s)
        self.t_dp = None                 # TMEM 128-255: ("dP", s), ("dS", s) or ("dQ", s)
        self.dkv = None                  # (unit, steps accumulated) in the dV, dK columns
        self.ds_box = [None, None]       # the dS region's halves: ("dS", s) or a staged dV/dK box
        self.reduce_reading = None       # step whose staged dQ the producer's reductions still read
        self.dq_read = set()             # warpgroups that have read the current dQ out of TMEM
        self.dkv_read = set()            # warpgroups that have written their half of dK/dV out
        self.pending, self.now, self.seq, self.last_done = [], 0, 0, {}

    def producer(self):
        s = 0
        for u, n in enumerate(self.units):
            def load_kv(u=u):
                self.kv = u
                self.b[("KV", 0)].arrive()
            # the unit's first Q/dO goes in before the wait for the previous unit's K/V release
            if n > 0:
                yield from self.load_q(s)
            if u > 0:
                yield from self.wait(("KVEmpty", 0), u - 1)
            self.later(load_kv)
            for st in range(n):
                if st > 0:
                    yield from self.load_q(s)
                if s > 0:
                    yield from self.wait(("PFull", 0), s - 1)

                def load_stats(s=s):
                    self.check(self.stats in (None, s - 1), "statistics overwritten early")
                    self.stats = s
                    self.b[("Stats", 0)].arrive()
                self.later(load_stats)
                s += 1
                yield ("step",)
        for t in range(max(s - 2, 0), s):
            yield from self.reduce(t)

    def load_q(self, s):
        """Refill ring stage s % 2 with step s's Q/dO once its previous occupant's GEMMs are
        done and the dQ staged there has been read by the reductions."""
        sg = s % 2
        if s >= 2:
            yield from self.wait(("QEmpty", sg), s // 2 - 1)
            yield from self.reduce(s - 2)
        self.check(self.qdo[sg] in (None, ("stage", s - 2)), "Q/dO stage overwritten early")
        self.check(self.reduce_reading != s - 2 or s < 2,
                   "Q/dO stage refilled while dQ reductions still read it")

        def load(sg=sg, s=s):
            self.qdo[sg] = s
            self.b[("QFull", sg)].arrive()
        self.later(load)

    def reduce(self, t):
        """The producer's TMA reductions of step t's staged dQ, then (normally) a wait for
        their reads of the stage."""
        yield from self.wait(("Staged", t % 2), t // 2)
        self.check(self.qdo[t % 2] == ("stage", t), "reductions read a stage not holding dQ")
        self.reduce_reading = t

        def reads_done(t=t):
            if self.reduce_reading == t:
                self.reduce_reading = None
        self.later(reads_done, channel="tma_reduce")
        while self.wait_reduce_reads and self.reduce_reading is not None:
            yield ("wait", "bulk read", t)

    def mma(self):
        s = 0
        for u, n in enumerate(self.units):
            yield from self.wait(("KV", 0), u)
            for st in range(n):
                sg = s % 2
                yield from self.wait(("QFull", sg), s // 2)

                def gemm_s(s=s, sg=sg, u=u):
                    self.check(self.kv == u and self.qdo[sg] == s, "S^T read the wrong K or Q")
                    self.check(self.t_sp in (None, ("P", s - 1)), "S^T overwrote P^T before dV read it")
                    self.t_sp = ("S", s)
                    self.b[("SFull", 0)].arrive()
                self.later(gemm_s, channel="mma")
                if s > 0:
                    yield from self.wait(("DQEmpty", 0), s - 1)

                def gemm_dp(s=s, sg=sg, u=u):
                    self.check(self.kv == u and self.qdo[sg] == s, "dP^T read the wrong V or dO")
                    self.check(self.t_dp in (None, ("dQ", s - 1, "read")), "dP^T overwrote an unread dQ")
                    self.t_dp = ("dP", s)
                    self.b[("DPFull", 0)].arrive()
                self.later(gemm_dp, channel="mma")
                yield from self.wait(("PFull", 0), s)
                if st == 0 and u > 0:
                    yield from self.wait(("DKVEmpty", 0), u - 1)

                def gemm_dvdk(s=s, sg=sg, u=u, st=st):
                    self.check(self.t_sp == ("P", s) and self.t_dp == ("dS", s), "dV/dK read the wrong P or dS")
                    self.check(self.qdo[sg] == s, "dV/dK read the wrong Q or dO")
                    if st == 0:
                        self.check(self.dkv is None, "dV/dK overwrote an unread accumulator")
                        self.dkv = (u, 0)
                    self.check(self.dkv == (u, st), "dV/dK accumulated out of order")
                    self.dkv = (u, st + 1)
                    self.b[("QEmpty", sg)].arrive()
                self.later(gemm_dvdk, channel="mma")

                def gemm_dq(s=s, u=u):
                    self.check(self.ds_box == [("dS", s), ("dS", s)] and self.kv == u, "dQ read the wrong dS or K")
                    self.t_dp = ("dQ", s)
                    self.b[("DQFull", 0)].arrive()
                self.later(gemm_dq, channel="mma")
                s += 1
                yield ("step",)
            if n == 0 and u > 0:
                yield from self.wait(("DKVEmpty", 0), u - 1)

            def unit_done(u=u, n=n):
                if n == 0:
                    self.check(self.dkv is None, "empty unit met an unread accumulator")
                    self.dkv = (u, 0)
                self.b[("DKVFull", 0)].arrive()
                self.b[("KVEmpty", 0)].arrive()
            self.later(unit_done, channel="mma")

    def pds(self, half, s, u):
        yield from self.wait(("Stats", 0), s)
        yield from self.wait(("SFull", 0), s)
        yield from self.wait(("DPFull", 0), s)
        self.check(self.stats == s, "P/dS read the wrong statistics")
        self.check(self.t_sp == ("S", s) and self.t_dp == ("dP", s), "P/dS read the wrong S^T or dP^T")
        yield ("step",)
        if self.read_barrier:
            self.b[("Read", 0)].arrive()
            yield from self.wait(("Read", 0), s)
        for box in self.ds_box:
            self.check(box is None or box[0] == "dS" or box[-1] == "read", "dS^T overwrote an unread dK/dV box")
        self.t_sp, self.t_dp, self.ds_box = ("P", s), ("dS", s), [("dS", s), ("dS", s)]
        self.b[("PFull", 0)].arrive()

    def wg(self, half):
        s = 0
        for u, n in enumerate(self.units):
            for _ in range(n):
                yield from self.pds(half, s, u)
                yield from self.wait(("DQFull", 0), s)
                self.check(self.t_dp == ("dQ", s), "dQ readout met the wrong TMEM contents")
                self.dq_read.add(half)
                if self.dq_read == {0, 1}:
                    self.t_dp, self.dq_read = ("dQ", s, "read"), set()
                self.b[("DQEmpty", 0)].arrive()
                # stage into its boxes of the step's Q/dO stage (its GEMMs are done) for the
                # producer's reductions
                sg = s % 2
                self.check(self.qdo[sg] in (s, ("stage", s)), "staging overwrote another step's Q/dO")
                self.qdo[sg] = ("stage", s)
                yield ("step",)
                self.b[("Staged", sg)].arrive()
                s += 1
                yield ("step",)
            # warpgroup 0 writes dV out, warpgroup 1 dK, each through its half (box) of the dS
            # region, 64 columns per round: stage, then a TMA store whose read of the box
            # completes later; the next round waits for it, and so (through the read barrier the
            # storing warp must reach) does the next unit's dS^T
            yield from self.wait(("DKVFull", 0), u)
            self.check(self.dkv == (u, n), "dK/dV read out unfinished")
            for cc in range(self.rounds):
                rnd = u * self.rounds + cc
                if rnd > 0 and self.box_free_wait:
                    yield from self.wait(("BoxFree", half), rnd - 1)
                box = self.ds_box[half]
                self.check(box is None or box[0] == "dS" or box[-1] == "read",
                           "dK/dV staging overwrote an unread box")
                self.ds_box[half] = ("out", u, half, cc)
                yield ("step",)
                if cc == self.rounds - 1:
                    self.dkv_read.add(half)
                    if self.dkv_read == {0, 1}:
                        self.dkv, self.dkv_read = None, set()
                    self.b[("DKVEmpty", 0)].arrive()

                def read_done(half=half, u=u, cc=cc):
                    self.check(self.ds_box[half] == ("out", u, half, cc), "dK/dV store read another box")
                    self.ds_box[half] = ("out", u, half, cc, "read")
                    self.b[("BoxFree", half)].arrive()
                self.later(read_done, channel="tma_store%d" % half)
                yield ("step",)
            yield from self.wait(("BoxFree", half), (u + 1) * self.rounds - 1)

    def run(self, max_events=200000):
        roles = {"producer": self.producer(), "mma": self.mma(), "wg0": self.wg(0), "wg1": self.wg(1)}
        self._schedule(roles, max_events)


BWD_PATTERNS = [[1], [4], [2, 0, 3], [1, 1, 1, 1, 1], [0, 2, 0, 0, 1], [3, 1, 4, 1, 2]]


@pytest.mark.parametrize("units", BWD_PATTERNS, ids=lambda u: "-".join(map(str, u)))
def test_backward_kernel_protocol(units):
    for seed in range(150):
        BwdModel(units, random.Random(seed * 31337 + len(units))).run()


def test_backward_random_unit_lengths():
    rng = random.Random(777)
    for _ in range(200):
        units = [rng.randint(0, 4) for _ in range(rng.randint(1, 8))]
        BwdModel(units, random.Random(rng.random())).run()


def test_backward_planted_early_stage_refill_is_caught():
    # the producer refilling a Q/dO stage before the dQ reductions issued from it have read
    # it: some schedule must expose it
    found = False
    for seed in range(400):
        try:
            BwdModel([3, 2], random.Random(seed), wait_reduce_reads=False).run()
        except (Violation, Deadlock):
            found = True
            break
    assert found


def test_backward_planted_early_p_store_is_caught():
    # a warpgroup storing P^T and dS^T over S^T and dP^T before the other warpgroup has loaded
    # its columns of them
    found = False
    for seed in range(400):
        try:
            BwdModel([2, 1], random.Random(seed), read_barrier=False).run()
        except (Violation, Deadlock):
            found = True
            break
    assert found


def test_backward_planted_early_box_restage_is_caught():
    # a warpgroup staging its next 64 columns of dV/dK before the previous box store has read
    # its half of the dS region
    found = False
    for seed in range(400):
        try:
            BwdModel([1, 0, 1], random.Random(seed), box_free_wait=False).run()
        except (Violation, Deadlock):
            found = True
            break
    assert found
