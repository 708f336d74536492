"""An executable model of the scaled-GEMM kernel's barrier-ring protocol.

The kernel (mxfp4_quantized_gemm_token_gb300/csrc/gemm_kernel.cuh) is a set of
warp roles handing work to each other through shared-memory rings, each slot
guarded by a pair of mbarriers (full / empty) that the roles wait on by phase
parity.  A parity wait cannot tell a phase that completed from one that is a
whole lap behind, so the protocol is only correct if no waiter can ever be
two phases away from the barrier it waits on.  These tests model the roles
as coroutines and the barriers with the hardware's arrival / phase / parity
rules, run them under many random interleavings (tensor-core and TMA
completions are asynchronous events completing later), and check at every
wait that the slot holds exactly the fill the waiter expects; they also
check that every accumulator the epilogue reads holds exactly the unit's
slices, and that nothing deadlocks.

Roles modelled, per CTA (names as in the kernel):
  producer      fills the A ring (weights) in slice order; an MXFP4 stage
                holds two consecutive slices of one unit (one copy), and a
                unit of odd length ends on a stage with one slice, whose
                decode group arrives on the stage's empty barrier twice
  B producer    fills the B ring (bf16 tokens) in slice order (bf16 kinds)
  scale loader  fills the scale ring in slice order (promoted kinds; the
                MXFP4 decode threads load their own scale bytes)
  decode warps  NDG groups; group g decodes the slices with ia % NDG == g
                into the C ring (TMEM); each warp arrives on its own
  MMA issuers   two; each takes alternate slices and commits asynchronously
  epilogue      reads the accumulators (per slice when promoted, per unit as
                a pair of buffers otherwise) and hands them back

The second test runs the model with the issuer rule the kernel first shipped
with (whole-K issuers taking a unit's slices by their parity within the unit)
and checks that the model finds the stale read that rule allows when the
decode runs as two groups and units have an odd number of slices.
"""
import random

import pytest


class Bar:
    """mbarrier: `count` arrivals complete a phase; try_wait.parity(P) is
    true while the number of completed phases has the other parity than P."""

    def __init__(self, name, count):
        self.name, self.count, self.pending, self.completed = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def passes(self, parity):
        return (self.completed & 1) != parity


class Violation(AssertionError):
    pass


def check(cond, msg):
    if not cond:
        raise Violation(msg)


class Cta:
    """State and roles of one persistent CTA processing `units` (slice counts)."""

    def __init__(self, units, promote, ndg, mxw, AS=12, BS=4, CS=4, SSL=8, NB=4,
                 old_issuer_rule=False, warps_per_group=2, f8f8=False, scale_ring=True,
                 a_per=None, double_arrival=True):
        # f8f8: FP8 x FP8 (dense and token-major W8A8): one producer loads both
        # operands of a slice into the A ring, which the MMA issuers read
        # directly; the scale ring feeds the promotion epilogue; no decode
        self.f8f8 = f8f8
        if f8f8:
            promote, ndg, mxw = True, 0, False
        self.units, self.promote, self.ndg, self.mxw = units, promote, ndg, mxw
        # the scale ring feeds the decode (MXFP4) or the promotion epilogue
        # (promoted kinds); per-tensor whole-K has none, and the token-major
        # epilogue reads its scales itself (scale_ring=False)
        self.epi_scales = promote and scale_ring
        self.AS, self.BS, self.CS, self.SSL, self.NB = AS, BS, CS, SSL, NB
        self.old = old_issuer_rule
        self.wpg = warps_per_group
        W = warps_per_group
        # K slices per A stage: two for MXFP4 (as the kernel), else one
        self.a_per = a_per if a_per is not None else (2 if mxw else 1)
        self.double_arrival = double_arrival
        self.a_full = [Bar("a_full%d" % i, 1) for i in range(AS)]
        self.a_empty = [Bar("a_empty%d" % i, 1 if f8f8 else W * self.a_per) for i in range(AS)]
        self.b_full = [Bar("b_full%d" % i, 1) for i in range(BS)]
        self.b_empty = [Bar("b_empty%d" % i, 1) for i in range(BS)]
        self.c_full = [Bar("c_full%d" % i, W) for i in range(CS)]
        self.c_empty = [Bar("c_empty%d" % i, 1) for i in range(CS)]
        self.s_full = [Bar("s_full%d" % i, 1) for i in range(SSL)]
        self.s_empty = [Bar("s_empty%d" % i, 1) for i in range(SSL)]
        self.t_full = [Bar("t_full%d" % i, 1) for i in range(NB)]
        self.t_empty = [Bar("t_empty%d" % i, 1) for i in range(NB)]
        # slot contents: which slice a slot holds, and how far it was consumed
        self.a_slot = [None] * AS
        self.a_reads = [0] * AS
        self.b_slot = [None] * BS
        self.b_used = [True] * BS
        self.c_slot = [[None] * W for _ in range(CS)]
        self.c_used = [True] * CS
        self.s_slot = [None] * SSL
        self.s_reads = [0] * SSL
        self.acc = [None] * NB          # slices summed into each TMEM accumulator
        self.events = []                # asynchronous completions: (order key, fn)
        self.mma_queue = {0: [], 1: []} # per issuer, completions in issue order
        self.nslices = sum(units)
        # A stages: a_per consecutive slices of one unit each
        self.stages, self.stage_of = [], {}
        base = 0
        for nsl in units:
            for l in range(0, nsl, self.a_per):
                sl = tuple(range(base + l, base + min(nsl, l + self.a_per)))
                for h, ia in enumerate(sl):
                    self.stage_of[ia] = (len(self.stages), h, len(sl))
                self.stages.append(sl)
            base += nsl

    # ------------------------------------------------------------- roles
    def producer_a(self):
        for st, sl in enumerate(self.stages):
            s = st % self.AS
            yield self.a_empty[s], ((st // self.AS) & 1) ^ 1
            check(st < self.AS or (self.a_slot[s] == self.stages[st - self.AS] and
                                   self.a_reads[s] == (1 if self.f8f8 else self.wpg * self.a_per)),
                  "A stage %d refilled with slices %s before slices %s were read by every "
                  "decode warp" % (s, sl, self.a_slot[s]))
            self.a_reads[s] = 0

            def fill(s=s, sl=sl):
                self.a_slot[s] = sl
                self.a_full[s].arrive()
            self.events.append(fill)

    def producer_b(self):
        for ib in range(self.nslices):
            s = ib % self.BS
            yield self.b_empty[s], ((ib // self.BS) & 1) ^ 1
            check(self.b_used[s], "B slot %d refilled for slice %d before the MMA read slice %s"
                  % (s, ib, self.b_slot[s]))

            def fill(s=s, ib=ib):
                self.b_slot[s], self.b_used[s] = ib, False
                self.b_full[s].arrive()
            self.events.append(fill)

    def scale_loader(self):
        for i in range(self.nslices):
            s = i % self.SSL
            yield self.s_empty[s], ((i // self.SSL) & 1) ^ 1
            check(i < self.SSL or (self.s_slot[s] == i - self.SSL and
                                   self.s_reads[s] == 1),
                  "scale slot %d republished before its slice was read" % s)
            self.s_slot[s], self.s_reads[s] = i, 0
            self.s_full[s].arrive()

    def decode_warp(self, grp, w):
        for ia in range(self.nslices):
            if ia % self.ndg != grp:
                continue
            st, h, n = self.stage_of[ia]
            sa, sc = st % self.AS, ia % self.CS
            yield self.a_full[sa], (st // self.AS) & 1
            check(self.a_slot[sa] is not None and len(self.a_slot[sa]) > h and
                  self.a_slot[sa][h] == ia,
                  "decode of slice %d read A stage %d holding slices %s" % (ia, sa, self.a_slot[sa]))
            yield self.c_empty[sc], ((ia // self.CS) & 1) ^ 1
            check(self.c_used[sc], "decode of slice %d overwrote C slot %d (slice %s) before "
                  "the MMA read it" % (ia, sc, self.c_slot[sc][w]))
            arrivals = 2 if (n < self.a_per and self.double_arrival) else 1
            for _ in range(arrivals):
                self.a_reads[sa] += 1
                self.a_empty[sa].arrive()
            yield None                                  # the decode itself
            self.c_slot[sc][w] = ia
            if all(v == ia for v in self.c_slot[sc]):
                self.c_used[sc] = False
            self.c_full[sc].arrive()

    def issuer(self, mine):
        ia = ib = au = 0
        for nsl in self.units:
            ubuf = None
            ia0 = ia
            if not self.promote:
                tb = 2 * au + mine
                ubuf = tb % self.NB
                yield self.t_empty[ubuf], ((tb // self.NB) & 1) ^ 1
                none = (nsl <= mine) if self.old else (nsl == 1 and ia0 % 2 != mine)
                if none:
                    self._commit(mine, self.t_full[ubuf])
            first = True
            for l in range(nsl):
                take = (ia % 2 == mine) if (self.promote or not self.old) else (l % 2 == mine)
                if not take:
                    ia += 1
                    ib += 1
                    if self.promote:
                        au += 1
                    continue
                buf = au % self.NB if self.promote else ubuf
                if self.promote:
                    yield self.t_empty[buf], ((au // self.NB) & 1) ^ 1
                if self.f8f8:
                    sa = ia % self.AS
                    yield self.a_full[sa], (ia // self.AS) & 1
                    check(self.a_slot[sa] is not None and self.a_slot[sa][0] == ia,
                          "MMA of slice %d read A slot %d holding slice %s" % (ia, sa, self.a_slot[sa]))

                    def done(sa=sa, buf=buf, ia=ia):
                        self.acc[buf] = [ia]
                        self.a_reads[sa] += 1
                        self.a_empty[sa].arrive()
                    self.mma_queue[mine].append(done)
                    ia += 1
                    ib += 1
                    self._commit(mine, self.t_full[buf])
                    au += 1
                    continue
                sa, sb = ia % self.CS, ib % self.BS
                yield self.c_full[sa], (ia // self.CS) & 1
                check(all(v == ia for v in self.c_slot[sa]),
                      "MMA of slice %d read C slot %d holding %s" % (ia, sa, self.c_slot[sa]))
                yield self.b_full[sb], (ib // self.BS) & 1
                check(self.b_slot[sb] == ib, "MMA of slice %d read B slot %d holding slice %s"
                      % (ib, sb, self.b_slot[sb]))
                fresh = self.promote or (first if not self.old else l == mine)
                first = False

                def done(sa=sa, sb=sb, buf=buf, ia=ia, fresh=fresh):
                    self.acc[buf] = [ia] if fresh else (self.acc[buf] or []) + [ia]
                    self.c_used[sa] = True
                    self.b_used[sb] = True
                    self.c_empty[sa].arrive()
                    self.b_empty[sb].arrive()
                self.mma_queue[mine].append(done)
                ia += 1
                ib += 1
                if self.promote:
                    self._commit(mine, self.t_full[buf])
                    au += 1
                elif l + 2 >= nsl:
                    self._commit(mine, self.t_full[buf])
            if not self.promote:
                au += 1

    def _commit(self, mine, bar):
        # tcgen05.commit: arrives once every earlier MMA of this thread is done
        self.mma_queue[mine].append(lambda bar=bar: bar.arrive())

    def epilogue(self):
        au = esl = 0
        base = 0
        for nsl in self.units:
            slices = list(range(base, base + nsl))
            if self.promote:
                for k in slices:
                    buf = au % self.NB
                    if self.epi_scales:
                        ss = k % self.SSL
                        yield self.s_full[ss], (k // self.SSL) & 1
                        check(self.s_slot[ss] == k, "epilogue of slice %d read scales of slice %s"
                              % (k, self.s_slot[ss]))
                        self.s_reads[ss] += 1
                        self.s_empty[ss].arrive()
                    yield self.t_full[buf], (au // self.NB) & 1
                    check(self.acc[buf] == [k], "epilogue of slice %d read accumulator %s"
                          % (k, self.acc[buf]))
                    self.t_empty[buf].arrive()
                    au += 1
            else:
                tb0, tb1 = 2 * au, 2 * au + 1
                b0, b1 = tb0 % self.NB, tb1 % self.NB
                yield self.t_full[b0], (tb0 // self.NB) & 1
                yield self.t_full[b1], (tb1 // self.NB) & 1
                two = nsl >= 2
                if two:
                    got = sorted((self.acc[b0] or []) + (self.acc[b1] or []))
                else:
                    rd = b1 if (not self.old and (esl & 1)) else b0
                    got = sorted(self.acc[rd] or [])
                check(got == slices, "epilogue of unit with slices %s read %s" % (slices, got))
                self.t_empty[b0].arrive()
                self.t_empty[b1].arrive()
                au += 1
                esl += nsl
            base += nsl

    # --------------------------------------------------------- scheduler
    def run(self, rng, max_steps=200000):
        actors = [self.producer_a(), self.issuer(0), self.issuer(1), self.epilogue()]
        if not self.f8f8:
            actors.append(self.producer_b())     # bf16 tokens
        if self.epi_scales:
            actors.append(self.scale_loader())
        for g in range(self.ndg):
            for w in range(self.wpg):
                actors.append(self.decode_warp(g, w))
        waits = {}
        for a in actors:
            waits[id(a)] = self._advance(a, None)
        live = [a for a in actors if waits[id(a)] is not StopIteration]
        for _ in range(max_steps):
            ready = [a for a in live if waits[id(a)] is None or waits[id(a)][0].passes(waits[id(a)][1])]
            choices = [("actor", a) for a in ready]
            choices += [("event", i) for i in range(len(self.events))]
            choices += [("mma", m) for m in (0, 1) if self.mma_queue[m]]
            if not choices:
                if live:
                    names = [waits[id(a)][0].name for a in live if waits[id(a)] is not None]
                    raise Violation("deadlock: roles wait on %s" % names)
                return
            kind, x = rng.choice(choices)
            if kind == "actor":
                waits[id(x)] = self._advance(x, True)
                if waits[id(x)] is StopIteration:
                    live.remove(x)
            elif kind == "event":
                self.events.pop(x)()
            else:
                self.mma_queue[x].pop(0)()
        raise Violation("no progress within the step budget")

    @staticmethod
    def _advance(gen, _):
        try:
            return next(gen)
        except StopIteration:
            return StopIteration


UNIT_PATTERNS = {
    "odd": [3, 3, 5, 3, 1, 3],
    "even": [2, 4, 2, 6],
    "mixed": [1, 2, 3, 1, 1, 4, 5, 2],
    "ones": [1, 1, 1, 1, 1],
}


@pytest.mark.parametrize("pattern", sorted(UNIT_PATTERNS))
@pytest.mark.parametrize("kind", ["mxfp4_whole_k", "fp8_block_promoted", "per_tensor_whole_k"])
@pytest.mark.parametrize("ndg", [1, 2])
@pytest.mark.parametrize("AS,BS,CS", [(12, 4, 4), (8, 8, 6), (4, 8, 4), (5, 4, 6)])
def test_ring_protocol_holds_under_random_interleavings(pattern, kind, ndg, AS, BS, CS):
    units = UNIT_PATTERNS[pattern]
    promote = kind == "fp8_block_promoted"
    mxw = kind == "mxfp4_whole_k"
    for seed in range(40):
        cta = Cta(units, promote=promote, ndg=ndg, mxw=mxw, AS=AS, BS=BS, CS=CS)
        cta.run(random.Random(seed))


def test_model_finds_the_lap_behind_read_of_a_three_stage_ring():
    """Two consumers taking alternate slices of one ring (the two decode
    groups, or the two MMA issuers of FP8 x FP8) with only three stages: a
    consumer can wait on a stage whose previous fill (the other consumer's
    slice) has not landed, and its parity wait passes one lap early.  The
    kernel's rings are four stages deep or more (asserted at compile time)."""
    found = 0
    for pat in UNIT_PATTERNS:
        for seed in range(100):
            try:
                Cta(UNIT_PATTERNS[pat], promote=True, ndg=2, mxw=False, AS=3, BS=8).run(random.Random(seed))
            except Violation:
                found += 1
    assert found > 0


def test_model_finds_a_missing_second_arrival_of_a_one_slice_stage():
    """MXFP4 stages of two slices of a unit: a unit of odd length ends on a
    stage with one slice.  Without its decode group's second arrival on the
    stage's empty barrier, the producer never gets the stage back, and the
    model reports the deadlock."""
    units = UNIT_PATTERNS["odd"]
    with pytest.raises(Violation, match="deadlock"):
        Cta(units, promote=False, ndg=2, mxw=True, AS=4, double_arrival=False).run(random.Random(0))
    Cta(units, promote=False, ndg=2, mxw=True, AS=4).run(random.Random(0))


def test_model_finds_the_stale_read_of_the_per_unit_issuer_rule():
    """Whole-K issuers taking a unit's slices by their parity inside the unit,
    with the decode in two groups taking global slice parity, and units of
    odd length: some interleaving lets an issuer pass a C-ring wait one lap
    early (or the epilogue read the wrong buffer), and the model says so."""
    found = 0
    for seed in range(300):
        cta = Cta(UNIT_PATTERNS["odd"], promote=False, ndg=2, mxw=True, old_issuer_rule=True)
        try:
            cta.run(random.Random(seed))
        except Violation:
            found += 1
    assert found > 0
    # the same schedules are clean with the rule the kernel uses now
    for seed in range(300):
        Cta(UNIT_PATTERNS["odd"], promote=False, ndg=2, mxw=True).run(random.Random(seed))


@pytest.mark.parametrize("AS,NB,ring", [(6, 4, False), (5, 2, False), (10, 4, True),
                                        (12, 4, True)])
@pytest.mark.parametrize("pattern", ["even", "odd", "mixed", "ones"])
def test_ring_protocol_fp8_x_fp8(AS, NB, ring, pattern):
    """FP8 x FP8 W8A8: token-major tiles of 128 (6 stages, 4 accumulator
    buffers) and 192 (5 stages, 2 buffers), whose epilogue reads its own slice
    scales, and weight-major decode tiles (10-12 stages, 4 buffers) fed by the
    scale ring."""
    for seed in range(40):
        cta = Cta(UNIT_PATTERNS[pattern], promote=True, ndg=0, mxw=False, AS=AS, NB=NB, f8f8=True,
                  scale_ring=ring)
        cta.run(random.Random(seed))
