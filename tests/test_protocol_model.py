"""A model of the prefix kernel's mbarrier protocol, run under random interleavings.

The kernel's roles (producers, the score-MMA issuer, two softmax sets, in both
CTAs of a pair, plus each CTA's in-order tensor pipe) are modelled as
generators that wait on barriers exactly where the kernel waits.  Barriers keep
the hardware's parity semantics: a wait for phase k succeeds when the
completed-phase count has the other parity; a wait that falls two or more
phases behind would misread, and the model reports it.  The model also checks
the buffers the barriers protect: the one P buffer, the one exchange buffer per
CTA, the two score buffers and the stage ring.  It finds no deadlock and no
hazard for many step counts, and it catches each of a set of planted protocol
mistakes (a dropped wait, a wrong parity) -- so the checks have teeth.

A CTA runs several passes (a unit's 16-bit pass and its 20-bit rerun, or the
units of the persistent launch) on the same barriers.  Arrivals that are
asynchronous in the kernel -- tensor-core commits and the relaxed remote arrive
that hands the exchange buffer back -- are delivered late and in any order, even
after the pass that made them has ended.  With barrier phases that run on across
passes (each pass numbers its steps from the CTA's running step count) no
hazard appears; re-initialising the barriers between passes, as a first version
did, is caught: a late arrival lands on the new pass's phases.
"""
import random

import pytest

K_STAGES = 5


class Hazard(Exception):
    pass


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.arr, self.done, self.tx = name, count, 0, 0, 0

    def arrive(self):
        self.arr += 1
        self._check()

    def expect(self, tx):
        self.tx += tx
        self.arrive()

    def complete_tx(self, tx):
        self.tx -= tx
        self._check()

    def _check(self):
        if self.arr == self.count and self.tx == 0:
            self.arr = 0
            self.done += 1


def wait(bar, k):
    def pred():
        if bar.done >= k + 2:
            raise Hazard(f"{bar.name}: wait for phase {k} with {bar.done} phases completed")
        return (bar.done & 1) != (k & 1) and bar.done >= k + 1
    return pred


class CTA:
    def __init__(self, name):
        B = lambda n, c=1: Bar(f"{name}.{n}", c)
        self.name = name
        self.k_full = [B(f"k_full{i}") for i in range(K_STAGES)]
        self.k_empty = [B(f"k_empty{i}") for i in range(K_STAGES)]
        self.s_full = [B(f"s_full{i}") for i in range(2)]
        self.s_free = [B(f"s_free{i}") for i in range(2)]
        self.p_ready = [B(f"p_ready{i}") for i in range(2)]
        self.m_ready = [B(f"m_ready{i}") for i in range(2)]
        self.x_full = [B(f"x_full{i}") for i in range(2)]
        self.x_free = [B(f"x_free{i}") for i in range(2)]
        self.q_ready = B("q_ready", 2)
        self.pipe = []
        self.pv_next = 0
        self.stage = [None] * K_STAGES   # step whose keys sit in each ring stage
        self.sbuf = [None, None]         # step whose scores sit in each S buffer
        self.sread = [True, True]
        self.pbuf = None                 # step whose P sits in the P buffer
        self.xbuf, self.xread = None, True
        self.o_steps = 0                 # P.V groups accumulated into O
        self.late = []                   # asynchronous arrivals still in flight

    def bars(self):
        return (self.k_full + self.k_empty + self.s_full + self.s_free + self.p_ready + self.m_ready + self.x_full
                + self.x_free + [self.q_ready])

    def reinit(self):
        for b in self.bars():
            b.arr = b.done = b.tx = 0
        self.pv_next = 0


def producer(c, passes, sync):
    for p, (G, n, _) in enumerate(passes):
        for g in range(G, G + n):
            st = g % K_STAGES
            if g >= K_STAGES:
                yield wait(c.k_empty[st], g // K_STAGES - 1)
            c.stage[st] = g
            c.k_full[st].arrive()
        yield from sync(p)


def s_issuer(c, passes, mut, sync):
    for p, (G, n, qp) in enumerate(passes):
        yield wait(c.q_ready, qp)
        for g in range(G, G + n):
            yield wait(c.k_full[g % K_STAGES], g // K_STAGES)
            if g > 1 and mut != "s_buffer_no_wait":
                yield wait(c.s_free[g % 2], (g - 2) // 2)
            c.pipe.append(("S", g))
            c.pipe.append(("commit", c.s_full[g % 2]))
        yield (lambda: not c.pipe)       # its MMAs have run (the drain); their arrivals may still travel
        yield from sync(p)


def softmax(c, peer, sset, passes, mut, sync):
    for p, (G, n, _) in enumerate(passes):
        c.q_ready.arrive()
        c.o_steps = 0
        for g in range(G + ((sset ^ G) & 1), G + n, 2):
            sb = g % 2
            c.x_full[sb].expect(1)
            yield wait(c.s_full[sb], g // 2)
            if c.sbuf[sb] != g:
                raise Hazard(f"{c.name}: S buffer {sb} holds step {c.sbuf[sb]}, set reads {g}")
            c.sread[sb] = True
            c.s_free[sb].arrive()
            if g >= 1 and mut != "exchange_no_wait":
                yield wait(c.x_free[sb ^ 1], (g - 1) // 2)
            if not peer.xread:
                raise Hazard(f"{c.name}: step {g} overwrote the peer's unread step {peer.xbuf}")
            peer.xbuf, peer.xread = g, False
            peer.x_full[sb].complete_tx(1)
            yield wait(c.x_full[sb], g // 2)
            if c.xbuf != g:
                raise Hazard(f"{c.name}: exchange buffer holds {c.xbuf}, step {g} expected")
            c.xread = True
            peer.late.append(peer.x_free[sb])          # relaxed remote arrive: in flight
            if g > 0:
                k = g - 1 if mut != "m_parity" else g
                yield wait(c.m_ready[k % 2], k // 2)
            c.m_ready[sb].arrive()
            if g >= 1 and mut != "p_buffer_no_wait":
                yield wait(c.k_empty[(g - 1) % K_STAGES], (g - 1) // K_STAGES)
            c.pbuf = g
            c.p_ready[sb].arrive()
            yield wait(c.p_ready[sb], g // 2)
            yield (lambda g=g: c.pv_next == g)
            c.pipe.append(("PV", g))
            c.pipe.append(("commit", c.k_empty[g % K_STAGES]))
            c.pv_next = g + 1
        last = G + n - 1
        yield wait(c.k_empty[last % K_STAGES], last // K_STAGES)
        if c.o_steps != n:
            raise Hazard(f"{c.name}: epilogue reads O after {c.o_steps} of {n} P.V groups")
        yield (lambda: not c.pipe)
        yield from sync(p)


def pipe_step(c):
    op = c.pipe.pop(0)
    if op[0] == "commit":
        c.late.append(op[1])             # the commit's arrive fires when the MMAs finish: in flight
    elif op[0] == "S":
        g = op[1]
        if c.stage[g % K_STAGES] != g:
            raise Hazard(f"{c.name}: S({g}) reads stage holding step {c.stage[g % K_STAGES]}")
        if not c.sread[g % 2]:
            raise Hazard(f"{c.name}: S({g}) overwrites unread scores of step {c.sbuf[g % 2]}")
        c.sbuf[g % 2], c.sread[g % 2] = g, False
    else:
        g = op[1]
        if c.pbuf != g:
            raise Hazard(f"{c.name}: P.V({g}) reads P of step {c.pbuf}")
        if c.stage[g % K_STAGES] != g:
            raise Hazard(f"{c.name}: P.V({g}) reads stage holding step {c.stage[g % K_STAGES]}")
        c.o_steps += 1


def run(n, seed, mut=None, passes=None, reinit=False, lag=1):
    """One unit of n steps, or the given passes [(steps, ...)] run back to back by both CTAs.

    reinit: set the barriers up again between passes (each pass then numbers its steps
    from 0) instead of letting their phases run on; "drained": the same, but only after every
    in-flight arrival has landed.  lag: how much likelier a role's move
    is than the delivery of one in-flight arrival."""
    rnd = random.Random(seed)
    A, B = CTA("A"), CTA("B")
    counts = passes or [n]
    plan, G = [], 0
    for p, m in enumerate(counts):
        # (first step, steps, phase of the q_ready barrier)
        plan.append((0, m, 0) if reinit else (G, m, p))
        G += m
    n_roles = 8
    arrived = [0] * len(plan)

    def sync(p):
        # the end-of-pass cluster barrier: every role of both CTAs; a re-initialising version sets the
        # barriers up again once all have arrived
        arrived[p] += 1
        if arrived[p] == n_roles and reinit:
            while reinit == "drained" and (A.late or B.late):
                (A.late or B.late).pop(0).arrive()
            A.reinit()
            B.reinit()
        yield (lambda p=p: arrived[p] == n_roles)

    roles = []
    for c, peer in ((A, B), (B, A)):
        roles += [producer(c, plan, sync), s_issuer(c, plan, mut, sync), softmax(c, peer, 0, plan, mut, sync),
                  softmax(c, peer, 1, plan, mut, sync)]
    waits = [None] * len(roles)
    alive = list(range(len(roles)))
    while alive or A.pipe or B.pipe or A.late or B.late:
        acts = [("role", i) for i in alive if waits[i] is None or waits[i]()]
        acts += [("pipe", c) for c in (A, B) if c.pipe]
        acts += [("late", c) for c in (A, B) if c.late]
        if not acts:
            raise Hazard(f"deadlock: roles {alive} all waiting")
        # in-flight arrivals are drawn less often than the roles' moves, so that some of them lag far
        kind, x = rnd.choices(acts, [1 if a[0] == "late" else lag for a in acts])[0]
        if kind == "pipe":
            pipe_step(x)
            continue
        if kind == "late":
            x.late.pop(rnd.randrange(len(x.late))).arrive()
            continue
        try:
            waits[x] = next(roles[x])
        except StopIteration:
            alive.remove(x)


@pytest.mark.parametrize("n", [1, 2, 3, 5, 6, 11, 16])
def test_protocol_has_no_deadlock_or_hazard(n):
    for seed in range(60):
        run(n, seed)


@pytest.mark.parametrize("mut", ["s_buffer_no_wait", "exchange_no_wait", "m_parity", "p_buffer_no_wait"])
def test_planted_protocol_mistakes_are_caught(mut):
    caught = False
    for n in (6, 11):
        for seed in range(60):
            try:
                run(n, seed, mut)
            except Hazard:
                caught = True
                break
        if caught:
            break
    assert caught, mut


@pytest.mark.parametrize("lag", [1, 16])
@pytest.mark.parametrize("passes", [[6, 6], [5, 11, 3], [1, 2, 7, 4]])
def test_passes_with_running_phases_survive_late_arrivals(passes, lag):
    for seed in range(60):
        run(0, seed, passes=passes, lag=lag)


def test_reinitialising_barriers_between_passes_is_caught():
    # a late arrival of one pass lands on the freshly set-up barriers of the next
    caught = []
    for passes in ([6, 6], [5, 11, 3]):
        for seed in range(60):
            try:
                run(0, seed, passes=passes, reinit=True, lag=16)
            except Hazard as e:
                caught.append(str(e))
    assert caught


def test_reinitialising_after_every_arrival_landed_is_safe():
    # the same set-up again is harmless once nothing is in flight: the hazard above is the late arrival
    for passes in ([6, 6], [5, 11, 3]):
        for seed in range(60):
            run(0, seed, passes=passes, reinit="drained", lag=16)
