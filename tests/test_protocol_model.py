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


def producer(c, n):
    for g in range(n):
        st = g % K_STAGES
        if g >= K_STAGES:
            yield wait(c.k_empty[st], g // K_STAGES - 1)
        c.stage[st] = g
        c.k_full[st].arrive()


def s_issuer(c, n, mut):
    yield wait(c.q_ready, 0)
    for g in range(n):
        yield wait(c.k_full[g % K_STAGES], g // K_STAGES)
        if g > 1 and mut != "s_buffer_no_wait":
            yield wait(c.s_free[g % 2], (g - 2) // 2)
        c.pipe.append(("S", g))
        c.pipe.append(("commit", c.s_full[g % 2]))


def softmax(c, peer, sset, n, mut):
    c.q_ready.arrive()
    for g in range(sset, n, 2):
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
        peer.x_free[sb].arrive()
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
    last = n - 1
    yield wait(c.k_empty[last % K_STAGES], last // K_STAGES)
    if c.o_steps != n:
        raise Hazard(f"{c.name}: epilogue reads O after {c.o_steps} of {n} P.V groups")


def pipe_step(c):
    op = c.pipe.pop(0)
    if op[0] == "commit":
        op[1].arrive()
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


def run(n, seed, mut=None):
    rnd = random.Random(seed)
    A, B = CTA("A"), CTA("B")
    roles = []
    for c, peer in ((A, B), (B, A)):
        roles += [producer(c, n), s_issuer(c, n, mut), softmax(c, peer, 0, n, mut), softmax(c, peer, 1, n, mut)]
    waits = [None] * len(roles)
    alive = list(range(len(roles)))
    while alive or A.pipe or B.pipe:
        acts = [("role", i) for i in alive if waits[i] is None or waits[i]()]
        acts += [("pipe", c) for c in (A, B) if c.pipe]
        if not acts:
            raise Hazard(f"deadlock: roles {alive} all waiting")
        kind, x = rnd.choice(acts)
        if kind == "pipe":
            pipe_step(x)
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
