"""A CPU model of the forward kernel's barrier protocol, run under adversarial interleavings.

The forward kernel's roles (the TMA copy thread, the MMA-issuing thread and the softmax
warpgroups) hand work to one another through mbarriers and wait with parity waits.  A parity
wait is only right while the barrier is at most one phase away from the phase it waits for;
beyond that it passes early or blocks forever.  The kernel's comments state, per wait, why
that window holds (e.g. "S(G) complete implies PV(G - 2) complete").  This test replays the
MMA issue order and the softmax loop of `fwd_kernel` (two query tiles per unit, including
one-tile units in the same CTA; and the d = 256 schedule with two S buffers).  MMAs complete in issue order after random delays; the
scheduler starves one role at a time.  At every parity wait the test asserts that the barrier
is exactly at the awaited phase, and it asserts that no run deadlocks.
"""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.pend, self.phase = count, 0, 0

    def arrive(self, n=1):
        self.pend += n
        assert self.pend <= self.count, "more arrivals than the barrier's count"
        if self.pend == self.count:
            self.pend = 0
            self.phase += 1

    def passes(self, parity):  # mbarrier.try_wait.parity
        return (self.phase & 1) != parity


def units_of_cta(cta, grid, bh, n, causal, rows_per_unit):
    """The units one persistent CTA walks (heaviest first when causal, boustrophedon)."""
    ncb = (n + rows_per_unit - 1) // rows_per_unit
    n_kv_all = (n + 127) // 128
    out, r = [], 0
    while True:
        u = r * grid + ((grid - 1 - cta) if (r & 1) else cta)
        if u >= bh * ncb:
            return out
        cb = (ncb - 1 - u // bh) if causal else u // bh
        q0 = cb * rows_per_unit
        last = min(q0 + rows_per_unit - 1, n - 1)
        n_kv = min(n_kv_all, last // 128 + 1) if causal else n_kv_all
        two = rows_per_unit == 256 and n - q0 > 128
        out.append(dict(n=max(1, n_kv), two=two))
        r += 1


class Machine:
    def __init__(self, seed, stages):
        self.rnd = random.Random(seed)
        self.stages = stages
        self.full = [Bar(1) for _ in range(stages)]
        self.empty = [Bar(1) for _ in range(stages)]
        self.q_full, self.q_empty = Bar(1), Bar(1)
        self.s_full = [Bar(1), Bar(1)]
        self.p_full = [Bar(128), Bar(128)]
        self.o_bar = [Bar(1), Bar(1)]
        self.o_free = [Bar(128), Bar(128)]
        self.now, self.last_done, self.queue = 0, 0, []

    def commit(self, bars):  # tcgen05.commit: arrives once every MMA issued so far has completed
        t = max(self.now, self.last_done) + self.rnd.randint(1, 4)
        self.last_done = t
        self.queue.append((t, bars))

    def wait(self, bar, index):
        """Yieldable parity wait for phase `index`; checks the one-phase window on passing."""
        def ready():
            return bar.passes(index & 1)
        return ready, (bar, index)

    def run(self, agents):
        waits = [None] * len(agents)
        alive = [True] * len(agents)
        starve, step = None, 0
        while any(alive):
            progressed = False
            while self.queue and self.queue[0][0] <= self.now:
                for b in self.queue.pop(0)[1]:
                    b.arrive()
                progressed = True
            if step % 150 == 0:
                starve = self.rnd.choice([None] + list(range(len(agents))))
            order = list(range(len(agents)))
            self.rnd.shuffle(order)
            for a in order:
                if not alive[a] or (a == starve and self.rnd.random() < 0.97):
                    continue
                if waits[a] is not None:
                    ready, (bar, index) = waits[a]
                    if not ready():
                        continue
                    assert bar.phase == index + 1, "parity wait passed outside its window"
                try:
                    waits[a] = next(agents[a])
                except StopIteration:
                    alive[a], waits[a] = False, None
                progressed = True
            self.now += 1
            step += 1
            if not progressed and not self.queue:
                if starve is None:
                    raise AssertionError("deadlock: %s" % alive)
                starve = None
            assert step < 2_000_000, "did not finish"


def two_tile_agents(m, units):
    """fwd_kernel with two query tiles per unit (d = 64 / 128): producer, MMA warp, 2 softmax WGs."""
    S = m.stages

    def producer():
        it = q = 0
        for u in units:
            if q:
                yield m.wait(m.q_empty, q - 1)
            m.q_full.arrive()
            q += 1
            for _ in range(2 * u["n"]):
                if it >= S:  # the slot's previous load has been consumed
                    yield m.wait(m.empty[it % S], it // S - 1)
                m.full[it % S].arrive()
                it += 1

    def mma():
        it = nu = nu2 = 0
        g = [0, 0]
        for u in units:
            n, two, it0 = u["n"], u["two"], it
            yield m.wait(m.q_full, nu)
            yield m.wait(m.full[it0 % S], it0 // S)
            m.commit([m.s_full[0]])
            if two:
                m.commit([m.s_full[1]])
            if n == 1:
                m.commit([m.q_empty])
            m.commit([m.empty[it0 % S]])
            if nu:
                yield m.wait(m.o_free[0], nu - 1)
            if two and nu2:
                yield m.wait(m.o_free[1], nu2 - 1)
            for j in range(n):
                more = j + 1 < n
                itv, itk = it0 + 2 * j + 1, it0 + 2 * j + 2
                yield m.wait(m.full[itv % S], itv // S)
                yield m.wait(m.p_full[0], g[0] + j)
                m.commit([m.o_bar[0]])  # PV0(j)
                if more:
                    yield m.wait(m.full[itk % S], itk // S)
                    m.commit([m.s_full[0]])  # S0(j + 1)
                if two:
                    yield m.wait(m.p_full[1], g[1] + j)
                    m.commit([m.o_bar[1]])
                m.commit([m.empty[itv % S]])
                if more:
                    if two:
                        m.commit([m.s_full[1]])
                    if j + 2 == n:
                        m.commit([m.q_empty])
                    m.commit([m.empty[itk % S]])
            it += 2 * n
            g[0] += n
            nu += 1
            if two:
                g[1] += n
                nu2 += 1

    def softmax(w):
        jg = 0
        for u in units:
            if w == 1 and not u["two"]:
                continue
            for j in range(u["n"]):
                yield m.wait(m.s_full[w], jg)
                if j > 0 and m.rnd.random() < 0.3:  # conditional rescale: PV(j - 1) complete
                    yield m.wait(m.o_bar[w], jg - 1)
                m.p_full[w].arrive(128)
                jg += 1
            yield m.wait(m.o_bar[w], jg - 1)  # epilogue
            m.o_free[w].arrive(128)

    return [producer(), mma(), softmax(0), softmax(1)]


def two_buffer_agents(m, units):
    """fwd_kernel at d = 256: one query tile, key tile G in S buffer G mod 2, K and V copied by
    two threads (ring slot 0 holds K, slot 1 holds V)."""
    def copier(kind):
        it = q = 0
        for u in units:
            if kind == 0:
                if q:
                    yield m.wait(m.q_empty, q - 1)
                m.q_full.arrive()
                q += 1
            for jj in range(2 * u["n"]):
                if (jj & 1) == kind:
                    if it >= 2:
                        yield m.wait(m.empty[it % 2], it // 2 - 1)
                    m.full[it % 2].arrive()
                it += 1

    def mma():
        it = nu = g = 0
        for u in units:
            n, it0 = u["n"], it
            yield m.wait(m.q_full, nu)
            yield m.wait(m.full[it0 % 2], it0 // 2)
            m.commit([m.s_full[g & 1]])
            if n == 1:
                m.commit([m.q_empty])
            m.commit([m.empty[it0 % 2]])
            if nu:
                yield m.wait(m.o_free[0], nu - 1)
            for j in range(n):
                G = g + j
                if j + 1 < n:
                    itk = it0 + 2 * (j + 1)
                    yield m.wait(m.full[itk % 2], itk // 2)
                    m.commit([m.s_full[(G + 1) & 1]])
                    if j + 2 == n:
                        m.commit([m.q_empty])
                    m.commit([m.empty[itk % 2]])
                itv = it0 + 2 * j + 1
                yield m.wait(m.full[itv % 2], itv // 2)
                yield m.wait(m.p_full[G & 1], G >> 1)
                m.commit([m.o_bar[G & 1]])
                m.commit([m.empty[itv % 2]])
            it += 2 * n
            g += n
            nu += 1

    def softmax():
        jg = 0
        for u in units:
            for j in range(u["n"]):
                yield m.wait(m.s_full[jg & 1], jg >> 1)
                if j > 0 and m.rnd.random() < 0.3:
                    yield m.wait(m.o_bar[(jg - 1) & 1], (jg - 1) >> 1)
                m.p_full[jg & 1].arrive(128)
                jg += 1
            yield m.wait(m.o_bar[(jg - 1) & 1], (jg - 1) >> 1)
            m.o_free[0].arrive(128)

    return [copier(0), copier(1), mma(), softmax()]


SHAPES = [(1, 3, 333), (2, 8, 640), (3, 50, 129), (1, 200, 300), (2, 40, 1100)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_two_tile_schedule_windows(shape, causal):
    B, H, N = shape
    grid = min(152, B * H * ((N + 255) // 256))
    for cta in range(0, grid, max(1, grid // 6)):
        units = units_of_cta(cta, grid, B * H, N, causal, 256)
        for seed in range(3):
            m = Machine(seed, stages=4)
            m.run(two_tile_agents(m, units))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_two_s_buffer_schedule_windows(shape, causal):
    B, H, N = shape
    grid = min(152, B * H * ((N + 127) // 128))
    for cta in range(0, grid, max(1, grid // 6)):
        units = units_of_cta(cta, grid, B * H, N, causal, 128)
        for seed in range(3):
            m = Machine(seed, stages=2)
            m.run(two_buffer_agents(m, units))


def test_model_catches_a_window_violation():
    """The checks have teeth: waiting the rescale on the wrong phase (PV(j - 2) instead of
    PV(j - 1), a plausible off-by-one) trips the window assertion or deadlocks."""
    units = units_of_cta(0, 1, 1, 2048, False, 256)
    m = Machine(0, stages=4)
    agents = two_tile_agents(m, units)

    def bad_softmax(w):
        jg = 0
        for u in units:
            for j in range(u["n"]):
                yield m.wait(m.s_full[w], jg)
                if j > 1:
                    yield m.wait(m.o_bar[w], jg - 2)
                    yield m.wait(m.o_bar[w], jg - 2)  # the same phase twice: the second is out of window
                m.p_full[w].arrive(128)
                jg += 1
            yield m.wait(m.o_bar[w], jg - 1)
            m.o_free[w].arrive(128)

    agents[2] = bad_softmax(0)
    with pytest.raises(AssertionError):
        m.run(agents)
