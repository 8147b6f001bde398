"""Host model of the attention kernel's barrier protocol (free_block_sparse_gb300/csrc/bsattn.cu).

A parity wait on an mbarrier (try_wait.parity with the parity of phase k) is only right when the
barrier has completed either exactly k phases (not yet: keep waiting) or k + 1 (done).  With k - 1
completed phases the parities alias and the wait passes early; with k + 2 it never passes.  This
model runs the kernel's roles - producer, score issuer, P.V issuer and the softmax warps - against
counters of completed phases, with the tensor-core products and TMA copies completing
asynchronously (each issuing thread's products in its own issue order, no order between the two
issuers), under random schedules, and checks that invariant at every wait and that every schedule
finishes.  A second model puts back the single P.V-completion barrier that the O rescale once
waited on and shows that with three score buffers the checker catches the aliasing."""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phases = 0  # completed phases

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.phases += 1
            self.pending = self.count


class Aliased(AssertionError):
    pass


class Model:
    """The kernel's protocol for one CTA and a row of T kept tiles."""

    def __init__(self, T, KST, VST, NSB=2, JRING=8, rescale_on="buffer", seed=0):
        self.T, self.KST, self.VST, self.NSB, self.J = T, KST, VST, NSB, JRING
        self.rescale_on = rescale_on
        self.rng = random.Random(seed)
        B = Barrier
        self.k_full = [B(1) for _ in range(KST)]
        self.k_empty = [B(1) for _ in range(KST)]
        self.v_full = [B(1) for _ in range(VST)]
        self.v_empty = [B(1) for _ in range(VST)]
        self.j_full = [B(1) for _ in range(JRING)]
        self.j_empty = [B(4) for _ in range(JRING)]
        self.s_full = [B(1) for _ in range(NSB)]
        self.p_full = [B(128) for _ in range(NSB)]
        self.pv_done = [B(1) for _ in range(NSB)]
        self.o_done = B(1)     # the former single P.V-completion barrier (second model only)
        self.q_full = B(128)
        self.mma_done = B(1)
        self.row_end = -1
        self.async_ops = []    # pending completions: (thread, list of barriers to arrive on)
        self.order = {"s": [], "pv": [], "tma": []}

    # a parity wait for phase k: returns True when done, False to keep waiting; raises on aliasing
    def wait(self, bar, k):
        c = bar.phases
        if c == k - 1 or c > k + 1 or c < k - 1:
            if c == k - 1 and k >= 1:
                raise Aliased("wait for phase %d found %d completed phases" % (k, c))
            if c > k + 1:
                raise Aliased("wait for phase %d found %d completed phases (would never pass)" % (k, c))
            return False
        return c == k + 1

    def issue(self, thread, bars):
        self.order[thread].append(bars)

    def complete_one(self):
        live = [t for t, q in self.order.items() if q]
        if not live:
            return False
        t = self.rng.choice(live)
        # each issuer's products complete in its issue order; TMA copies in any order
        i = self.rng.randrange(len(self.order[t])) if t == "tma" else 0
        for b in self.order[t].pop(i):
            b.arrive()
        return True

    # ---- roles as generators: each yield is one step; a wait yields until it passes
    def producer(self):
        T, KST, VST, J = self.T, self.KST, self.VST, self.J
        jprev = -1
        for t in range(T + 1):
            j = t if t < T else -1
            # K stage t % KST: free once the score product of tile t - KST completed
            while t >= KST and not self.wait(self.k_empty[t % KST], t // KST - 1):
                yield
            while t >= J and not self.wait(self.j_empty[t % J], t // J - 1):
                yield
            self.jring = getattr(self, "jring", {})
            self.jring[t % J] = j
            self.j_full[t % J].arrive()
            self.jk = getattr(self, "jk", {})
            self.jk[t % KST] = j
            if j >= 0:
                self.issue("tma", [self.k_full[t % KST]])
            else:
                self.k_full[t % KST].arrive()
            yield
            if jprev >= 0:
                u = t - 1
                while u >= VST and not self.wait(self.v_empty[u % VST], u // VST - 1):
                    yield
                self.issue("tma", [self.v_full[u % VST]])
                yield
            jprev = j
            if j < 0:
                return

    def score_issuer(self):
        KST, NSB = self.KST, self.NSB
        u = 0
        while True:
            while not self.wait(self.k_full[u % KST], u // KST):
                yield
            if self.jk[u % KST] < 0:
                break
            if u == 0:
                while not self.wait(self.q_full, 0):
                    yield
            elif u >= NSB:
                while not self.wait(self.pv_done[u % NSB], (u - NSB) // NSB):
                    yield
            self.issue("s", [self.s_full[u % NSB], self.k_empty[u % KST]])
            yield
            u += 1
        self.s_count = u

    def pv_issuer(self):
        NSB, VST = self.NSB, self.VST
        t = 0
        while True:
            while not self.wait(self.p_full[t % NSB], t // NSB):
                yield
            if self.row_end == t:
                break
            while not self.wait(self.v_full[t % VST], t // VST):
                yield
            self.issue("pv", [self.v_empty[t % VST], self.o_done, self.pv_done[t % NSB]])
            yield
            t += 1
        # the final completion, then the epilogue may read O
        self.issue("pv", [])
        while self.order["pv"]:
            yield
        self.mma_done.arrive()

    def softmax(self):
        NSB, J = self.NSB, self.J
        for _ in range(128):
            self.q_full.arrive()
        yield
        t = 0
        while True:
            while not self.wait(self.j_full[t % J], t // J):
                yield
            j = self.jring[t % J]
            for _ in range(4):
                self.j_empty[t % J].arrive()
            if j < 0:
                # the end mark is one more phase of p_full[t % NSB]: that buffer's previous phase
                # (tile t - NSB) must have been consumed by the P.V issuer first
                while t >= NSB and not self.wait(self.pv_done[t % NSB], (t - NSB) // NSB):
                    yield
                self.row_end = t
                for _ in range(128):
                    self.p_full[t % NSB].arrive()
                break
            while not self.wait(self.s_full[t % NSB], t // NSB):
                yield
            if t > 0 and self.rng.random() < 0.3:  # a rescale of O needs P.V of tile t - 1 complete
                if self.rescale_on == "buffer":
                    while not self.wait(self.pv_done[(t - 1) % NSB], (t - 1) // NSB):
                        yield
                else:
                    while not self.wait(self.o_done, t - 1):
                        yield
            yield
            for _ in range(128):
                self.p_full[t % NSB].arrive()
            yield
            t += 1
        if t > 0:
            while not self.wait(self.mma_done, 0):
                yield
        self.tiles = t

    def run(self, max_steps=200000):
        roles = [self.producer(), self.score_issuer(), self.pv_issuer(), self.softmax()]
        live = list(roles)
        for _ in range(max_steps):
            if not live and not any(self.order.values()):
                return
            # a role step or an asynchronous completion, in random order
            if any(self.order.values()) and (not live or self.rng.random() < 0.4):
                self.complete_one()
                continue
            r = self.rng.choice(live)
            try:
                next(r)
            except StopIteration:
                live.remove(r)
        raise AssertionError("no progress: the protocol did not finish")


@pytest.mark.parametrize("KST,VST", [(3, 2), (4, 3), (4, 2)])
@pytest.mark.parametrize("T", [0, 1, 2, 3, 5, 9, 17])
def test_protocol_waits_never_alias_and_finish(T, KST, VST):
    for seed in range(60):
        m = Model(T, KST, VST, seed=1000 * T + seed)
        m.run()
        assert m.tiles == T and m.s_count == T


def test_checker_catches_the_former_o_done_aliasing():
    """With three score buffers the score product of tile t can be issued once P.V of tile t - 3
    completed, so at the softmax of tile t the P.V of tile t - 2 may still be pending: a parity wait
    on one shared completion barrier for phase t - 1 then aliases phase t - 3."""
    caught = 0
    for seed in range(400):
        m = Model(12, 4, 3, NSB=3, rescale_on="o_done", seed=seed)
        try:
            m.run()
        except Aliased:
            caught += 1
    assert caught > 0
    for seed in range(200):   # the per-buffer barrier the kernel waits on instead
        Model(12, 4, 3, NSB=3, rescale_on="buffer", seed=seed).run()
