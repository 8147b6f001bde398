"""Host models of the barrier protocols of the two tcgen05 kernels (free_block_sparse_gb300/csrc/
bsattn.cu and score_gemm.cu).

A parity wait on an mbarrier (try_wait.parity with the parity of phase k) is only right when the
barrier has completed either exactly k phases (not yet: keep waiting) or k + 1 (done).  With k - 1
completed phases the parities alias and the wait passes early; with k + 2 it never passes.  The
models run each kernel's roles against counters of completed phases, with the tensor-core
products completing asynchronously in each issuing thread's order (no order between two issuers)
and TMA copies in any order, under random schedules.  They check that invariant at every wait,
that every schedule finishes, and the data hazards themselves (a buffer or stage overwritten while
a product or the softmax still uses it).  Planted mistakes - the former single P.V-completion
barrier with three score buffers, a score issuer that skips its wait, a GEMM stage released by one
arrival - show that the checks fire."""
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

    def __init__(self, T, KST, VST, NSB=2, JRING=8, rescale_on="buffer", seed=0, s_waits_pv=True):
        self.T, self.KST, self.VST, self.NSB, self.J = T, KST, VST, NSB, JRING
        self.s_waits_pv = s_waits_pv
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
        self.order = {"s": [], "pv": [], "tma": []}  # pending completions per issuing thread
        # data hazards: pending users of each score buffer, K and V stage, and pending P.V products
        self.sbuf = [set() for _ in range(NSB)]
        self.kst_busy = [set() for _ in range(KST)]
        self.vst_busy = [set() for _ in range(VST)]
        self.pv_pending = set()

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
            b() if callable(b) else b.arrive()
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
                assert not self.kst_busy[t % KST], ("K stage reloaded under a score product", t)
                self.issue("tma", [self.k_full[t % KST]])
            else:
                self.k_full[t % KST].arrive()
            yield
            if jprev >= 0:
                u = t - 1
                while u >= VST and not self.wait(self.v_empty[u % VST], u // VST - 1):
                    yield
                assert not self.vst_busy[u % VST], ("V stage reloaded under a P.V product", u)
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
            elif u >= NSB and self.s_waits_pv:
                while not self.wait(self.pv_done[u % NSB], (u - NSB) // NSB):
                    yield
            assert not self.sbuf[u % NSB], ("score buffer overwritten in use", u, self.sbuf[u % NSB])
            self.kst_busy[u % KST].add(u)
            self.issue("s", [lambda u=u: self.kst_busy[u % KST].discard(u), self.s_full[u % NSB],
                             self.k_empty[u % KST]])
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
            self.sbuf[t % NSB].add(("pv", t))
            self.vst_busy[t % VST].add(t)
            self.pv_pending.add(t)

            def pv_complete(t=t):
                self.sbuf[t % NSB].discard(("pv", t))
                self.vst_busy[t % VST].discard(t)
                self.pv_pending.discard(t)
            self.issue("pv", [pv_complete, self.v_empty[t % VST], self.o_done, self.pv_done[t % NSB]])
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
            self.sbuf[t % NSB].add(("softmax", t))
            if t > 0 and self.rng.random() < 0.3:  # a rescale of O needs P.V of tile t - 1 complete
                if self.rescale_on == "buffer":
                    while not self.wait(self.pv_done[(t - 1) % NSB], (t - 1) // NSB):
                        yield
                else:
                    while not self.wait(self.o_done, t - 1):
                        yield
                assert not any(x < t for x in self.pv_pending), ("O rescaled under a P.V product", t)
            yield
            self.sbuf[t % NSB].discard(("softmax", t))
            for _ in range(128):
                self.p_full[t % NSB].arrive()
            yield
            t += 1
        if t > 0:
            while not self.wait(self.mma_done, 0):
                yield
            assert not self.pv_pending, "epilogue reads O under a P.V product"
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


class GemmModel:
    """The pooled-score GEMM's protocol (free_block_sparse_gb300/csrc/score_gemm.cu) for one CTA of
    nch chunks: a producer loading K chunks into a 2-stage ring, an MMA issuer writing two TMEM
    accumulators in turn, and the epilogue warps that read an accumulator, stage the scores in the
    K stage whose products have completed and store them by TMA.  A stage returns to the producer
    only after both the chunk's products and the stores out of it are done (k_empty counts 2)."""

    def __init__(self, nch, seed=0, KST=2):
        self.nch, self.KST = nch, KST
        self.rng = random.Random(seed)
        B = Barrier
        self.q_full = B(1)
        self.k_full = [B(1) for _ in range(KST)]
        self.k_empty = [B(2) for _ in range(KST)]
        self.acc_full = [B(1) for _ in range(2)]
        self.acc_empty = [B(128) for _ in range(2)]
        self.order = {"mma": [], "tma": [], "store": []}
        self.stage_users = [set() for _ in range(KST)]  # who still reads or writes each K stage
        self.acc_users = [set() for _ in range(2)]
        self.wait = Model.wait.__get__(self)

    def complete_one(self):
        live = [t for t, q in self.order.items() if q]
        if not live:
            return False
        t = self.rng.choice(live)
        i = self.rng.randrange(len(self.order[t])) if t == "tma" else 0
        for f in self.order[t].pop(i):
            f()
        return True

    def producer(self):
        self.q_full.arrive()
        yield
        for ch in range(self.nch):
            st = ch % self.KST
            while ch >= self.KST and not self.wait(self.k_empty[st], ch // self.KST - 1):
                yield
            assert not self.stage_users[st], ("stage reloaded while in use", ch, self.stage_users[st])
            self.stage_users[st].add(("load", ch))

            def landed(st=st, ch=ch):
                self.stage_users[st].discard(("load", ch))
                self.k_full[st].arrive()
            self.order["tma"].append([landed])
            yield

    def mma(self):
        while not self.wait(self.q_full, 0):
            yield
        for ch in range(self.nch):
            st, ab = ch % self.KST, ch & 1
            while not self.wait(self.k_full[st], ch // self.KST):
                yield
            while ch >= 2 and not self.wait(self.acc_empty[ab], ch // 2 - 1):
                yield
            assert not self.acc_users[ab], ("accumulator overwritten while read", ch)
            self.stage_users[st].add(("mma", ch))

            def done(st=st, ab=ab, ch=ch):
                self.stage_users[st].discard(("mma", ch))
                self.k_empty[st].arrive()
                self.acc_users[ab].add(("epi", ch))
                self.acc_full[ab].arrive()
            self.order["mma"].append([done])
            yield

    def epilogue(self):
        for ch in range(self.nch):
            st, ab = ch % self.KST, ch & 1
            while not self.wait(self.acc_full[ab], ch // 2):
                yield
            yield  # reads the accumulator, writes the scores into the stage
            assert not any(u[0] != "store" for u in self.stage_users[st]), ("stage still in use", ch)
            self.acc_users[ab].discard(("epi", ch))
            for _ in range(128):
                self.acc_empty[ab].arrive()
            self.stage_users[st].add(("store", ch))

            def stored(st=st, ch=ch):
                self.stage_users[st].discard(("store", ch))
            self.order["store"].append([stored])
            while self.order["store"]:  # the stores have read the stage
                yield
            self.k_empty[st].arrive()

    def run(self, max_steps=100000):
        live = [self.producer(), self.mma(), self.epilogue()]
        for _ in range(max_steps):
            if not live and not any(self.order.values()):
                return
            if any(self.order.values()) and (not live or self.rng.random() < 0.4):
                self.complete_one()
                continue
            r = self.rng.choice(live)
            try:
                next(r)
            except StopIteration:
                live.remove(r)
        raise AssertionError("no progress: the protocol did not finish")


@pytest.mark.parametrize("nch", [1, 2, 3, 4, 7, 16])
def test_score_gemm_protocol(nch):
    for seed in range(80):
        GemmModel(nch, seed=100 * nch + seed).run()


def test_gemm_checker_catches_a_stage_returned_early():
    """With k_empty counting one arrival instead of two, the products' arrival alone returns a K
    stage to the producer while the previous chunk's scores may still be stored out of it (and
    the epilogue's own arrival then completes an extra phase): the model reports a stage reloaded
    in use or a parity wait off by a phase."""
    caught = 0
    for seed in range(300):
        m = GemmModel(8, seed=seed)
        m.k_empty = [Barrier(1) for _ in range(m.KST)]
        try:
            m.run()
        except AssertionError:
            caught += 1
    assert caught > 0


def test_checker_catches_a_score_product_over_a_pending_p():
    """A score issuer that did not wait for P.V of tile u - 2 would overwrite P while that product
    may still read it; the model's buffer bookkeeping reports it."""
    caught = 0
    for seed in range(300):
        try:
            Model(10, 3, 2, seed=seed, s_waits_pv=False).run()
        except AssertionError as e:
            caught += "overwritten" in str(e)
    assert caught > 0
