"""A model check of the kernels' barrier protocols (CPU).

The d = 64 / 128 forward kernel is modelled in full below; `D256Model` and
`BwdModel` at the end do the same for the d = 256 forward and the backward
kernels.

The roles of one CTA of `fa_fwd_f16_kernel` are written here as generators
that follow the kernel's waits, arrivals, commits and issues in program
order: the TMA producer, the MMA warp of each Q sub-tile (turns, P·V then S),
and the four softmax warps of each sub-tile. The tensor pipe executes the
CTA's MMAs in issue order; a commit fires once every MMA its warp issued
before it has completed; TMA copies land at any later time. A random
scheduler interleaves all of it, thousands of times per configuration.

Checked on every run:
  * no deadlock (some role can always make progress until all are done);
  * parity waits never alias: a wait for phase k of a barrier succeeds only
    when exactly k+1 phases have completed (a barrier one phase behind would
    satisfy the parity too, and two ahead would never release it);
  * the data dependencies the barriers stand for: S_i(j) runs on a landed
    K_j and after P_i(j-1)·V has read the columns it overwrites; P_i(j)·V
    runs on a landed V_j after all four softmax warps wrote P_i(j); the
    softmax reads S_i(j) after it completed, rescales O only with every
    earlier P·V complete and none later started, and writes P only after the
    previous P·V read those columns; a K or V stage is reloaded only after
    every MMA reading its previous tile has completed; the epilogue reads O
    after the last P·V.

Configurations: d = 128 (2-stage rings, stages freed by softmax-warp
arrivals) and d = 64 (3-stage rings, stages freed by commits), the default
order (P·V completion taken from the following S's commit) and the strict
order (every P·V committed and waited for), tile counts of both sub-tiles
equal, causal (one more tile for the second sub-tile), a single sub-tile,
and no key tile at all.
"""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.done = count, 0, 0  # done = completed phases

    def arrive(self, n=1):
        for _ in range(n):
            self.pending += 1
            assert self.pending <= self.count
            if self.pending == self.count:
                self.pending, self.done = 0, self.done + 1


class Model:
    def __init__(self, nkv0, nkv1, has1, stages, softmax_frees, strict, rng):
        self.rng = rng
        self.ST, self.SFREE, self.STRICT = stages, softmax_frees, strict
        self.nk = [nkv0, nkv1 if has1 else 0]
        self.has1 = has1
        self.nkv = max(self.nk)
        nsub = 2 if has1 else 1
        rel = 4 * nsub if softmax_frees else nsub
        self.bars = {"QF": Bar(1)}
        for s in range(stages):
            self.bars.update({f"KF{s}": Bar(1), f"KE{s}": Bar(rel), f"VF{s}": Bar(1), f"VE{s}": Bar(rel)})
        for i in range(2):
            self.bars.update({f"SF{i}": Bar(1), f"PF{i}": Bar(4), f"OD{i}": Bar(1), f"DR{i}": Bar(1),
                              f"T{i}": Bar(1)})
        self.kstage = [None] * stages   # tile landed in each K stage (None: empty or loading)
        self.vstage = [None] * stages
        self.landing = []               # (kind, stage, tile, bar) copies in flight
        self.pipe = []                  # MMAs issued, not yet complete: (warp, kind, sub, j)
        self.issued = {0: 0, 1: 0}      # MMAs issued per warp
        self.completed_by = {0: 0, 1: 0}
        self.commits = []               # (warp, count of its MMAs to wait for, bar)
        self.mma_done = set()           # ("S"|"PV", sub, j) completed
        self.mma_started = set()
        self.p_written = {}             # (sub, j) -> softmax warps that wrote P
        self.rescaled = {}              # (sub, j) -> softmax warps that rescaled O at tile j
        self.release_v = True           # softmax warps free V stages (planted-mistake switch)

    # -- barrier waits: runnable only when the parity says so; then no aliasing allowed
    def can_wait(self, name, k):
        return (self.bars[name].done & 1) != (k & 1)

    def check_wait(self, name, k):
        assert self.bars[name].done == k + 1, f"wait on {name} for phase {k} saw {self.bars[name].done} done"

    # ---------------------------------------------------------------- roles
    def producer(self):
        if self.nkv == 0:
            return
        self.landing.append(("Q", 0, 0, "QF"))
        for j in range(self.nkv):
            s = j % self.ST
            yield ("wait", f"KE{s}", j // self.ST - 1)
            # the stage's previous tile j-ST must have been read by every S
            if j >= self.ST:
                for i in range(2 if self.has1 else 1):
                    if j - self.ST < self.nk[i]:
                        assert ("S", i, j - self.ST) in self.mma_done, f"K stage {s} reloaded before S{i}({j - self.ST})"
            self.kstage[s] = None
            self.landing.append(("K", s, j, f"KF{s}"))
            yield ("step",)
            yield ("wait", f"VE{s}", j // self.ST - 1)
            if j >= self.ST:
                for i in range(2 if self.has1 else 1):
                    if j - self.ST < self.nk[i]:
                        assert ("PV", i, j - self.ST) in self.mma_done, f"V stage {s} reloaded before PV{i}({j - self.ST})"
            self.vstage[s] = None
            self.landing.append(("V", s, j, f"VF{s}"))
            yield ("step",)

    def mma(self, sub):
        nkv, nko = self.nk[sub], self.nk[sub ^ 1]
        if nkv > 0:
            yield ("wait", "QF", 0)
            for j in range(nkv + 1):
                other = j if sub == 1 else j - 1
                if self.has1 and 0 <= other <= nko and nko > 0:
                    yield ("wait", f"T{sub}", other)
                if j > 0:
                    s = (j - 1) % self.ST
                    yield ("wait", f"VF{s}", (j - 1) // self.ST)
                    yield ("wait", f"PF{sub}", j - 1)
                    self.issue(sub, "PV", j - 1)
                    if self.STRICT or j == nkv:
                        self.commit(sub, f"OD{sub}")
                    if not self.SFREE:
                        self.commit(sub, f"VE{s}")
                    yield ("step",)
                if j < nkv:
                    s = j % self.ST
                    yield ("wait", f"KF{s}", j // self.ST)
                    if self.STRICT and j > 0:
                        yield ("wait", f"OD{sub}", j - 1)
                    self.issue(sub, "S", j)
                    self.commit(sub, f"SF{sub}")
                    if not self.SFREE:
                        self.commit(sub, f"KE{s}")
                    yield ("step",)
                if self.has1:
                    self.bars[f"T{sub ^ 1}"].arrive()
                    yield ("step",)
        self.commit(sub, f"DR{sub}")
        yield ("wait", f"DR{sub}", 0)

    def softmax(self, sub, w):
        nkv = self.nk[sub]
        for j in range(nkv):
            yield ("wait", f"SF{sub}", j)
            if self.SFREE:
                if j > 0 and self.release_v:
                    self.bars[f"VE{(j - 1) % self.ST}"].arrive()
                self.bars[f"KE{j % self.ST}"].arrive()
            assert ("S", sub, j) in self.mma_done
            yield ("step",)
            if j > 0 and self.rng.random() < 0.3:   # a rescale of O at tile j
                if self.STRICT:
                    yield ("wait", f"OD{sub}", j - 1)
                assert ("PV", sub, j - 1) in self.mma_done, "O rescaled while an earlier P.V may run"
                assert ("PV", sub, j) not in self.mma_started
                self.rescaled.setdefault((sub, j), set()).add(w)
            # P overwrites S columns that P(j-1).V read
            assert j == 0 or ("PV", sub, j - 1) in self.mma_done
            self.p_written.setdefault((sub, j), set()).add(w)
            self.bars[f"PF{sub}"].arrive()
            yield ("step",)
        if nkv > 0:
            yield ("wait", f"OD{sub}", nkv - 1 if self.STRICT else 0)
            for j in range(nkv):
                assert ("PV", sub, j) in self.mma_done, "epilogue read O before the last P.V"

    # ---------------------------------------------------------------- async agents
    def issue(self, warp, kind, j):
        self.issued[warp] += 1
        self.pipe.append((warp, kind, warp, j))

    def commit(self, warp, bar):
        self.commits.append((warp, self.issued[warp], bar))

    def execute_head(self):
        warp, kind, sub, j = self.pipe.pop(0)
        self.mma_started.add((kind, sub, j))
        if kind == "S":
            assert self.kstage[j % self.ST] == j, f"S{sub}({j}) on a K stage without K_{j}"
            assert j == 0 or ("PV", sub, j - 1) in self.mma_done, "S overwrote P before P.V read it"
        else:
            assert self.vstage[j % self.ST] == j, f"PV{sub}({j}) on a V stage without V_{j}"
            assert self.p_written.get((sub, j)) == {0, 1, 2, 3}, "P.V before every softmax warp wrote P"
        self.mma_done.add((kind, sub, j))
        self.completed_by[warp] += 1

    def events(self):
        ev = []
        if self.pipe:
            ev.append(("pipe",))
        for n, c in enumerate(self.commits):
            if self.completed_by[c[0]] >= c[1]:
                ev.append(("commit", n))
        for n in range(len(self.landing)):
            ev.append(("land", n))
        return ev

    def fire(self, e):
        if e[0] == "pipe":
            self.execute_head()
        elif e[0] == "commit":
            _, _, bar = self.commits.pop(e[1])
            self.bars[bar].arrive()
        else:
            kind, s, j, bar = self.landing.pop(e[1])
            if kind == "K":
                self.kstage[s] = j
            elif kind == "V":
                self.vstage[s] = j
            self.bars[bar].arrive()

    # ---------------------------------------------------------------- scheduler
    def roles(self):
        roles = [self.producer(), self.mma(0)]
        roles += [self.softmax(0, w) for w in range(4)]
        if self.has1:
            roles += [self.mma(1)] + [self.softmax(1, w) for w in range(4)]
        return roles

    def run(self):
        roles = self.roles()
        state = {n: None for n in range(len(roles))}  # pending request of each live role
        live = set(range(len(roles)))

        def advance(n):
            try:
                state[n] = next(roles[n])
            except StopIteration:
                live.discard(n)
                state[n] = None

        for n in list(live):
            advance(n)
        for _ in range(200000):
            if not live and not self.pipe and not self.commits and not self.landing:
                return
            choices = []
            for n in live:
                req = state[n]
                if req[0] == "step" or self.can_wait(req[1], req[2]):
                    choices.append(("role", n))
            choices += self.events()
            assert choices, f"deadlock: {[state[n] for n in live]}"
            c = self.rng.choice(choices)
            if c[0] == "role":
                req = state[c[1]]
                if req[0] == "wait":
                    self.check_wait(req[1], req[2])
                advance(c[1])
            else:
                self.fire(c)
        raise AssertionError("did not finish")


CASES = [(1, 1, True), (2, 2, True), (5, 5, True), (3, 4, True), (1, 2, True), (4, 0, False), (0, 0, True),
         (0, 0, False)]


@pytest.mark.parametrize("stages,softmax_frees", [(2, True), (3, False)], ids=["d128", "d64"])
@pytest.mark.parametrize("strict", [False, True], ids=["default", "strict"])
@pytest.mark.parametrize("nkv0,nkv1,has1", CASES)
def test_forward_barrier_protocol(stages, softmax_frees, strict, nkv0, nkv1, has1):
    rng = random.Random(hash((stages, strict, nkv0, nkv1, has1)) & 0xFFFFFFFF)
    for _ in range(500):
        Model(nkv0, nkv1, has1, stages, softmax_frees, strict, rng).run()


def test_model_catches_a_missing_stage_release():
    """Planted mistake in the model: softmax warps that never free the V
    stage. The producer then waits on a phase that cannot complete."""
    m = Model(4, 4, True, 2, True, False, random.Random(1))
    m.release_v = False
    with pytest.raises(AssertionError, match="deadlock"):
        m.run()


def test_model_catches_a_parity_wait_that_skips_a_phase():
    """Planted mistake in the model: a softmax warp that waits for S-full
    only on odd tiles can observe the barrier two phases late, which the
    parity alone does not reveal."""
    class SkipWait(Model):
        def softmax(self, sub, w):
            for req in Model.softmax(self, sub, w):
                if req[0] == "wait" and req[1] == f"SF{sub}" and req[2] % 2 == 0 and req[2] > 0:
                    continue
                yield req
    with pytest.raises(AssertionError):
        for seed in range(50):
            SkipWait(6, 6, True, 2, True, False, random.Random(seed)).run()


def test_model_catches_a_stage_freed_too_early():
    """Planted mistake in the model: softmax warps that free V_j's stage as
    soon as S_j is complete (instead of V_{j-1}'s), before P_j·V_j has read
    it. The producer then reloads a V stage that an MMA still needs."""
    class EarlyV(Model):
        def softmax(self, sub, w):
            for j in range(self.nk[sub]):
                yield ("wait", f"SF{sub}", j)
                self.bars[f"VE{j % self.ST}"].arrive()
                self.bars[f"KE{j % self.ST}"].arrive()
                yield ("step",)
                self.p_written.setdefault((sub, j), set()).add(w)
                self.bars[f"PF{sub}"].arrive()
                yield ("step",)
            if self.nk[sub] > 0:
                yield ("wait", f"OD{sub}", 0)
    with pytest.raises(AssertionError, match="reloaded before"):
        EarlyV(6, 6, True, 2, True, False, random.Random(3)).run()


class D256Model(Model):
    """`fa_fwd_d256_kernel`: one 128-row Q tile, 64-key K/V tiles in 2-stage
    rings, two S buffers (S_{j+2} issued right behind P_j·V into the columns
    of P_j), K stages freed by the four softmax warps once S_j is complete, V
    stages by a commit behind each P·V, a per-P·V barrier (OD) for rescales
    and a barrier committed once after the last P·V (OL) for the epilogue."""

    def __init__(self, nkv, strict, rng):
        super().__init__(nkv, 0, False, 2, True, strict, rng)
        self.bars["OL"] = Bar(1)
        for s in range(2):
            self.bars[f"KE{s}"] = Bar(4)
            self.bars[f"VE{s}"] = Bar(1)
        self.bars["PF0"], self.bars["PF1"] = Bar(4), Bar(4)

    def roles(self):
        return [self.producer(), self.mma256()] + [self.softmax256(w) for w in range(4)]

    def mma256(self):
        nkv = self.nkv
        if nkv > 0:
            yield ("wait", "QF", 0)
            for j in range(min(nkv, 2)):
                yield ("wait", f"KF{j % 2}", j // 2)
                self.issue(0, "S", j)
                self.commit(0, f"SF{j & 1}")
                yield ("step",)
            for j in range(nkv):
                s = j % 2
                yield ("wait", f"VF{s}", j // 2)
                yield ("wait", f"PF{j & 1}", j // 2)
                self.issue(0, "PV", j)
                self.commit(0, "OD0")
                if j == nkv - 1:
                    self.commit(0, "OL")
                self.commit(0, f"VE{s}")
                yield ("step",)
                if j + 2 < nkv:
                    if self.STRICT:
                        yield ("wait", "OD0", j)
                    n = j + 2
                    yield ("wait", f"KF{n % 2}", n // 2)
                    self.issue(0, "S", n)
                    self.commit(0, f"SF{n & 1}")
                    yield ("step",)
        self.commit(0, "DR0")
        yield ("wait", "DR0", 0)

    def softmax256(self, w):
        nkv = self.nkv
        for j in range(nkv):
            yield ("wait", f"SF{j & 1}", j // 2)
            self.bars[f"KE{j % 2}"].arrive()
            assert ("S", 0, j) in self.mma_done
            yield ("step",)
            # P_j overwrites the buffer of S_j, whose previous P (P_{j-2}) P_{j-2}.V read
            assert j < 2 or ("PV", 0, j - 2) in self.mma_done
            self.p_written.setdefault((0, j), set()).add(w)
            if j > 0:
                # every phase of the per-P.V barrier is waited for in turn (not
                # only before a rescale), so its parity names one phase
                # whatever the order in which commits on different barriers land
                yield ("wait", "OD0", j - 1)
                if self.rng.random() < 0.3:   # a rescale of O at tile j
                    assert ("PV", 0, j - 1) in self.mma_done, "O rescaled while an earlier P.V may run"
                    assert ("PV", 0, j) not in self.mma_started
            self.bars[f"PF{j & 1}"].arrive()
            yield ("step",)
        if nkv > 0:
            yield ("wait", "OL", 0)
            for j in range(nkv):
                assert ("PV", 0, j) in self.mma_done, "epilogue read O before the last P.V"

    def execute_head(self):
        warp, kind, sub, j = self.pipe.pop(0)
        self.mma_started.add((kind, sub, j))
        if kind == "S":
            assert self.kstage[j % 2] == j, f"S({j}) on a K stage without K_{j}"
            assert j < 2 or ("PV", 0, j - 2) in self.mma_done, "S overwrote P before P.V read it"
        else:
            assert self.vstage[j % 2] == j, f"PV({j}) on a V stage without V_{j}"
            assert self.p_written.get((0, j)) == {0, 1, 2, 3}, "P.V before every softmax warp wrote P"
        self.mma_done.add((kind, sub, j))
        self.completed_by[warp] += 1


@pytest.mark.parametrize("strict", [False, True], ids=["default", "strict"])
@pytest.mark.parametrize("nkv", [0, 1, 2, 3, 7])
def test_d256_barrier_protocol(strict, nkv):
    rng = random.Random(1000 + 10 * nkv + strict)
    for _ in range(300):
        D256Model(nkv, strict, rng).run()


def test_model_catches_a_rescale_wait_that_relies_on_commit_order():
    """The d = 256 softmax used to wait on the per-P.V barrier only before a
    rescale, trusting that S_j's completion implies the arrival for the P.V
    issued before it. Commits on different barriers may land in any order, and
    then that parity can name a phase two behind."""
    class OnlyOnRescale(D256Model):
        def softmax256(self, w):
            for req in D256Model.softmax256(self, w):
                if req[0] == "wait" and req[1] == "OD0" and self.rng.random() < 0.7:
                    continue   # no rescale at this tile: the old code did not wait
                yield req
    with pytest.raises(AssertionError):
        for seed in range(200):
            OnlyOnRescale(7, False, random.Random(seed)).run()


class BwdModel(Model):
    """`fa_bwd_main_kernel`: the TMA producer (K, V once; Q_i with its rows
    in a QST-stage ring, dO_i in an OST-stage ring), MMA warp A (dQ_i, dK_i
    once dS_i is formed), MMA warp B (S^T_0, dP^T_0, dV_0, S^T_1, then per
    tile dP^T_{i+1}, dV_{i+1}, S^T_{i+2}), eight softmax warps (P_i over the
    S^T columns, then dS_i into shared memory) and four dQ warps (dQ_i out of
    TMEM). For d = 128 dQ_i reuses the dP^T columns; for d = 64 it has its own."""

    def __init__(self, nq, d, strict, rng):
        self.rng, self.STRICT, self.nq, self.d = rng, strict, nq, d
        self.QST, self.OST = (2, 1) if d == 128 else (3, 2)
        self.bars = {"K": Bar(1), "V": Bar(1), "SF": Bar(1), "DPF": Bar(1), "PF": Bar(8), "DSF": Bar(8),
                     "DQF": Bar(1), "DQE": Bar(4), "DSE": Bar(1), "DONE": Bar(2)}
        for s in range(self.QST):
            self.bars.update({f"QF{s}": Bar(1), f"QE{s}": Bar(1)})
        for s in range(self.OST):
            self.bars.update({f"OF{s}": Bar(1), f"OE{s}": Bar(1)})
        self.qstage, self.ostage = [None] * self.QST, [None] * self.OST
        self.kv = set()
        self.landing, self.pipe, self.commits = [], [], []
        self.issued = {0: 0, 1: 0}
        self.completed_by = {0: 0, 1: 0}
        self.mma_done, self.mma_started = set(), set()
        self.count = {}  # (event, i) -> number of warps that did it

    def bump(self, ev, i):
        self.count[(ev, i)] = self.count.get((ev, i), 0) + 1

    def roles(self):
        return ([self.producer(), self.mma_a(), self.mma_b()] + [self.softmax_bwd(w) for w in range(8)]
                + [self.dq_warp(w) for w in range(4)])

    def producer(self):
        self.landing += [("K", 0, 0, "K"), ("V", 0, 0, "V")]
        for i in range(self.nq):
            qs, os_ = i % self.QST, i % self.OST
            yield ("wait", f"QE{qs}", i // self.QST - 1)
            if i >= self.QST:  # readers of Q_{i-QST} and its rows: S^T, dK, the softmax's P and dS phases
                assert {("S", i - self.QST), ("DK", i - self.QST)} <= self.mma_done, "Q stage reloaded early"
                assert self.count.get(("ds", i - self.QST), 0) == 8, "Q rows reloaded before the softmax used them"
            self.qstage[qs] = None
            self.landing.append(("Q", qs, i, f"QF{qs}"))
            yield ("step",)
            yield ("wait", f"OE{os_}", i // self.OST - 1)
            if i >= self.OST:
                assert {("DP", i - self.OST), ("DV", i - self.OST)} <= self.mma_done, "dO stage reloaded early"
            self.ostage[os_] = None
            self.landing.append(("O", os_, i, f"OF{os_}"))
            yield ("step",)

    def mma_a(self):
        for i in range(self.nq):
            yield ("wait", "DSF", i)
            if self.d == 64 and i > 0:
                yield ("wait", "DQE", i - 1)
            self.issue(0, "DQ", i)
            self.commit(0, "DQF")
            self.issue(0, "DK", i)
            self.commit(0, f"QE{i % self.QST}")
            self.commit(0, "DSE")
            yield ("step",)
        self.commit(0, "DONE")
        yield ("wait", "DONE", 0)

    def mma_b(self):
        nq = self.nq
        yield ("wait", "K", 0)
        yield ("wait", "QF0", 0)
        self.issue(1, "S", 0)
        self.commit(1, "SF")
        yield ("wait", "V", 0)
        yield ("wait", "OF0", 0)
        self.issue(1, "DP", 0)
        self.commit(1, "DPF")
        yield ("wait", "PF", 0)
        self.issue(1, "DV", 0)
        self.commit(1, "OE0")
        yield ("step",)
        if nq > 1:
            if self.STRICT:
                yield ("wait", "OE0", 0)
            yield ("wait", f"QF{1 % self.QST}", 1 // self.QST)
            self.issue(1, "S", 1)
            self.commit(1, "SF")
            yield ("step",)
        for i in range(nq - 1):
            n1 = i + 1
            yield ("wait", "DQE", i) if self.d == 128 else ("wait", "DSF", i)
            yield ("wait", f"OF{n1 % self.OST}", n1 // self.OST)
            self.issue(1, "DP", n1)
            self.commit(1, "DPF")
            yield ("wait", "PF", n1)
            self.issue(1, "DV", n1)
            self.commit(1, f"OE{n1 % self.OST}")
            yield ("step",)
            if i + 2 < nq:
                n2 = i + 2
                if self.STRICT:
                    yield ("wait", f"OE{n1 % self.OST}", n1 // self.OST)
                yield ("wait", f"QF{n2 % self.QST}", n2 // self.QST)
                self.issue(1, "S", n2)
                self.commit(1, "SF")
                yield ("step",)
        self.commit(1, "DONE")
        yield ("wait", "DONE", 0)

    def softmax_bwd(self, w):
        for i in range(self.nq):
            yield ("wait", "SF", i)
            assert ("S", i) in self.mma_done and self.qstage[i % self.QST] == i
            # P^T_i over the S^T columns that dV_{i-1} read
            assert i == 0 or ("DV", i - 1) in self.mma_done
            self.bump("p", i)
            self.bars["PF"].arrive()
            yield ("step",)
            yield ("wait", "DPF", i)
            if i > 0:
                yield ("wait", "DSE", i - 1)
                assert {("DQ", i - 1), ("DK", i - 1)} <= self.mma_done, "dS overwritten while an MMA reads it"
            assert ("DP", i) in self.mma_done
            self.bump("ds", i)
            self.bars["DSF"].arrive()
            yield ("step",)
        yield ("wait", "DONE", 0)
        for i in range(self.nq):
            assert {("DV", i), ("DK", i)} <= self.mma_done, "epilogue read dV / dK before the last MMA"

    def dq_warp(self, w):
        for i in range(self.nq):
            yield ("wait", "DQF", i)
            assert ("DQ", i) in self.mma_done
            self.bump("dqread", i)
            self.bars["DQE"].arrive()
            yield ("step",)

    def issue(self, warp, kind, i):
        self.issued[warp] += 1
        self.pipe.append((warp, kind, 0, i))

    def execute_head(self):
        warp, kind, _, i = self.pipe.pop(0)
        self.mma_started.add((kind, i))
        c = self.count.get
        if kind == "S":
            assert "K" in self.kv and self.qstage[i % self.QST] == i
            if i > 0:  # over P^T_{i-1}: dV_{i-1} read it, every softmax warp wrote it
                assert ("DV", i - 1) in self.mma_done and c(("p", i - 1), 0) == 8
        elif kind == "DP":
            assert "V" in self.kv and self.ostage[i % self.OST] == i
            if i > 0:  # over dP^T_{i-1} (and, for d = 128, dQ_{i-1})
                assert c(("ds", i - 1), 0) == 8, "dP^T overwritten before the softmax read it"
                if self.d == 128:
                    assert c(("dqread", i - 1), 0) == 4, "dP^T overwrote dQ before it was read out"
        elif kind == "DV":
            assert c(("p", i), 0) == 8 and self.ostage[i % self.OST] == i
        elif kind == "DQ":
            assert c(("ds", i), 0) == 8, "dQ before dS was formed"
            if self.d == 64 and i > 0:
                assert c(("dqread", i - 1), 0) == 4, "dQ overwrote the previous dQ before it was read out"
            if self.d == 128:   # into the dP^T columns: the softmax read dP^T_i (it formed dS_i)
                assert ("DP", i) in self.mma_done
        elif kind == "DK":
            assert c(("ds", i), 0) == 8 and self.qstage[i % self.QST] == i
        self.mma_done.add((kind, i))
        self.completed_by[warp] += 1

    def fire(self, e):
        if e[0] == "land":
            kind, s, i, bar = self.landing.pop(e[1])
            if kind in ("K", "V"):
                self.kv.add(kind)
            elif kind == "Q":
                self.qstage[s] = i
            else:
                self.ostage[s] = i
            self.bars[bar].arrive()
        else:
            Model.fire(self, e)


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("strict", [False, True], ids=["default", "strict"])
@pytest.mark.parametrize("nq", [1, 2, 3, 6])
def test_backward_barrier_protocol(d, strict, nq):
    rng = random.Random(2000 + 10 * nq + d + strict)
    for _ in range(400):
        BwdModel(nq, d, strict, rng).run()


def test_model_catches_dp_overwriting_dq():
    """Planted mistake in the model: for d = 128, warp B issuing dP^T_{i+1}
    without waiting for the dQ warps to read dQ_i out of the same columns."""
    class NoDqWait(BwdModel):
        def mma_b(self):
            for req in BwdModel.mma_b(self):
                if req[0] == "wait" and req[1] == "DQE":
                    continue
                yield req
    with pytest.raises(AssertionError, match="dQ before it was read out"):
        for seed in range(100):
            NoDqWait(6, 128, False, random.Random(seed)).run()


class Bwd256DvModel(BwdModel):
    """`fa_bwd_dv256_kernel`: the producer (K once; Q_i with its LSE row and
    dO_i in 2-stage rings, Q stages freed by the four softmax warps once they
    have read the LSE row), the MMA warp (S^T_0, S^T_1, then dV_i and S^T_{i+2}
    into the buffer of P^T_i right behind it) and four softmax warps (P^T_i
    over S buffer i % 2)."""

    def __init__(self, nq, strict, rng):
        BwdModel.__init__(self, nq, 128, strict, rng)
        self.QST = self.OST = 2
        self.qstage, self.ostage = [None] * 2, [None] * 2
        self.bars = {"K": Bar(1), "DONE": Bar(1), "DR": Bar(1)}
        for s in range(2):
            self.bars.update({f"QF{s}": Bar(1), f"QE{s}": Bar(4), f"OF{s}": Bar(1), f"OE{s}": Bar(1),
                              f"SF{s}": Bar(1), f"PF{s}": Bar(4)})

    def roles(self):
        return [self.producer(), self.mma()] + [self.softmax(w) for w in range(4)]

    def producer(self):
        self.landing.append(("K", 0, 0, "K"))
        for i in range(self.nq):
            s = i % 2
            yield ("wait", f"QE{s}", i // 2 - 1)
            if i >= 2:
                assert ("S", i - 2) in self.mma_done and self.count.get(("p", i - 2), 0) == 4, "Q stage reloaded early"
            self.qstage[s] = None
            self.landing.append(("Q", s, i, f"QF{s}"))
            yield ("step",)
            yield ("wait", f"OE{s}", i // 2 - 1)
            if i >= 2:
                assert ("DV", i - 2) in self.mma_done, "dO stage reloaded early"
            self.ostage[s] = None
            self.landing.append(("O", s, i, f"OF{s}"))
            yield ("step",)

    def mma(self):
        nq = self.nq
        if nq > 0:
            yield ("wait", "K", 0)
            for i in range(min(nq, 2)):
                yield ("wait", f"QF{i % 2}", i // 2)
                self.issue(0, "S", i)
                self.commit(0, f"SF{i & 1}")
                yield ("step",)
            for i in range(nq):
                s = i % 2
                yield ("wait", f"OF{s}", i // 2)
                yield ("wait", f"PF{i & 1}", i // 2)
                self.issue(0, "DV", i)
                self.commit(0, f"OE{s}")
                if i == nq - 1:
                    self.commit(0, "DONE")
                yield ("step",)
                if i + 2 < nq:
                    n = i + 2
                    if self.STRICT:
                        yield ("wait", f"OE{s}", i // 2)
                    yield ("wait", f"QF{n % 2}", n // 2)
                    self.issue(0, "S", n)
                    self.commit(0, f"SF{n & 1}")
                    yield ("step",)
        self.commit(0, "DR")
        yield ("wait", "DR", 0)

    def softmax(self, w):
        for i in range(self.nq):
            yield ("wait", f"SF{i & 1}", i // 2)
            assert ("S", i) in self.mma_done and self.qstage[i % 2] == i
            # P^T_i over the buffer whose P^T_{i-2} dV_{i-2} read
            assert i < 2 or ("DV", i - 2) in self.mma_done
            self.bump("p", i)
            self.bars[f"PF{i & 1}"].arrive()
            self.bars[f"QE{i % 2}"].arrive()
            yield ("step",)
        if self.nq > 0:
            yield ("wait", "DONE", 0)
            for i in range(self.nq):
                assert ("DV", i) in self.mma_done, "epilogue read dV before the last MMA"

    def execute_head(self):
        warp, kind, _, i = self.pipe.pop(0)
        self.mma_started.add((kind, i))
        if kind == "S":
            assert "K" in self.kv and self.qstage[i % 2] == i
            if i >= 2:  # over P^T_{i-2}: dV_{i-2} read it, every softmax warp wrote it
                assert ("DV", i - 2) in self.mma_done and self.count.get(("p", i - 2), 0) == 4, \
                    "S^T overwrote P^T before dV read it"
        else:
            assert self.count.get(("p", i), 0) == 4 and self.ostage[i % 2] == i, "dV before P^T or dO"
        self.mma_done.add((kind, i))
        self.completed_by[warp] += 1


class Bwd256DkdqModel(BwdModel):
    """`fa_bwd_dkdq256_kernel`: the producer (K, V once; dO_i and Q_i with its
    rows, one stage each), the MMA warp (dP^T_0, then per tile S^T_i,
    dP^T_{i+1} once the softmax has read dP^T_i, dK_i and dQ^T_i once dS_i is
    written), four softmax warps (S^T_i and dP^T_i into registers, dS^T_i into
    shared memory) and four dQ warps (dQ^T_i out of TMEM)."""

    def __init__(self, nq, rng):
        BwdModel.__init__(self, nq, 128, False, rng)
        self.qstage, self.ostage = [None], [None]
        self.bars = {n: Bar(1) for n in ["K", "V", "QF", "QE", "OF", "OE", "SF", "DPF", "DSE", "DQF", "DONE", "DR"]}
        self.bars.update({"SC": Bar(4), "DSF": Bar(4), "DQE": Bar(4)})

    def roles(self):
        return ([self.producer(), self.mma()] + [self.softmax(w) for w in range(4)]
                + [self.dq_warp(w) for w in range(4)])

    def producer(self):
        self.landing += [("K", 0, 0, "K"), ("V", 0, 0, "V")]
        for i in range(self.nq):
            yield ("wait", "OE", i - 1)
            assert i == 0 or ("DP", i - 1) in self.mma_done, "dO reloaded early"
            self.ostage[0] = None
            self.landing.append(("O", 0, i, "OF"))
            yield ("step",)
            yield ("wait", "QE", i - 1)
            if i > 0:
                assert {("S", i - 1), ("DK", i - 1)} <= self.mma_done, "Q reloaded early"
                assert self.count.get(("ds", i - 1), 0) == 4, "Q rows reloaded before the softmax used them"
            self.qstage[0] = None
            self.landing.append(("Q", 0, i, "QF"))
            yield ("step",)

    def mma(self):
        nq = self.nq
        if nq > 0:
            yield ("wait", "V", 0)
            yield ("wait", "OF", 0)
            self.issue(0, "DP", 0)
            self.commit(0, "DPF")
            self.commit(0, "OE")
            yield ("wait", "K", 0)
            for i in range(nq):
                yield ("wait", "QF", i)
                self.issue(0, "S", i)
                self.commit(0, "SF")
                yield ("wait", "SC", i)
                if i + 1 < nq:
                    yield ("wait", "OF", i + 1)
                    self.issue(0, "DP", i + 1)
                    self.commit(0, "DPF")
                    self.commit(0, "OE")
                yield ("wait", "DSF", i)
                self.issue(0, "DK", i)
                self.commit(0, "QE")
                if i > 0:
                    yield ("wait", "DQE", i - 1)
                self.issue(0, "DQ", i)
                self.commit(0, "DQF")
                self.commit(0, "DSE")
                yield ("step",)
            self.commit(0, "DONE")
        self.commit(0, "DR")
        yield ("wait", "DR", 0)

    def softmax(self, w):
        for i in range(self.nq):
            yield ("wait", "SF", i)
            assert ("S", i) in self.mma_done
            yield ("wait", "DPF", i)
            assert ("DP", i) in self.mma_done
            self.bump("sc", i)
            self.bars["SC"].arrive()
            yield ("step",)
            if i > 0:
                yield ("wait", "DSE", i - 1)
                assert {("DQ", i - 1), ("DK", i - 1)} <= self.mma_done, "dS overwritten while an MMA reads it"
            self.bump("ds", i)
            self.bars["DSF"].arrive()
            yield ("step",)
        if self.nq > 0:
            yield ("wait", "DONE", 0)
            for i in range(self.nq):
                assert {("DK", i), ("DQ", i)} <= self.mma_done, "epilogue read dK before the last MMA"

    def dq_warp(self, w):
        for i in range(self.nq):
            yield ("wait", "DQF", i)
            assert ("DQ", i) in self.mma_done
            self.bump("dqread", i)
            self.bars["DQE"].arrive()
            yield ("step",)

    def execute_head(self):
        warp, kind, _, i = self.pipe.pop(0)
        self.mma_started.add((kind, i))
        c = self.count.get
        if kind == "DP":
            assert "V" in self.kv and self.ostage[0] == i
            assert i == 0 or c(("sc", i - 1), 0) == 4, "dP^T overwritten before the softmax read it"
        elif kind == "S":
            assert "K" in self.kv and self.qstage[0] == i
            assert i == 0 or c(("sc", i - 1), 0) == 4, "S^T overwritten before the softmax read it"
        elif kind == "DK":
            assert c(("ds", i), 0) == 4 and self.qstage[0] == i and "K" in self.kv
        else:
            assert c(("ds", i), 0) == 4, "dQ^T before dS was formed"
            assert i == 0 or c(("dqread", i - 1), 0) == 4, "dQ^T overwrote the previous one before it was read out"
        self.mma_done.add((kind, i))
        self.completed_by[warp] += 1


@pytest.mark.parametrize("strict", [False, True], ids=["default", "strict"])
@pytest.mark.parametrize("nq", [0, 1, 2, 3, 7])
def test_backward_d256_dv_barrier_protocol(strict, nq):
    rng = random.Random(3000 + 10 * nq + strict)
    for _ in range(400):
        Bwd256DvModel(nq, strict, rng).run()


@pytest.mark.parametrize("nq", [0, 1, 2, 3, 7])
def test_backward_d256_dkdq_barrier_protocol(nq):
    rng = random.Random(4000 + nq)
    for _ in range(400):
        Bwd256DkdqModel(nq, rng).run()


def test_model_catches_dq_overwrite_in_the_d256_dkdq_kernel():
    """Planted mistake: dQ^T_i issued without waiting for the dQ warps to read
    dQ^T_{i-1} out of the same columns."""
    class NoDqeWait(Bwd256DkdqModel):
        def mma(self):
            for req in Bwd256DkdqModel.mma(self):
                if req[0] == "wait" and req[1] == "DQE":
                    continue
                yield req
    with pytest.raises(AssertionError, match="before it was read out"):
        for seed in range(200):
            NoDqeWait(6, random.Random(seed)).run()


def test_model_catches_s_issued_before_dv_in_the_d256_dv_kernel():
    """Planted mistake: S^T_{i+2} issued before dV_i, whose P^T it overwrites."""
    class SBeforeDv(Bwd256DvModel):
        def issue(self, warp, kind, i):
            Bwd256DvModel.issue(self, warp, kind, i)
            if kind == "S" and i >= 2:
                # move S^T_i in front of dV_{i-2} while that is still queued
                for n, (_, k, _, j) in enumerate(self.pipe[:-1]):
                    if (k, j) == ("DV", i - 2):
                        self.pipe.insert(n, self.pipe.pop())
                        break
    with pytest.raises(AssertionError, match="overwrote P"):
        for seed in range(300):
            SBeforeDv(7, False, random.Random(seed)).run()


class OneWarpModel(Model):
    """The d = 64 kernel: one MMA warp issues both chains' blocks in the turn
    order B_0(0), B_1(0), B_0(1), ... by program order (no turn barriers); the
    rest as in Model with commit-freed stages."""

    def roles(self):
        roles = [self.producer(), self.mma_both()]
        roles += [self.softmax(0, w) for w in range(4)]
        if self.has1:
            roles += [self.softmax(1, w) for w in range(4)]
        return roles

    def block(self, sub, j):
        nkv = self.nk[sub]
        sv, sk = (j - 1) % self.ST, j % self.ST
        if j > 0:
            yield ("wait", f"VF{sv}", (j - 1) // self.ST)
            yield ("wait", f"PF{sub}", j - 1)
            self.issue(sub, "PV", j - 1)
            if self.STRICT or j == nkv:
                self.commit(sub, f"OD{sub}")
            if not self.SFREE:
                self.commit(sub, f"VE{sv}")
            yield ("step",)
        if j < nkv:
            yield ("wait", f"KF{sk}", j // self.ST)
            if self.STRICT and j > 0:
                yield ("wait", f"OD{sub}", j - 1)
            self.issue(sub, "S", j)
            self.commit(sub, f"SF{sub}")
            if not self.SFREE:
                self.commit(sub, f"KE{sk}")
            yield ("step",)

    def mma_both(self):
        n = max(self.nk)
        if n > 0:
            yield ("wait", "QF", 0)
            for j in range(n + 1):
                for sub in (0, 1):
                    if self.nk[sub] > 0 and j <= self.nk[sub]:
                        yield from self.block(sub, j)
        for sub in (0, 1):
            self.commit(sub, f"DR{sub}")
            yield ("wait", f"DR{sub}", 0)

    def issue(self, warp, kind, j):
        # one warp issues for both chains: one issue stream, in order
        self.issued[0] += 1
        self.pipe.append((0, kind, warp, j))

    def commit(self, warp, bar):
        self.commits.append((0, self.issued[0], bar))

    def execute_head(self):
        _, kind, sub, j = self.pipe.pop(0)
        self.pipe.insert(0, (sub, kind, sub, j))
        Model.execute_head(self)
        self.completed_by[sub] -= 1
        self.completed_by[0] += 1


@pytest.mark.parametrize("strict", [False, True], ids=["default", "strict"])
@pytest.mark.parametrize("nkv0,nkv1,has1", CASES)
def test_forward_d64_one_mma_warp_protocol(strict, nkv0, nkv1, has1):
    rng = random.Random(hash(("one", strict, nkv0, nkv1, has1)) & 0xFFFFFFFF)
    for _ in range(400):
        OneWarpModel(nkv0, nkv1, has1, 3, False, strict, rng).run()


class PersistModel(BwdModel):
    """The persistent form of the d = 128 forward kernel: one CTA walks a list
    of units (nkv0, nkv1); the producer (Q per unit once the previous unit's
    last S products of both sub-tiles completed; K/V tiles in a 2-stage ring
    numbered across units), one MMA warp (both chains' blocks in turn order;
    a unit's first P.V of sub-tile i waits until the previous unit's epilogue
    read O_i), four softmax warps per sub-tile (stage releases per tile, the
    tiles only the other sub-tile uses released once they have landed, the
    last V released after the unit's last P.V, the Q-free arrival after the
    last S, the O-free arrival after the epilogue read O)."""

    ST = 2

    def __init__(self, units, rng):
        BwdModel.__init__(self, 1, 128, False, rng)
        self.units = units
        self.bars = {"Q": Bar(1), "QE": Bar(8), "DR": Bar(1)}
        for s in range(self.ST):
            self.bars.update({f"KF{s}": Bar(1), f"KE{s}": Bar(8), f"VF{s}": Bar(1), f"VE{s}": Bar(8)})
        for i in range(2):
            self.bars.update({f"SF{i}": Bar(1), f"PF{i}": Bar(4), f"OD{i}": Bar(1), f"OF{i}": Bar(4)})
        self.kst, self.vst, self.qunit = [None] * self.ST, [None] * self.ST, None
        self.o_read = set()  # (sub, unit) epilogues that read O

    def base(self, k):
        return sum(max(a, b) for a, b in self.units[:k])

    def pending(self):
        """MMAs issued and not yet complete, as (kind, key)."""
        return [(kind, key) for _, kind, _, key in self.pipe]

    def roles(self):
        return [self.producer(), self.mma()] + [self.softmax(sub, w) for sub in (0, 1) for w in range(4)]

    def producer(self):
        g = 0
        for k, (n0, n1) in enumerate(self.units):
            nkv = max(n0, n1)
            if k > 0:
                yield ("wait", "QE", k - 1)
                p0, p1 = self.units[k - 1]
                b = self.base(k - 1)
                assert all(("S", (i, k - 1, j, b + j)) in self.mma_done for i, n in ((0, p0), (1, p1))
                           for j in range(n)), "Q reloaded before the last S read it"
            self.qunit = None
            self.landing.append(("Q", 0, k, "Q"))
            yield ("step",)
            for j in range(nkv):
                gg = g + j
                s = gg % self.ST
                yield ("wait", f"KE{s}", gg // self.ST - 1)
                if gg >= self.ST:
                    old_t = gg - self.ST
                    assert not any(x[0] == "S" and x[1][3] == old_t for x in self.pending()), \
                        "K stage reloaded while an S product may read it"
                self.kst[s] = None
                self.landing.append(("K", s, gg, f"KF{s}"))
                yield ("step",)
                yield ("wait", f"VE{s}", gg // self.ST - 1)
                if gg >= self.ST:
                    old_t = gg - self.ST
                    assert not any(x[0] == "PV" and x[1][3] == old_t for x in self.pending()), \
                        "V stage reloaded while a P.V may read it"
                self.vst[s] = None
                self.landing.append(("V", s, gg, f"VF{s}"))
                yield ("step",)
            g += nkv

    def mma(self):
        g, gp = 0, [0, 0]
        for k, (n0, n1) in enumerate(self.units):
            nkv = max(n0, n1)
            yield ("wait", "Q", k)
            for j in range(nkv + 1):
                for sub, n in ((0, n0), (1, n1)):
                    if j > n:
                        continue
                    if j == 1 and k > 0:
                        yield ("wait", f"OF{sub}", k - 1)
                    if j > 0:
                        gg = g + j - 1
                        yield ("wait", f"VF{gg % self.ST}", gg // self.ST)
                        yield ("wait", f"PF{sub}", gp[sub] + j - 1)
                        self.issue(0, "PV", (sub, k, j - 1, gg))
                        if j == n:
                            self.commit(0, f"OD{sub}")
                        yield ("step",)
                    if j < n:
                        gg = g + j
                        yield ("wait", f"KF{gg % self.ST}", gg // self.ST)
                        self.issue(0, "S", (sub, k, j, gg))
                        self.commit(0, f"SF{sub}")
                        yield ("step",)
            g += nkv
            gp[0] += n0
            gp[1] += n1
        self.commit(0, "DR")
        yield ("wait", "DR", 0)

    def softmax(self, sub, w):
        g, gs = 0, 0
        for k, (n0, n1) in enumerate(self.units):
            nkv, n = max(n0, n1), (n1 if sub else n0)
            for j in range(n):
                yield ("wait", f"SF{sub}", gs + j)
                assert ("S", (sub, k, j, g + j)) in self.mma_done
                if j > 0:
                    self.bars[f"VE{(g + j - 1) % self.ST}"].arrive()
                self.bars[f"KE{(g + j) % self.ST}"].arrive()
                self.bump(("p", sub, k), j)
                self.bars[f"PF{sub}"].arrive()
                if j == n - 1:
                    self.bars["QE"].arrive()
                yield ("step",)
            for jj in range(n, nkv):
                gg = g + jj
                yield ("wait", f"KF{gg % self.ST}", gg // self.ST)
                yield ("wait", f"VF{gg % self.ST}", gg // self.ST)
                self.bars[f"VE{gg % self.ST}"].arrive()
                self.bars[f"KE{gg % self.ST}"].arrive()
                yield ("step",)
            yield ("wait", f"OD{sub}", k)
            assert all(("PV", (sub, k, j, g + j)) in self.mma_done for j in range(n)), "epilogue before the last P.V"
            self.bars[f"VE{(g + n - 1) % self.ST}"].arrive()
            self.o_read.add((sub, k))
            self.bars[f"OF{sub}"].arrive()
            yield ("step",)
            g += nkv
            gs += n

    def execute_head(self):
        warp, kind, _, key = self.pipe.pop(0)
        sub, k, j, gg = key
        self.mma_started.add((kind, key))
        if kind == "S":
            assert self.qunit == k, "S on a Q buffer without this unit's Q"
            assert self.kst[gg % self.ST] == gg, "S on a K stage without its tile"
            # S overwrites the P columns that the previous P.V of this sub-tile read
            prev = [x for x in self.mma_started if x[0] == "PV" and x[1][0] == sub]
            assert all(x in self.mma_done for x in prev), "S overwrote P before P.V read it"
        else:
            assert self.vst[gg % self.ST] == gg, "P.V on a V stage without its tile"
            assert self.count.get((("p", sub, k), j), 0) == 4, "P.V before every softmax warp wrote P"
            if j == 0 and k > 0:
                assert (sub, k - 1) in self.o_read, "P.V overwrote O before the epilogue read it"
        self.mma_done.add((kind, key))
        self.completed_by[warp] += 1

    def fire(self, e):
        if e[0] == "land":
            kind, s, x, bar = self.landing.pop(e[1])
            if kind == "K":
                self.kst[s] = x
            elif kind == "V":
                self.vst[s] = x
            else:
                self.qunit = x
            self.bars[bar].arrive()
        else:
            Model.fire(self, e)


@pytest.mark.parametrize("units", [
    [(3, 3)], [(2, 2), (2, 2), (2, 2)], [(1, 2), (4, 5), (2, 3)], [(5, 6), (1, 2)], [(1, 1), (1, 1), (1, 1), (1, 1)],
    [(3, 4), (3, 4), (1, 2), (6, 7)],
    # the streamed tail: whole units, then pieces of a few tiles (equal on both sub-tiles)
    [(4, 4), (4, 4), (1, 1), (2, 2)], [(3, 3), (1, 1)],
], ids=lambda u: "-".join(f"{a}.{b}" for a, b in u))
def test_forward_persistent_barrier_protocol(units):
    rng = random.Random(hash(tuple(units)) & 0xFFFFFFFF)
    for _ in range(400):
        PersistModel(units, rng).run()


class PersistCommitModel(PersistModel):
    """The persistent form at d = 64 (unmasked units only): three K/V stages
    freed by commits behind the MMAs instead of softmax arrivals, one commit
    per sub-tile's S product (K) and P.V (V), so a stage's release barrier
    counts two; the softmax warps release nothing."""

    ST = 3

    def __init__(self, units, rng):
        PersistModel.__init__(self, units, rng)
        for s in range(self.ST):
            self.bars[f"KE{s}"] = Bar(2)
            self.bars[f"VE{s}"] = Bar(2)

    def mma(self):
        g, gp = 0, [0, 0]
        for k, (n0, n1) in enumerate(self.units):
            assert n0 == n1, "the commit-freed form takes units with equal sub-tiles"
            nkv = n0
            yield ("wait", "Q", k)
            for j in range(nkv + 1):
                for sub in (0, 1):
                    if j == 1 and k > 0:
                        yield ("wait", f"OF{sub}", k - 1)
                    if j > 0:
                        gg = g + j - 1
                        yield ("wait", f"VF{gg % self.ST}", gg // self.ST)
                        yield ("wait", f"PF{sub}", gp[sub] + j - 1)
                        self.issue(0, "PV", (sub, k, j - 1, gg))
                        if j == nkv:
                            self.commit(0, f"OD{sub}")
                        self.commit(0, f"VE{gg % self.ST}")
                        yield ("step",)
                    if j < nkv:
                        gg = g + j
                        yield ("wait", f"KF{gg % self.ST}", gg // self.ST)
                        self.issue(0, "S", (sub, k, j, gg))
                        self.commit(0, f"SF{sub}")
                        self.commit(0, f"KE{gg % self.ST}")
                        yield ("step",)
            g += nkv
            gp[0] += n0
            gp[1] += n1
        self.commit(0, "DR")
        yield ("wait", "DR", 0)

    def softmax(self, sub, w):
        g, gs = 0, 0
        for k, (n0, n1) in enumerate(self.units):
            n = n0
            for j in range(n):
                yield ("wait", f"SF{sub}", gs + j)
                assert ("S", (sub, k, j, g + j)) in self.mma_done
                self.bump(("p", sub, k), j)
                self.bars[f"PF{sub}"].arrive()
                if j == n - 1:
                    self.bars["QE"].arrive()
                yield ("step",)
            yield ("wait", f"OD{sub}", k)
            assert all(("PV", (sub, k, j, g + j)) in self.mma_done for j in range(n)), "epilogue before the last P.V"
            self.o_read.add((sub, k))
            self.bars[f"OF{sub}"].arrive()
            yield ("step",)
            g += n
            gs += n


@pytest.mark.parametrize("units", [
    [(3, 3)], [(2, 2), (2, 2), (2, 2)], [(1, 1), (1, 1), (1, 1), (1, 1)], [(4, 4), (1, 1), (5, 5)], [(6, 6), (2, 2)],
], ids=lambda u: "-".join(f"{a}.{b}" for a, b in u))
def test_forward_persistent_d64_barrier_protocol(units):
    rng = random.Random(hash(tuple(units)) ^ 0x64)
    for _ in range(400):
        PersistCommitModel(units, rng).run()


def test_model_catches_a_commit_freed_stage_released_twice():
    """Planted mistake: the softmax warps also release the stages (as at
    d = 128) on top of the commits; a stage then completes its phase before
    both chains have read it."""
    class DoubleRelease(PersistCommitModel):
        def softmax(self, sub, w):
            g = 0
            for req in PersistCommitModel.softmax(self, sub, w):
                if req[0] == "wait" and req[1].startswith("SF") and w == 0:
                    yield req
                    self.bars[f"KE{req[2] % self.ST}"].arrive()
                    continue
                yield req
    with pytest.raises(AssertionError):
        for seed in range(300):
            DoubleRelease([(3, 3), (2, 2), (4, 4)], random.Random(seed)).run()


class PersistTwoWarpModel(PersistModel):
    """The persistent form with one MMA warp per sub-tile whose blocks
    alternate by turns, as in the one-unit kernel: sub-tile 0's block j >= 1
    waits for sub-tile 1's block j-1, its first block of a unit for
    sub-tile 1's last block of the previous unit; sub-tile 1's block j waits
    for sub-tile 0's block j while sub-tile 0 has one; a warp passes the turn
    only for a block the other waits for. Turn phases are counted across
    units, so a turn barrier holding two arrivals would show up as an
    aliased parity wait."""

    def __init__(self, units, rng):
        PersistModel.__init__(self, units, rng)
        self.bars.update({"T0": Bar(1), "T1": Bar(1), "DR0": Bar(1), "DR1": Bar(1)})

    def roles(self):
        return ([self.producer(), self.mma_warp(0), self.mma_warp(1)]
                + [self.softmax(sub, w) for sub in (0, 1) for w in range(4)])

    def mma_warp(self, sub):
        g, gp, nt = 0, 0, 0
        for k, (n0, n1) in enumerate(self.units):
            nkv = max(n0, n1)
            n_me, n_other = (n1, n0) if sub else (n0, n1)
            yield ("wait", "Q", k)
            for j in range(n_me + 1):
                if (j > 0 or k > 0) if sub == 0 else (j <= n_other):
                    yield ("wait", f"T{sub}", nt)
                    nt += 1
                if j == 1 and k > 0:
                    yield ("wait", f"OF{sub}", k - 1)
                if j > 0:
                    gg = g + j - 1
                    yield ("wait", f"VF{gg % self.ST}", gg // self.ST)
                    yield ("wait", f"PF{sub}", gp + j - 1)
                    self.issue(sub, "PV", (sub, k, j - 1, gg))
                    if j == n_me:
                        self.commit(sub, f"OD{sub}")
                    yield ("step",)
                if j < n_me:
                    gg = g + j
                    yield ("wait", f"KF{gg % self.ST}", gg // self.ST)
                    self.issue(sub, "S", (sub, k, j, gg))
                    self.commit(sub, f"SF{sub}")
                    yield ("step",)
                if sub == 0 or j < n_other or j == n_me:
                    self.bars[f"T{sub ^ 1}"].arrive()
                    yield ("step",)
            g += nkv
            gp += n_me
        self.commit(sub, f"DR{sub}")
        yield ("wait", f"DR{sub}", 0)


@pytest.mark.parametrize("units", [
    [(3, 3)], [(2, 2), (2, 2), (2, 2)], [(1, 2), (4, 5), (2, 3)], [(5, 6), (1, 2)], [(1, 1), (1, 1), (1, 1), (1, 1)],
    [(3, 4), (3, 4), (1, 2), (6, 7)], [(4, 4), (4, 4), (1, 1), (2, 2)], [(3, 3), (1, 1)], [(1, 2), (1, 2), (1, 2)],
], ids=lambda u: "-".join(f"{a}.{b}" for a, b in u))
def test_forward_persistent_two_mma_warps_barrier_protocol(units):
    rng = random.Random(hash(tuple(units)) & 0xFFFFFFFF)
    for _ in range(400):
        PersistTwoWarpModel(units, rng).run()


def test_model_catches_a_turn_passed_for_every_block():
    """Planted mistake: sub-tile 1 passes the turn after every block, also
    the one sub-tile 0 does not wait for (a unit whose sub-tile 1 has one
    tile more); the extra arrival completes a turn phase early and a later
    parity wait aliases."""
    class EveryPass(PersistTwoWarpModel):
        def mma_warp(self, sub):
            if sub == 0:
                yield from PersistTwoWarpModel.mma_warp(self, 0)
                return
            units = self.units
            g, gp, nt = 0, 0, 0
            for k, (n0, n1) in enumerate(units):
                yield ("wait", "Q", k)
                for j in range(n1 + 1):
                    if j <= n0:
                        yield ("wait", "T1", nt)
                        nt += 1
                    if j == 1 and k > 0:
                        yield ("wait", "OF1", k - 1)
                    if j > 0:
                        gg = g + j - 1
                        yield ("wait", f"VF{gg % self.ST}", gg // self.ST)
                        yield ("wait", "PF1", gp + j - 1)
                        self.issue(1, "PV", (1, k, j - 1, gg))
                        if j == n1:
                            self.commit(1, "OD1")
                        yield ("step",)
                    if j < n1:
                        gg = g + j
                        yield ("wait", f"KF{gg % self.ST}", gg // self.ST)
                        self.issue(1, "S", (1, k, j, gg))
                        self.commit(1, "SF1")
                        yield ("step",)
                    self.bars["T0"].arrive()
                    yield ("step",)
                g += max(n0, n1)
                gp += n1
            self.commit(1, "DR1")
            yield ("wait", "DR1", 0)
    with pytest.raises(AssertionError):
        for seed in range(300):
            EveryPass([(1, 2), (4, 5), (2, 3), (3, 4)], random.Random(seed)).run()


def test_model_catches_an_early_release_of_an_unused_tile():
    """Planted mistake: the sub-tile that does not use a unit's last tile
    releases its stage at once instead of after the tile landed; its arrivals
    can then complete the stage's previous phase early."""
    class EarlyRelease(PersistModel):
        def softmax(self, sub, w):
            for req in PersistModel.softmax(self, sub, w):
                if req[0] == "wait" and req[1][:2] in ("KF", "VF") and self.rng.random() < 0.9:
                    continue
                yield req
    with pytest.raises(AssertionError):
        for seed in range(300):
            EarlyRelease([(1, 2), (4, 5), (2, 3), (3, 4)], random.Random(seed)).run()
