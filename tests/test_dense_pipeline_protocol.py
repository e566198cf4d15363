"""A model of the dense W4A16 GEMM's mbarrier protocol (dense_gemm.cu), run
under random interleavings on the CPU.

Each actor follows its warp's loop as the kernel writes it: the two TMA
producers (code stages with scales/zeros, token tiles), the MMA issuer (its
commits complete asynchronously, in issue order), the four epilogue warps and
the eight dequantisation warps in four groups.  Copies complete in any order
after they are issued.  At every wait the model evaluates the hardware's
parity test (the phase in progress has the other parity) and the exact
condition (the awaited phase has completed); they must agree, or a wait would
pass early or miss its phase.  A state where nothing can move before the end
is a deadlock.  Sizes: both shared-memory configurations (3 code + 3 token
stages, 7 + 4), units of 1 to 13 steps (partial last code stages), 1 to 4
units per CTA.
"""
import random

import pytest

GROUPS = 4            # dequantisation groups = A stages
GROUP_WARPS = 2
DQ_WARPS = GROUPS * GROUP_WARPS
EPI_WARPS = 4


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.arrived, self.completed = name, count, 0, 0

    def arrive(self):
        self.arrived += 1
        assert self.arrived <= self.count, self.name
        if self.arrived == self.count:
            self.arrived = 0
            self.completed += 1


class Sim:
    def __init__(self, sw, sb, units, rng):
        self.rng = rng
        self.units = units
        B = lambda name, n, c: [Bar(f"{name}{i}", c) for i in range(n)]
        self.w_full, self.w_empty = B("w_full", sw, 1), B("w_empty", sw, DQ_WARPS)
        self.a_full, self.a_empty = B("a_full", GROUPS, GROUP_WARPS), B("a_empty", GROUPS, 1)
        self.b_full, self.b_empty = B("b_full", sb, 1), B("b_empty", sb, 1)
        self.acc_full, self.acc_empty = B("acc_full", 2, 1), B("acc_empty", 2, EPI_WARPS)
        self.sz_full, self.sz_empty = B("sz_full", 1, 1), B("sz_empty", 1, DQ_WARPS)
        self.sw, self.sb = sw, sb
        self.copies = []        # pending copy completions (any order)
        self.commits = []       # pending MMA commits (issue order)

    # ---- operations an actor yields.  A wait carries the parity the kernel
    # passes and, counted separately from the kernel's parity variables, the
    # index of the phase it stands for (-1: nothing to wait for yet).
    @staticmethod
    def wait(bar, parity, target):
        return ("wait", bar, parity, target)

    @staticmethod
    def copy(bar):
        return ("copy", bar)

    @staticmethod
    def commit(bar):
        return ("commit", bar)

    @staticmethod
    def arrive(bar):
        return ("arrive", bar)

    # ---- actors, mirroring the kernel's loops; uses[...] count each stage's
    # fills / visits independently of the parity bookkeeping
    def producer_w(self):
        sw = szb = 0
        ph_w = ph_sz = 0
        w_fills, sz_fills = [0] * self.sw, [0]
        for kc0, kc1 in self.units:
            yield self.wait(self.sz_empty[szb], ph_sz ^ 1, sz_fills[szb] - 1)
            yield self.copy(self.sz_full[szb])
            sz_fills[szb] += 1
            szb += 1
            if szb == 1:
                szb, ph_sz = 0, ph_sz ^ 1
            for _ in range(kc0, kc1, GROUPS):
                yield self.wait(self.w_empty[sw], ph_w ^ 1, w_fills[sw] - 1)
                yield self.copy(self.w_full[sw])
                w_fills[sw] += 1
                sw += 1
                if sw == self.sw:
                    sw, ph_w = 0, ph_w ^ 1

    def producer_b(self):
        sb = ph_b = 0
        fills = [0] * self.sb
        for kc0, kc1 in self.units:
            for _ in range(kc0, kc1):
                yield self.wait(self.b_empty[sb], ph_b ^ 1, fills[sb] - 1)
                yield self.copy(self.b_full[sb])
                fills[sb] += 1
                sb += 1
                if sb == self.sb:
                    sb, ph_b = 0, ph_b ^ 1

    def mma(self):
        sb = ph_b = apar = 0
        a_uses, b_uses, acc_uses = [0] * GROUPS, [0] * self.sb, [0, 0]
        for n_unit, (kc0, kc1) in enumerate(self.units):
            st = n_unit & 1
            yield self.wait(self.acc_empty[st], ((n_unit >> 1) & 1) ^ 1, acc_uses[st] - 1)
            for kc in range(kc0, kc1):
                sa = (kc - kc0) % GROUPS
                yield self.wait(self.a_full[sa], (apar >> sa) & 1, a_uses[sa])
                yield self.wait(self.b_full[sb], ph_b, b_uses[sb])
                yield self.commit(self.a_empty[sa])
                yield self.commit(self.b_empty[sb])
                a_uses[sa] += 1
                b_uses[sb] += 1
                apar ^= 1 << sa
                sb += 1
                if sb == self.sb:
                    sb, ph_b = 0, ph_b ^ 1
            yield self.commit(self.acc_full[st])
            acc_uses[st] += 1

    def epilogue(self):
        uses = [0, 0]
        for n_unit, _ in enumerate(self.units):
            st = n_unit & 1
            yield self.wait(self.acc_full[st], (n_unit >> 1) & 1, uses[st])
            yield self.arrive(self.acc_empty[st])
            uses[st] += 1

    def dequant(self, grp):
        szb = sw = 0
        ph_sz = ph_w = apar = 0
        sz_uses, w_uses, a_fills = [0], [0] * self.sw, 0
        for kc0, kc1 in self.units:
            yield self.wait(self.sz_full[szb], ph_sz, sz_uses[szb])
            for kc4 in range(kc0, kc1, GROUPS):
                yield self.wait(self.w_full[sw], ph_w, w_uses[sw])
                w_uses[sw] += 1
                have = kc4 + grp < kc1
                yield self.arrive(self.w_empty[sw])
                sw += 1
                if sw == self.sw:
                    sw, ph_w = 0, ph_w ^ 1
                if not have:
                    continue
                yield self.wait(self.a_empty[grp], (apar & 1) ^ 1, a_fills - 1)
                apar ^= 1
                a_fills += 1
                yield self.arrive(self.a_full[grp])
            yield self.arrive(self.sz_empty[szb])
            sz_uses[szb] += 1
            szb += 1
            if szb == 1:
                szb, ph_sz = 0, ph_sz ^ 1

    # ---- scheduler
    def run(self):
        actors = [self.producer_w(), self.producer_b(), self.mma()]
        actors += [self.epilogue() for _ in range(EPI_WARPS)]
        actors += [self.dequant(w // GROUP_WARPS) for w in range(DQ_WARPS)]
        nxt = [next(a) for a in actors]
        done = [False] * len(actors)
        steps = 0
        while True:
            steps += 1
            assert steps < 200000
            choices = []
            for i, op in enumerate(nxt):
                if done[i]:
                    continue
                if op[0] == "wait":
                    bar, parity, target = op[1], op[2], op[3]
                    hw = (bar.completed & 1) != parity        # the hardware's parity test
                    exact = bar.completed >= target + 1       # the phase awaited is complete
                    assert hw == exact, (
                        f"{bar.name}: parity test {hw} but phase {target} "
                        f"{'complete' if exact else 'pending'} (completed {bar.completed})")
                    if hw:
                        choices.append(("actor", i))
                else:
                    choices.append(("actor", i))
            if self.copies:
                choices.append(("copy", None))
            if self.commits:
                choices.append(("commit", None))
            if not choices:
                assert all(done), "deadlock: " + ", ".join(
                    f"{op[1].name} phase {op[3]} (completed {op[1].completed})"
                    for i, op in enumerate(nxt) if not done[i])
                return
            kind, i = self.rng.choice(choices)
            if kind == "copy":
                self.copies.pop(self.rng.randrange(len(self.copies))).arrive()
                continue
            if kind == "commit":
                self.commits.pop(0).arrive()
                continue
            op = nxt[i]
            if op[0] == "arrive":
                op[1].arrive()
            elif op[0] == "copy":
                self.copies.append(op[1])
            elif op[0] == "commit":
                self.commits.append(op[1])
            try:
                nxt[i] = next(actors[i])
            except StopIteration:
                done[i] = True


@pytest.mark.parametrize("cfg", [(3, 3), (7, 4)])
@pytest.mark.parametrize("seed", range(40))
def test_dense_pipeline_protocol(cfg, seed):
    rng = random.Random(seed * 7919 + cfg[0])
    n_units = rng.randint(1, 4)
    units = []
    for _ in range(n_units):
        kc0 = rng.randint(0, 40)
        units.append((kc0, kc0 + rng.randint(1, 13)))
    Sim(cfg[0], cfg[1], units, rng).run()


def test_the_model_catches_a_broken_protocol():
    """Variants that break the protocol must fail, so the checks are not
    vacuous: (1) the code stages released after one group instead of all
    four (a stage is refilled while other groups still wait for it);
    (2) a wait whose parity does not follow the stage's uses."""
    class EarlyRelease(Sim):
        def __init__(self, *a):
            super().__init__(*a)
            self.w_empty = [Bar(f"w_empty{i}", GROUP_WARPS) for i in range(self.sw)]

        def dequant(self, grp):
            for op in Sim.dequant(self, grp):
                if op[0] == "arrive" and op[1] in self.w_empty and grp != 0:
                    continue            # only group 0 releases the code stages
                yield op

    class FixedParity(Sim):
        def dequant(self, grp):
            for op in Sim.dequant(self, grp):
                if op[0] == "wait" and op[1] in self.a_empty:
                    op = (op[0], op[1], 1, op[3])    # parity no longer tracks the uses
                yield op

    for cls in (EarlyRelease, FixedParity):
        failures = 0
        for seed in range(30):
            try:
                cls(3, 3, [(0, 13), (13, 26), (26, 30)], random.Random(seed)).run()
            except AssertionError:
                failures += 1
        assert failures > 0, cls.__name__
