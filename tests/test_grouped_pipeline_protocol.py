"""A model of the grouped W4A16 GEMM's mbarrier protocol (grouped_gemm.cu),
run under random interleavings on the CPU, in the manner of
test_dense_pipeline_protocol.py.

Roles as the kernel writes them, with the kernel's constants: the TMA warp for
codes and scales/zeros (5 code stages, 3 scale stages), the TMA warp for
activations (3 streamed slots, or 2 resident slots that hold a job's whole
activation block), four MMA issuers (two A buffers each in tensor memory, two
accumulator sets; their commits complete asynchronously in issue order per
issuer), sixteen dequantisation warps (lane quarter x sub-chunk) and four
epilogue warps.  Every wait is checked against the exact condition: the phase
it stands for, counted from per-stage uses kept apart from the kernel's
parity variables, has completed exactly when the parity test says so.  Unit
lists mix jobs of 16 and 32 slots over several panels; contraction sizes
cover gate_up (2816, streamed), down (704, resident) and short ones where an
issuer has no sub-chunk (192, 384).
"""
import random

import pytest

ISSUERS, BUFS, SETS = 4, 2, 2
STAGES_W, STAGES_B, STAGES_SZ = 5, 3, 3
DQ_WARPS, EPI_WARPS = 16, 4
CHUNK_K, SUB_K, MAX_N, RES_BYTES = 256, 64, 32, 49152


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.arrived, self.completed = name, count, 0, 0

    def arrive(self):
        self.arrived += 1
        assert self.arrived <= self.count, self.name
        if self.arrived == self.count:
            self.arrived = 0
            self.completed += 1


def b_kcols(n):
    return 16 if n == 16 else 8


class Grouped:
    def __init__(self, K, units, rng):
        self.K, self.units, self.rng = K, units, rng
        self.n_kchunks = (K + CHUNK_K - 1) // CHUNK_K
        self.n_sub = K // SUB_K
        self.resident = K // 64 <= 256 and K * 2 * MAX_N <= RES_BYTES
        B = lambda name, n, c: [Bar(f"{name}{i}", c) for i in range(n)]
        self.w_full, self.w_empty = B("w_full", STAGES_W, 1), B("w_empty", STAGES_W, DQ_WARPS)
        nb = 2 if self.resident else STAGES_B
        self.b_full, self.b_empty = B("b_full", nb, 1), B("b_empty", nb, ISSUERS)
        self.a_full = B("a_full", ISSUERS * BUFS, 4)
        self.a_empty = B("a_empty", ISSUERS * BUFS, 1)
        self.acc_full, self.acc_empty = B("acc_full", SETS, ISSUERS), B("acc_empty", SETS, EPI_WARPS)
        self.sz_full, self.sz_empty = B("sz_full", STAGES_SZ, 1), B("sz_empty", STAGES_SZ, DQ_WARPS)
        self.copies = []
        self.commits = [[] for _ in range(ISSUERS)]

    # ---- roles; each wait carries (parity as the kernel computes it, the
    # phase index it stands for from independent use counts; -1: none yet)
    def tma_w(self):
        sa = szb = ph_a = ph_sz = 0
        w_fill, sz_fill = [0] * STAGES_W, [0] * STAGES_SZ
        for _job, _n in self.units:
            yield ("wait", self.sz_empty[szb], ph_sz ^ 1, sz_fill[szb] - 1)
            yield ("copy", self.sz_full[szb])
            sz_fill[szb] += 1
            szb += 1
            if szb == STAGES_SZ:
                szb, ph_sz = 0, ph_sz ^ 1
            for _ in range(self.n_kchunks):
                yield ("wait", self.w_empty[sa], ph_a ^ 1, w_fill[sa] - 1)
                yield ("copy", self.w_full[sa])
                w_fill[sa] += 1
                sa += 1
                if sa == STAGES_W:
                    sa, ph_a = 0, ph_a ^ 1

    def tma_b(self):
        if self.resident:
            cur, b_seq, fill = None, 0, [0, 0]
            for job, _n in self.units:
                if job == cur:
                    continue
                cur = job
                s, ph = b_seq & 1, (b_seq >> 1) & 1
                yield ("wait", self.b_empty[s], ph ^ 1, fill[s] - 1)
                yield ("copy", self.b_full[s])
                fill[s] += 1
                b_seq += 1
            return
        sb = ph_b = 0
        fill = [0] * STAGES_B
        for _job, n in self.units:
            for _ in range(0, self.K, 64 * b_kcols(n)):
                yield ("wait", self.b_empty[sb], ph_b ^ 1, fill[sb] - 1)
                yield ("copy", self.b_full[sb])
                fill[sb] += 1
                sb += 1
                if sb == STAGES_B:
                    sb, ph_b = 0, ph_b ^ 1

    def issuer(self, me):
        a_slot = a_ph = 0
        a_use = [0] * BUFS
        acc_use, b_use = [0] * SETS, [0] * (2 if self.resident else STAGES_B)
        cur_job, res_slot, b_seq = None, 0, 0

        def issue():
            nonlocal a_slot, a_ph
            buf = me + ISSUERS * a_slot
            yield ("wait", self.a_full[buf], a_ph, a_use[a_slot])
            a_use[a_slot] += 1
            a_slot += 1
            if a_slot == BUFS:
                a_slot, a_ph = 0, a_ph ^ 1
            yield ("commit", me, self.a_empty[buf])

        for n_unit, (job, n) in enumerate(self.units):
            st, acc_ph = n_unit & 1, (n_unit >> 1) & 1
            yield ("wait", self.acc_empty[st], acc_ph ^ 1, acc_use[st] - 1)
            if self.resident:
                if job != cur_job:
                    if cur_job is not None:
                        yield ("commit", me, self.b_empty[res_slot])
                    res_slot = b_seq & 1
                    yield ("wait", self.b_full[res_slot], (b_seq >> 1) & 1, b_use[res_slot])
                    b_use[res_slot] += 1
                    b_seq += 1
                    cur_job = job
                for _j in range(me, self.n_sub, ISSUERS):
                    yield from issue()
            else:
                kb_cap = 64 * b_kcols(n)
                n_bslots = (self.K + kb_cap - 1) // kb_cap
                for t in range(n_bslots):
                    sb = (b_seq + t) % STAGES_B
                    yield ("wait", self.b_full[sb], ((b_seq + t) // STAGES_B) & 1, b_use[sb])
                    b_use[sb] += 1
                    j0 = t * (kb_cap // SUB_K)
                    j1 = min(self.n_sub, j0 + kb_cap // SUB_K)
                    j = j0 + ((me - j0) % ISSUERS + ISSUERS) % ISSUERS
                    while j < j1:
                        yield from issue()
                        j += ISSUERS
                    yield ("commit", me, self.b_empty[sb])
                b_seq += n_bslots
            yield ("commit", me, self.acc_full[st])
            acc_use[st] += 1

    def dequant(self, sub):
        sa = szb = ph_a = ph_sz = 0
        a_slot = a_ph = 0
        w_use, sz_use, a_fill = [0] * STAGES_W, [0] * STAGES_SZ, [0] * BUFS
        for _job, _n in self.units:
            yield ("wait", self.sz_full[szb], ph_sz, sz_use[szb])
            for kc in range(self.n_kchunks):
                yield ("wait", self.w_full[sa], ph_a, w_use[sa])
                w_use[sa] += 1
                mine = kc * (CHUNK_K // SUB_K) + sub < self.n_sub
                yield ("arrive", self.w_empty[sa])
                sa += 1
                if sa == STAGES_W:
                    sa, ph_a = 0, ph_a ^ 1
                if not mine:
                    continue
                buf = sub + ISSUERS * a_slot
                yield ("wait", self.a_empty[buf], a_ph ^ 1, a_fill[a_slot] - 1)
                a_fill[a_slot] += 1
                a_slot += 1
                if a_slot == BUFS:
                    a_slot, a_ph = 0, a_ph ^ 1
                yield ("arrive", self.a_full[buf])
            yield ("arrive", self.sz_empty[szb])
            sz_use[szb] += 1
            szb += 1
            if szb == STAGES_SZ:
                szb, ph_sz = 0, ph_sz ^ 1

    def epilogue(self):
        use = [0] * SETS
        for n_unit, _u in enumerate(self.units):
            st = n_unit & 1
            yield ("wait", self.acc_full[st], (n_unit >> 1) & 1, use[st])
            use[st] += 1
            yield ("arrive", self.acc_empty[st])

    def run(self):
        roles = [self.tma_w(), self.tma_b()] + [self.issuer(i) for i in range(ISSUERS)]
        roles += [self.dequant(w // 4) for w in range(DQ_WARPS)]      # 4 lane quarters per sub
        roles += [self.epilogue() for _ in range(EPI_WARPS)]
        nxt = [next(r, None) for r in roles]
        steps = 0
        while True:
            steps += 1
            assert steps < 500000
            choices = []
            for i, op in enumerate(nxt):
                if op is None:
                    continue
                if op[0] == "wait":
                    bar, parity, target = op[1], op[2], op[3]
                    hw = (bar.completed & 1) != parity
                    exact = bar.completed >= target + 1
                    assert hw == exact, (
                        f"{bar.name}: parity test {hw} but phase {target} "
                        f"{'complete' if exact else 'pending'} (completed {bar.completed})")
                    if hw:
                        choices.append(("role", i))
                else:
                    choices.append(("role", i))
            if self.copies:
                choices.append(("copy", None))
            for k in range(ISSUERS):
                if self.commits[k]:
                    choices.append(("commit", k))
            if not choices:
                assert all(op is None for op in nxt), "deadlock: " + ", ".join(
                    f"{op[1].name} phase {op[3]}" for op in nxt if op is not None)
                return
            kind, i = self.rng.choice(choices)
            if kind == "copy":
                self.copies.pop(self.rng.randrange(len(self.copies))).arrive()
                continue
            if kind == "commit":
                self.commits[i].pop(0).arrive()
                continue
            op = nxt[i]
            if op[0] == "arrive":
                op[1].arrive()
            elif op[0] == "copy":
                self.copies.append(op[1])
            elif op[0] == "commit":
                self.commits[op[1]].append(op[2])
            nxt[i] = next(roles[i], None)


def _units(rng, n_units):
    """A CTA's unit list: panels of jobs in the kernel's round-robin order,
    consecutive units sometimes of the same job (short expert lists)."""
    units, job = [], 0
    while len(units) < n_units:
        n = rng.choice((16, 32))
        for _ in range(rng.randint(1, 3)):
            units.append((job, n))
        job += 1
    return units[:n_units]


@pytest.mark.parametrize("K", [2816, 704, 384, 192])
@pytest.mark.parametrize("seed", range(12))
def test_grouped_pipeline_protocol(K, seed):
    rng = random.Random(seed * 104729 + K)
    Grouped(K, _units(rng, rng.randint(1, 7)), rng).run()


def test_the_grouped_model_catches_a_broken_protocol():
    """A dequant warp that waits on its A buffer with the parity of the
    wrong slot must fail the checks."""
    class Broken(Grouped):
        def dequant(self, sub):
            for op in Grouped.dequant(self, sub):
                if op[0] == "wait" and op[1] in self.a_empty:
                    op = (op[0], op[1], 1, op[3])
                yield op
    failures = 0
    for seed in range(20):
        rng = random.Random(seed)
        try:
            Broken(704, _units(rng, 6), rng).run()
        except AssertionError:
            failures += 1
    assert failures > 0
