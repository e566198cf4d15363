"""A model of the grouped W4A16 GEMM's mbarrier protocol (grouped_gemm.cu),
run under random interleavings on the CPU, in the manner of
test_dense_pipeline_protocol.py.

Roles as the kernel writes them, with the kernel's constants: the two TMA
threads for codes (one per parity of the CTA's stage sequence, 6 code stages
in all; the parity-0 one also issues the 2 or 3 scale/zero stages), the TMA
warp for activations (3 streamed slots, or 2 resident slots that hold a
job's whole activation block, the group-sum block included), four MMA
issuers (issuer r takes ring r: two A buffers in tensor memory that take the
ring's fills in turn, and its own accumulator in each of two sets; each
issuer's commits complete asynchronously in its issue order), sixteen
dequantisation warps (lane quarter x ring; ring r takes 64-code slice r of
every stage, i.e. the unit's blocks j with j % 4 == r, and ring blocks % 4
(ring unit % 4 when blocks % 4 == 0) also takes the unit's group-constant
correction) and
four epilogue warps (which also read the row scales the ring-0 dequant
warps publish per unit).  Every wait is checked against the exact
condition: the phase it stands for, counted from per-stage uses kept apart
from the kernel's parity variables, has completed exactly when the parity
test says so.  Unit lists mix jobs of 16 and 32 slots over several panels;
contraction sizes cover gate_up (2816, streamed, 11 stages per unit), down
(704, resident, a last stage with three of its four slices) and short ones
(384, 192, 320, 128, 64).
"""
import random

import pytest

RINGS, RING_BUFS, SETS, ISSUERS = 4, 2, 2, 4
# code stages (16 KB) and streamed activation slots (32 KB); resident mode
# has the same code stages and two job slots
STAGES_W_STREAMED, STAGES_W_RESIDENT, STAGES_B = 6, 6, 3
STAGE_B_BYTES = 32768
DQ_WARPS, EPI_WARPS = 16, 4
CHUNK_K, SLICE_K, MAX_N, RES_BYTES = 256, 64, 32, 49152
ROW_SCALE_SETS = 8


def sz_stages(G):
    return 2 if G > 16 else 3


def block_ring(j):
    return j & (RINGS - 1)


def corr_ring(n_unit, n_blocks):
    rest = n_blocks & (RINGS - 1)
    return rest if rest else n_unit & (RINGS - 1)


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
    return STAGE_B_BYTES // (n * 128)


class Grouped:
    def __init__(self, K, units, rng, group=None, big=False):
        """big: the big-job mode (jobs of up to 64 slots, activations always
        streamed, two issuers taking rings r and r + 2)."""
        self.K, self.units, self.rng = K, units, rng
        self.n_iss = 2 if big else ISSUERS
        group = group or (128 if K % 128 == 0 and K > 704 else 64)
        self.G = K // group
        self.n_sz = sz_stages(self.G)
        self.n_kchunks = (K + CHUNK_K - 1) // CHUNK_K
        self.n_blocks = K // SLICE_K
        self.resident = not big and (K + 64) * 2 * MAX_N <= RES_BYTES
        self.stages_w = STAGES_W_RESIDENT if self.resident else STAGES_W_STREAMED
        B = lambda name, n, c: [Bar(f"{name}{i}", c) for i in range(n)]
        self.w_full = B("w_full", self.stages_w, 1)
        self.w_empty = B("w_empty", self.stages_w, DQ_WARPS)
        nb = 2 if self.resident else STAGES_B
        self.b_full, self.b_empty = B("b_full", nb, 1), B("b_empty", nb, self.n_iss)
        # ring r's buffer b is a_full / a_empty [r * RING_BUFS + b]
        self.a_full = B("a_full", RINGS * RING_BUFS, 4)
        self.a_empty = B("a_empty", RINGS * RING_BUFS, 1)
        self.acc_full, self.acc_empty = B("acc_full", SETS, self.n_iss), B("acc_empty", SETS, EPI_WARPS)
        self.sz_full = B("sz_full", self.n_sz, 1)
        self.sz_empty = B("sz_empty", self.n_sz, DQ_WARPS)
        # row-scale tables (dequant -> epilogue), one entry per lane quarter
        self.row_scale = [[None] * 4 for _ in range(ROW_SCALE_SETS)]
        self.copies = []
        self.commits = [[] for _ in range(ISSUERS)]

    def tma_w(self, gp):
        """The code stages of parity gp of the CTA's stage sequence, unit by
        unit; the parity-0 thread issues each unit's scales and zeros before
        the unit's stages."""
        w_fill, sz_fill = [0] * self.stages_w, [0] * self.n_sz
        for n in range(len(self.units)):
            if gp == 0:
                szb = n % self.n_sz
                yield ("wait", self.sz_empty[szb], ((n // self.n_sz) & 1) ^ 1, sz_fill[szb] - 1)
                yield ("copy", self.sz_full[szb])
                sz_fill[szb] += 1
            gs0 = n * self.n_kchunks
            for kc in range(self.n_kchunks):
                g = gs0 + kc
                if self.stage_parity(g, kc) != gp:
                    continue
                sa = g % self.stages_w
                yield ("wait", self.w_empty[sa], ((g // self.stages_w) & 1) ^ 1, w_fill[sa] - 1)
                yield ("copy", self.w_full[sa])
                w_fill[sa] += 1

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
            for _ in range(0, self.K + 1, 64 * b_kcols(n)):     # blocks 0 .. K/64
                yield ("wait", self.b_empty[sb], ph_b ^ 1, fill[sb] - 1)
                yield ("copy", self.b_full[sb])
                fill[sb] += 1
                sb += 1
                if sb == STAGES_B:
                    sb, ph_b = 0, ph_b ^ 1

    def issuer(self, me):
        fill = {}               # per ring this issuer takes: its fills so far
        acc_use, b_use = [0] * SETS, [0] * (2 if self.resident else STAGES_B)
        cur_job, res_slot, b_seq = None, 0, 0
        nb = self.n_blocks

        def issue(ring):
            f = fill.get(ring, 0)
            buf = ring * RING_BUFS + f % RING_BUFS
            yield ("wait", self.a_full[buf], (f // RING_BUFS) & 1, f // RING_BUFS)
            fill[ring] = f + 1
            yield ("commit", me, self.a_empty[buf])

        def mine(ring):
            return ring % self.n_iss == me

        for n_unit, (job, n) in enumerate(self.units):
            st, acc_ph = n_unit & 1, (n_unit >> 1) & 1
            corr = corr_ring(n_unit, nb)
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
                for j in range(nb):
                    if mine(block_ring(j)):
                        yield from issue(block_ring(j))
                if mine(corr):
                    yield from issue(corr)
            else:
                kcols = b_kcols(n)
                n_bslots = nb // kcols + 1
                for t in range(n_bslots):
                    sb = (b_seq + t) % STAGES_B
                    yield ("wait", self.b_full[sb], ((b_seq + t) // STAGES_B) & 1, b_use[sb])
                    b_use[sb] += 1
                    for j in range(t * kcols, min(nb, (t + 1) * kcols)):
                        if mine(block_ring(j)):
                            yield from issue(block_ring(j))
                    if t == n_bslots - 1 and mine(corr):
                        yield from issue(corr)
                    yield ("commit", me, self.b_empty[sb])
                b_seq += n_bslots
            yield ("commit", me, self.acc_full[st])
            acc_use[st] += 1

    @staticmethod
    def stage_parity(g, kc):
        """Code producers by the stage's index in the CTA's stage sequence."""
        return g & 1

    def dequant(self, r, q=0):
        """Warp (q, r): slice r of every stage (block 4 kc + r of the unit),
        then the correction when r is the unit's correction ring."""
        szb = ph_sz = 0
        sz_use = [0] * self.n_sz
        w_use = [0] * self.stages_w
        fill = 0

        def fill_buffer(first):
            nonlocal fill
            buf = r * RING_BUFS + fill % RING_BUFS
            yield ("wait", self.a_empty[buf], ((fill // RING_BUFS) & 1) ^ 1,
                   fill // RING_BUFS - 1)
            if first:
                yield ("rs_write", n_unit, q)
            yield ("arrive", self.a_full[buf])
            fill += 1

        for n_unit, _u in enumerate(self.units):
            yield ("wait", self.sz_full[szb], ph_sz, sz_use[szb])
            gs0 = n_unit * self.n_kchunks
            for kc in range(self.n_kchunks):
                g = gs0 + kc
                sa = g % self.stages_w
                j = 4 * kc + r
                yield ("wait", self.w_full[sa], (g // self.stages_w) & 1, w_use[sa])
                w_use[sa] += 1
                yield ("arrive", self.w_empty[sa])
                if j >= self.n_blocks:
                    continue
                yield from fill_buffer(j == 0)
            if r == corr_ring(n_unit, self.n_blocks):
                yield from fill_buffer(False)
            yield ("arrive", self.sz_empty[szb])
            sz_use[szb] += 1
            szb += 1
            if szb == self.n_sz:
                szb, ph_sz = 0, ph_sz ^ 1

    def epilogue(self, q=0):
        use = [0] * SETS
        for n_unit, _u in enumerate(self.units):
            st = n_unit & 1
            yield ("wait", self.acc_full[st], (n_unit >> 1) & 1, use[st])
            use[st] += 1
            yield ("rs_read", n_unit, q)
            yield ("arrive", self.acc_empty[st])

    def run(self):
        roles = [self.tma_w(0), self.tma_w(1), self.tma_b()]
        roles += [self.issuer(i) for i in range(self.n_iss)]
        roles += [self.dequant(w // 4, w % 4) for w in range(DQ_WARPS)]   # 4 lane quarters per ring
        roles += [self.epilogue(q) for q in range(EPI_WARPS)]
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
            for q in range(ISSUERS):
                if self.commits[q]:
                    choices.append(("commit", q))
            if not choices:
                assert all(op is None for op in nxt), "deadlock: " + ", ".join(
                    f"{op[1].name} phase {op[3]}" for op in nxt if op is not None)
                return
            kind, i = self.rng.choice(choices)
            if kind == "copy":
                self.copies.pop(self.rng.randrange(len(self.copies))).arrive()
                continue
            if kind == "commit":
                self.commits[i].pop(0).arrive()   # an issuer's commits complete in order
                continue
            op = nxt[i]
            if op[0] == "arrive":
                op[1].arrive()
            elif op[0] == "copy":
                self.copies.append(op[1])
            elif op[0] == "rs_write":
                self.row_scale[op[1] % ROW_SCALE_SETS][op[2]] = op[1]
            elif op[0] == "rs_read":
                got = self.row_scale[op[1] % ROW_SCALE_SETS][op[2]]
                assert got == op[1], f"row scales of unit {op[1]} read as unit {got}'s"

            elif op[0] == "commit":
                self.commits[op[1]].append(op[2])
            nxt[i] = next(roles[i], None)


def _units(rng, n_units, big=False):
    """A CTA's unit list: panels of jobs in the kernel's round-robin order,
    consecutive units sometimes of the same job (short expert lists)."""
    units, job = [], 0
    while len(units) < n_units:
        n = rng.choice((16, 32, 48, 64) if big else (16, 32))
        for _ in range(rng.randint(1, 3)):
            units.append((job, n))
        job += 1
    return units[:n_units]


@pytest.mark.parametrize("K", [2816, 704, 384, 192, 320, 128, 64])
@pytest.mark.parametrize("seed", range(12))
def test_grouped_pipeline_protocol(K, seed):
    rng = random.Random(seed * 104729 + K)
    Grouped(K, _units(rng, rng.randint(1, 7)), rng).run()


@pytest.mark.parametrize("K", [2816, 704, 384, 192])
@pytest.mark.parametrize("seed", range(8))
def test_grouped_pipeline_protocol_big_jobs(K, seed):
    """Big-job mode: jobs of 16 to 64 slots, streamed activations, two
    issuers taking two rings each."""
    rng = random.Random(seed * 7919 + K)
    Grouped(K, _units(rng, rng.randint(1, 7), big=True), rng, big=True).run()


def test_the_grouped_model_catches_a_broken_protocol():
    """A dequant warp that waits on its A buffer with a fixed parity must
    fail the checks."""
    class Broken(Grouped):
        def dequant(self, r, q=0):
            for op in Grouped.dequant(self, r, q):
                if op[0] == "wait" and op[1] in self.a_empty:
                    op = (op[0], op[1], 1, op[3])
                yield op
    failures = 0
    for seed in range(20):
        rng = random.Random(seed)
        try:
            Broken(704, _units(rng, 6), rng).run()
        except AssertionError as e:
            assert "parity test" in str(e)
            failures += 1
    assert failures > 0


def test_the_grouped_model_catches_producers_by_stage_within_unit():
    """Splitting the code stages between the two producer threads by their
    index within the unit instead of in the CTA's stage sequence breaks the
    parity waits when a unit has an odd number of stages (gate_up: 11): both
    threads would fill the same stage slots."""
    class Broken(Grouped):
        @staticmethod
        def stage_parity(g, kc):
            return kc & 1                          # the broken rule
    failures = 0
    for seed in range(10):
        rng = random.Random(seed)
        try:
            Broken(2816, _units(rng, 4), rng).run()
        except AssertionError as e:
            # a skipped phase shows as a wrong parity test or as a deadlock
            assert "parity test" in str(e) or "deadlock" in str(e)
            failures += 1
    assert failures > 0


def test_the_grouped_model_catches_a_short_row_scale_table():
    """With two row-scale tables instead of eight, the ring-0 dequant warps
    of unit n + 2 can overwrite unit n's before its epilogue reads it."""
    global ROW_SCALE_SETS
    saved, ROW_SCALE_SETS = ROW_SCALE_SETS, 2
    failures = 0
    try:
        for seed in range(40):
            rng = random.Random(seed)
            try:
                Grouped(704, _units(rng, 7), rng).run()
            except AssertionError as e:
                assert "row scales" in str(e)
                failures += 1
    finally:
        ROW_SCALE_SETS = saved
    assert failures > 0
