"""A model of the grouped W4A16 GEMM's mbarrier protocol (grouped_gemm.cu),
run under random interleavings on the CPU, in the manner of
test_dense_pipeline_protocol.py.

Roles as the kernel writes them, with the kernel's constants: the TMA warp for
codes and scales/zeros (6 code stages, 2 or 3 scale stages), the TMA warp for
activations (3 streamed slots, or 2 resident slots that hold a job's whole
activation block, the group-sum block included), four MMA issuers (issuer
2h + p takes half p of every A buffer of ring h, two buffers per ring in
tensor memory; each has its own accumulator in each of two sets; each
issuer's commits complete asynchronously in its issue order), eight
dequantisation warps (lane quarter x half of each code stage, pipelined by
one item: a buffer's two halves are handed over only after the warp's next
item has been loaded and computed; the half whose ring takes sub-chunk n_sub
also produces the group-constant correction after its last sub-chunk of a
unit) and four epilogue warps.  Every wait is checked against the exact condition:
the phase it stands for, counted from per-stage uses kept apart from the
kernel's parity variables, has completed exactly when the parity test says
so.  Unit lists mix jobs of 16 and 32 slots over several panels; contraction
sizes cover gate_up (2816, streamed), down (704, resident, a 64-code last
sub-chunk) and short ones where one half has no sub-chunk in the last stage
(384, 192).
"""
import random

import pytest

RINGS, RING_BUFS, SETS, ISSUERS = 2, 2, 2, 4
STAGES_W, STAGES_B = 6, 3
DQ_WARPS, EPI_WARPS = 8, 4
CHUNK_K, SUB_K, MAX_N, RES_BYTES = 256, 128, 32, 49152


def sz_stages(G):
    return 2 if G > 16 else 3


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
    def __init__(self, K, units, rng, group=None):
        self.K, self.units, self.rng = K, units, rng
        group = group or (128 if K % 128 == 0 and K > 704 else 64)
        self.G = K // group
        self.n_sz = sz_stages(self.G)
        self.n_kchunks = (K + CHUNK_K - 1) // CHUNK_K
        self.n_sub = (K + SUB_K - 1) // SUB_K
        tail = K % SUB_K != 0
        self.corr_ring = (self.n_sub - 1) % 2 if tail else self.n_sub % 2
        self.resident = (K + 64) * 2 * MAX_N <= RES_BYTES
        B = lambda name, n, c: [Bar(f"{name}{i}", c) for i in range(n)]
        self.w_full, self.w_empty = B("w_full", STAGES_W, 1), B("w_empty", STAGES_W, DQ_WARPS)
        nb = 2 if self.resident else STAGES_B
        self.b_full, self.b_empty = B("b_full", nb, 1), B("b_empty", nb, ISSUERS)
        self.a_full = B("a_full", 2 * RINGS * RING_BUFS, 4)        # [buffer][half]
        self.a_empty = B("a_empty", RINGS * RING_BUFS, 2)
        self.acc_full, self.acc_empty = B("acc_full", SETS, ISSUERS), B("acc_empty", SETS, EPI_WARPS)
        self.sz_full = B("sz_full", self.n_sz, 1)
        self.sz_empty = B("sz_empty", self.n_sz, DQ_WARPS)
        self.copies = []
        self.commits = [[] for _ in range(ISSUERS)]

    # ---- roles; each wait carries (parity as the kernel computes it, the
    # phase index it stands for from independent use counts; -1: none yet)
    def tma_w(self):
        sa = szb = ph_a = ph_sz = 0
        w_fill, sz_fill = [0] * STAGES_W, [0] * self.n_sz
        for _job, _n in self.units:
            yield ("wait", self.sz_empty[szb], ph_sz ^ 1, sz_fill[szb] - 1)
            yield ("copy", self.sz_full[szb])
            sz_fill[szb] += 1
            szb += 1
            if szb == self.n_sz:
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
            for _ in range(0, self.K + 1, 64 * b_kcols(n)):     # blocks 0 .. K/64
                yield ("wait", self.b_empty[sb], ph_b ^ 1, fill[sb] - 1)
                yield ("copy", self.b_full[sb])
                fill[sb] += 1
                sb += 1
                if sb == STAGES_B:
                    sb, ph_b = 0, ph_b ^ 1

    def issuer(self, me):
        ring, part = me >> 1, me & 1
        ring_slot = ring_ph = 0
        a_use = [0] * RING_BUFS
        acc_use, b_use = [0] * SETS, [0] * (2 if self.resident else STAGES_B)
        cur_job, res_slot, b_seq = None, 0, 0

        def issue():
            nonlocal ring_slot, ring_ph
            buf = ring * RING_BUFS + ring_slot
            yield ("wait", self.a_full[2 * buf + part], ring_ph, a_use[ring_slot])
            a_use[ring_slot] += 1
            ring_slot += 1
            if ring_slot == RING_BUFS:
                ring_slot, ring_ph = 0, ring_ph ^ 1
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
                for _j in range(ring, self.n_sub, 2):
                    yield from issue()
                if ring == self.corr_ring:                   # the correction
                    yield from issue()
            else:
                kcols = b_kcols(n)
                subs = kcols // 2
                n_bslots = self.K // 64 // kcols + 1
                for t in range(n_bslots):
                    sb = (b_seq + t) % STAGES_B
                    yield ("wait", self.b_full[sb], ((b_seq + t) // STAGES_B) & 1, b_use[sb])
                    b_use[sb] += 1
                    for _j in range(t * subs + ring, min(self.n_sub, (t + 1) * subs), 2):
                        yield from issue()
                    if t == n_bslots - 1 and ring == self.corr_ring:
                        yield from issue()
                    yield ("commit", me, self.b_empty[sb])
                b_seq += n_bslots
            yield ("commit", me, self.acc_full[st])
            acc_use[st] += 1

    def dequant(self, h):
        # pipelined by one item: a buffer is handed over (both halves) only
        # after the next item of the same warp has been loaded and computed
        sa = szb = ph_a = ph_sz = 0
        ring_slot = ring_ph = 0
        w_use, sz_use, a_fill = [0] * STAGES_W, [0] * self.n_sz, [0] * RING_BUFS
        pend = None

        def flush():
            nonlocal pend
            if pend is not None:
                yield ("arrive", self.a_full[2 * pend])
                yield ("arrive", self.a_full[2 * pend + 1])
                pend = None

        def claim():
            nonlocal ring_slot, ring_ph, pend
            buf = h * RING_BUFS + ring_slot
            yield ("wait", self.a_empty[buf], ring_ph ^ 1, a_fill[ring_slot] - 1)
            a_fill[ring_slot] += 1
            ring_slot += 1
            if ring_slot == RING_BUFS:
                ring_slot, ring_ph = 0, ring_ph ^ 1
            pend = buf

        for _job, _n in self.units:
            yield ("wait", self.sz_full[szb], ph_sz, sz_use[szb])
            for kc in range(self.n_kchunks):
                yield ("wait", self.w_full[sa], ph_a, w_use[sa])
                w_use[sa] += 1
                mine = 2 * kc + h < self.n_sub
                yield ("arrive", self.w_empty[sa])
                sa += 1
                if sa == STAGES_W:
                    sa, ph_a = 0, ph_a ^ 1
                if not mine:
                    continue
                yield from flush()
                yield from claim()
            if self.corr_ring == h:          # the correction sub-chunk
                yield from flush()
                yield from claim()
            yield ("arrive", self.sz_empty[szb])
            sz_use[szb] += 1
            szb += 1
            if szb == self.n_sz:
                szb, ph_sz = 0, ph_sz ^ 1
        yield from flush()

    def epilogue(self):
        use = [0] * SETS
        for n_unit, _u in enumerate(self.units):
            st = n_unit & 1
            yield ("wait", self.acc_full[st], (n_unit >> 1) & 1, use[st])
            use[st] += 1
            yield ("arrive", self.acc_empty[st])

    def run(self):
        roles = [self.tma_w(), self.tma_b()] + [self.issuer(i) for i in range(ISSUERS)]
        roles += [self.dequant(w // 4) for w in range(DQ_WARPS)]      # 4 lane quarters per half
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


@pytest.mark.parametrize("K", [2816, 704, 384, 192, 320, 128, 64])
@pytest.mark.parametrize("seed", range(12))
def test_grouped_pipeline_protocol(K, seed):
    rng = random.Random(seed * 104729 + K)
    Grouped(K, _units(rng, rng.randint(1, 7)), rng).run()


def test_the_grouped_model_catches_a_broken_protocol():
    """A dequant warp that waits on its A buffer with the parity of the
    wrong slot must fail the checks."""
    class Broken(Grouped):
        def dequant(self, h):
            for op in Grouped.dequant(self, h):
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
