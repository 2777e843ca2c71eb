"""A model of the split-P two-tile attention kernel's barrier protocol, run on the CPU.

attn_f16_fwd3_kernel (csrc/attn3_kernels.cuh, head dimension 64) walks the
same units as the two-tile kernel (two query tiles A and B of one head, a last
unit of tile A alone on some CTAs, causal units whose tile A reads one block
fewer than B), but each tile's P has a tensor-memory buffer of its own.  So S
of block j + 1 may overwrite the score buffer as soon as the tile's softmax
warps have read S of block j into registers (they arrive on s_free), and it
runs on the tensor core while they compute P of block j.  A softmax warp
writes P of block j only once P V of block j - 1, which reads the P buffer,
has completed (pv_done).  K and V sit in rings of three slots; the MMA warp
frees a slot with a commit to its k_empty / v_empty barrier after the last
MMA that reads it (tile B's in a two-tile unit, which reads every block).

Every role is written as the sequence of its mbarrier waits and arrivals in
the kernel's order and with its phase arithmetic; a scheduler runs the roles,
the TMA completions (any order) and the tensor pipe (in issue order) in
seeded random interleavings.  Checked: no deadlock, no over-arrival, every
parity wait finding its barrier at exactly the phase it means, and no write
over data that is still to be read: S into a score buffer a softmax warp
reads, P into a buffer a queued P V reads, O rescaled under a queued P V or
overwritten by a unit's first P V before the output is read out (no barrier
of its own: each softmax warp arrives on p_full of a unit's first block only
after reading the previous unit's O, so that P V's wait on p_full covers
it), a K or V
slot loaded while a queued MMA reads its previous block, Q reloaded under a
queued S (the Q reload waits for q_empty, committed after a unit's last S:
a single s_full barrier per tile could be up to three phases behind the
producer).  Four planted defects must each fail.
"""
import random

import pytest

STAGES = 3


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.n = name, count, count, 0, 0

    def arrive(self, tx=0):
        self.tx += tx
        self.pending -= 1
        assert self.pending >= 0, f"over-arrival on {self.name} in phase {self.n}"
        self._complete()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.n += 1
            self.pending = self.count

    def passes(self, parity):
        return (self.n & 1) != parity


def run_protocol3(units, seed, nsoft=2, defect=None):
    """`units` as in the two-tile model: an int n (two tiles, n blocks each),
    (n, False) (tile A alone, last), or (a, b) with b = a + 1 (causal).
    `defect`: "s_before_free" (the next S issued without waiting for s_free),
    "p_unguarded" (P written without waiting for the previous P V),
    "k_empty_a" (a K slot of a two-tile unit freed after tile A's S, not B's),
    "q_unguarded" (Q reloaded without waiting for the previous unit's last S)."""
    units = [(u, u) if isinstance(u, int) else (u[0], 0 if u[1] is False else u[1]) for u in units]
    assert all(b == 0 or b >= a for a, b in units)
    assert all(a[1] or not b[1] for a, b in zip(units, units[1:])), "one-tile units come last"
    rnd = random.Random(seed)
    q_full, q_empty, drain = Barrier("q_full", 1), Barrier("q_empty", 1), Barrier("drain", 1)
    k_full = [Barrier(f"k_full{i}", 1) for i in range(STAGES)]
    v_full = [Barrier(f"v_full{i}", 1) for i in range(STAGES)]
    k_empty = [Barrier(f"k_empty{i}", 1) for i in range(STAGES)]
    v_empty = [Barrier(f"v_empty{i}", 1) for i in range(STAGES)]
    s_full = {t: Barrier(f"s_full{t}", 1) for t in "AB"}
    s_free = {t: Barrier(f"s_free{t}", nsoft) for t in "AB"}
    p_full = {t: Barrier(f"p_full{t}", nsoft) for t in "AB"}
    pv_done = {t: Barrier(f"pv_done{t}", 1) for t in "AB"}
    tma, pipe = [], []
    s_readers = {"A": 0, "B": 0}      # softmax warps reading each tile's score buffer
    reads = {"A": {}, "B": {}}        # per tile and unit: softmax warps that have read O out
    outputs_read = {"A": 0, "B": 0}   # units whose O every softmax warp of the tile has read out
    q_unit = [None]                   # the unit whose Q tiles shared memory holds (or is loading)

    def wait(bar, index, who):
        return (bar, index & 1, who, index)

    def queued(op, t=None, slot=None, before=None):
        for e in pipe:
            if e[0] != op or (t is not None and e[1] != t):
                continue
            if slot is not None and not (e[3] % STAGES == slot and e[3] < before):
                continue
            return True
        return False

    def producer(is_k):
        g = 0
        for u, (na, nb) in enumerate(units):
            nr = nb if nb else na
            if is_k:
                if u > 0 and defect != "q_unguarded":
                    # the previous unit's last S has read Q (a commit after it)
                    yield wait(q_empty, u - 1, "producer Q")
                    assert not queued("s"), "Q reloaded under a queued S"
                q_unit[0] = u                         # the Q tiles in shared memory from here on
                ntiles = 2 if nb else 1
                q_full.arrive(tx=ntiles)
                for _ in range(ntiles):
                    tma.append(q_full)
            for j in range(nr):
                gb = g + j
                s = gb % STAGES
                if gb >= STAGES:
                    yield wait(k_empty[s] if is_k else v_empty[s], gb // STAGES - 1, "producer slot")
                assert not queued("s" if is_k else "pv", slot=s, before=gb), \
                    f"{'K' if is_k else 'V'} block {gb} loaded into slot {s} under a queued MMA"
                full = k_full[s] if is_k else v_full[s]
                full.arrive(tx=1)
                tma.append(full)
            g += nr

    def mma():
        g = 0
        gt = {"A": 0, "B": 0}
        nu = {"A": 0, "B": 0}

        def issue(op, t, tb, rb, commits, outputs_needed=None):
            if op == "s":
                assert s_readers[t] == 0, f"S_{t} of block {tb} issued while a softmax warp reads the buffer"
            pipe.append((op, t, tb, rb, commits, outputs_needed, unit[0]))

        unit = [0]
        for u, (na, nb) in enumerate(units):
            unit[0] = u
            n = {"A": na, "B": nb}
            tiles = "AB" if nb else "A"
            last = tiles[-1]                      # the last reader of every block of the unit
            nr = max(na, nb)
            yield wait(q_full, u, "mma Q")
            yield wait(k_full[g % STAGES], g // STAGES, "mma K")
            for t in tiles:
                commits = [s_full[t]]
                k_last = "A" if defect == "k_empty_a" else last
                if t == k_last:
                    commits.append(k_empty[g % STAGES])
                if n[t] == 1 and t == last:
                    commits.append(q_empty)           # the unit's last S
                issue("s", t, gt[t], g, commits)
            for j in range(nr):
                rb = g + j
                for t in tiles:
                    if j + 1 < n[t]:
                        if defect != "s_before_free":
                            yield wait(s_free[t], gt[t] + j, f"mma S{t} free")
                        yield wait(k_full[(rb + 1) % STAGES], (rb + 1) // STAGES, "mma K")
                        commits = [s_full[t]]
                        k_last = "A" if defect == "k_empty_a" else last
                        if t == k_last:
                            commits.append(k_empty[(rb + 1) % STAGES])
                        if j + 2 == n[t] and t == last:
                            commits.append(q_empty)   # the unit's last S
                        issue("s", t, gt[t] + j + 1, rb + 1, commits)
                for t in tiles:
                    if j < n[t]:
                        yield wait(p_full[t], gt[t] + j, f"mma P{t}")
                        yield wait(v_full[rb % STAGES], rb // STAGES, "mma V")
                        commits = [pv_done[t]]
                        if t == last:
                            commits.append(v_empty[rb % STAGES])
                        # a unit's first P V overwrites O: every earlier output must be read out
                        issue("pv", t, gt[t] + j, rb, commits, nu[t] if j == 0 else None)
            g += nr
            for t in tiles:
                gt[t] += n[t]
                nu[t] += 1
        pipe.append(("drain", None, None, -1, [drain], None, None))
        yield wait(drain, 0, "mma drain")

    def softmax(t):
        g = 0
        for u, (na, nb) in enumerate(units):
            if t == "B" and not nb:
                break
            n = na if t == "A" else nb
            for j in range(n):
                gb = g + j
                yield wait(s_full[t], gb, f"softmax{t} S")
                s_readers[t] += 1
                yield None                              # S read into registers
                s_readers[t] -= 1
                s_free[t].arrive()
                yield None                              # maximum, exponentials
                if j >= 1 and defect != "p_unguarded":
                    yield wait(pv_done[t], gb - 1, f"softmax{t} P free")
                assert not queued("pv", t), f"P_{t} of block {gb} written under a queued P V"
                if j >= 1 and rnd.random() < 0.3:
                    assert not queued("pv", t), f"O_{t} rescaled under a queued P V"
                yield None                              # P written (and O rescaled)
                p_full[t].arrive()
            gl = g + n - 1
            yield wait(pv_done[t], gl, f"softmax{t} output")
            yield None                                  # O read out of tensor memory
            reads[t][u] = reads[t].get(u, 0) + 1
            if reads[t][u] == nsoft:
                outputs_read[t] += 1
            g += n

    roles = [producer(True), producer(False), mma()] + [softmax(t) for t in "AB" for _ in range(nsoft)]
    current = [None] * len(roles)
    live = [True] * len(roles)
    for _ in range(2_000_000):
        ready = []
        for i in range(len(roles)):
            if not live[i]:
                continue
            if current[i] is None:
                ready.append(("role", i))
                continue
            bar, parity, who, index = current[i]
            assert bar.n <= index + 1, f"{who}: {bar.name} is {bar.n - index - 1} phase(s) past the awaited one"
            if bar.passes(parity):
                assert bar.n == index + 1, f"{who}: {bar.name} passes {index + 1 - bar.n} phase(s) early"
                ready.append(("role", i))
        if tma:
            ready.append(("tma", None))
        if pipe:
            ready.append(("pipe", None))
        if not ready:
            stuck = [f"{current[i][2]} on {current[i][0].name}" for i in range(len(roles)) if live[i]]
            assert not stuck, "deadlock: " + "; ".join(stuck)
            return
        kind, i = rnd.choice(ready)
        if kind == "tma":
            tma.pop(rnd.randrange(len(tma))).complete_tx(1)
        elif kind == "pipe":
            op, t, tb, rb, commits, outputs_needed, u = pipe.pop(0)     # in issue order
            if op == "s":
                assert s_readers[t] == 0, f"S_{t} of block {tb} overwrote a score buffer a softmax still reads"
                assert q_unit[0] == u, f"S_{t} of unit {u} read the Q tiles of unit {q_unit[0]}"
            if outputs_needed is not None:
                assert outputs_read[t] >= outputs_needed, f"P V of tile {t} overwrote O before it was read out"
            for bar in commits:
                bar.arrive()
        else:
            try:
                current[i] = next(roles[i])
            except StopIteration:
                live[i], current[i] = False, None
    raise AssertionError("no progress bound reached")


CASES = [[1], [2], [3], [4], [5], [2, 2], [8, 8, 8], [32, 32], [3, 1, 4], [1, 1, 1, 1],
         [(1, False)], [(5, False)], [(3, False), (3, False)], [4, (4, False)], [8, 8, (8, False)],
         [1, (1, False)], [2, 2, (2, False), (2, False)], [32, 32, (32, False)],
         [(1, 2)], [(3, 4), (1, 2)], [(31, 32), (1, 2), (29, 30), (3, 4)], [(5, 6), (5, 6)], [(1, 2), (1, 2), (1, 2)]]


@pytest.mark.parametrize("units", CASES)
def test_attention3_barrier_protocol(units):
    for seed in range(8):
        run_protocol3(units, seed)


@pytest.mark.parametrize("defect", ["s_before_free", "p_unguarded", "k_empty_a", "q_unguarded"])
def test_attention3_model_catches_planted_defects(defect):
    with pytest.raises(AssertionError):
        for seed in range(100):
            run_protocol3([4, 4, 3], seed, defect=defect)
