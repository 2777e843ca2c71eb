"""A model of the split-P two-tile attention kernel's barrier protocol, run on the CPU.

attn_f16_fwd3_kernel (csrc/attn3_kernels.cuh, head dimension 64) walks the
same units as the two-tile kernel (two query tiles A and B of one head, a last
unit of tile A alone on some CTAs, causal units whose tile A reads one block
fewer than B), but each tile's P has a tensor-memory buffer of its own.  So S
of block j + 1 may overwrite the score buffer as soon as the tile's softmax
warps have read S of block j into registers (they arrive on s_free), and it
runs on the tensor core while they compute P of block j.  A softmax warp
writes P of block j only once P V of block j - 1, which reads the P buffer,
has completed (pv_done).  Each tile has an MMA warp of its own, whose MMAs the
tensor pipe runs in order; the two warps' MMAs interleave in any order, and a
commit arrives once its own warp's earlier MMAs have completed.  K and V sit in
rings of three slots, each freed by one commit from each tile's warp to its
k_empty / v_empty barrier (count two) after its last MMA reading the slot; in
a one-tile unit tile A's warp commits twice, and in a causal unit tile A's
warp arrives for the last block, which it does not read, once that block has
landed.  The Q tiles are freed the same way (q_empty, after each tile's last
S of the unit).

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
queued S (the Q reload waits for q_empty: a single s_full barrier per tile
could be up to three phases behind the producer), an MMA reading a ring slot
that holds another block.  Five planted defects must each fail.
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
    "k_empty_b_only" (tile A's MMA warp never arrives on k_empty, whose count
    is still two), "q_unguarded" (Q reloaded without waiting for q_empty), or
    "early_extra" (tile A's extra arrival for the last block of a causal unit,
    which it does not read, made without waiting for that block's load)."""
    units = [(u, u) if isinstance(u, int) else (u[0], 0 if u[1] is False else u[1]) for u in units]
    assert all(b == 0 or b >= a for a, b in units)
    assert all(a[1] or not b[1] for a, b in zip(units, units[1:])), "one-tile units come last"
    rnd = random.Random(seed)
    q_full, q_empty, drain = Barrier("q_full", 1), Barrier("q_empty", 2), Barrier("drain", 2)
    k_full = [Barrier(f"k_full{i}", 1) for i in range(STAGES)]
    v_full = [Barrier(f"v_full{i}", 1) for i in range(STAGES)]
    k_empty = [Barrier(f"k_empty{i}", 2) for i in range(STAGES)]
    v_empty = [Barrier(f"v_empty{i}", 2) for i in range(STAGES)]
    s_full = {t: Barrier(f"s_full{t}", 1) for t in "AB"}
    s_free = {t: Barrier(f"s_free{t}", nsoft) for t in "AB"}
    p_full = {t: Barrier(f"p_full{t}", nsoft) for t in "AB"}
    pv_done = {t: Barrier(f"pv_done{t}", 1) for t in "AB"}
    tma = []
    # tensor pipe: each MMA warp's operations complete in its issue order; the two
    # warps' operations interleave in any order.  A commit arrives once every
    # earlier operation of its warp has completed.
    ops = {"A": [], "B": []}
    s_readers = {"A": 0, "B": 0}      # softmax warps reading each tile's score buffer
    reads = {"A": {}, "B": {}}        # per tile and unit: softmax warps that have read O out
    outputs_read = {"A": 0, "B": 0}   # units whose O every softmax warp of the tile has read out
    q_unit = [None]                   # the unit whose Q tiles shared memory holds (or is loading)
    slot_block = {"k": [None] * STAGES, "v": [None] * STAGES}   # block each ring slot holds

    def wait(bar, index, who):
        return (bar, index & 1, who, index)

    def queued(kind, t=None, slot=None, before=None):
        for w in "AB":
            for e in ops[w]:
                if e[0] != kind or (t is not None and e[1] != t):
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
                    # both tiles' last S of the previous unit have read Q
                    yield wait(q_empty, u - 1, "producer Q")
                    assert not queued("s"), "Q reloaded under a queued S"
                q_unit[0] = u
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
                slot_block["k" if is_k else "v"][s] = gb
                full = k_full[s] if is_k else v_full[s]
                full.arrive(tx=1)
                tma.append(full)
            g += nr

    def mma(t):
        """Tile t's MMA warp: the S and P V of every unit the tile takes part in,
        per block S of the next block (once the softmax has read this one's)
        before P V of this one."""
        g = 0                      # blocks loaded
        gt = 0                     # blocks this tile reads
        nu = 0                     # units this tile took part in

        def issue(kind, tb, rb, commits, outputs_needed=None, unit=None):
            if kind == "s":
                assert s_readers[t] == 0, f"S_{t} of block {tb} issued while a softmax warp reads the buffer"
            ops[t].append((kind, t, tb, rb, list(commits), outputs_needed, unit))

        def commit_now(bars):
            # a commit arrives once the warp's earlier operations complete (at once if none)
            if ops[t]:
                ops[t][-1][4].extend(bars)
            else:
                for b in bars:
                    b.arrive()

        for u, (na, nb) in enumerate(units):
            if t == "B" and not nb:
                break                                  # tile B's MMA warp sits out the one-tile units
            n = na if t == "A" else nb
            nr = max(na, nb)
            reps = 2 if nb == 0 else 1                 # a one-tile unit: tile A arrives for both warps
            yield wait(q_full, u, f"mma{t} Q")

            def s_commits(j):
                c = [s_full[t]]
                if not (defect == "k_empty_b_only" and t == "A"):
                    c += [k_empty[(g + j) % STAGES]] * reps
                if j == n - 1:
                    c += [q_empty] * reps              # the tile's last S of the unit has read Q
                return c

            yield wait(k_full[g % STAGES], g // STAGES, f"mma{t} K")
            issue("s", gt, g, s_commits(0), unit=u)
            for j in range(n):
                rb = g + j
                if j + 1 < n:
                    if defect != "s_before_free":
                        yield wait(s_free[t], gt + j, f"mma{t} S free")
                    yield wait(k_full[(rb + 1) % STAGES], (rb + 1) // STAGES, f"mma{t} K")
                    issue("s", gt + j + 1, rb + 1, s_commits(j + 1), unit=u)
                yield wait(p_full[t], gt + j, f"mma{t} P")
                yield wait(v_full[rb % STAGES], rb // STAGES, f"mma{t} V")
                issue("pv", gt + j, rb, [pv_done[t]] + [v_empty[rb % STAGES]] * reps, nu if j == 0 else None)
            if n < nr:
                # causal: tile A does not read the unit's last block; it arrives for
                # that block's slots once the block has landed (an earlier arrival
                # could count toward the slot's previous block)
                lb = g + nr - 1
                if defect != "early_extra":
                    yield wait(k_full[lb % STAGES], lb // STAGES, f"mma{t} K extra")
                    yield wait(v_full[lb % STAGES], lb // STAGES, f"mma{t} V extra")
                commit_now([k_empty[lb % STAGES], v_empty[lb % STAGES]])
            g += nr
            gt += n
            nu += 1
        commit_now([drain])
        yield wait(drain, 0, f"mma{t} drain")

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

    roles = [producer(True), producer(False), mma("A"), mma("B")] + [softmax(t) for t in "AB" for _ in range(nsoft)]
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
        for w in "AB":
            if ops[w]:
                ready.append(("pipe", w))
        if not ready:
            stuck = [f"{current[i][2]} on {current[i][0].name}" for i in range(len(roles)) if live[i]]
            assert not stuck, "deadlock: " + "; ".join(stuck)
            return
        kind, i = rnd.choice(ready)
        if kind == "tma":
            tma.pop(rnd.randrange(len(tma))).complete_tx(1)
        elif kind == "pipe":
            op, t, tb, rb, commits, outputs_needed, u = ops[i].pop(0)     # this warp's oldest operation
            if op == "s":
                assert s_readers[t] == 0, f"S_{t} of block {tb} overwrote a score buffer a softmax still reads"
                assert q_unit[0] == u, f"S_{t} of unit {u} read the Q tiles of unit {q_unit[0]}"
                assert slot_block["k"][rb % STAGES] == rb, f"S_{t} read K slot {rb % STAGES} holding another block"
            if op == "pv":
                assert slot_block["v"][rb % STAGES] == rb, f"P V_{t} read V slot {rb % STAGES} holding another block"
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


@pytest.mark.parametrize("defect,units", [("s_before_free", [4, 4, 3]), ("p_unguarded", [4, 4, 3]),
                                          ("k_empty_b_only", [4, 4, 3]), ("q_unguarded", [4, 4, 3]),
                                          ("early_extra", [(5, 6), (1, 2), (3, 4)])])
def test_attention3_model_catches_planted_defects(defect, units):
    with pytest.raises(AssertionError):
        for seed in range(200):
            run_protocol3(units, seed, defect=defect)
