"""A model of the two-tile attention kernel's barrier protocol, run on the CPU.

attn_f16_fwd2_kernel (csrc/attn2_kernels.cuh) gives each CTA units of two
query tiles (A and B) of one head that share the K and V rings, and, when
the tiles do not divide evenly into two per CTA, a last unit of one tile
(A alone) on some CTAs.  Each tile
has one score buffer in tensor memory, which its P overwrites, and its own
output; the MMA thread issues S_A, S_B, then per key block P_A V, the next
S_A, P_B V, the next S_B, so one tile's MMAs run while the other tile's
softmax warps work.  Every role is written here as the sequence of its
mbarrier waits and arrivals in the kernel's order and with its phase
arithmetic; a scheduler runs the roles, the TMA completions (any order) and
the tensor pipe (in issue order) in seeded random interleavings.  Checked:
no deadlock, no barrier receiving more arrivals than its count in one phase,
every parity wait finding its barrier at exactly the phase it means, no
S writing a tile's score buffer while a softmax warp may still read it, and
no load overwriting a K or V ring slot that a queued or running MMA still
reads.  That P V of block j has read its P (in the score buffer) before S of
block j + 1 writes there rests on the tensor pipe executing one thread's
MMAs in issue order, which the model assumes as the kernel does.  Across
the switch from two-tile to one-tile units a ring slot's previous block may
have been read last by tile B's MMA; the producer then frees it on tile B's
barrier, later ones on tile A's.
"""
import random

import pytest


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


def run_protocol2(units, seed, nsoft=2, defect=None):
    """`units`: the units this CTA walks, each a number of key blocks (a unit
    of two tiles), a pair (key blocks, False) for a unit of tile A alone, or a
    pair (blocks of A, blocks of B) with B's one more (causal: tile A = 2k reads
    key blocks 0..2k, tile B = 2k + 1 reads 0..2k + 1, so B reads every block
    the unit loads); the one-tile units come last.  nsoft softmax warps per tile stand for the four.
    `defect` plants a mistake: "early_s" (the MMA thread issues the next S of a
    tile before that tile's P is written), "k_slot_a" (the producer frees a K
    slot on tile A's S instead of B's), "single_slot_a" (once the one-tile
    units begin, every slot is freed on tile A's barriers, also a slot whose
    previous block belonged to a two-tile unit), or "a_ring_phase" (the MMA
    thread takes tile A's barrier phases from the count of blocks loaded, which
    runs ahead of A's own count in causal units)."""
    # normalise to (blocks of A, blocks of B), B's 0 for a one-tile unit
    units = [(u, u) if isinstance(u, int) else (u[0], u[0] if u[1] is True else (0 if u[1] is False else u[1]))
             for u in units]
    assert all(b == 0 or b >= a for a, b in units), "tile B reads every block of a two-tile unit"
    assert all(a[1] or not b[1] for a, b in zip(units, units[1:])), "one-tile units come last"
    rnd = random.Random(seed)
    q_full, drain = Barrier("q_full", 1), Barrier("drain", 1)
    k_full = [Barrier(f"k_full{i}", 1) for i in range(2)]
    v_full = [Barrier(f"v_full{i}", 1) for i in range(2)]
    s_full = {"A": [Barrier(f"s_fullA{i}", 1) for i in range(2)], "B": [Barrier(f"s_fullB{i}", 1) for i in range(2)]}
    p_full = {t: Barrier(f"p_full{t}", nsoft) for t in "AB"}
    pv_done = {"A": [Barrier(f"pv_doneA{i}", 1) for i in range(2)], "B": [Barrier(f"pv_doneB{i}", 1) for i in range(2)]}
    o_free = {t: Barrier(f"o_free{t}", nsoft) for t in "AB"}
    tma, pipe = [], []
    # tensor-memory hazard: softmax warps that may still read each tile's score buffer
    s_readers = {"A": 0, "B": 0}

    def wait(bar, index, who):
        return (bar, index & 1, who, index)

    def producer(is_k):
        g = 0
        pair_end = 0                  # blocks of the two-tile units so far (they come first)
        prev_pair = True
        for u, (na, nbk) in enumerate(units):
            pair = nbk > 0
            nblk = nbk if pair else na      # blocks loaded: every block B reads, or A's
            if is_k:
                if g > 0:   # the previous unit's last S (S_B, issued after S_A, or S_A alone) has read Q
                    yield wait(s_full["B" if prev_pair else "A"][(g - 1) & 1], (g - 1) >> 1, "producer Q")
                ntiles = 2 if pair else 1
                q_full.arrive(tx=ntiles)
                for _ in range(ntiles):
                    tma.append(q_full)
            if pair:
                pair_end = g + nblk       # blocks below this one belong to two-tile units
            for j in range(nblk):
                gb = g + j
                s = gb & 1
                # the slot's previous block gb - 2 is done: both S (K) or both P V (V);
                # tile B's are issued after tile A's, so B's commits cover both; a
                # block of a one-tile unit was read by tile A alone
                t = "B" if gb - 2 < pair_end else "A"
                if is_k and defect == "k_slot_a":
                    t = "A"
                if defect == "single_slot_a" and not pair:
                    t = "A"
                yield wait(s_full[t][s] if is_k else pv_done[t][s], (gb >> 1) - 1, "producer slot")
                # the load overwrites ring slot s: no MMA reading its previous block may remain
                for op, _, _, rq in pipe:
                    assert not (rq is not None and rq & 1 == s and rq < gb and op == ("s" if is_k else "pv")), \
                        f"load of block {gb} into {'K' if is_k else 'V'} slot {s} while block {rq}'s MMA reads it"
                full = k_full[s] if is_k else v_full[s]
                full.arrive(tx=1)
                tma.append(full)
            g += nblk
            prev_pair = pair

    def mma():
        g = 0                          # ring blocks (every block loaded)
        gt = {"A": 0, "B": 0}          # each tile's own blocks: the phases of its barriers

        def issue_s(t, rb, tb):
            # S overwrites tile t's score buffer: no softmax may still read it and
            # no earlier P V may still read the P in it (the pipe is in order)
            pipe.append(("s", t, tb, rb))

        nb = 0                        # two-tile units so far
        for u, (na, nbk) in enumerate(units):
            n = {"A": na, "B": nbk}
            tiles = "AB" if nbk else "A"
            nr = max(na, nbk)
            yield wait(q_full, u, "mma Q")
            yield wait(k_full[g & 1], g >> 1, "mma K")
            for t in tiles:
                issue_s(t, g, gt[t])
            for j in range(nr):
                rb = g + j
                for t in tiles:
                    if j >= n[t]:
                        continue                   # tile A has no last block in a causal unit
                    tb = gt[t] + j
                    if defect == "a_ring_phase" and t == "A":
                        tb = rb
                    if defect == "early_s" and t == "A" and j + 1 < n[t]:
                        yield wait(k_full[(rb + 1) & 1], (rb + 1) >> 1, "mma K")
                        issue_s("A", rb + 1, tb + 1)
                    yield wait(p_full[t], tb, f"mma P{t}")
                    done = u if t == "A" else nb      # this tile's earlier units
                    if j == 0 and done > 0:
                        yield wait(o_free[t], done - 1, f"mma O{t} free")
                    yield wait(v_full[rb & 1], rb >> 1, "mma V")
                    pipe.append(("pv", t, tb, rb))
                    if j + 1 < n[t] and not (defect == "early_s" and t == "A"):
                        yield wait(k_full[(rb + 1) & 1], (rb + 1) >> 1, "mma K")
                        issue_s(t, rb + 1, tb + 1)
            g += nr
            for t in tiles:
                gt[t] += n[t]
            nb += nbk > 0
        pipe.append(("drain", None, None, None))
        yield wait(drain, 0, "mma drain")

    def softmax(t):
        g = 0                                        # this tile's blocks
        for u, (na, nbk) in enumerate(units):
            if t == "B" and not nbk:
                break                                # tile B's warps sit out the one-tile units
            nblk = na if t == "A" else nbk
            for j in range(nblk):
                gb = g + j
                yield wait(s_full[t][gb & 1], gb >> 1, f"softmax{t} S")
                s_readers[t] += 1
                yield None                           # S read into registers, P written over it
                if j >= 1 and rnd.random() < 0.3:   # a raise: O rescaled after the previous P V
                    yield wait(pv_done[t][(gb - 1) & 1], (gb - 1) >> 1, f"softmax{t} rescale")
                s_readers[t] -= 1
                p_full[t].arrive()
            gl = g + nblk - 1
            yield wait(pv_done[t][gl & 1], gl >> 1, f"softmax{t} output")
            o_free[t].arrive()                       # O read out of tensor memory
            g += nblk

    roles = [producer(True), producer(False), mma()] + [softmax(t) for t in "AB" for _ in range(nsoft)]
    current = [None] * len(roles)
    live = [True] * len(roles)
    for _ in range(1_000_000):
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
            op, t, gb, _ = pipe.pop(0)     # the tensor pipe completes in issue order (gb: the tile's block)
            if op == "s":
                assert s_readers[t] == 0, f"S_{t} of block {gb} overwrote a score buffer a softmax still reads"
                s_full[t][gb & 1].arrive()
            elif op == "pv":
                pv_done[t][gb & 1].arrive()
            else:
                drain.arrive()
        else:
            try:
                current[i] = next(roles[i])   # None: a step with no wait, a scheduling point
            except StopIteration:
                live[i], current[i] = False, None
    raise AssertionError("no progress bound reached")


CASES = [[1], [2], [5], [2, 2], [8, 8, 8], [32, 32], [3, 1, 4], [1, 1, 1, 1],
         [(1, False)], [(5, False)], [(3, False), (3, False)], [4, (4, False)], [8, 8, (8, False)],
         [1, (1, False)], [2, 2, (2, False), (2, False)], [32, 32, (32, False)],
         # causal units: tile A 2k + 1 blocks, tile B 2k + 2 (two pairs of one head, heavy then light)
         [(1, 2)], [(3, 4), (1, 2)], [(31, 32), (1, 2), (29, 30), (3, 4)], [(5, 6), (5, 6)], [(1, 2), (1, 2), (1, 2)]]


@pytest.mark.parametrize("units", CASES)
def test_attention2_barrier_protocol(units):
    for seed in range(8):
        run_protocol2(units, seed)


@pytest.mark.parametrize("defect", ["early_s", "k_slot_a"])
def test_attention2_model_catches_planted_defects(defect):
    with pytest.raises(AssertionError):
        for seed in range(60):
            run_protocol2([4, 4, 3], seed, defect=defect)


def test_attention2_model_catches_slot_freed_on_the_wrong_tile_at_the_switch():
    # the last two-tile unit's blocks are read last by tile B: freeing their
    # slots on tile A's barriers lets a load overwrite K or V under S_B / P_B V
    with pytest.raises(AssertionError):
        for seed in range(200):
            run_protocol2([4, 4, (3, False)], seed, defect="single_slot_a")


def test_attention2_model_catches_tile_a_phases_from_the_ring_count():
    # in causal units tile A reads one block fewer than is loaded: its barrier
    # phases must follow its own block count
    with pytest.raises(AssertionError):
        for seed in range(50):
            run_protocol2([(3, 4), (1, 2), (5, 6)], seed, defect="a_ring_phase")
