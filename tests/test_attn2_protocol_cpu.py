"""A model of the two-tile attention kernel's barrier protocol, run on the CPU.

attn_f16_fwd2_kernel (csrc/attn2_kernels.cuh) gives each CTA units of two
query tiles (A and B) of one head that share the K and V rings.  Each tile
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
MMAs in issue order, which the model assumes as the kernel does.
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
    """`units`: key blocks of each unit this CTA walks.  nsoft softmax warps per
    tile stand for the eight.  `defect` plants a mistake: "early_s" (the MMA
    thread issues the next S of a tile before that tile's P is written) or
    "k_slot_a" (the producer frees a K slot on tile A's S instead of B's)."""
    rnd = random.Random(seed)
    q_full, drain = Barrier("q_full", 1), Barrier("drain", 1)
    k_full = [Barrier(f"k_full{i}", 1) for i in range(2)]
    v_full = [Barrier(f"v_full{i}", 1) for i in range(2)]
    s_full = {"A": [Barrier(f"s_fullA{i}", 1) for i in range(2)], "B": [Barrier(f"s_fullB{i}", 1) for i in range(2)]}
    p_full = {t: Barrier(f"p_full{t}", nsoft) for t in "AB"}
    pv_done = {"A": [Barrier(f"pv_doneA{i}", 1) for i in range(2)], "B": [Barrier(f"pv_doneB{i}", 1) for i in range(2)]}
    o_free = {t: Barrier(f"o_free{t}", nsoft) for t in "AB"}
    xch = {t: [Barrier(f"xch{t}{i}", nsoft) for i in range(2)] for t in "AB"}
    tma, pipe = [], []
    # tensor-memory hazard: softmax warps that may still read each tile's score buffer
    s_readers = {"A": 0, "B": 0}

    def wait(bar, index, who):
        return (bar, index & 1, who, index)

    def producer(is_k):
        g = 0
        for u, nblk in enumerate(units):
            if is_k:
                if g > 0:   # the previous unit's last S (S_B, issued after S_A) has read both Q tiles
                    yield wait(s_full["B"][(g - 1) & 1], (g - 1) >> 1, "producer Q")
                q_full.arrive(tx=2)
                tma.append(q_full)
                tma.append(q_full)
            for j in range(nblk):
                gb = g + j
                s = gb & 1
                # the slot's previous block gb - 2 is done: both S (K) or both P V (V);
                # tile B's are issued after tile A's, so B's commits cover both
                t = "A" if (is_k and defect == "k_slot_a") else "B"
                yield wait(s_full[t][s] if is_k else pv_done["B"][s], (gb >> 1) - 1, "producer slot")
                # the load overwrites ring slot s: no MMA reading its previous block may remain
                for op, _, gq in pipe:
                    assert not (gq is not None and gq & 1 == s and gq < gb and op == ("s" if is_k else "pv")), \
                        f"load of block {gb} into {'K' if is_k else 'V'} slot {s} while block {gq}'s MMA reads it"
                full = k_full[s] if is_k else v_full[s]
                full.arrive(tx=1)
                tma.append(full)
            g += nblk

    def mma():
        g = 0

        def issue_s(t, gb):
            # S overwrites tile t's score buffer: no softmax may still read it and
            # no earlier P V may still read the P in it (the pipe is in order)
            pipe.append(("s", t, gb))

        for u, nblk in enumerate(units):
            yield wait(q_full, u, "mma Q")
            yield wait(k_full[g & 1], g >> 1, "mma K")
            issue_s("A", g)
            issue_s("B", g)
            for j in range(nblk):
                gb = g + j
                for t in "AB":
                    if defect == "early_s" and t == "A" and j + 1 < nblk:
                        yield wait(k_full[(gb + 1) & 1], (gb + 1) >> 1, "mma K")
                        issue_s("A", gb + 1)
                    yield wait(p_full[t], gb, f"mma P{t}")
                    if j == 0 and u > 0:
                        yield wait(o_free[t], u - 1, f"mma O{t} free")
                    yield wait(v_full[gb & 1], gb >> 1, "mma V")
                    pipe.append(("pv", t, gb))
                    if j + 1 < nblk and not (defect == "early_s" and t == "A"):
                        yield wait(k_full[(gb + 1) & 1], (gb + 1) >> 1, "mma K")
                        issue_s(t, gb + 1)
            g += nblk
        pipe.append(("drain", None, None))
        yield wait(drain, 0, "mma drain")

    def softmax(t):
        g = x = 0
        for u, nblk in enumerate(units):
            for j in range(nblk):
                gb = g + j
                yield wait(s_full[t][gb & 1], gb >> 1, f"softmax{t} S")
                s_readers[t] += 1
                slot, use = x & 1, x >> 1
                x += 1
                xch[t][slot].arrive()
                yield wait(xch[t][slot], use, f"softmax{t} exchange")
                if j >= 1 and rnd.random() < 0.3:   # a raise: O rescaled after the previous P V
                    yield wait(pv_done[t][(gb - 1) & 1], (gb - 1) >> 1, f"softmax{t} rescale")
                yield None                           # pass 2 reads S again and writes P into it
                s_readers[t] -= 1
                p_full[t].arrive()
            gl = g + nblk - 1
            yield wait(pv_done[t][gl & 1], gl >> 1, f"softmax{t} output")
            slot, use = x & 1, x >> 1
            x += 1
            xch[t][slot].arrive()
            yield wait(xch[t][slot], use, f"softmax{t} row sum")
            o_free[t].arrive()
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
            op, t, gb = pipe.pop(0)        # the tensor pipe completes in issue order
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


CASES = [[1], [2], [5], [2, 2], [8, 8, 8], [32, 32], [3, 1, 4], [1, 1, 1, 1]]


@pytest.mark.parametrize("units", CASES)
def test_attention2_barrier_protocol(units):
    for seed in range(8):
        run_protocol2(units, seed)


@pytest.mark.parametrize("defect", ["early_s", "k_slot_a"])
def test_attention2_model_catches_planted_defects(defect):
    with pytest.raises(AssertionError):
        for seed in range(60):
            run_protocol2([4, 4, 3], seed, defect=defect)
