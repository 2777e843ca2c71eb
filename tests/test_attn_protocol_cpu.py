"""A model of the attention kernel's barrier protocol, run on the CPU.

Each role of the one-tile attention kernel attn_f16_fwd4_kernel
(csrc/attn4_kernels.cuh) is written here as
the sequence of its mbarrier waits, arrivals, expect-tx arrivals, TMA loads
and tensor-core commits, in the kernel's order and with its phase-parity
arithmetic; a scheduler runs the roles, the TMA completions (any order) and
the tensor pipe (in issue order) in seeded random interleavings.  Checked:
no deadlock, no barrier receiving more arrivals than its count in one phase,
every parity wait finding its barrier at exactly the phase it means (a
barrier one phase behind or two ahead would pass or block wrongly), and no
score buffer overwritten while a softmax warp reads it: a block's scores are
read once after its S commit and, when the block's sum of P exceeds 2^8 (the
maximum then taken exactly), a second time before P is signalled; the MMA
thread issues the next S into that buffer only after the signal.  The
work lists are those the kernel walks: one tile per unit (head-major,
heaviest causal tile first) or causal pairs (tile nq-1-k, then tile k).

An mbarrier here: `count` arrivals and zero pending transaction bytes
complete a phase; `try_wait.parity(P)` succeeds when the current phase's
parity differs from P (the phase with parity P has completed).
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


def work_list(units, grid, cta, nq, causal, paired):
    """(query tile, key blocks) of CTA `cta` of `grid`, as the kernel's tile_of() walks them."""
    tiles, u = [], cta
    while u < units:
        if not paired:
            tiles.append(nq - 1 - u % nq)
        else:
            npairs = (nq + 1) // 2
            k = u % npairs
            tiles.append(nq - 1 - k)
            if k != nq - 1 - k:
                tiles.append(k)
        u += grid
    return [(qt, min(nq, qt + 1) if causal else nq) for qt in tiles]


def run_protocol(tiles, seed, nsoft=2, misnumbered_producer=False, early_s=False):
    """One CTA: producer K and V lanes, the MMA thread and `nsoft` softmax warps
    (standing for the four, which all arrive on the same barriers).
    `misnumbered_producer` plants a defect an early build had: the producer
    advanced its block count inside the block loop.  `early_s` plants another:
    the MMA thread issues S of block gb + 2 before P of block gb is signalled."""
    rnd = random.Random(seed)
    q_full, drain, o_free = Barrier("q_full", 1), Barrier("drain", 1), Barrier("o_free", nsoft)
    k_full = [Barrier(f"k_full{i}", 1) for i in range(2)]
    v_full = [Barrier(f"v_full{i}", 1) for i in range(2)]
    s_full = [Barrier(f"s_full{i}", 1) for i in range(2)]
    p_full = [Barrier(f"p_full{i}", nsoft) for i in range(2)]
    pv_done = [Barrier(f"pv_done{i}", 1) for i in range(2)]
    tma, pipe = [], []
    s_block = [None, None]       # the block whose S the MMA thread last issued into each buffer

    def wait(bar, index, who):
        # the phase the wait means and the parity the kernel passes for it
        return (bar, index & 1, who, index)

    def producer(is_k):
        g = ntile = 0
        for qt, nblk in tiles:
            if is_k:
                if g > 0:   # the previous tile's last S has read Q
                    yield wait(s_full[(g - 1) & 1], (g - 1) >> 1, "producer Q")
                q_full.arrive(tx=1)
                tma.append(q_full)
            ntile += 1
            for j in range(nblk):
                gb = g + j
                s = gb & 1
                # parity ((gb >> 1) & 1) ^ 1: the phase of block gb - 2
                yield wait(s_full[s] if is_k else pv_done[s], (gb >> 1) - 1, "producer slot")
                full = k_full[s] if is_k else v_full[s]
                full.arrive(tx=1)
                tma.append(full)
                if misnumbered_producer:
                    g = gb + 1
            if not misnumbered_producer:
                g += nblk

    def mma():
        g = ntile = 0

        def issue_s(gb):
            yield wait(k_full[gb & 1], gb >> 1, "mma K")
            s_block[gb & 1] = gb
            pipe.append(s_full[gb & 1])

        for qt, nblk in tiles:
            yield wait(q_full, ntile, "mma Q")
            yield from issue_s(g)
            if nblk > 1:
                yield from issue_s(g + 1)
            for j in range(nblk):
                gb = g + j
                s = gb & 1
                if early_s and j + 2 < nblk:
                    yield from issue_s(gb + 2)
                yield wait(p_full[s], gb >> 1, "mma P")
                if j == 0 and ntile > 0:
                    yield wait(o_free, ntile - 1, "mma O free")
                yield wait(v_full[s], gb >> 1, "mma V")
                pipe.append(pv_done[s])
                if j + 2 < nblk and not early_s:
                    yield from issue_s(gb + 2)
            g += nblk
            ntile += 1
        pipe.append(drain)
        yield wait(drain, 0, "mma drain")

    def softmax():
        g = 0
        for qt, nblk in tiles:
            for j in range(nblk):
                gb = g + j
                s = gb & 1
                yield wait(s_full[s], gb >> 1, "softmax S")
                assert s_block[s] == gb, f"score buffer {s} overwritten while block {gb} is read"
                yield None                           # S read, P computed in registers
                if j >= 1 and rnd.random() < 0.3:   # a block sum above 2^8: the scores read again
                    yield None
                    assert s_block[s] == gb, f"score buffer {s} overwritten before block {gb} is read again"
                if j >= 1 and rnd.random() < 0.3:   # a raise of the running maximum
                    yield wait(pv_done[(gb - 1) & 1], (gb - 1) >> 1, "softmax rescale")
                p_full[s].arrive()
            gl = g + nblk - 1
            yield wait(pv_done[gl & 1], gl >> 1, "softmax output")
            o_free.arrive()
            g += nblk

    roles = [producer(True), producer(False), mma()] + [softmax() for _ in range(nsoft)]
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
            pipe.pop(0).arrive()           # the tensor pipe completes in issue order
        else:
            try:
                current[i] = next(roles[i])
            except StopIteration:
                live[i], current[i] = False, None
    raise AssertionError("no progress bound reached")


CASES = []
for S, causal in [(128, False), (300, True), (700, False), (1300, True), (4096, False), (4096, True), (129, True)]:
    nq = (S + 127) // 128
    for heads in (1, 3):
        for paired in ((False, True) if causal else (False,)):
            units = heads * ((nq + 1) // 2 if paired else nq)
            for grid in sorted({1, 2, 5, units}):
                if grid <= units:
                    CASES.append((S, causal, paired, units, grid))


@pytest.mark.parametrize("S,causal,paired,units,grid", CASES)
def test_attention_barrier_protocol(S, causal, paired, units, grid):
    nq = (S + 127) // 128
    for cta in range(min(grid, 2)):
        tiles = work_list(units, grid, cta, nq, causal, paired)
        for seed in range(6):
            run_protocol(tiles, seed)


def test_protocol_model_catches_a_misnumbered_producer():
    # the defect of an early persistent build (block numbers advanced inside the
    # producer's block loop, so its loads went to the wrong slots and phases):
    # the model must reject it
    tiles = work_list(2, 1, 0, 3, False, False)
    with pytest.raises(AssertionError):
        run_protocol(tiles, 0, misnumbered_producer=True)


def test_protocol_model_catches_an_early_score_issue():
    # S of block gb + 2 issued into the buffer of block gb before that block's
    # P is signalled would overwrite scores the softmax may still be reading
    tiles = work_list(1, 1, 0, 4, False, False)
    with pytest.raises(AssertionError):
        for seed in range(20):
            run_protocol(tiles, seed, early_s=True)

