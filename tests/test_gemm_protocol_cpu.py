"""A model of the CTA-pair GEMM kernel's barrier protocol, run on the CPU.

gemm_f16_tc2_kernel and the grouped kernel (csrc/gemm_kernels_pair.cuh) run a
pair of CTAs on one 256 x 256 tile: each CTA's producer waits for its own
`empty[s]` and loads its half of the operands, completing CTA 0's `full[s]`
(CTA 0's producer posts the expected bytes of both); CTA 0's MMA thread waits
for `full[s]` and a free accumulator `acc_empty[b]`, and its commits are
multicast to both CTAs' `empty[s]` and `acc_full[b]`; the epilogue warps of
both CTAs wait for their own `acc_full[b]` and arrive on CTA 0's
`acc_empty[b]`.  At the end CTA 0's producer waits for the last stages' bytes
and the MMA thread for a drain commit.  Here every role is the sequence of
those waits and arrivals, with the kernel's stage / phase / accumulator
arithmetic, run with the tensor pipe completing in issue order and the TMA
loads in any order (the peer's bytes may land before CTA 0 posts the count).
Checked under seeded random interleavings: no deadlock, no barrier receiving
more arrivals than its count in one phase, and every parity wait finding its
barrier at exactly the phase it means.
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


def run_pair(units, stages, seed, epi_warps=2, defect=None):
    """units: the K blocks of each unit the pair walks (whole tiles and half tiles
    alike: each unit is one accumulator's worth); epi_warps per CTA.  `defect`
    plants a mistake: "producer_parity" (a producer waits for the current use of
    its stage instead of the previous one) or "no_acc_wait" (the MMA thread does
    not wait for a free accumulator)."""
    rnd = random.Random(seed)
    full = [Barrier(f"full{s}", 1) for s in range(stages)]                      # CTA 0
    empty = [[Barrier(f"empty{s}@cta{c}", 1) for s in range(stages)] for c in range(2)]
    acc_full = [[Barrier(f"acc_full{b}@cta{c}", 1) for b in range(2)] for c in range(2)]
    acc_empty = [Barrier(f"acc_empty{b}", 2 * epi_warps) for b in range(2)]      # CTA 0
    drain = Barrier("drain", 1)
    tma, pipe = [], []

    def wait(bar, index, who):
        return (bar, index & 1, who, index)

    def producer(cta):
        stage = phase = issued = 0
        count = [0] * stages          # loads issued per stage: the phase of the next one
        for kblocks in units:
            for _ in range(kblocks):
                # parity phase ^ 1: the phase of the stage's previous use (none at first)
                late = 1 if defect == "producer_parity" else 0
                yield wait(empty[cta][stage], count[stage] - 1 + late, f"producer {cta}")
                if cta == 0:
                    full[stage].arrive(tx=2)                  # both CTAs' bytes
                tma.append(full[stage])
                count[stage] += 1
                issued += 1
                stage += 1
                if stage == stages:
                    stage, phase = 0, phase ^ 1
        if cta == 0:                  # CTA 0's full barriers count both CTAs' bytes
            for _ in range(min(issued, stages)):
                stage -= 1
                if stage < 0:
                    stage, phase = stages - 1, phase ^ 1
                yield wait(full[stage], count[stage] - 1, "producer drain")

    def mma():
        stage = acc = 0
        count = [0] * stages
        acc_count = [0, 0]
        for kblocks in units:
            if defect != "no_acc_wait":
                yield wait(acc_empty[acc], acc_count[acc] - 1, "mma acc_empty")
            for _ in range(kblocks):
                yield wait(full[stage], count[stage], "mma full")
                count[stage] += 1
                pipe.append(("mma", None))
                pipe.append(("commit", [empty[0][stage], empty[1][stage]]))
                stage = (stage + 1) % stages
            pipe.append(("commit", [acc_full[0][acc], acc_full[1][acc]]))
            acc_count[acc] += 1
            acc ^= 1
        pipe.append(("commit", [drain]))
        yield wait(drain, 0, "mma drain")

    def epilogue(cta):
        acc = 0
        acc_count = [0, 0]
        for _ in units:
            yield wait(acc_full[cta][acc], acc_count[acc], f"epilogue {cta}")
            acc_empty[acc].arrive()
            acc_count[acc] += 1
            acc ^= 1

    roles = [producer(0), producer(1), mma()] + [epilogue(c) for c in (0, 1) for _ in range(epi_warps)]
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
            tma.pop(rnd.randrange(len(tma))).complete_tx(1)   # one CTA's bytes of a stage
        elif kind == "pipe":
            op, bars = pipe.pop(0)                             # completes in issue order
            if op == "commit":
                for bar in bars:
                    bar.arrive()
        else:
            try:
                current[i] = next(roles[i])
            except StopIteration:
                live[i], current[i] = False, None
    raise AssertionError("no progress bound reached")


def pair_units(tiles_m, tiles_n, pairs, pair, kblocks, tail_split):
    """The units of one pair as PairUnitIter walks them: whole tiles pair, pair +
    pairs, ... below the whole-tile count, then half tiles of the rest."""
    tiles = tiles_m * tiles_n
    rest = tiles % pairs if tail_split else 0
    whole = tiles - rest
    units = [kblocks for _ in range(pair, whole, pairs)]
    units += [kblocks for _ in range(pair, 2 * rest, pairs)]
    return units


@pytest.mark.parametrize("stages", [2, 3, 4])
@pytest.mark.parametrize("tiles_m,tiles_n,pairs,kblocks,tail", [
    (1, 1, 1, 1, False), (1, 1, 1, 5, False), (2, 3, 2, 3, True), (4, 4, 3, 2, True), (3, 5, 4, 7, True),
    (32, 32, 76, 64, True), (12, 20, 76, 8, True), (1, 2, 76, 1, True)])
def test_gemm_pair_barrier_protocol(stages, tiles_m, tiles_n, pairs, kblocks, tail):
    for pair in sorted({0, pairs // 2, pairs - 1}):
        units = pair_units(tiles_m, tiles_n, pairs, pair, kblocks, tail)
        if not units:
            continue
        if sum(units) > 400:           # a long list: its first units exercise the same steady state
            units = units[:max(1, 400 // kblocks)]
        for seed in range(4):
            run_pair(units, stages, seed)


@pytest.mark.parametrize("defect", ["producer_parity", "no_acc_wait"])
def test_gemm_protocol_model_catches_planted_defects(defect):
    units = pair_units(4, 4, 1, 0, 1, False)     # 16 one-block units: the MMA thread can run ahead
    with pytest.raises(AssertionError):
        for seed in range(40):
            run_pair(units, 3, seed, defect=defect)


# ---------------------------------------------------------------- a stage's loads never arrive

def run_pair_lost_load(units, stages, seed, lost_cta, lost_pos, epi_warps=2, defect=None):
    """The protocol of run_pair with its abort paths: one CTA's producer never
    issues the loads of position `lost_pos` (the leader then posts no expected
    bytes for it either), so that stage's `full` phase never completes.  Every
    wait is bounded: a wait may run out only when nothing else can move (a
    load or a tensor-core operation still in flight always lands first), and
    then sets its CTA's abort flag (the final drains have no abort flag and
    only give up); a wait in a CTA whose flag is up may give up at any time.
    Each role then takes the kernel's exit path.  Checked: every role ends,
    no load is in flight and the tensor pipe is empty when the CTAs exit (the
    shared memory the loads write and the tensor memory the MMAs write are
    released only then), no barrier over-arrives, and a timeout was reported.
    `defect` = "no_mma_drain" plants a mistake: the MMA thread leaves without
    waiting for its drain commit."""
    rnd = random.Random(seed)
    full = [Barrier(f"full{s}", 1) for s in range(stages)]
    empty = [[Barrier(f"empty{s}@cta{c}", 1) for s in range(stages)] for c in range(2)]
    acc_full = [[Barrier(f"acc_full{b}@cta{c}", 1) for b in range(2)] for c in range(2)]
    acc_empty = [Barrier(f"acc_empty{b}", 2 * epi_warps) for b in range(2)]
    drain = Barrier("drain", 1)
    tma, pipe = [], []
    abort = [False, False]
    status = []

    def wait(bar, index, who, cta, honours_abort=True):
        return (bar, index & 1, who, index, cta, honours_abort)

    def producer(cta):
        stage = issued = 0
        count = [0] * stages
        ok = True
        pos = 0
        for kblocks in units:
            for _ in range(kblocks):
                ok = yield wait(empty[cta][stage], count[stage] - 1, f"producer {cta}", cta)
                if not ok:
                    break
                if not (cta == lost_cta and pos == lost_pos):
                    if cta == 0:
                        full[stage].arrive(tx=2)
                    tma.append(full[stage])
                count[stage] += 1
                issued += 1
                pos += 1
                stage = (stage + 1) % stages
            if not ok:
                break
        if cta == 0:
            for _ in range(min(issued, stages)):
                stage = (stage - 1) % stages
                yield wait(full[stage], count[stage] - 1, "producer drain", cta, honours_abort=False)

    def mma():
        stage = acc = 0
        count = [0] * stages
        acc_count = [0, 0]
        ok = True
        for kblocks in units:
            ok = yield wait(acc_empty[acc], acc_count[acc] - 1, "mma acc_empty", 0)
            if not ok:
                break
            for _ in range(kblocks):
                ok = yield wait(full[stage], count[stage], "mma full", 0)
                if not ok:
                    break
                count[stage] += 1
                pipe.append(("mma", None))
                pipe.append(("commit", [empty[0][stage], empty[1][stage]]))
                stage = (stage + 1) % stages
            if not ok:
                break
            pipe.append(("commit", [acc_full[0][acc], acc_full[1][acc]]))
            acc_count[acc] += 1
            acc ^= 1
        pipe.append(("commit", [drain]))
        if defect != "no_mma_drain":
            yield wait(drain, 0, "mma drain", 0, honours_abort=False)

    def epilogue(cta):
        acc = 0
        acc_count = [0, 0]
        for _ in units:
            ok = yield wait(acc_full[cta][acc], acc_count[acc], f"epilogue {cta}", cta)
            if not ok:
                break
            acc_empty[acc].arrive()
            acc_count[acc] += 1
            acc ^= 1

    roles = [producer(0), producer(1), mma()] + [epilogue(c) for c in (0, 1) for _ in range(epi_warps)]
    current = [None] * len(roles)
    live = [True] * len(roles)

    def resume(i, value):
        try:
            current[i] = roles[i].send(value) if current[i] is not None else next(roles[i])
        except StopIteration:
            live[i], current[i] = False, None

    for _ in range(2_000_000):
        if not any(live):                               # the CTAs exit here
            break
        ready, stuck = [], []
        for i in range(len(roles)):
            if not live[i]:
                continue
            if current[i] is None:
                ready.append(("role", i))
                continue
            bar, parity, who, index, cta, honours = current[i]
            assert bar.n <= index + 1, f"{who}: {bar.name} is {bar.n - index - 1} phase(s) past the awaited one"
            if bar.passes(parity):
                assert bar.n == index + 1, f"{who}: {bar.name} passes {index + 1 - bar.n} phase(s) early"
                ready.append(("role", i))
            else:
                stuck.append(i)
                if honours and abort[cta]:
                    ready.append(("give_up", i))
        if tma:
            ready.append(("tma", None))
        if pipe:
            ready.append(("pipe", None))
        if not ready:
            i = rnd.choice(stuck)                       # nothing can move: one wait runs out
            bar, parity, who, index, cta, honours = current[i]
            status.append(who)
            if honours:
                abort[cta] = True
            resume(i, False)
            continue
        kind, i = rnd.choice(ready)
        if kind == "tma":
            tma.pop(rnd.randrange(len(tma))).complete_tx(1)
        elif kind == "pipe":
            op, bars = pipe.pop(0)
            if op == "commit":
                for bar in bars:
                    bar.arrive()
        elif kind == "give_up":
            resume(i, False)
        else:
            resume(i, True)
    else:
        raise AssertionError("no progress bound reached")
    assert not any(live), "a role never ended"
    assert not tma, "a load still in flight when the CTAs exit"
    assert not pipe, "tensor-core work still in flight when tensor memory is freed"
    assert status, "the lost load went unnoticed"


@pytest.mark.parametrize("stages", [2, 3])
@pytest.mark.parametrize("lost_cta", [0, 1])
@pytest.mark.parametrize("units,lost_pos", [([1], 0), ([4], 1), ([3, 3, 2], 4), ([2] * 6, 9), ([5, 5], 9)])
def test_gemm_pair_lost_load_ends_cleanly(stages, lost_cta, units, lost_pos):
    for seed in range(12):
        run_pair_lost_load(units, stages, seed, lost_cta, lost_pos)


def test_lost_load_model_catches_a_missing_drain():
    with pytest.raises(AssertionError, match="tensor-core work still in flight"):
        for seed in range(40):
            run_pair_lost_load([2] * 6, 3, seed, 1, 9, defect="no_mma_drain")
