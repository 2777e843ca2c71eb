"""The attention forward's host plan (attn_f16_plan: kernel choice and work
split), checked on the CPU through the C ABI.

Pinned: the routing decisions that same-box GPU measurements settled (the
figures are in the library's comments), and invariants that hold for every
plan: the units of each mode account for every query tile exactly once, the
CTAs are min(units, SMs), and argument errors are reported as for
attn_f16_fwd.  Page: "writing-tilelang-kernels", Flash Attention Forward
(the computation the plan splits into tiles of 128 query rows).
"""
import itertools

import pytest

g = pytest.importorskip("dense_fp16_tensor_tma_gb300")

ONE, TWO128, TWO64 = 1, 2, 3


def plan(B, H, S, D, causal, sms=152):
    return g.attn_f16_plan(B, H, S, D, causal, sms)


@pytest.mark.parametrize("B,H,S,D,causal,kernel", [
    (4, 32, 4096, 128, False, TWO128),     # the bench workload
    (4, 32, 4096, 64, False, TWO64),
    (4, 32, 4096, 128, True, TWO128),      # 32 tiles per head: steps of two pairs
    (4, 32, 4096, 64, True, TWO64),
    (4, 32, 1024, 128, True, TWO128),      # 8 tiles per head (687 against 627 TFLOP/s)
    (4, 32, 1792, 128, True, ONE),         # 14 tiles: an odd pair count (827 against 935)
    (4, 32, 2048, 128, True, ONE),         # 512 steps split unevenly (1059 against 1055: a tie)
    (4, 32, 3072, 128, True, TWO128),      # 768 steps (1183 against 1149)
    (2, 32, 1500, 64, True, TWO64),        # 192 steps: two on some CTAs against three units (473 against 454)
    (4, 32, 512, 128, True, ONE),          # 4 tiles per head: below the minimum of 8
    (8, 16, 1300, 64, False, TWO64),       # odd tiles at D = 64 (703 against 575)
    (4, 16, 2100, 128, False, TWO128),     # 17 tiles at D = 128 (1225 against 1143)
    (8, 16, 1300, 128, False, TWO128),     # 11 tiles at D = 128 (988 against 986)
    (16, 16, 1300, 128, False, TWO128),    # (1014 against 999)
    (2, 3, 100, 64, False, ONE),           # one tile per head
])
def test_measured_routing(B, H, S, D, causal, kernel):
    assert plan(B, H, S, D, causal)["kernel"] == kernel


def test_units_cover_every_tile_once():
    sms = 152
    for B, H, S, D, causal in itertools.product((1, 2, 4), (1, 7, 32, 64), (1, 127, 129, 300, 1000, 1300, 2100, 4096),
                                                (64, 128), (False, True)):
        nq = (S + 127) // 128
        tiles = B * H * nq
        p = plan(B, H, S, D, causal, sms)
        units, pairs = p["units"], p["pair_units"]
        assert p["ctas"] == min(units, sms)
        if p["kernel"] == ONE:
            assert pairs == 0
            if p["causal_pairs"]:
                assert causal and units == B * H * ((nq + 1) // 2)
            else:
                assert units == tiles
        elif causal:
            # steps of two adjacent pairs of one head: a multiple of 4 tiles
            assert nq % 4 == 0 and nq >= 8 and units == pairs == B * H * nq // 4
        else:
            # pairs (2k, 2k + 1) of a head, the rest one tile each
            assert 0 <= pairs <= B * H * (nq // 2)
            assert 2 * pairs + (units - pairs) == tiles


def test_sm_count_moves_the_causal_split():
    # the same problem splits evenly over 128 SMs (1024 steps = 8 rounds), so
    # it keeps the two-tile kernel there too
    assert plan(4, 32, 4096, 128, True, 128)["kernel"] == TWO128
    # too few steps for the SMs: the one-tile kernel
    assert plan(1, 4, 4096, 128, True, 152)["kernel"] == ONE


def test_empty_and_invalid_arguments():
    assert plan(0, 4, 128, 64, False)["kernel"] == 0
    assert plan(2, 4, 0, 128, True)["units"] == 0
    for bad in [(1, 1, 128, 96, False), (-1, 1, 128, 64, False), (1, 1, 1 << 31, 64, False)]:
        with pytest.raises(g.GemmError):
            plan(*bad)
    with pytest.raises(g.GemmError):
        plan(1, 1, 128, 64, False, sms=0)
