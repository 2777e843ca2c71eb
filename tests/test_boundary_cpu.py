"""Host-only tests of the C-ABI library: it loads, exports every declared
symbol, rejects bad arguments before touching a device, and plans as designed."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def g():
    import __graft_entry__
    __graft_entry__.build()
    import dense_fp16_tensor_tma_gb300 as mod
    return mod


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(gemm_f16\w*)\s*\(", text))
    return names


def test_exports_every_declared_symbol(g):
    declared = _declared_functions()
    assert {"gemm_f16", "gemm_f16_status_string", "gemm_f16_debug_status"} <= declared
    lib = ctypes.CDLL(g.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert set(g.EXPORTS) == declared


def test_status_strings(g):
    assert g.gemm_f16_status_string(0) == "ok"
    for s in range(1, 7):
        assert g.gemm_f16_status_string(s) not in ("ok", "unknown status")
    assert g.gemm_f16_status_string(99) == "unknown status"


GOOD = 0x10000  # a 16-byte aligned fake device address: never dereferenced on the error paths


@pytest.mark.parametrize("args, expect", [
    ((GOOD, GOOD, GOOD, GOOD, -1, 8, 8, 0), 1),          # negative M
    ((GOOD, GOOD, GOOD, GOOD, 8, -2, 8, 0), 1),          # negative N
    ((GOOD, GOOD, GOOD, GOOD, 8, 8, -3, 0), 1),          # negative K
    ((GOOD, GOOD, GOOD, GOOD, 8, 8, 8, 6), 1),           # unknown epilogue
    ((GOOD, GOOD, GOOD, GOOD, 8, 8, 8, -1), 1),
    ((GOOD, GOOD, GOOD, 0, 8, 8, 8, 0), 1),              # C null
    ((0, GOOD, GOOD, GOOD, 8, 8, 8, 0), 1),              # A null with K > 0
    ((GOOD, 0, GOOD, GOOD, 8, 8, 8, 0), 1),              # B null
    ((GOOD, GOOD, 0, GOOD, 8, 8, 8, 3), 1),              # bias null with GELU
    ((GOOD, GOOD, 0, GOOD, 8, 8, 8, 1), 1),              # bias null with bias
    ((GOOD, GOOD, GOOD, GOOD, 1 << 31, 8, 8, 0), 1),     # M too large
    ((GOOD + 1, GOOD, GOOD, GOOD, 8, 8, 8, 0), 3),       # A odd address
    ((GOOD, GOOD, GOOD, GOOD + 1, 8, 8, 8, 0), 3),       # C odd address
    ((GOOD, GOOD, GOOD + 1, GOOD, 8, 8, 8, 2), 3),       # bias odd address
    ((GOOD, GOOD, GOOD, GOOD, 0, 8, 8, 3), 0),           # M == 0: no-op
    ((GOOD, GOOD, GOOD, GOOD, 8, 0, 8, 3), 0),           # N == 0: no-op
    ((0, 0, 0, 0, 0, 0, 0, 0), 0),                       # everything empty
])
def test_argument_errors_need_no_device(g, args, expect):
    a, b, bias, c, M, N, K, epi = args
    assert g.gemm_f16_ptr(a, b, bias, c, M, N, K, epi, 0) == expect


def test_plan_large_square_uses_cta_pairs(g):
    p = g.gemm_f16_plan(8192, 8192, 8192, "bias_gelu_erf", num_sms=152)
    # 1024 tiles on 76 pairs: 988 whole tiles, then the last 36 as 72 half tiles
    assert p == {"path": 2, "tile_m": 256, "tile_n": 256, "stages": 3, "ctas": 152,
                 "pack_a": 0, "pack_b": 0, "vec_store": 1, "splits": 1, "scratch": 0, "whole_tiles": 988}
    # an exact number of waves needs no half tiles
    assert g.gemm_f16_plan(8192, 9728, 8192, "none", num_sms=152)["whole_tiles"] == -1
    p = g.gemm_f16_plan(4096, 4096, 4096, "bias_gelu_erf", num_sms=152)
    assert p["tile_m"] == 256 and p["ctas"] == 152


def test_plan_mid_size_uses_single_cta_tiles(g):
    # 18 pair tiles < 76 pairs: single-CTA 128-row tiles give more CTAs
    p = g.gemm_f16_plan(1536, 768, 4096, "none", num_sms=152)
    assert p["tile_m"] == 128 and p["tile_n"] == 64 and p["ctas"] == 144


def test_force_config_overrides_and_restores(g):
    prev = g.gemm_f16_force_config("128x256")
    try:
        p = g.gemm_f16_plan(8192, 8192, 8192, "none", num_sms=152)
        assert (p["tile_m"], p["tile_n"], p["stages"]) == (128, 256, 4)
        g.gemm_f16_force_config("pair256x256")
        p = g.gemm_f16_plan(200, 300, 64, "none", num_sms=152)
        # 2 tiles, far fewer than pairs: run as 4 half tiles on 4 pairs
        assert (p["tile_m"], p["tile_n"], p["ctas"], p["whole_tiles"]) == (256, 256, 8, 0)
    finally:
        g.gemm_f16_force_config(prev)
    with pytest.raises(ValueError):
        g.gemm_f16_force_config(9)
    assert g.gemm_f16_plan(8192, 8192, 8192, "none", num_sms=152)["tile_m"] == 256


def test_plan_small_problem_uses_narrow_tiles(g):
    p = g.gemm_f16_plan(1024, 1024, 1024, "none", num_sms=152)
    assert p["tile_n"] == 64 and p["ctas"] == 128
    p = g.gemm_f16_plan(256, 256, 256, "none", num_sms=152)
    assert p["tile_n"] == 64 and p["ctas"] == 8


def test_plan_ragged_n_repacks_b_and_stores_narrow(g):
    p = g.gemm_f16_plan(3001, 5003, 1000, "bias_relu", num_sms=152)
    assert p["pack_b"] == 1 and p["pack_a"] == 0 and p["vec_store"] == 0 and p["path"] == 2
    assert p["tile_m"] == 256 and p["ctas"] == 152      # 12 x 20 pair tiles


def test_plan_unaligned_pointers_repack(g):
    p = g.gemm_f16_plan(64, 64, 64, "none", num_sms=152, a_addr=GOOD + 2, b_addr=GOOD + 8, c_addr=GOOD + 2)
    assert p["pack_a"] == 1 and p["pack_b"] == 1 and p["vec_store"] == 0
    p = g.gemm_f16_plan(64, 64, 60, "none", num_sms=152)
    assert p["pack_a"] == 1 and p["pack_b"] == 0


def test_plan_k_zero_is_bias_only(g):
    assert g.gemm_f16_plan(16, 16, 0, "bias", num_sms=152)["path"] == 1
    assert g.gemm_f16_plan(0, 16, 16, "none", num_sms=152)["path"] == 0


def test_python_binding_rejects_bad_tensors(g):
    torch = pytest.importorskip("torch")
    A = torch.zeros(4, 8, dtype=torch.float16)
    B = torch.zeros(8, 4, dtype=torch.float16)
    C = torch.zeros(4, 4, dtype=torch.float16)
    with pytest.raises(ValueError):
        g.gemm_f16(A, B, None, C)            # CPU tensors
    with pytest.raises(ValueError):
        g.gemm_f16(A, B, None, torch.zeros(4, 5, dtype=torch.float16))


def test_plan_short_a_uses_swap_ab(g):
    p = g.gemm_f16_plan(16, 8192, 8192, "none", num_sms=152)
    # 64 tiles of 128 columns, K split in two: 128 CTAs stream B
    assert (p["path"], p["tile_m"], p["tile_n"], p["splits"], p["ctas"]) == (3, 16, 128, 2, 128)
    assert p["scratch"] == 64 * 2 * 16 * 128 * 4 + 1024
    p = g.gemm_f16_plan(16, 16384, 8192, "none", num_sms=152)
    assert (p["splits"], p["ctas"], p["scratch"]) == (1, 128, 0)
    assert g.gemm_f16_plan(33, 1000, 64, "none", num_sms=152)["tile_m"] == 64
    assert g.gemm_f16_plan(65, 1000, 64, "none", num_sms=152)["path"] == 2
