"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Bar: relative Frobenius error <= 1e-3 and |err| <= 1e-2 (1 + |ref|) per
element (oracle/compare.py); bit-exact where every step is exact (small
integer operands).  Inputs come from workloads.py (seeded, shared by both
sides).
"""
import numpy as np
import pytest

import workloads
from oracle.compare import parity

pytestmark = pytest.mark.gpu

EPIS = ("none", "bias", "bias_relu", "bias_gelu_erf", "bias_sigmoid", "bias_gelu_tanh")


@pytest.fixture(scope="module")
def torch_dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch, torch.device("cuda:0")


@pytest.fixture(scope="module")
def g(torch_dev):
    import dense_fp16_tensor_tma_gb300 as mod
    return mod


def _dev(torch, x, dev):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(dev)


def run(g, torch_dev, A, B, bias, epi, check_status=True):
    torch, dev = torch_dev
    M, K = A.shape
    N = B.shape[1]
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    g.gemm_f16(_dev(torch, A, dev), _dev(torch, B, dev), _dev(torch, bias, dev) if epi != "none" else None, C, epi)
    if check_status:
        st, word = g.gemm_f16_debug_status()
        assert st == 0, f"device status {st} word {word:#x}"
    return C.cpu().numpy()


def rand16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def assert_parity(got, ref, what=""):
    res = parity(got, ref)
    assert res["ok"], f"{what}: {res}"
    return res


# ---------------------------------------------------------------- exact (integer) cases first

@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (128, 64, 64), (256, 512, 128), (200, 300, 136), (129, 257, 65)])
@pytest.mark.parametrize("epi", ["none", "bias", "bias_relu"])
def test_integer_inputs_bit_exact(g, torch_dev, oracle_mod, M, N, K, epi):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A = rng.integers(-2, 3, (M, K)).astype(np.float16)
    B = rng.integers(-2, 3, (K, N)).astype(np.float16)
    bias = rng.integers(-8, 9, N).astype(np.float16)
    got = run(g, torch_dev, A, B, bias, epi)
    ref = oracle_mod.gemm(A, B, bias, epi)
    assert np.array_equal(got, ref), f"max diff {np.nanmax(np.abs(got.astype(np.float64) - ref.astype(np.float64)))}"


def test_identity_and_permutation_B(g, torch_dev, oracle_mod):
    rng = np.random.default_rng(12)
    K = 320
    A = rand16(rng, (300, K))
    eye = np.eye(K, dtype=np.float16)
    assert np.array_equal(run(g, torch_dev, A, eye, None, "none").view(np.uint16), A.view(np.uint16))
    perm = rng.permutation(K)
    P = np.zeros((K, K), np.float16)
    P[perm, np.arange(K)] = 1.0
    assert np.array_equal(run(g, torch_dev, A, P, None, "none").view(np.uint16), A[:, perm].view(np.uint16))


# ---------------------------------------------------------------- the five workloads

def _check_full(g, torch_dev, oracle_mod, w, epi):
    A, B, bias = w.make()
    got = run(g, torch_dev, A, B, bias, epi)
    ref = oracle_mod.gemm(A, B, bias if epi != "none" else None, epi)
    return assert_parity(got, ref, f"{w.name} {epi}")


@pytest.mark.parametrize("epi", ["none", "bias_gelu_erf"])
def test_workload_gemm256(g, torch_dev, oracle_mod, epi):
    _check_full(g, torch_dev, oracle_mod, workloads.WORKLOADS["gemm256"], epi)


def test_workload_gemm1024(g, torch_dev, oracle_mod):
    _check_full(g, torch_dev, oracle_mod, workloads.WORKLOADS["gemm1024"], "none")


def test_workload_ragged_3001x5003x1000(g, torch_dev, oracle_mod):
    _check_full(g, torch_dev, oracle_mod, workloads.WORKLOADS["ragged3001x5003x1000"], "bias_relu")


def test_workload_skinny_16x8192x8192(g, torch_dev, oracle_mod):
    _check_full(g, torch_dev, oracle_mod, workloads.WORKLOADS["skinny16x8192x8192"], "none")


def _check_sampled(g, torch_dev, oracle_mod, w, epi, n_rows_extra=0):
    A, B, bias = w.make()
    got = run(g, torch_dev, A, B, bias, epi)
    b = bias if epi != "none" else None
    rows = [0, w.M - 1] + list(workloads.sample_coords(w.seed + 1000, w.M, 1, n_rows_extra)[0])
    ref_rows = oracle_mod.gemm_rows(A, B, b, epi, rows)
    assert_parity(got[rows], ref_rows, f"{w.name} rows")
    ii, jj = workloads.sample_coords(w.seed, w.M, w.N, workloads.SAMPLED_ELEMS)
    ref_el = oracle_mod.gemm_elems(A, B, b, epi, ii, jj)
    assert_parity(got[ii, jj], ref_el, f"{w.name} elems")
    assert np.all(np.isfinite(got))


def test_workload_fused4096(g, torch_dev, oracle_mod):
    _check_sampled(g, torch_dev, oracle_mod, workloads.WORKLOADS["fused4096"], "bias_gelu_erf", n_rows_extra=62)


def test_workload_fused8192(g, torch_dev, oracle_mod):
    _check_sampled(g, torch_dev, oracle_mod, workloads.WORKLOADS["fused8192"], "bias_gelu_erf")


# ---------------------------------------------------------------- tails, epilogues, paths

SHAPES = [(1, 1, 1), (1, 15, 8), (15, 16, 16), (16, 17, 63), (17, 127, 64), (127, 128, 65),
          (128, 129, 1000), (129, 255, 16), (255, 257, 8), (257, 1, 63), (64, 1000, 200),
          (300, 520, 77), (513, 384, 128), (33, 4097, 24)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_shape_sweep(g, torch_dev, oracle_mod, M, N, K):
    rng = np.random.default_rng(M * 1009 + N * 17 + K)
    A, B, bias = rand16(rng, (M, K), 0.5), rand16(rng, (K, N), 0.5), rand16(rng, N)
    epi = EPIS[(M + N + K) % len(EPIS)]
    got = run(g, torch_dev, A, B, bias, epi)
    assert_parity(got, oracle_mod.gemm(A, B, bias if epi != "none" else None, epi), f"{M}x{N}x{K} {epi}")


@pytest.mark.parametrize("epi", EPIS)
def test_each_epilogue_multi_tile(g, torch_dev, oracle_mod, epi):
    rng = np.random.default_rng(99)
    M, N, K = 384, 768, 320
    A, B, bias = rand16(rng, (M, K), 0.3), rand16(rng, (K, N), 0.3), rand16(rng, N)
    got = run(g, torch_dev, A, B, bias, epi)
    assert_parity(got, oracle_mod.gemm(A, B, bias if epi != "none" else None, epi), epi)


def test_large_tiles_persistent_many_waves(g, torch_dev, oracle_mod):
    # > 2 tiles per CTA on the 128x256 configuration, every tile checked on sampled rows
    rng = np.random.default_rng(5)
    M, N, K = 2048, 4096, 256
    A, B, bias = rand16(rng, (M, K), 0.2), rand16(rng, (K, N), 0.2), rand16(rng, N)
    got = run(g, torch_dev, A, B, bias, "bias_gelu_erf")
    rows = np.arange(0, M, 37)
    assert_parity(got[rows], oracle_mod.gemm_rows(A, B, bias, "bias_gelu_erf", rows), "rows")


def test_unaligned_pointers_use_repack_and_narrow_stores(g, torch_dev, oracle_mod):
    torch, dev = torch_dev
    rng = np.random.default_rng(6)
    M, N, K = 200, 136, 96
    A, B, bias = rand16(rng, (M, K)), rand16(rng, (K, N)), rand16(rng, N)
    # offset every operand by one element inside a larger buffer: 2-byte but not 16-byte aligned
    def offset(x):
        buf = torch.zeros(x.size + 8, dtype=torch.float16, device=dev)
        buf[1:1 + x.size] = torch.from_numpy(x.ravel()).to(dev)
        return buf, buf[1:1 + x.size]
    _, a1 = offset(A)
    _, b1 = offset(B)
    _, bias1 = offset(bias)
    cbuf = torch.full((M * N + 8,), -7.0, dtype=torch.float16, device=dev)
    c1 = cbuf[1:1 + M * N]
    assert g.gemm_f16_ptr(a1.data_ptr(), b1.data_ptr(), bias1.data_ptr(), c1.data_ptr(), M, N, K,
                          "bias_gelu_erf", torch.cuda.current_stream().cuda_stream) == 0
    got = c1.view(M, N).cpu().numpy()
    assert_parity(got, oracle_mod.gemm(A, B, bias, "bias_gelu_erf"))
    c = cbuf.cpu().numpy()
    assert c[0] == -7.0 and np.all(c[1 + M * N:] == -7.0)


@pytest.mark.parametrize("shift", [1, 2, 3, 4, 5, 6, 7])
def test_repack_every_base_offset_integer_exact(g, torch_dev, oracle_mod, shift):
    # A and B start `shift` elements (2 * shift bytes) past a 16-byte boundary and
    # have odd row pitches (lda = K, ldb = N with K, N odd): the repack must cut
    # every 8-element piece out of its two aligned 16-byte chunks correctly, at
    # every byte offset, and copy each row's short last piece.  Small integers:
    # every step is exact, so the result must equal the oracle's bit for bit.
    torch, dev = torch_dev
    rng = np.random.default_rng(40 + shift)
    M, N, K = 136, 203, 77
    A = rng.integers(-2, 3, (M, K)).astype(np.float16)
    B = rng.integers(-2, 3, (K, N)).astype(np.float16)
    bias = rng.integers(-4, 5, N).astype(np.float16)
    def at_offset(x):
        buf = torch.zeros(x.size + 16, dtype=torch.float16, device=dev)
        buf[shift:shift + x.size] = torch.from_numpy(x.ravel()).to(dev)
        return buf, buf[shift:shift + x.size]
    bufa, a1 = at_offset(A)
    bufb, b1 = at_offset(B)
    plan = g.gemm_f16_plan(M, N, K, "bias", a_addr=a1.data_ptr(), b_addr=b1.data_ptr())
    assert plan["pack_a"] == 1 and plan["pack_b"] == 1
    tb = torch.from_numpy(bias).to(dev)
    C = torch.empty((M, N), dtype=torch.float16, device=dev)
    assert g.gemm_f16_ptr(a1.data_ptr(), b1.data_ptr(), tb.data_ptr(), C.data_ptr(), M, N, K, "bias",
                          torch.cuda.current_stream().cuda_stream) == 0
    st, word = g.gemm_f16_debug_status()
    assert st == 0, hex(word)
    ref = oracle_mod.gemm(A, B, bias, "bias")
    assert np.array_equal(C.cpu().numpy().view(np.uint16), ref.view(np.uint16))


def test_odd_k_repacks_a(g, torch_dev, oracle_mod):
    rng = np.random.default_rng(7)
    M, N, K = 150, 264, 77
    A, B, bias = rand16(rng, (M, K)), rand16(rng, (K, N)), rand16(rng, N)
    assert g.gemm_f16_plan(M, N, K, "bias")["pack_a"] == 1
    assert_parity(run(g, torch_dev, A, B, bias, "bias"), oracle_mod.gemm(A, B, bias, "bias"))


def test_guard_zones_untouched(g, torch_dev, oracle_mod):
    torch, dev = torch_dev
    rng = np.random.default_rng(8)
    M, N, K = 130, 264, 72
    A, B, bias = rand16(rng, (M, K)), rand16(rng, (K, N)), rand16(rng, N)
    pad = 4096
    sentinel = np.float16(-12345.0)
    buf = torch.full((pad + M * N + pad,), float(sentinel), dtype=torch.float16, device=dev)
    C = buf[pad:pad + M * N].view(M, N)
    tA, tB, tb = _dev(torch, A, dev), _dev(torch, B, dev), _dev(torch, bias, dev)
    g.gemm_f16(tA, tB, tb, C, "bias_relu")
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    assert np.all(host[:pad] == sentinel) and np.all(host[pad + M * N:] == sentinel)
    assert_parity(host[pad:pad + M * N].reshape(M, N), oracle_mod.gemm(A, B, bias, "bias_relu"))
    # inputs unchanged
    assert np.array_equal(tA.cpu().numpy().view(np.uint16), A.view(np.uint16))
    assert np.array_equal(tB.cpu().numpy().view(np.uint16), B.view(np.uint16))


def test_deterministic(g, torch_dev):
    rng = np.random.default_rng(9)
    A, B, bias = rand16(rng, (777, 999)), rand16(rng, (999, 1234)), rand16(rng, 1234)
    c1 = run(g, torch_dev, A, B, bias, "bias_gelu_erf")
    c2 = run(g, torch_dev, A, B, bias, "bias_gelu_erf")
    assert np.array_equal(c1.view(np.uint16), c2.view(np.uint16))


def test_k_zero_and_empty(g, torch_dev):
    torch, dev = torch_dev
    bias = np.array([-2.0, -0.5, 0.0, 1.0, 3.0, 0.25, -1.0, 2.0], np.float16)
    tb = _dev(torch, bias, dev)
    C = torch.full((5, 8), 9.0, dtype=torch.float16, device=dev)
    empty_a = torch.empty((5, 0), dtype=torch.float16, device=dev)
    empty_b = torch.empty((0, 8), dtype=torch.float16, device=dev)
    g.gemm_f16(empty_a, empty_b, tb, C, "bias_relu")
    assert np.array_equal(C.cpu().numpy(), np.tile(np.maximum(bias, 0), (5, 1)))
    g.gemm_f16(empty_a, empty_b, None, C, "none")
    assert np.all(C.cpu().numpy() == 0)
    C0 = torch.empty((0, 8), dtype=torch.float16, device=dev)
    g.gemm_f16(torch.empty((0, 4), dtype=torch.float16, device=dev),
               torch.empty((4, 8), dtype=torch.float16, device=dev), None, C0, "none")


def test_runs_on_a_side_stream(g, torch_dev, oracle_mod):
    torch, dev = torch_dev
    rng = np.random.default_rng(10)
    A, B, bias = rand16(rng, (256, 512)), rand16(rng, (512, 384)), rand16(rng, 384)
    s = torch.cuda.Stream()
    tA, tB, tb = _dev(torch, A, dev), _dev(torch, B, dev), _dev(torch, bias, dev)
    C = torch.empty((256, 384), dtype=torch.float16, device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g.gemm_f16(tA, tB, tb, C, "bias")
    s.synchronize()
    assert_parity(C.cpu().numpy(), oracle_mod.gemm(A, B, bias, "bias"))


def test_bounded_wait_reports_timeout_and_context_survives(g, torch_dev, oracle_mod):
    # a barrier nothing arrives on: the wait gives up after 2 ms and reports it
    assert g.gemm_f16_selftest_timeout(2000) == g.GEMM_ERR_TIMEOUT
    assert g.gemm_f16_debug_status()[0] == g.GEMM_OK          # cleared
    rng = np.random.default_rng(11)
    A, B = rand16(rng, (128, 64)), rand16(rng, (64, 128))
    assert_parity(run(g, torch_dev, A, B, None, "none"), oracle_mod.gemm(A, B, None, "none"))


# ---------------------------------------------------------------- every kernel configuration

CONFIGS = ["pair256x256", "pair_whole", "128x256", "128x128", "128x64", "swap"]


@pytest.fixture
def forced(g):
    prev = g.gemm_f16_force_config("auto")
    yield g
    g.gemm_f16_force_config(prev)


@pytest.mark.parametrize("cfg", CONFIGS)
@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (512, 768, 320), (300, 200, 136), (129, 520, 1000)])
def test_forced_config_integer_exact(forced, torch_dev, oracle_mod, cfg, M, N, K):
    g = forced
    g.gemm_f16_force_config(cfg)
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    A = rng.integers(-2, 3, (M, K)).astype(np.float16)
    B = rng.integers(-2, 3, (K, N)).astype(np.float16)
    bias = rng.integers(-8, 9, N).astype(np.float16)
    got = run(g, torch_dev, A, B, bias, "bias")
    assert np.array_equal(got, oracle_mod.gemm(A, B, bias, "bias"))


@pytest.mark.parametrize("cfg", CONFIGS)
@pytest.mark.parametrize("M,N,K,epi", [(1, 1, 1, "bias_gelu_erf"), (257, 129, 65, "bias_relu"),
                                       (700, 1100, 333, "bias_gelu_erf"), (2000, 600, 96, "none"),
                                       (40, 5003, 200, "bias")])
def test_forced_config_random(forced, torch_dev, oracle_mod, cfg, M, N, K, epi):
    g = forced
    g.gemm_f16_force_config(cfg)
    rng = np.random.default_rng(M * 5 + N + K)
    A, B, bias = rand16(rng, (M, K), 0.5), rand16(rng, (K, N), 0.5), rand16(rng, N)
    got = run(g, torch_dev, A, B, bias, epi)
    assert_parity(got, oracle_mod.gemm(A, B, bias if epi != "none" else None, epi), f"{cfg} {M}x{N}x{K}")


@pytest.mark.parametrize("cfg", CONFIGS)
def test_forced_config_many_tiles_per_cta(forced, torch_dev, oracle_mod, cfg):
    # several tiles per persistent CTA (both TMEM accumulators reused repeatedly)
    g = forced
    g.gemm_f16_force_config(cfg)
    rng = np.random.default_rng(17)
    M, N, K = 4096, 4096, 128
    A, B, bias = rand16(rng, (M, K), 0.3), rand16(rng, (K, N), 0.3), rand16(rng, N)
    got = run(g, torch_dev, A, B, bias, "bias_gelu_erf")
    rows = np.arange(3, M, 61)
    assert_parity(got[rows], oracle_mod.gemm_rows(A, B, bias, "bias_gelu_erf", rows), cfg)


# ---------------------------------------------------------------- short A: the swap-AB kernel

@pytest.mark.parametrize("M,N,K,epi", [(1, 128, 64, "bias"), (7, 300, 77, "bias_gelu_erf"), (16, 1024, 512, "none"),
                                       (17, 5003, 1000, "bias_relu"), (33, 264, 130, "bias_gelu_erf"),
                                       (64, 2048, 4096, "bias"), (48, 129, 8, "none")])
def test_short_a_swap_path(g, torch_dev, oracle_mod, M, N, K, epi):
    assert g.gemm_f16_plan(M, N, K, epi)["path"] == 3
    rng = np.random.default_rng(M * 31 + N + K)
    A, B, bias = rand16(rng, (M, K), 0.5), rand16(rng, (K, N), 0.5), rand16(rng, N)
    got = run(g, torch_dev, A, B, bias, epi)
    assert_parity(got, oracle_mod.gemm(A, B, bias if epi != "none" else None, epi), f"{M}x{N}x{K} {epi}")


@pytest.mark.parametrize("M", [1, 16, 40, 64])
def test_short_a_integer_exact(g, torch_dev, oracle_mod, M):
    rng = np.random.default_rng(M)
    N, K = 520, 264
    A = rng.integers(-2, 3, (M, K)).astype(np.float16)
    B = rng.integers(-2, 3, (K, N)).astype(np.float16)
    bias = rng.integers(-8, 9, N).astype(np.float16)
    got = run(g, torch_dev, A, B, bias, "bias_relu")
    assert np.array_equal(got, oracle_mod.gemm(A, B, bias, "bias_relu"))


@pytest.mark.parametrize("M,N,K", [(16, 256, 4096), (40, 1000, 2000), (64, 384, 8192), (3, 130, 1024)])
def test_short_a_split_k_integer_exact(g, torch_dev, oracle_mod, M, N, K):
    plan = g.gemm_f16_plan(M, N, K, "bias")
    assert plan["path"] == 3 and plan["splits"] > 1
    rng = np.random.default_rng(M + N + K)
    A = rng.integers(-1, 2, (M, K)).astype(np.float16)      # |C| <= K: exact in fp32 and, here, fp16 for K <= 2048
    B = rng.integers(-1, 2, (K, N)).astype(np.float16)
    bias = rng.integers(-8, 9, N).astype(np.float16)
    got = run(g, torch_dev, A, B, bias, "bias")
    ref = oracle_mod.gemm(A, B, bias, "bias")
    if K <= 2048:
        assert np.array_equal(got, ref)
    else:
        assert_parity(got, ref, f"{M}x{N}x{K}")


@pytest.mark.parametrize("epi", EPIS)
def test_short_a_split_k_random_and_deterministic(g, torch_dev, oracle_mod, epi):
    M, N, K = 24, 1536, 6000
    assert g.gemm_f16_plan(M, N, K, epi)["splits"] > 1
    rng = np.random.default_rng(21)
    A, B, bias = rand16(rng, (M, K), 0.1), rand16(rng, (K, N), 0.1), rand16(rng, N)
    c1 = run(g, torch_dev, A, B, bias, epi)
    c2 = run(g, torch_dev, A, B, bias, epi)
    assert np.array_equal(c1.view(np.uint16), c2.view(np.uint16))
    assert_parity(c1, oracle_mod.gemm(A, B, bias if epi != "none" else None, epi), epi)


# ---------------------------------------------------------------- K split across a cluster (128-row tiles)

@pytest.fixture
def ksplit(g):
    prev_cfg = g.gemm_f16_force_config("auto")
    prev = g.gemm_f16_force_ksplit(0)
    yield g
    g.gemm_f16_force_ksplit(prev)
    g.gemm_f16_force_config(prev_cfg)


@pytest.mark.parametrize("S", [2, 4])
@pytest.mark.parametrize("cfg", ["128x64", "128x128", "128x256"])
@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (300, 200, 1000), (129, 264, 1000)])
def test_ksplit_integer_exact(ksplit, torch_dev, oracle_mod, S, cfg, M, N, K):
    g = ksplit
    g.gemm_f16_force_config(cfg)
    g.gemm_f16_force_ksplit(S)
    assert g.gemm_f16_plan(M, N, K, "bias")["splits"] == S
    rng = np.random.default_rng(M * 7 + N + K + S)
    A = rng.integers(-1, 2, (M, K)).astype(np.float16)
    B = rng.integers(-1, 2, (K, N)).astype(np.float16)
    bias = rng.integers(-8, 9, N).astype(np.float16)
    got = run(g, torch_dev, A, B, bias, "bias")
    assert np.array_equal(got.view(np.uint16), oracle_mod.gemm(A, B, bias, "bias").view(np.uint16))


@pytest.mark.parametrize("epi", EPIS)
def test_ksplit_every_epilogue_ragged_and_unaligned_c(ksplit, torch_dev, oracle_mod, epi):
    # N % 8 != 0: B repacked and C rows not 16-byte aligned (element-wise stores)
    g = ksplit
    M, N, K = 333, 1003, 2000
    g.gemm_f16_force_ksplit(4)
    plan = g.gemm_f16_plan(M, N, K, epi)
    assert plan["splits"] == 4 and plan["vec_store"] == 0
    rng = np.random.default_rng(77)
    A, B, bias = rand16(rng, (M, K), 0.05), rand16(rng, (K, N), 0.05), rand16(rng, N)
    got = run(g, torch_dev, A, B, bias if epi != "none" else None, epi)
    assert_parity(got, oracle_mod.gemm(A, B, bias if epi != "none" else None, epi), epi)


def test_ksplit_automatic_choice_matches_oracle(ksplit, torch_dev, oracle_mod):
    g = ksplit
    for (M, N, K) in [(1024, 1024, 1024), (1536, 768, 4096), (512, 512, 512)]:
        plan = g.gemm_f16_plan(M, N, K, "bias_gelu_erf")
        rng = np.random.default_rng(M + K)
        A, B, bias = rand16(rng, (M, K), 1 / 32), rand16(rng, (K, N), 1 / 32), rand16(rng, N)
        got = run(g, torch_dev, A, B, bias, "bias_gelu_erf")
        rows = np.array([0, 1, M // 2, M - 1])
        assert_parity(got[rows], oracle_mod.gemm_rows(A, B, bias, "bias_gelu_erf", rows), f"{M}x{N}x{K} {plan}")
        c2 = run(g, torch_dev, A, B, bias, "bias_gelu_erf")
        assert np.array_equal(got.view(np.uint16), c2.view(np.uint16))   # a fixed summation order


# ---------------------------------------------------------------- the device GELU itself

@pytest.mark.parametrize("epi", ["bias_gelu_erf", "bias_gelu_tanh", "bias_sigmoid"])
def test_device_activation_on_every_fp16_value_in_range(g, torch_dev, oracle_mod, epi):
    # C[i, j] = x_i exactly (x_i * 1 + zeros), so the epilogue sees every fp16 value in
    # [-10, 10].  The device activations run in fp32 (erfc by Abramowitz & Stegun 7.1.26,
    # tanh and the sigmoid through the fast exponential), each written so that no
    # difference of nearly equal terms occurs in the negative tail: every result, the
    # fp16 subnormals included, lies within 1 fp16 ulp of the fp64 definition, and
    # almost all are bit-equal.
    bits = np.arange(1 << 16, dtype=np.uint16)
    xs = bits.view(np.float16)
    xs = xs[np.isfinite(xs)]
    xs = np.unique(xs[np.abs(xs.astype(np.float64)) <= 10.0])
    M, N, K = xs.size, 16, 8
    A = np.zeros((M, K), np.float16)
    A[:, 0] = xs
    B = np.zeros((K, N), np.float16)
    B[0, :] = 1.0
    bias = np.zeros(N, np.float16)
    got = run(g, torch_dev, A, B, bias, epi)[:, 0]
    ref = oracle_mod.gemm(A, B, bias, epi)[:, 0]
    gb = got.view(np.uint16).astype(np.int64)
    rb = ref.view(np.uint16).astype(np.int64)
    # ulp distance on the sign-magnitude fp16 encoding (+0 and -0 are 0 apart)
    def ordered(b):
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    dist = np.abs(ordered(gb) - ordered(rb))
    bad = dist > 1
    assert not bad.any(), (xs[bad][:5], got[bad][:5], ref[bad][:5], dist.max())
    assert (dist == 0).mean() >= 0.99
    # where |result| >= 2^-10 the fp16 spacing dwarfs the fp32 error: nearly all bit-equal
    big = np.abs(ref.astype(np.float64)) >= 2.0 ** -10
    assert (dist[big] == 0).mean() >= 0.995



# ---------------------------------------------------------------- CTA pair: half-tile units for a partial last wave

@pytest.mark.parametrize("M,N,K", [(2560, 2560, 1920), (2304, 2816, 1536), (4096, 4096, 640), (300, 4003, 200)])
def test_pair_half_tile_tail_integer_exact(forced, torch_dev, oracle_mod, M, N, K):
    g = forced
    g.gemm_f16_force_config("pair256x256")
    assert g.gemm_f16_plan(M, N, K, "bias")["whole_tiles"] >= 0
    rng = np.random.default_rng(M + N + K)
    A = rng.integers(-1, 2, (M, K)).astype(np.float16)   # |C| <= K + 4 <= 1924: exact in fp32 and fp16
    B = rng.integers(-1, 2, (K, N)).astype(np.float16)
    bias = rng.integers(-4, 5, N).astype(np.float16)
    assert np.array_equal(run(g, torch_dev, A, B, bias, "bias"), oracle_mod.gemm(A, B, bias, "bias"))


def test_pair_half_tile_tail_gelu(g, torch_dev, oracle_mod):
    M, N, K = 2816, 2560, 1280
    assert g.gemm_f16_plan(M, N, K, "bias_gelu_erf")["whole_tiles"] > 0
    rng = np.random.default_rng(33)
    A, B, bias = rand16(rng, (M, K), 0.05), rand16(rng, (K, N), 0.05), rand16(rng, N)
    assert_parity(run(g, torch_dev, A, B, bias, "bias_gelu_erf"), oracle_mod.gemm(A, B, bias, "bias_gelu_erf"))
