"""GPU parity of the strided / transposed operand layouts (gemm_f16_ex).

The tile GEMM primitive of "writing-tilelang-kernels" (Key API Patterns,
T.gemm) takes transpose_A / transpose_B; gemm_f16_ex offers the same for the
operands in global memory, plus row pitches.  Every case here computes the
LOGICAL matrices A [M,K] and B [K,N] on the host, hands the oracle those
(row-major, contiguous), and hands the CUDA path a differently stored copy of
the same values: transposed (A as K x M, B as N x K) and/or with padded rows.
The bar is the one of test_gpu_parity.py: bit-exact where every step is
exact (small integers), else the oracle.compare tolerance.
"""
import numpy as np
import pytest

import workloads
from oracle.compare import parity

pytestmark = pytest.mark.gpu

LAYOUTS = ("nn", "nt", "tn", "tt")   # first letter A, second B: n = as is, t = stored transposed
CONFIGS = ["auto", "pair256x256", "pair_whole", "128x256", "128x128", "128x64", "swap"]
SENTINEL = 0x7E5A   # a NaN pattern no computed element can take


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


@pytest.fixture
def forced(g):
    prev = g.gemm_f16_force_config("auto")
    yield g
    g.gemm_f16_force_config(prev)


def stored(torch, dev, X, trans, pad=0):
    """The logical matrix X as a device view of X's shape whose storage is
    row-major with `pad` spare elements per stored row, holding X itself or
    (trans) X^T.  Returns (view, backing buffer)."""
    S = np.ascontiguousarray(X.T if trans else X)
    r, c = S.shape
    buf = torch.empty((r, c + pad), dtype=torch.float16, device=dev)
    buf.view(torch.int16).fill_(SENTINEL)   # NaN in the padding: reading it would show in C
    buf[:, :c] = torch.from_numpy(S).to(dev)
    v = buf[:, :c]
    return (v.t() if trans else v), buf


def run_layout(g, torch_dev, A, B, bias, epi, layout, pad_a=0, pad_b=0, pad_c=0):
    torch, dev = torch_dev
    M, K = A.shape
    N = B.shape[1]
    Av, _ = stored(torch, dev, A, layout[0] == "t", pad_a)
    Bv, _ = stored(torch, dev, B, layout[1] == "t", pad_b)
    Cbuf = torch.empty((M, N + pad_c), dtype=torch.float16, device=dev)
    Cbuf.view(torch.int16).fill_(SENTINEL)
    C = Cbuf[:, :N]
    bias_d = torch.from_numpy(bias).to(dev) if epi != "none" else None
    g.gemm_f16(Av, Bv, bias_d, C, epi)
    st, word = g.gemm_f16_debug_status()
    assert st == 0, f"device status {st} word {word:#x}"
    out = Cbuf.cpu().numpy()
    if pad_c:
        assert np.all(out[:, N:].view(np.uint16) == SENTINEL), "C padding was written"
    return out[:, :N]


def ints(rng, shape, lo=-2, hi=3):
    return rng.integers(lo, hi, shape).astype(np.float16)


def rand16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


# ---------------------------------------------------------------- every layout on every kernel, exact

@pytest.mark.parametrize("cfg", CONFIGS)
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("M,N,K", [(256, 512, 128), (200, 300, 136), (129, 257, 72), (40, 1000, 200)])
def test_layout_integer_exact(forced, torch_dev, oracle_mod, cfg, layout, M, N, K):
    g = forced
    g.gemm_f16_force_config(cfg)
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    A, B, bias = ints(rng, (M, K)), ints(rng, (K, N)), ints(rng, N, -8, 9)
    got = run_layout(g, torch_dev, A, B, bias, "bias", layout)
    ref = oracle_mod.gemm(A, B, bias, "bias")
    assert np.array_equal(got, ref), f"{cfg} {layout}: max diff {np.abs(got.astype(float) - ref).max()}"


# ---------------------------------------------------------------- 3-D operand maps
# MN-major operands (B stored K x N, A stored K x M) whose MN extent and pitch are
# multiples of 64 load both 64-wide boxes of a CTA's slice with one 3-D tensor-map
# load: an odd number of 64-wide groups leaves the last slice's second box past
# the end (read as zeros); a pitch of MN + 64 keeps the 3-D path with rows longer
# than MN; a pitch of MN + 8 falls back to 2-D boxes.  Small shapes run as CTA-pair
# half tiles, larger ones as whole tiles.

@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("M,N,K,pad", [(192, 320, 128, 0), (320, 192, 200, 0), (448, 576, 264, 64),
                                       (576, 448, 128, 8), (2304, 2624, 192, 0)])
def test_mn3d_maps_integer_exact(forced, torch_dev, oracle_mod, layout, M, N, K, pad):
    forced.gemm_f16_force_config("pair256x256")
    rng = np.random.default_rng(M + N + K + pad)
    A, B, bias = ints(rng, (M, K)), ints(rng, (K, N)), ints(rng, N, -8, 9)
    got = run_layout(forced, torch_dev, A, B, bias, "bias", layout, pad, pad)
    ref = oracle_mod.gemm(A, B, bias, "bias")
    assert np.array_equal(got, ref), f"{layout} {M}x{N}x{K} pad {pad}: max diff {np.abs(got.astype(float) - ref).max()}"


# ---------------------------------------------------------------- row pitches

@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("pads", [(8, 16, 8), (3, 5, 1), (0, 0, 7), (64, 8, 0)])
def test_pitches_integer_exact_and_c_padding_untouched(g, torch_dev, oracle_mod, layout, pads):
    # pads of a multiple of 8 keep the operands TMA-readable in place; odd pads
    # take the repack; an odd C pitch takes the staged (narrow) stores
    rng = np.random.default_rng(sum(pads) + 11)
    M, N, K = 300, 520, 200
    A, B, bias = ints(rng, (M, K)), ints(rng, (K, N)), ints(rng, N, -8, 9)
    got = run_layout(g, torch_dev, A, B, bias, "bias_relu", layout, *pads)
    assert np.array_equal(got, oracle_mod.gemm(A, B, bias, "bias_relu"))


@pytest.mark.parametrize("layout", ("nt", "tn"))
def test_pitches_short_a_swap_path(g, torch_dev, oracle_mod, layout):
    rng = np.random.default_rng(5)
    for M in (1, 16, 33, 64):
        A, B, bias = ints(rng, (M, 1024)), ints(rng, (1024, 384)), ints(rng, 384, -8, 9)
        got = run_layout(g, torch_dev, A, B, bias, "bias", layout, 8, 8, 8)
        assert np.array_equal(got, oracle_mod.gemm(A, B, bias, "bias")), f"M={M}"


# ---------------------------------------------------------------- random values, every epilogue

@pytest.mark.parametrize("layout", ("nt", "tn", "tt"))
@pytest.mark.parametrize("epi", ["bias_gelu_erf", "bias_sigmoid", "none"])
@pytest.mark.parametrize("M,N,K", [(700, 1100, 333), (1, 1, 1), (3001, 260, 96), (17, 5003, 1000)])
def test_layout_random(g, torch_dev, oracle_mod, layout, epi, M, N, K):
    rng = np.random.default_rng(M * 5 + N + K)
    A, B, bias = rand16(rng, (M, K), 0.5), rand16(rng, (K, N), 0.5), rand16(rng, N)
    got = run_layout(g, torch_dev, A, B, bias, epi, layout)
    res = parity(got, oracle_mod.gemm(A, B, bias if epi != "none" else None, epi))
    assert res["ok"], f"{layout} {epi} {M}x{N}x{K}: {res}"


def test_linear_layer_weight_view(g, torch_dev, oracle_mod):
    # y = x W^T + b with W stored [N, K], as a Linear layer keeps it: B = W.t()
    torch, dev = torch_dev
    rng = np.random.default_rng(21)
    M, N, K = 1000, 3072, 768
    X, W, bias = rand16(rng, (M, K), 0.5), rand16(rng, (N, K), 0.05), rand16(rng, N)
    Wd = torch.from_numpy(W).to(dev)
    C = torch.empty((M, N), dtype=torch.float16, device=dev)
    g.gemm_f16(torch.from_numpy(X).to(dev), Wd.t(), torch.from_numpy(bias).to(dev), C, "bias_gelu_tanh")
    assert g.gemm_f16_debug_status()[0] == 0
    res = parity(C.cpu().numpy(), oracle_mod.gemm(X, np.ascontiguousarray(W.T), bias, "bias_gelu_tanh"))
    assert res["ok"], res


# ---------------------------------------------------------------- the large workloads, sampled

@pytest.mark.parametrize("name,layout", [("fused8192", "nt"), ("fused4096", "tn"), ("fused4096", "tt"),
                                         ("skinny16x8192x8192", "nt"), ("skinny16x8192x8192", "tn"),
                                         ("ragged3001x5003x1000", "tt")])
def test_workload_layouts_sampled(g, torch_dev, oracle_mod, name, layout):
    w = workloads.WORKLOADS[name]
    A, B, bias = w.make()
    epi = w.epilogues[-1]
    got = run_layout(g, torch_dev, A, B, bias, epi, layout)
    b = bias if epi != "none" else None
    rows = [0, w.M - 1] + list(workloads.sample_coords(w.seed + 2000, w.M, 1, 2)[0])
    res = parity(got[rows], oracle_mod.gemm_rows(A, B, b, epi, rows))
    assert res["ok"], f"{name} {layout} rows: {res}"
    ii, jj = workloads.sample_coords(w.seed + 1, w.M, w.N, workloads.SAMPLED_ELEMS)
    res = parity(got[ii, jj], oracle_mod.gemm_elems(A, B, b, epi, ii, jj))
    assert res["ok"], f"{name} {layout} elems: {res}"
