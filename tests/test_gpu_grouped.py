"""GPU parity of gemm_f16_grouped: many independent problems in one persistent
launch, each checked against the oracle's definition of a grouped GEMM (every
problem on its own).  Bit-exact with small-integer operands, else the
oracle.compare tolerance."""
import numpy as np
import pytest

from oracle.compare import parity

pytestmark = pytest.mark.gpu


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


SENTINEL = 0x7E5A


def ints(rng, shape, lo=-2, hi=3):
    return rng.integers(lo, hi, shape).astype(np.float16)


def rand16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def device_problems(torch, dev, probs, layout="nn"):
    """Device views (A, B, bias, C) of host problems (A, B, bias), A / B stored
    transposed where `layout` says so; C pre-filled with a NaN sentinel."""
    out = []
    for A, B, bias in probs:
        Ad = torch.from_numpy(np.ascontiguousarray(A.T if layout[0] == "t" else A)).to(dev)
        Bd = torch.from_numpy(np.ascontiguousarray(B.T if layout[1] == "t" else B)).to(dev)
        Ad = Ad.t() if layout[0] == "t" else Ad
        Bd = Bd.t() if layout[1] == "t" else Bd
        C = torch.empty((A.shape[0], B.shape[1]), dtype=torch.float16, device=dev)
        C.view(torch.int16).fill_(SENTINEL)
        out.append((Ad, Bd, torch.from_numpy(bias).to(dev) if bias is not None else None, C))
    return out


def run_grouped(g, torch_dev, probs, epi, layout="nn"):
    torch, dev = torch_dev
    dp = device_problems(torch, dev, probs, layout)
    g.gemm_f16_grouped(dp, epi)
    st, word = g.gemm_f16_debug_status()
    assert st == 0, f"device status {st} word {word:#x}"
    return [C.cpu().numpy() for _, _, _, C in dp]


@pytest.mark.parametrize("layout", ["nn", "nt", "tn", "tt"])
def test_grouped_integer_exact_ragged_sizes(g, torch_dev, oracle_mod, layout):
    rng = np.random.default_rng(50 + len(layout))
    shapes = [(256, 256, 128), (300, 200, 136), (1, 64, 64), (700, 1100, 72), (129, 257, 200), (64, 8, 1000),
              (512, 520, 64), (0, 128, 64), (96, 0, 64), (1000, 33, 512)]
    probs = [(ints(rng, (M, K)), ints(rng, (K, N)), ints(rng, N, -8, 9)) for M, N, K in shapes]
    got = run_grouped(g, torch_dev, probs, "bias", layout)
    for i, (c, r) in enumerate(zip(got, oracle_mod.gemm_grouped(probs, "bias"))):
        assert c.shape == r.shape
        assert np.array_equal(c, r), f"problem {i} {shapes[i]} {layout}"


@pytest.mark.parametrize("epi", ["none", "bias", "bias_relu", "bias_gelu_erf", "bias_sigmoid", "bias_gelu_tanh"])
def test_grouped_random_every_epilogue(g, torch_dev, oracle_mod, epi):
    rng = np.random.default_rng(60)
    shapes = [(512, 768, 320), (257, 129, 65), (40, 1000, 200), (1024, 256, 1024), (3, 5, 7)]
    probs = [(rand16(rng, (M, K), 0.5), rand16(rng, (K, N), 0.5), rand16(rng, N)) for M, N, K in shapes]
    got = run_grouped(g, torch_dev, probs, epi)
    for i, (c, r) in enumerate(zip(got, oracle_mod.gemm_grouped(probs, epi))):
        res = parity(c, r)
        assert res["ok"], f"problem {i} {shapes[i]} {epi}: {res}"


@pytest.mark.parametrize("layout", ["nn", "tt"])
def test_grouped_whole_and_half_tiles(g, torch_dev, oracle_mod, layout):
    # 100 tiles of 256 x 256 over ten problems: with 76 CTA pairs (152 SMs)
    # the first 76 run whole and the last 24 as 48 halves of 256 x 128, the
    # halves spanning three problems; integer operands, so bit-exact
    rng = np.random.default_rng(66)
    shapes = [(512, 1280, 64)] * 7 + [(300, 1100, 72), (512, 1280, 64), (257, 1203, 64)]
    probs = [(ints(rng, (M, K)), ints(rng, (K, N)), ints(rng, N, -8, 9)) for M, N, K in shapes]
    got = run_grouped(g, torch_dev, probs, "bias", layout)
    for i, (c, r) in enumerate(zip(got, oracle_mod.gemm_grouped(probs, "bias"))):
        assert np.array_equal(c, r), f"problem {i} {shapes[i]} {layout}"


def test_grouped_k_zero_and_repacked_operands(g, torch_dev, oracle_mod):
    rng = np.random.default_rng(61)
    shapes = [(100, 60, 0), (300, 1003, 136), (257, 300, 61), (64, 64, 64)]   # K=0; N % 8; K % 8
    probs = [(ints(rng, (M, K)), ints(rng, (K, N)), ints(rng, N, -8, 9)) for M, N, K in shapes]
    got = run_grouped(g, torch_dev, probs, "bias_relu")
    for i, (c, r) in enumerate(zip(got, oracle_mod.gemm_grouped(probs, "bias_relu"))):
        assert np.array_equal(c, r), f"problem {i} {shapes[i]}"


def test_grouped_more_problems_than_one_launch(g, torch_dev, oracle_mod):
    # 150 problems: three launches of at most 64
    rng = np.random.default_rng(62)
    probs = []
    for i in range(150):
        M, N, K = int(rng.integers(1, 300)), int(rng.integers(1, 300)), int(rng.integers(8, 200))
        probs.append((ints(rng, (M, K)), ints(rng, (K, N)), ints(rng, N, -8, 9)))
    got = run_grouped(g, torch_dev, probs, "bias")
    for i, (c, r) in enumerate(zip(got, oracle_mod.gemm_grouped(probs, "bias"))):
        assert np.array_equal(c, r), f"problem {i} {probs[i][0].shape} x {probs[i][1].shape}"


def test_grouped_mixed_layouts_in_one_call(g, torch_dev, oracle_mod):
    torch, dev = torch_dev
    rng = np.random.default_rng(63)
    probs = [(ints(rng, (300, 256)), ints(rng, (256, 520)), ints(rng, 520, -8, 9)) for _ in range(4)]
    dp = []
    for layout, p in zip(["nn", "nt", "tn", "tt"], probs):
        dp += device_problems(torch, dev, [p], layout)
    g.gemm_f16_grouped(dp, "bias")
    for i, (c, r) in enumerate(zip(dp, oracle_mod.gemm_grouped(probs, "bias"))):
        assert np.array_equal(c[3].cpu().numpy(), r), f"problem {i}"


def test_grouped_expert_shapes_sampled(g, torch_dev, oracle_mod):
    # mixture-of-experts shape: 8 experts, one weight [N, K] each (a Linear
    # layer's layout, so B = W^T), token counts from empty to 3000
    torch, dev = torch_dev
    rng = np.random.default_rng(64)
    N, K = 1024, 2048
    Ms = [0, 37, 256, 1000, 3000, 3, 512, 700]
    probs = [(rand16(rng, (M, K), K ** -0.5), rand16(rng, (K, N)), rand16(rng, N)) for M in Ms]
    got = run_grouped(g, torch_dev, probs, "bias_gelu_erf", "nt")
    for i, (M, (A, B, bias)) in enumerate(zip(Ms, probs)):
        if M == 0:
            assert got[i].shape == (0, N)
            continue
        rows = sorted({0, M - 1, M // 2, M // 3})
        res = parity(got[i][rows], oracle_mod.gemm_rows(A, B, bias, "bias_gelu_erf", rows))
        assert res["ok"], f"expert {i} (M={M}): {res}"


def test_grouped_under_graph_capture(g, torch_dev, oracle_mod):
    torch, dev = torch_dev
    rng = np.random.default_rng(65)
    shapes = [(256, 512, 256), (100, 300, 64), (512, 256, 128)]
    probs = [(ints(rng, (M, K)), ints(rng, (K, N)), ints(rng, N, -8, 9)) for M, N, K in shapes]
    dp = device_problems(torch, dev, probs)
    g.gemm_f16_grouped(dp, "bias")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.gemm_f16_grouped(dp, "bias")
    for _, _, _, C in dp:
        C.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for i, (c, r) in enumerate(zip(dp, oracle_mod.gemm_grouped(probs, "bias"))):
        assert np.array_equal(c[3].cpu().numpy(), r), f"problem {i}"
