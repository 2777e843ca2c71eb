"""GPU tests of how calls are launched: dependent chains with programmatic
dependent launch on and off, write-after-read reuse of buffers, and CUDA-graph
capture and replay.

Every chain uses small-integer or dyadic inputs whose products and sums are
exact in fp32, so each intermediate C is the exactly rounded fp16 of an exact
value on both sides.  The oracle's chain is computed from its own outputs
(never from the GPU's), and the two chains agree bit for bit.
"""
import numpy as np
import pytest

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


@pytest.fixture
def pdl_restore(g):
    prev = g.gemm_f16_set_pdl(True)
    yield g
    g.gemm_f16_set_pdl(prev)


def tern(rng, shape, scale=1.0):
    """Entries in {-1, 0, 1} * scale (scale a power of two)."""
    return (rng.integers(-1, 2, shape) * scale).astype(np.float16)


def two_per_column(rng, K, N):
    """Each column: +1 in one random row and +-1 in another (x W is then a
    signed sum of two columns of x: exact, and at most doubles magnitudes)."""
    W = np.zeros((K, N), np.float16)
    for j in range(N):
        k1, k2 = rng.choice(K, 2, replace=False)
        W[k1, j] = 1.0
        W[k2, j] = rng.choice([-1.0, 1.0])
    return W


def chain_inputs(seed, M, K1=64, N1=256, N2=384, N3=200):
    rng = np.random.default_rng(seed)
    return dict(
        X=tern(rng, (M, K1)),                 # |C1| <= 64
        W1=tern(rng, (K1, N1)), b1=rng.integers(-4, 5, N1).astype(np.float16),
        W2=tern(rng, (N1, N2)), b2=rng.integers(-4, 5, N2).astype(np.float16),   # |C2| <= 17000
        W3=tern(rng, (N2, N3), 1.0 / 128.0),  # |C3| <= 17000 * 384 / 128 ~ 51000, sums exact in fp32
    )


def oracle_chain(o, d):
    c1 = o.gemm(d["X"], d["W1"], d["b1"], "bias_relu")
    c2 = o.gemm(c1, d["W2"], d["b2"], "bias")
    c3 = o.gemm(c2, d["W3"], None, "none")
    return c1, c2, c3


def to_dev(torch, dev, d):
    return {k: torch.from_numpy(v).to(dev) for k, v in d.items()}


def gpu_chain(g, torch, dev, t, out=None):
    M = t["X"].shape[0]
    if out is None:
        out = (torch.empty((M, t["W1"].shape[1]), dtype=torch.float16, device=dev),
               torch.empty((M, t["W2"].shape[1]), dtype=torch.float16, device=dev),
               torch.empty((M, t["W3"].shape[1]), dtype=torch.float16, device=dev))
    c1, c2, c3 = out
    g.gemm_f16(t["X"], t["W1"], t["b1"], c1, "bias_relu")
    g.gemm_f16(c1, t["W2"], t["b2"], c2, "bias")
    g.gemm_f16(c2, t["W3"], None, c3, "none")
    return out


@pytest.mark.parametrize("pdl", [True, False])
@pytest.mark.parametrize("M", [256, 48, 1000, 4096])
def test_dependent_chain_exact(pdl_restore, torch_dev, oracle_mod, pdl, M):
    g = pdl_restore
    torch, dev = torch_dev
    g.gemm_f16_set_pdl(pdl)
    d = chain_inputs(M, M)
    ref = oracle_chain(oracle_mod, d)
    t = to_dev(torch, dev, d)
    for rep in range(3):
        got = gpu_chain(g, torch, dev, t)
        assert g.gemm_f16_debug_status()[0] == 0
        for i, (a, b) in enumerate(zip(got, ref)):
            assert np.array_equal(a.cpu().numpy(), b), f"step {i + 1} of the chain, repeat {rep}"


def test_write_after_read_reuse(pdl_restore, torch_dev, oracle_mod):
    # each call overwrites the buffer the previous call read from: a call that
    # wrote before its predecessor finished reading would corrupt the chain
    g = pdl_restore
    torch, dev = torch_dev
    rng = np.random.default_rng(3)
    M, K = 512, 256
    X = tern(rng, (M, K))
    Ws = [two_per_column(rng, K, K) for _ in range(6)]   # integer values at most double per layer
    bs = [rng.integers(-2, 3, K).astype(np.float16) for _ in range(6)]
    ref = X
    for W, b in zip(Ws, bs):
        ref = oracle_mod.gemm(ref, W, b, "bias_relu")
    P = torch.from_numpy(X).to(dev)
    Q = torch.empty_like(P)
    Wd = [torch.from_numpy(W).to(dev) for W in Ws]
    bd = [torch.from_numpy(b).to(dev) for b in bs]
    src, dst = P, Q
    for W, b in zip(Wd, bd):
        g.gemm_f16(src, W, b, dst, "bias_relu")   # dst was the source two calls ago
        src, dst = dst, src
    assert g.gemm_f16_debug_status()[0] == 0
    assert np.array_equal(src.cpu().numpy(), ref)


@pytest.mark.parametrize("pdl", [True, False])
def test_graph_capture_and_replay(pdl_restore, torch_dev, oracle_mod, pdl):
    g = pdl_restore
    torch, dev = torch_dev
    g.gemm_f16_set_pdl(pdl)
    M = 256
    d0 = chain_inputs(100, M)
    t = to_dev(torch, dev, d0)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = gpu_chain(g, torch, dev, t)          # eager first: per-device set-up happens outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gpu_chain(g, torch, dev, t, out)
    for seed in (101, 102, 103):
        d = chain_inputs(seed, M)
        for k, v in d.items():
            t[k].copy_(torch.from_numpy(v).to(dev))   # new values in the captured buffers
        graph.replay()
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(out, oracle_chain(oracle_mod, d))):
            assert np.array_equal(a.cpu().numpy(), b), f"replay seed {seed}, step {i + 1}"
    assert g.gemm_f16_debug_status()[0] == 0


def test_graph_capture_with_repack_scratch(pdl_restore, torch_dev, oracle_mod):
    # N % 8 != 0 repacks B into stream-ordered scratch: under capture the
    # allocation and its free become graph memory nodes
    g = pdl_restore
    torch, dev = torch_dev
    rng = np.random.default_rng(9)
    M, N, K = 300, 1003, 136
    A, B, bias = tern(rng, (M, K)), tern(rng, (K, N)), rng.integers(-4, 5, N).astype(np.float16)
    tA, tB, tb = (torch.from_numpy(x).to(dev) for x in (A, B, bias))
    C = torch.empty((M, N), dtype=torch.float16, device=dev)
    assert g.gemm_f16_plan(M, N, K, "bias")["pack_b"] == 1
    g.gemm_f16(tA, tB, tb, C, "bias")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.gemm_f16(tA, tB, tb, C, "bias")
    C.zero_()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle_mod.gemm(A, B, bias, "bias"))


def test_side_stream_pdl_does_not_cross_streams(pdl_restore, torch_dev, oracle_mod):
    # a call on stream s2 that consumes a result of stream s1 is ordered by an
    # event, not by the launch attribute
    g = pdl_restore
    torch, dev = torch_dev
    d = chain_inputs(7, 512)
    ref = oracle_chain(oracle_mod, d)
    t = to_dev(torch, dev, d)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    c1 = torch.empty((512, 256), dtype=torch.float16, device=dev)
    c2 = torch.empty((512, 384), dtype=torch.float16, device=dev)
    s1.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        g.gemm_f16(t["X"], t["W1"], t["b1"], c1, "bias_relu")
    s2.wait_stream(s1)
    with torch.cuda.stream(s2):
        g.gemm_f16(c1, t["W2"], t["b2"], c2, "bias")
    torch.cuda.synchronize()
    assert np.array_equal(c2.cpu().numpy(), ref[1])


def test_one_buffer_many_shapes_same_address(g, torch_dev, oracle_mod):
    # the same base addresses with other extents and pitches: every call must
    # see its own operand shape (encoded tensor maps are reused only on an
    # exact match of address, extents, pitch and box)
    torch, dev = torch_dev
    rng = np.random.default_rng(31)
    bufA = torch.zeros(1 << 20, dtype=torch.float16, device=dev)
    bufB = torch.zeros(1 << 20, dtype=torch.float16, device=dev)
    for M, N, K, lda, ldb in [(256, 256, 256, 256, 256), (256, 128, 512, 512, 128), (128, 256, 256, 512, 256),
                              (256, 256, 256, 264, 256), (256, 256, 256, 256, 256), (64, 1024, 128, 128, 1024)]:
        A, B = tern(rng, (M, K)), tern(rng, (K, N))
        Av = bufA[:M * lda].view(M, lda)[:, :K]
        Bv = bufB[:K * ldb].view(K, ldb)[:, :N]
        Av.copy_(torch.from_numpy(A).to(dev))
        Bv.copy_(torch.from_numpy(B).to(dev))
        C = torch.empty((M, N), dtype=torch.float16, device=dev)
        g.gemm_f16(Av, Bv, None, C, "none")
        assert np.array_equal(C.cpu().numpy(), oracle_mod.gemm(A, B, None, "none")), (M, N, K, lda, ldb)
