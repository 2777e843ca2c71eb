"""The error paths of the product kernels, driven on the GPU without a fault.

A bounded wait runs out inside a real kernel launch because the test hook
(gemm_f16_debug_inject / attn_f16_debug_inject) makes the producer skip one
stage's loads: nothing is ever in flight for that stage, the MMA thread's
wait for it gives up after 2 ms, every role leaves through its abort path and
tensor memory is freed.  The kernel reports the timeout in its status word;
the next call on the same context must match the oracle again.  A failed
tensor-map encoding must return GEMM_ERR_CUDA and enqueue nothing.  The
CTA-pair kernels are not driven this way: their abort path is covered by the
barrier-protocol model in test_gemm_protocol_cpu.py.
"""
import numpy as np
import pytest

from oracle.compare import parity

pytestmark = pytest.mark.gpu

WAIT_US = 2000
CUDA_ERROR_INVALID_VALUE = 1


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp16_tensor_tma_gb300 as g
    import oracle
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    yield torch, dev, g, oracle
    g.gemm_f16_debug_inject(g.GEMM_F16_FAULT_NONE)
    g.attn_f16_debug_inject(g.GEMM_F16_FAULT_NONE)


def _problem(rng, M, N, K):
    A = (rng.standard_normal((M, K)) * 0.25).astype(np.float16)
    B = (rng.standard_normal((K, N)) * 0.25).astype(np.float16)
    bias = rng.standard_normal(N).astype(np.float16)
    return A, B, bias


def _gemm(env, A, B, bias, epi, C=None):
    torch, dev, g, _ = env
    tA, tB, tb = (torch.from_numpy(x).to(dev) for x in (A, B, bias))
    if C is None:
        C = torch.full((A.shape[0], B.shape[1]), 7.0, dtype=torch.float16, device=dev)
    st = g.gemm_f16_ptr(tA.data_ptr(), tB.data_ptr(), tb.data_ptr(), C.data_ptr(), A.shape[0], B.shape[1],
                        A.shape[1], epi, torch.cuda.current_stream().cuda_stream)
    return st, C


# Status word (ptx.cuh): bit 31, role << 8, barrier.  With every wait of the
# faulty launch limited to 2 ms, whichever stuck wait started first records
# itself: the epilogue's wait for the accumulator (from the kernel's start),
# the MMA thread's for the skipped stage, or the producer's final wait for it.
GEMM_TIMEOUT_WORDS = {0x80000000 | (3 << 8) | 3, 0x80000000 | (2 << 8) | 1, 0x80000000 | (5 << 8) | 1}


@pytest.mark.parametrize("M,N,K,path,tile_m", [(128, 64, 256, 2, 128), (300, 200, 256, 2, 128),
                                               (16, 128, 256, 3, 16), (40, 300, 192, 3, 64)])
def test_skipped_loads_time_out_and_the_context_survives(env, M, N, K, path, tile_m):
    torch, dev, g, oracle = env
    plan = g.gemm_f16_plan(M, N, K, "bias_gelu_erf")
    assert (plan["path"], plan["tile_m"], plan["splits"]) == (path, tile_m, 1), plan
    rng = np.random.default_rng(M + N + K)
    A, B, bias = _problem(rng, M, N, K)
    assert g.gemm_f16_debug_inject(g.GEMM_F16_FAULT_SKIP_LOADS, WAIT_US) == g.GEMM_OK
    st, _ = _gemm(env, A, B, bias, "bias_gelu_erf")
    assert st == g.GEMM_OK                       # enqueued; the failure shows on the device
    st, word = g.gemm_f16_debug_status()
    assert st == g.GEMM_ERR_TIMEOUT and word in GEMM_TIMEOUT_WORDS, hex(word)
    assert g.gemm_f16_debug_status()[0] == g.GEMM_OK          # read and cleared
    # the next call on the same context, with the same buffers' shapes, is right again
    st, C = _gemm(env, A, B, bias, "bias_gelu_erf")
    assert st == g.GEMM_OK
    st, word = g.gemm_f16_debug_status()
    assert st == g.GEMM_OK, hex(word)
    res = parity(C.cpu().numpy(), oracle.gemm(A, B, bias, "bias_gelu_erf"))
    assert res["ok"], res


def test_skip_fault_is_not_taken_by_a_cta_pair_launch(env):
    torch, dev, g, oracle = env
    M = N = 2560                 # 100 pair tiles: the CTA-pair kernel
    K = 256
    assert g.gemm_f16_plan(M, N, K, "bias")["tile_m"] == 256
    rng = np.random.default_rng(5)
    A, B, bias = _problem(rng, M, N, K)
    assert g.gemm_f16_debug_inject(g.GEMM_F16_FAULT_SKIP_LOADS, WAIT_US) == g.GEMM_OK
    try:
        st, C = _gemm(env, A, B, bias, "bias")
        assert st == g.GEMM_OK
        st, word = g.gemm_f16_debug_status()
        assert st == g.GEMM_OK, hex(word)
        rows = np.array([0, 1, 777, M - 1])
        res = parity(C.cpu().numpy()[rows], oracle.gemm_rows(A, B, bias, "bias", rows))
        assert res["ok"], res
        # still armed: the next single-CTA launch takes it
        A2, B2, bias2 = _problem(rng, 128, 64, 256)
        assert _gemm(env, A2, B2, bias2, "bias")[0] == g.GEMM_OK
        assert g.gemm_f16_debug_status()[0] == g.GEMM_ERR_TIMEOUT
    finally:
        g.gemm_f16_debug_inject(g.GEMM_F16_FAULT_NONE)


def test_failed_encoding_returns_cuda_error_and_enqueues_nothing(env):
    torch, dev, g, oracle = env
    rng = np.random.default_rng(9)
    # dense (no repack), then one that repacks both operands (through the no-alloc entry point)
    for M, N, K in [(256, 256, 128), (300, 1003, 203)]:
        A, B, bias = _problem(rng, M, N, K)
        tA, tB, tb = (torch.from_numpy(x).to(dev) for x in (A, B, bias))
        C = torch.full((M, N), 7.0, dtype=torch.float16, device=dev)
        stream = torch.cuda.current_stream().cuda_stream
        for call in (g.gemm_f16_ptr, g.gemm_f16_noalloc_ptr):
            assert g.gemm_f16_debug_inject(g.GEMM_F16_FAULT_ENCODE) == g.GEMM_OK
            st = call(tA.data_ptr(), tB.data_ptr(), tb.data_ptr(), C.data_ptr(), M, N, K, "bias_relu", stream)
            assert st == g.GEMM_ERR_CUDA
            assert g.lib.gemm_f16_last_cuda_error() == CUDA_ERROR_INVALID_VALUE
            torch.cuda.synchronize()
            assert bool(torch.all(C == 7.0)), "a failed call wrote C"
            assert g.gemm_f16_debug_status()[0] == g.GEMM_OK
        st, C = _gemm(env, A, B, bias, "bias_relu", C)
        assert st == g.GEMM_OK and g.gemm_f16_debug_status()[0] == g.GEMM_OK
        res = parity(C.cpu().numpy(), oracle.gemm(A, B, bias, "bias_relu"))
        assert res["ok"], res


def _attn_inputs(torch, dev, shape, seed):
    rng = np.random.default_rng(seed)
    Q, K, V = (rng.standard_normal(shape).astype(np.float16) for _ in range(3))
    return (Q, K, V), [torch.from_numpy(x).to(dev) for x in (Q, K, V)]


# D = 64, the two-tile kernel with P buffers of its own: (1,1,256,64) with
# one-tile units only; (4,40,256,64) two-tile units then one-tile units
# (152 + 16); (1,76,2048,64) causal pairs (16 tiles per head, 304 steps).
# D = 128, the two-tile kernel with P over the scores: the same two non-causal
# cases and (1,76,1024,128) causal pairs (8 tiles per head, 152 steps).
# (1,2,384,128) causal: the one-tile kernel (3 tiles per head).
@pytest.mark.parametrize("shape,causal", [((1, 1, 256, 64), False), ((4, 40, 256, 64), False),
                                          ((1, 76, 2048, 64), True), ((1, 1, 256, 128), False),
                                          ((4, 40, 256, 128), False), ((1, 76, 1024, 128), True),
                                          ((1, 2, 384, 128), True)])
def test_attention_skipped_key_block_times_out_and_the_context_survives(env, shape, causal):
    torch, dev, g, oracle = env
    (Q, K, V), (tq, tk, tv) = _attn_inputs(torch, dev, shape, 3)
    O = torch.zeros_like(tq)
    assert g.attn_f16_debug_inject(g.GEMM_F16_FAULT_SKIP_LOADS, WAIT_US) == g.GEMM_OK
    g.attn_f16_fwd(tq, tk, tv, O, causal)
    st, word = g.attn_f16_debug_status()
    # the first stuck wait to run out records itself (the MMA thread's for the
    # skipped key block, the softmax's for its scores, a producer's)
    assert st == g.GEMM_ERR_TIMEOUT and word & 0x80000000, hex(word)
    assert g.attn_f16_debug_status()[0] == g.GEMM_OK
    g.attn_f16_fwd(tq, tk, tv, O, causal)
    st, word = g.attn_f16_debug_status()
    assert st == g.GEMM_OK, hex(word)
    D = shape[-1]
    res = parity(O.cpu().numpy().reshape(-1, D), oracle.attention(Q, K, V, causal).reshape(-1, D))
    assert res["ok"], res


def test_attention_failed_encoding_enqueues_nothing(env):
    torch, dev, g, oracle = env
    (Q, K, V), (tq, tk, tv) = _attn_inputs(torch, dev, (1, 2, 256, 128), 4)
    O = torch.full_like(tq, 7.0)
    assert g.attn_f16_debug_inject(g.GEMM_F16_FAULT_ENCODE) == g.GEMM_OK
    st = g.attn_f16_fwd_ptr(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), O.data_ptr(), 1, 2, 256, 128, False, 0.0,
                            torch.cuda.current_stream().cuda_stream)
    assert st == g.GEMM_ERR_CUDA and g.lib.attn_f16_last_cuda_error() == CUDA_ERROR_INVALID_VALUE
    torch.cuda.synchronize()
    assert bool(torch.all(O == 7.0))
    assert g.attn_f16_debug_status()[0] == g.GEMM_OK
