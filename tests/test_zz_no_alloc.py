"""gemm_f16_noalloc: the entry point for callers that must not allocate device memory.

Such callers are plugins running inside a framework that owns the device
memory, serving loops that cannot afford the device-wide synchronisation of
cudaMalloc/cudaFree, and deployments that forbid allocation after start-up.
The variant keeps any operand repack in a fixed 32 MiB buffer compiled into
the library, so these tests check that its results agree with gemm_f16 on
problems that do need the repack, on consecutive calls that reuse the
buffer, and that a repack larger than the buffer is refused cleanly.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest

from oracle.compare import parity

GOOD = 0x10000


def test_noalloc_rejects_bad_arguments_without_a_device():
    import __graft_entry__
    __graft_entry__.build()
    import dense_fp16_tensor_tma_gb300 as g
    assert g.gemm_f16_noalloc_ptr(GOOD, GOOD, GOOD, GOOD, -1, 8, 8, 0, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_f16_noalloc_ptr(GOOD, GOOD, 0, GOOD, 8, 8, 8, 3, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_f16_noalloc_ptr(GOOD + 1, GOOD, GOOD, GOOD, 8, 8, 8, 0, 0) == g.GEMM_ERR_MISALIGNED
    assert g.gemm_f16_noalloc_ptr(GOOD, GOOD, GOOD, GOOD, 0, 8, 8, 0, 0) == g.GEMM_OK
    assert "32 MiB" in g.gemm_f16_status_string(g.GEMM_ERR_SCRATCH_LIMIT)


@pytest.mark.gpu
def test_noalloc_matches_gemm_f16_on_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp16_tensor_tma_gb300 as g

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream().cuda_stream
    # both problems need a repack: N % 8 != 0 (B) and K % 8 != 0 (A)
    cases = [(300, 1003, 203, "bias_gelu_erf", 1), (517, 777, 129, "bias_relu", 2)]
    for M, N, K, epi, seed in cases:
        rng = np.random.default_rng(seed)
        A = torch.from_numpy((rng.standard_normal((M, K)) * 0.5).astype(np.float16)).to(dev)
        B = torch.from_numpy((rng.standard_normal((K, N)) * 0.5).astype(np.float16)).to(dev)
        bias = torch.from_numpy(rng.standard_normal(N).astype(np.float16)).to(dev)
        plan = g.gemm_f16_plan(M, N, K, epi, a_addr=A.data_ptr(), b_addr=B.data_ptr(),
                               c_addr=A.data_ptr(), bias_addr=bias.data_ptr())
        assert plan["pack_a"] == 1 and plan["pack_b"] == 1
        C_ref = torch.empty((M, N), dtype=torch.float16, device=dev)
        C_new = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
        assert g.gemm_f16_ptr(A.data_ptr(), B.data_ptr(), bias.data_ptr(), C_ref.data_ptr(),
                              M, N, K, epi, stream) == g.GEMM_OK
        assert g.gemm_f16_noalloc_ptr(A.data_ptr(), B.data_ptr(), bias.data_ptr(), C_new.data_ptr(),
                                      M, N, K, epi, stream) == g.GEMM_OK
        st, word = g.gemm_f16_debug_status()
        assert st == g.GEMM_OK, hex(word)
        res = parity(C_new.cpu().numpy(), C_ref.cpu().numpy())
        assert res["ok"], res

    # a repack bigger than the fixed buffer is refused and enqueues nothing
    big_M, big_K = 8192, 2049            # A repack: 8192 * 2056 * 2 bytes > 32 MiB
    A = torch.zeros((big_M, big_K), dtype=torch.float16, device=dev)
    B = torch.zeros((big_K, 64), dtype=torch.float16, device=dev)
    C = torch.full((big_M, 64), 3.0, dtype=torch.float16, device=dev)
    assert g.gemm_f16_noalloc_ptr(A.data_ptr(), B.data_ptr(), 0, C.data_ptr(), big_M, 64, big_K,
                                  "none", stream) == g.GEMM_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert bool(torch.all(C == 3.0))
