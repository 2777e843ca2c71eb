"""gemm_f16_noalloc: the entry point for callers that must not allocate device memory.

Such callers are plugins running inside a framework that owns the device
memory, serving loops that cannot afford the device-wide synchronisation of
cudaMalloc/cudaFree, and deployments that forbid allocation after start-up.
The variant keeps its scratch (operand repacks, and the split-K partial sums
and counters of short-A problems) in a fixed 32 MiB buffer compiled into the
library.  These tests check its plans on the host, and on the GPU its results
against the fp64 oracle and against gemm_f16, on consecutive calls of
different shapes that reuse the buffer: a repack of both operands, a short-A
problem that repacks B and splits K inside the buffer, one whose partial sums
do not fit beside the repack (so it runs unsplit), and a repack larger than
the buffer, which is refused cleanly.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest

from oracle.compare import parity

GOOD = 0x10000
LIMIT = 32 << 20


def _lib():
    import __graft_entry__
    __graft_entry__.build()
    import dense_fp16_tensor_tma_gb300 as g
    return g


def test_noalloc_rejects_bad_arguments_without_a_device():
    g = _lib()
    assert g.gemm_f16_noalloc_ptr(GOOD, GOOD, GOOD, GOOD, -1, 8, 8, 0, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_f16_noalloc_ptr(GOOD, GOOD, 0, GOOD, 8, 8, 8, 3, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_f16_noalloc_ptr(GOOD + 1, GOOD, GOOD, GOOD, 8, 8, 8, 0, 0) == g.GEMM_ERR_MISALIGNED
    assert "32 MiB" in g.gemm_f16_status_string(g.GEMM_ERR_SCRATCH_LIMIT)


def test_noalloc_empty_problem_runs_the_device_set_up():
    # valid arguments with nothing to compute: the call sets up the device (and
    # with it the fixed buffer) and enqueues nothing, so without a device it
    # reports the failed CUDA call instead of succeeding silently
    g = _lib()
    import torch
    st = g.gemm_f16_noalloc_ptr(GOOD, GOOD, GOOD, GOOD, 0, 8, 8, 0, 0)
    if torch.cuda.is_available():
        assert st in (g.GEMM_OK, g.GEMM_ERR_UNSUPPORTED_DEVICE)
    else:
        assert st == g.GEMM_ERR_CUDA


def test_noalloc_plans_fit_the_fixed_buffer():
    g = _lib()
    # short A, B repacked (N % 8 != 0) and K split four ways: repack 16.8 MB plus
    # 1 MiB of partial sums fit, so the no-alloc plan is gemm_f16's
    p = g.gemm_f16_plan(16, 4090, 2048, "bias_gelu_erf", noalloc=True)
    assert p == g.gemm_f16_plan(16, 4090, 2048, "bias_gelu_erf")
    assert p["path"] == 3 and p["pack_b"] == 1 and p["splits"] == 4 and p["scratch"] <= LIMIT
    # repack 32.8 MB (31.25 MiB) plus 4 MiB of partial sums do not fit: unsplit
    full = g.gemm_f16_plan(64, 8190, 2000, "bias")
    assert full["splits"] == 2 and full["scratch"] > LIMIT
    p = g.gemm_f16_plan(64, 8190, 2000, "bias", noalloc=True)
    assert p["path"] == 3 and p["pack_b"] == 1 and p["splits"] == 1 and p["scratch"] <= LIMIT
    # no repack at all: no scratch, no size limit
    assert g.gemm_f16_plan(8192, 8192, 8192, "bias_gelu_erf", noalloc=True)["scratch"] == 0
    # a repack alone larger than the buffer
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_plan(8192, 64, 2049, "none", noalloc=True)
    assert e.value.status == g.GEMM_ERR_SCRATCH_LIMIT


CASES = [
    # M, N, K, epilogue, seed: what the fixed buffer holds
    (300, 1003, 203, "bias_gelu_erf", 1),   # A repack (K % 8) and B repack (N % 8)
    (16, 4090, 2048, "bias_gelu_erf", 2),   # B repack + split-K partials and counters
    (16, 4090, 2048, "bias_gelu_erf", 3),   # the same plan again on other inputs
    (64, 8190, 2000, "bias", 4),            # B repack only: the split is dropped
    (517, 777, 129, "bias_relu", 5),        # both repacks again, a smaller problem
]


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_gemm_f16_on_consecutive_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp16_tensor_tma_gb300 as g
    import oracle

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream().cuda_stream
    # set-up at "start-up": an empty problem, then real calls
    assert g.gemm_f16_noalloc_ptr(GOOD, GOOD, GOOD, GOOD, 0, 8, 8, 0, stream) == g.GEMM_OK
    for M, N, K, epi, seed in CASES:
        rng = np.random.default_rng(seed)
        A = (rng.standard_normal((M, K)) * 0.5).astype(np.float16)
        B = (rng.standard_normal((K, N)) * 0.5).astype(np.float16)
        bias = rng.standard_normal(N).astype(np.float16)
        tA, tB, tb = (torch.from_numpy(x).to(dev) for x in (A, B, bias))
        plan = g.gemm_f16_plan(M, N, K, epi, a_addr=tA.data_ptr(), b_addr=tB.data_ptr(),
                               c_addr=tA.data_ptr(), bias_addr=tb.data_ptr(), noalloc=True)
        assert plan["scratch"] > 0 and plan["scratch"] <= LIMIT, plan
        C_ref = torch.empty((M, N), dtype=torch.float16, device=dev)
        C_new = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
        assert g.gemm_f16_ptr(tA.data_ptr(), tB.data_ptr(), tb.data_ptr(), C_ref.data_ptr(),
                              M, N, K, epi, stream) == g.GEMM_OK
        assert g.gemm_f16_noalloc_ptr(tA.data_ptr(), tB.data_ptr(), tb.data_ptr(), C_new.data_ptr(),
                                      M, N, K, epi, stream) == g.GEMM_OK
        st, word = g.gemm_f16_debug_status()
        assert st == g.GEMM_OK, hex(word)
        got = C_new.cpu().numpy()
        res = parity(got, oracle.gemm(A, B, bias, epi))
        assert res["ok"], (M, N, K, plan, res)
        res = parity(got, C_ref.cpu().numpy())
        assert res["ok"], (M, N, K, plan, "vs gemm_f16", res)

    # a repack bigger than the fixed buffer is refused and enqueues nothing
    big_M, big_K = 8192, 2049            # A repack: 8192 * 2056 * 2 bytes > 32 MiB
    A = torch.zeros((big_M, big_K), dtype=torch.float16, device=dev)
    B = torch.zeros((big_K, 64), dtype=torch.float16, device=dev)
    C = torch.full((big_M, 64), 3.0, dtype=torch.float16, device=dev)
    assert g.gemm_f16_noalloc_ptr(A.data_ptr(), B.data_ptr(), 0, C.data_ptr(), big_M, 64, big_K,
                                  "none", stream) == g.GEMM_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert bool(torch.all(C == 3.0))
