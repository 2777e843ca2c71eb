"""The pipelined end-to-end steps of bench.py (copies in, kernel, copies out on
three streams over two device buffer sets) produce every step's own result:
each step gets different inputs from pinned host memory and writes its result
to its own host buffer, and every result is checked against the oracle (a race
between the buffer sets would show as a result of the wrong step)."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch, torch.device("cuda:0")


def test_pipelined_gemm_steps_each_get_their_own_result(torch_dev, oracle_mod):
    torch, dev = torch_dev
    import bench
    import dense_fp16_tensor_tma_gb300 as g
    M, N, K, steps = 384, 512, 320, 7
    total = 3 + steps                      # the helper's warm-up steps come first
    rng = np.random.default_rng(91)
    # integer entries: exact in fp32 and fp16, so every result must match bit for bit
    As = [rng.integers(-2, 3, (M, K)).astype(np.float16) for _ in range(total)]
    B = rng.integers(-2, 3, (K, N)).astype(np.float16)
    bias = rng.integers(-8, 9, N).astype(np.float16)
    hA = [torch.from_numpy(a).pin_memory() for a in As]
    hC = [torch.empty((M, N), dtype=torch.float16).pin_memory() for _ in range(total)]
    dA = [torch.empty((M, K), dtype=torch.float16, device=dev) for _ in range(2)]
    dC = [torch.empty((M, N), dtype=torch.float16, device=dev) for _ in range(2)]
    dB = torch.from_numpy(B).to(dev)
    db = torch.from_numpy(bias).to(dev)
    n_in, n_out = [0], [0]

    def copy_in(b):
        dA[b].copy_(hA[n_in[0]], non_blocking=True)
        n_in[0] += 1

    def compute(b):
        st = g.gemm_f16_ex_ptr(dA[b].data_ptr(), K, dB.data_ptr(), N, db.data_ptr(), dC[b].data_ptr(), N, M, N, K,
                               g.EPILOGUES["bias_relu"], 0, torch.cuda.current_stream().cuda_stream)
        assert st == 0

    def copy_out(b):
        hC[n_out[0]].copy_(dC[b], non_blocking=True)
        n_out[0] += 1

    comp = torch.cuda.Stream(device=dev)
    bench.pipelined_e2e(torch, dev, 1, steps, comp, copy_in, compute, copy_out)
    torch.cuda.synchronize()
    assert n_in[0] == n_out[0] == total
    assert g.gemm_f16_debug_status()[0] == 0
    for i in range(total):
        ref = oracle_mod.gemm(As[i], B, bias, "bias_relu")
        assert np.array_equal(hC[i].numpy(), ref), f"step {i}"


def test_pipelined_attention_steps_each_get_their_own_result(torch_dev, oracle_mod):
    torch, dev = torch_dev
    import bench
    from oracle.compare import parity
    import dense_fp16_tensor_tma_gb300 as g
    B, H, S, D, steps = 1, 2, 300, 64, 5
    total = 3 + steps
    rng = np.random.default_rng(92)
    Qs = [rng.standard_normal((B, H, S, D)).astype(np.float16) for _ in range(total)]
    K = rng.standard_normal((B, H, S, D)).astype(np.float16)
    V = rng.standard_normal((B, H, S, D)).astype(np.float16)
    hQ = [torch.from_numpy(q).pin_memory() for q in Qs]
    hO = [torch.empty((B, H, S, D), dtype=torch.float16).pin_memory() for _ in range(total)]
    dQ = [torch.empty((B, H, S, D), dtype=torch.float16, device=dev) for _ in range(2)]
    dO = [torch.empty((B, H, S, D), dtype=torch.float16, device=dev) for _ in range(2)]
    dK, dV = torch.from_numpy(K).to(dev), torch.from_numpy(V).to(dev)
    n_in, n_out = [0], [0]

    def copy_in(b):
        dQ[b].copy_(hQ[n_in[0]], non_blocking=True)
        n_in[0] += 1

    def compute(b):
        st = g.attn_f16_fwd_ptr(dQ[b].data_ptr(), dK.data_ptr(), dV.data_ptr(), dO[b].data_ptr(), B, H, S, D, 1, 0.0,
                                torch.cuda.current_stream().cuda_stream)
        assert st == 0

    def copy_out(b):
        hO[n_out[0]].copy_(dO[b], non_blocking=True)
        n_out[0] += 1

    comp = torch.cuda.Stream(device=dev)
    bench.pipelined_e2e(torch, dev, 1, steps, comp, copy_in, compute, copy_out)
    torch.cuda.synchronize()
    assert n_in[0] == n_out[0] == total
    assert g.attn_f16_debug_status()[0] == 0
    for i in range(total):
        ref = oracle_mod.attention(Qs[i], K, V, True)
        res = parity(hO[i].numpy().reshape(-1, D), ref.reshape(-1, D))
        assert res["ok"], (i, res)
