"""Seeded random GEMM problems on the GPU against the fp64 oracle.

The host plan picks, per call, among the swap-AB kernel (M <= 64, with split-K
over CTAs), 128-row tiles of width 64, 128 or 256 (with K split over a
cluster), and the CTA pair with its half-tile tail; operands it cannot hand to
TMA (a pitch that is not a multiple of 8 elements) are first repacked, and C
rows that are not 16-byte aligned go out through the narrow-store path.  Forty
problems drawn over shape regimes, K tails, operand layouts (row-major with a
padded pitch, or stored transposed), C pitches and the six epilogues exercise
the combinations a fixed list misses.  Bar: the oracle.compare tolerance on
sampled elements (2048 seeded positions and the first and last row and column).
Inputs: A ~ U(-1, 1), B ~ N(0, 1) / sqrt(K), bias ~ N(0, 1), seeded.
RANDOM_GEMM_PROBLEMS and RANDOM_SEED in the environment draw a longer or
different sample (a soak run); the defaults are 40 problems from seed 7.
"""
import os

import numpy as np
import pytest

from oracle.compare import parity

pytestmark = pytest.mark.gpu

EPILOGUES = ["none", "bias", "bias_relu", "bias_gelu_erf", "bias_sigmoid", "bias_gelu_tanh"]


def problems(count=int(os.environ.get("RANDOM_GEMM_PROBLEMS", "40")),
             seed=int(os.environ.get("RANDOM_SEED", "7"))):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        regime = int(rng.integers(0, 4))
        if regime == 0:      # skinny: the swap-AB kernel
            M = int(rng.integers(1, 65))
            N = int(rng.integers(64, 6000))
            K = int(rng.integers(16, 6000))
        elif regime == 1:    # small and mid: single-CTA tiles, split-K clusters
            M = int(rng.integers(65, 1500))
            N = int(rng.integers(16, 1500))
            K = int(rng.integers(1, 5000))
        elif regime == 2:    # large: the CTA pair
            M = int(rng.integers(1500, 5000))
            N = int(rng.integers(1500, 5000))
            K = int(rng.integers(64, 2500))
        else:                # tall or wide
            M = int(rng.integers(64, 8000)) if rng.integers(0, 2) else int(rng.integers(64, 400))
            N = int(rng.integers(64, 400)) if M > 1000 else int(rng.integers(1000, 8000))
            K = int(rng.integers(32, 3000))
        out.append(dict(M=M, N=N, K=K, epi=EPILOGUES[int(rng.integers(0, len(EPILOGUES)))],
                        ta=bool(rng.integers(0, 4) == 0), tb=bool(rng.integers(0, 3) == 0),
                        pad_a=int(rng.choice([0, 0, 8, 3])), pad_b=int(rng.choice([0, 0, 8, 5])),
                        pad_c=int(rng.choice([0, 0, 8, 1]))))
    return out


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp16_tensor_tma_gb300 as g
    return torch, torch.device("cuda:0"), g


def stored(torch, dev, X, transposed, pad):
    """A device view of the fp16 matrix X (rows x cols): row-major with pitch
    cols + pad, or stored transposed (X^T row-major, pitch rows + pad) and
    viewed back as X."""
    rows, cols = X.shape
    if transposed:
        buf = torch.zeros((cols, rows + pad), dtype=torch.float16, device=dev)
        buf[:, :rows] = torch.from_numpy(np.ascontiguousarray(X.T)).to(dev)
        return buf[:, :rows].t()
    buf = torch.zeros((rows, cols + pad), dtype=torch.float16, device=dev)
    buf[:, :cols] = torch.from_numpy(X).to(dev)
    return buf[:, :cols]


@pytest.mark.parametrize("case", list(enumerate(problems())),
                         ids=lambda c: "M{M}N{N}K{K}_{epi}_{ta:d}{tb:d}_{pad_a}{pad_b}{pad_c}".format(**c[1]))
def test_random_gemm_problem(env, oracle_mod, case):
    torch, dev, g = env
    i, pb = case
    M, N, K, epi = pb["M"], pb["N"], pb["K"], pb["epi"]
    rng = np.random.default_rng(500 + i)
    A = rng.uniform(-1.0, 1.0, (M, K)).astype(np.float16)
    B = (rng.standard_normal((K, N)) / np.sqrt(max(K, 1))).astype(np.float16)
    bias = rng.standard_normal(N).astype(np.float16) if epi != "none" else None
    tA = stored(torch, dev, A, pb["ta"], pb["pad_a"])
    tB = stored(torch, dev, B, pb["tb"], pb["pad_b"])
    cbuf = torch.full((M, N + pb["pad_c"]), float("nan"), dtype=torch.float16, device=dev)
    tC = cbuf[:, :N]
    tbias = torch.from_numpy(bias).to(dev) if bias is not None else None
    g.gemm_f16(tA, tB, tbias, tC, epi)
    st, word = g.gemm_f16_debug_status()
    assert st == 0, f"device status {st} word {word:#x}"
    got = tC.cpu().numpy()
    if pb["pad_c"]:
        # the padding between C's rows is never written
        assert np.isnan(cbuf[:, N:].cpu().numpy()).all()
    ii = np.concatenate([rng.integers(0, M, 2048), [0, M - 1, 0, M - 1]]).astype(np.int64)
    jj = np.concatenate([rng.integers(0, N, 2048), [0, N - 1, N - 1, 0]]).astype(np.int64)
    ref = oracle_mod.gemm_elems(A, B, bias, epi, ii, jj)
    res = parity(got[ii, jj], ref)
    assert res["ok"], f"{pb}: {res}"
