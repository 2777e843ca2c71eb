"""Pins for the CPU oracle: each check ties it to something other than itself.

* fp16 conversion: every one of the 65 536 bit patterns against numpy's
  float16 decoding, round trips, numpy's float64->float16 rounding on random
  and exactly-halfway values, and hand-worked IEEE-754 binary16 cases.
* GELU: textbook standard-normal CDF values (tests/golden), a numerical
  integral of the normal density (independent of erf), the odd-part identity
  GELU(x) - GELU(-x) = x, and the large-|x| limits.
* GEMM: closed forms (identity, permutation, rank-1, zero K tail, small
  integers where every step is exact), numpy's fp64 matmul, and a brute-force
  pure-Python triple loop on tiny shapes.
* Planted mistakes (a transposed operand, a dropped bias) must fail the
  closed forms.
"""
import math
import os

import numpy as np
import pytest

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- fp16 conversion

def test_half_to_double_exhaustive(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint16)
    got = oracle_mod.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signs of zeros and infinities
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_half_round_trip_identity(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    keep = ~np.isnan(vals)
    back = oracle_mod.double_to_half(vals[keep])
    assert np.array_equal(back, bits[keep])


def test_double_to_half_matches_numpy_random(oracle_mod):
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(200_000) * 10.0 ** rng.integers(-9, 6, 200_000),
        rng.uniform(-70000, 70000, 50_000),
        rng.uniform(-1e-6, 1e-6, 50_000),           # subnormal range
    ])
    got = oracle_mod.double_to_half(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_double_to_half_exact_halfway_points(oracle_mod):
    # midpoints between consecutive finite fp16 values must tie to even
    bits = np.arange(0, 0x7bff, dtype=np.uint16)            # positive finite, < max
    lo = bits.view(np.float16).astype(np.float64)
    hi = (bits + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2.0                                     # exact in double
    got = oracle_mod.double_to_half(mid)
    even = np.where(bits % 2 == 0, bits, bits + 1).astype(np.uint16)
    assert np.array_equal(got, even)
    assert np.array_equal(oracle_mod.double_to_half(-mid), even | np.uint16(0x8000))
    # and numpy agrees
    assert np.array_equal(got, mid.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("x, expect", [
    (1.0 + 2.0 ** -11, 0x3C00),          # tie -> even (1.0)
    (1.0 + 3 * 2.0 ** -11, 0x3C02),      # tie -> even (1 + 2^-9)
    (65504.0, 0x7BFF),                   # max finite
    (65519.999, 0x7BFF),
    (65520.0, 0x7C00),                   # tie at the top rounds to infinity
    (-1e6, 0xFC00),
    (2.0 ** -24, 0x0001),                # smallest subnormal
    (2.0 ** -25, 0x0000),                # tie between 0 and 2^-24 -> even (0)
    (3 * 2.0 ** -26, 0x0001),            # 0.75 quantum -> 1 quantum
    (2.0 ** -14, 0x0400),                # smallest normal
    (2.0 ** -14 - 2.0 ** -25, 0x0400),   # tie between 0x03ff and 0x0400 -> even
    (-0.0, 0x8000),
    (float("inf"), 0x7C00),
])
def test_double_to_half_hand_cases(oracle_mod, x, expect):
    assert int(oracle_mod.double_to_half(np.array([x]))[0]) == expect


def test_nan_maps_to_nan(oracle_mod):
    h = int(oracle_mod.double_to_half(np.array([float("nan")]))[0])
    assert (h & 0x7C00) == 0x7C00 and (h & 0x03FF) != 0


# ---------------------------------------------------------------- epilogues

def _golden_phi():
    rows = []
    with open(os.path.join(GOLDEN, "normal_cdf_table.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                x, p = line.split()
                rows.append((float(x), float(p)))
    return rows


def test_gelu_textbook_phi_values(oracle_mod):
    for x, phi in _golden_phi():
        assert oracle_mod.epilogue_scalar(x, "bias_gelu_erf") == pytest.approx(x * phi, abs=1e-13)


def _simpson(f, a, b, n):
    h = (b - a) / n
    s = 0.0
    for i in range(n + 1):
        w = 1 if i in (0, n) else (4 if i % 2 else 2)
        s += w * f(a + i * h)
    return s * h / 3.0


def _phi_by_simpson(x, n=40000):
    # Phi(x) from the normal density phi(t) = exp(-t^2/2)/sqrt(2 pi) alone:
    # x >= 0: 1/2 + integral_0^x phi; x < 0: integral_{x-30}^x phi (no cancellation)
    phi = lambda t: math.exp(-0.5 * t * t) / math.sqrt(2.0 * math.pi)
    if x >= 0:
        return 0.5 + _simpson(phi, 0.0, x, n)
    return _simpson(phi, x - 30.0, x, 4 * n)


@pytest.mark.parametrize("x", [-5.0, -2.7, -1.3, -0.4, 0.1, 0.77, 1.5, 3.3, 6.0])
def test_gelu_against_normal_density_integral(oracle_mod, x):
    assert oracle_mod.epilogue_scalar(x, "bias_gelu_erf") == pytest.approx(
        x * _phi_by_simpson(x), rel=1e-11, abs=1e-14)


def test_gelu_identities(oracle_mod):
    g = lambda v: oracle_mod.epilogue_scalar(v, "bias_gelu_erf")
    assert g(0.0) == 0.0
    for x in np.linspace(-8, 8, 161):
        assert g(x) - g(-x) == pytest.approx(x, abs=1e-14)
    # GELU(x) -> x above ~6 and -> 0 below ~-6, exactly once rounded to fp16
    xs = np.array([6.0, 7.5, 12.0, 100.0])
    ys = np.array([g(v) for v in xs])
    assert np.array_equal(oracle_mod.double_to_half(ys), xs.astype(np.float16).view(np.uint16))
    assert abs(g(-9.0)) < 1e-17


def test_relu_and_identity_epilogues(oracle_mod):
    for x in (-3.5, -1e-30, 0.0, 2.25, 1e6):
        assert oracle_mod.epilogue_scalar(x, "bias_relu") == max(x, 0.0)
        assert oracle_mod.epilogue_scalar(x, "bias") == x
        assert oracle_mod.epilogue_scalar(x, "none") == x
    assert math.isnan(oracle_mod.epilogue_scalar(float("nan"), "bias_relu"))


def test_sigmoid_closed_forms(oracle_mod):
    sg = lambda v: oracle_mod.epilogue_scalar(v, "bias_sigmoid")
    assert sg(0.0) == 0.5
    assert sg(math.log(3.0)) == pytest.approx(0.75, abs=1e-15)       # 1 / (1 + 1/3)
    assert sg(-math.log(4.0)) == pytest.approx(0.2, abs=1e-15)       # 1 / (1 + 4)
    for x in np.linspace(-20, 20, 81):
        assert sg(x) + sg(-x) == pytest.approx(1.0, abs=1e-15)
    assert sg(-800.0) == 0.0 and sg(800.0) == 1.0


def test_gelu_tanh_against_exact_gelu(oracle_mod):
    # the tanh form approximates x Phi(x) to a few 1e-4 everywhere; a dropped cubic
    # term or a wrong scale is off by > 1e-2 near |x| = 2
    gt = lambda v: oracle_mod.epilogue_scalar(v, "bias_gelu_tanh")
    ge = lambda v: oracle_mod.epilogue_scalar(v, "bias_gelu_erf")
    assert gt(0.0) == 0.0
    xs = np.linspace(-8, 8, 321)
    assert max(abs(gt(x) - ge(x)) for x in xs) < 1e-3
    for x in xs:
        assert gt(x) - gt(-x) == pytest.approx(x, abs=1e-13)     # tanh odd
    assert abs(gt(8.0) - 8.0) < 1e-12 and abs(gt(-8.0)) < 1e-12


# ---------------------------------------------------------------- GEMM closed forms

def _rand16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def test_identity_B(oracle_mod):
    rng = np.random.default_rng(1)
    M, K = 37, 40
    A = _rand16(rng, (M, K), 3.0)
    eye = np.eye(K, dtype=np.float16)
    bias = _rand16(rng, (K,))
    assert np.array_equal(oracle_mod.gemm(A, eye, None, "none").view(np.uint16), A.view(np.uint16))
    ref = (A.astype(np.float64) + bias.astype(np.float64)).astype(np.float16)
    assert np.array_equal(oracle_mod.gemm(A, eye, bias, "bias").view(np.uint16), ref.view(np.uint16))


def test_permutation_B(oracle_mod):
    rng = np.random.default_rng(2)
    M, K = 19, 33
    A = _rand16(rng, (M, K))
    perm = rng.permutation(K)
    P = np.zeros((K, K), np.float16)
    P[perm, np.arange(K)] = 1.0           # C[i, j] = A[i, perm[j]]
    C = oracle_mod.gemm(A, P, None, "none")
    assert np.array_equal(C.view(np.uint16), A[:, perm].view(np.uint16))


def test_rank1(oracle_mod):
    rng = np.random.default_rng(3)
    M, N, K = 21, 45, 17
    u, v = _rand16(rng, M), _rand16(rng, N)
    A = np.zeros((M, K), np.float16)
    B = np.zeros((K, N), np.float16)
    A[:, 0] = u
    B[0, :] = v
    ref = np.outer(u.astype(np.float64), v.astype(np.float64)).astype(np.float16)  # products exact
    assert np.array_equal(oracle_mod.gemm(A, B, None, "none").view(np.uint16), ref.view(np.uint16))


def test_zero_k_tail(oracle_mod):
    rng = np.random.default_rng(4)
    M, N, K = 13, 29, 24
    A, B, bias = _rand16(rng, (M, K)), _rand16(rng, (K, N)), _rand16(rng, N)
    A2 = np.concatenate([A, np.zeros((M, 9), np.float16)], axis=1)
    B2 = np.concatenate([B, np.zeros((9, N), np.float16)], axis=0)
    for epi in ("none", "bias", "bias_relu", "bias_gelu_erf"):
        b = None if epi == "none" else bias
        assert np.array_equal(oracle_mod.gemm(A, B, b, epi).view(np.uint16),
                              oracle_mod.gemm(A2, B2, b, epi).view(np.uint16))


@pytest.mark.parametrize("epi", ["none", "bias", "bias_relu"])
def test_integer_inputs_exact(oracle_mod, epi):
    rng = np.random.default_rng(5)
    M, N, K = 40, 56, 300
    Ai = rng.integers(-2, 3, (M, K))
    Bi = rng.integers(-2, 3, (K, N))
    bi = rng.integers(-8, 9, N)
    ref = Ai @ Bi + (0 if epi == "none" else bi)
    if epi == "bias_relu":
        ref = np.maximum(ref, 0)
    assert np.abs(ref).max() <= 2048
    C = oracle_mod.gemm(Ai.astype(np.float16), Bi.astype(np.float16),
                        None if epi == "none" else bi.astype(np.float16), epi)
    assert np.array_equal(C.astype(np.int64), ref)


def test_matches_numpy_fp64_matmul(oracle_mod):
    rng = np.random.default_rng(6)
    M, N, K = 64, 96, 200
    A, B, bias = _rand16(rng, (M, K)), _rand16(rng, (K, N)), _rand16(rng, N)
    _, y = oracle_mod.gemm(A, B, bias, "bias", want_f64=True)
    ref = A.astype(np.float64) @ B.astype(np.float64) + bias.astype(np.float64)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def _brute(A, B, bias, epi):
    M, K = A.shape
    N = B.shape[1]
    out = np.zeros((M, N), np.float64)
    for i in range(M):
        for j in range(N):
            s = 0.0
            for k in range(K):
                s += float(A[i, k]) * float(B[k, j])
            x = s + (float(bias[j]) if epi != "none" else 0.0)
            if epi == "bias_relu":
                x = max(x, 0.0)
            elif epi == "bias_gelu_erf":
                x = 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0)))
            elif epi == "bias_sigmoid":
                x = 1.0 / (1.0 + math.exp(-x))
            elif epi == "bias_gelu_tanh":
                x = 0.5 * x * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))
            out[i, j] = x
    return out.astype(np.float16)


def test_brute_force_tiny(oracle_mod):
    rng = np.random.default_rng(8)
    epis = ["none", "bias", "bias_relu", "bias_gelu_erf", "bias_sigmoid", "bias_gelu_tanh"]
    n = 0
    for M in (1, 2, 3, 5, 8):
        for N in (1, 2, 4, 7):
            for K in (1, 3, 6, 8):
                epi = epis[n % len(epis)]
                n += 1
                A, B, bias = _rand16(rng, (M, K)), _rand16(rng, (K, N)), _rand16(rng, N)
                b = None if epi == "none" else bias
                got = oracle_mod.gemm(A, B, b, epi)
                assert np.array_equal(got.view(np.uint16), _brute(A, B, bias, epi).view(np.uint16)), (M, N, K, epi)


def test_rows_and_elems_agree(oracle_mod):
    rng = np.random.default_rng(9)
    M, N, K = 50, 70, 130
    A, B, bias = _rand16(rng, (M, K)), _rand16(rng, (K, N)), _rand16(rng, N)
    full = oracle_mod.gemm(A, B, bias, "bias_gelu_erf")
    ii, jj = workloads.sample_coords(11, M, N, 300)
    el = oracle_mod.gemm_elems(A, B, bias, "bias_gelu_erf", ii, jj)
    assert np.array_equal(el.view(np.uint16), full[ii, jj].view(np.uint16))
    rows = np.array([0, 17, 49])
    assert np.array_equal(oracle_mod.gemm_rows(A, B, bias, "bias_gelu_erf", rows).view(np.uint16),
                          full[rows].view(np.uint16))


def test_k_zero_is_epilogue_of_bias(oracle_mod):
    bias = np.array([-2.0, -0.5, 0.0, 1.0, 3.0], np.float16)
    A = np.zeros((3, 0), np.float16)
    B = np.zeros((0, 5), np.float16)
    C = oracle_mod.gemm(A, B, bias, "bias_relu")
    assert np.array_equal(C, np.tile(np.maximum(bias, 0), (3, 1)))
    assert np.all(oracle_mod.gemm(A, B, None, "none") == 0)


def test_bad_arguments_rejected(oracle_mod):
    A = np.zeros((2, 3), np.float16)
    B = np.zeros((3, 4), np.float16)
    with pytest.raises(ValueError):
        oracle_mod.gemm(A, B, None, "bias")            # bias missing
    with pytest.raises(ValueError):
        oracle_mod.gemm_rows(A, B, None, "none", [5])   # row out of range


# ---------------------------------------------------------------- grouped GEMM

def _block_diag(blocks, rows_cols):
    R = sum(r for r, _ in rows_cols)
    C = sum(c for _, c in rows_cols)
    out = np.zeros((R, C), np.float16)
    r0 = c0 = 0
    for b, (r, c) in zip(blocks, rows_cols):
        out[r0:r0 + r, c0:c0 + c] = b
        r0, c0 = r0 + r, c0 + c
    return out


@pytest.mark.parametrize("epi", ["none", "bias_relu", "bias_gelu_erf"])
def test_grouped_is_the_block_diagonal_product(oracle_mod, epi):
    # stacking the problems block-diagonally turns them into ONE GEMM whose
    # diagonal blocks are the problems' products and whose off-diagonal
    # blocks are epilogue(0 + bias): an independent construction of what a
    # grouped call must return (a mixed-up operand or bias fails it)
    rng = np.random.default_rng(40)
    shapes = [(5, 7, 3), (1, 9, 12), (8, 2, 5), (4, 6, 1)]
    probs = [(_rand16(rng, (M, K)), _rand16(rng, (K, N)), _rand16(rng, N)) for M, N, K in shapes]
    got = oracle_mod.gemm_grouped(probs, epi)
    Abig = _block_diag([a for a, _, _ in probs], [(M, K) for M, N, K in shapes])
    Bbig = _block_diag([b for _, b, _ in probs], [(K, N) for M, N, K in shapes])
    bias_big = np.concatenate([c for _, _, c in probs])
    big = oracle_mod.gemm(Abig, Bbig, bias_big if epi != "none" else None, epi)
    r0 = c0 = 0
    for (M, N, K), g in zip(shapes, got):
        assert np.array_equal(g.view(np.uint16), big[r0:r0 + M, c0:c0 + N].view(np.uint16))
        r0, c0 = r0 + M, c0 + N


def test_grouped_empty_and_k_zero_problems(oracle_mod):
    rng = np.random.default_rng(41)
    bias = _rand16(rng, 4)
    out = oracle_mod.gemm_grouped([(np.zeros((0, 3), np.float16), np.zeros((3, 4), np.float16), bias),
                                   (np.zeros((2, 0), np.float16), np.zeros((0, 4), np.float16), bias)], "bias_relu")
    assert out[0].shape == (0, 4)
    assert np.array_equal(out[1].view(np.uint16), np.broadcast_to(np.maximum(bias, 0), (2, 4)).view(np.uint16))


# ---------------------------------------------------------------- attention

def _qkv(rng, B, H, S, D, scale=1.0):
    return tuple((rng.standard_normal((B, H, S, D)) * scale).astype(np.float16) for _ in range(3))


def test_attention_single_key_is_v(oracle_mod):
    # one admissible key: its weight is exp(0)/exp(0) = 1 exactly
    rng = np.random.default_rng(70)
    Q, K, V = _qkv(rng, 2, 3, 1, 16)
    assert np.array_equal(oracle_mod.attention(Q, K, V, False).view(np.uint16), V.view(np.uint16))
    Q, K, V = _qkv(rng, 1, 2, 9, 16)
    O = oracle_mod.attention(Q, K, V, True)             # causal: query 0 sees key 0 only
    assert np.array_equal(O[:, :, 0].view(np.uint16), V[:, :, 0].view(np.uint16))


@pytest.mark.parametrize("causal", [False, True])
def test_attention_equal_scores_average_v(oracle_mod, causal):
    # Q = 0: every score is 0, the weights 1/n, O the mean of the admissible V rows
    rng = np.random.default_rng(71)
    B, H, S, D = 1, 2, 11, 8
    _, K, V = _qkv(rng, B, H, S, D)
    Q = np.zeros_like(V)
    _, f64 = oracle_mod.attention(Q, K, V, causal, want_f64=True)
    v = V.astype(np.float64)
    ref = np.cumsum(v, axis=2) / np.arange(1, S + 1)[None, None, :, None] if causal else \
        np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
    assert np.allclose(f64, ref, rtol=1e-13, atol=1e-15)


def test_attention_constant_v_is_returned(oracle_mod):
    rng = np.random.default_rng(72)
    Q, K, _ = _qkv(rng, 2, 2, 13, 32, 2.0)
    c = rng.standard_normal(32).astype(np.float16)
    V = np.broadcast_to(c, Q.shape).astype(np.float16)
    for causal in (False, True):
        O = oracle_mod.attention(Q, K, V, causal)
        assert np.array_equal(O.view(np.uint16), V.view(np.uint16))


def test_attention_one_hot_keys_closed_form(oracle_mod):
    # K rows = unit vectors e_j, Q row i = alpha e_{pi(i)}, scale 1: query i
    # scores alpha on key pi(i) and 0 elsewhere, so
    # O[i] = (e^alpha V[pi(i)] + sum_{j != pi(i)} V[j]) / (e^alpha + S - 1)
    rng = np.random.default_rng(73)
    S, D, alpha = 6, 8, 3.0
    K = np.zeros((1, 1, S, D), np.float16)
    K[0, 0, np.arange(S), np.arange(S)] = 1.0
    perm = rng.permutation(S)
    Q = np.zeros((1, 1, S, D), np.float16)
    Q[0, 0, np.arange(S), perm] = alpha
    V = rng.standard_normal((1, 1, S, D)).astype(np.float16)
    _, f64 = oracle_mod.attention(Q, K, V, False, scale=1.0, want_f64=True)
    v = V[0, 0].astype(np.float64)
    e = math.exp(alpha)
    for i in range(S):
        ref = (e * v[perm[i]] + (v.sum(axis=0) - v[perm[i]])) / (e + S - 1)
        assert np.allclose(f64[0, 0, i], ref, rtol=1e-13, atol=1e-15)


def test_attention_brute_force_tiny(oracle_mod):
    # plain Python: exp of the raw scores (no max subtraction), then the ratio
    rng = np.random.default_rng(74)
    for B, H, S, D, causal in [(1, 1, 3, 4, False), (2, 1, 5, 3, True), (1, 2, 4, 8, False), (1, 1, 7, 2, True)]:
        Q, K, V = _qkv(rng, B, H, S, D, 0.5)
        scale = 0.7
        _, f64 = oracle_mod.attention(Q, K, V, causal, scale=scale, want_f64=True)
        q, k, v = (x.astype(np.float64).tolist() for x in (Q, K, V))
        for b in range(B):
            for h in range(H):
                for i in range(S):
                    keys = range(i + 1) if causal else range(S)
                    w = [math.exp(scale * sum(q[b][h][i][d] * k[b][h][j][d] for d in range(D))) for j in keys]
                    tot = sum(w)
                    for d in range(D):
                        ref = sum(w[n] * v[b][h][j][d] for n, j in enumerate(keys)) / tot
                        assert abs(f64[b, h, i, d] - ref) <= 1e-13 * max(1.0, abs(ref))


def test_attention_causal_row_is_the_prefix_problem(oracle_mod):
    # causal query i sees exactly the non-causal problem over the first i + 1 rows
    rng = np.random.default_rng(75)
    Q, K, V = _qkv(rng, 1, 2, 10, 16)
    Oc = oracle_mod.attention(Q, K, V, True)
    for i in (0, 3, 9):
        On = oracle_mod.attention(Q[:, :, :i + 1], K[:, :, :i + 1], V[:, :, :i + 1], False)
        assert np.array_equal(Oc[:, :, i].view(np.uint16), On[:, :, i].view(np.uint16))


def test_attention_key_permutation_and_scale_invariances(oracle_mod):
    rng = np.random.default_rng(76)
    Q, K, V = _qkv(rng, 1, 2, 12, 16)
    _, f0 = oracle_mod.attention(Q, K, V, False, want_f64=True)
    perm = rng.permutation(12)
    _, f1 = oracle_mod.attention(Q, K[:, :, perm], V[:, :, perm], False, want_f64=True)
    assert np.allclose(f0, f1, rtol=1e-13, atol=1e-15)       # keys and values moved together
    Q2 = (Q.astype(np.float32) * 2).astype(np.float16)        # exact doubling
    a = oracle_mod.attention(Q, K, V, True, scale=0.5)
    b = oracle_mod.attention(Q2, K, V, True, scale=0.25)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_attention_planted_missing_mask_is_caught(oracle_mod):
    # without the causal mask, query 0 averages over every key and is no longer V[0]
    rng = np.random.default_rng(77)
    Q, K, V = _qkv(rng, 1, 1, 8, 16)
    O = oracle_mod.attention(Q, K, V, False)
    assert not np.array_equal(O[:, :, 0].view(np.uint16), V[:, :, 0].view(np.uint16))


# ---------------------------------------------------------------- planted mistakes

def test_planted_transpose_is_caught(oracle_mod):
    # feeding B^T (a transposed operand) must break the permutation closed form
    rng = np.random.default_rng(10)
    K = 24
    A = _rand16(rng, (6, K))
    perm = rng.permutation(K)
    P = np.zeros((K, K), np.float16)
    P[perm, np.arange(K)] = 1.0
    C = oracle_mod.gemm(A, np.ascontiguousarray(P.T), None, "none")
    assert not np.array_equal(C.view(np.uint16), A[:, perm].view(np.uint16))


def test_planted_dropped_bias_is_caught(oracle_mod):
    rng = np.random.default_rng(11)
    A = _rand16(rng, (4, 8))
    eye = np.eye(8, dtype=np.float16)
    bias = np.full(8, 0.5, np.float16)
    ref = (A.astype(np.float64) + 0.5).astype(np.float16)
    dropped = oracle_mod.gemm(A, eye, bias, "none")      # "none" ignores the bias
    assert not np.array_equal(dropped.view(np.uint16), ref.view(np.uint16))


# ---------------------------------------------------------------- input generator

def test_generator_is_deterministic_and_shaped():
    w = workloads.WORKLOADS["gemm256"]
    A1, B1, b1 = w.make()
    A2, B2, b2 = w.make()
    assert A1.dtype == np.float16 and A1.shape == (256, 256) and b1.shape == (256,)
    assert np.array_equal(A1.view(np.uint16), A2.view(np.uint16))
    assert np.array_equal(B1.view(np.uint16), B2.view(np.uint16))
    assert not np.array_equal(A1.view(np.uint16), B1.view(np.uint16))
    # N(0,1)/16 statistics
    a = A1.astype(np.float64).ravel()
    assert abs(a.mean()) < 0.002 and abs(a.std() - 1 / 16) < 0.002
    u = workloads.fp16_tensor((100000,), "uniform", 1.0, 4, 2).astype(np.float64)
    assert u.min() >= -1 and u.max() <= 1 and abs(u.mean()) < 0.01 and abs(u.var() - 1 / 3) < 0.01


def test_generator_is_counter_based():
    # any slice of a stream equals the same slice of a longer draw
    full = workloads.raw_draws(3, 1, 0, 1000)
    assert np.array_equal(full[500:600], workloads.raw_draws(3, 1, 500, 100))
    # first splitmix64 output for state 0 is the published value
    z = workloads._mix(np.array([0x9E3779B97F4A7C15], dtype=np.uint64))[0]
    assert int(z) == 0xE220A8397B1DCDAF
