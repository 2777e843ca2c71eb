"""GPU parity of the attention forward (attn_f16_fwd) against the fp64 oracle.

Bar: the oracle.compare tolerance (relative Frobenius error <= 1e-3, per
element |err| <= 1e-2 (1 + |ref|)); bit-exact where the method is exact (one
admissible key, constant V).  Inputs: workloads.ATTN_WORKLOADS (seeded) and
seeded numpy draws for the special cases.
"""
import numpy as np
import pytest

import workloads
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


def run_attn(g, torch_dev, Q, K, V, causal, scale=None):
    torch, dev = torch_dev
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x)).to(dev) for x in (Q, K, V))
    O = torch.full(Q.shape, float("nan"), dtype=torch.float16, device=dev)
    g.attn_f16_fwd(tq, tk, tv, O, causal, scale)
    st, word = g.attn_f16_debug_status()
    assert st == 0, f"device status {st} word {word:#x}"
    return O.cpu().numpy()


def qkv(rng, shape, scale=1.0):
    return tuple((rng.standard_normal(shape) * scale).astype(np.float16) for _ in range(3))


def check(got, ref, what):
    res = parity(got.reshape(-1, got.shape[-1]), ref.reshape(-1, ref.shape[-1]))
    assert res["ok"], f"{what}: {res}"
    return res


# ---------------------------------------------------------------- the workloads

@pytest.mark.parametrize("name", ["attn_small", "attn_small_causal", "attn_ragged_causal"])
def test_attention_workloads_full(g, torch_dev, oracle_mod, name):
    w = workloads.ATTN_WORKLOADS[name]
    Q, K, V = w.make()
    got = run_attn(g, torch_dev, Q, K, V, w.causal)
    check(got, oracle_mod.attention(Q, K, V, w.causal), name)


@pytest.mark.parametrize("name", ["attn_prefill", "attn_prefill_causal", "attn_prefill_d64",
                                  "attn_prefill_d64_causal", "attn_odd_causal"])
def test_attention_prefill_sampled_rows(g, torch_dev, oracle_mod, name):
    w = workloads.ATTN_WORKLOADS[name]
    Q, K, V = w.make()
    got = run_attn(g, torch_dev, Q, K, V, w.causal)
    rows = w.sample_rows(384)
    ref = oracle_mod.attention_rows(Q, K, V, w.causal, 1.0 / np.sqrt(w.D), rows)
    check(got.reshape(-1, w.D)[rows], ref, name)


# ---------------------------------------------------------------- many tiles per CTA
# More query tiles than SMs, so every CTA walks several tiles.  Non-causal
# problems run two tiles per CTA (S 2100: 17 tiles per head, the last one
# alone; S 1300: 11 tiles, alone at D = 64, one tile per CTA at D = 128);
# causal ones too with a multiple of 4 tiles per head, at least 8 (adjacent
# pairs, two pairs of a head per step; S 1500: 12 tiles, S 1000: 8, the last
# partial); otherwise one tile per CTA, causal tiles paired nq - 1 - k with k
# (S 1300: 11 tiles, the middle one alone); ragged S makes every head's last
# tile partial.

@pytest.mark.parametrize("B,H,S,D,causal", [(4, 32, 1300, 128, True), (4, 32, 1300, 64, True),
                                            (8, 16, 1000, 128, False), (8, 24, 700, 64, True),
                                            (4, 32, 4096, 64, True), (4, 32, 4096, 64, False),
                                            (16, 16, 1024, 128, False), (4, 32, 1500, 64, True),
                                            (2, 76, 1000, 128, True), (4, 32, 1300, 128, False),
                                            (4, 32, 1300, 64, False), (4, 16, 2100, 128, False)])
def test_attention_many_tiles_per_cta_sampled_rows(g, torch_dev, oracle_mod, B, H, S, D, causal):
    rng = np.random.default_rng(S + D + 7 * causal)
    Q, K, V = qkv(rng, (B, H, S, D))
    got = run_attn(g, torch_dev, Q, K, V, causal)
    # O starts as NaN: every row of every query tile is written (no unit skipped)
    assert np.isfinite(got).all()
    total = B * H * S
    # rows of the first, a middle and the last head, each head's first and last
    # query tile, and a seeded sample
    heads = [0, (B * H) // 2, B * H - 1]
    rows = [h * S + i for h in heads for i in (0, 1, 127, 128, S - 129, S - 128, S - 2, S - 1)]
    rows = np.unique(np.concatenate([np.array(rows, np.int64), rng.integers(0, total, 256)]))
    ref = oracle_mod.attention_rows(Q, K, V, causal, 1.0 / np.sqrt(D), rows)
    check(got.reshape(-1, D)[rows], ref, f"B{B} H{H} S{S} D{D} causal={causal}")


# ---------------------------------------------------------------- shapes

@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 7, 127, 128, 129, 256, 300, 513, 1000])
def test_attention_shape_sweep(g, torch_dev, oracle_mod, D, causal, S):
    rng = np.random.default_rng(S * 3 + D + causal)
    Q, K, V = qkv(rng, (2, 3, S, D))
    got = run_attn(g, torch_dev, Q, K, V, causal)
    check(got, oracle_mod.attention(Q, K, V, causal), f"S={S} D={D} causal={causal}")


# ---------------------------------------------------------------- exact special cases

@pytest.mark.parametrize("D", [64, 128])
def test_attention_single_key_is_exactly_v(g, torch_dev, D):
    # one key: p = 2^0 = 1 exactly, the sum is 1, O = V
    rng = np.random.default_rng(80 + D)
    Q, K, V = qkv(rng, (3, 2, 1, D))
    got = run_attn(g, torch_dev, Q, K, V, False)
    assert np.array_equal(got.view(np.uint16), V.view(np.uint16))
    # causal: query 0 of every head sees key 0 only
    Q, K, V = qkv(rng, (1, 2, 300, D))
    got = run_attn(g, torch_dev, Q, K, V, True)
    assert np.array_equal(got[:, :, 0].view(np.uint16), V[:, :, 0].view(np.uint16))


@pytest.mark.parametrize("causal", [False, True])
def test_attention_constant_v_is_exact(g, torch_dev, causal):
    # sum_j p_j c / sum_j p_j = c up to a few fp32 ulps: rounds back to c
    rng = np.random.default_rng(81)
    Q, K, _ = qkv(rng, (2, 2, 700, 128), 2.0)
    c = rng.standard_normal(128).astype(np.float16)
    V = np.broadcast_to(c, Q.shape).astype(np.float16)
    got = run_attn(g, torch_dev, Q, K, V, causal)
    assert np.array_equal(got.view(np.uint16), V.view(np.uint16))


def test_attention_equal_scores_average(g, torch_dev, oracle_mod):
    rng = np.random.default_rng(82)
    _, K, V = qkv(rng, (1, 2, 500, 64))
    Q = np.zeros_like(K)
    for causal in (False, True):
        check(run_attn(g, torch_dev, Q, K, V, causal), oracle_mod.attention(Q, K, V, causal), f"Q=0 {causal}")


# ---------------------------------------------------------------- the online maximum

@pytest.mark.parametrize("D", [64, 128])
def test_attention_running_max_raised_every_block(g, torch_dev, oracle_mod, D):
    # scores rise along the keys for even query rows and fall for odd ones:
    # the even rows raise their running maximum (and rescale O) in every
    # block, the odd rows never do, within the same warps
    rng = np.random.default_rng(83)
    S = 640
    sign = np.where(np.arange(S) % 2 == 0, 1.0, -1.0)
    Q = np.broadcast_to((sign[:, None] * np.ones(D))[None, None], (1, 2, S, D)).astype(np.float16)
    ramp = (np.arange(S) * 0.1)[:, None] * np.ones(D)
    K = np.broadcast_to(ramp[None, None], (1, 2, S, D)).astype(np.float16)
    V = rng.standard_normal((1, 2, S, D)).astype(np.float16)
    scale = 1.0 / D   # scores +-0.1 j: 12.8 (18 in log2 units) more per block of 128 keys
    for causal in (False, True):
        got = run_attn(g, torch_dev, Q, K, V, causal, scale)
        check(got, oracle_mod.attention(Q, K, V, causal, scale=scale), f"ramp causal={causal}")


# Score levels (log2 units) of successive key blocks for the even query rows:
# after block 0 sets the running maximum m = 0, block 1's P sum 128 * 2^6 and
# block 2's 128 * 2^7.75 exceed 2^8 with no raise due (the exact maximum is
# taken and the first P kept), block 3 raises m to 9, blocks 4, 5 and 9 again
# sum above 2^8 without a raise, block 6 raises to 20, block 7's P is tiny,
# block 8's sum is exactly 2^8 (no second look) and block 10 raises to 30.
# The odd rows see the negated scores and never leave the first pass, in the
# same warps.
SUM_CHECK_LEVELS = [0.0, 6.0, 7.75, 9.0, 14.0, 12.0, 20.0, 1.0, 21.0, 27.0, 30.0]


@pytest.mark.parametrize("B,H,S,D,causal,kernel", [
    (1, 2, 1024, 128, False, "attn_f16_fwd2_kernel"),
    (1, 76, 1024, 128, True, "attn_f16_fwd2_kernel"),
    (1, 3, 1300, 128, False, "attn_f16_fwd4_kernel"),
    (1, 3, 1300, 128, True, "attn_f16_fwd4_kernel"),
    (1, 2, 1300, 64, True, "attn_f16_fwd4_kernel"),
    (1, 2, 1300, 64, False, "attn_f16_fwd3_kernel"),
])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_attention_block_sum_check(g, torch_dev, oracle_mod, B, H, S, D, causal, kernel, sign):
    # Q = +-1 and every key of block b equal to SUM_CHECK_LEVELS[b]: with scale
    # ln 2 / D the log2-unit score of a key is +-its level.  A negative scale
    # (Q negated with it) takes the kernels' minimum-score branch.
    assert g.attn_f16_plan(B, H, S, D, causal)["kernel_name"] == kernel
    rng = np.random.default_rng(86)
    row_sign = np.where(np.arange(S) % 2 == 0, 1.0, -1.0) * sign
    Q = np.broadcast_to((row_sign[:, None] * np.ones(D))[None, None], (B, H, S, D)).astype(np.float16)
    level = np.array(SUM_CHECK_LEVELS)[np.arange(S) // 128]
    K = np.broadcast_to((level[:, None] * np.ones(D))[None, None], (B, H, S, D)).astype(np.float16)
    V = rng.standard_normal((B, H, S, D)).astype(np.float16)
    scale = sign * np.log(2.0) / D
    got = run_attn(g, torch_dev, Q, K, V, causal, scale).reshape(B * H * S, D)
    assert np.isfinite(got).all()
    heads = B * H
    rows = np.unique(np.concatenate([h * S + np.arange(S) for h in sorted({0, heads - 1})] +
                                    [rng.integers(0, heads * S, 256)]))
    ref = oracle_mod.attention_rows(Q, K, V, causal, scale, rows)
    check(got[rows], ref, f"levels {B}x{H}x{S}x{D} causal={causal} sign={sign}")


@pytest.mark.parametrize("scale", [0.05, -0.1, 0.3, -1.0])
def test_attention_explicit_scale(g, torch_dev, oracle_mod, scale):
    rng = np.random.default_rng(84)
    Q, K, V = qkv(rng, (2, 2, 384, 64))
    got = run_attn(g, torch_dev, Q, K, V, True, scale)
    check(got, oracle_mod.attention(Q, K, V, True, scale=scale), f"scale {scale}")


def test_attention_deterministic_and_pdl_chain(g, torch_dev, oracle_mod):
    # attention then a GEMM that reads its output, back to back on one stream,
    # twice: bit-identical results, and the GEMM sees the finished O
    torch, dev = torch_dev
    rng = np.random.default_rng(85)
    B, H, S, D = 1, 4, 512, 64
    Q, K, V = qkv(rng, (B, H, S, D))
    W = (rng.standard_normal((D, 96)) * 0.1).astype(np.float16)
    tq, tk, tv, tw = (torch.from_numpy(x).to(dev) for x in (Q, K, V, W))
    outs = []
    for _ in range(2):
        O = torch.empty((B, H, S, D), dtype=torch.float16, device=dev)
        C = torch.empty((B * H * S, 96), dtype=torch.float16, device=dev)
        g.attn_f16_fwd(tq, tk, tv, O, True)
        g.gemm_f16(O.view(B * H * S, D), tw, None, C, "none")
        torch.cuda.synchronize()
        outs.append((O.cpu().numpy(), C.cpu().numpy()))
    assert np.array_equal(outs[0][0].view(np.uint16), outs[1][0].view(np.uint16))
    assert np.array_equal(outs[0][1].view(np.uint16), outs[1][1].view(np.uint16))
    O_ref = oracle_mod.attention(Q, K, V, True)
    check(outs[0][0], O_ref, "attention")
    # the composition, all on the oracle's side
    res = parity(outs[0][1], oracle_mod.gemm(O_ref.reshape(B * H * S, D), W, None, "none"))
    assert res["ok"], res
    assert g.attn_f16_debug_status()[0] == 0 and g.gemm_f16_debug_status()[0] == 0
