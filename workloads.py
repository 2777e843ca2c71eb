"""Seeded synthetic inputs for the fused fp16 GEMM workloads.

This module holds no GEMM or epilogue arithmetic.  It only draws the inputs
(A, B, bias, sampled output coordinates) that the CUDA path and the CPU oracle
both consume, so the two sides see bit-identical operands.

Generator (counter based, so any element can be drawn independently):

* splitmix64 finaliser ``mix(z)``: z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
  z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31   (all mod 2^64).
* stream key for tensor t of a workload with seed s:
  ``key = mix((s << 8) + t + 1)`` with t = 0 (A), 1 (B), 2 (bias),
  3 (sampled coordinates).
* draw i of a stream: ``x_i = mix(key + (i+1) * 0x9E3779B97F4A7C15)``.
* uniform in [0,1): ``u_i = (x_i >> 11) * 2^-53``.
* U(-1,1): ``2 u_i - 1``.
* N(0,1) by Box-Muller on draw pairs (2p, 2p+1):
  ``r = sqrt(-2 ln(1 - u_2p))``, ``z_2p = r cos(2 pi u_2p+1)``,
  ``z_2p+1 = r sin(2 pi u_2p+1)``.
* element e of a row-major tensor takes draw e; the scaled double value is
  rounded to fp16 (round to nearest even, numpy's conversion).

The five workloads are the fused-GEMM configurations: shapes, distributions
and seeds as listed in ``WORKLOADS``.  ``ATTN_WORKLOADS`` are the attention
forward configurations: Q, K, V drawn from streams t = 4, 5, 6 of their seed,
N(0,1) rounded to fp16; query rows to check drawn from stream 7.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

T_A, T_B, T_BIAS, T_SAMPLES = 0, 1, 2, 3
T_Q, T_K, T_V, T_ROWS = 4, 5, 6, 7


def _mix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _C1
    z = z ^ (z >> np.uint64(27))
    z = z * _C2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor: int) -> np.uint64:
    z = np.array([((seed << 8) + tensor + 1) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return _mix(z)[0]


def raw_draws(seed: int, tensor: int, start: int, count: int) -> np.ndarray:
    """Draws x_start .. x_{start+count-1} of one stream (uint64)."""
    key = stream_key(seed, tensor)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + idx * _GAMMA)


def uniform01(seed: int, tensor: int, start: int, count: int) -> np.ndarray:
    return (raw_draws(seed, tensor, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _normal_chunk(seed, tensor, start, count):
    # start is even: draws come in Box-Muller pairs
    n_pairs = (count + 1) // 2
    u = uniform01(seed, tensor, start, 2 * n_pairs)
    r = np.sqrt(-2.0 * np.log1p(-u[0::2]))
    th = 2.0 * math.pi * u[1::2]
    z = np.empty(2 * n_pairs, np.float64)
    z[0::2] = r * np.cos(th)
    z[1::2] = r * np.sin(th)
    return z[:count]


def fp16_tensor(shape, dist: str, scale: float, seed: int, tensor: int) -> np.ndarray:
    """Row-major fp16 tensor of `shape`, element e = round_fp16(scale * draw_e)."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, np.float16)
    for lo in range(0, n, _CHUNK):
        cnt = min(_CHUNK, n - lo)
        if dist == "normal":
            v = _normal_chunk(seed, tensor, lo, cnt)
        elif dist == "uniform":
            v = 2.0 * uniform01(seed, tensor, lo, cnt) - 1.0
        else:
            raise ValueError(dist)
        out[lo:lo + cnt] = (v * scale).astype(np.float16)
    return out.reshape(shape)


def sample_coords(seed: int, M: int, N: int, count: int):
    """`count` seeded (i, j) output coordinates (duplicates allowed)."""
    x = raw_draws(seed, T_SAMPLES, 0, 2 * count)
    ii = (x[0::2] % np.uint64(M)).astype(np.int64)
    jj = (x[1::2] % np.uint64(N)).astype(np.int64)
    return ii, jj


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    ab_dist: str          # "normal" or "uniform"
    ab_scale: str         # "1", "1/16", "1/sqrtK"
    bias_dist: Optional[str]
    epilogues: tuple
    seed: int
    check: str            # "full" or "sampled"

    def scale(self) -> float:
        return {"1": 1.0, "1/16": 1.0 / 16.0, "1/sqrtK": 1.0 / math.sqrt(self.K)}[self.ab_scale]

    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def alg_bytes(self) -> float:
        b = 2.0 * (self.M * self.K + self.K * self.N + self.M * self.N)
        return b + (2.0 * self.N if self.bias_dist else 0.0)

    def make(self, with_bias: bool = True):
        """(A, B, bias|None) as numpy fp16 arrays."""
        A = fp16_tensor((self.M, self.K), self.ab_dist, self.scale(), self.seed, T_A)
        B = fp16_tensor((self.K, self.N), self.ab_dist, self.scale(), self.seed, T_B)
        bias = None
        if with_bias and self.bias_dist:
            bias = fp16_tensor((self.N,), self.bias_dist, 1.0, self.seed, T_BIAS)
        return A, B, bias


WORKLOADS = {
    "gemm256": Workload("gemm256", 256, 256, 256, "normal", "1/16", "normal",
                        ("none", "bias_gelu_erf"), 0, "full"),
    "gemm1024": Workload("gemm1024", 1024, 1024, 1024, "normal", "1", None,
                         ("none",), 1, "full"),
    "fused4096": Workload("fused4096", 4096, 4096, 4096, "normal", "1/sqrtK", "uniform",
                          ("bias_gelu_erf",), 2, "full"),
    "fused8192": Workload("fused8192", 8192, 8192, 8192, "normal", "1/sqrtK", "uniform",
                          ("bias_gelu_erf",), 3, "sampled"),
    "ragged3001x5003x1000": Workload("ragged3001x5003x1000", 3001, 5003, 1000, "uniform", "1",
                                     "normal", ("bias_relu",), 4, "full"),
    "skinny16x8192x8192": Workload("skinny16x8192x8192", 16, 8192, 8192, "uniform", "1", None,
                                   ("none",), 4, "full"),
}

# the 8192^3 check: 4096 seeded elements plus full rows 0 and M-1
SAMPLED_ELEMS = 4096


@dataclass(frozen=True)
class AttnWorkload:
    """Attention forward O = softmax(Q K^T / sqrt(D)) V on (B, H, S, D) fp16
    tensors; Q, K, V ~ N(0, 1).  The pages give the operation and its FLOP
    model but no sizes: the shapes are those of a long-context prefill (S 4096,
    head dimension 128) and small and ragged cases for full checks."""
    name: str
    B: int
    H: int
    S: int
    D: int
    causal: bool
    seed: int
    check: str            # "full" or "sampled"

    def flops(self) -> float:
        return 4.0 * self.B * self.H * self.S * self.S * self.D * (0.5 if self.causal else 1.0)

    def alg_bytes(self) -> float:
        return 4.0 * 2.0 * self.B * self.H * self.S * self.D   # Q, K, V read once, O written once

    def make(self):
        shape = (self.B, self.H, self.S, self.D)
        return tuple(fp16_tensor(shape, "normal", 1.0, self.seed, t) for t in (T_Q, T_K, T_V))

    def sample_rows(self, count: int) -> np.ndarray:
        """`count` seeded flattened query rows (b * H + h) * S + i, plus the
        first and last row of the first and last head."""
        total = self.B * self.H * self.S
        x = raw_draws(self.seed, T_ROWS, 0, count)
        extra = [0, self.S - 1, total - self.S, total - 1]
        return np.unique(np.concatenate([(x % np.uint64(total)).astype(np.int64), np.array(extra, np.int64)]))


ATTN_WORKLOADS = {
    "attn_small": AttnWorkload("attn_small", 1, 2, 256, 64, False, 10, "full"),
    "attn_small_causal": AttnWorkload("attn_small_causal", 1, 2, 256, 128, True, 11, "full"),
    "attn_ragged_causal": AttnWorkload("attn_ragged_causal", 2, 3, 1000, 128, True, 12, "full"),
    "attn_prefill": AttnWorkload("attn_prefill", 4, 32, 4096, 128, False, 13, "sampled"),
    "attn_prefill_causal": AttnWorkload("attn_prefill_causal", 4, 32, 4096, 128, True, 14, "sampled"),
    "attn_prefill_d64": AttnWorkload("attn_prefill_d64", 4, 32, 4096, 64, False, 15, "sampled"),
    "attn_prefill_d64_causal": AttnWorkload("attn_prefill_d64_causal", 4, 32, 4096, 64, True, 16, "sampled"),
    # an odd number of query tiles per head (11): the one-tile kernel, causal pairs
    "attn_odd_causal": AttnWorkload("attn_odd_causal", 8, 16, 1300, 128, True, 17, "sampled"),
}
