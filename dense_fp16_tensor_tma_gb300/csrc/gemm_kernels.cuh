// Fused fp16 GEMM kernels for sm_103a:  C = epilogue(A.B + bias).
//
// The method: "writing-tilelang-kernels", Kernel Anatomy / GEMM (Minimal)
// (tile loop over K with global->shared copies of an A tile and a B tile and
// a tensor-core tile product into a float accumulator, then one write-back),
// and "TileLang: Write, Autotune, and Ship Fused Tensor-Core Kernels from
// Python", Why tile-level control matters (bias + activation applied to the
// on-chip accumulator before the single write of C).
//
// GB300 design (not the pages' Ampere/Hopper templates):
//   * persistent CTAs, one per SM, walking output tiles in grouped order so
//     that concurrently running CTAs share A row-panels and B column-panels
//     in L2;
//   * warp 0: TMA producer filling a STAGES-deep ring of (A, B) tiles with
//     128-byte-swizzled boxes; OOB elements of ragged M/N/K tails arrive as
//     zeros;
//   * warp 1: allocates tensor memory and issues tcgen05.mma (M=128, N=BN,
//     K=16) from one thread into one of two TMEM accumulators;
//   * warps 2..9: epilogue (two warps per TMEM lane quarter, each taking half
//     of the columns), reading the accumulator with tcgen05.ld while the MMA
//     warp already fills the other accumulator for the next tile.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace gemm_f16_dev {

enum : int { EPI_NONE = 0, EPI_BIAS = 1, EPI_BIAS_RELU = 2, EPI_BIAS_GELU_ERF = 3, EPI_BIAS_SIGMOID = 4,
             EPI_BIAS_GELU_TANH = 5 };

__device__ unsigned int g_status;  // bounded-wait status word, read by the host

constexpr int kBM = 128;                 // tile rows = MMA M = TMEM lanes
constexpr int kBK = 64;                  // K per stage: one 128-byte swizzle row of fp16
constexpr int kUMMA_K = 16;              // K per tcgen05.mma kind::f16
constexpr int kThreads = 320;            // 10 warps: producer, MMA, 8 epilogue
constexpr int kEpiWarps = 8;             // two per TMEM lane quarter, each half of the columns
constexpr uint32_t kATileBytes = kBM * kBK * 2;  // 16 KiB
constexpr uint32_t kBBoxBytes = 64 * kBK * 2;    // one 64(N) x 64(K) box, 8 KiB
// Per epilogue warp: a 32 x 32 fp16 block, rows padded to 17 words so that
// both the row-wise writes and the column-wise reads are bank-conflict free,
// then the bias of the warp's (up to 128) columns as 64 packed fp16 pairs.
constexpr uint32_t kStageRowWords = 17;
constexpr uint32_t kStageBlockWords = 32 * kStageRowWords;
constexpr uint32_t kStageBiasWords = 64;
constexpr uint32_t kStageWarpBytes = (kStageBlockWords + kStageBiasWords) * 4;
constexpr uint32_t kStageBytes = kEpiWarps * kStageWarpBytes;   // 19 KiB for the eight epilogue warps

template <int BN, int STAGES>
struct SmemPlan {
    static constexpr uint32_t kBTileBytes = BN * kBK * 2;
    static constexpr uint32_t kA = 0;                                   // STAGES A tiles
    static constexpr uint32_t kB = kA + STAGES * kATileBytes;           // STAGES B tiles
    static constexpr uint32_t kStage = kB + STAGES * kBTileBytes;       // epilogue staging (narrow stores)
    static constexpr uint32_t kBars = kStage + kStageBytes;             // mbarriers (8 B each)
    static constexpr uint32_t kNumBars = 2 * STAGES + 2 + 2 + 1;        // full, empty, acc_full, acc_empty, drain
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kEnd = kAbort + 4;
    static constexpr uint32_t kDynamicBytes = kEnd + 1024;             // + alignment slack
    static_assert(kBTileBytes % 1024 == 0 && kATileBytes % 1024 == 0, "swizzle atoms need 1 KiB alignment");
};

struct TileCoord { int m0, n0; };

// Grouped rasterisation: `group_m` consecutive tile-rows are walked column by
// column, so a wave of CTAs covers a compact group_m x (wave/group_m) block.
__device__ __forceinline__ TileCoord tile_coord(int t, int tiles_m, int tiles_n, int group_m, int BN) {
    const int per_group = group_m * tiles_n;
    const int g = t / per_group;
    const int first_m = g * group_m;
    const int rows = min(tiles_m - first_m, group_m);
    const int r = t - g * per_group;
    TileCoord c;
    c.m0 = (first_m + r % rows) * kBM;
    c.n0 = (r / rows) * BN;
    return c;
}

// erfc(z) for z >= 0 by Abramowitz & Stegun, Handbook of Mathematical
// Functions, eq. 7.1.26: erfc(z) = (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5)
// exp(-z^2), t = 1 / (1 + p z), with |error| <= 1.5e-7 over z >= 0 (absolute;
// relative to erfc itself it stays below 8e-4 for z <= 3.1, where GELU's
// negative tail leaves the fp16 normal range).  It costs about half the
// instructions of erff, which matters because the epilogue shares the SM's
// issue slots with the MMA and load warps.
__device__ __forceinline__ float erfc_as_7_1_26(float z) {
    const float t = __fdividef(1.0f, fmaf(0.3275911f, z, 1.0f));
    float q = fmaf(1.061405429f, t, -1.453152027f);
    q = fmaf(q, t, 1.421413741f);
    q = fmaf(q, t, -0.284496736f);
    q = fmaf(q, t, 0.254829592f);
    q *= t;
    return q * __expf(-z * z);
}

// GELU(x) = x Phi(x) = 0.5 x (1 + erf(x / sqrt 2)).  With z = |x| / sqrt 2 and
// c = erfc(z): 1 + erf = 2 - c for x >= 0 and 1 - erf(z) = c for x < 0.  The
// negative tail is thus the product 0.5 x c, with no cancellation: it keeps
// the relative accuracy of c down to the fp16 subnormals.
__device__ __forceinline__ float gelu_erf(float x) {
    const float c = erfc_as_7_1_26(fabsf(x) * 0.70710678118654752440f);
    const float hx = 0.5f * x;
    return hx * (x < 0.0f ? c : 2.0f - c);
}

// 1 / (1 + e^-x): e^-x overflows to +inf for x < -88, giving 0.
__device__ __forceinline__ float sigmoid_f(float x) {
    return __fdividef(1.0f, 1.0f + __expf(-x));
}

// GELU, tanh form: 0.5 x (1 + tanh(u)), u = sqrt(2/pi) (x + 0.044715 x^3),
// with 1 + tanh(u) = 2 / (1 + e^(-2u)): a quotient, never a difference, so
// the negative tail keeps its relative accuracy (e^(-2u) = 0 gives 2,
// e^(-2u) = inf gives 0).
__device__ __forceinline__ float gelu_tanh_f(float x) {
    const float u = 0.7978845608028654f * fmaf(0.044715f * x, x * x, x);
    const float one_plus_t = __fdividef(2.0f, 1.0f + __expf(-2.0f * u));
    return 0.5f * x * one_plus_t;
}

// The activation of epilogue kind ACT (a compile-time constant: no branch).
template <int ACT>
__device__ __forceinline__ float act(float x) {
    if (ACT == EPI_BIAS_RELU) return fmaxf(x, 0.0f);
    if (ACT == EPI_BIAS_GELU_ERF) return gelu_erf(x);
    if (ACT == EPI_BIAS_SIGMOID) return sigmoid_f(x);
    if (ACT == EPI_BIAS_GELU_TANH) return gelu_tanh_f(x);
    return x;
}

__device__ __forceinline__ float apply_act(float x, int epi) {
    switch (epi) {
        case EPI_BIAS_RELU: return act<EPI_BIAS_RELU>(x);
        case EPI_BIAS_GELU_ERF: return act<EPI_BIAS_GELU_ERF>(x);
        case EPI_BIAS_SIGMOID: return act<EPI_BIAS_SIGMOID>(x);
        case EPI_BIAS_GELU_TANH: return act<EPI_BIAS_GELU_TANH>(x);
        default: return x;
    }
}

struct GemmParams {
    __half* C;
    const __half* bias;
    int M, N, K;
    int ldc;
    int epi;
    int vec_store;       // C base 16-byte aligned and ldc % 8 == 0
    int mn3d_a, mn3d_b;  // MN-major operand map is 3-D (64, K, MN / 64): two 64-wide boxes per load
    int bias_vec;        // bias base 16-byte aligned (8-wide bias loads)
    int group_m;
    int group_n;         // CTA-pair tile order: blocks of group_n tile-columns (0: whole width)
    int snake;           // CTA-pair tile order: odd bands of group_m tile-rows walk from the right
    uint64_t timeout_ns;
    // CTA-pair kernel: tiles [0, dp_tiles) whole; with tail_split the rest are
    // computed as two 256 x 128 halves each (a partial last wave costs half a tile)
    int dp_tiles;
    int tail_split;
    // split-K (swap-AB kernel): K of every tile divided among `splits` CTAs
    int splits;
    float* partials;          // [tile][split][MT][128] fp32 partial sums
    unsigned int* counters;   // [tile][4]: parts finished per 32-column slice (zero before the launch)
    // operand layouts: trans_a = A stored K x M (M contiguous, MN-major);
    // trans_b = B stored N x K (K contiguous, K-major)
    int trans_a;
    int trans_b;
    // Fault injection for the tests of the bounded waits (single-CTA kernels
    // only; -1 in every normal call): the producer never issues the loads of
    // K block `fault_skip_kb` of its first tile, so the MMA thread's wait for
    // that stage runs out and the abort path runs with no copy in flight.
    int fault_skip_kb;
};

// One 64 (M or N) x 64 (K) box of an operand tile.  The tensor map of a
// K-major operand has K as its inner coordinate, that of an MN-major one M
// (or N).  Either way the box is 8 KiB, and boxes placed 8 KiB apart extend
// the tile along M (or N): for K-major that continues the run of 8-row
// swizzle atoms, for MN-major it is the next 64-element atom column (LBO).
__device__ __forceinline__ void tma_load_box(uint32_t dst, const CUtensorMap* tm, uint32_t bar, bool k_major,
                                             int mn, int k) {
    if (k_major) tma_load_2d(dst, tm, bar, k, mn);
    else tma_load_2d(dst, tm, bar, mn, k);
}

// Shared-memory descriptor of an operand tile at `base`, and its increment
// per 16-deep K step (the MMA of step k takes desc_base + k * desc_step).
// K-major: 128-byte rows, 8-row atoms 1 KiB apart (SBO), a step is 32 bytes
// into the swizzled row.  MN-major: 64-element atom columns 8 KiB apart
// (LBO), 8-deep K groups 1 KiB apart (SBO), a step is 16 rows = 2 KiB.  The
// step adds to the start-address field (bits 0-13, address >> 4) without a
// carry into the next field: shared-memory addresses stay below 2^18.
__device__ __forceinline__ uint64_t desc_base(uint32_t base, bool mn_major) {
    return mn_major ? smem_desc_sw128(base, kBBoxBytes, 1024) : smem_desc_sw128(base, 0, 1024);
}
__device__ __forceinline__ uint64_t desc_step(bool mn_major) { return mn_major ? (2048u >> 4) : (32u >> 4); }

// Stage the bias of columns n0 .. n0 + ncol - 1 (zero past N) as packed fp16
// pairs in this warp's shared memory: done before the accumulator wait, so
// the global loads overlap it.
__device__ __forceinline__ void stage_bias(const GemmParams& p, uint32_t* bias_w, int n0, int ncol) {
    const int lane = threadIdx.x & 31;
    const uint16_t* b16 = reinterpret_cast<const uint16_t*>(p.bias);
    __syncwarp();
    for (int i = lane; i < ncol / 2; i += 32) {
        const int n = n0 + 2 * i;
        const uint32_t lo = n < p.N ? b16[n] : 0u;
        const uint32_t hi = n + 1 < p.N ? b16[n + 1] : 0u;
        bias_w[i] = lo | (hi << 16);
    }
    __syncwarp();
}

// Bias, activation ACT and fp16 rounding of one 32-column chunk of this
// thread's row: r = 32 fp32 accumulator columns; bw = the chunk's 16 staged
// bias pairs.
template <int ACT, bool BIAS>
__device__ __forceinline__ void epilogue_math_fixed(const uint32_t (&r)[32], const uint32_t* bw, uint32_t (&h)[16]) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        float x0 = __uint_as_float(r[2 * j]);
        float x1 = __uint_as_float(r[2 * j + 1]);
        if (BIAS) {
            const uint32_t w = bw[j];
            const float2 b2 = __half22float2(*reinterpret_cast<const __half2*>(&w));
            x0 += b2.x;
            x1 += b2.y;
        }
        const __half2 hv = __floats2half2_rn(act<ACT>(x0), act<ACT>(x1));
        h[j] = *reinterpret_cast<const uint32_t*>(&hv);
    }
}

// Epilogue kind read from the parameters at run time (see epilogue_math_act).
constexpr int EPI_DYNAMIC = -1;

// epilogue_math_fixed for a compile-time kind, or, for EPI_DYNAMIC, for the
// kind in p.epi, dispatched once per chunk.
template <int ACT, bool BIAS>
__device__ __forceinline__ void epilogue_math_act(const GemmParams& p, const uint32_t (&r)[32], const uint32_t* bw,
                                                  uint32_t (&h)[16]) {
    if (ACT != EPI_DYNAMIC) {
        epilogue_math_fixed<ACT, BIAS>(r, bw, h);
        return;
    }
    switch (p.epi) {
        case EPI_BIAS: epilogue_math_fixed<EPI_NONE, true>(r, bw, h); break;
        case EPI_BIAS_RELU: epilogue_math_fixed<EPI_BIAS_RELU, true>(r, bw, h); break;
        case EPI_BIAS_GELU_ERF: epilogue_math_fixed<EPI_BIAS_GELU_ERF, true>(r, bw, h); break;
        case EPI_BIAS_SIGMOID: epilogue_math_fixed<EPI_BIAS_SIGMOID, true>(r, bw, h); break;
        case EPI_BIAS_GELU_TANH: epilogue_math_fixed<EPI_BIAS_GELU_TANH, true>(r, bw, h); break;
        default: epilogue_math_fixed<EPI_NONE, false>(r, bw, h); break;
    }
}


// Store one 32 x 32 fp16 block: rows row0..row0+31 (one per lane, h = that
// lane's 32 columns from col0).  Where C rows are 16-byte aligned and the
// chunk is whole, each thread writes its own 64-byte row segment with 16-byte
// stores; otherwise (N % 8 != 0, unaligned C, or the ragged last chunk) the
// block goes through `stage` (this warp's shared-memory tile) and all 32
// lanes write one row at a time, 64 contiguous bytes per store.
__device__ __forceinline__ void epilogue_store(const GemmParams& p, const uint32_t (&h)[16], int row0, int col0,
                                               uint32_t* stage) {
    const int lane = threadIdx.x & 31;
    if (p.vec_store && col0 + 32 <= p.N) {
        const int row = row0 + lane;
        if (row < p.M) {
            uint4* dst = reinterpret_cast<uint4*>(p.C + static_cast<int64_t>(row) * p.ldc + col0);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) stage[lane * kStageRowWords + j] = h[j];
    __syncwarp();
    const bool col_ok = col0 + lane < p.N;
    uint16_t* cbase = reinterpret_cast<uint16_t*>(p.C + static_cast<int64_t>(row0) * p.ldc + col0 + lane);
    if (row0 + 32 <= p.M) {
#pragma unroll 8
        for (int rr = 0; rr < 32; ++rr) {
            const uint32_t w = stage[rr * kStageRowWords + (lane >> 1)];
            if (col_ok) cbase[static_cast<int64_t>(rr) * p.ldc] = static_cast<uint16_t>(w >> (16 * (lane & 1)));
        }
    } else {
        const int rows_here = p.M - row0;   // may be <= 0: nothing to store
        for (int rr = 0; rr < rows_here; ++rr) {
            const uint32_t w = stage[rr * kStageRowWords + (lane >> 1)];
            if (col_ok) cbase[static_cast<int64_t>(rr) * p.ldc] = static_cast<uint16_t>(w >> (16 * (lane & 1)));
        }
    }
    __syncwarp();
}

// Epilogue of NCOL accumulator columns for this warp's 32 TMEM lanes (tile
// rows row0..row0+31, one per thread), starting at TMEM address t_base and
// output column n0, with epilogue kind ACT (bias added if BIAS; EPI_DYNAMIC:
// the kind in p.epi).  `stage` is
// the warp's shared-memory block, followed by its staged bias (stage_bias).
// The TMEM load of chunk c+1 is in flight while chunk c is processed.
template <int NCOL, int ACT, bool BIAS>
__device__ __forceinline__ void epilogue_rows_act(const GemmParams& p, uint32_t t_base, int row0, int n0,
                                                  uint32_t* stage) {
    constexpr int kChunks = NCOL / 32;
    const uint32_t* bias_w = stage + kStageBlockWords;
    uint32_t ra[32], rb[32];
    tmem_ld_32x32b_x32(t_base, ra);
    tmem_wait_ld(ra);
    // chunks two at a time: the even one in ra, the odd one in rb
#pragma unroll 1
    for (int c = 0; c < kChunks; c += 2) {
        const int col0 = n0 + 32 * c;
        if (col0 >= p.N) break;   // warp-uniform: the remaining chunks are right of N
        const bool odd = c + 1 < kChunks && col0 + 32 < p.N;
        if (odd) tmem_ld_32x32b_x32(t_base + 32u * (c + 1), rb);
        uint32_t h[16];
        epilogue_math_act<ACT, BIAS>(p, ra, bias_w + 16 * c, h);
        epilogue_store(p, h, row0, col0, stage);
        if (!odd) break;
        tmem_wait_ld(rb);
        const bool even = c + 2 < kChunks && col0 + 64 < p.N;
        if (even) tmem_ld_32x32b_x32(t_base + 32u * (c + 2), ra);
        epilogue_math_act<ACT, BIAS>(p, rb, bias_w + 16 * (c + 1), h);
        epilogue_store(p, h, row0, col0 + 32, stage);
        if (!even) break;
        tmem_wait_ld(ra);
    }
}

// epilogue_rows_act with the epilogue kind read at run time, chosen once per
// 32-column chunk (outside the element loop): a switch inside the element
// loop (one dispatch per element) measured 14 % slower on 4096^3 with GELU.
// The CTA-pair kernel takes the kind as a template argument instead.
template <int NCOL>
__device__ __forceinline__ void epilogue_rows(const GemmParams& p, uint32_t t_base, int row0, int n0,
                                              uint32_t* stage) {
    epilogue_rows_act<NCOL, EPI_DYNAMIC, true>(p, t_base, row0, n0, stage);
}

// ---------------------------------------------------------------- split K across a cluster
// The S CTAs of a cluster compute one tile, each over its share of K.  CTA o
// finishes rows o * 128 / S .. of the tile: every CTA pushes its partial rows
// of that slice straight from tensor memory into CTA o's shared memory
// (remote 16-byte stores; the operand ring, idle by then in every CTA of the
// cluster), slot `source rank`, and after a cluster barrier CTA o sums its S
// slots locally, in rank order.  Row pitch (fp32 words) of the received
// rows: 4 words of padding put a warp's 16-byte stores on different banks.
template <int BN>
struct SplitPlan {
    static constexpr int kPitch = BN + 4;
    static constexpr uint32_t kBytes = 128u * kPitch * 4u;
};

// This warp's 32 accumulator rows (row0 = 32 q ..) x BN/2 columns (col0 ..)
// from tensor memory to the CTA that finishes them.  All 32 rows go to one
// CTA (a slice is 128 / S >= 32 rows, and slices start at multiples of 32).
template <int BN>
__device__ __forceinline__ void split_push(uint32_t recv, uint32_t t_base, int row0, int col0, int rank, int S) {
    const int lane = threadIdx.x & 31;
    const int rows = 128 / S;
    const int row = row0 + lane;
    const uint32_t owner = static_cast<uint32_t>(row / rows);
    const int slot_row = rank * rows + row % rows;
    const uint32_t dst = mapa_shared(recv + static_cast<uint32_t>(slot_row * SplitPlan<BN>::kPitch + col0) * 4u, owner);
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_base + 32u * c, r);
        tmem_wait_ld(r);
#pragma unroll
        for (int v = 0; v < 8; ++v)
            st_shared_cluster_v4(dst + (32u * c + 4u * v) * 4u, r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
    }
}

// After the cluster barrier that follows every push: this CTA's slice of
// tile tc (rows rank * 128 / S ..), the S received partials summed in rank
// order (a fixed order), plus bias, activation, fp16, stored (16 bytes where
// C allows).  tid runs over the 256 epilogue threads; SS is S.
template <int BN, int SS>
__device__ __forceinline__ void split_reduce(const GemmParams& p, uint32_t recv, TileCoord tc, int rank, int tid) {
    constexpr int kGroups = BN / 8;                 // 8-column groups per row
    constexpr int kRows = 128 / SS;
    for (int g = tid; g < kRows * kGroups; g += 256) {
        const int lr = g / kGroups;
        const int cc = (g % kGroups) * 8;
        const int row = tc.m0 + rank * kRows + lr, col = tc.n0 + cc;
        if (row >= p.M || col >= p.N) continue;
        float4 part[SS][2];
#pragma unroll
        for (int src = 0; src < SS; ++src) {
            const uint32_t a = recv + static_cast<uint32_t>((src * kRows + lr) * SplitPlan<BN>::kPitch + cc) * 4u;
            part[src][0] = ld_shared_v4(a);
            part[src][1] = ld_shared_v4(a + 16u);
        }
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = 0.0f;
#pragma unroll
        for (int src = 0; src < SS; ++src) {
            x[0] += part[src][0].x; x[1] += part[src][0].y; x[2] += part[src][0].z; x[3] += part[src][0].w;
            x[4] += part[src][1].x; x[5] += part[src][1].y; x[6] += part[src][1].z; x[7] += part[src][1].w;
        }
        if (p.epi != EPI_NONE) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (col + i < p.N) x[i] += __half2float(p.bias[col + i]);
        }
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 hv = __floats2half2_rn(apply_act(x[2 * i], p.epi), apply_act(x[2 * i + 1], p.epi));
            h[i] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        __half* dst = p.C + static_cast<int64_t>(row) * p.ldc + col;
        if (p.vec_store && col + 8 <= p.N) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(h[0], h[1], h[2], h[3]);
        } else {
            for (int i = 0; i < 8 && col + i < p.N; ++i)
                reinterpret_cast<uint16_t*>(dst)[i] = static_cast<uint16_t>(h[i >> 1] >> (16 * (i & 1)));
        }
    }
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
gemm_f16_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
    using SP = SmemPlan<BN, STAGES>;
    static_assert(SplitPlan<BN>::kBytes <= SP::kStage - SP::kA, "a partial tile fits in the operand ring");
    constexpr int kBoxesB = BN / 64;
    constexpr uint32_t kTmemCols = 2 * BN;   // two accumulators, power of two >= 32
    const bool ta = p.trans_a != 0, tb = p.trans_b != 0;

    extern __shared__ uint8_t smem_raw[];
    // 1 KiB alignment of the shared-window address (128-byte swizzle atoms).
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);

    const uint32_t sA = base_s + SP::kA;
    const uint32_t sB = base_s + SP::kB;
    const uint32_t bars = base_s + SP::kBars;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bars + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bars + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bars + 8u * (2 * STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + SP::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + SP::kAbort);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // set-up above overlaps the previous kernel; global memory only from here
    grid_dependency_wait();
    grid_launch_dependents();

    const int tiles_m = (p.M + kBM - 1) / kBM;
    const int tiles_n = (p.N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int kblocks = (p.K + kBK - 1) / kBK;
    unsigned int* status = &g_status;
    // Split K across a cluster (p.splits = S > 1, launched as clusters of S
    // CTAs, one tile per cluster): CTA `rank` multiplies the tile's K blocks
    // [kb_lo, kb_hi); the S fp32 partial tiles are summed through distributed
    // shared memory after the mainloop (split_reduce below).
    const int S = p.splits;
    const int rank = S > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int t_first = static_cast<int>(blockIdx.x) / S;
    const int t_stride = S > 1 ? num_tiles : static_cast<int>(gridDim.x);   // split: this cluster's tile only
    const int kb_per = (kblocks + S - 1) / S;
    const int kb_lo = rank * kb_per;
    const int kb_hi = min(kblocks, kb_lo + kb_per);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            int skip_kb = p.fault_skip_kb;   // -1 except in fault-injection tests
            for (int t = t_first; ok && t < num_tiles; t += t_stride) {
                const TileCoord tc = tile_coord(t, tiles_m, tiles_n, p.group_m, BN);
                // B boxes entirely right of N are skipped: the stale smem they
                // leave only feeds accumulator columns >= N, which are never stored.
                const int live_boxes = min(kBoxesB, (p.N - tc.n0 + 63) / 64);
                // A: one 128-row K-major box, or (A stored K x M) two 64-row
                // boxes, the second skipped when it starts past M
                const int a_boxes = ta ? (tc.m0 + 64 < p.M ? 2 : 1) : 1;
                const uint32_t bytes = (ta ? static_cast<uint32_t>(a_boxes) * kBBoxBytes : kATileBytes) +
                                       static_cast<uint32_t>(live_boxes) * kBBoxBytes;
                for (int kb = kb_lo; kb < kb_hi; ++kb) {
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag, status,
                                           ROLE_PRODUCER, BAR_EMPTY)) { ok = false; break; }
                    if (kb - kb_lo == skip_kb) {   // injected fault: this stage's loads never come
                        ++issued;
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                        continue;
                    }
                    mbar_arrive_expect_tx(full_bar(stage), bytes);
                    if (ta) {
                        for (int c = 0; c < a_boxes; ++c)
                            tma_load_box(sA + stage * kATileBytes + c * kBBoxBytes, &tmA, full_bar(stage), false,
                                         tc.m0 + 64 * c, kb * kBK);
                    } else {
                        tma_load_2d(sA + stage * kATileBytes, &tmA, full_bar(stage), kb * kBK, tc.m0);
                    }
                    for (int c = 0; c < live_boxes; ++c)
                        tma_load_box(sB + stage * SP::kBTileBytes + c * kBBoxBytes, &tmB, full_bar(stage), tb,
                                     tc.n0 + 64 * c, kb * kBK);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                skip_kb = -1;
            }
            // Let the last (up to STAGES) loads land before the CTA can exit:
            // earlier ones were consumed, which the empty-barrier waits proved.
            const int pending = min(issued, STAGES);
            for (int i = 0; i < pending; ++i) {
                if (--stage < 0) { stage = STAGES - 1; phase ^= 1u; }
                mbar_wait_bounded(full_bar(stage), phase, p.timeout_ns, nullptr, status, ROLE_DRAIN, BAR_FULL);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        {
            const uint32_t idesc = idesc_f16_f32(kBM, BN, /*b_mn_major=*/!tb, /*a_mn_major=*/ta);
            const uint64_t a_step = desc_step(ta), b_step = desc_step(!tb);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = t_first; ok && t < num_tiles; t += t_stride) {
                if (!mbar_wait_bounded(acce_bar(acc), acc_phase ^ 1u, p.timeout_ns, abort_flag, status,
                                            ROLE_MMA, BAR_ACC_EMPTY)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = kb_lo; kb < kb_hi; ++kb) {
                    if (!mbar_wait_bounded(full_bar(stage), phase, p.timeout_ns, abort_flag, status,
                                                ROLE_MMA, BAR_FULL)) { ok = false; break; }
                    tc_fence_after();
                    // A K-major unless stored K x M; B MN-major unless stored N x K
                    const uint64_t a_desc = desc_base(sA + stage * kATileBytes, ta);
                    const uint64_t b_desc = desc_base(sB + stage * SP::kBTileBytes, !tb);
#pragma unroll
                    for (int k = 0; k < kBK / kUMMA_K; ++k)
                        tc_mma_f16(d_tmem, a_desc + k * a_step, b_desc + k * b_step, idesc,
                                   (kb != kb_lo || k != 0) ? 1u : 0u);
                    tc_commit(empty_bar(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit(accf_bar(acc));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // Every MMA issued has completed before the accumulator is freed.
            tc_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, p.timeout_ns, nullptr, status, ROLE_DRAIN, BAR_DRAIN);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;            // TMEM lane quarter this warp may access
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = t_first; t < num_tiles; t += t_stride) {
            const TileCoord tc = tile_coord(t, tiles_m, tiles_n, p.group_m, BN);
            const int half = (warp - 2) >> 2;   // which half of the tile's columns
            uint32_t* stage = reinterpret_cast<uint32_t*>(base + SP::kStage + (warp - 2) * kStageWarpBytes);
            if (p.epi != EPI_NONE && S == 1)
                stage_bias(p, stage + kStageBlockWords, tc.n0 + half * (BN / 2), BN / 2);
            // tcgen05.ld is warp-collective: the go/no-go decision must be warp-uniform.
            const bool ready = mbar_wait_bounded(accf_bar(acc), acc_phase, p.timeout_ns, abort_flag, status,
                                                 ROLE_EPILOGUE, BAR_ACC_FULL);
            if (!__all_sync(0xffffffffu, ready)) break;
            tc_fence_after();
            const uint32_t t_base = tmem_base + static_cast<uint32_t>(acc * BN + half * (BN / 2)) +
                                    (static_cast<uint32_t>(32 * q) << 16);
            if (S > 1) break;   // the partial stays in tensor memory until every CTA's ring is idle
            epilogue_rows<BN / 2>(p, t_base, tc.m0 + 32 * q, tc.n0 + half * (BN / 2), stage);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(acc));
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    __syncthreads();
    if (S > 1) {
        // every CTA of the cluster is done with its operand ring (its MMAs completed)
        cluster_sync_all();
        if (warp >= 2) {
            const int q = warp & 3, half = (warp - 2) >> 2;
            tc_fence_after();
            split_push<BN>(base_s + SP::kA, tmem_base + static_cast<uint32_t>(half * (BN / 2)) +
                                               (static_cast<uint32_t>(32 * q) << 16),
                           32 * q, half * (BN / 2), rank, S);
        }
        // every partial slice has landed where it is summed; no CTA touches a
        // peer's shared memory after this
        cluster_sync_all();
        if (warp >= 2) {
            const TileCoord tc = tile_coord(t_first, tiles_m, tiles_n, p.group_m, BN);
            const int tid = static_cast<int>(threadIdx.x) - 64;
            if (S == 2) split_reduce<BN, 2>(p, base_s + SP::kA, tc, rank, tid);
            else split_reduce<BN, 4>(p, base_s + SP::kA, tc, rank, tid);
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// K == 0: C = epilogue(bias) (zeros for NONE).
__global__ void gemm_f16_bias_only_kernel(__half* C, const __half* bias, int64_t M, int64_t N, int64_t ldc, int epi) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t total = M * N;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = e / N, j = e - i * N;
        const float x = epi == EPI_NONE ? 0.0f : __half2float(bias[j]);
        C[i * ldc + j] = __float2half_rn(apply_act(x, epi));
    }
}

// Row repack: dst[r, 0:cols] = src[r, 0:cols] with a 16-byte-multiple pitch,
// so the tensor map can describe the copy (columns >= cols are left as is;
// the tensor map's extent stops at `cols`, so TMA never reads them).  Each
// thread writes 16-byte pieces, elements c .. c+7 of `group` rows (ld_dst
// % 8 == 0 and dst is 256-byte aligned).  A source piece is only 2-byte
// aligned: it lies within the aligned 16-byte chunk holding its first element
// and, unless it starts on a chunk boundary, the next chunk; each of these
// holds at least one element of the piece, so neither load reaches outside
// the memory pages the source occupies.  The piece is cut out of the two
// chunks by a funnel shift (odd element offset) and a word offset picked by
// selects.  All of a thread's loads are issued before its first store, so
// each thread keeps up to 2 x kRepackRows loads in flight (large copies use
// groups of kRepackRows rows; small ones, where blocks are scarce, single
// rows).  A row's last piece, if shorter than 8 elements, is copied element
// by element.  grid.x covers a row in 2048-element pieces, grid.y strides
// over groups of rows.
constexpr int kRepackRows = 4;

__device__ __forceinline__ uint4 repack_cut(const uint4 v0, const uint4 v1, uint32_t off) {
    const uint32_t x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    const uint32_t sh = (off & 2u) ? 16u : 0u;   // an odd element offset
    const uint32_t wo = off >> 2;                  // whole words to skip: 0 .. 3
    uint32_t z[7];
#pragma unroll
    for (int i = 0; i < 7; ++i) z[i] = __funnelshift_r(x[i], x[i + 1], sh);
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t lo = (wo & 1u) ? z[j + 1] : z[j];
        const uint32_t hi = (wo & 1u) ? z[j + 3] : z[j + 2];
        w[j] = (wo & 2u) ? hi : lo;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void gemm_f16_repack_kernel(uint16_t* __restrict__ dst, const uint16_t* __restrict__ src,
                                       int64_t rows, int64_t cols, int64_t ld_src, int64_t ld_dst, int group) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t c = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
    if (c >= cols) return;
    const bool whole = c + 8 <= cols;
    for (int64_t r0 = static_cast<int64_t>(blockIdx.y) * group; r0 < rows;
         r0 += static_cast<int64_t>(gridDim.y) * group) {
        const int64_t r_end = min(rows, r0 + group);
        if (whole) {
            uint4 v0[kRepackRows], v1[kRepackRows];
            uint32_t off[kRepackRows];
#pragma unroll
            for (int i = 0; i < kRepackRows; ++i) {
                v0[i] = v1[i] = make_uint4(0u, 0u, 0u, 0u);
                off[i] = 0u;
                if (r0 + i < r_end) {
                    const uintptr_t a = reinterpret_cast<uintptr_t>(src + (r0 + i) * ld_src + c);
                    off[i] = static_cast<uint32_t>(a & 15u);       // bytes past the chunk boundary, even
                    const uint4* chunk = reinterpret_cast<const uint4*>(a - off[i]);
                    v0[i] = __ldg(chunk);
                    if (off[i] != 0u) v1[i] = __ldg(chunk + 1);
                }
            }
#pragma unroll
            for (int i = 0; i < kRepackRows; ++i)
                if (r0 + i < r_end)
                    *reinterpret_cast<uint4*>(dst + (r0 + i) * ld_dst + c) = repack_cut(v0[i], v1[i], off[i]);
        } else {
            for (int64_t r = r0; r < r_end; ++r)
                for (int64_t j = 0; j < cols - c; ++j) dst[r * ld_dst + c + j] = src[r * ld_src + c + j];
        }
    }
}

// One CTA, one thread waits on a barrier nobody arrives on.
__global__ void gemm_f16_selftest_timeout_kernel(uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbarrier_init();
        mbar_wait_bounded(smem_u32(&bar), 0, timeout_ns, nullptr, &g_status, ROLE_SELFTEST, BAR_TEST);
    }
}

}  // namespace gemm_f16_dev
