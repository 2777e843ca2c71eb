// Swap-AB variant of the fused fp16 GEMM for short A (small M):
//
//   C^T = B^T . A^T,   then C = epilogue(C + bias) written transposed back.
//
// Same method as gemm_kernels.cuh ("writing-tilelang-kernels", GEMM
// (Minimal); "TileLang: Write, Autotune, and Ship Fused Tensor-Core Kernels
// from Python", Why tile-level control matters).  The tensor core's M side
// must be 128 rows; with M of 64 or less, putting N on that side instead keeps
// every MMA row useful and keeps the A tile (now the MMA's N side, MT rows)
// small, so most of shared memory holds B, the operand this shape streams
// from HBM:
//
//   * tile = 128 columns of C (MMA M, one TMEM lane each) x MT rows of C
//     (MMA N = 16, 32 or 64);
//   * MMA "A" operand = B^T: the same two 64 x 64 boxes as the regular
//     kernel's B (MN-major; K-major when B is stored N x K);
//   * MMA "B" operand = A^T: an MT x 64 box of A rows (K-major; when A is
//     stored K x M, MT = 64 and the box is MN-major);
//   * stage = 16 KiB of B + MT x 128 B of A, 9 to 12 stages deep;
//   * epilogue: thread = one output column n (its TMEM lane), registers = MT
//     rows; bias[n] is one value per thread; every store of a warp covers 32
//     consecutive columns of one row of C (64 contiguous bytes);
//   * split-K: a CTA streams HBM at a bounded rate (its outstanding TMA
//     requests), so when there are fewer tiles than SMs each tile's K range
//     is divided among `splits` CTAs.  Every part writes its fp32 partial
//     tile to scratch and counts itself in per-slice counters; the last part
//     of a slice to finish sums all parts in part order (so the result does
//     not depend on which finished last), then applies bias and activation
//     and writes C.  No CTA waits for another.
#pragma once

#include "gemm_kernels.cuh"

namespace gemm_f16_dev {

constexpr int kSwapThreads = 192;   // producer, MMA, 4 epilogue warps

// The 64 accumulator columns of this thread's TMEM lane in one load, and its
// wait (the registers as read-write operands: no use is scheduled before it).
__device__ __forceinline__ void swap_tmem_ld_x64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
        "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
        "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63"
        "}, [%64];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr));
}
__device__ __forceinline__ void swap_tmem_wait_ld_x64(uint32_t (&r)[64]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
          "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
          "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
          "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]),
          "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]),
          "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]),
          "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]),
          "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63]) : : "memory");
}
// This thread's MT accumulator columns in one load (MT / 16 loads, each waited
// for in turn, measured the same or up to 4 % slower: 48x4096x4096 20.4 -> 19.5 us).
template <int MT>
__device__ __forceinline__ void swap_ld_acc(uint32_t taddr, uint32_t (&r)[MT]) {
    if constexpr (MT == 16) tmem_ld_32x32b_x16(taddr, r);
    else if constexpr (MT == 32) tmem_ld_32x32b_x32(taddr, r);
    else swap_tmem_ld_x64(taddr, r);
    if constexpr (MT == 64) swap_tmem_wait_ld_x64(r);
    else tmem_wait_ld(r);
}

template <int MT, int STAGES>
struct SmemPlanSwap {
    static constexpr uint32_t kBtBytes = 2 * kBBoxBytes;       // 128 columns of B x 64 K
    static constexpr uint32_t kAtBytes = MT * kBK * 2;         // MT rows of A x 64 K
    static constexpr uint32_t kStage = kBtBytes + kAtBytes;    // multiple of 1 KiB for MT % 8 == 0
    static constexpr uint32_t kBars = STAGES * kStage;
    static constexpr uint32_t kNumBars = 2 * STAGES + 2 + 2 + 1;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kEnd = kAbort + 4;
    static constexpr uint32_t kDynamicBytes = kEnd + 1024;
    static_assert(kStage % 1024 == 0, "swizzle atoms need 1 KiB alignment");
};

// Column n of rows m0 .. m0 + MT - 1 of C (one thread): activation ACT of
// v[i] + b, rounded to fp16; rows past M and columns past N are not stored.
template <int ACT, int MT>
__device__ __forceinline__ void swap_store(const GemmParams& p, const float (&v)[MT], float b, int m0, int n,
                                           bool col_ok) {
#pragma unroll
    for (int i = 0; i < MT; ++i) {
        const int m = m0 + i;
        if (col_ok && m < p.M) p.C[static_cast<int64_t>(m) * p.ldc + n] = __float2half_rn(act<ACT>(v[i] + b));
    }
}

template <int MT, int STAGES>
__global__ void __launch_bounds__(kSwapThreads, 1)
gemm_f16_swap_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmParams p) {
    using SP = SmemPlanSwap<MT, STAGES>;
    constexpr int TN = 128;                                      // columns of C per tile
    // A stored K x M takes MT = 64 (the host plans it so): one MN-major box
    const bool ta = p.trans_a != 0, tb = p.trans_b != 0;
    constexpr uint32_t kTmemCols = 2 * MT < 32 ? 32 : 2 * MT;    // two accumulators

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
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
            mbar_init(acce_bar(b), 4);
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

    const int tiles_m = (p.M + MT - 1) / MT;
    const int tiles_n = (p.N + TN - 1) / TN;
    const int num_tiles = tiles_m * tiles_n;
    const int kblocks = (p.K + kBK - 1) / kBK;
    const int S = p.splits;                          // >= 1; no part is empty (host guarantees)
    const int kb_per = (kblocks + S - 1) / S;
    const int num_units = num_tiles * S;             // unit u: tile u / S, part u % S
    unsigned int* status = &g_status;
    // tile t: row block t % tiles_m, column block t / tiles_m (consecutive CTAs share a B panel)
    auto tile_m0 = [&](int t) { return (t % tiles_m) * MT; };
    auto tile_n0 = [&](int t) { return (t / tiles_m) * TN; };
    auto kb_begin = [&](int u) { return (u % S) * kb_per; };
    auto kb_end = [&](int u) { return min(kblocks, (u % S + 1) * kb_per); };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            int skip_kb = p.fault_skip_kb;   // -1 except in fault-injection tests
            for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
                const int t = u / S;
                const int m0 = tile_m0(t), n0 = tile_n0(t);
                // a B box wholly right of N is skipped: its stale columns only
                // reach TMEM lanes that are never stored
                const int live_b = min(2, (p.N - n0 + 63) / 64);
                const uint32_t bytes = static_cast<uint32_t>(live_b) * kBBoxBytes + SP::kAtBytes;
                for (int kb = kb_begin(u); kb < kb_end(u); ++kb) {
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag, status,
                                           ROLE_PRODUCER, BAR_EMPTY)) { ok = false; break; }
                    if (kb - kb_begin(u) == skip_kb) {   // injected fault: this stage's loads never come
                        ++issued;
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                        continue;
                    }
                    const uint32_t st = base_s + stage * SP::kStage;
                    mbar_arrive_expect_tx(full_bar(stage), bytes);
                    for (int c = 0; c < live_b; ++c)
                        tma_load_box(st + c * kBBoxBytes, &tmB, full_bar(stage), tb, n0 + 64 * c, kb * kBK);
                    if (ta) tma_load_2d(st + SP::kBtBytes, &tmA, full_bar(stage), m0, kb * kBK);
                    else tma_load_2d(st + SP::kBtBytes, &tmA, full_bar(stage), kb * kBK, m0);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                skip_kb = -1;
            }
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
            // MMA A = B^T (MN-major unless B is stored N x K), MMA B = A^T (K-major unless A is stored K x M)
            const uint32_t idesc = idesc_f16_f32(TN, MT, /*b_mn_major=*/ta, /*a_mn_major=*/!tb);
            const uint64_t a_step = desc_step(!tb), b_step = desc_step(ta);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
                if (!mbar_wait_bounded(acce_bar(acc), acc_phase ^ 1u, p.timeout_ns, abort_flag, status,
                                            ROLE_MMA, BAR_ACC_EMPTY)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * MT);
                const int kb0 = kb_begin(u);
                for (int kb = kb0; kb < kb_end(u); ++kb) {
                    if (!mbar_wait_bounded(full_bar(stage), phase, p.timeout_ns, abort_flag, status,
                                                ROLE_MMA, BAR_FULL)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t st = base_s + stage * SP::kStage;
                    const uint64_t a_desc = desc_base(st, !tb);
                    const uint64_t b_desc = desc_base(st + SP::kBtBytes, ta);
#pragma unroll
                    for (int k = 0; k < kBK / kUMMA_K; ++k)
                        tc_mma_f16(d_tmem, a_desc + k * a_step, b_desc + k * b_step, idesc,
                                   (kb != kb0 || k != 0) ? 1u : 0u);
                    tc_commit(empty_bar(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit(accf_bar(acc));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            tc_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, p.timeout_ns, nullptr, status, ROLE_DRAIN, BAR_DRAIN);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;   // TMEM lane quarter = columns n0 + 32q .. n0 + 32q + 31
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
            const int t = u / S, part = u % S;
            const int m0 = tile_m0(t), n0 = tile_n0(t);
            const int nl = 32 * q + lane;                // column within the tile
            const int n = n0 + nl;
            const bool col_ok = n < p.N;
            const bool ready = mbar_wait_bounded(accf_bar(acc), acc_phase, p.timeout_ns, abort_flag, status,
                                                 ROLE_EPILOGUE, BAR_ACC_FULL);
            if (!__all_sync(0xffffffffu, ready)) break;
            tc_fence_after();
            const uint32_t t_base = tmem_base + static_cast<uint32_t>(acc * MT) + (static_cast<uint32_t>(32 * q) << 16);
            float v[MT];
            {
                uint32_t r[MT];
                swap_ld_acc<MT>(t_base, r);
#pragma unroll
                for (int i = 0; i < MT; ++i) v[i] = __uint_as_float(r[i]);
            }
            // the accumulator is in registers now: hand the TMEM buffer back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(acc));
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }

            bool finish = true;
            if (S > 1) {
                float* mine = p.partials + static_cast<int64_t>(u) * MT * TN;
#pragma unroll
                for (int i = 0; i < MT; ++i) __stcg(mine + i * TN + nl, v[i]);
                __threadfence();
                __syncwarp();
                unsigned int before = 0;
                if (lane == 0) before = atomicAdd(p.counters + 4 * t + q, 1u);
                before = __shfl_sync(0xffffffffu, before, 0);
                finish = before == static_cast<unsigned int>(S - 1);
                if (finish) {
                    __threadfence();
                    // all parts, in part order: the sum does not depend on arrival order
                    float sum[MT];
#pragma unroll
                    for (int i = 0; i < MT; ++i) sum[i] = 0.0f;
                    for (int sp = 0; sp < S; ++sp) {
                        const float* src = p.partials + static_cast<int64_t>(t * S + sp) * MT * TN;
#pragma unroll
                        for (int i = 0; i < MT; ++i) sum[i] += sp == part ? v[i] : __ldcg(src + i * TN + nl);
                    }
#pragma unroll
                    for (int i = 0; i < MT; ++i) v[i] = sum[i];
                    if (lane == 0) p.counters[4 * t + q] = 0u;   // ready for the next launch
                }
            }
            if (finish) {
                const float b = (p.epi != EPI_NONE && col_ok) ? __half2float(p.bias[n]) : 0.0f;
                switch (p.epi) {   // once per tile, not per element
                    case EPI_BIAS_RELU: swap_store<EPI_BIAS_RELU, MT>(p, v, b, m0, n, col_ok); break;
                    case EPI_BIAS_GELU_ERF: swap_store<EPI_BIAS_GELU_ERF, MT>(p, v, b, m0, n, col_ok); break;
                    case EPI_BIAS_SIGMOID: swap_store<EPI_BIAS_SIGMOID, MT>(p, v, b, m0, n, col_ok); break;
                    case EPI_BIAS_GELU_TANH: swap_store<EPI_BIAS_GELU_TANH, MT>(p, v, b, m0, n, col_ok); break;
                    default: swap_store<EPI_NONE, MT>(p, v, b, m0, n, col_ok); break;
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace gemm_f16_dev
