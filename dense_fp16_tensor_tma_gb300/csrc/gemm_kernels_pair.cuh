// CTA-pair variant of the fused fp16 GEMM:  C = epilogue(A.B + bias).
//
// Same method as gemm_kernels.cuh (tile loop over K, tensor-core tile product
// into an on-chip fp32 accumulator, fused bias + activation, one write of C:
// "writing-tilelang-kernels", GEMM (Minimal); "TileLang: Write, Autotune, and
// Ship Fused Tensor-Core Kernels from Python", Why tile-level control
// matters), mapped onto two SMs that cooperate on one 256 x 256 output tile:
//
//   * a cluster of 2 CTAs; CTA r (r = 0, 1) owns output rows m0 + 128r ..
//     m0 + 128r + 127 and loads only its own 128 rows of A and its own 128
//     columns of B: 16 KiB + 16 KiB per 64-deep K sub-block, KSUB sub-blocks
//     per pipeline stage (8 MMAs per barrier round trip at KSUB = 2: each
//     stage hand-over costs the tensor pipe a short bubble, so fewer, deeper
//     stages keep it busier);
//   * one thread of CTA 0 issues tcgen05.mma.cta_group::2 (M = 256, N = 256,
//     K = 16): each SM's tensor core computes its 128 rows against all 256
//     columns, taking B from both SMs' shared memory, so per SM the operand
//     traffic is 2/3 of the single-SM 128 x 256 tile for the same FLOPs;
//   * both CTAs' TMA loads complete on CTA 0's "full" barrier; MMA completion
//     is multicast to both CTAs' "empty" and "accumulator full" barriers;
//     both CTAs' epilogues arrive on CTA 0's "accumulator empty" barrier;
//   * each CTA's epilogue reads its own tensor memory (its 128 rows x 256
//     fp32 columns, double-buffered) and writes its own rows of C.
#pragma once

#include <type_traits>

#include "gemm_kernels.cuh"

namespace gemm_f16_dev {

constexpr uint32_t kBHalfSubBytes = 128 * kBK * 2;   // this CTA's 128 columns of a 64-deep K sub-block: 16 KiB

// tma_load_box for the pair: the bytes complete on the leader CTA's barrier.
__device__ __forceinline__ void tma_load_box_pair(uint32_t dst, const CUtensorMap* tm, uint32_t bar_leader,
                                                  bool k_major, int mn, int k) {
    if (k_major) tma_load_2d_pair(dst, tm, bar_leader, k, mn);
    else tma_load_2d_pair(dst, tm, bar_leader, mn, k);
}

template <int STAGES, int KSUB>
struct SmemPlanPair {
    static constexpr uint32_t kAStage = KSUB * kATileBytes;        // KSUB A boxes
    static constexpr uint32_t kBStage = KSUB * kBHalfSubBytes;     // KSUB x two 64-column B boxes
    static constexpr uint32_t kA = 0;
    static constexpr uint32_t kB = kA + STAGES * kAStage;
    static constexpr uint32_t kStage = kB + STAGES * kBStage;   // epilogue staging (narrow stores)
    static constexpr uint32_t kBars = kStage + kStageBytes;
    static constexpr uint32_t kNumBars = 2 * STAGES + 2 + 2 + 1;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kEnd = kAbort + 4;
    static constexpr uint32_t kDynamicBytes = kEnd + 1024;
};

// Tile t of a tiles_m x tiles_n grid in grouped order: bands of group_m
// tile-rows, each walked in blocks of group_n tile-columns (the whole width
// when group_n == 0), column by column inside a block, so a wave of
// concurrent pairs covers a compact block of tiles that share A row-panels
// and B column-panels in L2.  With `snake`, odd bands walk their columns from
// the right: a band starts on the B panels its predecessor ended with.
__device__ __forceinline__ TileCoord tile_coord_bm(int t, int tiles_m, int tiles_n, int group_m, int BM, int BN,
                                                   int group_n = 0, int snake = 0) {
    const int band_tiles = group_m * tiles_n;
    const int band = t / band_tiles;
    const int first_m = band * group_m;
    const int rows = min(tiles_m - first_m, group_m);
    const int r = t - band * band_tiles;           // inside the band: rows x tiles_n tiles
    const int gn = group_n > 0 ? group_n : tiles_n;
    const int blk = r / (rows * gn);
    const int i = r - blk * rows * gn;             // inside the block: rows x (<= gn) tiles
    int n = blk * gn + i / rows;
    if (snake && (band & 1)) n = tiles_n - 1 - n;
    TileCoord c;
    c.m0 = (first_m + i % rows) * BM;
    c.n0 = n * BN;
    return c;
}

// One unit of a CTA pair's work: a whole 256 x 256 tile (half < 0) or the
// 256 x 128 column half `half` of a tile.
struct PairUnit {
    int tile, half;
};

// The units of CTA pair w out of G, in order: whole tiles w, w + G, ...
// below dp_tiles, then half-tile units w, w + G, ... of the remaining tiles.
// A partial last wave of R tiles thus becomes 2R half-tiles spread over the
// pairs (the host splits only when 2R <= G), each worth half a tile.  Every
// role of both CTAs walks the same sequence.
struct PairUnitIter {
    int w, G, D, halves;
    int t, u;
    __device__ PairUnitIter(int w_, int G_, int D_, int num_tiles, int split)
        : w(w_), G(G_), D(D_), halves(split ? 2 * (num_tiles - D_) : 0), t(w_), u(w_) {}
    __device__ bool next(PairUnit& x) {
        if (t < D) {
            x.tile = t;
            x.half = -1;
            t += G;
            return true;
        }
        if (u < halves) {
            x.tile = D + (u >> 1);
            x.half = u & 1;
            u += G;
            return true;
        }
        return false;
    }
};

// EPI: the epilogue kind (p.epi), fixed at compile time so that the
// epilogue warps run one activation with no dispatch.
template <int STAGES, int KSUB, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
gemm_f16_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmParams p) {
    using SP = SmemPlanPair<STAGES, KSUB>;
    constexpr int kStageK = KSUB * kBK;      // K per pipeline stage
    constexpr int PM = 256;                  // pair tile rows = MMA M
    constexpr int BN = 256;                  // pair tile columns = MMA N
    constexpr uint32_t kTmemCols = 2 * BN;   // two accumulators of 256 fp32 columns
    const bool ta = p.trans_a != 0, tb = p.trans_b != 0;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;   // identical in both CTAs of the pair
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
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);      // CTA 0's producer arrives; both CTAs' bytes complete it
            mbar_init(empty_bar(s), 1);     // one multicast MMA commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);      // one multicast MMA commit
            mbar_init(acce_bar(b), 2 * kEpiWarps);   // epilogue warps of both CTAs (used on CTA 0)
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
        tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish_pair();
        tc_fence_before();
    }
    __syncthreads();
    cluster_sync_all();     // both CTAs' barriers exist before any cross-CTA arrive or complete_tx
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // set-up above overlaps the previous kernel; global memory only from here
    grid_dependency_wait();
    grid_launch_dependents();

    const int tiles_m = (p.M + PM - 1) / PM;
    const int tiles_n = (p.N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int kblocks = (p.K + kStageK - 1) / kStageK;   // pipeline stages per tile
    const int cid = blockIdx.x >> 1;
    const int nclusters = gridDim.x >> 1;
    auto units = [&]() { return PairUnitIter(cid, nclusters, p.dp_tiles, num_tiles, p.tail_split); };
    unsigned int* status = &g_status;

    // Boxes each CTA loads for a tile: its A rows unless all are past M (one
    // 128-row K-major box, or, with A stored K x M, those of its two 64-row
    // boxes that start before M), and those of its two 64-column B boxes that
    // start before N.  The skipped ones would only feed accumulator rows /
    // columns that are never stored.
    auto a_boxes = [&](int m0, int r) {
        return ta ? max(0, min(2, (p.M - (m0 + 128 * r) + 63) / 64)) : ((m0 + 128 * r) < p.M ? 1 : 0);
    };
    auto a_bytes = [&](int m0, int r) {
        return static_cast<uint32_t>(a_boxes(m0, r)) * (ta ? kBBoxBytes : kATileBytes);
    };
    auto b_live = [&](int n0, int r) { return max(0, min(2, (p.N - (n0 + 128 * r) + 63) / 64)); };

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            PairUnitIter it = units();
            PairUnit un;
            while (ok && it.next(un)) {
                const TileCoord tc = tile_coord_bm(un.tile, tiles_m, tiles_n, p.group_m, PM, BN, p.group_n, p.snake);
                const int my_a = a_boxes(tc.m0, rank);
                // a whole tile: CTA r loads columns n0 + 128r (two boxes); a half
                // tile h: CTA r loads the one box at n0 + 128h + 64r
                const int bcol = un.half < 0 ? tc.n0 + 128 * static_cast<int>(rank) : tc.n0 + 128 * un.half + 64 * static_cast<int>(rank);
                auto live = [&](int r) {
                    return un.half < 0 ? b_live(tc.n0, r) : (tc.n0 + 128 * un.half + 64 * r < p.N ? 1 : 0);
                };
                const int my_b = live(rank);
                // One instantiation of the tile's load loop per combination of 3-D
                // MN-major operand maps (both 64-wide boxes of a CTA in one load):
                // runtime branches for them inside the loop measured 5-11 % slower on
                // the layouts that do not use them (B stored N x K).
                auto stream_tile = [&](auto a3c, auto b3c) {
                    constexpr bool A3 = decltype(a3c)::value, B3 = decltype(b3c)::value;
                    auto a_load_bytes = [&](int r) {
                        return A3 ? (a_boxes(tc.m0, r) > 0 ? 2u * kBBoxBytes : 0u) : a_bytes(tc.m0, r);
                    };
                    auto b_load_bytes = [&](int r) {
                        return B3 ? (live(r) > 0 ? 2u * kBBoxBytes : 0u) : static_cast<uint32_t>(live(r)) * kBBoxBytes;
                    };
                    // every sub-block's boxes are issued, also those starting past K
                    // (they arrive as zeros), so each stage carries the same bytes
                    const uint32_t pair_bytes =
                        KSUB * (a_load_bytes(0) + a_load_bytes(1) + b_load_bytes(0) + b_load_bytes(1));
                    for (int kb = 0; kb < kblocks; ++kb) {
                        if (!mbar_wait_cluster_bounded(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag, status,
                                                       ROLE_PRODUCER, BAR_EMPTY)) { ok = false; break; }
                        const uint32_t full_leader = mapa_shared(full_bar(stage), 0);
                        if (leader) mbar_arrive_expect_tx(full_bar(stage), pair_bytes);
                        for (int ks = 0; ks < KSUB; ++ks) {
                            const int k0 = kb * kStageK + ks * kBK;
                            const uint32_t a_dst = sA + stage * SP::kAStage + ks * kATileBytes;
                            const int arow = tc.m0 + 128 * static_cast<int>(rank);
                            if (A3) {
                                if (my_a) tma_load_3d_pair(a_dst, &tmA, full_leader, 0, k0, arow >> 6);
                            } else if (ta) {
                                for (int c = 0; c < my_a; ++c)
                                    tma_load_box_pair(a_dst + c * kBBoxBytes, &tmA, full_leader, false, arow + 64 * c, k0);
                            } else if (my_a) {
                                tma_load_2d_pair(a_dst, &tmA, full_leader, k0, arow);
                            }
                            const uint32_t b_dst = sB + stage * SP::kBStage + ks * kBHalfSubBytes;
                            if (B3) {
                                if (my_b) tma_load_3d_pair(b_dst, &tmB, full_leader, 0, k0, bcol >> 6);
                            } else {
                                for (int c = 0; c < my_b; ++c)
                                    tma_load_box_pair(b_dst + c * kBBoxBytes, &tmB, full_leader, tb, bcol + 64 * c, k0);
                            }
                        }
                        ++issued;
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                };
                using T = std::true_type;
                using F = std::false_type;
                if (ta && p.mn3d_a) {
                    if (!tb && p.mn3d_b) stream_tile(T{}, T{});
                    else stream_tile(T{}, F{});
                } else {
                    if (!tb && p.mn3d_b) stream_tile(F{}, T{});
                    else stream_tile(F{}, F{});
                }
            }
            // CTA 0's full barriers count both CTAs' bytes: draining them there
            // covers every load of the pair still in flight.
            if (leader) {
                const int pending = min(issued, STAGES);
                for (int i = 0; i < pending; ++i) {
                    if (--stage < 0) { stage = STAGES - 1; phase ^= 1u; }
                    mbar_wait_cluster_bounded(full_bar(stage), phase, p.timeout_ns, nullptr, status, ROLE_DRAIN,
                                              BAR_FULL);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (CTA 0 only)
        if (leader) {
            const uint32_t idesc_whole = idesc_f16_f32(PM, BN, /*b_mn_major=*/!tb, /*a_mn_major=*/ta);
            const uint32_t idesc_half = idesc_f16_f32(PM, BN / 2, !tb, ta);   // 256 x 128 units
            const uint64_t a_step = desc_step(ta), b_step = desc_step(!tb);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            PairUnitIter it = units();
            PairUnit un;
            while (ok && it.next(un)) {
                if (!mbar_wait_cluster_bounded(acce_bar(acc), acc_phase ^ 1u, p.timeout_ns, abort_flag, status,
                                                    ROLE_MMA, BAR_ACC_EMPTY)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                const uint32_t idesc = un.half < 0 ? idesc_whole : idesc_half;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_cluster_bounded(full_bar(stage), phase, p.timeout_ns, abort_flag, status,
                                                        ROLE_MMA, BAR_FULL)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < KSUB; ++ks) {
                        // same layouts as the single-SM kernel; B here is this
                        // CTA's 128 columns (two 64-column boxes)
                        const uint64_t a_desc = desc_base(sA + stage * SP::kAStage + ks * kATileBytes, ta);
                        const uint64_t b_desc = desc_base(sB + stage * SP::kBStage + ks * kBHalfSubBytes, !tb);
#pragma unroll
                        for (int k = 0; k < kBK / kUMMA_K; ++k)
                            tc_mma_f16_pair(d_tmem, a_desc + k * a_step, b_desc + k * b_step, idesc,
                                            (kb | ks | k) != 0 ? 1u : 0u);
                    }
                    tc_commit_pair_mc(empty_bar(stage), 0x3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit_pair_mc(accf_bar(acc), 0x3);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            tc_commit_pair_mc(drain_bar, 0x1);
            mbar_wait_bounded(drain_bar, 0, p.timeout_ns, nullptr, status, ROLE_DRAIN, BAR_DRAIN);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
        const uint32_t acce_leader1 = mapa_shared(acce_bar(1), 0);
        PairUnitIter it = units();
        PairUnit un;
        while (it.next(un)) {
            const TileCoord tc = tile_coord_bm(un.tile, tiles_m, tiles_n, p.group_m, PM, BN, p.group_n, p.snake);
            const int half = (warp - 2) >> 2;   // which half of the unit's columns this warp takes
            const int ucols = un.half < 0 ? BN : BN / 2;                       // the unit's width
            const int un0 = un.half < 0 ? tc.n0 : tc.n0 + (BN / 2) * un.half;  // its first column
            uint32_t* stage = reinterpret_cast<uint32_t*>(base + SP::kStage + (warp - 2) * kStageWarpBytes);
            if (EPI != EPI_NONE) stage_bias(p, stage + kStageBlockWords, un0 + half * (ucols / 2), ucols / 2);
            const bool ready = mbar_wait_cluster_bounded(accf_bar(acc), acc_phase, p.timeout_ns, abort_flag, status,
                                                         ROLE_EPILOGUE, BAR_ACC_FULL);
            if (!__all_sync(0xffffffffu, ready)) break;
            tc_fence_after();
            const uint32_t t_base = tmem_base + static_cast<uint32_t>(acc * BN + half * (ucols / 2)) +
                                    (static_cast<uint32_t>(32 * q) << 16);
            const int row0 = tc.m0 + 128 * static_cast<int>(rank) + 32 * q;
            if (un.half < 0)
                epilogue_rows_act<BN / 2, EPI, EPI != EPI_NONE>(p, t_base, row0, un0 + half * (BN / 2), stage);
            else
                epilogue_rows_act<BN / 4, EPI, EPI != EPI_NONE>(p, t_base, row0, un0 + half * (BN / 4), stage);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc == 0 ? acce_leader0 : acce_leader1);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    __syncthreads();
    cluster_sync_all();     // the peer no longer touches this CTA's shared or tensor memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}


// ---------------------------------------------------------------- grouped launch

// A unit of a CTA pair's work as a work source hands it out.
struct PairJob {
    const CUtensorMap* tmA;
    const CUtensorMap* tmB;
    int prob;     // which problem (its GemmParams)
    int m0, n0;   // the tile's first row and column
    int half;     // -1: the whole 256 x 256 tile; 0 / 1: its 256 x 128 column half
};

// Independent problems of one grouped launch (at most kMaxGroupProblems, all
// with the same epilogue and operand layouts), passed by value as the kernel
// parameter: their tensor maps, their GemmParams, the prefix sums of their
// 256 x 256 tile counts, and how the concatenated tiles split into whole
// tiles and half tiles (as for one problem: the tiles from dp_tiles on run as
// two 256 x 128 halves when tail_split is set).
constexpr int kMaxGroupProblems = 64;
struct GroupedParams {
    CUtensorMap tmA[kMaxGroupProblems];
    CUtensorMap tmB[kMaxGroupProblems];
    GemmParams prob[kMaxGroupProblems];
    int tile_start[kMaxGroupProblems + 1];
    int count;
    int dp_tiles;
    int tail_split;
};

// Work source of a grouped launch: the concatenated tile lists of all
// problems, strided over the CTA pairs, whole tiles below dp_tiles and then
// (tail_split) half tiles of the rest, in the order PairUnitIter gives one
// problem's units.  Tile indices only grow along the sequence, so the
// problem of each is found by a forward scan of the prefix sums.
struct GroupedPairSource {
    const GroupedParams* gp;
    int t, u, G, g, halves;
    __device__ GroupedPairSource(const GroupedParams* gp_, int cid, int G_)
        : gp(gp_), t(cid), u(cid), G(G_), g(0),
          halves(gp_->tail_split ? 2 * (gp_->tile_start[gp_->count] - gp_->dp_tiles) : 0) {}
    __device__ bool next(PairJob& j) {
        int tile, half;
        if (t < gp->dp_tiles) {
            tile = t;
            half = -1;
            t += G;
        } else if (u < halves) {
            tile = gp->dp_tiles + (u >> 1);
            half = u & 1;
            u += G;
        } else {
            return false;
        }
        while (tile >= gp->tile_start[g + 1]) ++g;
        const GemmParams& q = gp->prob[g];
        const TileCoord tc = tile_coord_bm(tile - gp->tile_start[g], (q.M + 255) / 256, (q.N + 255) / 256, q.group_m,
                                           256, 256);
        j.tmA = &gp->tmA[g];
        j.tmB = &gp->tmB[g];
        j.prob = g;
        j.m0 = tc.m0;
        j.n0 = tc.n0;
        j.half = half;
        return true;
    }
    __device__ const GemmParams& params(int g) const { return gp->prob[g]; }
};

// The CTA-pair GEMM over the units of a work source (the grouped launch).
// `cp` holds the settings every unit shares (epilogue kind, operand
// layouts, wait limit).  Same roles, barriers and layouts as
// gemm_f16_tc2_kernel above, with each unit's operands and parameters taken
// from the source.  The single-problem kernel keeps its own body: routing it
// through this template measured 1-3 % slower on the large squares.
template <int STAGES, int KSUB, int EPI, class Src>
__device__ __forceinline__ void pair_gemm(const Src& src, const GemmParams cp) {

    using SP = SmemPlanPair<STAGES, KSUB>;
    constexpr int kStageK = KSUB * kBK;      // K per pipeline stage
    constexpr int PM = 256;                  // pair tile rows = MMA M
    constexpr int BN = 256;                  // pair tile columns = MMA N
    constexpr uint32_t kTmemCols = 2 * BN;   // two accumulators of 256 fp32 columns
    const bool ta = cp.trans_a != 0, tb = cp.trans_b != 0;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;   // identical in both CTAs of the pair
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
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);      // CTA 0's producer arrives; both CTAs' bytes complete it
            mbar_init(empty_bar(s), 1);     // one multicast MMA commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);      // one multicast MMA commit
            mbar_init(acce_bar(b), 2 * kEpiWarps);   // epilogue warps of both CTAs (used on CTA 0)
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        Src first = src;   // descriptors of this pair's first unit (kernel parameters: no dependency)
        PairJob j;
        if (first.next(j)) {
            tma_prefetch_desc(j.tmA);
            tma_prefetch_desc(j.tmB);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish_pair();
        tc_fence_before();
    }
    __syncthreads();
    cluster_sync_all();     // both CTAs' barriers exist before any cross-CTA arrive or complete_tx
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // set-up above overlaps the previous kernel; global memory only from here
    grid_dependency_wait();
    grid_launch_dependents();

    auto kblocks_of = [&](const GemmParams& q) { return (q.K + kStageK - 1) / kStageK; };   // stages per unit
    unsigned int* status = &g_status;

    // Boxes each CTA loads for a tile: its A rows unless all are past M (one
    // 128-row K-major box, or, with A stored K x M, those of its two 64-row
    // boxes that start before M), and those of its two 64-column B boxes that
    // start before N.  The skipped ones would only feed accumulator rows /
    // columns that are never stored.
    auto a_boxes = [&](int M, int m0, int r) {
        return ta ? max(0, min(2, (M - (m0 + 128 * r) + 63) / 64)) : ((m0 + 128 * r) < M ? 1 : 0);
    };
    auto a_bytes = [&](int M, int m0, int r) {
        return static_cast<uint32_t>(a_boxes(M, m0, r)) * (ta ? kBBoxBytes : kATileBytes);
    };
    auto b_live = [&](int N, int n0, int r) { return max(0, min(2, (N - (n0 + 128 * r) + 63) / 64)); };

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            Src it = src;
            PairJob un;
            while (ok && it.next(un)) {
                const GemmParams pp = it.params(un.prob);   // by value: kept in registers
                const TileCoord tc{un.m0, un.n0};
                const int kblocks = kblocks_of(pp);
                const int my_a = a_boxes(pp.M, tc.m0, rank);
                // a whole tile: CTA r loads columns n0 + 128r (two boxes); a half
                // tile h: CTA r loads the one box at n0 + 128h + 64r
                const int bcol = un.half < 0 ? tc.n0 + 128 * static_cast<int>(rank) : tc.n0 + 128 * un.half + 64 * static_cast<int>(rank);
                auto live = [&](int r) {
                    return un.half < 0 ? b_live(pp.N, tc.n0, r) : (tc.n0 + 128 * un.half + 64 * r < pp.N ? 1 : 0);
                };
                const int my_b = live(rank);
                // one instantiation of the load loop per combination of 3-D MN-major maps
                // (as in gemm_f16_tc2_kernel)
                auto stream_tile = [&](auto a3c, auto b3c) {
                    constexpr bool A3 = decltype(a3c)::value, B3 = decltype(b3c)::value;
                    auto a_load_bytes = [&](int r) {
                        return A3 ? (a_boxes(pp.M, tc.m0, r) > 0 ? 2u * kBBoxBytes : 0u) : a_bytes(pp.M, tc.m0, r);
                    };
                    auto b_load_bytes = [&](int r) {
                        return B3 ? (live(r) > 0 ? 2u * kBBoxBytes : 0u) : static_cast<uint32_t>(live(r)) * kBBoxBytes;
                    };
                    // every sub-block's boxes are issued, also those starting past K
                    // (they arrive as zeros), so each stage carries the same bytes
                    const uint32_t pair_bytes =
                        KSUB * (a_load_bytes(0) + a_load_bytes(1) + b_load_bytes(0) + b_load_bytes(1));
                    for (int kb = 0; kb < kblocks; ++kb) {
                        if (!mbar_wait_cluster_bounded(empty_bar(stage), phase ^ 1u, cp.timeout_ns, abort_flag, status,
                                                       ROLE_PRODUCER, BAR_EMPTY)) { ok = false; break; }
                        const uint32_t full_leader = mapa_shared(full_bar(stage), 0);
                        if (leader) mbar_arrive_expect_tx(full_bar(stage), pair_bytes);
                        for (int ks = 0; ks < KSUB; ++ks) {
                            const int k0 = kb * kStageK + ks * kBK;
                            const uint32_t a_dst = sA + stage * SP::kAStage + ks * kATileBytes;
                            const int arow = tc.m0 + 128 * static_cast<int>(rank);
                            if (A3) {
                                if (my_a) tma_load_3d_pair(a_dst, un.tmA, full_leader, 0, k0, arow >> 6);
                            } else if (ta) {
                                for (int c = 0; c < my_a; ++c)
                                    tma_load_box_pair(a_dst + c * kBBoxBytes, un.tmA, full_leader, false, arow + 64 * c, k0);
                            } else if (my_a) {
                                tma_load_2d_pair(a_dst, un.tmA, full_leader, k0, arow);
                            }
                            const uint32_t b_dst = sB + stage * SP::kBStage + ks * kBHalfSubBytes;
                            if (B3) {
                                if (my_b) tma_load_3d_pair(b_dst, un.tmB, full_leader, 0, k0, bcol >> 6);
                            } else {
                                for (int c = 0; c < my_b; ++c)
                                    tma_load_box_pair(b_dst + c * kBBoxBytes, un.tmB, full_leader, tb, bcol + 64 * c, k0);
                            }
                        }
                        ++issued;
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                };
                using T = std::true_type;
                using F = std::false_type;
                if (ta && pp.mn3d_a) {
                    if (!tb && pp.mn3d_b) stream_tile(T{}, T{});
                    else stream_tile(T{}, F{});
                } else {
                    if (!tb && pp.mn3d_b) stream_tile(F{}, T{});
                    else stream_tile(F{}, F{});
                }
            }
            // CTA 0's full barriers count both CTAs' bytes: draining them there
            // covers every load of the pair still in flight.
            if (leader) {
                const int pending = min(issued, STAGES);
                for (int i = 0; i < pending; ++i) {
                    if (--stage < 0) { stage = STAGES - 1; phase ^= 1u; }
                    mbar_wait_cluster_bounded(full_bar(stage), phase, cp.timeout_ns, nullptr, status, ROLE_DRAIN,
                                              BAR_FULL);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (CTA 0 only)
        if (leader) {
            const uint32_t idesc_whole = idesc_f16_f32(PM, BN, /*b_mn_major=*/!tb, /*a_mn_major=*/ta);
            const uint32_t idesc_half = idesc_f16_f32(PM, BN / 2, !tb, ta);   // 256 x 128 units
            const uint64_t a_step = desc_step(ta), b_step = desc_step(!tb);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            Src it = src;
            PairJob un;
            while (ok && it.next(un)) {
                const int kblocks = kblocks_of(it.params(un.prob));
                if (!mbar_wait_cluster_bounded(acce_bar(acc), acc_phase ^ 1u, cp.timeout_ns, abort_flag, status,
                                                    ROLE_MMA, BAR_ACC_EMPTY)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                const uint32_t idesc = un.half < 0 ? idesc_whole : idesc_half;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_cluster_bounded(full_bar(stage), phase, cp.timeout_ns, abort_flag, status,
                                                        ROLE_MMA, BAR_FULL)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < KSUB; ++ks) {
                        // same layouts as the single-SM kernel; B here is this
                        // CTA's 128 columns (two 64-column boxes)
                        const uint64_t a_desc = desc_base(sA + stage * SP::kAStage + ks * kATileBytes, ta);
                        const uint64_t b_desc = desc_base(sB + stage * SP::kBStage + ks * kBHalfSubBytes, !tb);
#pragma unroll
                        for (int k = 0; k < kBK / kUMMA_K; ++k)
                            tc_mma_f16_pair(d_tmem, a_desc + k * a_step, b_desc + k * b_step, idesc,
                                            (kb | ks | k) != 0 ? 1u : 0u);
                    }
                    tc_commit_pair_mc(empty_bar(stage), 0x3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit_pair_mc(accf_bar(acc), 0x3);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            tc_commit_pair_mc(drain_bar, 0x1);
            mbar_wait_bounded(drain_bar, 0, cp.timeout_ns, nullptr, status, ROLE_DRAIN, BAR_DRAIN);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
        const uint32_t acce_leader1 = mapa_shared(acce_bar(1), 0);
        Src it = src;
        PairJob un;
        while (it.next(un)) {
            const GemmParams pp = it.params(un.prob);   // by value: kept in registers
            const TileCoord tc{un.m0, un.n0};
            const int half = (warp - 2) >> 2;   // which half of the unit's columns this warp takes
            const int ucols = un.half < 0 ? BN : BN / 2;                       // the unit's width
            const int un0 = un.half < 0 ? tc.n0 : tc.n0 + (BN / 2) * un.half;  // its first column
            uint32_t* stage = reinterpret_cast<uint32_t*>(base + SP::kStage + (warp - 2) * kStageWarpBytes);
            if (EPI != EPI_NONE) stage_bias(pp, stage + kStageBlockWords, un0 + half * (ucols / 2), ucols / 2);
            const bool ready = mbar_wait_cluster_bounded(accf_bar(acc), acc_phase, cp.timeout_ns, abort_flag, status,
                                                         ROLE_EPILOGUE, BAR_ACC_FULL);
            if (!__all_sync(0xffffffffu, ready)) break;
            tc_fence_after();
            const uint32_t t_base = tmem_base + static_cast<uint32_t>(acc * BN + half * (ucols / 2)) +
                                    (static_cast<uint32_t>(32 * q) << 16);
            const int row0 = tc.m0 + 128 * static_cast<int>(rank) + 32 * q;
            if (un.half < 0)
                epilogue_rows_act<BN / 2, EPI, EPI != EPI_NONE>(pp, t_base, row0, un0 + half * (BN / 2), stage);
            else
                epilogue_rows_act<BN / 4, EPI, EPI != EPI_NONE>(pp, t_base, row0, un0 + half * (BN / 4), stage);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc == 0 ? acce_leader0 : acce_leader1);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    __syncthreads();
    cluster_sync_all();     // the peer no longer touches this CTA's shared or tensor memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}


// Grouped GEMM: C_g = epilogue(A_g . B_g + bias_g) for every problem g of
// `gp` in one persistent launch.
template <int STAGES, int KSUB, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
gemm_f16_tc2_grouped_kernel(const __grid_constant__ GroupedParams gp) {
    const GroupedPairSource src(&gp, static_cast<int>(blockIdx.x >> 1), static_cast<int>(gridDim.x >> 1));
    pair_gemm<STAGES, KSUB, EPI>(src, gp.prob[0]);
}

}  // namespace gemm_f16_dev
