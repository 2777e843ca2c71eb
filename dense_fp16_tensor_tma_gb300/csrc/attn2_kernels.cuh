// Attention forward, two query tiles per CTA:  O = softmax(scale * Q K^T) V.
//
// The method is that of attn_kernels.cuh ("writing-tilelang-kernels", Flash
// Attention Forward and its Online Softmax pattern; "TileLang: Write,
// Autotune, and Ship Fused Tensor-Core Kernels from Python", FlashAttention:
// the FLOP model): blocks of 128 query rows, key blocks of 128 streamed
// through shared memory, the running maximum and sum kept online, the S x S
// scores never written to memory.  What differs is the schedule.  With one
// query tile per CTA the tensor core waits for each block's softmax and the
// softmax for each block's MMAs.  Here a CTA takes a unit of two adjacent
// query tiles, A and B, of one head (or, for a tail of the work, tile A
// alone); both read the K and V blocks loaded for the unit (half the K/V
// traffic per query row; causal: tile B reads one block more than A), each
// has one score buffer and one output in tensor memory, and the MMA warp
// issues
//
//     S_A(0) S_B(0) | P_A(0)V S_A(1) | P_B(0)V S_B(1) | P_A(1)V S_A(2) | ...
//
// so the tensor core computes one tile's P V and next scores while the other
// tile's softmax warps work.  Each softmax warp owns 32 whole rows of its
// tile (one TMEM lane quarter): a thread reads all 128 scores of its row's
// block into registers once, takes the exact block maximum before any
// exponential (no partner warp, no exchange), and writes its row's P (fp16,
// 64 columns) over the first half of its row's score columns, after it has
// read them; S of the next block overwrites the buffer only after the P V
// that reads that P, both issued by the MMA warp, whose MMAs the tensor pipe
// executes in issue order.  (Two warps per row, 64 keys each, exchanging
// their block maxima through shared memory with P computed speculatively
// meanwhile, measured the same at D = 128 and 2-4 % slower elsewhere.)
//
// Roles: warp 0 lane 0 loads each unit's Q tiles and the K blocks, lane 1
// the V blocks (two-slot rings; a slot is free once the last MMA reading the
// block two back has completed: tile B's, issued after A's, or tile A's in a
// one-tile unit); warp 1
// allocates tensor memory and issues every MMA (the whole warp runs the
// loop, one lane elected per instruction: tc_mma_f16); warps 2..5 run tile
// A's softmax, warps 6..9 tile B's (one warp per TMEM lane quarter); 320
// threads leave 168 registers per thread.  Every wait is bounded.
#pragma once

#include "attn_kernels.cuh"

namespace attn_dev {

constexpr int kAttn2Threads = 320;   // producer, MMA, 2 x 4 softmax warps

// Units of the two-tile kernels.  Non-causal: a head's query tiles form pairs
// (2k, 2k + 1), numbered head-major; unit u below pair_units holds pair u, each
// later unit one tile (A alone): first the tiles of the pairs not taken as
// pairs, then, with an odd number of tiles per head, each head's last tile.
// The host takes the pairs in whole rounds over the CTAs and leaves the rest
// as one-tile units when they fit one per CTA (13 pairs and a single rather
// than 14 pairs on some CTAs).  Causal: units of tiles 2k and 2k + 1 of one head; tile
// A reads key blocks 0..2k, tile B 0..2k + 1 (every block the unit loads); a
// CTA takes them two at a time from one head, pair np - 1 - m and then pair m
// (np pairs per head, even: the host launches causal problems here only with a
// multiple of 4 query tiles per head), so every such step costs the same.
// Units in flight share a few heads, whose K and V stay in L2.
struct UnitWalk {
    int U, i;                                   // step (unit) index, unit within a causal step
    // the next unit: head, tile A's index, key blocks of A and of B (0: A alone);
    // nblk key blocks per tile (non-causal), np pairs and sp causal steps per head
    __device__ bool next(const AttnParams& p, int nblk, int np, int sp, int& bh, int& qa, int& na, int& nb) {
        if (U >= p.units) return false;
        if (!p.causal) {
            const int u = U;
            U += static_cast<int>(gridDim.x);
            const int pph = p.nq >> 1;                  // pairs (2k, 2k + 1) per head
            na = nblk;
            if (u < p.pair_units) {                     // pair u
                bh = u / pph;
                qa = 2 * (u - bh * pph);
                nb = nblk;
                return true;
            }
            // the tiles of the pairs not taken as pairs, then (odd nq) each
            // head's last tile
            nb = 0;
            const int s = u - p.pair_units;
            const int split = 2 * (p.BH * pph - p.pair_units);
            if (s < split) {
                const int pi = p.pair_units + (s >> 1);
                bh = pi / pph;
                qa = 2 * (pi - bh * pph) + (s & 1);
            } else {
                bh = s - split;
                qa = p.nq - 1;
            }
            return true;
        }
        bh = U / sp;
        const int m = U - bh * sp;
        int k;
        if (i == 0) {
            k = np - 1 - m;
            i = 1;
        } else {
            k = m;
            i = 0;
            U += static_cast<int>(gridDim.x);
        }
        qa = 2 * k;
        na = 2 * k + 1;
        nb = 2 * k + 2;
        return true;
    }
};

template <int D>
struct Attn2Smem {
    static constexpr uint32_t kTile = (D / 64) * kBox;     // one 128-row tile of Q, K or V
    // D = 64: a V slot is the block's 64 columns and then a box of fp16 ones,
    // columns 64.. of the P V operand, so O's column 64 accumulates the row sum
    static constexpr uint32_t kVSlot = D == 64 ? 2 * kBox : kTile;
    static constexpr uint32_t kQ = 0;                        // Q_A, Q_B
    static constexpr uint32_t kK = kQ + 2 * kTile;           // 2 slots
    static constexpr uint32_t kV = kK + 2 * kTile;           // 2 slots
    static constexpr uint32_t kBars = kV + 2 * kVSlot;
    // q_full, k_full[2], v_full[2], s_full[2 tiles][2], p_full[2], pv_done[2][2], o_free[2], drain
    static constexpr uint32_t kNumBars = 1 + 2 + 2 + 4 + 2 + 4 + 2 + 1;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kEnd = kAbort + 4;
    static constexpr uint32_t kNeed = kEnd + 1024;           // + alignment of the swizzled tiles
    // one CTA per SM: it allocates all 512 tensor-memory columns
    static constexpr uint32_t kOnePerSm = 120 * 1024;
    static constexpr uint32_t kDynamicBytes = kNeed > kOnePerSm ? kNeed : kOnePerSm;
    static_assert(kDynamicBytes <= kMaxDynSmem, "shared memory plan too large");
};

template <int D>
__global__ void __launch_bounds__(kAttn2Threads, 1)
attn_f16_fwd2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    static_assert(D == 64 || D == 128, "head dimension 64 or 128");
    using SM = Attn2Smem<D>;
    constexpr int kDB = D / 64;
    constexpr uint32_t kTileBytes = SM::kTile;
    // D = 64: the P V MMA also multiplies P by a column of ones (N = 80), so the
    // tensor core sums each row's fp16 P into O's column 64 in fp32, rescaled
    // with O; D = 128 leaves no tensor-memory columns for it and the softmax
    // warps sum P themselves
    constexpr bool kSumByMma = D == 64;
    constexpr int kON = kSumByMma ? D + 16 : D;
    constexpr uint32_t kIdescS = idesc_f16_f32(kQRows, kKeys, /*b_mn_major=*/false);
    constexpr uint32_t kIdescO = idesc_f16_f32(kQRows, kON, /*b_mn_major=*/true);
    constexpr uint32_t kSCol = 0;             // S_A at 0, S_B at 128
    constexpr uint32_t kOCol2 = 256;          // O_A at 256, O_B at 384 (kON <= 128 columns each)

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
    const uint32_t sQ = base_s + SM::kQ, sK = base_s + SM::kK, sV = base_s + SM::kV;
    const uint32_t bars = base_s + SM::kBars;
    const uint32_t q_full = bars;
    auto k_full = [&](int s) { return bars + 8u * (1 + s); };
    auto v_full = [&](int s) { return bars + 8u * (3 + s); };
    auto s_full = [&](int t, int s) { return bars + 8u * (5 + 2 * t + s); };    // S of tile t, block parity s
    auto p_full = [&](int t) { return bars + 8u * (9 + t); };                   // P of tile t written
    auto pv_done = [&](int t, int s) { return bars + 8u * (11 + 2 * t + s); };  // P V of tile t completed
    auto o_free = [&](int t) { return bars + 8u * (15 + t); };                  // tile t's output read out
    const uint32_t drain_bar = bars + 8u * 17;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + SM::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + SM::kAbort);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int nblk = (p.S + kKeys - 1) / kKeys;    // key blocks per tile, non-causal
    const int np = p.nq >> 1;                       // pairs per head
    const int sp = np >> 1;                         // causal steps per head

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(v_full(s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            for (int s = 0; s < 2; ++s) {
                mbar_init(s_full(t, s), 1);
                mbar_init(pv_done(t, s), 1);
            }
            mbar_init(p_full(t), 4);
            mbar_init(o_free(t), 4);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if constexpr (kSumByMma) {
        // the boxes of ones after each V slot, written once; never loaded over
        for (int s = 0; s < 2; ++s) {
            uint4* ones = reinterpret_cast<uint4*>(base + SM::kV + s * SM::kVSlot + kBox);
            for (int i = threadIdx.x; i < static_cast<int>(kBox / 16); i += kAttn2Threads)
                ones[i] = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);   // fp16 1.0
        }
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();      // set-up above overlaps the previous kernel
    grid_launch_dependents();
    unsigned int* status = &g_attn_status;

    // Key blocks loaded are numbered g = 0, 1, ... over all of this CTA's units:
    // block g uses ring slot g & 1 and phase (g >> 1) & 1 of the ring barriers.
    // Each tile numbers the blocks it reads (A fewer than loaded in causal
    // units): its block b uses phase (b >> 1) & 1 of its s_full(t, b & 1) and
    // pv_done(t, b & 1), phase b & 1 of p_full(t).  Unit n uses phase n & 1 of
    // q_full, each tile's own unit count the phases of its o_free.
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane < 2) {
            const bool is_k = lane == 0;
            const CUtensorMap* tm = is_k ? &tmK : &tmV;
            const uint32_t ring = is_k ? sK : sV;
            const uint32_t slot_bytes = is_k ? kTileBytes : SM::kVSlot;
            const uint32_t which = is_k ? BAR_K : BAR_V;
            bool ok = true;
            int g = 0, nu = 0, issued = 0;
            int pair_end = 0;            // key blocks of the two-tile units so far (they come first)
            bool prev_two = true;
            UnitWalk walk{static_cast<int>(blockIdx.x), 0};
            int bh, qa, na, nb;
            while (ok && walk.next(p, nblk, np, sp, bh, qa, na, nb)) {
                const bool two = nb > 0;
                const int nr = two ? nb : na;   // blocks loaded: all of B's (B reads every one), or A's
                if (is_k) {
                    // the Q tiles are operands of every S of the previous unit: reload
                    // once the last of those (tile B's, issued last, or tile A's in a
                    // one-tile unit) has completed
                    if (g > 0 && !mbar_wait_bounded(s_full(prev_two ? 1 : 0, (g - 1) & 1), ((g - 1) >> 1) & 1,
                                                    p.timeout_ns, abort_flag, status, ROLE_PRODUCER, BAR_Q))
                        break;
                    const int ntiles = two ? 2 : 1;
                    mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(ntiles) * kTileBytes);
                    for (int t = 0; t < ntiles; ++t)
                        for (int c = 0; c < kDB; ++c)
                            tma_load_3d(sQ + t * kTileBytes + c * kBox, &tmQ, q_full, 64 * c, (qa + t) * kQRows, bh);
                }
                ++nu;
                if (two) pair_end = g + nr;
                prev_two = two;
                for (int j = 0; j < nr; ++j) {
                    const int gb = g + j;
                    const int s = gb & 1;
                    // slot s is free once the last MMA reading block gb - 2 completed:
                    // tile B's S (for K) or P V (for V) in a two-tile unit (tile A's
                    // were issued before it), tile A's in a one-tile unit.  Tile B
                    // reads every block of a two-tile unit and the two-tile units come
                    // first, so B's count of that block is gb - 2; one-tile units
                    // come only without causal masking, where A reads every block.
                    const int tb = gb - 2 < pair_end ? 1 : 0;
                    const uint32_t empty = is_k ? s_full(tb, s) : pv_done(tb, s);
                    if (!mbar_wait_bounded(empty, static_cast<uint32_t>((gb >> 1) & 1) ^ 1u, p.timeout_ns,
                                           abort_flag, status, ROLE_PRODUCER, which)) {
                        ok = false;
                        break;
                    }
                    if (is_k && gb == p.fault_skip_block) continue;   // injected fault: never loaded
                    const uint32_t full = is_k ? k_full(s) : v_full(s);
                    mbar_arrive_expect_tx(full, kTileBytes);
                    for (int c = 0; c < kDB; ++c)
                        tma_load_3d(ring + s * slot_bytes + c * kBox, tm, full, 64 * c, j * kKeys, bh);
                    issued = gb + 1;
                }
                g += nr;
            }
            // every issued load lands before the CTA can exit (the last Q pair and the
            // last one or two blocks of each ring; earlier ones were waited for by the
            // MMA thread before it issued what freed their slots)
            if (is_k && nu > 0)
                mbar_wait_bounded(q_full, (nu - 1) & 1, p.timeout_ns, nullptr, status, ROLE_DRAIN, BAR_Q);
            for (int gb = max(0, issued - 2); gb < issued; ++gb)
                mbar_wait_bounded(is_k ? k_full(gb & 1) : v_full(gb & 1), (gb >> 1) & 1, p.timeout_ns, nullptr,
                                  status, ROLE_DRAIN, which);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        {
            const uint64_t k_desc = smem_desc_sw128(sK, 0, 1024);
            const uint64_t v_desc = smem_desc_sw128(sV, kBox, 1024);   // MN-major: 64-column boxes kBox apart
            constexpr uint32_t kSlotUnits = kTileBytes >> 4;
            constexpr uint32_t kVSlotUnits = SM::kVSlot >> 4;
            // S_t of loaded block rb (tile t's block tb) = Q_t K^T into t's score buffer
            auto issue_s = [&](int t, int rb, int tb) -> bool {
                const int s = rb & 1;
                if (!mbar_wait_bounded(k_full(s), (rb >> 1) & 1, p.timeout_ns, abort_flag, status, ROLE_MMA, BAR_K))
                    return false;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + kSCol + static_cast<uint32_t>(t * kKeys);
                const uint64_t qd = smem_desc_sw128(sQ + t * kTileBytes, 0, 1024);
                const uint64_t kd = k_desc + static_cast<uint64_t>(s * kSlotUnits);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t off = static_cast<uint64_t>(((k >> 2) * kBox + (k & 3) * 32) >> 4);
                    tc_mma_f16(d_tmem, qd + off, kd + off, kIdescS, k != 0 ? 1u : 0u);
                }
                tc_commit(s_full(t, tb & 1));
                return true;
            };
            // O_t += P_t V of loaded block rb (tile t's block tb; j: its index in the
            // unit, nu: the tile's earlier units)
            auto issue_pv = [&](int t, int rb, int tb, int j, int nu) -> bool {
                const int s = rb & 1;
                if (!mbar_wait_bounded(p_full(t), tb & 1, p.timeout_ns, abort_flag, status, ROLE_MMA, BAR_P))
                    return false;
                // the unit's first P V overwrites O_t: the previous unit's output must be read out
                if (j == 0 && nu > 0 &&
                    !mbar_wait_bounded(o_free(t), (nu - 1) & 1, p.timeout_ns, abort_flag, status, ROLE_MMA, BAR_P))
                    return false;
                if (!mbar_wait_bounded(v_full(s), (rb >> 1) & 1, p.timeout_ns, abort_flag, status, ROLE_MMA, BAR_V))
                    return false;
                tc_fence_after();
                const uint32_t o_tmem = tmem_base + kOCol2 + static_cast<uint32_t>(t * 128);
                const uint32_t pa = tmem_base + kSCol + static_cast<uint32_t>(t * kKeys);
                const uint64_t vd = v_desc + static_cast<uint64_t>(s * kVSlotUnits);
#pragma unroll
                for (int k = 0; k < kKeys / 16; ++k) {
                    // keys 16k..: P at columns 8k .. 8k + 7 of the tile's score buffer
                    const uint32_t pcol = static_cast<uint32_t>(k * 8);
                    tc_mma_f16_ta(o_tmem, pa + pcol, vd + static_cast<uint64_t>(k * 2048 >> 4), kIdescO,
                                  (j | k) != 0 ? 1u : 0u);
                }
                tc_commit(pv_done(t, tb & 1));
                return true;
            };
            bool ok = true;
            int g = 0, gA = 0, gB = 0;   // blocks loaded; blocks tile A and tile B read
            int nu = 0, nuB = 0;         // units; units with a tile B
            UnitWalk walk{static_cast<int>(blockIdx.x), 0};
            int bh, qa, na, nb;
            while (ok && walk.next(p, nblk, np, sp, bh, qa, na, nb)) {
                const int nr = nb > 0 ? nb : na;
                ok = mbar_wait_bounded(q_full, nu & 1, p.timeout_ns, abort_flag, status, ROLE_MMA, BAR_Q);
                if (ok) {
                    tc_fence_after();
                    ok = issue_s(0, g, gA) && (nb == 0 || issue_s(1, g, gB));
                }
                // S of a tile's next block overwrites its buffer after the P V just
                // issued has read its P: the pipe runs them in order.  In a causal
                // unit tile A has no last block.
                for (int j = 0; ok && j < nr; ++j) {
                    if (j < na) {
                        ok = issue_pv(0, g + j, gA + j, j, nu);
                        if (ok && j + 1 < na) ok = issue_s(0, g + j + 1, gA + j + 1);
                    }
                    if (ok && j < nb) {
                        ok = issue_pv(1, g + j, gB + j, j, nuB);
                        if (ok && j + 1 < nb) ok = issue_s(1, g + j + 1, gB + j + 1);
                    }
                }
                g += nr;
                gA += na;
                gB += nb;
                ++nu;
                nuB += nb > 0 ? 1 : 0;
            }
            tc_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, p.timeout_ns, nullptr, status, ROLE_DRAIN, BAR_DRAIN);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + output
        const int t = (warp - 2) >> 2;               // query tile A (0) or B (1)
        const int quarter = warp & 3;                // TMEM lanes 32 * quarter ..: this warp's rows
        const int r = 32 * quarter + lane;           // this thread's row of the tile
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16);
        const uint32_t s_cols = lane_base + kSCol + static_cast<uint32_t>(t * kKeys);
        const uint32_t o_cols = lane_base + kOCol2 + static_cast<uint32_t>(t * 128);
        const bool pos = p.scale_log2 >= 0.0f;
        const uint32_t lose = __float_as_uint(pos ? -INFINITY : INFINITY);
        bool ok = true;
        int g = 0;
        UnitWalk walk{static_cast<int>(blockIdx.x), 0};
        int bh, qa, na, nb;
        while (ok && walk.next(p, nblk, np, sp, bh, qa, na, nb)) {
            if (t == 1 && nb == 0) break;                 // tile B's warps sit out the one-tile units
            const int n = t == 0 ? na : nb;               // key blocks this tile reads
            const int q = (qa + t) * kQRows + r;          // this thread's query index
            // keys past S, and (causal) keys after this query, do not count
            const int key_end = p.causal ? min(p.S, q + 1) : p.S;
            float m = -INFINITY, l = 0.0f;
            for (int j = 0; j < n; ++j) {
                const int gb = g + j;                     // this tile's block number
                const int k0 = j * kKeys;
                ok = mbar_wait_bounded(s_full(t, gb & 1), (gb >> 1) & 1, p.timeout_ns, abort_flag, status,
                                       ROLE_SOFTMAX, BAR_S);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                // the row's 128 scores of the block, all in registers
                uint32_t v[128];
                tmem_ld_32x32b_x128(s_cols, v);   // one load: four 32-column loads took longer
                tmem_wait_ld(v);
                if (k0 + kKeys > p.S || (p.causal && j == n - 1)) {
                    const int key_lim = key_end - k0;         // valid: column < key_lim
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (i >= key_lim) v[i] = lose;
                }
                float bm[4];
                bm[0] = bm[1] = bm[2] = bm[3] = pos ? -INFINITY : INFINITY;
                if (pos) {
#pragma unroll
                    for (int i = 0; i < 128; i += 2)
                        bm[(i >> 1) & 3] = max3f(bm[(i >> 1) & 3], __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
                } else {
#pragma unroll
                    for (int i = 0; i < 128; i += 2)
                        bm[(i >> 1) & 3] = min3f(bm[(i >> 1) & 3], __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
                }
                float bmax = pos ? fmaxf(fmaxf(bm[0], bm[1]), fmaxf(bm[2], bm[3]))
                                 : fminf(fminf(bm[0], bm[1]), fminf(bm[2], bm[3]));
                bmax *= p.scale_log2;
                float m_new = m;
                bool raise = false;
                if (bmax > m + kRaise || m == -INFINITY) {
                    m_new = fmaxf(m, bmax);
                    raise = m != -INFINITY && m_new != m;
                }
                // P = 2^(x * scale_log2 - m) as fp16 over the first 64 of the row's
                // score columns (keys 32c .. 32c + 31 into columns 16c ..), and (D =
                // 128) its sum over the fp16 values the tensor core multiplies
                const float mm = (m_new == -INFINITY) ? 0.0f : m_new;
                float rs0 = 0.0f, rs1 = 0.0f;
                // P written 32 columns (keys 64 c2 ..) at a time: one 64-column store
                // after the whole pass measured 1 % faster non-causal and 3 % slower
                // causal, four 16-column stores 1-2 % slower than this
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t h2[32];
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int c = 2 * c2 + cc;
                        uint32_t (&h)[16] = *reinterpret_cast<uint32_t(*)[16]>(h2 + 16 * cc);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float2 xs = fma2_bc(__uint_as_float(v[32 * c + 2 * i]),
                                                      __uint_as_float(v[32 * c + 2 * i + 1]), p.scale_log2, -mm);
                            const __half2 hv = __floats2half2_rn(fast_exp2(xs.x), fast_exp2(xs.y));
                            h[i] = *reinterpret_cast<const uint32_t*>(&hv);
                            if constexpr (!kSumByMma) {
                                if (i & 1) rs1 = add_f16x2_to_f32(rs1, h[i]);
                                else rs0 = add_f16x2_to_f32(rs0, h[i]);
                            }
                        }
                    }
                    tmem_st_32x32b_x32(s_cols + 32u * c2, h2);
                }
                // O rescaled (a raise needs an earlier block of the unit) after the
                // tile's previous P V has completed
                if (__any_sync(0xffffffffu, raise)) {
                    ok = mbar_wait_bounded(pv_done(t, (gb - 1) & 1), ((gb - 1) >> 1) & 1, p.timeout_ns, abort_flag,
                                           status, ROLE_SOFTMAX, BAR_PV);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                    const float alpha = raise ? fast_exp2(m - m_new) : 1.0f;
                    l *= alpha;
                    // D = 64: columns 64..95, the row sum among them
#pragma unroll 1
                    for (int c = 0; c < (kSumByMma ? D / 32 + 1 : D / 32); ++c) {
                        uint32_t w[32];
                        tmem_ld_32x32b_x32(o_cols + 32u * c, w);
                        tmem_wait_ld(w);
#pragma unroll
                        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha);
                        tmem_st_32x32b_x32(o_cols + 32u * c, w);
                    }
                }
                m = m_new;
                if constexpr (!kSumByMma) l += rs0 + rs1;
                tmem_wait_st();
                tc_fence_before();           // P and the O rescale, if any, before the signal
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(t));
            }
            if (!ok) break;
            // output: O / l after the unit's last P V of this tile; O read into
            // registers and its tensor memory released before the stores
            const int gl = g + n - 1;
            ok = mbar_wait_bounded(pv_done(t, gl & 1), (gl >> 1) & 1, p.timeout_ns, abort_flag, status,
                                   ROLE_SOFTMAX, BAR_PV);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            uint32_t w[D];
            tmem_ld_row<D>(o_cols, w);
            uint32_t lw[16];
            if constexpr (kSumByMma) tmem_ld_32x32b_x16(o_cols + D, lw);
            tmem_wait_ld(w);
            if constexpr (kSumByMma) {
                tmem_wait_ld(lw);
                l = __uint_as_float(lw[0]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free(t));
            const float inv = 1.0f / l;
            if (q < p.S) {
                uint4* dst = reinterpret_cast<uint4*>(p.O + (static_cast<int64_t>(bh) * p.S + q) * D);
#pragma unroll
                for (int i = 0; i < D / 8; ++i) {
                    uint32_t hh[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __half2 hv = __floats2half2_rn(__uint_as_float(w[8 * i + 2 * e]) * inv,
                                                             __uint_as_float(w[8 * i + 2 * e + 1]) * inv);
                        hh[e] = *reinterpret_cast<const uint32_t*>(&hv);
                    }
                    dst[i] = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                }
            }
            g += n;
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace attn_dev
