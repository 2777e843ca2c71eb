// Attention forward at head dimension 64, two query tiles per CTA, each tile's
// P in a tensor-memory buffer of its own:  O = softmax(scale * Q K^T) V.
//
// What it computes and the units it walks are those of attn_f16_fwd2_kernel
// ("writing-tilelang-kernels", Flash Attention Forward and its Online Softmax
// pattern; the FLOP model of "TileLang: Write, Autotune, and Ship Fused
// Tensor-Core Kernels from Python", FlashAttention).  What differs is the
// schedule.  There P is written over its tile's scores, so S of the next key
// block can only start once P V has read that P: each tile runs softmax, then
// its own MMAs, then softmax again, and at D = 64 the other tile's MMAs
// (about 600 cycles a block) are too short to cover a softmax.  Here the
// score buffer is free as soon as the tile's softmax warps have read S into
// registers (they arrive on s_free): the MMA warp then issues S of the next
// block, which runs on the tensor core while they compute P of this block.
// A softmax warp writes P only once P V of the previous block, which reads
// the P buffer, has completed (pv_done).  Tensor memory: S_A, S_B at columns
// 0 and 128, P_A, P_B (fp16 pairs) at 256 and 320, O_A, O_B at 384 and 448:
// all 512 columns, which is why this schedule is for D = 64 only.
//
// Each tile has an MMA warp of its own (warps 1 and 2): one warp issuing all
// 24 MMAs of a block pair spent most of its time issuing (about 75 cycles an
// MMA with its commits) and held back the other tile's next P V.  Per block a
// tile's warp issues S of the next block (once the softmax has read this
// block's) and then P V of this block; the tensor pipe runs each warp's MMAs
// in order and may interleave the two warps'.  K and V blocks sit in rings of
// three slots.  A commit covers only its own warp's MMAs, so a slot's k_empty
// / v_empty barrier and the Q tiles' q_empty take one commit from each tile's
// warp after its last MMA reading them; in a one-tile unit tile A's warp
// commits twice, and in a causal unit, whose last block tile A does not read,
// tile A's warp arrives for that block once it has landed (earlier, the
// arrival could count toward the slot's previous block).  A unit's first P V
// overwrites O without a barrier of its own: each softmax warp arrives on
// p_full of the unit's first block only after it has read the previous
// unit's O out.  The protocol (every wait's
// phase, no deadlock, no write over data still to be read, planted defects
// caught) is checked by a CPU model in tests/test_attn3_protocol_cpu.py.
//
// Every wait is bounded (globaltimer); on a timeout or an abort raised by
// another role the CTA records the role and barrier in g_attn_status, drains
// what it issued and frees its tensor memory.
#pragma once

#include "attn2_kernels.cuh"

namespace attn_dev {

constexpr int kAttn3Stages = 3;
constexpr int kAttn3Threads = 352;   // producer, two MMA warps, 2 x 4 softmax warps

template <int D>
struct Attn3Smem {
    static constexpr uint32_t kTile = (D / 64) * kBox;     // one 128-row tile of Q, K or V
    static constexpr uint32_t kQ = 0;                        // Q_A, Q_B
    static constexpr uint32_t kK = kQ + 2 * kTile;           // kAttn3Stages slots
    static constexpr uint32_t kV = kK + kAttn3Stages * kTile;
    static constexpr uint32_t kBars = kV + kAttn3Stages * kTile;
    // q_full, q_empty, k_full[3], k_empty[3], v_full[3], v_empty[3],
    // s_full[2], s_free[2], p_full[2], pv_done[2], drain
    static constexpr uint32_t kNumBars = 2 + 4 * kAttn3Stages + 4 * 2 + 1;
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
__global__ void __launch_bounds__(kAttn3Threads, 1)
attn_f16_fwd3_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    static_assert(D == 64, "separate P buffers leave tensor memory for D = 64 only");
    using SM = Attn3Smem<D>;
    constexpr int kSt = kAttn3Stages;
    constexpr uint32_t kTileBytes = SM::kTile;
    constexpr uint32_t kIdescS = idesc_f16_f32(kQRows, kKeys, /*b_mn_major=*/false);
    constexpr uint32_t kIdescO = idesc_f16_f32(kQRows, D, /*b_mn_major=*/true);
    constexpr uint32_t kSCol = 0;             // S_t at 128 t
    constexpr uint32_t kPCol = 256;           // P_t at 256 + 64 t
    constexpr uint32_t kOCol = 384;           // O_t at 384 + 64 t

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
    const uint32_t sQ = base_s + SM::kQ, sK = base_s + SM::kK, sV = base_s + SM::kV;
    const uint32_t bars = base_s + SM::kBars;
    const uint32_t q_full = bars, q_empty = bars + 8u;
    auto k_full = [&](int s) { return bars + 8u * (2 + s); };
    auto k_empty = [&](int s) { return bars + 8u * (2 + kSt + s); };
    auto v_full = [&](int s) { return bars + 8u * (2 + 2 * kSt + s); };
    auto v_empty = [&](int s) { return bars + 8u * (2 + 3 * kSt + s); };
    auto s_full = [&](int t) { return bars + 8u * (2 + 4 * kSt + t); };       // S of tile t landed
    auto s_free = [&](int t) { return bars + 8u * (4 + 4 * kSt + t); };       // S of tile t read out
    auto p_full = [&](int t) { return bars + 8u * (6 + 4 * kSt + t); };       // P of tile t written
    auto pv_done = [&](int t) { return bars + 8u * (8 + 4 * kSt + t); };      // P V of tile t completed
    const uint32_t drain_bar = bars + 8u * (10 + 4 * kSt);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + SM::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + SM::kAbort);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nblk = (p.S + kKeys - 1) / kKeys;    // key blocks per tile, non-causal
    const int np = p.nq >> 1;                       // pairs per head
    const int sp = np >> 1;                         // causal steps per head

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 2);                       // one commit from each tile's MMA warp
        for (int s = 0; s < kSt; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 2);
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 2);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(s_full(t), 1);
            mbar_init(s_free(t), 4);
            mbar_init(p_full(t), 4);
            mbar_init(pv_done(t), 1);
        }
        mbar_init(drain_bar, 2);
        *abort_flag = 0;
        fence_mbarrier_init();
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
    // block g uses ring slot g % 3 and phase (g / 3) & 1 of its full and empty
    // barriers.  Each tile numbers the blocks it reads (A fewer than loaded in
    // causal units): its block b uses phase b & 1 of s_full, s_free, p_full and
    // pv_done.  Unit n uses phase n & 1 of q_full and q_empty.
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane < 2) {
            const bool is_k = lane == 0;
            const CUtensorMap* tm = is_k ? &tmK : &tmV;
            const uint32_t ring = is_k ? sK : sV;
            const uint32_t which = is_k ? BAR_K : BAR_V;
            bool ok = true;
            int g = 0, nu = 0, issued = 0;
            UnitWalk walk{static_cast<int>(blockIdx.x), 0};
            int bh, qa, na, nb;
            while (ok && walk.next(p, nblk, np, sp, bh, qa, na, nb)) {
                const int nr = nb > 0 ? nb : na;   // blocks loaded: all of B's (B reads every one), or A's
                if (is_k) {
                    // the previous unit's last S has read the Q tiles
                    if (nu > 0 && !mbar_wait_bounded(q_empty, (nu - 1) & 1, p.timeout_ns, abort_flag, status,
                                                     ROLE_PRODUCER, BAR_Q))
                        break;
                    const int ntiles = nb > 0 ? 2 : 1;
                    mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(ntiles) * kTileBytes);
                    for (int t = 0; t < ntiles; ++t)
                        tma_load_3d(sQ + t * kTileBytes, &tmQ, q_full, 0, (qa + t) * kQRows, bh);
                }
                ++nu;
                for (int j = 0; j < nr; ++j) {
                    const int gb = g + j;
                    const int s = gb % kSt;
                    if (gb >= kSt && !mbar_wait_bounded(is_k ? k_empty(s) : v_empty(s),
                                                        static_cast<uint32_t>((gb / kSt - 1) & 1), p.timeout_ns,
                                                        abort_flag, status, ROLE_PRODUCER, which)) {
                        ok = false;
                        break;
                    }
                    if (is_k && gb == p.fault_skip_block) continue;   // injected fault: never loaded
                    const uint32_t full = is_k ? k_full(s) : v_full(s);
                    mbar_arrive_expect_tx(full, kTileBytes);
                    tma_load_3d(ring + s * kTileBytes, tm, full, 0, j * kKeys, bh);
                    issued = gb + 1;
                }
                g += nr;
            }
            // every issued load lands before the CTA can exit (the last Q tiles
            // and the last three blocks of each ring; earlier ones were read by
            // MMAs whose completion freed their slots)
            if (is_k && nu > 0)
                mbar_wait_bounded(q_full, (nu - 1) & 1, p.timeout_ns, nullptr, status, ROLE_DRAIN, BAR_Q);
            for (int gb = max(0, issued - kSt); gb < issued; ++gb)
                mbar_wait_bounded(is_k ? k_full(gb % kSt) : v_full(gb % kSt), (gb / kSt) & 1, p.timeout_ns, nullptr,
                                  status, ROLE_DRAIN, which);
        }
        __syncwarp();
    } else if (warp <= 2) {
        // ------------------------------------------------------------ MMA issuers, one per tile
        {
            const int t = warp - 1;
            const uint64_t k_desc = smem_desc_sw128(sK, 0, 1024);
            const uint64_t v_desc = smem_desc_sw128(sV, kBox, 1024);   // MN-major, one 64-column box
            const uint64_t qd = smem_desc_sw128(sQ + t * kTileBytes, 0, 1024);
            const uint32_t s_tmem = tmem_base + kSCol + static_cast<uint32_t>(t * kKeys);
            const uint32_t o_tmem = tmem_base + kOCol + static_cast<uint32_t>(t * D);
            const uint32_t pa = tmem_base + kPCol + static_cast<uint32_t>(t * (kKeys / 2));
            constexpr uint32_t kSlotUnits = kTileBytes >> 4;
            // S_t of loaded block rb = Q_t K^T into the tile's score buffer; the
            // commits free the K slot and, after the tile's last S of the unit, the
            // Q tiles (reps: 2 in a one-tile unit, arriving for tile B's warp too)
            auto issue_s = [&](int rb, bool last_s, int reps) -> bool {
                const int s = rb % kSt;
                if (!mbar_wait_bounded(k_full(s), (rb / kSt) & 1, p.timeout_ns, abort_flag, status, ROLE_MMA, BAR_K))
                    return false;
                tc_fence_after();
                const uint64_t kd = k_desc + static_cast<uint64_t>(s * kSlotUnits);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t off = static_cast<uint64_t>((k * 32) >> 4);
                    tc_mma_f16(s_tmem, qd + off, kd + off, kIdescS, k != 0 ? 1u : 0u);
                }
                tc_commit(s_full(t));
                for (int r = 0; r < reps; ++r) tc_commit(k_empty(s));
                if (last_s)
                    for (int r = 0; r < reps; ++r) tc_commit(q_empty);
                return true;
            };
            // O_t += P_t V of loaded block rb (the tile's block tb, j-th of the unit)
            auto issue_pv = [&](int rb, int tb, int j, int reps) -> bool {
                const int s = rb % kSt;
                if (!mbar_wait_bounded(p_full(t), tb & 1, p.timeout_ns, abort_flag, status, ROLE_MMA, BAR_P))
                    return false;
                if (!mbar_wait_bounded(v_full(s), (rb / kSt) & 1, p.timeout_ns, abort_flag, status, ROLE_MMA, BAR_V))
                    return false;
                tc_fence_after();
                const uint64_t vd = v_desc + static_cast<uint64_t>(s * kSlotUnits);
#pragma unroll
                for (int k = 0; k < kKeys / 16; ++k) {
                    // keys 16k..: P at columns 8k .. 8k + 7 of the tile's P buffer
                    tc_mma_f16_ta(o_tmem, pa + static_cast<uint32_t>(k * 8), vd + static_cast<uint64_t>(k * 2048 >> 4),
                                  kIdescO, (j | k) != 0 ? 1u : 0u);
                }
                tc_commit(pv_done(t));
                for (int r = 0; r < reps; ++r) tc_commit(v_empty(s));
                return true;
            };
            bool ok = true;
            int g = 0, gt = 0, nu = 0;   // blocks loaded, blocks this tile read, units
            UnitWalk walk{static_cast<int>(blockIdx.x), 0};
            int bh, qa, na, nb;
            while (ok && walk.next(p, nblk, np, sp, bh, qa, na, nb)) {
                if (t == 1 && nb == 0) break;         // tile B's warp sits out the one-tile units
                const int n = t == 0 ? na : nb;       // blocks this tile reads
                const int nr = nb > 0 ? nb : na;      // blocks loaded
                const int reps = nb > 0 ? 1 : 2;
                ok = mbar_wait_bounded(q_full, nu & 1, p.timeout_ns, abort_flag, status, ROLE_MMA, BAR_Q);
                if (ok) {
                    tc_fence_after();
                    ok = issue_s(g, n == 1, reps);
                }
                for (int j = 0; ok && j < n; ++j) {
                    const int rb = g + j;
                    // the next S, once the softmax warps have read this one
                    if (j + 1 < n) {
                        ok = mbar_wait_bounded(s_free(t), (gt + j) & 1, p.timeout_ns, abort_flag, status, ROLE_MMA,
                                               BAR_S);
                        if (ok) {
                            tc_fence_after();
                            ok = issue_s(rb + 1, j + 2 == n, reps);
                        }
                    }
                    if (ok) ok = issue_pv(rb, gt + j, j, reps);
                }
                if (ok && n < nr) {
                    // causal: tile A does not read the unit's last block; it arrives
                    // for that block's ring slots once the block has landed
                    const int lb = g + nr - 1;
                    ok = mbar_wait_bounded(k_full(lb % kSt), (lb / kSt) & 1, p.timeout_ns, abort_flag, status,
                                           ROLE_MMA, BAR_K) &&
                         mbar_wait_bounded(v_full(lb % kSt), (lb / kSt) & 1, p.timeout_ns, abort_flag, status,
                                           ROLE_MMA, BAR_V);
                    if (ok) {
                        tc_commit(k_empty(lb % kSt));
                        tc_commit(v_empty(lb % kSt));
                    }
                }
                g += nr;
                gt += n;
                ++nu;
            }
            tc_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, p.timeout_ns, nullptr, status, ROLE_DRAIN, BAR_DRAIN);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + output
        const int t = (warp - 3) >> 2;               // query tile A (0, warps 3..6) or B (1, warps 7..10)
        const int quarter = warp & 3;                // TMEM lanes 32 * quarter ..: this warp's rows
        const int r = 32 * quarter + lane;           // this thread's row of the tile
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16);
        const uint32_t s_cols = lane_base + kSCol + static_cast<uint32_t>(t * kKeys);
        const uint32_t p_cols = lane_base + kPCol + static_cast<uint32_t>(t * (kKeys / 2));
        const uint32_t o_cols = lane_base + kOCol + static_cast<uint32_t>(t * D);
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
                ok = mbar_wait_bounded(s_full(t), gb & 1, p.timeout_ns, abort_flag, status, ROLE_SOFTMAX, BAR_S);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                // the row's 128 scores of the block into registers; then the score
                // buffer is free for the next block's S
                uint32_t v[128];
                tmem_ld_32x32b_x128(s_cols, v);   // one load: four 32-column loads took longer
                tmem_wait_ld(v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_free(t));
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
                // P = 2^(x * scale_log2 - m) as fp16 pairs, all in registers (each
                // pair replaces two scores), and its sum over the fp16 values the
                // tensor core multiplies
                const float mm = (m_new == -INFINITY) ? 0.0f : m_new;
                float rs0 = 0.0f, rs1 = 0.0f;
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const float2 xs = fma2_bc(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]), p.scale_log2, -mm);
                    const __half2 hv = __floats2half2_rn(fast_exp2(xs.x), fast_exp2(xs.y));
                    v[i] = *reinterpret_cast<const uint32_t*>(&hv);
                    if (i & 1) rs1 = add_f16x2_to_f32(rs1, v[i]);
                    else rs0 = add_f16x2_to_f32(rs0, v[i]);
                }
                // into the P buffer (keys 32c .. 32c + 31 at columns 16c ..) once the
                // tile's previous P V, which reads it, has completed; O is then
                // settled for a rescale too (a unit's first block: the previous
                // unit's output already waited for its last P V)
                if (j > 0) {
                    ok = mbar_wait_bounded(pv_done(t), (gb - 1) & 1, p.timeout_ns, abort_flag, status, ROLE_SOFTMAX,
                                           BAR_PV);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                }
                // one store of the row's 64 columns (four 16-column stores measured 2-3 % slower)
                tmem_st_32x32b_x64(p_cols, *reinterpret_cast<const uint32_t(*)[64]>(v));
                // O rescaled on a raise (which needs an earlier block of the unit)
                if (__any_sync(0xffffffffu, raise)) {
                    const float alpha = raise ? fast_exp2(m - m_new) : 1.0f;
                    l *= alpha;
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t w[32];
                        tmem_ld_32x32b_x32(o_cols + 32u * c, w);
                        tmem_wait_ld(w);
#pragma unroll
                        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha);
                        tmem_st_32x32b_x32(o_cols + 32u * c, w);
                    }
                }
                m = m_new;
                l += rs0 + rs1;
                tmem_wait_st();
                tc_fence_before();           // P and the O rescale, if any, before the signal
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(t));
            }
            if (!ok) break;
            // output: O / l after the unit's last P V of this tile
            const int gl = g + n - 1;
            ok = mbar_wait_bounded(pv_done(t), gl & 1, p.timeout_ns, abort_flag, status, ROLE_SOFTMAX, BAR_PV);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            uint32_t w[D];
            tmem_ld_row<D>(o_cols, w);
            tmem_wait_ld(w);
            tc_fence_before();           // O read before this warp's next p_full arrival
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
