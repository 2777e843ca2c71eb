// Attention forward, one query tile per CTA and one softmax warp per TMEM lane
// quarter:  O = softmax(scale * Q K^T) V.
//
// The method and the roles common to the attention kernels are described in
// attn_kernels.cuh ("writing-tilelang-kernels", Flash Attention Forward and
// its Online Softmax pattern; the FLOP model of "TileLang: Write, Autotune,
// and Ship Fused Tensor-Core Kernels from Python", FlashAttention).  This
// kernel takes units of single query tiles, head-major, or causal pairs
// nq - 1 - k and k of one head (the middle tile of an odd count alone), so
// every unit costs the same; the host uses it where the two-tile kernels do
// not apply (an odd number of tiles, short or unevenly split causal problems).
// Two score buffers, so S of block j + 1 runs on the tensor core while the
// softmax works on block j (the MMA warp issues S of block j + 2 right after
// P V of block j), and two P buffers, so a softmax warp never waits for the
// previous P V before writing P.  A thread owns a whole row of the tile and
// holds the row's 128 scores of a block in registers: no exchange of row
// maxima or sums between warps (an earlier form split each row over two warps
// of 64 keys, 320 threads, exchanging maxima and sums through shared memory;
// same-box A/B at 4x32x4096x128: 1215 -> 1316 TFLOP/s, 4x32x4096x64 701 ->
// 800, causal 1058 -> 1124).  It computes all of P in registers before storing
// it, each pair of scores' registers then holding their P; where a block's sum
// of P calls for the exact maximum, the thread reads the block's scores from
// tensor memory again (the buffer is overwritten only after P is signalled).
// 192 threads: warp 0 the TMA producer, warp 1 the MMA warp, warps 2..5
// the softmax.  (Keeping P in tensor memory instead of shared memory measured
// 3 % faster and frees 64 KiB of shared memory; spending that on a third K
// and V ring slot did not pay.)
//
// Tensor memory: score buffers at columns 0 and 128, O at 256 (D columns),
// P buffers (fp16 pairs) at 384 and 448.  The barrier protocol is checked by
// a CPU model (tests/test_attn_protocol_cpu.py).
// Every wait is bounded (globaltimer); on a timeout or an abort raised by
// another role the CTA records the role and barrier in g_attn_status, drains
// what it issued and frees its tensor memory.
#pragma once

#include "attn_kernels.cuh"

namespace attn_dev {

constexpr int kAttn4Threads = 192;   // producer, MMA, 4 softmax warps

template <int D>
struct Attn4Smem {
    static constexpr uint32_t kQ = 0;                        // D/64 boxes
    static constexpr uint32_t kK = kQ + (D / 64) * kBox;     // 2 slots x D/64 boxes
    static constexpr uint32_t kV = kK + 2 * (D / 64) * kBox; // 2 slots x D/64 boxes
    static constexpr uint32_t kBars = kV + 2 * (D / 64) * kBox;
    // q_full, k_full[2], v_full[2], s_full[2], p_full[2], pv_done[2], drain, o_free
    static constexpr uint32_t kNumBars = 13;
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
__global__ void __launch_bounds__(kAttn4Threads, 1)
attn_f16_fwd4_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    static_assert(D == 64 || D == 128, "head dimension 64 or 128");
    using SM = Attn4Smem<D>;
    constexpr int kDB = D / 64;                     // 64-wide boxes per row of Q, K, V
    constexpr uint32_t kTileBytes = kDB * kBox;     // one Q, K or V tile
    // S = Q K^T: M 128, N 128, both K-major.  O += P V: M 128, N D, V MN-major.
    constexpr uint32_t kIdescS = idesc_f16_f32(kQRows, kKeys, /*b_mn_major=*/false);
    constexpr uint32_t kIdescO = idesc_f16_f32(kQRows, D, /*b_mn_major=*/true);
    constexpr uint32_t kOCol = 256;                 // O: D columns
    constexpr uint32_t kPCol = 384;                 // two 64-column P buffers (fp16 pairs)

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
    const uint32_t sQ = base_s + SM::kQ, sK = base_s + SM::kK, sV = base_s + SM::kV;
    const uint32_t bars = base_s + SM::kBars;
    const uint32_t q_full = bars;
    auto k_full = [&](int s) { return bars + 8u * (1 + s); };
    auto v_full = [&](int s) { return bars + 8u * (3 + s); };
    // S_j completed (block j in score buffer j & 1; K slot j & 1 free again)
    auto s_full = [&](int b) { return bars + 8u * (5 + b); };
    // P_j written (and O rescaled) for blocks b, b + 2, ...
    auto p_full = [&](int b) { return bars + 8u * (7 + b); };
    // P V of blocks b, b + 2, ... completed (V slot b free again)
    auto pv_done = [&](int b) { return bars + 8u * (9 + b); };
    const uint32_t drain_bar = bars + 8u * 11;
    // the softmax warps have read a tile's O: the next tile's first P V may overwrite it
    const uint32_t o_free = bars + 8u * 12;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + SM::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + SM::kAbort);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Work units in head-major order: unit u is query tile nq - 1 - u % nq of
    // head u / nq (causal: the heaviest tiles of a head first), or, when causal
    // tiles are paired, tiles nq - 1 - k and k of a head, so that every unit
    // costs the same nq + 1 key blocks, the pairs of every head first and then,
    // with an odd nq, each head's middle tile alone (half a unit: dealt last,
    // they fall on the CTAs with one pair fewer).  The units in flight belong to a few heads,
    // whose K and V stay in L2 (ordering by tile across heads made every query
    // tile read its head's K and V from HBM again: 7.4 GB per launch at B 4,
    // H 32, S 4096, D 128).
    const int kblocks_all = (p.S + kKeys - 1) / kKeys;
    auto tile_of = [&](int u, int i, int& bh, int& qt) -> bool {
        if (!p.pair) {
            if (i > 0) return false;
            bh = u / p.nq;
            qt = p.nq - 1 - u % p.nq;
            return true;
        }
        // pairs of every head first, then (odd nq) each head's middle tile
        const int hp = p.nq >> 1;                  // pairs per head
        const int pair_units = p.BH * hp;
        if (u >= pair_units) {
            if (i > 0) return false;
            bh = u - pair_units;
            qt = hp;                                // the middle tile (nq - 1) / 2
            return true;
        }
        bh = u / hp;
        const int k = u - bh * hp;
        qt = i == 0 ? p.nq - 1 - k : k;
        return true;
    };
    auto blocks_of = [&](int qt) { return p.causal ? min(kblocks_all, qt + 1) : kblocks_all; };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(v_full(s), 1);
            mbar_init(s_full(s), 1);
            mbar_init(p_full(s), 4);   // the four softmax warps
            mbar_init(pv_done(s), 1);
        }
        mbar_init(o_free, 4);
        mbar_init(drain_bar, 1);
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

    // Key blocks are numbered g = 0, 1, ... over all of this CTA's tiles: block g
    // uses ring slot, score buffer and P buffer g & 1, and phase (g >> 1) & 1 of
    // their barriers; tile t uses phase t & 1 of q_full and o_free.
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // lane 0 streams Q and K, lane 1 streams V
        if (lane < 2) {
            const bool is_k = lane == 0;
            const CUtensorMap* tm = is_k ? &tmK : &tmV;
            const uint32_t ring = is_k ? sK : sV;
            const uint32_t which = is_k ? BAR_K : BAR_V;
            bool ok = true;
            int g = 0, ntile = 0, issued = 0;
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                for (int i = 0; ok && i < 2; ++i) {
                    int bh, qt;
                    if (!tile_of(u, i, bh, qt)) break;
                    const int nblk = blocks_of(qt);
                    if (is_k) {
                        // Q is the A operand of every S of the previous tile: reload it once
                        // the last of those (block g - 1) has completed
                        if (g > 0 && !mbar_wait_bounded(s_full((g - 1) & 1), ((g - 1) >> 1) & 1, p.timeout_ns,
                                                        abort_flag, status, ROLE_PRODUCER, BAR_Q)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(q_full, kTileBytes);
                        for (int c = 0; c < kDB; ++c) tma_load_3d(sQ + c * kBox, &tmQ, q_full, 64 * c, qt * kQRows, bh);
                    }
                    ++ntile;
                    for (int j = 0; j < nblk; ++j) {
                        const int gb = g + j;
                        const int s = gb & 1;
                        // slot s is free once S (for K) or P V (for V) of block gb - 2 completed
                        const uint32_t empty = is_k ? s_full(s) : pv_done(s);
                        if (!mbar_wait_bounded(empty, static_cast<uint32_t>((gb >> 1) & 1) ^ 1u, p.timeout_ns,
                                               abort_flag, status, ROLE_PRODUCER, which)) {
                            ok = false;
                            break;
                        }
                        if (is_k && gb == p.fault_skip_block) continue;   // injected fault: never loaded
                        const uint32_t full = is_k ? k_full(s) : v_full(s);
                        mbar_arrive_expect_tx(full, kTileBytes);
                        for (int c = 0; c < kDB; ++c)
                            tma_load_3d(ring + (s * kDB + c) * kBox, tm, full, 64 * c, j * kKeys, bh);
                        issued = gb + 1;
                    }
                    g += nblk;
                }
            }
            // every issued load lands before the CTA can exit
            if (is_k && ntile > 0)
                mbar_wait_bounded(q_full, (ntile - 1) & 1, p.timeout_ns, nullptr, status, ROLE_DRAIN, BAR_Q);
            for (int gb = max(0, issued - 2); gb < issued; ++gb)
                mbar_wait_bounded(is_k ? k_full(gb & 1) : v_full(gb & 1), (gb >> 1) & 1, p.timeout_ns, nullptr,
                                  status, ROLE_DRAIN, which);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        {
            const uint64_t q_desc = smem_desc_sw128(sQ, 0, 1024);
            const uint64_t k_desc = smem_desc_sw128(sK, 0, 1024);
            const uint64_t v_desc = smem_desc_sw128(sV, kBox, 1024);   // MN-major: 64-column boxes kBox apart
            constexpr uint32_t kSlotUnits = kTileBytes >> 4;           // one ring slot, in 16-byte units
            auto issue_s = [&](int gb) -> bool {   // S of block gb = Q K^T into score buffer gb & 1
                const int s = gb & 1;
                if (!mbar_wait_bounded(k_full(s), (gb >> 1) & 1, p.timeout_ns, abort_flag, status, ROLE_MMA, BAR_K))
                    return false;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(s * kKeys);
                const uint64_t kd = k_desc + static_cast<uint64_t>(s * kSlotUnits);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    // K-major: box k / 4, 32 bytes per 16-deep step inside the swizzled row
                    const uint64_t off = static_cast<uint64_t>(((k >> 2) * kBox + (k & 3) * 32) >> 4);
                    tc_mma_f16(d_tmem, q_desc + off, kd + off, kIdescS, k != 0 ? 1u : 0u);
                }
                tc_commit(s_full(s));        // also frees K slot s
                return true;
            };
            bool ok = true;
            int g = 0, ntile = 0;
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                for (int i = 0; ok && i < 2; ++i) {
                    int bh, qt;
                    if (!tile_of(u, i, bh, qt)) break;
                    const int nblk = blocks_of(qt);
                    ok = mbar_wait_bounded(q_full, ntile & 1, p.timeout_ns, abort_flag, status, ROLE_MMA, BAR_Q);
                    if (ok) {
                        tc_fence_after();
                        ok = issue_s(g);
                    }
                    if (ok && nblk > 1) ok = issue_s(g + 1);
                    for (int j = 0; ok && j < nblk; ++j) {
                        const int gb = g + j;
                        const int s = gb & 1;
                        if (!mbar_wait_bounded(p_full(s), (gb >> 1) & 1, p.timeout_ns, abort_flag, status, ROLE_MMA,
                                               BAR_P)) {
                            ok = false;
                            break;
                        }
                        // the first P V of a tile overwrites O: the previous tile's output
                        // must have been read out of tensor memory
                        if (j == 0 && ntile > 0 &&
                            !mbar_wait_bounded(o_free, (ntile - 1) & 1, p.timeout_ns, abort_flag, status, ROLE_MMA,
                                               BAR_P)) {
                            ok = false;
                            break;
                        }
                        if (!mbar_wait_bounded(v_full(s), (gb >> 1) & 1, p.timeout_ns, abort_flag, status, ROLE_MMA,
                                               BAR_V)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t o_tmem = tmem_base + kOCol;
                        const uint32_t pa = tmem_base + kPCol + static_cast<uint32_t>(s * 64);
                        const uint64_t vd = v_desc + static_cast<uint64_t>(s * kSlotUnits);
#pragma unroll
                        for (int k = 0; k < kKeys / 16; ++k)
                            tc_mma_f16_ta(o_tmem, pa + static_cast<uint32_t>(k * 8),
                                          vd + static_cast<uint64_t>(k * 2048 >> 4), kIdescO, (j | k) != 0 ? 1u : 0u);
                        tc_commit(pv_done(s));       // also frees V slot s
                        // score buffer s was read before this P was written
                        if (j + 2 < nblk) ok = issue_s(gb + 2);
                    }
                    g += nblk;
                    ++ntile;
                }
            }
            tc_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, p.timeout_ns, nullptr, status, ROLE_DRAIN, BAR_DRAIN);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + output
        const int quarter = warp & 3;                // TMEM lanes 32 * quarter ..: this warp's rows
        const int r = 32 * quarter + lane;           // this thread's row of the tile
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16);
        const uint32_t o_cols = lane_base + kOCol;
        const bool pos = p.scale_log2 >= 0.0f;
        const uint32_t lose = __float_as_uint(pos ? -INFINITY : INFINITY);
        bool ok = true;
        int g = 0;
        for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
            for (int i = 0; ok && i < 2; ++i) {
                int bh, qt;
                if (!tile_of(u, i, bh, qt)) break;
                const int nblk = blocks_of(qt);
                const int q = qt * kQRows + r;               // this thread's query index
                // keys past S, and (causal) keys after this query, do not count
                const int key_end = p.causal ? min(p.S, q + 1) : p.S;
                float m = -INFINITY, l = 0.0f;
                for (int j = 0; j < nblk; ++j) {
                    const int gb = g + j;
                    const int k0 = j * kKeys;
                    const int s = gb & 1;
                    const uint32_t s_cols = lane_base + static_cast<uint32_t>(s * kKeys);
                    ok = mbar_wait_bounded(s_full(s), (gb >> 1) & 1, p.timeout_ns, abort_flag, status, ROLE_SOFTMAX,
                                           BAR_S);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                    // the row's 128 scores of the block, all in registers.  The largest
                    // scaled score comes from the largest raw score when the scale is
                    // positive and from the smallest when it is negative; keys that do
                    // not count get the raw score that loses that comparison, so their
                    // weight is 2^-inf = 0.
                    uint32_t v[128];
                    auto load_scores = [&]() {
                        tmem_ld_32x32b_x128(s_cols, v);   // one load: four 32-column loads took longer
                        tmem_wait_ld(v);
                        if (k0 + kKeys > p.S || (p.causal && j == nblk - 1)) {
                            const int key_lim = key_end - k0;         // valid: column < key_lim
#pragma unroll
                            for (int t = 0; t < 128; ++t)
                                if (t >= key_lim) v[t] = lose;
                        }
                    };
                    // the largest scaled score (log2 units); -inf if no key counts
                    auto block_max = [&]() -> float {
                        float bm[4];
                        bm[0] = bm[1] = bm[2] = bm[3] = pos ? -INFINITY : INFINITY;
                        if (pos) {
#pragma unroll
                            for (int t = 0; t < 128; t += 2)
                                bm[(t >> 1) & 3] = max3f(bm[(t >> 1) & 3], __uint_as_float(v[t]), __uint_as_float(v[t + 1]));
                        } else {
#pragma unroll
                            for (int t = 0; t < 128; t += 2)
                                bm[(t >> 1) & 3] = min3f(bm[(t >> 1) & 3], __uint_as_float(v[t]), __uint_as_float(v[t + 1]));
                        }
                        const float b = pos ? fmaxf(fmaxf(bm[0], bm[1]), fmaxf(bm[2], bm[3]))
                                            : fminf(fminf(bm[0], bm[1]), fminf(bm[2], bm[3]));
                        return b * p.scale_log2;
                    };
                    // P = 2^(x * scale_log2 - mm) as fp16 pairs, all in registers (each
                    // pair replaces two scores); returns the block's sum of those fp16
                    // values, in fp32
                    auto p_pass = [&](float mm) -> float {
                        float rs0 = 0.0f, rs1 = 0.0f;
#pragma unroll
                        for (int t = 0; t < 64; ++t) {
                            const float2 xs = fma2_bc(__uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1]),
                                                      p.scale_log2, -mm);
                            const __half2 hv = __floats2half2_rn(fast_exp2(xs.x), fast_exp2(xs.y));
                            v[t] = *reinterpret_cast<const uint32_t*>(&hv);
                            if (t & 1) rs1 = add_f16x2_to_f32(rs1, v[t]);
                            else rs0 = add_f16x2_to_f32(rs0, v[t]);
                        }
                        return rs0 + rs1;
                    };
                    // The running maximum m is raised when the block maximum exceeds it
                    // by more than kRaise, so that every P stays within 2^kRaise.  At a
                    // tile's first block (m not yet set) the maximum is taken first.
                    // Otherwise P is formed with m at once and its sum decides: a sum
                    // within 2^kRaise bounds every P, so the maximum cannot have exceeded
                    // the limit; above it the scores are read again from tensor memory,
                    // the maximum taken and P formed again (with the raised maximum,
                    // where there is a raise).
                    load_scores();
                    float m_new = m;
                    bool raise = false;
                    const bool first = __any_sync(0xffffffffu, m == -INFINITY);
                    if (first) {
                        const float bmax = block_max();
                        if (bmax > m + kRaise || m == -INFINITY) {
                            m_new = fmaxf(m, bmax);
                            raise = m != -INFINITY && m_new != m;
                        }
                    }
                    float bsum = p_pass((m_new == -INFINITY) ? 0.0f : m_new);
                    if (!first && __any_sync(0xffffffffu, bsum > kRaiseSum)) {
                        load_scores();
                        const float bmax = block_max();
                        if (bmax > m + kRaise) {
                            m_new = fmaxf(m, bmax);
                            raise = m_new != m;
                        }
                        bsum = p_pass(m_new);
                    }
                    // O is rescaled only after P V of block gb - 1 (of this tile: a raise
                    // needs an earlier block) has finished.  P V of block gb - 3 was issued
                    // before S of block gb, whose completion this thread has seen, and P V
                    // of block gb + 1 needs this block's P first: the barrier is within one
                    // phase of the one waited for, so its parity names it.
                    if (__any_sync(0xffffffffu, raise)) {
                        ok = mbar_wait_bounded(pv_done((gb - 1) & 1), ((gb - 1) >> 1) & 1, p.timeout_ns, abort_flag,
                                               status, ROLE_SOFTMAX, BAR_PV);
                        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                        tc_fence_after();
                        const float alpha = raise ? fast_exp2(m - m_new) : 1.0f;
                        l *= alpha;
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t w[32];
                            tmem_ld_32x32b_x32(o_cols + 32u * c, w);
                            tmem_wait_ld(w);
#pragma unroll
                            for (int t = 0; t < 32; ++t) w[t] = __float_as_uint(__uint_as_float(w[t]) * alpha);
                            tmem_st_32x32b_x32(o_cols + 32u * c, w);
                        }
                    }
                    m = m_new;
                    l += bsum;
                    // P buffer s (keys 32c .. 32c + 31 at columns 16c ..) was last read by
                    // P V of block gb - 2, issued before S of block gb: complete
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        tmem_st_32x32b_x16(lane_base + kPCol + static_cast<uint32_t>(s * 64 + 16 * c),
                                           *reinterpret_cast<const uint32_t(*)[16]>(v + 16 * c));
                    tmem_wait_st();
                    tc_fence_before();           // P and the O rescale, if any, before the signal
                    __syncwarp();
                    if (lane == 0) mbar_arrive(p_full(s));
                }
                if (!ok) break;
                // output: O / l after the tile's last P V (its commit also covers every
                // earlier MMA); O read into registers and released before the stores
                const int gl = g + nblk - 1;
                ok = mbar_wait_bounded(pv_done(gl & 1), (gl >> 1) & 1, p.timeout_ns, abort_flag, status,
                                       ROLE_SOFTMAX, BAR_PV);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t w[D];
                tmem_ld_row<D>(o_cols, w);
                tmem_wait_ld(w);
                tc_fence_before();           // O read out before the next tile may overwrite it
                __syncwarp();
                if (lane == 0) mbar_arrive(o_free);
                const float inv = 1.0f / l;
                if (q < p.S) {
                    uint4* dst = reinterpret_cast<uint4*>(p.O + (static_cast<int64_t>(bh) * p.S + q) * D);
#pragma unroll
                    for (int t = 0; t < D / 8; ++t) {
                        uint32_t hh[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __half2 hv = __floats2half2_rn(__uint_as_float(w[8 * t + 2 * e]) * inv,
                                                                 __uint_as_float(w[8 * t + 2 * e + 1]) * inv);
                            hh[e] = *reinterpret_cast<const uint32_t*>(&hv);
                        }
                        dst[t] = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                    }
                }
                g += nblk;
            }
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
