// Attention forward for sm_103a:  O = softmax(scale * Q K^T) V  per (batch, head).
//
// The method: "writing-tilelang-kernels", Flash Attention Forward (Q, K, V, O
// as (B, H, S, D) fp16 tensors; one program per block of query rows) and its
// pattern table's "Online Softmax" row (running max, exp, rescaling);
// "TileLang: Write, Autotune, and Ship Fused Tensor-Core Kernels from
// Python", FlashAttention: the FLOP model (softmax computed online, the S x S
// score matrix never written to memory; causal and non-causal).
//
// GB300 design: persistent, one CTA per SM, each taking a sequence of query
// tiles of 128 rows of one head (tensor memory, barriers and the rings carry
// over from tile to tile: the next tile's Q and first two S products overlap
// the current tile's last blocks and output):
//   * warp 0: TMA producers (lane 0: each tile's Q, then K; lane 1: V), blocks
//     of 128 keys through two 2-slot rings; 3-D tensor maps
//     (D, S, B*H), so rows past S arrive as zeros and never come from the
//     next head;
//   * warp 1: allocates tensor memory and issues tcgen05.mma from one thread:
//     S_j = Q K_j^T (M = 128, N = 128, K = D; both operands K-major) into one
//     of two TMEM score buffers, and O += P_j V_j (M = 128, N = D, K = 128;
//     P read by the tensor core straight from tensor memory, V MN-major from
//     shared memory) into the TMEM output;
//     S_{j+1} is computed while the softmax of block j runs;
//   * warps 2..9: softmax, one query row per thread pair (its TMEM lane; the
//     two warps of a lane quarter each take 64 keys of a block): pass 1
//     reads the row of S_j for the block maximum, pass 2 reads it again,
//     forms p = 2^(s * scale * log2 e - m) in fp32, sums it and writes it as
//     fp16 pairs into one of two tensor-memory P buffers (one row per lane,
//     the layout the MMA reads its A operand in), so the softmax of block
//     j + 1 never waits for the P V product of block j (keeping P in tensor
//     memory instead of shared memory measured 3 % faster and frees 64 KiB of
//     shared memory; spending that on a third K and V ring slot did not pay).
//     The running maximum m is raised only when a
//     block's maximum exceeds it by more than 8 (in log2 units); O and the
//     running sum l are then rescaled in place (TMEM load, multiply, store).
//     Between raises p stays below 2^8, which fp16 and the fp32 sums hold
//     exactly enough, and the final O / l is the same ratio;
//   * after a tile's last block: O / l rounded to fp16, 16-byte stores of
//     each thread's row; then the tile's O may be overwritten.
// Every wait is bounded (as in the GEMM kernels): on a timeout the role
// records itself in the status word, raises a shared abort flag, drains what
// it issued and leaves; tensor memory is always freed.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace attn_dev {

using namespace gemm_f16_dev;

__device__ unsigned int g_attn_status;   // bounded-wait status word of the attention kernels

constexpr int kQRows = 128;              // query rows per CTA = MMA M = TMEM lanes
constexpr int kKeys = 128;               // keys per block = N of S = K of P V
constexpr int kAttnThreads = 320;        // producer, MMA, 8 softmax warps (two per TMEM lane quarter)
constexpr uint32_t kMaxDynSmem = 232448;  // 227 KiB: the most dynamic shared memory a CTA may have
constexpr uint32_t kBox = 64 * 128 * 2;  // one 64 (D or keys) x 128 (rows) fp16 box: 16 KiB
constexpr uint32_t kTmemCols = 512;      // two 128-column score buffers, O (<= 128 columns), two P buffers
constexpr uint32_t kOCol = 256;          // first TMEM column of O
constexpr uint32_t kPCol = 384;          // two 64-column P buffers (fp16 pairs), columns 384 .. 511
constexpr float kRaise = 8.0f;           // raise the running max only past 2^8 growth

enum : uint32_t { ROLE_SOFTMAX = 6, BAR_Q = 7, BAR_K = 8, BAR_V = 9, BAR_S = 10, BAR_P = 11, BAR_PV = 12,
                  BAR_X = 13, BAR_ALIGN = 14 };

struct AttnParams {
    __half* O;
    int S;              // sequence length (queries = keys)
    int BH;             // batch * heads
    int nq;             // query tiles per head
    int causal;
    int units;          // work units: query tiles, or pairs of query tiles
    int pair;           // causal, with at least two tiles per SM: a unit is a pair of tiles
    int pair_units;     // two-tile kernel: units below this hold two tiles, the rest one
    float scale_log2;   // softmax scale * log2(e)
    uint64_t timeout_ns;
    // Fault injection for the tests of the bounded waits (-1 in every normal
    // call): the K producer never loads key block `fault_skip_block` of the
    // CTA's block sequence, so the MMA thread's wait for it runs out and the
    // abort path runs with no copy in flight for that block.
    int fault_skip_block;
};

template <int D>
struct AttnSmem {
    static constexpr uint32_t kQ = 0;                        // D/64 boxes
    static constexpr uint32_t kK = kQ + (D / 64) * kBox;     // 2 slots x D/64 boxes
    static constexpr uint32_t kV = kK + 2 * (D / 64) * kBox; // 2 slots x D/64 boxes
    static constexpr uint32_t kX = kV + 2 * (D / 64) * kBox; // row-maximum exchange [2 parity][2 half][128]
    static constexpr uint32_t kBars = kX + 2 * 2 * 128 * 4;
    // q_full, k_full[2], v_full[2], s_full[2], p_full[2], pv_done[2], drain, o_free,
    // xch[4 quarters][2 parity]
    static constexpr uint32_t kNumBars = 13 + 8;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kEnd = kAbort + 4;
    // 1 KiB of slack aligns the base to the 128-byte swizzle's 1 KiB atoms
    // when it fits; otherwise (D = 128) the kernel checks that the base is
    // already aligned (the dynamic window starts after the 1 KiB the system
    // reserves) and reports BAR_ALIGN instead of running if it is not.
    static constexpr bool kSlack = kEnd + 1024 <= kMaxDynSmem;
    // The CTA allocates all 512 tensor-memory columns, so a second CTA on the
    // same SM would only wait in its allocation: ask for enough shared memory
    // (> half of the SM's 228 KiB) that one CTA fits per SM.
    static constexpr uint32_t kOnePerSm = 120 * 1024;
    static constexpr uint32_t kNeed = kEnd + (kSlack ? 1024 : 0);
    static constexpr uint32_t kDynamicBytes = kNeed > kOnePerSm ? kNeed : kOnePerSm;
    static_assert(kDynamicBytes <= kMaxDynSmem, "shared memory plan too large");
};

// 3-D tiled load (D, S, B*H) global -> shared, completing `bar`.  c0 (the D
// offset) is 0 or 64: a multiple of 8 elements (16 bytes).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                                            int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns from registers to tensor memory.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
          "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
          "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]: A (M x 16, fp16) held in tensor memory,
// one row per lane, two fp16 per 32-bit column (issued from a converged warp,
// as tc_mma_f16).
__device__ __forceinline__ void tc_mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\t"
        "elect.sync r|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// acc + the two fp16 halves of w, each widened exactly to fp32 (the
// mixed-precision add of sm_100 and later: no separate conversion)
__device__ __forceinline__ float add_f16x2_to_f32(float acc, uint32_t w) {
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "add.f32.f16 %0, lo, %0;\n\tadd.f32.f16 %0, hi, %0;\n\t}"
        : "+f"(acc) : "r"(w));
    return acc;
}

// Generic-proxy writes to shared memory made visible to the async proxy (the
// tensor core, TMA) before a barrier that orders them with its reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Three-input maximum / minimum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float m;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
    return m;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
    float m;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
    return m;
}
// (a.x * b + c, a.y * b + c) as one paired fp32 FMA (sm_100 and later).
__device__ __forceinline__ float2 fma2_bc(float ax, float ay, float b, float c) {
    uint64_t x, y, z, d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(ax), "f"(ay));
    asm("mov.b64 %0, {%1, %1};" : "=l"(y) : "f"(b));
    asm("mov.b64 %0, {%1, %1};" : "=l"(z) : "f"(c));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(x), "l"(y), "l"(z));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_f16_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    static_assert(D == 64 || D == 128, "head dimension 64 or 128");
    using SM = AttnSmem<D>;
    constexpr int kDB = D / 64;                     // 64-wide boxes per row of Q, K, V
    constexpr uint32_t kTileBytes = kDB * kBox;     // one Q, K or V tile
    // S = Q K^T: M 128, N 128, both K-major.  O += P V: M 128, N D, V MN-major.
    constexpr uint32_t kIdescS = idesc_f16_f32(kQRows, kKeys, /*b_mn_major=*/false);
    constexpr uint32_t kIdescO = idesc_f16_f32(kQRows, D, /*b_mn_major=*/true);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    if (!SM::kSlack && (raw_s & 1023u) != 0) {   // uniform over the CTA: nothing started yet
        if (threadIdx.x == 0) atomicCAS(&g_attn_status, 0u, 0x80000000u | (ROLE_SOFTMAX << 8) | BAR_ALIGN);
        return;
    }
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
    const uint32_t sQ = base_s + SM::kQ, sK = base_s + SM::kK, sV = base_s + SM::kV;
    const uint32_t bars = base_s + SM::kBars;
    const uint32_t q_full = bars;
    auto k_full = [&](int s) { return bars + 8u * (1 + s); };
    auto v_full = [&](int s) { return bars + 8u * (3 + s); };
    // S_j completed (block j in score buffer j & 1; K slot j & 1 free again)
    auto s_full = [&](int b) { return bars + 8u * (5 + b); };
    // P_j written (and O rescaled) for blocks b, b + 2, ...: one barrier per P
    // buffer, so the softmax of block j + 1 cannot complete a phase before the
    // MMA thread has seen the one of block j (its next arrival on the same
    // barrier, block j + 2, needs S_{j+2}, issued only after that)
    auto p_full = [&](int b) { return bars + 8u * (7 + b); };
    // P V of blocks b, b + 2, ... completed (V slot b free again)
    auto pv_done = [&](int b) { return bars + 8u * (9 + b); };
    const uint32_t drain_bar = bars + 8u * 11;
    // the softmax warps have read a tile's O: the next tile's first P V may overwrite it
    const uint32_t o_free = bars + 8u * 12;
    auto xch_bar = [&](int quarter, int b) { return bars + 8u * (13 + 2 * quarter + b); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + SM::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + SM::kAbort);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Work units in head-major order: unit u is query tile nq - 1 - u % nq
    // of head u / nq (causal: the heaviest tiles of a head first), or, when
    // causal tiles are paired, the two tiles nq - 1 - k and k of head
    // u / npairs (k = u % npairs; the middle tile of an odd count alone), so
    // that every unit costs the same nq + 1 key blocks.  One CTA per
    // SM takes units blockIdx.x, blockIdx.x + gridDim.x, ...: the units in
    // flight belong to a few heads, whose K and V stay in L2 (ordering by
    // tile across heads made every query tile read its head's K and V from
    // HBM again: 7.4 GB per launch at B 4, H 32, S 4096, D 128).  Staying
    // resident lets the next tile's Q load and first two S products overlap
    // the current tile's last blocks and output.
    const int kblocks_all = (p.S + kKeys - 1) / kKeys;
    auto tile_of = [&](int u, int i, int& bh, int& qt) -> bool {
        if (!p.pair) {
            if (i > 0) return false;
            bh = u / p.nq;
            qt = p.nq - 1 - u % p.nq;
            return true;
        }
        const int npairs = (p.nq + 1) >> 1;
        bh = u / npairs;
        const int k = u % npairs;
        if (i == 0) {
            qt = p.nq - 1 - k;
            return true;
        }
        if (k == p.nq - 1 - k) return false;
        qt = k;
        return true;
    };
    auto blocks_of = [&](int qt) { return p.causal ? min(kblocks_all, qt + 1) : kblocks_all; };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(v_full(s), 1);
            mbar_init(s_full(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(p_full(b), 8);   // the eight softmax warps
            mbar_init(pv_done(b), 1);
        }
        mbar_init(o_free, 8);
        for (int q = 0; q < 4; ++q)
            for (int b = 0; b < 2; ++b) mbar_init(xch_bar(q, b), 64);   // both warps of a lane quarter
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
        // lane 0 streams Q and K, lane 1 streams V: a K load never waits behind
        // a V slot (V of block g frees after P V of block g - 2, K after S_{g-2})
        if (lane < 2) {
            const bool is_k = lane == 0;
            const CUtensorMap* tm = is_k ? &tmK : &tmV;
            const uint32_t ring = is_k ? sK : sV;
            const uint32_t which = is_k ? BAR_K : BAR_V;
            bool ok = true;
            int g = 0, ntile = 0, issued = 0;   // issued: blocks loaded (= g + j while streaming)
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
                        // slot s is free once S (for K) or P V (for V) of block g - 2
                        // completed: the barriers the softmax waits on serve the producer
                        // as well (one commit fewer per group of MMAs)
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
            // every issued load lands before the CTA can exit (the last Q and the last
            // one or two blocks of each ring; earlier ones were waited for by the MMA
            // thread before it issued what freed their slots)
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
            // The whole warp runs this loop and one elected lane issues each MMA
            // (tc_mma_f16); the tensor pipe stays fed only if the work between
            // two MMAs (64 cycles each at N = 128) stays short: the descriptors
            // are built once, and each MMA adds a constant to the start-address
            // field (in 16-byte units; every shared address is below 2^18, so
            // the 14-bit field never carries).
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
                    // this tile's Q (its first two S need nothing else of the previous tile)
                    ok = mbar_wait_bounded(q_full, ntile & 1, p.timeout_ns, abort_flag, status, ROLE_MMA, BAR_Q);
                    if (ok) {
                        tc_fence_after();
                        ok = issue_s(g);
                    }
                    if (ok && nblk > 1) ok = issue_s(g + 1);
                    for (int j = 0; ok && j < nblk; ++j) {
                        const int gb = g + j;
                        const int s = gb & 1;
                        // P of block gb written (and O rescaled) by the softmax warps
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
                        for (int k = 0; k < kKeys / 16; ++k) {
                            // P from tensor memory (16 keys = 8 columns of fp16 pairs per step);
                            // V: MN-major, 16 key rows = 2 KiB per step
                            tc_mma_f16_ta(o_tmem, pa + static_cast<uint32_t>(k * 8),
                                          vd + static_cast<uint64_t>(k * 2048 >> 4), kIdescO, (j | k) != 0 ? 1u : 0u);
                        }
                        tc_commit(pv_done(s));       // also frees V slot s
                        // score buffer s was read before this P was written; the next
                        // tile's first two S wait for its Q, after this tile's last P V
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
        // Two warps per TMEM lane quarter: warp half h takes keys 64h .. 64h + 63
        // of every block (it writes P box h) and O columns h D/2 .. (h + 1) D/2.
        // The pair combines its row maxima (and, at the end of a tile, its row
        // sums) through shared memory behind a 64-thread mbarrier with a bounded
        // wait; the exchanges alternate between two buffers, so a warp never
        // overwrites a value its partner has not read yet.
        const int quarter = warp & 3;                // TMEM lanes 32 * quarter ..
        const int half = (warp - 2) >> 2;
        const int r = 32 * quarter + lane;           // this thread's row of the tile
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16);
        volatile float* xch = reinterpret_cast<volatile float*>(base + SM::kX);
        int x = 0;                                   // exchanges so far
        auto exchange = [&](float mine, float& theirs) -> bool {
            const int slot = x & 1, use = x >> 1;    // use: earlier uses of this slot
            ++x;
            xch[(slot * 2 + half) * 128 + r] = mine;
            mbar_arrive(xch_bar(quarter, slot));
            const bool got = mbar_wait_bounded(xch_bar(quarter, slot), use & 1, p.timeout_ns, abort_flag, status,
                                               ROLE_SOFTMAX, BAR_X);
            theirs = xch[(slot * 2 + (1 - half)) * 128 + r];
            return got;
        };
        constexpr int kOCols = D / 2;                // this warp's O columns
        const uint32_t o_cols = lane_base + kOCol + static_cast<uint32_t>(half * kOCols);
        bool ok = true;
        int g = 0;
        for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
            for (int i = 0; ok && i < 2; ++i) {
                int bh, qt;
                if (!tile_of(u, i, bh, qt)) break;
                const int nblk = blocks_of(qt);
                const int q = qt * kQRows + r;               // this thread's query index
                float m = -INFINITY, l = 0.0f;
                for (int j = 0; j < nblk; ++j) {
                    const int gb = g + j;
                    const int k0 = j * kKeys;
                    const int s = gb & 1;
                    const uint32_t s_tmem = lane_base + static_cast<uint32_t>(s * kKeys + 64 * half);
                    ok = mbar_wait_bounded(s_full(s), (gb >> 1) & 1, p.timeout_ns, abort_flag, status, ROLE_SOFTMAX,
                                           BAR_S);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                    // keys past S, and (causal) keys after this query, do not count
                    const bool masked_block = (k0 + kKeys > p.S) || (p.causal && j == nblk - 1);
                    const int key_lim = (p.causal ? min(p.S, q + 1) - k0 : p.S - k0) - 64 * half;   // valid: col < key_lim
                    // this warp's 64 scores of the row: two loads in flight, one wait, kept
                    // in registers for both passes (each wait call ties one chunk's registers)
                    uint32_t v[64];
                    tmem_ld_32x32b_x32(s_tmem, *reinterpret_cast<uint32_t(*)[32]>(v));
                    tmem_ld_32x32b_x32(s_tmem + 32u, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
                    tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(v));
                    tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(v + 32));
                    // The largest scaled score comes from the largest raw score when the
                    // scale is positive and from the smallest when it is negative.  Keys
                    // that do not count get the raw score that loses that comparison
                    // (-inf, or +inf for a negative scale): their scaled score is -inf
                    // and their weight 2^-inf = 0.
                    const bool pos = p.scale_log2 >= 0.0f;
                    if (masked_block) {
                        const uint32_t lose = __float_as_uint(pos ? -INFINITY : INFINITY);
#pragma unroll
                        for (int t = 0; t < 64; ++t)
                            if (t >= key_lim) v[t] = lose;
                    }
                    // pass 1: the row's largest scaled score over this warp's 64 keys, then the pair's
                    float bm[4];   // four independent chains, two new values per three-input step
                    if (pos) {
                        bm[0] = bm[1] = bm[2] = bm[3] = -INFINITY;
#pragma unroll
                        for (int t = 0; t < 64; t += 2)
                            bm[(t >> 1) & 3] = max3f(bm[(t >> 1) & 3], __uint_as_float(v[t]), __uint_as_float(v[t + 1]));
                    } else {
                        bm[0] = bm[1] = bm[2] = bm[3] = INFINITY;
#pragma unroll
                        for (int t = 0; t < 64; t += 2)
                            bm[(t >> 1) & 3] = min3f(bm[(t >> 1) & 3], __uint_as_float(v[t]), __uint_as_float(v[t + 1]));
                    }
                    float bmax = pos ? fmaxf(fmaxf(bm[0], bm[1]), fmaxf(bm[2], bm[3]))
                                     : fminf(fminf(bm[0], bm[1]), fminf(bm[2], bm[3]));
                    bmax *= p.scale_log2;   // the largest scaled score (log2 units); -inf if no key counts
                    float other = -INFINITY;
                    ok = exchange(bmax, other);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    const float bmax2 = fmaxf(bmax, other);
                    float m_new = m;
                    bool raise = false;
                    if (bmax2 > m + kRaise || m == -INFINITY) {
                        m_new = fmaxf(m, bmax2);
                        raise = m != -INFINITY && m_new != m;
                    }
                    // O is rescaled only after P V of block gb - 1 (of this tile: a raise
                    // needs an earlier block) has finished.  P V of block gb - 3 was issued
                    // before S of block gb, whose completion this thread has seen, and P V
                    // of block gb + 1 needs this block's P first: the barrier is within one
                    // phase of the one waited for, so its parity names it.  P buffer s was
                    // last read by P V of block gb - 2, issued before S of block gb.
                    if (__any_sync(0xffffffffu, raise)) {
                        ok = mbar_wait_bounded(pv_done((gb - 1) & 1), ((gb - 1) >> 1) & 1, p.timeout_ns, abort_flag,
                                               status, ROLE_SOFTMAX, BAR_PV);
                        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                        tc_fence_after();
                        const float alpha = raise ? fast_exp2(m - m_new) : 1.0f;
                        l *= alpha;
#pragma unroll 1
                        for (int c = 0; c < kOCols / 32; ++c) {
                            uint32_t w[32];
                            tmem_ld_32x32b_x32(o_cols + 32u * c, w);
                            tmem_wait_ld(w);
#pragma unroll
                            for (int t = 0; t < 32; ++t) w[t] = __float_as_uint(__uint_as_float(w[t]) * alpha);
                            tmem_st_32x32b_x32(o_cols + 32u * c, w);
                        }
                        tmem_wait_st();
                    }
                    m = m_new;
                    // pass 2: p = 2^(x * scale_log2 - m) as fp16 into box `half` of P buffer s
                    const float mm = (m == -INFINITY) ? 0.0f : m;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t h[16];
                        float rs0 = 0.0f, rs1 = 0.0f;
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            // masked keys hold -inf: 2^-inf = 0
                            const float2 xs = fma2_bc(__uint_as_float(v[32 * c + 2 * t]),
                                                      __uint_as_float(v[32 * c + 2 * t + 1]), p.scale_log2, -mm);
                            const float e0 = fast_exp2(xs.x);
                            const float e1 = fast_exp2(xs.y);
                            const __half2 hv = __floats2half2_rn(e0, e1);
                            h[t] = *reinterpret_cast<const uint32_t*>(&hv);
                            // the sum takes the fp16 values the tensor core multiplies
                            if (t & 1) rs1 = add_f16x2_to_f32(rs1, h[t]);
                            else rs0 = add_f16x2_to_f32(rs0, h[t]);
                        }
                        l += rs0 + rs1;
                        // keys 64 half + 32c .. + 31: P buffer s columns 32 half + 16c .. + 15
                        tmem_st_32x32b_x16(lane_base + kPCol + static_cast<uint32_t>(s * 64 + 32 * half + 16 * c), h);
                    }
                    tmem_wait_st();
                    tc_fence_before();           // P and the O rescale, if any, before the signal
                    __syncwarp();
                    if (lane == 0) mbar_arrive(p_full(s));
                }
                if (!ok) break;
                // output: O / l after the tile's last P V product (its commit also
                // covers every earlier MMA)
                const int gl = g + nblk - 1;
                ok = mbar_wait_bounded(pv_done(gl & 1), (gl >> 1) & 1, p.timeout_ns, abort_flag, status,
                                       ROLE_SOFTMAX, BAR_PV);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                float l_other = 0.0f;   // the row sum: both halves of the keys
                ok = exchange(l, l_other);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                const float inv = 1.0f / (l + l_other);
                __half* orow = p.O + (static_cast<int64_t>(bh) * p.S + q) * D + half * kOCols;
#pragma unroll 1
                for (int c = 0; c < kOCols / 32; ++c) {
                    uint32_t w[32];
                    tmem_ld_32x32b_x32(o_cols + 32u * c, w);
                    tmem_wait_ld(w);
                    uint32_t h[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        const __half2 hv = __floats2half2_rn(__uint_as_float(w[2 * t]) * inv,
                                                             __uint_as_float(w[2 * t + 1]) * inv);
                        h[t] = *reinterpret_cast<const uint32_t*>(&hv);
                    }
                    if (q < p.S) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
                        for (int t = 0; t < 4; ++t) dst[t] = make_uint4(h[4 * t], h[4 * t + 1], h[4 * t + 2], h[4 * t + 3]);
                    }
                }
                tc_fence_before();           // O read out before the next tile may overwrite it
                __syncwarp();
                if (lane == 0) mbar_arrive(o_free);
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
