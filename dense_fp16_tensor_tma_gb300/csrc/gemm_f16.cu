// C-ABI boundary of the fused fp16 GEMM (declared in include/gemm_f16.h):
// argument checks, device check, execution plan, TMA tensor-map encoding,
// operand repack into scratch (stream-ordered pool, or the fixed buffer of
// the no-alloc entry point), and kernel launch on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <type_traits>

#include "gemm_f16.h"
#include "gemm_kernels.cuh"
#include "gemm_kernels_pair.cuh"
#include "gemm_kernels_swap.cuh"

namespace {

using namespace gemm_f16_dev;

thread_local int t_last_cuda_error = 0;

// Kernel configurations.  The CTA pair (256 x 256 per pair, 3 x 64 KiB ring
// per CTA, 128-deep K stages) is the throughput shape; single-CTA tiles of
// 128 x {256,128,64} give small problems more CTAs; the swap-AB kernel
// (C^T = B^T A^T, tiles of 128 columns x 16/32/64 rows) serves short A.
enum Config : int {
    CFG_AUTO = 0, CFG_PAIR_256 = 1, CFG_128x256 = 2, CFG_128x128 = 3, CFG_128x64 = 4, CFG_SWAP = 5,
    CFG_PAIR_256_WHOLE = 6   // the CTA pair without half-tile tail units (diagnostic)
};
#ifndef GEMM_F16_PAIR_STAGES
#define GEMM_F16_PAIR_STAGES 3
#endif
#ifndef GEMM_F16_PAIR_KSUB
#define GEMM_F16_PAIR_KSUB 2
#endif
#ifndef GEMM_F16_GROUP_M
#define GEMM_F16_GROUP_M 8
#endif
#ifndef GEMM_F16_GROUP_N
#define GEMM_F16_GROUP_N 0
#endif
#ifndef GEMM_F16_SNAKE
#define GEMM_F16_SNAKE 1   // measured: 8192^3 DRAM reads 1.065 -> 1.018 GB per launch, 0.3-0.5 % faster
#endif
constexpr int kStagesPair = GEMM_F16_PAIR_STAGES;   // 3 stages x 64 KiB per CTA
constexpr int kKSubPair = GEMM_F16_PAIR_KSUB;       // 64-deep K sub-blocks per stage
constexpr int kStages256 = 4;   // 4 x 48 KiB ring
constexpr int kStages128 = 6;   // 6 x 32 KiB
constexpr int kStages64 = 8;    // 8 x 24 KiB
constexpr int kGroupM = GEMM_F16_GROUP_M;   // tile-rows per rasterisation group
constexpr int kStagesSwap16 = 12;   // 12 x 18 KiB
constexpr int kStagesSwap32 = 11;   // 11 x 20 KiB
constexpr int kStagesSwap64 = 9;    //  9 x 24 KiB

constexpr int kMaxDevices = 64;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
    bool ready = false;
    int status = GEMM_OK;        // result of the one-time checks
    int num_sms = 0;
    int pair_clusters = 0;       // CTA pairs of the pair kernel that fit on the device at once
    cudaMemPool_t pool = nullptr;  // repack scratch of gemm_f16, created on first use
    bool noalloc_ready = false;
    uint8_t* noalloc_scratch = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
// 2 s per bounded wait; written once at set-up (under g_mu), read by every
// calling thread when it fills kernel parameters
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_force_config{CFG_AUTO};
std::atomic<int> g_force_ksplit{0};   // 0 automatic, 1 never, 2 / 4 that many CTAs per tile
// Programmatic dependent launch on every kernel of the library (GEMM_F16_PDL=0
// in the environment, or gemm_f16_set_pdl(0), turns it off).
std::atomic<int> g_pdl{-1};   // -1: not yet read from the environment

bool pdl_enabled() {
    int v = g_pdl.load(std::memory_order_relaxed);
    if (v < 0) {
        const char* env = std::getenv("GEMM_F16_PDL");
        v = (env != nullptr && env[0] == '0') ? 0 : 1;
        int expected = -1;
        g_pdl.compare_exchange_strong(expected, v);
        v = g_pdl.load(std::memory_order_relaxed);
    }
    return v != 0;
}

// Fault injection for the tests of the error paths (gemm_f16_debug_inject):
// one-shot and process-wide.  GEMM_F16_FAULT_SKIP_LOADS: the next launch of a
// single-CTA tensor-core kernel (128-row tiles or swap-AB) never loads the
// second K block of each CTA's first tile and waits at most g_fault_wait_ns;
// GEMM_F16_FAULT_ENCODE: the next tensor-map encoding fails.
std::atomic<int> g_fault{GEMM_F16_FAULT_NONE};
std::atomic<uint64_t> g_fault_wait_ns{0};

bool take_fault(int kind) {
    if (g_fault.load(std::memory_order_relaxed) != kind) return false;   // the usual case: one load
    int expected = kind;
    return g_fault.compare_exchange_strong(expected, GEMM_F16_FAULT_NONE);
}

// Calls f(std::integral_constant<int, E>) for every epilogue kind E in
// order; stops at and returns the first error.
template <class F>
cudaError_t for_each_epilogue(F f) {
    cudaError_t e = f(std::integral_constant<int, GEMM_EPI_NONE>());
    if (e == cudaSuccess) e = f(std::integral_constant<int, GEMM_EPI_BIAS>());
    if (e == cudaSuccess) e = f(std::integral_constant<int, GEMM_EPI_BIAS_RELU>());
    if (e == cudaSuccess) e = f(std::integral_constant<int, GEMM_EPI_BIAS_GELU_ERF>());
    if (e == cudaSuccess) e = f(std::integral_constant<int, GEMM_EPI_BIAS_SIGMOID>());
    if (e == cudaSuccess) e = f(std::integral_constant<int, GEMM_EPI_BIAS_GELU_TANH>());
    return e;
}

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return GEMM_ERR_CUDA;
}

struct Plan {
    int path = 0;          // 0 none, 1 bias-only, 2 tiled tensor-core kernel, 3 swap-AB kernel
    int cfg = CFG_AUTO;
    int tile_m = 0, tile_n = 0, stages = 0, ctas = 0;
    bool pack_a = false, pack_b = false, vec_store = false;
    int64_t lda_packed = 0, ldb_packed = 0;
    int splits = 1;                        // swap-AB: split-K parts per tile; 128-row tiles: CTAs per cluster
    int dp_tiles = 0, tail_split = 0;      // CTA pair: whole tiles, then half-tile units
    // scratch layout: [A repack][B repack][split-K partials][split-K counters], each 256-aligned
    size_t a_scratch = 0, b_scratch = 0, p_scratch = 0, c_scratch = 0;
    size_t scratch_bytes() const { return a_scratch + b_scratch + p_scratch + c_scratch; }
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// The operands of one call as stored: A is M x K with row pitch lda, or, with
// trans_a, K x M (A^T row-major, pitch lda); B is K x N with pitch ldb, or,
// with trans_b, N x K; C is M x N with pitch ldc.  Pitches in elements.
struct Operands {
    const void* A = nullptr;
    const void* B = nullptr;
    void* C = nullptr;
    int64_t lda = 0, ldb = 0, ldc = 0;
    bool ta = false, tb = false;
    // stored rows x contiguous extent of each operand
    int64_t a_rows(int64_t M, int64_t K) const { return ta ? K : M; }
    int64_t a_cols(int64_t M, int64_t K) const { return ta ? M : K; }
    int64_t b_rows(int64_t N, int64_t K) const { return tb ? N : K; }
    int64_t b_cols(int64_t N, int64_t K) const { return tb ? K : N; }
};

Operands dense_operands(const void* A, const void* B, void* C, int64_t N, int64_t K) {
    Operands op;
    op.A = A;
    op.B = B;
    op.C = C;
    op.lda = K;
    op.ldb = N;
    op.ldc = N;
    return op;
}

int check_args(const Operands& op, const void* bias, int64_t M, int64_t N, int64_t K, int epilogue) {
    constexpr int64_t kLim = int64_t(1) << 31;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M >= kLim || N >= kLim || K >= kLim) return GEMM_ERR_INVALID_ARG;
    if (epilogue < GEMM_EPI_NONE || epilogue > GEMM_EPI_BIAS_GELU_TANH) return GEMM_ERR_INVALID_ARG;
    if (op.lda >= kLim || op.ldb >= kLim || op.ldc >= kLim) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (op.C == nullptr || op.ldc < N) return GEMM_ERR_INVALID_ARG;
    if (K > 0 && (op.A == nullptr || op.B == nullptr)) return GEMM_ERR_INVALID_ARG;
    if (K > 0 && (op.lda < op.a_cols(M, K) || op.ldb < op.b_cols(N, K))) return GEMM_ERR_INVALID_ARG;
    if (epilogue != GEMM_EPI_NONE && bias == nullptr) return GEMM_ERR_INVALID_ARG;
    if (!aligned(op.C, 2) || (K > 0 && (!aligned(op.A, 2) || !aligned(op.B, 2))) ||
        (epilogue != GEMM_EPI_NONE && !aligned(bias, 2)))
        return GEMM_ERR_MISALIGNED;
    // every tile index of the smallest tile shape must fit an int
    if (((M + 127) / 128) * ((N + 63) / 64) >= kLim) return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

// Kernel choice for problems with too few 256 x 256 tiles for the CTA pair to
// take them by rule (and M > 64): 128-row tiles of width 64, 128 or 256,
// possibly with K split across a cluster of 2 or 4 CTAs, and, with at least 32
// K blocks, the CTA pair itself.  Each candidate is costed by the operand bytes
// it moves: the busiest SM's bytes at its intake rate, or every SM's bytes at
// the L2's aggregate rate, whichever takes longer, plus a fixed cost per call
// and, for a split, the cluster reduction (proportional to the tile's width).
// The rates were fitted on a GB300 to replayed-graph timings of every
// candidate on 26 shapes (per SM: 98.7 GB/s single-CTA, 134.4 GB/s in the
// pair; L2 12.2 TB/s; 4.0 us fixed, 5.1 in the pair; 2.5 us per split of a
// 128-wide tile), with the MMAs issued from a converged warp; the fitted model
// then picked the fastest candidate on all 26 and on 7 of 8 further shapes
// (the eighth 3 % slower).  The pair at fewer than 32 K blocks was slower than
// the best single-CTA tile on every shape measured.
struct Choice {
    int cfg;
    int splits;
};

Choice choose_tiles(int64_t M, int64_t N, int64_t K, int num_sms, int pair_clusters, int force, bool allow_split) {
    constexpr double kBytesPerUs = 98.7e3, kPairBytesPerUs = 134.4e3, kL2BytesPerUs = 12.19e6;
    constexpr double kFixedUs = 4.0, kPairFixedUs = 5.14, kSplitUs = 2.5;
    const int64_t kblocks = (K + kBK - 1) / kBK;
    const int64_t tiles_m = (M + 127) / 128;
    const int forced_split = g_force_ksplit.load();
    Choice best{force == CFG_AUTO ? CFG_128x64 : force, 1};
    double best_t = 1e300;
    for (int bn : {64, 128, 256}) {
        const int cfg = bn == 256 ? CFG_128x256 : (bn == 128 ? CFG_128x128 : CFG_128x64);
        if (force != CFG_AUTO && cfg != force) continue;
        const int64_t tiles = tiles_m * ((N + bn - 1) / bn);
        const double per_k = (128.0 + bn) * 128.0;   // operand bytes per K block of a tile
        for (int sp : {1, 2, 4}) {
            if (forced_split == 1 && sp > 1) continue;
            if (forced_split > 1 && sp != forced_split) continue;
            double per_sm, total;
            if (sp > 1) {
                const int64_t kb_per = (kblocks + sp - 1) / sp;
                // one tile per cluster, >= 4 K blocks per CTA, no empty part
                if (!allow_split || tiles * sp > num_sms || kb_per < 4 || kb_per * (sp - 1) >= kblocks) continue;
                per_sm = per_k * kb_per;
                total = per_sm * tiles * sp;
            } else {
                per_sm = per_k * kblocks * ((tiles + num_sms - 1) / num_sms);
                total = per_k * kblocks * tiles;
            }
            const double t = std::max(per_sm / kBytesPerUs, total / kL2BytesPerUs) + kFixedUs +
                             (sp > 1 ? kSplitUs * bn / 128.0 : 0.0);
            if (t < best_t || (forced_split > 1 && best.splits == 1)) {
                best_t = t;
                best = Choice{cfg, sp};
            }
        }
    }
    if (force == CFG_AUTO && forced_split <= 1 && kblocks >= 32 && pair_clusters > 0) {
        // the pair's units: whole 256 x 256 tiles, a partial last wave of R <= G/2
        // tiles as 2R half tiles (256 x 128), as make_plan lays them out; per SM
        // and K block a whole tile moves 128 rows of A and 128 columns of B, a
        // half tile 128 rows and 64 columns
        const int64_t G = pair_clusters;
        const int64_t T = ((M + 255) / 256) * ((N + 255) / 256);
        const int64_t R = T % G;
        const int64_t halves = (R > 0 && 2 * R <= G) ? 2 * R : 0;
        const int64_t whole = T - halves / 2;
        const double per_sm = static_cast<double>(kblocks) *
                              (32768.0 * static_cast<double>((whole + G - 1) / G) + (halves ? 24576.0 : 0.0));
        const double total = static_cast<double>(kblocks) *
                             (65536.0 * static_cast<double>(whole) + 49152.0 * static_cast<double>(halves));
        const double t = std::max(per_sm / kPairBytesPerUs, total / kL2BytesPerUs) + kPairFixedUs;
        if (t < best_t) best = Choice{CFG_PAIR_256, 1};
    }
    return best;
}

Plan make_plan(const Operands& op, int64_t M, int64_t N, int64_t K, int num_sms, int pair_clusters, int force,
               bool allow_split = true) {
    Plan pl;
    if (M == 0 || N == 0) return pl;
    if (K == 0) {
        pl.path = 1;
        pl.ctas = static_cast<int>(std::min<int64_t>((M * N + 255) / 256, int64_t(num_sms) * 8));
        return pl;
    }
    pl.path = 2;
    // TMA wants a 16-byte aligned base and a pitch of a multiple of 16 bytes;
    // otherwise the operand is first copied, in its own layout, to scratch
    pl.pack_a = !(aligned(op.A, 16) && op.lda % 8 == 0);
    pl.pack_b = !(aligned(op.B, 16) && op.ldb % 8 == 0);
    pl.lda_packed = pl.pack_a ? round_up(op.a_cols(M, K), 8) : op.lda;
    pl.ldb_packed = pl.pack_b ? round_up(op.b_cols(N, K), 8) : op.ldb;
    pl.a_scratch = pl.pack_a ? align256(static_cast<size_t>(op.a_rows(M, K) * pl.lda_packed * 2)) : 0;
    pl.b_scratch = pl.pack_b ? align256(static_cast<size_t>(op.b_rows(N, K) * pl.ldb_packed * 2)) : 0;
    pl.vec_store = aligned(op.C, 16) && op.ldc % 8 == 0;
    const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
    int cfg = force;
    bool tail_halves = true;
    if (cfg == CFG_PAIR_256_WHOLE) {
        cfg = CFG_PAIR_256;
        tail_halves = false;
    }
    int ksplit = 1;   // 128-row tiles: CTAs per cluster sharing a tile's K
    if (cfg == CFG_AUTO) {
        if (M <= 64) {
            cfg = CFG_SWAP;
        } else if (4 * pair_tiles >= pair_clusters && g_force_ksplit.load() <= 1) {
            // the CTA pair, also with a partial first wave: it loads half the
            // operand bytes per output of a 128 x 128 tile per SM (measured
            // fastest down to a quarter of the pairs busy, e.g. 2048 x 2048 x
            // 1024: 12.0 us against 13.9 for the best single-CTA tile)
            cfg = CFG_PAIR_256;
        } else {
            const Choice c = choose_tiles(M, N, K, num_sms, pair_clusters, CFG_AUTO, allow_split);
            cfg = c.cfg;
            ksplit = c.splits;
        }
    } else if (cfg == CFG_128x256 || cfg == CFG_128x128 || cfg == CFG_128x64) {
        ksplit = choose_tiles(M, N, K, num_sms, pair_clusters, cfg, allow_split).splits;
    }
    pl.cfg = cfg;
    switch (cfg) {
        case CFG_PAIR_256: {
            pl.tile_m = 256; pl.tile_n = 256; pl.stages = kStagesPair;
            const int64_t G = std::max(1, pair_clusters);
            // A partial last wave of R tiles (R <= G/2) runs as 2R half tiles
            // (256 x 128) on the pairs: it then costs half a tile, not a whole one.
            const int64_t R = pair_tiles % G;
            pl.dp_tiles = static_cast<int>(pair_tiles);
            if (tail_halves && R > 0 && 2 * R <= G) {
                pl.dp_tiles = static_cast<int>(pair_tiles - R);
                pl.tail_split = 1;
            }
            const int64_t units = pl.dp_tiles + (pl.tail_split ? 2 * (pair_tiles - pl.dp_tiles) : 0);
            pl.ctas = 2 * static_cast<int>(std::min<int64_t>(units, G));
            break;
        }
        case CFG_SWAP:
            pl.path = 3;
            // A stored K x M is one MN-major box of 64 rows (a 128-byte swizzle row)
            pl.tile_m = (M <= 16 && !op.ta) ? 16 : ((M <= 32 && !op.ta) ? 32 : 64);
            pl.tile_n = 128;
            pl.stages = pl.tile_m == 16 ? kStagesSwap16 : (pl.tile_m == 32 ? kStagesSwap32 : kStagesSwap64);
            break;
        case CFG_128x256: pl.tile_m = 128; pl.tile_n = 256; pl.stages = kStages256; break;
        case CFG_128x128: pl.tile_m = 128; pl.tile_n = 128; pl.stages = kStages128; break;
        default: pl.tile_m = 128; pl.tile_n = 64; pl.stages = kStages64; break;
    }
    if (cfg != CFG_PAIR_256 && cfg != CFG_SWAP) pl.splits = ksplit;
    if (cfg != CFG_PAIR_256) {
        const int64_t tiles = ((M + pl.tile_m - 1) / pl.tile_m) * ((N + pl.tile_n - 1) / pl.tile_n);
        if (cfg == CFG_SWAP && allow_split && tiles < num_sms) {
            // a CTA streams HBM at a bounded rate: spread each tile's K over
            // more CTAs, keeping at least 8 K-blocks (512) per part
            const int64_t kblocks = (K + kBK - 1) / kBK;
            int64_t S = std::min<int64_t>({num_sms / tiles, kblocks / 8, 16});
            if (S > 1) {
                const int64_t kb_per = (kblocks + S - 1) / S;
                S = (kblocks + kb_per - 1) / kb_per;   // no empty part
            }
            pl.splits = static_cast<int>(std::max<int64_t>(1, S));
        }
        if (pl.splits > 1 && cfg == CFG_SWAP) {
            pl.p_scratch = align256(static_cast<size_t>(tiles) * pl.splits * pl.tile_m * pl.tile_n * 4);
            pl.c_scratch = align256(static_cast<size_t>(tiles) * 4 * 4);
        }
        pl.ctas = static_cast<int>(std::min<int64_t>(tiles * pl.splits, num_sms));
    }
    return pl;
}

cudaLaunchConfig_t launch_config(int ctas, uint32_t smem, cudaStream_t s) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cfg;
}

// Launch attributes of a kernel of this library: a cluster of `cluster` CTAs
// (if > 1) and programmatic stream serialization (if enabled): the kernel may
// start while the previous one in the stream finishes; every kernel here
// calls grid_dependency_wait() before touching global memory.
struct LaunchAttrs {
    cudaLaunchAttribute a[2];
    unsigned n = 0;
    LaunchAttrs(int cluster, bool pdl) {
        std::memset(a, 0, sizeof(a));
        if (cluster > 1) {
            a[n].id = cudaLaunchAttributeClusterDimension;
            a[n].val.clusterDim.x = static_cast<unsigned>(cluster);
            a[n].val.clusterDim.y = 1;
            a[n].val.clusterDim.z = 1;
            ++n;
        }
        if (pdl) {
            a[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            a[n].val.programmaticStreamSerializationAllowed = 1;
            ++n;
        }
    }
    void apply(cudaLaunchConfig_t& cfg) {
        cfg.attrs = n ? a : nullptr;
        cfg.numAttrs = n;
    }
};

// One-time per-device checks and kernel attributes (allocates nothing).
// Called with g_mu held.
int init_common_locked(int dev, DeviceState& st) {
    if (st.ready) return st.status;
    int major = 0, minor = 0, sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (major != 10 || minor != 3) {
        st.ready = true;
        st.status = GEMM_ERR_UNSUPPORTED_DEVICE;
        return st.status;
    }
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return cuda_fail(e != cudaSuccess ? e : cudaErrorSymbolNotFound);
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    e = for_each_epilogue([](auto epi) {
        constexpr int E = decltype(epi)::value;
        constexpr uint32_t smem = SmemPlanPair<kStagesPair, kKSubPair>::kDynamicBytes;
        cudaError_t r = cudaFuncSetAttribute(gemm_f16_tc2_kernel<kStagesPair, kKSubPair, E>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(gemm_f16_tc2_grouped_kernel<kStagesPair, kKSubPair, E>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        return r;
    });
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_f16_tc_kernel<256, kStages256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SmemPlan<256, kStages256>::kDynamicBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_f16_tc_kernel<128, kStages128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SmemPlan<128, kStages128>::kDynamicBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_f16_tc_kernel<64, kStages64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SmemPlan<64, kStages64>::kDynamicBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_f16_swap_kernel<16, kStagesSwap16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SmemPlanSwap<16, kStagesSwap16>::kDynamicBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_f16_swap_kernel<32, kStagesSwap32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SmemPlanSwap<32, kStagesSwap32>::kDynamicBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_f16_swap_kernel<64, kStagesSwap64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SmemPlanSwap<64, kStagesSwap64>::kDynamicBytes);
    if (e != cudaSuccess) return cuda_fail(e);
    // How many CTA pairs fit at once decides the persistent grid of the pair kernel.
    {
        cudaLaunchConfig_t cfg = launch_config(sms, SmemPlanPair<kStagesPair, kKSubPair>::kDynamicBytes, nullptr);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(
                                               gemm_f16_tc2_kernel<kStagesPair, kKSubPair, GEMM_EPI_BIAS_GELU_ERF>),
                                           &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = sms / 2;
        }
        st.pair_clusters = n;
    }
    if (const char* env = std::getenv("GEMM_F16_TIMEOUT_MS")) {
        const long ms = std::strtol(env, nullptr, 10);
        if (ms > 0) g_timeout_ns.store(static_cast<uint64_t>(ms) * 1000000ull, std::memory_order_relaxed);
    }
    st.num_sms = sms;
    st.ready = true;
    st.status = GEMM_OK;
    return GEMM_OK;
}

int init_device(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    return init_common_locked(dev, g_dev[dev]);
}

// The library-owned pool for gemm_f16's repack scratch (keeps memory cached
// between calls without touching the device's default pool).
int ensure_pool(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[dev];
    if (st.pool != nullptr) return GEMM_OK;
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaError_t e = cudaMemPoolCreate(&st.pool, &props);
    if (e != cudaSuccess) {
        st.pool = nullptr;
        return cuda_fail(e);
    }
    uint64_t keep = ~0ull;
    cudaMemPoolSetAttribute(st.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    return GEMM_OK;
}

// Encoded tensor maps of recent calls.  A map is a pure function of its
// arguments (address, extents, pitch, box; the rest is fixed), so a hit is
// exactly the map a new encoding would give; repeated calls on the same
// buffers (a layer's weights, a serving loop) skip the encoder.
struct TensorMapCache {
    static constexpr int kWays = 16;
    struct Entry {
        const void* ptr = nullptr;
        int64_t inner = 0, outer = 0, ld = 0;
        int box_inner = 0, box_outer = 0;
        CUtensorMap map;
    };
    Entry e[kWays];
    int next = 0;
};
thread_local TensorMapCache t_maps;

// 3-D view of an MN-major operand whose MN extent and pitch are multiples of
// 64: (64 elements, K rows, MN / 64 groups of 64), box 64 x 64 x 2, so one
// load brings the two 64-wide boxes of a 128-wide operand slice (laid out in
// shared memory exactly as two 2-D boxes 8 KiB apart) and reads 256
// contiguous bytes of each K row instead of two 128-byte pieces: measured
// 2-3 % faster with B stored K x N and 13-22 % with A stored K x M (the
// CTA-pair kernels).  Every element of the view lies inside a row of the
// operand (64 j + i < MN <= pitch), which is why MN must be a multiple of 64;
// coordinates past K or past MN / 64 read as zeros without touching memory.
bool mn3d_ok(bool mn_major, int64_t mn, int64_t ld) { return mn_major && mn % 64 == 0 && ld % 64 == 0; }

// An injected encoding failure (what the driver returns for an invalid map).
int injected_encode_failure() {
    t_last_cuda_error = static_cast<int>(CUDA_ERROR_INVALID_VALUE);
    return GEMM_ERR_CUDA;
}

int encode_mn3d(CUtensorMap* m, const void* ptr, int64_t mn, int64_t k, int64_t ld) {
    if (take_fault(GEMM_F16_FAULT_ENCODE)) return injected_encode_failure();
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(mn / 64)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, 128};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBK), 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

// 2-D fp16 tensor map: `inner` contiguous elements per row, `outer` rows,
// row pitch `ld` elements, box `box_inner` x `box_outer`, 128-byte swizzle,
// zero fill outside the tensor.
int encode_2d(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int64_t ld, int box_inner,
              int box_outer) {
    if (take_fault(GEMM_F16_FAULT_ENCODE)) return injected_encode_failure();
    for (const TensorMapCache::Entry& c : t_maps.e) {
        if (c.ptr == ptr && ptr != nullptr && c.inner == inner && c.outer == outer && c.ld == ld &&
            c.box_inner == box_inner && c.box_outer == box_outer) {
            *m = c.map;
            return GEMM_OK;
        }
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return GEMM_ERR_CUDA;
    }
    TensorMapCache::Entry& c = t_maps.e[t_maps.next];
    t_maps.next = (t_maps.next + 1) % TensorMapCache::kWays;
    c.ptr = ptr;
    c.inner = inner;
    c.outer = outer;
    c.ld = ld;
    c.box_inner = box_inner;
    c.box_outer = box_outer;
    c.map = *m;
    return GEMM_OK;
}

int launch_repack(uint16_t* dst, const void* src, int64_t rows, int64_t cols, int64_t ld_src, int64_t ld_dst,
                  cudaStream_t s) {
    // 256 threads, 8 elements per thread: 2048 per block along a row; groups of
    // kRepackRows rows per thread once there are blocks enough for every SM
    // several times over (measured: 8192 x 8191 and 1000 x 5003 copies gain,
    // a 300 x 203 one loses with groups)
    const int64_t col_blocks = (cols + 2047) / 2048;
    const int group = col_blocks * rows >= 2048 ? kRepackRows : 1;
    cudaLaunchConfig_t cfg = launch_config(1, 0, s);
    cfg.gridDim = dim3(static_cast<unsigned>(col_blocks),
                       static_cast<unsigned>(std::min<int64_t>((rows + group - 1) / group, 65535)));
    cfg.blockDim = dim3(256);
    LaunchAttrs la(1, pdl_enabled());
    la.apply(cfg);
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_f16_repack_kernel, dst, static_cast<const uint16_t*>(src), rows,
                                       cols, ld_src, ld_dst, group);
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
}

template <int BN, int STAGES>
int launch_tc(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& prm, int ctas, cudaStream_t s) {
    cudaLaunchConfig_t cfg = launch_config(ctas, SmemPlan<BN, STAGES>::kDynamicBytes, s);
    LaunchAttrs la(prm.splits, pdl_enabled());   // split K: clusters of `splits` CTAs
    la.apply(cfg);
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_f16_tc_kernel<BN, STAGES>, ta, tb, prm);
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
}

template <int MT, int STAGES>
int launch_swap(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& prm, int ctas, cudaStream_t s) {
    cudaLaunchConfig_t cfg = launch_config(ctas, SmemPlanSwap<MT, STAGES>::kDynamicBytes, s);
    cfg.blockDim = dim3(kSwapThreads);
    LaunchAttrs la(1, pdl_enabled());
    la.apply(cfg);
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_f16_swap_kernel<MT, STAGES>, ta, tb, prm);
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
}

int launch_tc_pair(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& prm, int ctas, cudaStream_t s) {
    cudaLaunchConfig_t cfg = launch_config(ctas, SmemPlanPair<kStagesPair, kKSubPair>::kDynamicBytes, s);
    LaunchAttrs la(2, pdl_enabled());
    la.apply(cfg);
    cudaError_t e = cudaErrorInvalidValue;
    switch (prm.epi) {
        case GEMM_EPI_NONE: e = cudaLaunchKernelEx(&cfg, gemm_f16_tc2_kernel<kStagesPair, kKSubPair, 0>, ta, tb, prm); break;
        case GEMM_EPI_BIAS: e = cudaLaunchKernelEx(&cfg, gemm_f16_tc2_kernel<kStagesPair, kKSubPair, 1>, ta, tb, prm); break;
        case GEMM_EPI_BIAS_RELU:
            e = cudaLaunchKernelEx(&cfg, gemm_f16_tc2_kernel<kStagesPair, kKSubPair, 2>, ta, tb, prm);
            break;
        case GEMM_EPI_BIAS_GELU_ERF:
            e = cudaLaunchKernelEx(&cfg, gemm_f16_tc2_kernel<kStagesPair, kKSubPair, 3>, ta, tb, prm);
            break;
        case GEMM_EPI_BIAS_SIGMOID:
            e = cudaLaunchKernelEx(&cfg, gemm_f16_tc2_kernel<kStagesPair, kKSubPair, 4>, ta, tb, prm);
            break;
        case GEMM_EPI_BIAS_GELU_TANH:
            e = cudaLaunchKernelEx(&cfg, gemm_f16_tc2_kernel<kStagesPair, kKSubPair, 5>, ta, tb, prm);
            break;
        default: break;
    }
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
}

// Kernel parameters of one problem (split-K and tail fields left empty).
GemmParams kernel_params(const Operands& op, const __half* biasp, int64_t M, int64_t N, int64_t K, int epilogue) {
    GemmParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.C = static_cast<__half*>(op.C);
    prm.bias = biasp;
    prm.M = static_cast<int>(M);
    prm.N = static_cast<int>(N);
    prm.K = static_cast<int>(K);
    prm.ldc = static_cast<int>(op.ldc);
    prm.trans_a = op.ta ? 1 : 0;
    prm.trans_b = op.tb ? 1 : 0;
    prm.epi = epilogue;
    prm.vec_store = (aligned(op.C, 16) && op.ldc % 8 == 0) ? 1 : 0;
    prm.bias_vec = (biasp != nullptr && aligned(biasp, 16)) ? 1 : 0;
    prm.group_m = kGroupM;
    prm.group_n = GEMM_F16_GROUP_N;
    prm.snake = GEMM_F16_SNAKE;
    prm.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    prm.splits = 1;
    prm.fault_skip_kb = -1;
    return prm;
}

// Everything after scratch is settled, all on stream `s`: the tensor maps
// (encoded first, so that an encoding failure enqueues nothing), the repacks
// (into `scratch`, which holds pl.a_scratch + pl.b_scratch bytes when a
// repack is planned), the split-K counters' reset, and the tensor-core kernel.
int enqueue_plan(const Plan& pl, const Operands& op, const __half* biasp, int64_t M, int64_t N, int64_t K,
                 int epilogue, uint8_t* scratch, cudaStream_t s) {
    const void* a_src = pl.pack_a ? static_cast<const void*>(scratch) : op.A;
    uint16_t* bdst = pl.pack_b ? reinterpret_cast<uint16_t*>(scratch + pl.a_scratch) : nullptr;
    const void* b_src = pl.pack_b ? static_cast<const void*>(bdst) : op.B;
    CUtensorMap ta, tb;
    // A boxes: 64 K x 128 rows (64 K x MT rows for the swap-AB kernel), or,
    // for A stored K x M, 64 rows x 64 K; B boxes: 64 x 64 in either layout
    const bool pair = pl.cfg == CFG_PAIR_256;
    const bool a3 = pair && mn3d_ok(op.ta, M, pl.lda_packed);
    const bool b3 = pair && mn3d_ok(!op.tb, N, pl.ldb_packed);
    int st = a3 ? encode_mn3d(&ta, a_src, M, K, pl.lda_packed)
             : op.ta ? encode_2d(&ta, a_src, M, K, pl.lda_packed, 64, kBK)
                     : encode_2d(&ta, a_src, K, M, pl.lda_packed, kBK, pl.path == 3 ? pl.tile_m : kBM);
    if (st == GEMM_OK) {
        st = b3 ? encode_mn3d(&tb, b_src, N, K, pl.ldb_packed)
             : op.tb ? encode_2d(&tb, b_src, K, N, pl.ldb_packed, kBK, 64)
                     : encode_2d(&tb, b_src, N, K, pl.ldb_packed, 64, kBK);
    }
    if (st != GEMM_OK) return st;
    if (pl.pack_a)
        st = launch_repack(reinterpret_cast<uint16_t*>(scratch), op.A, op.a_rows(M, K), op.a_cols(M, K), op.lda,
                           pl.lda_packed, s);
    if (st == GEMM_OK && pl.pack_b)
        st = launch_repack(bdst, op.B, op.b_rows(N, K), op.b_cols(N, K), op.ldb, pl.ldb_packed, s);
    float* partials = nullptr;
    unsigned int* counters = nullptr;
    if (st == GEMM_OK && pl.splits > 1) {
        partials = reinterpret_cast<float*>(scratch + pl.a_scratch + pl.b_scratch);
        counters = reinterpret_cast<unsigned int*>(scratch + pl.a_scratch + pl.b_scratch + pl.p_scratch);
        const cudaError_t e = cudaMemsetAsync(counters, 0, pl.c_scratch, s);   // every slice starts at zero parts
        if (e != cudaSuccess) st = cuda_fail(e);
    }
    if (st != GEMM_OK) return st;
    GemmParams prm = kernel_params(op, biasp, M, N, K, epilogue);
    prm.mn3d_a = a3 ? 1 : 0;
    prm.mn3d_b = b3 ? 1 : 0;
    prm.dp_tiles = pl.dp_tiles;
    prm.tail_split = pl.tail_split;
    prm.splits = pl.splits;
    prm.partials = partials;
    prm.counters = counters;
    if (!pair && take_fault(GEMM_F16_FAULT_SKIP_LOADS)) {
        prm.fault_skip_kb = 1;
        prm.timeout_ns = g_fault_wait_ns.load(std::memory_order_relaxed);
    }
    switch (pl.cfg) {
        case CFG_PAIR_256: return launch_tc_pair(ta, tb, prm, pl.ctas, s);
        case CFG_SWAP:
            if (pl.tile_m == 16) return launch_swap<16, kStagesSwap16>(ta, tb, prm, pl.ctas, s);
            if (pl.tile_m == 32) return launch_swap<32, kStagesSwap32>(ta, tb, prm, pl.ctas, s);
            return launch_swap<64, kStagesSwap64>(ta, tb, prm, pl.ctas, s);
        case CFG_128x256: return launch_tc<256, kStages256>(ta, tb, prm, pl.ctas, s);
        case CFG_128x128: return launch_tc<128, kStages128>(ta, tb, prm, pl.ctas, s);
        default: return launch_tc<64, kStages64>(ta, tb, prm, pl.ctas, s);
    }
}

int enqueue_bias_only(const Plan& pl, const __half* biasp, void* C, int64_t ldc, int64_t M, int64_t N, int epilogue,
                      cudaStream_t s) {
    cudaLaunchConfig_t cfg = launch_config(pl.ctas, 0, s);
    cfg.blockDim = dim3(256);
    LaunchAttrs la(1, pdl_enabled());
    la.apply(cfg);
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_f16_bias_only_kernel, static_cast<__half*>(C), biasp, M, N, ldc,
                                       epilogue);
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
}

// ---------------------------------------------------------------- grouped GEMM
Operands problem_operands(const gemm_f16_problem_t& q, int flags) {
    Operands op;
    op.A = q.A;
    op.B = q.B;
    op.C = q.C;
    op.lda = q.lda;
    op.ldb = q.ldb;
    op.ldc = q.ldc;
    op.ta = (flags & GEMM_F16_TRANS_A) != 0;
    op.tb = (flags & GEMM_F16_TRANS_B) != 0;
    return op;
}

int launch_grouped(const GroupedParams& gp, int ctas, cudaStream_t s) {
    cudaLaunchConfig_t cfg = launch_config(ctas, SmemPlanPair<kStagesPair, kKSubPair>::kDynamicBytes, s);
    LaunchAttrs la(2, pdl_enabled());
    la.apply(cfg);
    cudaError_t e = cudaErrorInvalidValue;
    switch (gp.prob[0].epi) {
        case GEMM_EPI_NONE: e = cudaLaunchKernelEx(&cfg, gemm_f16_tc2_grouped_kernel<kStagesPair, kKSubPair, 0>, gp); break;
        case GEMM_EPI_BIAS: e = cudaLaunchKernelEx(&cfg, gemm_f16_tc2_grouped_kernel<kStagesPair, kKSubPair, 1>, gp); break;
        case GEMM_EPI_BIAS_RELU:
            e = cudaLaunchKernelEx(&cfg, gemm_f16_tc2_grouped_kernel<kStagesPair, kKSubPair, 2>, gp);
            break;
        case GEMM_EPI_BIAS_GELU_ERF:
            e = cudaLaunchKernelEx(&cfg, gemm_f16_tc2_grouped_kernel<kStagesPair, kKSubPair, 3>, gp);
            break;
        case GEMM_EPI_BIAS_SIGMOID:
            e = cudaLaunchKernelEx(&cfg, gemm_f16_tc2_grouped_kernel<kStagesPair, kKSubPair, 4>, gp);
            break;
        case GEMM_EPI_BIAS_GELU_TANH:
            e = cudaLaunchKernelEx(&cfg, gemm_f16_tc2_grouped_kernel<kStagesPair, kKSubPair, 5>, gp);
            break;
        default: break;
    }
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
}

// Kernel parameter of one grouped launch, filled per launch (the launch call
// copies it).
thread_local GroupedParams t_grouped;

// ---------------------------------------------------------------- no-alloc variant
// Fixed repack buffer for gemm_f16_noalloc, part of the module image: every
// device that loads this library holds it until the process exits.  In host
// code `g_noalloc_scratch` names a host-side stand-in, never the device
// buffer; its device address comes from cudaGetSymbolAddress in
// init_device_noalloc and is what the kernels and tensor maps receive.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Per-device set-up of the no-alloc path: the common checks plus the device
// address of the fixed buffer.  Allocates nothing.
int init_device_noalloc(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[dev];
    const int s = init_common_locked(dev, st);
    if (s != GEMM_OK) return s;
    if (st.noalloc_ready) return GEMM_OK;
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    st.noalloc_scratch = static_cast<uint8_t*>(ptr);
    st.noalloc_ready = true;
    return GEMM_OK;
}

// The plan gemm_f16_noalloc runs: gemm_f16's, inside the fixed buffer.
// Without room for the split-K partials the problem runs unsplit; if even
// the repacks alone do not fit, *fits is false.
Plan make_noalloc_plan(const Operands& op, int64_t M, int64_t N, int64_t K, int num_sms, int pair_clusters,
                       int force, bool* fits) {
    Plan pl = make_plan(op, M, N, K, num_sms, pair_clusters, force);
    if (pl.scratch_bytes() > kNoAllocScratchBytes) pl = make_plan(op, M, N, K, num_sms, pair_clusters, force, false);
    *fits = pl.scratch_bytes() <= kNoAllocScratchBytes;
    return pl;
}

}  // namespace

extern "C" {

const char* gemm_f16_status_string(int status) {
    switch (status) {
        case GEMM_OK: return "ok";
        case GEMM_ERR_INVALID_ARG: return "invalid argument";
        case GEMM_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3, sm_103a)";
        case GEMM_ERR_MISALIGNED: return "pointer not 2-byte aligned";
        case GEMM_ERR_CUDA: return "CUDA error";
        case GEMM_ERR_TIMEOUT: return "device-side bounded wait timed out";
        case GEMM_ERR_NO_MEMORY: return "out of device memory for repack scratch";
        case GEMM_ERR_SCRATCH_LIMIT:
            return "repack needs more than the 32 MiB fixed buffer of gemm_f16_noalloc (use gemm_f16)";
        default: return "unknown status";
    }
}

int gemm_f16_last_cuda_error(void) { return t_last_cuda_error; }

int gemm_f16_set_pdl(int enable) {
    const int prev = pdl_enabled() ? 1 : 0;
    g_pdl.store(enable ? 1 : 0);
    return prev;
}

int gemm_f16_force_config(int config) {
    if (config < CFG_AUTO || config > CFG_PAIR_256_WHOLE) return -1;
    return g_force_config.exchange(config);
}

int gemm_f16_force_ksplit(int splits) {
    if (splits != 0 && splits != 1 && splits != 2 && splits != 4) return -1;
    return g_force_ksplit.exchange(splits);
}

int gemm_f16_plan_ex(const void* A, int64_t lda, const void* B, int64_t ldb, const void* bias, const void* C,
                     int64_t ldc, int64_t M, int64_t N, int64_t K, int epilogue, int flags, int num_sms,
                     int64_t plan[11]) {
    if (plan == nullptr || num_sms <= 0) return GEMM_ERR_INVALID_ARG;
    if (flags & ~(GEMM_F16_TRANS_A | GEMM_F16_TRANS_B | GEMM_F16_PLAN_NOALLOC)) return GEMM_ERR_INVALID_ARG;
    Operands op;
    op.A = A;
    op.B = B;
    op.C = const_cast<void*>(C);
    op.lda = lda;
    op.ldb = ldb;
    op.ldc = ldc;
    op.ta = (flags & GEMM_F16_TRANS_A) != 0;
    op.tb = (flags & GEMM_F16_TRANS_B) != 0;
    const int st = check_args(op, bias, M, N, K, epilogue);
    if (st != GEMM_OK) return st;
    Plan pl;
    if (flags & GEMM_F16_PLAN_NOALLOC) {
        bool fits = true;
        pl = make_noalloc_plan(op, M, N, K, num_sms, num_sms / 2, g_force_config.load(), &fits);
        if (!fits) return GEMM_ERR_SCRATCH_LIMIT;
    } else {
        pl = make_plan(op, M, N, K, num_sms, num_sms / 2, g_force_config.load());
    }
    plan[0] = pl.path;
    plan[1] = pl.tile_m;
    plan[2] = pl.tile_n;
    plan[3] = pl.stages;
    plan[4] = pl.ctas;
    plan[5] = pl.pack_a;
    plan[6] = pl.pack_b;
    plan[7] = pl.vec_store;
    plan[8] = pl.splits;
    plan[9] = static_cast<int64_t>(pl.scratch_bytes());
    plan[10] = pl.tail_split ? static_cast<int64_t>(pl.dp_tiles) : -1;
    return GEMM_OK;
}

int gemm_f16_plan(const void* A, const void* B, const void* bias, const void* C, int64_t M, int64_t N, int64_t K,
                  int epilogue, int num_sms, int64_t plan[11]) {
    return gemm_f16_plan_ex(A, K, B, N, bias, C, N, M, N, K, epilogue, 0, num_sms, plan);
}

int gemm_f16_ex(const void* A, int64_t lda, const void* B, int64_t ldb, const void* bias, void* C, int64_t ldc,
                int64_t M, int64_t N, int64_t K, int epilogue, int flags, void* cuda_stream) {
    if (flags & ~(GEMM_F16_TRANS_A | GEMM_F16_TRANS_B)) return GEMM_ERR_INVALID_ARG;
    Operands op;
    op.A = A;
    op.B = B;
    op.C = C;
    op.lda = lda;
    op.ldb = ldb;
    op.ldc = ldc;
    op.ta = (flags & GEMM_F16_TRANS_A) != 0;
    op.tb = (flags & GEMM_F16_TRANS_B) != 0;
    int st = check_args(op, bias, M, N, K, epilogue);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    st = init_device(dev);
    if (st != GEMM_OK) return st;
    const DeviceState& ds = g_dev[dev];
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const Plan pl = make_plan(op, M, N, K, ds.num_sms, ds.pair_clusters, g_force_config.load());
    const __half* biasp = epilogue == GEMM_EPI_NONE ? nullptr : static_cast<const __half*>(bias);
    if (pl.path == 1) return enqueue_bias_only(pl, biasp, C, ldc, M, N, epilogue, s);

    void* scratch = nullptr;
    const size_t scratch_bytes = pl.scratch_bytes();
    if (scratch_bytes > 0) {
        st = ensure_pool(dev);
        if (st != GEMM_OK) return st;
        e = cudaMallocFromPoolAsync(&scratch, scratch_bytes, ds.pool, s);
        if (e != cudaSuccess) {
            t_last_cuda_error = static_cast<int>(e);
            cudaGetLastError();
            return GEMM_ERR_NO_MEMORY;
        }
    }
    st = enqueue_plan(pl, op, biasp, M, N, K, epilogue, static_cast<uint8_t*>(scratch), s);
    if (scratch != nullptr) {
        e = cudaFreeAsync(scratch, s);   // stream-ordered: freed after the GEMM has read it
        if (e != cudaSuccess && st == GEMM_OK) st = cuda_fail(e);
    }
    return st;
}

int gemm_f16(const void* A, const void* B, const void* bias, void* C, int64_t M, int64_t N, int64_t K, int epilogue,
             void* cuda_stream) {
    return gemm_f16_ex(A, K, B, N, bias, C, N, M, N, K, epilogue, 0, cuda_stream);
}

int gemm_f16_noalloc(const void* A, const void* B, const void* bias, void* C, int64_t M, int64_t N, int64_t K,
                     int epilogue, void* cuda_stream) {
    const Operands op = dense_operands(A, B, C, N, K);
    int st = check_args(op, bias, M, N, K, epilogue);
    if (st != GEMM_OK) return st;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    // the set-up (and with it the fixed buffer's reservation) also runs for an
    // empty problem, so that a caller can take it at start-up
    st = init_device_noalloc(dev);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    const DeviceState& ds = g_dev[dev];
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    // Same scratch layout as gemm_f16, inside the fixed buffer.  The repacks
    // need no zeroed memory (the tensor maps stop at the true extents); the
    // split-K counters are zeroed by a stream-ordered memset in enqueue_plan.
    bool fits = true;
    const Plan pl = make_noalloc_plan(op, M, N, K, ds.num_sms, ds.pair_clusters, g_force_config.load(), &fits);
    const __half* biasp = epilogue == GEMM_EPI_NONE ? nullptr : static_cast<const __half*>(bias);
    if (pl.path == 1) return enqueue_bias_only(pl, biasp, C, N, M, N, epilogue, s);
    if (!fits) return GEMM_ERR_SCRATCH_LIMIT;
    return enqueue_plan(pl, op, biasp, M, N, K, epilogue, ds.noalloc_scratch, s);
}

int gemm_f16_grouped(const gemm_f16_problem_t* problems, int count, int epilogue, int flags, void* cuda_stream) {
    if (count < 0 || (count > 0 && problems == nullptr)) return GEMM_ERR_INVALID_ARG;
    if (flags & ~(GEMM_F16_TRANS_A | GEMM_F16_TRANS_B)) return GEMM_ERR_INVALID_ARG;
    for (int i = 0; i < count; ++i) {
        const gemm_f16_problem_t& q = problems[i];
        const int st = check_args(problem_operands(q, flags), q.bias, q.M, q.N, q.K, epilogue);
        if (st != GEMM_OK) return st;
    }
    bool any = false;
    for (int i = 0; i < count; ++i) any = any || (problems[i].M > 0 && problems[i].N > 0);
    if (!any) return GEMM_OK;   // nothing to compute: no CUDA call
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    int st = init_device(dev);
    if (st != GEMM_OK) return st;
    const DeviceState& ds = g_dev[dev];
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);

    // Repack scratch for every operand a tensor map cannot describe, in one
    // stream-ordered allocation: [problem 0 A][problem 0 B][problem 1 A] ...
    struct Prep {
        Operands op;
        Plan pl;          // repack decisions and pitches (tile fields unused)
        size_t off = 0;   // this problem's scratch offset
    };
    Prep* prep = new (std::nothrow) Prep[count > 0 ? count : 1];
    if (prep == nullptr) return GEMM_ERR_NO_MEMORY;
    size_t scratch_bytes = 0;
    for (int i = 0; i < count; ++i) {
        const gemm_f16_problem_t& q = problems[i];
        prep[i].op = problem_operands(q, flags);
        prep[i].pl = make_plan(prep[i].op, q.M, q.N, q.K, ds.num_sms, ds.pair_clusters, CFG_PAIR_256_WHOLE, false);
        prep[i].off = scratch_bytes;
        scratch_bytes += prep[i].pl.a_scratch + prep[i].pl.b_scratch;
    }
    uint8_t* scratch = nullptr;
    if (scratch_bytes > 0) {
        st = ensure_pool(dev);
        if (st == GEMM_OK) {
            void* ptr = nullptr;
            e = cudaMallocFromPoolAsync(&ptr, scratch_bytes, ds.pool, s);
            if (e != cudaSuccess) {
                t_last_cuda_error = static_cast<int>(e);
                cudaGetLastError();
                st = GEMM_ERR_NO_MEMORY;
            }
            scratch = static_cast<uint8_t*>(ptr);
        }
    }
    GroupedParams& gp = t_grouped;
    gp.count = 0;
    gp.tile_start[0] = 0;
    auto flush = [&]() -> int {
        if (gp.count == 0) return GEMM_OK;
        const int tiles = gp.tile_start[gp.count];
        const int G = std::max(1, ds.pair_clusters);
        // a partial last wave of R tiles (R <= G/2) runs as 2R half tiles, as
        // for one problem
        const int R = tiles % G;
        const bool halves = R > 0 && 2 * R <= G;
        gp.dp_tiles = halves ? tiles - R : tiles;
        gp.tail_split = halves ? 1 : 0;
        const int ctas = 2 * std::min(gp.dp_tiles + (halves ? 2 * R : 0), G);
        const int r = launch_grouped(gp, ctas, s);
        gp.count = 0;
        return r;
    };
    for (int i = 0; st == GEMM_OK && i < count; ++i) {
        const gemm_f16_problem_t& q = problems[i];
        const Prep& pr = prep[i];
        if (q.M == 0 || q.N == 0) continue;
        const __half* biasp = epilogue == GEMM_EPI_NONE ? nullptr : static_cast<const __half*>(q.bias);
        if (q.K == 0) {
            Plan bl;
            bl.path = 1;
            bl.ctas = static_cast<int>(std::min<int64_t>((q.M * q.N + 255) / 256, int64_t(ds.num_sms) * 8));
            st = enqueue_bias_only(bl, biasp, q.C, q.ldc, q.M, q.N, epilogue, s);
            continue;
        }
        const int64_t tiles = ((q.M + 255) / 256) * ((q.N + 255) / 256);   // < 2^28 by check_args
        if (int64_t(gp.tile_start[gp.count]) + tiles >= (int64_t(1) << 31)) {
            st = flush();   // keep every tile index of a launch an int
            if (st != GEMM_OK) break;
        }
        const void* a_src = q.A;
        const void* b_src = q.B;
        if (pr.pl.pack_a) {
            uint16_t* dst = reinterpret_cast<uint16_t*>(scratch + pr.off);
            st = launch_repack(dst, q.A, pr.op.a_rows(q.M, q.K), pr.op.a_cols(q.M, q.K), q.lda, pr.pl.lda_packed, s);
            a_src = dst;
        }
        if (st == GEMM_OK && pr.pl.pack_b) {
            uint16_t* dst = reinterpret_cast<uint16_t*>(scratch + pr.off + pr.pl.a_scratch);
            st = launch_repack(dst, q.B, pr.op.b_rows(q.N, q.K), pr.op.b_cols(q.N, q.K), q.ldb, pr.pl.ldb_packed, s);
            b_src = dst;
        }
        if (st != GEMM_OK) break;
        const int j = gp.count;
        const bool a3 = mn3d_ok(pr.op.ta, q.M, pr.pl.lda_packed);
        const bool b3 = mn3d_ok(!pr.op.tb, q.N, pr.pl.ldb_packed);
        st = a3 ? encode_mn3d(&gp.tmA[j], a_src, q.M, q.K, pr.pl.lda_packed)
             : pr.op.ta ? encode_2d(&gp.tmA[j], a_src, q.M, q.K, pr.pl.lda_packed, 64, kBK)
                        : encode_2d(&gp.tmA[j], a_src, q.K, q.M, pr.pl.lda_packed, kBK, kBM);
        if (st == GEMM_OK)
            st = b3 ? encode_mn3d(&gp.tmB[j], b_src, q.N, q.K, pr.pl.ldb_packed)
                 : pr.op.tb ? encode_2d(&gp.tmB[j], b_src, q.K, q.N, pr.pl.ldb_packed, kBK, 64)
                            : encode_2d(&gp.tmB[j], b_src, q.N, q.K, pr.pl.ldb_packed, 64, kBK);
        if (st != GEMM_OK) break;
        gp.prob[j] = kernel_params(pr.op, biasp, q.M, q.N, q.K, epilogue);
        gp.prob[j].mn3d_a = a3 ? 1 : 0;
        gp.prob[j].mn3d_b = b3 ? 1 : 0;
        gp.tile_start[j + 1] = gp.tile_start[j] + static_cast<int>(tiles);
        gp.count = j + 1;
        if (gp.count == kMaxGroupProblems) st = flush();
    }
    if (st == GEMM_OK) st = flush();
    if (scratch != nullptr) {
        e = cudaFreeAsync(scratch, s);   // stream-ordered: after every launch above has read it
        if (e != cudaSuccess && st == GEMM_OK) st = cuda_fail(e);
    }
    delete[] prep;
    return st;
}

int gemm_f16_debug_status(void* cuda_stream, uint32_t* detail) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int word = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&word, g_status, sizeof(word));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e);
    if (detail) *detail = word;
    return word != 0 ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

int gemm_f16_release_workspace(void) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_dev[dev].pool != nullptr) {
        e = cudaMemPoolTrimTo(g_dev[dev].pool, 0);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return GEMM_OK;
}

int gemm_f16_debug_inject(int fault, uint32_t wait_us) {
    if (fault < GEMM_F16_FAULT_NONE || fault > GEMM_F16_FAULT_ENCODE) return GEMM_ERR_INVALID_ARG;
    if (fault == GEMM_F16_FAULT_SKIP_LOADS && wait_us == 0) return GEMM_ERR_INVALID_ARG;
    g_fault_wait_ns.store(static_cast<uint64_t>(wait_us) * 1000ull, std::memory_order_relaxed);
    g_fault.store(fault);
    return GEMM_OK;
}

int gemm_f16_selftest_timeout(void* cuda_stream, uint32_t timeout_us) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    int st = init_device(dev);
    if (st != GEMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    gemm_f16_selftest_timeout_kernel<<<1, 32, 0, s>>>(static_cast<uint64_t>(timeout_us) * 1000ull);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return gemm_f16_debug_status(cuda_stream, nullptr);
}

}  // extern "C"
