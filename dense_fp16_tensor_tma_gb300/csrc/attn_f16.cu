// C-ABI boundary of the attention forward (declared in include/attn_f16.h):
// argument checks, device check, 3-D TMA tensor maps over (D, S, B*H), and
// and the launch of the attention kernel the problem's shape selects on the
// caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "attn_f16.h"
#include "attn3_kernels.cuh"
#include "attn4_kernels.cuh"

#ifndef ATTN_PINGPONG
#define ATTN_PINGPONG 1   // two query tiles per CTA where the problem allows it
#endif
#ifndef ATTN_CAUSAL_MIN_TILES
#define ATTN_CAUSAL_MIN_TILES 8   // causal heads of fewer query tiles run one tile per CTA
#endif
#ifndef ATTN_ODD_TILES
#define ATTN_ODD_TILES 1   // non-causal heads of an odd number of query tiles too (their last tile alone)
#endif
#ifndef ATTN_CAUSAL_PAIRS
#define ATTN_CAUSAL_PAIRS 1   // causal problems too
#endif
#ifndef ATTN_SPLIT_P
#define ATTN_SPLIT_P 1   // D = 64: the two-tile kernel with P buffers of its own (attn_f16_fwd3_kernel)
#endif
// Routing costs (see plan_attention): a causal key block of the two-tile kernels
// in percent of the one-tile kernel's, and a tile of the one-tile kernel in
// thousandths of a two-tile unit, at D = 128 and D = 64
#ifndef ATTN_CAUSAL_PCT_D128
#define ATTN_CAUSAL_PCT_D128 89
#endif
#ifndef ATTN_CAUSAL_PCT_D64
#define ATTN_CAUSAL_PCT_D64 73
#endif
#ifndef ATTN_ODD_TILE_MILLI_D128
#define ATTN_ODD_TILE_MILLI_D128 525
#endif
#ifndef ATTN_ODD_TILE_MILLI_D64
#define ATTN_ODD_TILE_MILLI_D64 640
#endif

namespace {

using namespace attn_dev;

thread_local int t_last_cuda_error = 0;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;
struct AttnDevice {
    bool ready = false;
    int status = GEMM_OK;
    int sms = 0;          // streaming multiprocessors: one persistent CTA each
};
std::mutex g_mu;
AttnDevice g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
std::atomic<uint64_t> g_timeout_ns{2000000000ull};   // set once at set-up, read by every caller
std::atomic<bool> g_pdl{true};   // programmatic dependent launch unless GEMM_F16_PDL=0

// Fault injection for the tests of the error paths (attn_f16_debug_inject):
// one-shot and process-wide, like the GEMM library's.
std::atomic<int> g_fault{GEMM_F16_FAULT_NONE};
std::atomic<uint64_t> g_fault_wait_ns{0};

bool take_fault(int kind) {
    if (g_fault.load(std::memory_order_relaxed) != kind) return false;
    int expected = kind;
    return g_fault.compare_exchange_strong(expected, GEMM_F16_FAULT_NONE);
}

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return GEMM_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int init_device(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    AttnDevice& st = g_dev[dev];
    if (st.ready) return st.status;
    int major = 0, minor = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (major != 10 || minor != 3) {
        st.ready = true;
        st.status = GEMM_ERR_UNSUPPORTED_DEVICE;
        return st.status;
    }
    e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return cuda_fail(e != cudaSuccess ? e : cudaErrorSymbolNotFound);
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    e = cudaFuncSetAttribute(attn_f16_fwd4_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Attn4Smem<64>::kDynamicBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_f16_fwd4_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Attn4Smem<128>::kDynamicBytes);
#if ATTN_SPLIT_P
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_f16_fwd3_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Attn3Smem<64>::kDynamicBytes);
#else
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_f16_fwd2_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Attn2Smem<64>::kDynamicBytes);
#endif
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_f16_fwd2_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Attn2Smem<128>::kDynamicBytes);
    if (e != cudaSuccess) return cuda_fail(e);
    if (const char* env = std::getenv("GEMM_F16_TIMEOUT_MS")) {
        const long ms = std::strtol(env, nullptr, 10);
        if (ms > 0) g_timeout_ns.store(static_cast<uint64_t>(ms) * 1000000ull, std::memory_order_relaxed);
    }
    if (const char* env = std::getenv("GEMM_F16_PDL")) g_pdl.store(env[0] != '0', std::memory_order_relaxed);
    st.ready = true;
    st.status = GEMM_OK;
    return GEMM_OK;
}

// (D, S, B*H) fp16 tensor with box 64 x 128 x 1, 128-byte swizzle, zeros
// outside the tensor (rows past S of a head never come from the next head).
int encode_3d(CUtensorMap* m, const void* ptr, int64_t D, int64_t S, int64_t BH) {
    if (take_fault(GEMM_F16_FAULT_ENCODE)) {   // injected: what the encoder returns for an invalid map
        t_last_cuda_error = static_cast<int>(CUDA_ERROR_INVALID_VALUE);
        return GEMM_ERR_CUDA;
    }
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(S * D) * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kQRows), 1};
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

// The kernel and the work units of one call: 1 attn_f16_fwd4_kernel (one query
// tile per CTA), 2 attn_f16_fwd2_kernel (two tiles, P over the scores, D = 128),
// 3 attn_f16_fwd3_kernel (two tiles, P buffers of its own, D = 64).  Host only.
struct AttnPlan {
    int kernel = 1;
    int64_t units = 0, pair_units = 0;
    int pair = 0;        // one-tile kernel: causal pairs of tiles nq - 1 - k and k
    int ctas = 0;
};

AttnPlan plan_attention(int64_t B, int64_t H, int64_t nq, int64_t D, bool causal, int sms) {
    AttnPlan pl;
    // Work units: query tiles, or, causal with at least two tiles per SM, pairs
    // of a head's tiles nq - 1 - k and k (equal cost per unit; with fewer tiles
    // pairing would only halve the parallelism).
    // Non-causal: two tiles per CTA whose softmax and MMAs interleave
    // (attn_f16_fwd2_kernel; at D = 64 attn_f16_fwd3_kernel), a head's tiles
    // paired (2k, 2k + 1) and, with an odd number per head, its last tile run
    // alone.  Causal (same-box A/B against the one-tile kernel, attn_f16_fwd4_kernel,
    // which pairs tiles k and nq - 1 - k, so its units cost half a step each):
    // with a multiple of 4 tiles per head (an even number of pairs, so every
    // step of two pairs costs the same; with an odd number the cheaper one-pair
    // steps fell on the same CTAs: 4x32x1792x128 827 against 935 TFLOP/s), from
    // 8 tiles per head (4x32x1024: 687 against 627 at D = 128, 574 against 414
    // at D = 64), with at least one step per SM, and only where the busiest
    // CTA's steps cost less than its share of the one-tile kernel's units.  A
    // key block of the two-tile kernels takes 0.89 (D = 128) and 0.73 (D = 64)
    // of the one-tile kernel's time, fitted to same-box A/B runs of both
    // kernels forced in turn (D = 128: 4x32x3072 1183 against 1149 TFLOP/s,
    // 2x32x3072 1162 against 1068, 8x16x1536 933 against 844, 4x32x2048 1059
    // against 1055, which the rule leaves to the one-tile kernel; D = 64:
    // 4x32x3072 828 against 671, 4x32x2048 749 against 622, 2x32x1500 473
    // against 454).  Otherwise one tile per CTA.
    // Non-causal with an odd number of tiles per head (at least 3): pairs of a
    // head's tiles and its last tile alone, where the busiest CTA's units cost
    // less than the one-tile kernel's tiles.  Costs in pair units: a one-tile
    // unit of the two-tile kernels 0.6, a tile of the one-tile kernel 0.525 at
    // D = 128 and 0.64 at D = 64, fitted to the same runs (D = 128: 4x16x2100
    // 1225 against 1143, 16x16x1300 1014 against 999, 8x16x1300 988 against
    // 986; D = 64: 8x16x1300 703 against 575, 4x32x300 251 against 214).  The
    // number of pairs taken (all of them, or one of the last three whole rounds
    // over the CTAs) is the one that leaves the busiest CTA the least work.
    const int64_t tiles_all = B * H * nq;
    const int64_t head_pairs = B * H * (nq / 2);
    // the busiest CTA's cost with p pair units first and then s one-tile units,
    // dealt round-robin to min(p + s, sms) CTAs
    auto busiest = [&](int64_t p, int64_t s1) -> double {
        const int64_t G = std::min<int64_t>(p + s1, sms);
        double worst = 0.0;
        for (int64_t c = 0; c < G; ++c) {
            const int64_t pc = p / G + (c < p % G ? 1 : 0);
            const int64_t first = (c - p % G + G) % G;   // the first one-tile unit dealt to CTA c
            const int64_t sc = first < s1 ? (s1 - first + G - 1) / G : 0;
            worst = std::max(worst, static_cast<double>(pc) + 0.6 * static_cast<double>(sc));
        }
        return worst;
    };
    int64_t odd_pairs = head_pairs;
    bool odd_two = false;
    if (!causal && nq % 2 == 1 && nq >= 3 && ATTN_ODD_TILES) {
        double best = busiest(head_pairs, tiles_all - 2 * head_pairs);
        const int64_t rounds = tiles_all / (2 * static_cast<int64_t>(sms));   // whole rounds of pairs that fit
        for (int64_t j = std::max<int64_t>(0, rounds - 2); j <= rounds && j * sms < head_pairs; ++j) {
            const double c = busiest(j * sms, tiles_all - 2 * j * sms);
            if (c < best) {
                best = c;
                odd_pairs = j * sms;
            }
        }
        const int64_t one_tile = (tiles_all + sms - 1) / sms;
        odd_two = best < static_cast<double>(one_tile) *
                             (D == 64 ? ATTN_ODD_TILE_MILLI_D64 : ATTN_ODD_TILE_MILLI_D128) / 1000.0;
    }
    const int64_t causal_steps = B * H * (nq / 4);
    const int64_t steps_busiest = (causal_steps + sms - 1) / sms;
    const int64_t units1_busiest = (2 * causal_steps + sms - 1) / sms;
    const int64_t block_cost_pct = D == 64 ? ATTN_CAUSAL_PCT_D64 : ATTN_CAUSAL_PCT_D128;
    const bool two_tiles = ATTN_PINGPONG &&
                           (causal ? (ATTN_CAUSAL_PAIRS && nq % 4 == 0 && nq >= ATTN_CAUSAL_MIN_TILES &&
                                      causal_steps >= static_cast<int64_t>(sms) &&
                                      2 * steps_busiest * block_cost_pct < 100 * units1_busiest)
                                   : (nq % 2 == 0 || odd_two));
    pl.pair = !two_tiles && causal && B * H * nq >= 2 * static_cast<int64_t>(sms) ? 1 : 0;
    int64_t units = pl.pair ? B * H * ((nq + 1) / 2) : B * H * nq;
    pl.pair_units = 0;
    if (two_tiles && causal) {
        // steps of two pairs of one head (np - 1 - m, then m; np is even here)
        units = causal_steps;
        pl.pair_units = units;
    } else if (two_tiles) {
        // Two tiles per unit; when the tiles left over after k full rounds of
        // pairs (k per CTA) fit one per CTA, they run as one-tile units (k pairs
        // and at most one single per CTA instead of k + 1 pairs on some CTAs);
        // otherwise every pair a head has is a unit (and, with an odd number of
        // tiles per head, each head's last tile runs alone).
        const int64_t tiles = tiles_all;
        const int64_t k = tiles / (2 * static_cast<int64_t>(sms));
        const int64_t rest = tiles - 2 * k * sms;
        const int64_t pairs = nq % 2 == 1 ? odd_pairs : (rest <= sms ? k * sms : head_pairs);
        pl.pair_units = pairs;
        units = pairs + (tiles - 2 * pairs);
    }
    pl.kernel = !two_tiles ? 1 : (D == 64 ? 3 : 2);
    pl.units = units;
    pl.ctas = static_cast<int>(std::min<int64_t>(units, sms));
    return pl;
}

template <int D>
cudaError_t launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const AttnParams& prm, int ctas,
                   bool two_tiles, cudaStream_t s) {
    constexpr bool split_p = D == 64 && ATTN_SPLIT_P;
    constexpr int one_threads = kAttn4Threads;
    constexpr uint32_t one_smem = Attn4Smem<D>::kDynamicBytes;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(!two_tiles ? one_threads : split_p ? kAttn3Threads : kAttn2Threads);
    if constexpr (split_p) cfg.dynamicSmemBytes = two_tiles ? Attn3Smem<D>::kDynamicBytes : one_smem;
    else cfg.dynamicSmemBytes = two_tiles ? Attn2Smem<D>::kDynamicBytes : one_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    std::memset(attr, 0, sizeof(attr));
    if (g_pdl.load(std::memory_order_relaxed)) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if constexpr (split_p) {
        if (two_tiles) return cudaLaunchKernelEx(&cfg, attn_f16_fwd3_kernel<D>, q, k, v, prm);
    } else {
        if (two_tiles) return cudaLaunchKernelEx(&cfg, attn_f16_fwd2_kernel<D>, q, k, v, prm);
    }
    return cudaLaunchKernelEx(&cfg, attn_f16_fwd4_kernel<D>, q, k, v, prm);
}

}  // namespace

extern "C" {

int attn_f16_fwd(const void* Q, const void* K, const void* V, void* O, int64_t B, int64_t H, int64_t S, int64_t D,
                 int causal, float scale, void* cuda_stream) {
    if (B < 0 || H < 0 || S < 0) return GEMM_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return GEMM_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return GEMM_ERR_INVALID_ARG;
    if (S >= (int64_t(1) << 31) || B >= (int64_t(1) << 31) || H >= (int64_t(1) << 31)) return GEMM_ERR_INVALID_ARG;
    if (B * H >= (int64_t(1) << 31)) return GEMM_ERR_INVALID_ARG;
    if (B == 0 || H == 0 || S == 0) return GEMM_OK;
    const int64_t nq = (S + kQRows - 1) / kQRows;
    if (B * H * nq >= (int64_t(1) << 31)) return GEMM_ERR_INVALID_ARG;
    if (!Q || !K || !V || !O) return GEMM_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return GEMM_ERR_MISALIGNED;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    int st = init_device(dev);
    if (st != GEMM_OK) return st;
    CUtensorMap tq, tk, tv;
    st = encode_3d(&tq, Q, D, S, B * H);
    if (st == GEMM_OK) st = encode_3d(&tk, K, D, S, B * H);
    if (st == GEMM_OK) st = encode_3d(&tv, V, D, S, B * H);
    if (st != GEMM_OK) return st;
    AttnParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.O = static_cast<__half*>(O);
    prm.S = static_cast<int>(S);
    prm.BH = static_cast<int>(B * H);
    prm.nq = static_cast<int>(nq);
    prm.causal = causal ? 1 : 0;
    const double sc = scale == 0.0f ? 1.0 / std::sqrt(static_cast<double>(D)) : static_cast<double>(scale);
    prm.scale_log2 = static_cast<float>(sc * 1.4426950408889634);
    prm.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    prm.fault_skip_block = -1;
    if (take_fault(GEMM_F16_FAULT_SKIP_LOADS)) {
        prm.fault_skip_block = 1;
        prm.timeout_ns = g_fault_wait_ns.load(std::memory_order_relaxed);
    }
    const AttnPlan pl = plan_attention(B, H, nq, D, causal != 0, g_dev[dev].sms);
    prm.pair = pl.pair;
    prm.pair_units = static_cast<int>(pl.pair_units);
    prm.units = static_cast<int>(pl.units);
    const int ctas = pl.ctas;
    const bool two_tiles = pl.kernel != 1;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    e = D == 64 ? launch<64>(tq, tk, tv, prm, ctas, two_tiles, s) : launch<128>(tq, tk, tv, prm, ctas, two_tiles, s);
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
}

int attn_f16_plan(int64_t B, int64_t H, int64_t S, int64_t D, int causal, int num_sms, int64_t plan[5]) {
    if (plan == nullptr || num_sms <= 0) return GEMM_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || S < 0) return GEMM_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return GEMM_ERR_INVALID_ARG;
    if (S >= (int64_t(1) << 31) || B >= (int64_t(1) << 31) || H >= (int64_t(1) << 31)) return GEMM_ERR_INVALID_ARG;
    if (B * H >= (int64_t(1) << 31)) return GEMM_ERR_INVALID_ARG;
    for (int i = 0; i < 5; ++i) plan[i] = 0;
    if (B == 0 || H == 0 || S == 0) return GEMM_OK;
    const int64_t nq = (S + kQRows - 1) / kQRows;
    if (B * H * nq >= (int64_t(1) << 31)) return GEMM_ERR_INVALID_ARG;
    const AttnPlan pl = plan_attention(B, H, nq, D, causal != 0, num_sms);
    plan[0] = pl.kernel;
    plan[1] = pl.units;
    plan[2] = pl.pair_units;
    plan[3] = pl.pair;
    plan[4] = pl.ctas;
    return GEMM_OK;
}

int attn_f16_last_cuda_error(void) { return t_last_cuda_error; }

int attn_f16_debug_inject(int fault, uint32_t wait_us) {
    if (fault < GEMM_F16_FAULT_NONE || fault > GEMM_F16_FAULT_ENCODE) return GEMM_ERR_INVALID_ARG;
    if (fault == GEMM_F16_FAULT_SKIP_LOADS && wait_us == 0) return GEMM_ERR_INVALID_ARG;
    g_fault_wait_ns.store(static_cast<uint64_t>(wait_us) * 1000ull, std::memory_order_relaxed);
    g_fault.store(fault);
    return GEMM_OK;
}

int attn_f16_debug_status(void* cuda_stream, uint32_t* detail) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int word = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&word, g_attn_status, sizeof(word));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e);
    if (detail) *detail = word;
    return word != 0 ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

}  // extern "C"
