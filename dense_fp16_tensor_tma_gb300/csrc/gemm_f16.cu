// C-ABI boundary of the fused fp16 GEMM (declared in include/gemm_f16.h):
// argument checks, device check, execution plan, TMA tensor-map encoding,
// stream-ordered repack scratch, and kernel launch on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "gemm_f16.h"
#include "gemm_kernels.cuh"

namespace {

using namespace gemm_f16_dev;

thread_local int t_last_cuda_error = 0;

// Tile configurations (tile_n, stages): 128 x 256 is the throughput shape;
// narrower tiles give small problems more CTAs.
constexpr int kStages256 = 4;   // 4 x 48 KiB ring
constexpr int kStages128 = 6;   // 6 x 32 KiB
constexpr int kStages64 = 8;    // 8 x 24 KiB

constexpr int kMaxDevices = 64;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
    bool ready = false;
    int status = GEMM_OK;      // result of the one-time checks
    int num_sms = 0;
    cudaMemPool_t pool = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
uint64_t g_timeout_ns = 2000000000ull;   // 2 s per bounded wait

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return GEMM_ERR_CUDA;
}

struct Plan {
    int path = 0;          // 0 none, 1 bias-only, 2 tiled tensor-core kernel
    int tile_n = 0, stages = 0, ctas = 0;
    bool pack_a = false, pack_b = false, vec_store = false;
    int64_t lda_packed = 0, ldb_packed = 0;
};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

int check_args(const void* A, const void* B, const void* bias, const void* C, int64_t M, int64_t N, int64_t K,
               int epilogue) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return GEMM_ERR_INVALID_ARG;
    if (epilogue < GEMM_EPI_NONE || epilogue > GEMM_EPI_BIAS_GELU_ERF) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (C == nullptr) return GEMM_ERR_INVALID_ARG;
    if (K > 0 && (A == nullptr || B == nullptr)) return GEMM_ERR_INVALID_ARG;
    if (epilogue != GEMM_EPI_NONE && bias == nullptr) return GEMM_ERR_INVALID_ARG;
    if (!aligned(C, 2) || (K > 0 && (!aligned(A, 2) || !aligned(B, 2))) ||
        (epilogue != GEMM_EPI_NONE && !aligned(bias, 2)))
        return GEMM_ERR_MISALIGNED;
    return GEMM_OK;
}

Plan make_plan(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K, int num_sms) {
    Plan pl;
    if (M == 0 || N == 0) return pl;
    if (K == 0) {
        pl.path = 1;
        pl.ctas = static_cast<int>(std::min<int64_t>((M * N + 255) / 256, int64_t(num_sms) * 8));
        return pl;
    }
    pl.path = 2;
    pl.pack_a = !(aligned(A, 16) && K % 8 == 0);
    pl.pack_b = !(aligned(B, 16) && N % 8 == 0);
    pl.lda_packed = pl.pack_a ? round_up(K, 8) : K;
    pl.ldb_packed = pl.pack_b ? round_up(N, 8) : N;
    pl.vec_store = aligned(C, 16) && N % 8 == 0;
    const int64_t tiles_m = (M + kBM - 1) / kBM;
    // Widest tile that still gives every SM work; otherwise the narrowest.
    pl.tile_n = 64;
    for (int bn : {256, 128}) {
        if (tiles_m * ((N + bn - 1) / bn) >= num_sms) { pl.tile_n = bn; break; }
    }
    pl.stages = pl.tile_n == 256 ? kStages256 : (pl.tile_n == 128 ? kStages128 : kStages64);
    const int64_t tiles = tiles_m * ((N + pl.tile_n - 1) / pl.tile_n);
    pl.ctas = static_cast<int>(std::min<int64_t>(tiles, num_sms));
    return pl;
}

int init_device(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[dev];
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
    e = cudaFuncSetAttribute(gemm_f16_tc_kernel<256, kStages256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SmemPlan<256, kStages256>::kDynamicBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_f16_tc_kernel<128, kStages128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SmemPlan<128, kStages128>::kDynamicBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_f16_tc_kernel<64, kStages64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SmemPlan<64, kStages64>::kDynamicBytes);
    if (e != cudaSuccess) return cuda_fail(e);
    // A library-owned pool keeps repack scratch cached between calls without
    // changing the device's default pool.
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    e = cudaMemPoolCreate(&st.pool, &props);
    if (e != cudaSuccess) return cuda_fail(e);
    uint64_t keep = ~0ull;
    cudaMemPoolSetAttribute(st.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (const char* env = std::getenv("GEMM_F16_TIMEOUT_MS")) {
        const long ms = std::strtol(env, nullptr, 10);
        if (ms > 0) g_timeout_ns = static_cast<uint64_t>(ms) * 1000000ull;
    }
    st.num_sms = sms;
    st.ready = true;
    st.status = GEMM_OK;
    return GEMM_OK;
}

// 2-D fp16 tensor map: `inner` contiguous elements per row, `outer` rows,
// row pitch `ld` elements, box `box_inner` x `box_outer`, 128-byte swizzle,
// zero fill outside the tensor.
int encode_2d(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int64_t ld, int box_inner,
              int box_outer) {
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
    return GEMM_OK;
}

int launch_repack(uint16_t* dst, const void* src, int64_t rows, int64_t cols, int64_t ld_src, int64_t ld_dst,
                  cudaStream_t s) {
    dim3 block(256);
    dim3 grid(static_cast<unsigned>(std::min<int64_t>((cols + 255) / 256, 64)),
              static_cast<unsigned>(std::min<int64_t>(rows, 65535)));
    gemm_f16_repack_kernel<<<grid, block, 0, s>>>(dst, static_cast<const uint16_t*>(src), rows, cols, ld_src,
                                                  ld_dst);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
}

template <int BN, int STAGES>
int launch_tc(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& prm, int ctas, cudaStream_t s) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SmemPlan<BN, STAGES>::kDynamicBytes;
    cfg.stream = s;
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_f16_tc_kernel<BN, STAGES>, ta, tb, prm);
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
}

// ---------------------------------------------------------------- no-alloc variant
// Fixed repack buffer for gemm_f16_noalloc, part of the module image: every
// device that loads this library holds it until the process exits.  In host
// code `g_noalloc_scratch` names a host-side stand-in, never the device
// buffer; its device address comes from cudaGetSymbolAddress in
// init_device_noalloc and is what the kernels and tensor maps receive.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocState {
    bool ready = false;
    int status = GEMM_OK;
    int num_sms = 0;
    uint8_t* scratch = nullptr;   // device address of g_noalloc_scratch on this device
};
NoAllocState g_noalloc[kMaxDevices];

// Per-device set-up of the no-alloc path: device check, tensor-map encoder,
// kernel attributes and the scratch address.  Allocates nothing.
int init_device_noalloc(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    NoAllocState& st = g_noalloc[dev];
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
    e = cudaFuncSetAttribute(gemm_f16_tc_kernel<256, kStages256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SmemPlan<256, kStages256>::kDynamicBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_f16_tc_kernel<128, kStages128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SmemPlan<128, kStages128>::kDynamicBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_f16_tc_kernel<64, kStages64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SmemPlan<64, kStages64>::kDynamicBytes);
    if (e != cudaSuccess) return cuda_fail(e);
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    if (const char* env = std::getenv("GEMM_F16_TIMEOUT_MS")) {
        const long ms = std::strtol(env, nullptr, 10);
        if (ms > 0) g_timeout_ns = static_cast<uint64_t>(ms) * 1000000ull;
    }
    st.scratch = static_cast<uint8_t*>(ptr);
    st.num_sms = sms;
    st.ready = true;
    st.status = GEMM_OK;
    return GEMM_OK;
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

int gemm_f16_plan(const void* A, const void* B, const void* bias, const void* C, int64_t M, int64_t N, int64_t K,
                  int epilogue, int num_sms, int64_t plan[8]) {
    if (plan == nullptr || num_sms <= 0) return GEMM_ERR_INVALID_ARG;
    const int st = check_args(A, B, bias, C, M, N, K, epilogue);
    if (st != GEMM_OK) return st;
    const Plan pl = make_plan(A, B, C, M, N, K, num_sms);
    plan[0] = pl.path;
    plan[1] = pl.path == 2 ? kBM : 0;
    plan[2] = pl.tile_n;
    plan[3] = pl.stages;
    plan[4] = pl.ctas;
    plan[5] = pl.pack_a;
    plan[6] = pl.pack_b;
    plan[7] = pl.vec_store;
    return GEMM_OK;
}

int gemm_f16(const void* A, const void* B, const void* bias, void* C, int64_t M, int64_t N, int64_t K, int epilogue,
             void* cuda_stream) {
    int st = check_args(A, B, bias, C, M, N, K, epilogue);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    st = init_device(dev);
    if (st != GEMM_OK) return st;
    DeviceState& ds = g_dev[dev];
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const Plan pl = make_plan(A, B, C, M, N, K, ds.num_sms);
    const __half* biasp = epilogue == GEMM_EPI_NONE ? nullptr : static_cast<const __half*>(bias);

    if (pl.path == 1) {
        gemm_f16_bias_only_kernel<<<pl.ctas, 256, 0, s>>>(static_cast<__half*>(C), biasp, M, N, N, epilogue);
        e = cudaGetLastError();
        return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
    }

    // Repack operands the tensor map cannot describe (unaligned base or row pitch).
    const void* a_src = A;
    const void* b_src = B;
    void* scratch = nullptr;
    size_t a_bytes = pl.pack_a ? static_cast<size_t>(M * pl.lda_packed * 2) : 0;
    size_t b_bytes = pl.pack_b ? static_cast<size_t>(K * pl.ldb_packed * 2) : 0;
    a_bytes = (a_bytes + 255) & ~size_t(255);
    if (a_bytes + b_bytes > 0) {
        e = cudaMallocFromPoolAsync(&scratch, a_bytes + b_bytes, ds.pool, s);
        if (e != cudaSuccess) {
            t_last_cuda_error = static_cast<int>(e);
            cudaGetLastError();
            return GEMM_ERR_NO_MEMORY;
        }
        if (pl.pack_a) {
            st = launch_repack(static_cast<uint16_t*>(scratch), A, M, K, K, pl.lda_packed, s);
            a_src = scratch;
        }
        if (st == GEMM_OK && pl.pack_b) {
            uint16_t* bdst = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(scratch) + a_bytes);
            st = launch_repack(bdst, B, K, N, N, pl.ldb_packed, s);
            b_src = bdst;
        }
    }

    CUtensorMap ta, tb;
    if (st == GEMM_OK) st = encode_2d(&ta, a_src, K, M, pl.lda_packed, kBK, kBM);
    if (st == GEMM_OK) st = encode_2d(&tb, b_src, N, K, pl.ldb_packed, 64, kBK);
    if (st == GEMM_OK) {
        GemmParams prm;
        prm.C = static_cast<__half*>(C);
        prm.bias = biasp;
        prm.M = static_cast<int>(M);
        prm.N = static_cast<int>(N);
        prm.K = static_cast<int>(K);
        prm.ldc = static_cast<int>(N);
        prm.epi = epilogue;
        prm.vec_store = pl.vec_store ? 1 : 0;
        prm.group_m = 8;
        prm.timeout_ns = g_timeout_ns;
        if (pl.tile_n == 256)
            st = launch_tc<256, kStages256>(ta, tb, prm, pl.ctas, s);
        else if (pl.tile_n == 128)
            st = launch_tc<128, kStages128>(ta, tb, prm, pl.ctas, s);
        else
            st = launch_tc<64, kStages64>(ta, tb, prm, pl.ctas, s);
    }
    if (scratch != nullptr) {
        e = cudaFreeAsync(scratch, s);   // stream-ordered: freed after the GEMM reads it
        if (e != cudaSuccess && st == GEMM_OK) st = cuda_fail(e);
    }
    return st;
}

int gemm_f16_noalloc(const void* A, const void* B, const void* bias, void* C, int64_t M, int64_t N, int64_t K,
                     int epilogue, void* cuda_stream) {
    int st = check_args(A, B, bias, C, M, N, K, epilogue);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    st = init_device_noalloc(dev);
    if (st != GEMM_OK) return st;
    const NoAllocState& ns = g_noalloc[dev];
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const Plan pl = make_plan(A, B, C, M, N, K, ns.num_sms);
    const __half* biasp = epilogue == GEMM_EPI_NONE ? nullptr : static_cast<const __half*>(bias);

    if (pl.path == 1) {
        gemm_f16_bias_only_kernel<<<pl.ctas, 256, 0, s>>>(static_cast<__half*>(C), biasp, M, N, N, epilogue);
        e = cudaGetLastError();
        return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
    }

    // Same repack layout as gemm_f16 (A first, 256-byte aligned, then B), but
    // inside the fixed buffer; nothing in it has to start at zero because the
    // tensor maps stop at the true extents.
    size_t a_bytes = pl.pack_a ? static_cast<size_t>(M * pl.lda_packed * 2) : 0;
    const size_t b_bytes = pl.pack_b ? static_cast<size_t>(K * pl.ldb_packed * 2) : 0;
    a_bytes = (a_bytes + 255) & ~size_t(255);
    if (a_bytes + b_bytes > kNoAllocScratchBytes) return GEMM_ERR_SCRATCH_LIMIT;
    const void* a_src = A;
    const void* b_src = B;
    if (pl.pack_a) {
        st = launch_repack(reinterpret_cast<uint16_t*>(ns.scratch), A, M, K, K, pl.lda_packed, s);
        a_src = ns.scratch;
    }
    if (st == GEMM_OK && pl.pack_b) {
        uint16_t* bdst = reinterpret_cast<uint16_t*>(ns.scratch + a_bytes);
        st = launch_repack(bdst, B, K, N, N, pl.ldb_packed, s);
        b_src = bdst;
    }
    CUtensorMap ta, tb;
    if (st == GEMM_OK) st = encode_2d(&ta, a_src, K, M, pl.lda_packed, kBK, kBM);
    if (st == GEMM_OK) st = encode_2d(&tb, b_src, N, K, pl.ldb_packed, 64, kBK);
    if (st != GEMM_OK) return st;
    GemmParams prm;
    prm.C = static_cast<__half*>(C);
    prm.bias = biasp;
    prm.M = static_cast<int>(M);
    prm.N = static_cast<int>(N);
    prm.K = static_cast<int>(K);
    prm.ldc = static_cast<int>(N);
    prm.epi = epilogue;
    prm.vec_store = pl.vec_store ? 1 : 0;
    prm.group_m = 8;
    prm.timeout_ns = g_timeout_ns;
    if (pl.tile_n == 256) return launch_tc<256, kStages256>(ta, tb, prm, pl.ctas, s);
    if (pl.tile_n == 128) return launch_tc<128, kStages128>(ta, tb, prm, pl.ctas, s);
    return launch_tc<64, kStages64>(ta, tb, prm, pl.ctas, s);
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
