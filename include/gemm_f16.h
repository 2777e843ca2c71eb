/*
 * gemm_f16.h -- C ABI of the fused fp16 tensor-core GEMM for GB300 (sm_103a).
 *
 *   C[M,N] = epilogue(A[M,K] . B[K,N] + bias[N])
 *
 * The operation: "writing-tilelang-kernels", Kernel Anatomy and GEMM (Minimal)
 * (A an (M,K) fp16 tensor, B a (K,N) fp16 tensor, C an (M,N) fp16 tensor,
 * float accumulator, one write-back of C); the same page's Pre-flight
 * Checklist ("GEMM + fusion": an activation epilogue after the GEMM); and
 * "TileLang: Write, Autotune, and Ship Fused Tensor-Core Kernels from
 * Python", Why tile-level control matters (bias add and GELU applied while
 * the accumulator is on chip, C written once, no M x N intermediate in HBM).
 *
 * Numerics: A and B are fp16; products are accumulated in fp32 in tensor
 * memory; bias is added and the activation applied in fp32; C is rounded
 * once to fp16 (round to nearest even).  GELU is the exact form
 * 0.5 x (1 + erf(x / sqrt 2)); its tanh approximation and the sigmoid (the
 * checklist's other "GEMM + fusion" activation) are also offered.
 *
 * Layout: gemm_f16 takes dense row-major matrices (lda = K, ldb = N,
 * ldc = N); gemm_f16_ex takes any row pitches and either operand stored
 * transposed.  Element type IEEE binary16 passed as raw pointers.  bias is a
 * length-N vector broadcast over the rows of C.
 *
 * Pointers: A, B, bias and C are DEVICE pointers on the current CUDA device.
 * The caller owns them; the library never frees or retains them.  C must not
 * overlap A, B or bias.  Every pointer must be at least 2-byte aligned.
 * Operands whose base is not 16-byte aligned, or whose row pitch in bytes is
 * not a multiple of 16 (e.g. K % 8 != 0 for a dense A, N % 8 != 0 for a
 * dense B), are repacked, in their own layout, into a library-owned,
 * stream-ordered scratch buffer before the GEMM.
 *
 * Streams: every call is asynchronous on `cuda_stream` (a cudaStream_t, or
 * NULL for the legacy default stream) and returns once the work is enqueued.
 * Errors detected while the kernel runs appear at the caller's next
 * synchronisation; gemm_f16_debug_status reports bounded-wait timeouts.
 */
#ifndef GEMM_F16_H
#define GEMM_F16_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Epilogue applied to x = acc + bias[n] (bias ignored for NONE). */
typedef enum {
    GEMM_EPI_NONE = 0,          /* C = acc                              */
    GEMM_EPI_BIAS = 1,          /* C = acc + bias                       */
    GEMM_EPI_BIAS_RELU = 2,     /* C = max(acc + bias, 0)               */
    GEMM_EPI_BIAS_GELU_ERF = 3, /* C = 0.5 x (1 + erf(x/sqrt2)), x = acc + bias */
    GEMM_EPI_BIAS_SIGMOID = 4,  /* C = 1 / (1 + exp(-x))                 */
    GEMM_EPI_BIAS_GELU_TANH = 5 /* C = 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */
} gemm_epilogue_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,        /* negative size, bad epilogue, null pointer, overflow */
    GEMM_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not compute capability 10.3 */
    GEMM_ERR_MISALIGNED = 3,         /* a pointer is not 2-byte aligned */
    GEMM_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed; see gemm_f16_last_cuda_error */
    GEMM_ERR_TIMEOUT = 5,            /* a kernel's bounded wait ran out (reported by gemm_f16_debug_status) */
    GEMM_ERR_NO_MEMORY = 6,          /* the repack scratch buffer could not be allocated */
    GEMM_ERR_SCRATCH_LIMIT = 7       /* gemm_f16_noalloc: repack needs more than its fixed buffer */
} gemm_status_t;

/*
 * gemm_f16 -- C = epilogue(A.B + bias) on the current device.
 *
 *   A        device pointer, fp16 [M, K] row-major
 *   B        device pointer, fp16 [K, N] row-major
 *   bias     device pointer, fp16 [N]; required for epilogue >= GEMM_EPI_BIAS,
 *            ignored (may be NULL) for GEMM_EPI_NONE
 *   C        device pointer, fp16 [M, N] row-major, written (never read)
 *   M, N, K  sizes, each >= 0 and < 2^31; M*N, M*K, K*N < 2^62
 *   epilogue a gemm_epilogue_t value
 *   cuda_stream  cudaStream_t to enqueue on (NULL = legacy default stream)
 *
 * Returns GEMM_OK once enqueued.  M == 0 or N == 0 is a no-op; K == 0 writes
 * C = epilogue(bias) (zeros for NONE).  Argument errors return before any
 * CUDA call and enqueue nothing.
 */
int gemm_f16(const void* A, const void* B, const void* bias, void* C,
             int64_t M, int64_t N, int64_t K, int epilogue, void* cuda_stream);

/* Operand layout flags of gemm_f16_ex (bitwise or). */
typedef enum {
    GEMM_F16_TRANS_A = 1,     /* A is stored transposed: K x M, M contiguous */
    GEMM_F16_TRANS_B = 2,     /* B is stored transposed: N x K, K contiguous */
    GEMM_F16_PLAN_NOALLOC = 4 /* gemm_f16_plan_ex only: the plan of gemm_f16_noalloc */
} gemm_f16_flags_t;

/*
 * gemm_f16_ex -- gemm_f16 with row pitches and transposed operands: the
 * transpose_A / transpose_B options of the tile GEMM primitive in
 * "writing-tilelang-kernels", Key API Patterns (T.gemm), applied to the
 * operands in global memory.  Computes the same C[M,N] = epilogue(A.B + bias)
 * where, with pitches in elements,
 *
 *   A[i,k] = A_ptr[i*lda + k]   (lda >= K)   or, with GEMM_F16_TRANS_A,
 *            A_ptr[k*lda + i]   (lda >= M)
 *   B[k,j] = B_ptr[k*ldb + j]   (ldb >= N)   or, with GEMM_F16_TRANS_B,
 *            B_ptr[j*ldb + k]   (ldb >= K)   (a Linear layer's weight W[N,K]: C = A.W^T)
 *   C[i,j] = C_ptr[i*ldc + j]   (ldc >= N; elements between rows untouched)
 *
 * The tensor cores read both layouts directly (K-major or MN-major shared-
 * memory operands); only a base not 16-byte aligned or a pitch not a multiple
 * of 8 elements costs a repack, as in gemm_f16.  Pitches are < 2^31; the
 * pitch checks apply only to operands that are read (K > 0, M, N > 0).
 * Unknown flag bits, a pitch below its minimum, or the gemm_f16 argument
 * errors return GEMM_ERR_INVALID_ARG (or GEMM_ERR_MISALIGNED) before any
 * CUDA call.  Otherwise as gemm_f16; gemm_f16(A, B, bias, C, M, N, K, e, s)
 * is gemm_f16_ex(A, K, B, N, bias, C, N, M, N, K, e, 0, s).
 */
int gemm_f16_ex(const void* A, int64_t lda, const void* B, int64_t ldb, const void* bias, void* C,
                int64_t ldc, int64_t M, int64_t N, int64_t K, int epilogue, int flags,
                void* cuda_stream);

/*
 * One problem of a grouped call: the arguments of gemm_f16_ex (pitches in
 * elements; the layout flags are the call's).
 */
typedef struct gemm_f16_problem {
    const void* A;
    int64_t lda;
    const void* B;
    int64_t ldb;
    const void* bias;   /* required unless the epilogue is GEMM_EPI_NONE */
    void* C;
    int64_t ldc;
    int64_t M, N, K;
} gemm_f16_problem_t;

/*
 * gemm_f16_grouped -- many independent GEMMs in one persistent launch (the
 * "grouped GEMM" of the tilelang documentation's advanced examples):
 *
 *   C_g = epilogue(A_g . B_g + bias_g)   for g = 0 .. count-1,
 *
 * each problem with its own sizes, pointers and pitches, all with the same
 * epilogue and operand-layout flags (see gemm_f16_ex).  `problems` is a HOST
 * array, read during the call only.  Every problem is checked first; any
 * argument error returns before anything is enqueued.  Problems with M or N
 * of 0 are skipped; K == 0 problems get C_g = epilogue(bias_g).  The tiles of
 * all problems (256 x 256, CTA pairs) are scheduled together, up to 64
 * problems per launch (more take further launches on the same stream); a
 * partial last wave of at most half the pairs runs as 256 x 128 half tiles.
 * Problems must not write each other's C or read another problem's C.
 * No counterpart beyond the name on the pages; the numerics are gemm_f16's.
 */
int gemm_f16_grouped(const gemm_f16_problem_t* problems, int count, int epilogue, int flags,
                     void* cuda_stream);

/* Static, human-readable name of a status code. */
const char* gemm_f16_status_string(int status);

/* cudaError_t value behind the calling thread's most recent GEMM_ERR_CUDA. */
int gemm_f16_last_cuda_error(void);

/*
 * Synchronises `cuda_stream`, then reads and clears the device-side status
 * word of the current device.  Returns GEMM_ERR_TIMEOUT if any kernel of
 * this library gave up a bounded wait since the last call, GEMM_ERR_CUDA if
 * the synchronisation failed, GEMM_OK otherwise.  `detail` (nullable)
 * receives the raw status word (role and barrier of the first timeout).
 */
int gemm_f16_debug_status(void* cuda_stream, uint32_t* detail);

/* Returns the library's cached repack scratch memory on the current device
 * to the system (the scratch is stream-ordered; call after synchronising). */
int gemm_f16_release_workspace(void);

/*
 * Host-only planning query (no device access): the execution plan that
 * gemm_f16 would choose for these sizes and base addresses on a device with
 * `num_sms` SMs (assuming num_sms/2 co-resident CTA pairs).  plan[0..7]
 * receive: path (0 none, 1 bias-only K==0, 2 tiled tensor-core kernel,
 * 3 swap-AB kernel for M <= 64), tile_m (256 for the CTA-pair kernel),
 * tile_n,
 * pipeline stages, CTAs launched, repack A (0/1), repack B (0/1), vector
 * stores of C (0/1), split-K parts per tile (swap-AB: CTAs sharing a tile's
 * K through scratch; 128-row tiles: CTAs of a cluster), scratch bytes, and for the CTA
 * pair the number of whole tiles before the half-tile units (-1: no split).
 * Returns a status
 * code like gemm_f16 (argument errors only).  Diagnostic; it has no
 * counterpart on the pages.
 */
int gemm_f16_plan(const void* A, const void* B, const void* bias, const void* C,
                  int64_t M, int64_t N, int64_t K, int epilogue, int num_sms,
                  int64_t plan[11]);

/* gemm_f16_plan for the arguments of gemm_f16_ex (same plan[] entries).
 * With GEMM_F16_PLAN_NOALLOC in `flags`: the plan gemm_f16_noalloc takes
 * (all of its scratch inside the fixed buffer, split-K dropped when the
 * partial sums do not fit beside the repacks), or GEMM_ERR_SCRATCH_LIMIT
 * when the repacks alone exceed the buffer. */
int gemm_f16_plan_ex(const void* A, int64_t lda, const void* B, int64_t ldb, const void* bias,
                     const void* C, int64_t ldc, int64_t M, int64_t N, int64_t K, int epilogue,
                     int flags, int num_sms, int64_t plan[11]);

/*
 * Diagnostic (no counterpart on the pages): pins the kernel configuration
 * that every later call in this process uses, for tests and tile sweeps.
 *   0 automatic (the default), 1 CTA pair with a 256 x 256 tile,
 *   2 single CTA 128 x 256, 3 single CTA 128 x 128, 4 single CTA 128 x 64,
 *   5 swap-AB (C^T = B^T A^T; tiles of 128 columns x 16, 32 or 64 rows),
 *   6 CTA pair with whole tiles only (no half-tile units for a partial last wave).
 * Returns the previous setting, or -1 (nothing changed) for an unknown
 * value.  Process-wide; set it while no other host thread is calling.
 */
int gemm_f16_force_config(int config);

/*
 * Diagnostic (no counterpart on the pages): pins whether later calls that
 * run 128-row tiles split K across a cluster of CTAs (each CTA multiplies a
 * share of the tile's K blocks; the fp32 partial tiles are summed through
 * distributed shared memory before the epilogue).  0 automatic (the
 * default: split where it lowers the operand bytes per SM), 1 never, 2 or 4
 * that many CTAs per tile wherever the problem allows it (one tile per
 * cluster, at least 4 K blocks per CTA).  Returns the previous setting, or -1
 * (nothing changed) for another value.  Process-wide.
 */
int gemm_f16_force_ksplit(int splits);

/*
 * Programmatic dependent launch (on by default; the environment variable
 * GEMM_F16_PDL=0 turns it off at start-up).  Every kernel of this library is
 * launched with programmatic stream serialization: it may begin while the
 * previous kernel in the stream is still finishing, runs its set-up (barrier
 * initialisation, tensor-memory allocation, descriptor prefetch) meanwhile,
 * and waits for that kernel's completion and memory before its first access
 * to global memory.  Results are the same either way; back-to-back small
 * calls (and their CUDA graphs) lose part of the launch latency.  No
 * counterpart on the pages.  Returns the previous setting (0/1).
 * Process-wide; set it while no other host thread is calling.
 */
int gemm_f16_set_pdl(int enable);

/* Faults gemm_f16_debug_inject can arm. */
typedef enum {
    GEMM_F16_FAULT_NONE = 0,
    GEMM_F16_FAULT_SKIP_LOADS = 1,  /* next single-CTA tensor-core launch skips one stage's loads */
    GEMM_F16_FAULT_ENCODE = 2       /* next TMA tensor-map encoding fails */
} gemm_f16_fault_t;

/*
 * Test hook for the library's error paths (no counterpart on the pages; not
 * for production use).  Arms one fault, process-wide, consumed by the first
 * call that reaches it; GEMM_F16_FAULT_NONE disarms.
 *
 *   GEMM_F16_FAULT_SKIP_LOADS: the next launch of a single-CTA tensor-core
 *     kernel (128-row tiles or swap-AB; CTA-pair launches neither use nor
 *     consume it) never issues the loads of the second K block of each CTA's
 *     first tile, and every bounded wait of that launch gives up after
 *     `wait_us` microseconds (> 0).  The MMA thread's wait for that stage
 *     runs out; the kernel records the timeout in the status word, every role
 *     leaves, in-flight loads and MMAs are drained and tensor memory is freed.
 *     Nothing is ever in flight for the skipped stage.  C is left partly
 *     written; gemm_f16_debug_status then reports GEMM_ERR_TIMEOUT, and the
 *     context stays usable.  The problem must have at least two K blocks
 *     (K > 64), or nothing is skipped.
 *   GEMM_F16_FAULT_ENCODE: the next tensor-map encoding fails as the driver's
 *     encoder would for an invalid map: that call returns GEMM_ERR_CUDA
 *     (gemm_f16_last_cuda_error = CUDA_ERROR_INVALID_VALUE).  gemm_f16,
 *     gemm_f16_ex and gemm_f16_noalloc encode their maps before enqueueing
 *     any work, so such a call enqueues no kernel.
 *
 * Returns GEMM_OK, or GEMM_ERR_INVALID_ARG for an unknown fault or a zero
 * wait with GEMM_F16_FAULT_SKIP_LOADS.
 */
int gemm_f16_debug_inject(int fault, uint32_t wait_us);

/*
 * Diagnostic for the bounded-wait machinery (no counterpart on the pages):
 * launches one CTA that waits on an mbarrier nothing ever arrives on, with a
 * limit of `timeout_us` microseconds, and returns what gemm_f16_debug_status
 * then reports (GEMM_ERR_TIMEOUT when the limit worked).  The context stays
 * usable afterwards.
 */
int gemm_f16_selftest_timeout(void* cuda_stream, uint32_t timeout_us);

/*
 * gemm_f16_noalloc -- the same operation as gemm_f16, for callers that must
 * not allocate device memory.  The tutorial pages have no counterpart; this entry
 * point exists for the library's users.
 *
 * Who needs it: code that runs inside a host framework which owns the
 * device memory (its caching allocator has reserved nearly all of it, so a
 * plugin's own cudaMalloc fails or fragments that pool), latency-critical
 * serving loops where cudaMalloc/cudaFree would synchronise the device and
 * stall every other stream, and deployments whose rules forbid dynamic
 * allocation after start-up.
 *
 * Arguments, layout, ownership and asynchrony are those of gemm_f16; the
 * caller still passes A, B, bias and C.  The only difference: when an operand
 * must be repacked (base not 16-byte aligned, or K % 8 != 0 for A,
 * N % 8 != 0 for B), the repacked copy goes into a fixed 32 MiB buffer that
 * is part of the library's device image (a static __device__ array, so every
 * GPU that loads the library holds it until the process exits) instead of
 * memory obtained from the allocator.  This function calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 *   - Sizes: the repack needs 2*M*round8(K) bytes for A plus 2*K*round8(N)
 *     bytes for B (each rounded up to 256); a problem needing more than
 *     32 MiB returns GEMM_ERR_SCRATCH_LIMIT and enqueues nothing.  Problems
 *     that need no repack have no size limit.  The split-K partial sums of
 *     short-A problems use the same buffer when they fit, and are skipped
 *     (the problem runs unsplit) when they do not.
 *   - Set-up: the first call on each device (with that device current) looks
 *     up the buffer's device address and sets kernel attributes; make that
 *     first call before any stream capture.  The buffer is reserved when the
 *     library's device code is loaded onto the device; with CUDA's lazy
 *     module loading (the default) that happens during this set-up, so on a
 *     device whose memory another allocator has already claimed the first
 *     call can fail with GEMM_ERR_CUDA.  A call with M == 0 or N == 0 (valid
 *     arguments, nothing to compute) runs the set-up and enqueues nothing:
 *     make one at start-up to take the buffer before the device fills up.
 *   - Sharing: every call on a device uses the same buffer, which keeps the
 *     previous call's contents (nothing in it needs to start at zero).  Calls
 *     whose GPU work overlaps (e.g. on two streams without ordering between
 *     them) race on the buffer; order them on one stream or with events.
 */
int gemm_f16_noalloc(const void* A, const void* B, const void* bias, void* C,
                     int64_t M, int64_t N, int64_t K, int epilogue, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F16_H */
