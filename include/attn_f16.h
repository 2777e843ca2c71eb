/*
 * attn_f16.h -- C ABI of the fused fp16 attention forward for GB300 (sm_103a).
 *
 *   O[b,h] = softmax(scale * Q[b,h] K[b,h]^T) V[b,h]      for every batch b, head h
 *
 * The operation: "writing-tilelang-kernels", Flash Attention Forward (Q, K,
 * V and O as (B, H, S, D) float16 tensors) and the pattern table's Online
 * Softmax / Flash Attention rows; "TileLang: Write, Autotune, and Ship Fused
 * Tensor-Core Kernels from Python", FlashAttention: the FLOP model and what
 * the example measures (softmax computed online, the S x S score matrix never
 * stored; causal and non-causal; FLOP model 4 B H S^2 D, halved when causal;
 * validated against scaled-dot-product attention, whose default scale is
 * 1/sqrt(D) and whose causal mask keeps key j for query i when j <= i).
 *
 * Numerics: Q K^T and P V on the tensor cores with fp32 accumulation in
 * tensor memory; the softmax in fp32 with the row maximum tracked online; P
 * rounded to fp16 before P V (the row sums use those same fp16 values); O
 * divided by the row sum in fp32 and rounded once to fp16.
 *
 * Status codes are those of gemm_f16.h (gemm_status_t).
 */
#ifndef ATTN_F16_H
#define ATTN_F16_H

#include <stdint.h>

#include "gemm_f16.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_f16_fwd -- attention forward on the current device.
 *
 *   Q, K, V  device pointers, fp16 [B, H, S, D] row-major (D contiguous),
 *            16-byte aligned; read only
 *   O        device pointer, fp16 [B, H, S, D] row-major, 16-byte aligned;
 *            written (never read); must not overlap Q, K or V
 *   B, H, S  batch, heads, sequence length (queries = keys), each >= 0;
 *            B * H < 2^31, S < 2^31
 *   D        head dimension: 64 or 128
 *   causal   0: every key; nonzero: key j only for queries i >= j
 *   scale    the softmax scale; 0 selects 1 / sqrt(D)
 *   cuda_stream  cudaStream_t to enqueue on (NULL = legacy default stream)
 *
 * Returns GEMM_OK once enqueued (B, H or S of 0 is a no-op).  Argument errors
 * (GEMM_ERR_INVALID_ARG, or GEMM_ERR_MISALIGNED for a pointer not 16-byte
 * aligned) return before any CUDA call; GEMM_ERR_UNSUPPORTED_DEVICE unless
 * the current device is compute capability 10.3.  Launched with programmatic
 * stream serialization (set-up overlaps the previous kernel in the stream)
 * unless the environment variable GEMM_F16_PDL=0 is set at the first call.
 */
int attn_f16_fwd(const void* Q, const void* K, const void* V, void* O, int64_t B, int64_t H, int64_t S,
                 int64_t D, int causal, float scale, void* cuda_stream);

/*
 * attn_f16_plan -- host only, touches no device (a diagnostic with no
 * counterpart on the pages): the kernel and work split attn_f16_fwd would use
 * for these arguments on a device of `num_sms` SMs.  On GEMM_OK,
 *
 *   plan[0]  kernel: 1 one query tile per CTA (attn_f16_fwd4_kernel);
 *            2 two tiles per CTA, P over the scores (attn_f16_fwd2_kernel,
 *            D = 128); 3 two tiles per CTA, P buffers of its own
 *            (attn_f16_fwd3_kernel, D = 64); 0 for an empty problem
 *   plan[1]  work units (a unit: one tile, a pair of tiles, or, causal on a
 *            two-tile kernel, a step of two pairs of one head)
 *   plan[2]  two-tile kernels: units that hold two tiles (or causal steps)
 *   plan[3]  one-tile kernel: 1 when causal tiles run in pairs nq - 1 - k, k
 *   plan[4]  CTAs launched (persistent: min(units, SMs))
 *
 * `plan` is caller-owned, 5 entries.  GEMM_ERR_INVALID_ARG for a null plan,
 * num_sms <= 0 or the argument errors of attn_f16_fwd (pointers aside).
 */
int attn_f16_plan(int64_t B, int64_t H, int64_t S, int64_t D, int causal, int num_sms, int64_t plan[5]);

/* cudaError_t value behind the calling thread's most recent GEMM_ERR_CUDA from attn_f16_fwd. */
int attn_f16_last_cuda_error(void);

/*
 * Synchronises `cuda_stream`, then reads and clears the attention kernels'
 * device-side status word (like gemm_f16_debug_status for the GEMM kernels):
 * GEMM_ERR_TIMEOUT if a bounded wait gave up since the last call.
 */
int attn_f16_debug_status(void* cuda_stream, uint32_t* detail);

/*
 * Test hook for the attention forward's error paths (no counterpart on the
 * pages; not for production use), like gemm_f16_debug_inject and with the
 * same gemm_f16_fault_t values, armed separately for this entry point:
 *
 *   GEMM_F16_FAULT_SKIP_LOADS: the next attn_f16_fwd launch never loads the
 *     second key block of each CTA's block sequence (S must exceed 128), and
 *     its bounded waits give up after `wait_us` microseconds (> 0): the MMA
 *     thread's wait for that block runs out, every role leaves, the rest is
 *     drained and tensor memory freed; attn_f16_debug_status then reports
 *     GEMM_ERR_TIMEOUT and the context stays usable.  O is left partly
 *     written.
 *   GEMM_F16_FAULT_ENCODE: the next tensor-map encoding fails: that
 *     attn_f16_fwd call returns GEMM_ERR_CUDA and enqueues nothing.
 *
 * Returns GEMM_OK, or GEMM_ERR_INVALID_ARG for an unknown fault or a zero
 * wait with GEMM_F16_FAULT_SKIP_LOADS.
 */
int attn_f16_debug_inject(int fault, uint32_t wait_us);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_F16_H */
