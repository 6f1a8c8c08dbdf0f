/*
 * gbgemm.h - C ABI of the projection GEMM that sits on either side of the
 * attention forward in libgbattn.so (the QKV and O projections of the
 * decoder chain on "CS149 L11: Programming Specialized Hardware", section 6;
 * the matrix multiply of its section 4).
 *
 * All pointers are device pointers on the current CUDA device; the caller
 * owns all memory.  Calls are asynchronous on `stream`; device-side failures
 * (a bounded wait that gave up) are reported by attn_check_device() in
 * gbattn.h.
 */
#ifndef GBGEMM_H
#define GBGEMM_H

#include "gbattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gemm_bf16_nt - C = A B^T with fp32 accumulation.
 *
 *  a  bf16 [M, K], row-major (activations: one row per token).
 *  b  bf16 [N, K], row-major (a linear layer's weight: one row per output
 *     feature).
 *  c  [M, N], row-major, written: fp32 when c_fp32 != 0, else bf16 (each
 *     fp32 sum rounded once, to nearest even).
 *  M, N, K > 0; K % 8 == 0 (rows of A and B are whole 16-byte units, the
 *  tensor-memory-accelerator rule) and N % 2 == 0.  Pointers 16-byte
 *  aligned.
 *
 * For M > 128 the two CTAs of a thread-block cluster share each 256 x 256
 * output tile (the environment variable ATTN_GEMM_SINGLE_CTA=1 selects the
 * one-CTA kernel with 128 x 256 tiles instead, for comparison).
 *
 * Returns ATTN_OK once the kernel is enqueued, ATTN_ERR_INVALID_ARG for a
 * null or misaligned pointer or a size outside the rules above,
 * ATTN_ERR_UNSUPPORTED for sizes past 32-bit row indexing, ATTN_ERR_CUDA /
 * ATTN_ERR_NO_DEVICE as attn_fwd does.
 */
int gemm_bf16_nt(const void* a, const void* b, void* c, int M, int N, int K, int c_fp32,
                 attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GBGEMM_H */
