/*
 * gblayer.h - C ABI of one attention layer slice in libgbattn.so: the Q/K/V
 * projection, the attention forward and the output projection of a decoder
 * layer, in the order "CS149 L11: Programming Specialized Hardware",
 * section 6 lists them (Q/K/V GEMMs, Q K^T, scale, mask, softmax, x V, the O
 * GEMM).  No normalisation, rotary embedding or bias: the slice is exactly
 * these three contractions.
 *
 * All pointers are device pointers on the current CUDA device, 16-byte
 * aligned; the caller owns all memory.  The call enqueues three kernels on
 * `stream` and returns; device-side failures are reported by
 * attn_check_device() in gbattn.h.
 */
#ifndef GBLAYER_H
#define GBLAYER_H

#include "gbattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_layer_fwd - Y = Attn(X W_qkv^T) W_o^T for B sequences of N tokens.
 *
 *  x      bf16 [B * N, d_model], one row per token (sequence-major).
 *  w_qkv  bf16 [(Hq + 2 * Hkv) * d, d_model]: the Hq * d rows of W_q, then
 *         the Hkv * d rows of W_k, then the Hkv * d rows of W_v (PyTorch's
 *         Linear weight layout, one row per output feature).
 *  w_o    bf16 [d_model, Hq * d].
 *  qkv    written, bf16 [B * N, (Hq + 2 * Hkv) * d]: X W_qkv^T with fp32
 *         accumulation, rounded once to bf16.  Feature h * d + c of a row is
 *         head h's feature c of Q; the K heads start at column Hq * d and the
 *         V heads at (Hq + Hkv) * d.
 *  o      written, bf16 [B * N, Hq * d]: the attention output of each token,
 *         head h at columns [h * d, (h + 1) * d), each value rounded once.
 *  y      written, [B * N, d_model]: o W_o^T, fp32 when y_fp32 != 0, else bf16.
 *  lse    fp32 [B, Hq, N] natural-log LSE of the scaled logits, or NULL.
 *  Attention is self-attention (Nq == Nkv == N) with attn_fwd's GQA map,
 *  causal alignment and scale.  d is 64 or 128; d_model % 8 == 0.
 *
 * Returns the first failing step's status: ATTN_ERR_INVALID_ARG for a null
 * pointer or a size rule of gemm_bf16_nt or attn_fwd_bshd,
 * ATTN_ERR_UNSUPPORTED for another d or sizes past 32-bit indexing,
 * ATTN_ERR_CUDA / ATTN_ERR_NO_DEVICE as attn_fwd.  Steps before a failing one
 * stay enqueued.
 */
int attn_layer_fwd(const void* x, const void* w_qkv, const void* w_o, void* qkv, void* o, void* y, float* lse,
                   int B, int N, int d_model, int Hq, int Hkv, int d, int causal, float scale, int y_fp32,
                   attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GBLAYER_H */
