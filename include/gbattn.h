/*
 * gbattn.h - fused attention forward for one NVIDIA GB300 (sm_103a), C ABI.
 *
 * The operation is the FlashAttention forward
 *
 *     O = softmax(mask(scale * Q K^T)) V,     LSE_i = log sum_j exp(scale * q_i . k_j)
 *
 * computed tile by tile without materialising the score matrix.  Its stage
 * order (QK^T -> Mask -> Softmax -> x V) is the FlashAttention metapipeline of
 * "CS149 L11: Programming Specialized Hardware", section 5; the softmax is the
 * Map(exp) / Reduce(+) / Zip(/) chain of the same section, evaluated online
 * with a running row maximum and normaliser as in the FA2-style kernel of
 * "Distilling a 4.5 hour CUDA talk", section 7, with log2(e) folded into the
 * scale (sections 2 and 7 of that page).
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers on the current CUDA device; the
 *    caller owns every buffer.  Nothing is freed or retained after return.
 *  - Layouts are dense row-major [batch, head, sequence, feature], the
 *    {batch, head, seq, col} four-dimensional global layout of "Distilling a
 *    4.5 hour CUDA talk", sections 7 and 10.
 *  - Work is enqueued on `stream` (NULL = the legacy default stream) and the
 *    call returns without waiting for it.  The caller synchronises.
 *  - Errors are returned as attn_status codes; nothing prints, throws or exits.
 *  - Host threads may call concurrently on different streams; the library
 *    keeps no mutable device state across calls except the device error word
 *    read by attn_check_device().
 */
#ifndef GBATTN_H
#define GBATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, spelled without the CUDA headers. */
typedef struct CUstream_st* attn_stream_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, Hq % Hkv != 0,
                                  misaligned pointer, bad scale, bad aliasing   */
    ATTN_ERR_UNSUPPORTED = 2,  /* head dims not built, or a 576/512 shape whose
                                  V is not the first 512 features of K          */
    ATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed             */
    ATTN_ERR_TIMEOUT = 4,      /* a kernel gave up on a bounded wait            */
    ATTN_ERR_NO_DEVICE = 5,    /* no sm_103 device is current                   */
    ATTN_ERR_SCRATCH_LIMIT = 6 /* attn_decode_fwd_noalloc: problem needs more
                                  scratch than its fixed static array holds     */
} attn_status;

/*
 * attn_fwd - attention forward, O and LSE.
 *
 *  q    bf16 [B, Hq,  Nq,  d_qk], contiguous.
 *  k    bf16 [B, Hkv, Nkv, d_qk], contiguous.
 *  v    bf16 [B, Hkv, Nkv, d_v], contiguous; OR v == k with d_v < d_qk, in
 *       which case V is the first d_v features of each K row (row stride d_qk),
 *       the head-dim 576/512 latent layout of "Distilling a 4.5 hour CUDA
 *       talk", sections 12-13.
 *  o    fp32 [B, Hq, Nq, d_v], written.
 *  lse  fp32 [B, Hq, Nq], written: natural-log log-sum-exp of the scaled
 *       logits over the visible keys; -inf for a row with no visible key (its
 *       O row is 0).  May be NULL to skip it.
 *  Hq % Hkv == 0; query head h reads KV head h / (Hq / Hkv).
 *  causal != 0: key j is visible to query i iff j <= i + (Nkv - Nq)
 *       (aligned at the bottom-right corner; the plain lower triangle when
 *       Nq == Nkv).
 *  scale >= 0 and finite; the logits are scale * q_i . k_j.
 *
 * Supported (d_qk, d_v): (64, 64) and (128, 128) through the prefill kernel,
 * any Nq and Nkv >= 1.  (576, 512) with V aliased to the first 512 features
 * of K (v == k): Nq == 1 and Hq / Hkv <= 128 through the split-KV decode
 * kernel plus a combine kernel (one query sees every key under the
 * bottom-right causal alignment, so the causal flag changes nothing there);
 * any other Nq, causal or not, through the same kernel in prefill mode on
 * blocks of 128 query rows, which writes O and LSE directly.  The decode
 * path takes a
 * stream-ordered workspace (cudaMallocFromPoolAsync / cudaFreeAsync on
 * `stream`) from a memory pool the library creates per device on the first
 * decode call; the pool
 * keeps freed memory for the next call (it never shrinks below the largest
 * workspace used so far), so repeated calls map no new memory.
 *
 * Pointers must be 16-byte aligned (the tensor-memory-accelerator rule).
 * Returns ATTN_OK once the kernels are enqueued.  Device-side failures are
 * reported later by attn_check_device().  With the environment variable
 * ATTN_CHECK=1 the call synchronises `stream` and reports them itself.
 */
int attn_fwd(const void* q, const void* k, const void* v, float* o, float* lse,
             int B, int Hq, int Hkv, int Nq, int Nkv, int d_qk, int d_v,
             int causal, float scale, attn_stream_t stream);

/*
 * attn_fwd_bf16out - attn_fwd with O written as bf16 (round to nearest even)
 * instead of fp32: same arguments, layouts, supported shapes, LSE (fp32) and
 * errors, with o a bf16 [B, Hq, Nq, d_v] buffer (16-byte aligned).  It
 * halves O's share of the HBM traffic; the arithmetic is unchanged (fp32
 * accumulation, one rounding of each normalised output).
 */
int attn_fwd_bf16out(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int Nq, int Nkv, int d_qk, int d_v,
                     int causal, float scale, attn_stream_t stream);

/*
 * attn_fwd_dropout - attn_fwd with dropout on the softmax weights, the stage
 * between Softmax and x V in the FlashAttention pipeline on "CS149 L11:
 * Programming Specialized Hardware", section 5 (the training forward).
 *
 *   O = (P * Keep) V * 256 / (256 - t),  P = softmax(mask(scale Q K^T)),
 *   t = floor(p_drop * 256 + 1/2),
 *
 * where Keep[b, h, i, j] is 1 iff the 8-bit uniform of key j of query row i
 * (its position in the sequence) in head h of batch b is >= t.  That uniform
 * is byte (j & 3) (the least significant for j & 3 = 0) of word
 * ((j >> 2) & 3) of Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC 2011) at
 * counter (j >> 4, i, h, b) and key (seed mod 2^32, seed >> 32): a pure
 * function of the position and the seed, so a backward pass can redraw the
 * same mask.  The realised drop probability is t / 256 and the scale keeps
 * E[O] equal to attn_fwd's O.  LSE is attn_fwd's (dropout does not change
 * it).
 *
 * Arguments, layouts and errors as attn_fwd, O fp32, for the prefill shapes
 * (d_qk == d_v, 64 or 128); ATTN_ERR_UNSUPPORTED for the latent shape and
 * ATTN_ERR_INVALID_ARG unless p_drop == 0 or 1/512 <= p_drop with t < 256:
 * a nonzero p_drop below 1/512 would round to t = 0 and silently drop
 * nothing, so it is refused rather than run.  p_drop == 0 runs the same
 * kernel as attn_fwd.
 */
int attn_fwd_dropout(const void* q, const void* k, const void* v, float* o, float* lse,
                     int B, int Hq, int Hkv, int Nq, int Nkv, int d_qk, int d_v,
                     int causal, float scale, float p_drop, unsigned long long seed,
                     attn_stream_t stream);

/*
 * attn_fwd_bshd - attn_fwd (head dims 64 and 128) on token-major tensors:
 * the layout in which a projection GEMM writes Q, K and V (one row per token,
 * the heads side by side), so attention reads them in place and writes O in
 * the layout the output projection reads ("CS149 L11: Programming
 * Specialized Hardware", section 6: the Q/K/V GEMMs, attention and the O
 * GEMM of one decoder layer).
 *
 *  q  bf16, element (b, h, i, c) at q[(b * Nq + i) * q_ld + h * d + c],
 *     h < Hq, i < Nq, c < d.
 *  k  bf16, element (b, g, j, c) at k[(b * Nkv + j) * k_ld + g * d + c],
 *     g < Hkv.
 *  v  bf16, same form with v_ld.
 *  o  written, element (b, h, i, c) at o[(b * Nq + i) * o_ld + h * d + c]:
 *     fp32 when o_fp32 != 0, else bf16 (each value rounded once, to nearest
 *     even).  Elements of a row past Hq * d are not touched.  o must not
 *     overlap q, k or v.
 *  lse  fp32 [B, Hq, Nq] (head-major, as in attn_fwd), or NULL.
 *  d is 64 or 128 (d_qk == d_v == d).  Each ld counts elements, is a multiple
 *  of 8 and at least the heads' width (Hq * d for q and o, Hkv * d for k and
 *  v); pointers are 16-byte aligned, so Q, K and V may be column slices of
 *  one [B * N, (Hq + 2 * Hkv) * d] buffer.
 *  Heads, GQA map, causal alignment, scale and errors as in attn_fwd;
 *  ATTN_ERR_UNSUPPORTED for another d, or sizes past the tensor map's 2^40-byte
 *  strides or 32-bit row indexing.
 */
int attn_fwd_bshd(const void* q, const void* k, const void* v, void* o, float* lse,
                  int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                  long long q_ld, long long k_ld, long long v_ld, long long o_ld,
                  int o_fp32, int causal, float scale, attn_stream_t stream);

/*
 * attn_check_device - synchronise `stream` and read the device error word
 * that the kernels set when a bounded wait gives up (see
 * ATTN_ERR_TIMEOUT).  reset != 0 clears the word.  Returns ATTN_OK,
 * ATTN_ERR_TIMEOUT or ATTN_ERR_CUDA.
 */
int attn_check_device(attn_stream_t stream, int reset);

/* attn_status_string - static text for a status code (never NULL). */
const char* attn_status_string(int status);

/* attn_last_cuda_error - static text of the last CUDA error seen by this
 * thread's most recent failing call ("" if none). */
const char* attn_last_cuda_error(void);

/* attn_version - 100 * major + minor of this library. */
int attn_version(void);

/*
 * attn_decode_workspace_bytes - bytes of stream-ordered workspace attn_fwd
 * allocates (and frees, on the same stream) for a (576, 512) decode shape
 * with B * Hkv KV planes and Nkv keys on the current device.  0 if the
 * arguments are not positive or no sm_103 device is current.
 */
size_t attn_decode_workspace_bytes(int B, int Hkv, int Nkv);

/*
 * attn_decode_fwd_noalloc - the (576, 512) split-KV decode of attn_fwd,
 * without any memory allocation.  The paper has no counterpart; it is a
 * library service.
 *
 * Who needs it: callers that cannot let a library allocate device memory at
 * call time - a host framework whose caching allocator already holds the
 * GPU's free memory, a serving loop with a fixed memory budget that must not
 * fail in the middle of a request, or a plug-in whose host forbids
 * allocation.  attn_fwd takes its decode workspace from a stream-ordered
 * pool (cudaMallocFromPoolAsync), which it creates on its first decode call
 * on a device; this entry point neither creates nor uses that pool, and
 * calls no cudaMalloc, cudaFree or any allocating routine.
 *
 * Its split partials go to one static device array of 48 MiB declared in
 * the library.  Every GPU that loads the library holds that array until the
 * process exits.  Problems whose partials would not fit return
 * ATTN_ERR_SCRATCH_LIMIT (the 64 x 128-head x 8192-key shape needs about
 * 40 MB on a 152-SM GB300).
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture.  All calls on a device share the one array and it keeps
 * the last call's contents; no call relies on it starting at zero.  Calls
 * whose work overlaps on the GPU (e.g. on two streams at once) race on the
 * array: serialise them.
 *
 *  q   bf16 [B, Hq, 1, 576];  kv bf16 [B, Hkv, Nkv, 576] holding K, with V
 *      the first 512 features of each row;  o fp32 [B, Hq, 1, 512];
 *  lse fp32 [B, Hq, 1] or NULL.  Hq / Hkv <= 128.  Same numbers, layouts,
 *  errors and asynchrony as attn_fwd(q, kv, kv, o, lse, B, Hq, Hkv, 1, Nkv,
 *  576, 512, 0, scale, stream).
 */
int attn_decode_fwd_noalloc(const void* q, const void* kv, float* o, float* lse,
                            int B, int Hq, int Hkv, int Nkv, float scale,
                            attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H */
