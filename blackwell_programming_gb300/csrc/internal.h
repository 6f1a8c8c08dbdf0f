// internal.h - launch interfaces between the C-ABI layer and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gbattn {

// Prefill: one persistent CTA per SM walks "units" of two 128-row query
// tiles of one (batch, head) pair.
struct PrefillParams {
  float* o;            // fp32 O, or null when o_bf16 is set
  uint16_t* o_bf16;    // bf16 O (same layout), or null
  float* lse;          // may be null; [B, Hq, Nq]
  int B, Hq, Hkv, Nq, Nkv, d_v;
  // Layout of Q, K and V in their 4-D tensor maps: 0 = (features, rows,
  // heads, batch), i.e. [B, H, N, d]; 1 = (features, heads, rows, batch),
  // i.e. token-major [B, N, H, d] with any token stride.
  int token_major;
  // O element (b, h, row, c) is at o[b * o_sb + h * o_sh + row * o_sr + c].
  long long o_sb, o_sh, o_sr;
  int causal;
  float scale_log2;    // scale * log2(e)
  // Dropout on P (drop_t == 0: none).  Key j of query row i in head (b, h)
  // is dropped iff its 8-bit uniform is below drop_t; the uniform is byte
  // (j & 3) of word ((j >> 2) & 3) of Philox4x32-10 at counter
  // (j >> 4, i, h, b) and key (seed_lo, seed_hi).  Kept weights are scaled
  // by drop_scale = 256 / (256 - drop_t) in the epilogue.
  uint32_t seed_lo, seed_hi, drop_t;
  float drop_scale;
  // The generator's key for each of its ten rounds, (k0, k1) of round r at
  // [2r], [2r + 1]: the key schedule is the same for every call, so the
  // kernel reads it from its parameters instead of advancing the key.
  uint32_t round_keys[20];
  // Exponentials on the FMA pipe: one pair in every exp2_split (0, 4 or 8;
  // 0 = all on the SFU), dropout-free kernels only.
  int exp2_split;
  int tiles_per_unit;  // 128-row query tiles per work unit: 2, or 1 for problems under one wave
  // 1: a unit is one 128-row query tile and both tile slots take it, slot 0
  // the first ceil(n / 2) of its n key tiles and slot 1 the rest; the two
  // partial softmax states are merged in the epilogue (tiles_per_unit 1, D 64)
  int kv_split;
  int num_units;       // B * Hq * nqb
  int nqb;             // ceil(Nq / (128 * tiles_per_unit))
  int nkv_tiles;       // ceil(Nkv / 128)
  unsigned* err;       // device error word
};

cudaError_t launch_prefill(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int num_sms, cudaStream_t stream);

// Split-KV decode for the latent head-dim 576 / 512 shape (V = first 512
// features of K).  The Hq / Hkv query heads that share a KV head form the
// rows of one 128-row tile; a "plane" is one (batch, KV head) pair.
struct DecodeParams {
  const uint16_t* q;   // bf16 Q [planes * group, 576] (the kernel loads part of it into TMEM)
  float* o_part;       // [grid * max_seg, 128, 256] partial O (normalised), per half
  float* lse_part;     // [grid * max_seg, 128] partial LSE (natural log)
  int planes;          // B * Hkv
  int group;           // Hq / Hkv, <= 128
  int Nkv;
  int tiles;           // ceil(Nkv / decode_key_tile())
  int max_seg;         // partial slots per CTA
  float scale_log2;    // scale * log2(e)
  unsigned* err;
};

// Prefill (Nq > 1, causal or not) for the same latent shape, run by the
// decode kernel on blocks of 128 query rows of one (batch, query head); each
// work item writes its half of O and (half 0) the LSE directly.
struct LatentPrefillParams {
  const uint16_t* q;   // bf16 Q [B * Hq, Nq, 576]
  float* o;            // fp32 O [B * Hq, Nq, 512], or null when o_bf16 is set
  uint16_t* o_bf16;    // bf16 O (same layout), or null
  float* lse;          // fp32 LSE [B * Hq, Nq], may be null
  int B, Hq, Hkv, Nq, Nkv;
  int causal;
  int tiles;           // ceil(Nkv / decode_key_tile())
  int nqb;             // ceil(Nq / 128)
  int num_units;       // 2 * B * Hq * nqb
  float scale_log2;    // scale * log2(e)
  unsigned* err;
};

// The latent kernel reads Q and K through tensor maps of a [planes, rows,
// 576] bf16 tensor seen as (64 features, rows, 9 chunks of 64 features,
// planes): Q in boxes of kLatentQRows rows x kLatentQChunks chunks (the
// shared-memory part of Q, chunks 6..8), K in boxes of kLatentKeyRows keys x
// 5, 4 or 1 chunks.
constexpr int kLatentQRows = 128;
constexpr int kLatentQChunks = 3;
constexpr int kLatentKeyRows = 64;
struct LatentMaps {
  CUtensorMap q, k5, k4, k1;
};

cudaError_t launch_latent_prefill(const LatentMaps& m, const LatentPrefillParams& p, int num_sms,
                                  cudaStream_t stream);

// The CTA-pair decode (decode_pair_sm103.cu): one CTA of each cluster of two
// computes the score tiles and the softmax, the other holds O and computes
// P V.  K is read through the same 4-D view as above, in boxes of
// kLatentKeyRows keys x kPairKeyChunks chunks (score CTA) and x
// kPairValueChunks chunks (value CTA: V, the first 512 features), and Q in
// boxes of kLatentKeyRows rows x kPairKeyChunks chunks (rows past the group
// read as zeros).  The
// pieces go to decode_pair_slots(planes, pairs) slots of [128, 512] floats
// and 128 LSEs, which launch_combine_pair merges.
constexpr int kPairKeyChunks = 3;
constexpr int kPairValueChunks = 8;
int decode_pair_slots(int planes, int pairs);
// Clusters of the pair kernel that fit on the device at once (0 on success).
int decode_pair_max_pairs(int num_sms, int* out);
// `tq` maps Q [planes, group, 576] in boxes of 64 rows x 3 chunks.
cudaError_t launch_decode_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, int pairs, cudaStream_t stream);
cudaError_t launch_combine_pair(const DecodeParams& p, int pairs, float* o, uint16_t* o_bf16, float* lse,
                                cudaStream_t stream);
// The latent prefill on the same CTA pairs (num_units = B * Hq * nqb), with
// Q mapped as [B * Hq, Nq, 576] and K as [B * Hkv, Nkv, 576] like the decode.
cudaError_t launch_latent_prefill_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                       const LatentPrefillParams& p, int pairs, cudaStream_t stream);

// Number of partial slots each CTA needs for a grid of `grid` CTAs.
int decode_max_segments(int planes, int tiles, int grid);
int decode_tiles(int Nkv);
int decode_key_tile();   // keys per K tile of the decode kernel (TMA box rows)

cudaError_t launch_decode(const LatentMaps& m, const DecodeParams& p, int grid, cudaStream_t stream);

// Merge the partials of every row into O [planes * group, 512] and LSE; O is
// fp32 (o) or, when o is null, bf16 (o_bf16).
cudaError_t launch_combine(const DecodeParams& p, int grid, float* o, uint16_t* o_bf16, float* lse,
                           cudaStream_t stream);

// Projection GEMM: C [M, N] = A [M, K] B [N, K]^T, bf16 in, fp32 accumulate,
// bf16 or fp32 out; 128 x 256 output tiles walked by persistent CTAs.
struct GemmParams {
  void* c;             // bf16 or fp32 C [M, N]
  int M, N, K;
  int c_fp32;          // 1: C is fp32, 0: bf16
  int tiles_m, tiles_n, num_tiles;
  int group_m;         // CTA-pair kernel: 256-row blocks per raster group
  unsigned* err;
};

int gemm_tile_rows();
int gemm_tile_cols();
int gemm_tile_depth();
// CTA-pair GEMM (256 x 256 tiles over two SMs), chosen for M > 128.  Its B
// map takes boxes of gemm_b_box_rows(true) rows; tiles_m counts 256-row
// blocks.
bool gemm_use_pair(int M);
int gemm_b_box_rows(bool use_pair);
// `tc` (or null): C as a 2-D map (N, M) with boxes of 32 rows x 128 bytes and
// the 128-byte swizzle, for the TMA-store epilogue (C's row pitch a multiple
// of 16 bytes); null: the epilogue stores from registers.
cudaError_t launch_gemm_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap* tc,
                             const GemmParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, int num_sms,
                        cudaStream_t stream);

}  // namespace gbattn
