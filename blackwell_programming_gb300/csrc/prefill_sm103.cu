// prefill_sm103.cu - fused attention forward (prefill), head dims 64 and 128.
//
// What it computes: O = softmax(mask(scale * Q K^T)) V and the row LSE,
// streaming K/V tiles through the QK^T -> Mask -> Softmax -> x V pipeline of
// "CS149 L11: Programming Specialized Hardware", section 5, with the online
// softmax (running max and normaliser) of the FA2-style kernel in
// "Distilling a 4.5 hour CUDA talk", section 7, and log2(e) folded into the
// scale (same page, sections 2 and 7).
//
// How, on sm_103a (a design for this chip, not the pages' RTX 4090 / H100
// kernels):
//  * One persistent CTA per SM walks a static longest-first list of units; a
//    unit is two 128-row query tiles (t = 0, 1) of one (batch, head).  The
//    query heads that share a KV head are adjacent in the list so their K/V
//    tiles are reused from L2 ("Distilling...", section 5, L2 super-blocks).
//  * Warp 9 is the TMA producer: Q tiles once per unit, then a ring of K and
//    a ring of V stages, each stage guarded by a full / empty mbarrier pair
//    (expect-tx on full, tcgen05.commit on empty) - the producer/consumer
//    template of "Distilling...", section 12, with the mbarrier handoff of
//    section 13.
//  * Warps 8 and 10 issue the tcgen05.mma of query tile 0 and 1 (warp-uniform
//    code, one elected lane per instruction).  S_t = Q_t K_j^T lands in
//    tensor memory (TMEM); the softmax writes P_t (bf16) over S_t and the
//    MMA computes O_t += P_t V_j with P read straight from TMEM.  The two
//    query tiles ping-pong: the tensor core works on one tile while the
//    softmax warpgroup of the other one runs.  P_t is published in two
//    halves (keys 0..63, then 64..127), and P V starts on the first half
//    while the softmax computes the second.
//  * Warpgroups 0 and 1 own query tile 0 and 1.  TMEM lane i is row i, so a
//    thread owns a whole row: max, exp2 and sum stay in-thread.  They also
//    rescale O (only when the running max grew by more than 2^8, which keeps
//    the result exact) and run the epilogue: O / l and LSE to global memory.
//  * Problems under one wave at D = 64 run key-split units (KSPLIT): both
//    query tiles are the same rows over two halves of the key tiles, and the
//    epilogue merges the two partial softmax states.
//
// TMEM columns: S0 [0,128)  S1 [128,256)  O0 [256,256+D)  O1 [256+D,256+2D).
#include <cmath>

#include "internal.h"
#include "philox.cuh"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int BM = 128;               // query rows per tile (TMEM lanes)
constexpr int BN = 128;               // keys per K/V tile
constexpr int kThreads = 384;         // 3 warpgroups
constexpr int kMmaWarp0 = 8;    // MMA issuer for query tile 0 (also owns the TMEM allocation)
constexpr int kTmaWarp = 9;
constexpr int kMmaWarp1 = 10;   // MMA issuer for query tile 1
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O only past 2^8
constexpr uint32_t kFull = 0xFFFFFFFFu;
// Register split: the MMA / TMA warpgroup gives registers to the two softmax
// warpgroups.  128 * 96 + 256 * 200 = 63488 must not exceed the launch
// allocation (384 threads x registers per thread), which the host checks.
constexpr uint32_t kRegsLow = 96;
constexpr uint32_t kRegsHigh = 200;
constexpr int kRegsNeededAtLaunch = (128 * kRegsLow + 256 * kRegsHigh + kThreads - 1) / kThreads;

template <int D>
struct Cfg {
  static constexpr int KCH = D / 64;                 // 128-byte column chunks per row
  static constexpr uint32_t Q_BYTES = BM * D * 2;
  static constexpr uint32_t KV_BYTES = BN * D * 2;
  static constexpr uint32_t CHUNK_Q = BM * 128;      // one 64-column chunk of a Q tile
  static constexpr uint32_t CHUNK_KV = BN * 128;
  static constexpr int KS = (D == 128) ? 2 : 4;      // K stages
  static constexpr int VS = (D == 128) ? 3 : 4;      // V stages
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + KS * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + VS * KV_BYTES;
  // barrier indices
  static constexpr int B_QFULL = 0, B_QEMPTY = 2, B_KFULL = 4, B_KEMPTY = 4 + KS, B_VFULL = 4 + 2 * KS,
                       B_VEMPTY = 4 + 2 * KS + VS, B_SFULL = 4 + 2 * KS + 2 * VS, B_PFULL = B_SFULL + 2,
                       B_OFULL = B_PFULL + 2, B_OEMPTY = B_OFULL + 2, B_DRAIN = B_OEMPTY + 2,
                       B_TURN = B_DRAIN + 1, B_PHALF = B_TURN + 2, B_MERGE = B_PHALF + 2, NUM_BARS = B_MERGE + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  // (m, l) of every row of both tile slots for the merge of key-split units
  // (D = 64 only: at D = 128 the rings leave no room)
  static constexpr uint32_t MRG_BYTES = (D == 64) ? 2u * BM * 8u : 0u;
  static constexpr uint32_t OFF_MRG = OFF_MISC + 16;
  static constexpr uint32_t SMEM_BYTES = OFF_MRG + MRG_BYTES + 1024;   // + slack for 1024-byte alignment
  // TMEM column of S_t and O_t
  __device__ static constexpr uint32_t col_s(int t) { return static_cast<uint32_t>(t) * 128u; }
  __device__ static constexpr uint32_t col_o(int t) { return 256u + static_cast<uint32_t>(t) * D; }
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, false, true);
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct Unit {
  int b, h;
  int row0[2];   // first query row of tile 0 / 1 (Nq: the tile does not exist)
  int n[2];      // K/V tiles visited by query tile 0 / 1
  int k0[2];     // index of the first of them
};

__device__ __forceinline__ int kv_tiles_for(int q0, const PrefillParams& p) {
  if (q0 >= p.Nq) return 0;
  if (!p.causal) return p.nkv_tiles;
  const int last_row = min(q0 + BM - 1, p.Nq - 1);
  const int last_key = last_row + (p.Nkv - p.Nq);
  if (last_key < 0) return 0;
  return min(last_key / BN + 1, p.nkv_tiles);
}

// Unit u: query-block index descending (longest causal work first), then
// (batch, head) with the heads of one KV group adjacent.  A block is two
// 128-row tiles, or one when the problem has fewer two-tile blocks than the
// GPU has SMs: then tile 1 does not exist and its warps idle, or, in a
// key-split kernel, both tile slots take the one tile and share out its key
// tiles (slot 0 the first ceil(n / 2), slot 1 the rest).
__device__ __forceinline__ Unit decode_unit(int u, const PrefillParams& p, bool ksplit) {
  Unit U;
  const int bh_count = p.B * p.Hq;
  const int qb_rev = u / bh_count;
  const int bh = u - qb_rev * bh_count;
  const int qb = p.nqb - 1 - qb_rev;
  U.b = bh / p.Hq;
  U.h = bh - U.b * p.Hq;
  U.k0[0] = U.k0[1] = 0;
  if (ksplit) {
    // both slots take the same rows; slot 0 the first half of the key tiles
    U.row0[0] = U.row0[1] = qb * BM;
    const int n = kv_tiles_for(U.row0[0], p);
    U.n[0] = (n + 1) / 2;
    U.n[1] = n - U.n[0];
    U.k0[1] = U.n[0];
    return U;
  }
  if (p.tiles_per_unit == 1) {
    U.row0[0] = qb * BM;
    U.row0[1] = p.Nq;
  } else {
    U.row0[0] = qb * 2 * BM;
    U.row0[1] = qb * 2 * BM + BM;
  }
  U.n[0] = kv_tiles_for(U.row0[0], p);
  U.n[1] = kv_tiles_for(U.row0[1], p);
  return U;
}

// Snake order over rounds of gridDim.x units.
__device__ __forceinline__ int unit_at(int it) {
  const int base = it * static_cast<int>(gridDim.x);
  return (it & 1) ? base + static_cast<int>(gridDim.x - 1 - blockIdx.x) : base + static_cast<int>(blockIdx.x);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(kFull, ok);
}

// Dropout keep flags.  Key 4m + k of a generator word w is kept iff its byte
// u_k = byte k of w satisfies u_k >= t, i.e. iff u_k + (256 - t) reaches 256.
// Each 16-bit lane takes one byte shifted up by 7 (the even bytes, then the
// odd ones), so with cdrop = (256 - t) * (2^7 + 2^23) that carry lands on bit
// 15 or 31 and no lane overflows into the next (u + 256 - t < 512).  One byte
// permute then gathers the four carries into the top bits of the result's
// bytes: byte 0 <- key 1, byte 1 <- key 0, byte 2 <- key 3, byte 3 <- key 2.
__device__ __forceinline__ uint32_t keep_flags(uint32_t w, uint32_t cdrop) {
  uint32_t wo, f;
  asm("prmt.b32 %0, %1, 0, 0x4341;" : "=r"(wo) : "r"(w));   // bytes 1 and 3 down to 0 and 2
  const uint32_t ev = (w & 0x00FF00FFu) * 128u + cdrop;
  const uint32_t od = wo * 128u + cdrop;
  asm("prmt.b32 %0, %1, %2, 0x3715;" : "=r"(f) : "r"(ev), "r"(od));
  return f;
}

// Two flag words in one register: fa's flags stay on bit 7 of each byte,
// fb's move to bit 6 (the other bits are don't-care).
__device__ __forceinline__ uint32_t keep_flags2(uint32_t fa, uint32_t fb) {
  return (fa & 0x80808080u) | ((fb >> 1) & 0x40404040u);
}

// AND masks for the two bf16 pairs of a flag word's keys (m01: keys 0 and 1
// in the low and high half; m23: keys 2 and 3): a sign-replicating byte
// permute spreads each flag bit over the 16 bits of its key's half.
__device__ __forceinline__ void keep_pair_masks(uint32_t f, uint32_t& m01, uint32_t& m23) {
  asm("prmt.b32 %0, %1, 0, 0x8899;" : "=r"(m01) : "r"(f));
  asm("prmt.b32 %0, %1, 0, 0xAABB;" : "=r"(m23) : "r"(f));
}

// Epilogue of a key-split unit: slots 0 and 1 hold the same rows' partial
// states (O_t relative to the reference m_t, normaliser l_t) over the first
// and second part of the key tiles.  With m = max(m_0, m_1) and
// L = sum_t 2^(m_t - m) l_t, the row's output is sum_t 2^(m_t - m) O_t / L
// (the same merge of partial softmax states as the split-KV combine), and
// LSE = (m + log2 L) ln 2.  Each slot's warps write their rows' (m, l) to
// shared memory, meet the other slot on an mbarrier, then merge and store
// half of the columns (slot t: columns t D/2 .. (t+1) D/2 - 1), reading both
// O tiles from TMEM (warps q and 4 + q reach the same TMEM lanes).  A second
// meeting keeps both O tiles in TMEM until both halves are read.
template <int D, bool DROP>
__device__ __forceinline__ bool merge_epilogue(const PrefillParams& p, const Unit& U, int t, uint32_t quad,
                                               uint32_t lane, int row_in_tile, float m_used, float l, uint32_t tm,
                                               float2* mrg, uint32_t merge_bar, uint32_t& mph, const WaitCtx& wctx) {
  using C = Cfg<D>;
  mrg[t * BM + row_in_tile] = make_float2(m_used, l);
  __syncwarp();
  if (lane == 0) mbar_arrive(merge_bar);
  if (!warp_wait(merge_bar, mph, wctx)) return false;
  mph ^= 1u;
  tc_fence_after();   // the other slot's O is complete (it waited for its commit before arriving)
  const float2 oth = mrg[(t ^ 1) * BM + row_in_tile];
  const float m0 = t ? oth.x : m_used, l0 = t ? oth.y : l;
  const float m1 = t ? m_used : oth.x, l1 = t ? l : oth.y;
  const float mm = fmaxf(m0, m1);
  const float a0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - mm);
  const float a1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - mm);
  const float L = a0 * l0 + a1 * l1;
  const float inv = (L > 0.f) ? (DROP ? p.drop_scale : 1.f) / L : 0.f;
  const float f0 = a0 * inv, f1 = a1 * inv;
  const int q0 = U.row0[0];
  const long long ohead = U.b * p.o_sb + U.h * p.o_sh;
  const bool bf = p.o_bf16 != nullptr;
  const bool use0 = U.n[0] > 0, use1 = U.n[1] > 0;   // a slot with no key tile holds no O
#pragma unroll 1
  for (int hl = 0; hl < 2; ++hl) {
    const int ra = static_cast<int>(quad * 32 + hl * 16 + (lane >> 2));   // rows ra and ra + 8 of the tile
    const int src = hl * 16 + static_cast<int>(lane >> 2);
    const float f0a = __shfl_sync(kFull, f0, src), f0b = __shfl_sync(kFull, f0, src + 8);
    const float f1a = __shfl_sync(kFull, f1, src), f1b = __shfl_sync(kFull, f1, src + 8);
    const bool la = q0 + ra < p.Nq, lb = q0 + ra + 8 < p.Nq;
    const long long oa = ohead + (la ? q0 + ra : 0) * p.o_sr + 2 * (lane & 3);
    const long long ob = ohead + (lb ? q0 + ra + 8 : 0) * p.o_sr + 2 * (lane & 3);
    const uint32_t lanes16 = (quad * 32u + hl * 16u) << 16;
#pragma unroll 1
    for (int cc = 0; cc < D / 64; ++cc) {
      const int col = t * (D / 2) + cc * 32;
      uint32_t x0[16], x1[16];
      if (use0) {
        tmem_ld16x256b_x4(tm + lanes16 + C::col_o(0) + col, x0);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) x0[i] = 0u;
      }
      if (use1) {
        tmem_ld16x256b_x4(tm + lanes16 + C::col_o(1) + col, x1);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) x1[i] = 0u;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float y0 = __uint_as_float(x0[4 * k]) * f0a + __uint_as_float(x1[4 * k]) * f1a;
        const float y1 = __uint_as_float(x0[4 * k + 1]) * f0a + __uint_as_float(x1[4 * k + 1]) * f1a;
        const float z0 = __uint_as_float(x0[4 * k + 2]) * f0b + __uint_as_float(x1[4 * k + 2]) * f1b;
        const float z1 = __uint_as_float(x0[4 * k + 3]) * f0b + __uint_as_float(x1[4 * k + 3]) * f1b;
        const int c = col + 8 * k;
        if (bf) {
          if (la) *reinterpret_cast<uint32_t*>(p.o_bf16 + oa + c) = pack_bf16x2(y0, y1);
          if (lb) *reinterpret_cast<uint32_t*>(p.o_bf16 + ob + c) = pack_bf16x2(z0, z1);
        } else {
          if (la) *reinterpret_cast<float2*>(p.o + oa + c) = make_float2(y0, y1);
          if (lb) *reinterpret_cast<float2*>(p.o + ob + c) = make_float2(z0, z1);
        }
      }
    }
  }
  const int row = q0 + row_in_tile;
  if (t == 0 && row < p.Nq && p.lse != nullptr)
    p.lse[static_cast<size_t>(U.b * p.Hq + U.h) * p.Nq + row] =
        (L > 0.f) ? (mm + __log2f(L)) * 0.69314718055994531f : -INFINITY;
  // both slots have read both O tiles before either is handed back
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(merge_bar);
  if (!warp_wait(merge_bar, mph, wctx)) return false;
  mph ^= 1u;
  return true;
}

// SPLIT > 0: one exponential pair in every SPLIT on the FMA pipe (ex2_fma2),
// the others on the SFU.  KSPLIT: key-split units (D = 64 only).
template <int D, bool DROP, int SPLIT, bool KSPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);
  const WaitCtx wctx{abort_flag, p.err};

  const uint32_t warp = warp_id(), lane = lane_id();
  static_assert(!KSPLIT || C::MRG_BYTES > 0, "key-split units need the merge buffer");
  constexpr bool ksplit = KSPLIT;

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::B_QFULL + t), 1);
      mbar_init(bar(C::B_QEMPTY + t), 1);
      mbar_init(bar(C::B_SFULL + t), 1);
      mbar_init(bar(C::B_PFULL + t), 4);
      mbar_init(bar(C::B_PHALF + t), 4);
      mbar_init(bar(C::B_OFULL + t), 1);
      mbar_init(bar(C::B_OEMPTY + t), 4);
    }
    for (int s = 0; s < C::KS; ++s) {
      mbar_init(bar(C::B_KFULL + s), 1);
      mbar_init(bar(C::B_KEMPTY + s), 2);   // released by both MMA warps
    }
    for (int s = 0; s < C::VS; ++s) {
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), 2);
    }
    mbar_init(bar(C::B_DRAIN), 2);
    mbar_init(bar(C::B_TURN + 0), 1);
    mbar_init(bar(C::B_TURN + 1), 1);
    if constexpr (KSPLIT) mbar_init(bar(C::B_MERGE), 8);   // the eight softmax warps
    fence_mbar_init();
  }
  if (warp == kMmaWarp0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  if (warp >= 8) {
   regs_dec<kRegsLow>();
   if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t pol_kv = l2_policy_evict_last();
      const uint64_t pol_q = l2_policy_evict_first();
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0, qph = 0u;   // bit t: parity of Q tile t
      // Buffers filled so far (bit b) and the parity of their last fill, for
      // the drain at exit.  Bits: Q tile t -> t, K stage s -> 2 + s,
      // V stage s -> 2 + KS + s.
      uint32_t filled = 0u, fill_par = 0u;
      auto note_fill = [&](int b, uint32_t par) {
        filled |= 1u << b;
        fill_par = (fill_par & ~(1u << b)) | (par << b);
      };
      const int group = p.Hq / p.Hkv;
      for (int it = 0;; ++it) {
        const int u = unit_at(it);
        if (u >= p.num_units) break;
        const Unit U = decode_unit(u, p, ksplit);
        bool ok = true;
        for (int t = 0; t < 2 && ok; ++t) {
          if (U.n[t] == 0) continue;
          if (!(ok = mbar_wait(bar(C::B_QEMPTY + t), ((qph >> t) & 1u) ^ 1u, wctx))) break;
          qph ^= 1u << t;
          mbar_arrive_expect_tx(bar(C::B_QFULL + t), C::Q_BYTES);
          note_fill(t, ((qph >> t) & 1u) ^ 1u);
          const int qrow = U.row0[t];
          for (int kc = 0; kc < C::KCH; ++kc)
            tma_load_4d(sQ + t * C::Q_BYTES + kc * C::CHUNK_Q, &tmQ, bar(C::B_QFULL + t), kc * 64,
                        p.token_major ? U.h : qrow, p.token_major ? qrow : U.h, U.b, pol_q);
        }
        if (!ok) break;
        const int nmax = max(U.n[0], U.n[1]);
        const int kvh = U.h / group;
        if constexpr (KSPLIT) {
          // Two ring positions per step: slot 0's key tile, then slot 1's.
          // A slot with no key tile at a step gets its position completed by
          // a plain arrive, so both MMA warps still walk every position in
          // order.
          for (int j = 0; j < nmax && ok; ++j) {
            for (int tt = 0; tt < 2; ++tt) {
              if (!(ok = mbar_wait(bar(C::B_KEMPTY + ks), kph ^ 1u, wctx))) break;
              note_fill(2 + ks, kph);
              const int kt = U.k0[tt] + j;
              if (j < U.n[tt]) {
                mbar_arrive_expect_tx(bar(C::B_KFULL + ks), C::KV_BYTES);
                for (int kc = 0; kc < C::KCH; ++kc)
                  tma_load_4d(sK + ks * C::KV_BYTES + kc * C::CHUNK_KV, &tmK, bar(C::B_KFULL + ks), kc * 64,
                              p.token_major ? kvh : kt * BN, p.token_major ? kt * BN : kvh, U.b, pol_kv);
              } else {
                mbar_arrive(bar(C::B_KFULL + ks));
              }
              if (++ks == C::KS) { ks = 0; kph ^= 1u; }
            }
            for (int tt = 0; tt < 2 && ok; ++tt) {
              if (!(ok = mbar_wait(bar(C::B_VEMPTY + vs), vph ^ 1u, wctx))) break;
              note_fill(2 + C::KS + vs, vph);
              const int kt = U.k0[tt] + j;
              if (j < U.n[tt]) {
                mbar_arrive_expect_tx(bar(C::B_VFULL + vs), C::KV_BYTES);
                for (int kc = 0; kc < C::KCH; ++kc)
                  tma_load_4d(sV + vs * C::KV_BYTES + kc * C::CHUNK_KV, &tmV, bar(C::B_VFULL + vs), kc * 64,
                              p.token_major ? kvh : kt * BN, p.token_major ? kt * BN : kvh, U.b, pol_kv);
              } else {
                mbar_arrive(bar(C::B_VFULL + vs));
              }
              if (++vs == C::VS) { vs = 0; vph ^= 1u; }
            }
          }
        } else {
          for (int j = 0; j < nmax && ok; ++j) {
            if (!(ok = mbar_wait(bar(C::B_KEMPTY + ks), kph ^ 1u, wctx))) break;
            mbar_arrive_expect_tx(bar(C::B_KFULL + ks), C::KV_BYTES);
            note_fill(2 + ks, kph);
            for (int kc = 0; kc < C::KCH; ++kc)
              tma_load_4d(sK + ks * C::KV_BYTES + kc * C::CHUNK_KV, &tmK, bar(C::B_KFULL + ks), kc * 64,
                          p.token_major ? kvh : j * BN, p.token_major ? j * BN : kvh, U.b, pol_kv);
            if (++ks == C::KS) { ks = 0; kph ^= 1u; }
            if (!(ok = mbar_wait(bar(C::B_VEMPTY + vs), vph ^ 1u, wctx))) break;
            mbar_arrive_expect_tx(bar(C::B_VFULL + vs), C::KV_BYTES);
            note_fill(2 + C::KS + vs, vph);
            for (int kc = 0; kc < C::KCH; ++kc)
              tma_load_4d(sV + vs * C::KV_BYTES + kc * C::CHUNK_KV, &tmV, bar(C::B_VFULL + vs), kc * 64,
                          p.token_major ? kvh : j * BN, p.token_major ? j * BN : kvh, U.b, pol_kv);
            if (++vs == C::VS) { vs = 0; vph ^= 1u; }
          }
        }
        if (!ok) break;
      }
      // Every issued copy must have landed before the CTA may exit.
      for (int b = 0; b < 2 + C::KS + C::VS; ++b) {
        if (!((filled >> b) & 1u)) continue;
        const int full = b < 2 ? C::B_QFULL + b : (b < 2 + C::KS ? C::B_KFULL + (b - 2) : C::B_VFULL + (b - 2 - C::KS));
        mbar_wait_drain(bar(full), (fill_par >> b) & 1u);
      }
    }
    __syncwarp();
   } else if (warp == kMmaWarp0 || warp == kMmaWarp1) {
    // --------------------------------------------------------- MMA issuers
    // One issuing warp per query tile.  tcgen05.mma issue blocks while the
    // tensor core's queue is full, so a single issuer leaves the tensor core
    // idle whenever it waits on a barrier; with two, one tile's issuer waits
    // for its P while the other issues.  The two pass an issue turn (a pair
    // of mbarriers) once per K/V step, so the tensor core runs tile 0's
    // group [PV_0, S_0] and then tile 1's [PV_1, S_1]: the tiles stay half a
    // period apart and each softmax overlaps the other tile's MMAs instead
    // of running at the same time.  Both walk the same K/V stages and both
    // release each stage (empty barriers count 2).
    const int t = (warp == kMmaWarp0) ? 0 : 1;
    // The whole warp runs this loop (warp-uniform control flow); one elected
    // lane issues each tcgen05 instruction.
    {
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0, qph = 0, pph = 0, oeph = 0;
      // Tile 0 holds the turn first: its first wait is on the phase before
      // the barrier's first one, which counts as complete.
      uint32_t tph = (t == 0) ? 1u : 0u;
      const uint32_t dS = tm + C::col_s(t), dO = tm + C::col_o(t);
      // Base descriptors; a K step adds its byte offset / 16 to the start
      // address field (offsets stay inside the 256 KB window).
      const uint64_t q_desc = smem_desc_sw128(sQ + t * C::Q_BYTES, 16, 1024);
      const uint64_t k_desc0 = smem_desc_sw128(sK, 16, 1024);
      const uint64_t v_desc0 = smem_desc_sw128(sV, C::CHUNK_KV, 1024);
      for (int it = 0;; ++it) {
        const int u = unit_at(it);
        if (u >= p.num_units) break;
        const Unit U = decode_unit(u, p, ksplit);
        const int n = t ? U.n[1] : U.n[0];
        const int nmax = max(U.n[0], U.n[1]);
        // ring positions per step (two in a key-split unit: slot 0's, then
        // slot 1's); both warps wait for and release every position, and
        // each uses its own
        const int lanes = ksplit ? 2 : 1;
        const int own = ksplit ? t : 0;
        bool o_waited = false;
        bool ok = true;
        for (int j = 0; j <= nmax && ok; ++j) {
          const bool do_pv = j >= 1 && j - 1 < n;
          const bool do_s = j < n;
          // every wait of this step first, then the turn
          int vs_own = vs, ks_own = ks;
          if constexpr (KSPLIT) {
            if (j >= 1)
              for (int o = 0; o < lanes && ok; ++o)
                ok = warp_wait(bar(C::B_VFULL + (vs + o) % C::VS), vph ^ ((vs + o) >= C::VS ? 1u : 0u), wctx);
            if (!ok) break;
            if (j < nmax)
              for (int o = 0; o < lanes && ok; ++o)
                ok = warp_wait(bar(C::B_KFULL + (ks + o) % C::KS), kph ^ ((ks + o) >= C::KS ? 1u : 0u), wctx);
            if (!ok) break;
            vs_own = (vs + own) % C::VS;
            ks_own = (ks + own) % C::KS;
          } else {
            if (j >= 1 && !(ok = warp_wait(bar(C::B_VFULL + vs), vph, wctx))) break;
            if (j < nmax && !(ok = warp_wait(bar(C::B_KFULL + ks), kph, wctx))) break;
          }
          if (do_pv) {
            if (!o_waited) {
              if (!(ok = warp_wait(bar(C::B_OEMPTY + t), oeph ^ 1u, wctx))) break;
              oeph ^= 1u;
              o_waited = true;
            }
          }
          if (do_s && j == 0) {
            if (!(ok = warp_wait(bar(C::B_QFULL + t), qph, wctx))) break;
            qph ^= 1u;
          }
          // The turn before P: it is normally free long before P is ready,
          // and taking it first leaves only the P wait between the softmax
          // and the first P V.
          if (!(ok = warp_wait(bar(C::B_TURN + t), tph, wctx))) break;
          tph ^= 1u;
          if (do_pv && !(ok = warp_wait(bar(C::B_PHALF + t), pph, wctx))) break;
          tc_fence_after();
          if (do_pv) {
            // O_t += P_t(j-1) V_{j-1}; P read from TMEM over S_t
            // keys 0..63 as soon as their P is in TMEM, keys 64..127 after
            const uint64_t vd = v_desc0 + ((vs_own * C::KV_BYTES) >> 4);
            {
              uint32_t a[4];
              uint64_t b[4];
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) { a[kk] = dS + kk * 8; b[kk] = vd + ((kk * 16 * 128) >> 4); }
              mma_ts_warp4(dO, a, b, C::IDESC_PV, j - 1 > 0 ? 1u : 0u);
            }
            if (!(ok = warp_wait(bar(C::B_PFULL + t), pph, wctx))) break;
            pph ^= 1u;
            tc_fence_after();
            {
              uint32_t a[4];
              uint64_t b[4];
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) { a[kk] = dS + (4 + kk) * 8; b[kk] = vd + (((4 + kk) * 16 * 128) >> 4); }
              mma_ts_warp4(dO, a, b, C::IDESC_PV, 1u);
            }
          }
          if (do_s) {
            // S_t = Q_t K_j^T, one 64-feature chunk (four MMAs) per elect
            const uint64_t kd = k_desc0 + ((ks_own * C::KV_BYTES) >> 4);
#pragma unroll
            for (int kc = 0; kc < C::KCH; ++kc) {
              uint64_t a[4], b[4];
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                a[kk] = q_desc + ((kc * C::CHUNK_Q + kk * 32) >> 4);
                b[kk] = kd + ((kc * C::CHUNK_KV + kk * 32) >> 4);
              }
              mma_ss_warp4(dS, a, b, C::IDESC_S, kc > 0 ? 1u : 0u);
            }
          }
          mbar_arrive_warp(bar(C::B_TURN + (t ^ 1)));
          if (do_s) {
            mma_commit_warp(bar(C::B_SFULL + t));
            if (j == n - 1) mma_commit_warp(bar(C::B_QEMPTY + t));
          }
          if (j == n && n > 0) mma_commit_warp(bar(C::B_OFULL + t));
          if constexpr (KSPLIT) {
            if (j < nmax)
              for (int o = 0; o < lanes; ++o) {
                mma_commit_warp(bar(C::B_KEMPTY + ks));
                if (++ks == C::KS) { ks = 0; kph ^= 1u; }
              }
            if (j >= 1)
              for (int o = 0; o < lanes; ++o) {
                mma_commit_warp(bar(C::B_VEMPTY + vs));
                if (++vs == C::VS) { vs = 0; vph ^= 1u; }
              }
          } else {
            if (j < nmax) {
              mma_commit_warp(bar(C::B_KEMPTY + ks));
              if (++ks == C::KS) { ks = 0; kph ^= 1u; }
            }
            if (j >= 1) {
              mma_commit_warp(bar(C::B_VEMPTY + vs));
              if (++vs == C::VS) { vs = 0; vph ^= 1u; }
            }
          }
        }
        if (!ok) break;
        // A tile with no K/V tile still takes one o_empty / o_full turn, so
        // its epilogue can never run a barrier phase ahead of this warp.
        if (!o_waited) {
          if (!(ok = warp_wait(bar(C::B_OEMPTY + t), oeph ^ 1u, wctx))) break;
          oeph ^= 1u;
        }
        if (n == 0) mma_commit_warp(bar(C::B_OFULL + t));
      }
      // Let every MMA this warp issued finish before TMEM is released.
      mma_commit_warp(bar(C::B_DRAIN));
      mbar_wait_drain(bar(C::B_DRAIN), 0);
    }
    __syncwarp();
   }
  } else {
    regs_inc<kRegsHigh>();
    // ------------------------------------------------ softmax + epilogue
    const int t = static_cast<int>(warp >> 2);
    const uint32_t quad = warp & 3u;
    const int row_in_tile = static_cast<int>(quad * 32 + lane);
    const uint32_t lane_addr = (quad * 32u) << 16;
    const uint32_t tS = tm + lane_addr + C::col_s(t);
    const uint32_t tO = tm + lane_addr + C::col_o(t);
    const float sl2 = p.scale_log2;
    const uint32_t cdrop = (256u - p.drop_t) * 0x00800080u;
    const int delta = p.Nkv - p.Nq;
    uint32_t sph = 0, ofph = 0, mph = 0;
    for (int it = 0;; ++it) {
      const int u = unit_at(it);
      if (u >= p.num_units) break;
      const Unit U = decode_unit(u, p, ksplit);
      const int n = t ? U.n[1] : U.n[0];
      const int q0 = U.row0[t];
      const int row = q0 + row_in_tile;
      const int kt0 = KSPLIT ? (t ? U.k0[1] : U.k0[0]) : 0;   // first key tile of this slot
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        // Dropout: the keep flags of this row's 128 keys, drawn while the
        // tensor core computes S (one generator call per 16 keys), so the
        // exp loop after the S wait only expands them into pair masks.
        uint32_t rw[DROP ? BN / 8 : 1];
        if constexpr (DROP) {
#pragma unroll
          for (int g = 0; g < BN / 16; ++g) {
            const uint4 r = philox4x32_10_rk(make_uint4(static_cast<uint32_t>((kt0 + j) * (BN / 16) + g),
                                                        static_cast<uint32_t>(row), static_cast<uint32_t>(U.h),
                                                        static_cast<uint32_t>(U.b)),
                                             p.round_keys);
            // two words' flags per register: the first word's on bit 7 of
            // each byte, the second's on bit 6
            rw[2 * g] = keep_flags2(keep_flags(r.x, cdrop), keep_flags(r.y, cdrop));
            rw[2 * g + 1] = keep_flags2(keep_flags(r.z, cdrop), keep_flags(r.w, cdrop));
          }
        }
        if (!(ok = warp_wait(bar(C::B_SFULL + t), sph, wctx))) break;
        sph ^= 1u;
        tc_fence_after();
        const int key0 = (kt0 + j) * BN;
        const bool need_mask = (key0 + BN > p.Nkv) || (p.causal && key0 + BN - 1 > q0 + delta);
        const int key_lim = p.causal ? min(row + delta, p.Nkv - 1) : p.Nkv - 1;   // last visible key
        // The whole 128-column S row in registers: one TMEM load per tile.
        float v[BN];
        tmem_ld128(tS, v);
        if (need_mask) {
#pragma unroll
          for (int i = 0; i < BN; ++i)
            if (key0 + i > key_lim) v[i] = -INFINITY;
        }
        // Row maximum: eight independent three-input max chains, then merge.
        float mx8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = fmaxf(v[2 * a], v[2 * a + 1]);
#pragma unroll
        for (int i = 8; i < BN / 2; ++i) mx8[i & 7] = fmax3(mx8[i & 7], v[2 * i], v[2 * i + 1]);
        const float mx = fmaxf(fmax3(fmax3(mx8[0], mx8[1], mx8[2]), mx8[3], mx8[4]),
                               fmax3(mx8[5], mx8[6], mx8[7]));
        const float m_new = (mx == -INFINITY) ? -INFINITY : mx * sl2;
        float alpha = 1.f;
        const bool grow = m_new > m_used + kRescaleThreshold;
        if (grow) {
          alpha = ex2(m_used - m_new);
          m_used = m_new;
        }
        l *= alpha;
        if (j > 0 && __any_sync(kFull, grow)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(tO + c * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tO + c * 32, o);
          }
        }
        const float base = (m_used == -INFINITY) ? 0.f : m_used;
        // P = 2^(s * scale * log2 e - m): the argument with paired FMAs, the
        // exponential on the SFU, the row sum in four paired accumulators,
        // P as bf16 pairs written over S.  Masked keys need no second test
        // here: their logit is -inf and ex2(-inf) = 0.  The one exception is
        // scale 0 (0 * -inf): then the visible logits become 0 with a unit
        // factor.  The loop itself carries no mask code, so the compiler
        // emits nothing per element for it.
        float csl = sl2;
        if (need_mask && sl2 == 0.f) {
#pragma unroll
          for (int i = 0; i < BN; ++i) v[i] = (v[i] == -INFINITY) ? -INFINITY : 0.f;
          csl = 1.f;
        }
        const uint64_t c2 = f2_pack(csl, csl);
        const uint64_t nb2 = f2_pack(-base, -base);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        // P in two halves: keys 0..63 are published first, so the MMA warp
        // can start P V on them while keys 64..127 are computed.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[BN / 4];
#pragma unroll
          for (int i = 0; i < BN / 4; ++i) {
            const int e = h * (BN / 4) + i;
            const uint64_t x = f2_fma(f2_pack(v[2 * e], v[2 * e + 1]), c2, nb2);
            // ex2_fma2 gives 2^-125 rather than 0 for -inf, so masked tiles
            // (where a row may see no key at all) keep every exponential on the SFU
            uint64_t pp;
            if (SPLIT > 0 && !need_mask && i % (SPLIT > 0 ? SPLIT : 1) == SPLIT - 1) {
              pp = ex2_fma2(x);
            } else {
              pp = f2_pack(ex2(f2_lo(x)), ex2(f2_hi(x)));
            }
            acc[i & 3] = f2_add(acc[i & 3], pp);
            pk[i] = pack_bf16x2(f2_lo(pp), f2_hi(pp));
          }
          if constexpr (DROP) {
            // dropout after the row sum: the normaliser counts every key,
            // P V sees only the kept ones
#pragma unroll
            for (int q = 0; q < BN / 16; ++q) {
              const uint32_t fa = rw[h * (BN / 16) + q];
              uint32_t m01, m23;
              keep_pair_masks(fa, m01, m23);
              pk[4 * q] &= m01;
              pk[4 * q + 1] &= m23;
              keep_pair_masks(fa << 1, m01, m23);
              pk[4 * q + 2] &= m01;
              pk[4 * q + 3] &= m23;
            }
          }
          tmem_st32u(tS + h * (BN / 4), pk);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(h == 0 ? C::B_PHALF + t : C::B_PFULL + t));
        }
        const uint64_t a01 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
        l += f2_lo(a01) + f2_hi(a01);
      }
      if (!ok) break;
      // epilogue: O / l and LSE, then hand O_t back to the MMA warp
      if (!(ok = warp_wait(bar(C::B_OFULL + t), ofph, wctx))) break;
      ofph ^= 1u;
      tc_fence_after();
      const bool live = row < p.Nq;
      if constexpr (KSPLIT) {
        if (ksplit) {
          if (!(ok = merge_epilogue<D, DROP>(p, U, t, quad, lane, row_in_tile, m_used, l, tm,
                                             reinterpret_cast<float2*>(smem + C::OFF_MRG), bar(C::B_MERGE), mph,
                                             wctx)))
            break;
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::B_OEMPTY + t));
          continue;
        }
      }
      const float inv_l = (l > 0.f) ? (DROP ? p.drop_scale : 1.f) / l : 0.f;
      // O leaves TMEM in the 16x256b shape: each store instruction of the
      // warp then writes 8 rows x 32 contiguous bytes (whole sectors),
      // instead of 32 rows x 16 bytes with one row per thread.
      // fp32 O, or bf16 O when the call asked for it (p.o_bf16)
      const long long ohead = U.b * p.o_sb + U.h * p.o_sh;
      const bool bf = p.o_bf16 != nullptr;
#pragma unroll 1
      for (int hl = 0; hl < 2; ++hl) {
        const int ra = static_cast<int>(quad * 32 + hl * 16 + (lane >> 2));   // rows ra and ra + 8 of the tile
        const float ia = __shfl_sync(kFull, inv_l, hl * 16 + (lane >> 2));
        const float ib = __shfl_sync(kFull, inv_l, hl * 16 + (lane >> 2) + 8);
        const bool la = q0 + ra < p.Nq, lb = q0 + ra + 8 < p.Nq;
        const long long oa = ohead + (la ? q0 + ra : 0) * p.o_sr + 2 * (lane & 3);
        const long long ob = ohead + (lb ? q0 + ra + 8 : 0) * p.o_sr + 2 * (lane & 3);
#pragma unroll 1
        for (int ch = 0; ch < D / 64; ++ch) {
          uint32_t r[32];
          if (n > 0) {
            tmem_ld16x256b_x8(tm + ((quad * 32u + hl * 16u) << 16) + C::col_o(t) + ch * 64, r);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float a0 = __uint_as_float(r[4 * k]) * ia, a1 = __uint_as_float(r[4 * k + 1]) * ia;
            const float b0 = __uint_as_float(r[4 * k + 2]) * ib, b1 = __uint_as_float(r[4 * k + 3]) * ib;
            const int c = ch * 64 + 8 * k;
            if (bf) {
              if (la) *reinterpret_cast<uint32_t*>(p.o_bf16 + oa + c) = pack_bf16x2(a0, a1);
              if (lb) *reinterpret_cast<uint32_t*>(p.o_bf16 + ob + c) = pack_bf16x2(b0, b1);
            } else {
              if (la) *reinterpret_cast<float2*>(p.o + oa + c) = make_float2(a0, a1);
              if (lb) *reinterpret_cast<float2*>(p.o + ob + c) = make_float2(b0, b1);
            }
          }
        }
      }
      if (live && p.lse != nullptr) {
        const float lse = (l > 0.f) ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        p.lse[static_cast<size_t>(U.b * p.Hq + U.h) * p.Nq + row] = lse;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_OEMPTY + t));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp0) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

template <int D, bool DROP, int SPLIT, bool KSPLIT = false>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                     int num_sms, cudaStream_t stream) {
  using C = Cfg<D>;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, DROP, SPLIT, KSPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM_BYTES));
  if (e != cudaSuccess) return e;
  const int grid = min(p.num_units, num_sms);
  if (grid <= 0) return cudaSuccess;
  // The register split needs the kernel to be launched with enough registers;
  // otherwise setmaxnreg.inc could never be served, so refuse to launch.
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, prefill_kernel<D, DROP, SPLIT, KSPLIT>)) != cudaSuccess) return e;
  if (((fa.numRegs + 7) / 8) * 8 < kRegsNeededAtLaunch) return cudaErrorInvalidConfiguration;
  prefill_kernel<D, DROP, SPLIT, KSPLIT><<<grid, kThreads, C::SMEM_BYTES, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int num_sms, cudaStream_t stream) {
  const bool drop = p.drop_t != 0u;
  if (d == 64 && p.kv_split) {
    if (drop) return launch_d<64, true, 0, true>(tq, tk, tv, p, num_sms, stream);
    switch (p.exp2_split) {
      case 0: return launch_d<64, false, 0, true>(tq, tk, tv, p, num_sms, stream);
      case 4: return launch_d<64, false, 4, true>(tq, tk, tv, p, num_sms, stream);
      case 8: return launch_d<64, false, 8, true>(tq, tk, tv, p, num_sms, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (p.kv_split) return cudaErrorInvalidValue;   // key-split units exist at d = 64 only
  if (drop) {
    if (d == 64) return launch_d<64, true, 0>(tq, tk, tv, p, num_sms, stream);
    if (d == 128) return launch_d<128, true, 0>(tq, tk, tv, p, num_sms, stream);
    return cudaErrorInvalidValue;
  }
  switch (d * 100 + p.exp2_split) {
    case 6400: return launch_d<64, false, 0>(tq, tk, tv, p, num_sms, stream);
    case 6404: return launch_d<64, false, 4>(tq, tk, tv, p, num_sms, stream);
    case 6408: return launch_d<64, false, 8>(tq, tk, tv, p, num_sms, stream);
    case 12800: return launch_d<128, false, 0>(tq, tk, tv, p, num_sms, stream);
    case 12804: return launch_d<128, false, 4>(tq, tk, tv, p, num_sms, stream);
    case 12808: return launch_d<128, false, 8>(tq, tk, tv, p, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gbattn
