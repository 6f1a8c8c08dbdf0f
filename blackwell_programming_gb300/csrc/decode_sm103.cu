// decode_sm103.cu - attention for the latent head-dim shape (d_qk = 576,
// d_v = 512, V = the first 512 features of K): the split-KV decode with the
// combine kernel that merges its splits, and the prefill (causal or not,
// Nq > 1) that runs the same kernel on blocks of 128 query rows.
//
// The shape is the DeepSeek MLA case of "Distilling a 4.5 hour CUDA talk",
// sections 12-13: Q/K are 576 wide and V/O are the first 512 features.  That
// page repartitions the work along the head dimension; here the repartition
// is chosen for tensor memory (TMEM, 512 columns of 32 bits per lane): a full
// 128 x 512 fp32 O accumulator would fill all of TMEM and leave no room for
// the scores, so every work item computes the whole score tile S = Q K^T but
// only one 256-column half of O.  Nq = 1, so the Hq / Hkv query heads that
// share a KV head become the 128 rows (TMEM lanes) of the tile.
//
// Parallel split ("stream-K" style): the (half, sequence, key-tile) space is
// cut into gridDim.x contiguous equal ranges, one per persistent CTA, so every
// SM gets the same number of K tiles whatever the batch size (no wave
// quantisation, "Distilling..." section 5 and the bootcamp talks' 133-block
// example).  A range that ends inside a (sequence, half) produces a partial
// (normalised O over its keys, and its LSE) in its own slot of the workspace;
// partials of different CTAs never share a slot, so there are no races
// (section 5's rule that disjoint outputs need no atomics).  The combine
// kernel then merges the partials of each row:
//   LSE = log sum_s exp(lse_s),   O = sum_s exp(lse_s - LSE) O_s.
//
// Prefill mode: a work item is (value half, batch, query head, block of 128
// query rows) and covers every K tile the block sees (all of them, or up to
// the causal diagonal with bottom-right alignment), so it writes O and LSE
// directly.  Items are handed out longest first (query blocks from the
// bottom), the two halves of a block and the heads that share a KV head
// side by side so that their K tiles come from L2.
//
// Roles: warp 5 = TMA producer (the shared-memory part of Q once per
// segment, K tiles through two rings), warp 4 = tcgen05 MMA issuer (whole
// warp, one elected lane per instruction), warps 0-3 = the TMEM part of Q,
// softmax (one row per thread), O rescale and epilogue.
//
// Copies are few and large: each TMA copy costs its issuing thread a few
// hundred cycles of round trip, so the tensor maps see a [planes, rows, 576]
// tensor as (64 features, rows, 9 chunks, planes) (the 128-byte chunk stride
// inside the 1152-byte row stride) and one box of r rows x c chunks lands as c
// consecutive r x 128-byte chunk images with the 128-byte swizzle, the layout
// the MMA descriptors read.  A K tile then takes two or three copies instead
// of nine.
#include <cmath>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int DQK = 576;
constexpr int DVH = 256;              // O columns per work item (half of d_v)
constexpr int BM = 128;               // rows = query heads of one KV head
constexpr int BN = 64;                // keys per K tile
constexpr int QCH = DQK / 64;         // 9 chunks of 64 features (128 bytes)
constexpr int Q_TMEM_FEATS = 384;     // Q features 0..383 live in TMEM, 384..575 in shared memory
constexpr int Q_SMEM_CH = (DQK - Q_TMEM_FEATS) / 64;   // 3 chunks
constexpr int A_CH = 5;               // K chunks outside this item's value half
constexpr int B_CH = 4;               // K chunks of this item's value half (= V)
constexpr int AS = 2;                 // ring A stages (released after Q K^T)
constexpr int BS = 3;                 // ring B stages (released after P V)
constexpr int kThreads = 192;
constexpr int kMmaWarp = 4;
constexpr int kTmaWarp = 5;
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kFull = 0xFFFFFFFFu;

constexpr uint32_t CHUNK_Q = BM * 128;              // 16 KB
constexpr uint32_t CHUNK_K = BN * 128;              // 8 KB
constexpr uint32_t QS_BYTES = Q_SMEM_CH * CHUNK_Q;  // 48 KB
constexpr uint32_t A_BYTES = A_CH * CHUNK_K;        // 40 KB
constexpr uint32_t B_BYTES = B_CH * CHUNK_K;        // 32 KB
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_A = OFF_Q + QS_BYTES;
constexpr uint32_t OFF_B = OFF_A + AS * A_BYTES;
constexpr uint32_t OFF_BAR = OFF_B + BS * B_BYTES;
constexpr int B_QFULL = 0, B_QEMPTY = 1, B_QTFULL = 2, B_AFULL = 3, B_AEMPTY = B_AFULL + AS, B_BFULL = B_AEMPTY + AS,
              B_BEMPTY = B_BFULL + BS, B_SFULL = B_BEMPTY + BS, B_PFULL = B_SFULL + 1, B_PHALF = B_PFULL + 1, B_OFULL = B_PHALF + 1,
              B_OEMPTY = B_OFULL + 1, B_DRAIN = B_OEMPTY + 1, NUM_BARS = B_DRAIN + 1;
constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(Q_SMEM_CH == kLatentQChunks && BN == kLatentKeyRows && A_CH == B_CH + 1 && QCH == 2 * B_CH + 1,
              "box shapes shared with the host");

// TMEM: O half [0,256), S [256,320) (P as bf16 pairs in its first 32
// columns), Q features 0..383 as bf16 pairs [320,512).
constexpr uint32_t COL_O = 0;
constexpr uint32_t COL_S = 256;
constexpr uint32_t COL_Q = 320;
constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, DVH, false, true);

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(kFull, ok);
}

// The (half, plane, key-tile) space is numbered g = (half * planes + plane) *
// tiles + tile and cut into gridDim.x equal contiguous ranges.
__host__ __device__ __forceinline__ long long range_begin(long long total, int c, int grid) {
  return total * c / grid;
}

// One contiguous run of K tiles of one (half, plane) inside a CTA's range.
struct Segment {
  int plane, half;
  int t0, n;    // first tile, tile count
  int slot;     // partial slot within this CTA (decode)
  int kplane;   // K plane (batch * Hkv + KV head)
  int qplane;   // plane of the Q map: decode = KV plane (rows = heads), prefill = batch * Hq + head
  int qrow0;    // first query row of the tile in that plane
};

struct SegmentWalker {
  long long g, g0, g1, tiles;
  int planes;
  __device__ SegmentWalker(const DecodeParams& p) {
    const long long total = 2LL * p.planes * p.tiles;
    g0 = range_begin(total, blockIdx.x, gridDim.x);
    g1 = range_begin(total, blockIdx.x + 1, gridDim.x);
    g = g0;
    tiles = p.tiles;
    planes = p.planes;
  }
  __device__ bool next(Segment& s) {
    if (g >= g1) return false;
    const long long sg = g / tiles;
    s.half = static_cast<int>(sg / planes);
    s.plane = static_cast<int>(sg - static_cast<long long>(s.half) * planes);
    s.t0 = static_cast<int>(g - sg * tiles);
    const long long end = min(g1, (sg + 1) * tiles);
    s.n = static_cast<int>(end - g);
    s.slot = static_cast<int>(sg - g0 / tiles);
    s.kplane = s.qplane = s.plane;
    s.qrow0 = 0;
    g = end;
    return true;
  }
};

// Prefill mode: unit u = ((query block from the bottom) * B * Hq + batch *
// Hq + head) * 2 + half, handed to the persistent CTAs in rounds of
// gridDim.x with every other round reversed (snake), so each CTA gets a
// similar mix of long and short blocks.
struct UnitWalker {
  const LatentPrefillParams& p;
  int it = 0;
  __device__ UnitWalker(const LatentPrefillParams& prm) : p(prm) {}
  __device__ bool next(Segment& s) {
    const int base = it * static_cast<int>(gridDim.x);
    const int u = (it & 1) ? base + static_cast<int>(gridDim.x - 1 - blockIdx.x) : base + static_cast<int>(blockIdx.x);
    ++it;
    if (u >= p.num_units) return false;
    const int bh_count = p.B * p.Hq;
    s.half = u & 1;
    const int rest = u >> 1;
    const int qb = p.nqb - 1 - rest / bh_count;
    const int bh = rest - (rest / bh_count) * bh_count;
    const int b = bh / p.Hq, h = bh - b * p.Hq;
    s.qplane = bh;
    s.kplane = b * p.Hkv + h / (p.Hq / p.Hkv);
    s.plane = s.kplane;
    s.qrow0 = qb * BM;
    s.t0 = 0;
    s.slot = 0;
    int n = p.tiles;
    if (p.causal) {
      const int last_key = min(s.qrow0 + BM - 1, p.Nq - 1) + (p.Nkv - p.Nq);
      n = last_key < 0 ? 0 : min(last_key / BN + 1, p.tiles);
    }
    s.n = n;
    return true;
  }
};

template <class P> struct WalkerFor;
template <> struct WalkerFor<DecodeParams> { using type = SegmentWalker; };
template <> struct WalkerFor<LatentPrefillParams> { using type = UnitWalker; };

// Row r of a tile's Q: its global address, and whether it exists.
__device__ __forceinline__ const uint16_t* q_row(const DecodeParams& p, const Segment& s, int r) {
  return p.q + (static_cast<size_t>(s.qplane) * p.group + r) * DQK;
}
__device__ __forceinline__ bool q_live(const DecodeParams& p, const Segment&, int r) { return r < p.group; }
__device__ __forceinline__ const uint16_t* q_row(const LatentPrefillParams& p, const Segment& s, int r) {
  return p.q + (static_cast<size_t>(s.qplane) * p.Nq + s.qrow0 + r) * DQK;
}
__device__ __forceinline__ bool q_live(const LatentPrefillParams& p, const Segment& s, int r) {
  return s.qrow0 + r < p.Nq;
}

// K chunk c (features 64c .. 64c+63) of a tile lives in ring B when it belongs
// to the item's value half (chunks 4*half .. 4*half+3), else in ring A.
__device__ __forceinline__ bool in_ring_b(int c, int half) { return c >= 4 * half && c < 4 * half + 4; }
__device__ __forceinline__ int a_index(int c, int half) { return c < 4 * half ? c : c - 4; }

// Why this layout: an MMA whose A operand comes from shared memory pays
// about 32 cycles for the A read whatever N is, so a 64-key score tile
// (N = 64) runs at two thirds of the tensor rate with A in shared memory and
// at full rate with A in TMEM.  Two thirds of Q therefore sits in TMEM.
// The 576-feature K tile is split into the five chunks the item needs only
// for Q K^T (ring A, freed as soon as S is computed) and the four chunks that
// are also its V half (ring B, freed after P V), so the shared memory left
// beside Q's last third holds enough tiles in flight to cover the memory
// latency.
template <class P>
__global__ void __launch_bounds__(kThreads, 1)
    latent_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK5,
                  const __grid_constant__ CUtensorMap tmK4, const __grid_constant__ CUtensorMap tmK1, const P p) {
  constexpr bool kPrefill = std::is_same<P, LatentPrefillParams>::value;
  using Walker = typename WalkerFor<P>::type;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + OFF_Q, sA = sbase + OFF_A, sB = sbase + OFF_B;
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC + 4);
  const WaitCtx wctx{abort_flag, p.err};
  const uint32_t warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    mbar_init(bar(B_QTFULL), 4);
    for (int s = 0; s < AS; ++s) {
      mbar_init(bar(B_AFULL + s), 1);
      mbar_init(bar(B_AEMPTY + s), 1);
    }
    for (int s = 0; s < BS; ++s) {
      mbar_init(bar(B_BFULL + s), 1);
      mbar_init(bar(B_BEMPTY + s), 1);
    }
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_PFULL), 4);
    mbar_init(bar(B_PHALF), 4);
    mbar_init(bar(B_OFULL), 1);
    mbar_init(bar(B_OEMPTY), 4);
    mbar_init(bar(B_DRAIN), 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK5);
      tma_prefetch_desc(&tmK4);
      tma_prefetch_desc(&tmK1);
      // decode: each K tile is read by the two halves, then dead; prefill: K
      // is read again by every query head of its KV head and every block
      const uint64_t pol_k = kPrefill ? l2_policy_evict_last() : l2_policy_evict_first();
      const uint64_t pol_q = l2_policy_evict_last();
      int as = 0, bs = 0;
      uint32_t aph = 0, bph = 0, qph = 0;
      // buffers filled (bit) and the parity of their last fill, for the drain
      uint32_t filled = 0u, fill_par = 0u;
      auto note_fill = [&](int b, uint32_t par) {
        filled |= 1u << b;
        fill_par = (fill_par & ~(1u << b)) | (par << b);
      };
      Walker walk(p);
      Segment S;
      bool ok = true;
      while (ok && walk.next(S)) {
        if (S.n == 0) continue;   // a prefill block that sees no key: the softmax warps write it
        if (!(ok = mbar_wait(bar(B_QEMPTY), qph ^ 1u, wctx))) break;
        qph ^= 1u;
        mbar_arrive_expect_tx(bar(B_QFULL), QS_BYTES);
        note_fill(0, qph ^ 1u);
        tma_load_4d(sQ, &tmQ, bar(B_QFULL), 0, S.qrow0, Q_TMEM_FEATS / 64, S.qplane, pol_q);
        for (int j = 0; j < S.n; ++j) {
          const int y = (S.t0 + j) * BN;
          if (!(ok = mbar_wait(bar(B_AEMPTY + as), aph ^ 1u, wctx))) break;
          mbar_arrive_expect_tx(bar(B_AFULL + as), A_BYTES);
          note_fill(1 + as, aph);
          // ring A: the five chunks outside this item's value half (4..8 for
          // half 0; 0..3 and 8 for half 1), in chunk order
          if (S.half == 0) {
            tma_load_4d(sA + as * A_BYTES, &tmK5, bar(B_AFULL + as), 0, y, B_CH, S.kplane, pol_k);
          } else {
            tma_load_4d(sA + as * A_BYTES, &tmK4, bar(B_AFULL + as), 0, y, 0, S.kplane, pol_k);
            tma_load_4d(sA + as * A_BYTES + B_CH * CHUNK_K, &tmK1, bar(B_AFULL + as), 0, y, 2 * B_CH, S.kplane,
                        pol_k);
          }
          if (++as == AS) { as = 0; aph ^= 1u; }
          if (!(ok = mbar_wait(bar(B_BEMPTY + bs), bph ^ 1u, wctx))) break;
          mbar_arrive_expect_tx(bar(B_BFULL + bs), B_BYTES);
          note_fill(1 + AS + bs, bph);
          tma_load_4d(sB + bs * B_BYTES, &tmK4, bar(B_BFULL + bs), 0, y, B_CH * S.half, S.kplane, pol_k);
          if (++bs == BS) { bs = 0; bph ^= 1u; }
        }
      }
      // Every issued copy must have landed before the CTA may exit.
      for (int b = 0; b < 1 + AS + BS; ++b) {
        if (!((filled >> b) & 1u)) continue;
        const int full = b == 0 ? B_QFULL : (b < 1 + AS ? B_AFULL + (b - 1) : B_BFULL + (b - 1 - AS));
        mbar_wait_drain(bar(full), (fill_par >> b) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issuer (whole warp)
    int as = 0, bs = 0;
    uint32_t aph = 0, bph = 0, qph = 0, qtph = 0, pph = 0, oeph = 0;
    const uint64_t qs_desc = smem_desc_sw128(sQ, 16, 1024);
    const uint64_t a_desc0 = smem_desc_sw128(sA, 16, 1024);
    const uint64_t b_desc0 = smem_desc_sw128(sB, 16, 1024);
    const uint64_t v_desc0 = smem_desc_sw128(sB, CHUNK_K, 1024);
    const uint32_t dS = tm + COL_S, dO = tm + COL_O, aQ = tm + COL_Q;
    Walker walk(p);
    Segment S;
    bool ok = true;
    while (ok && walk.next(S)) {
      if (S.n == 0) continue;
      if (!(ok = warp_wait(bar(B_QFULL), qph, wctx))) break;
      qph ^= 1u;
      if (!(ok = warp_wait(bar(B_QTFULL), qtph, wctx))) break;
      qtph ^= 1u;
      tc_fence_after();
      for (int j = 0; j < S.n && ok; ++j) {
        if (!(ok = warp_wait(bar(B_AFULL + as), aph, wctx))) break;
        if (!(ok = warp_wait(bar(B_BFULL + bs), bph, wctx))) break;
        // S = Q K^T over 36 K steps of 16 features
        const uint64_t ad = a_desc0 + ((as * A_BYTES) >> 4);
        const uint64_t bd = b_desc0 + ((bs * B_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const int c = kk >> 2;
          const uint32_t in_chunk = ((kk & 3) * 32) >> 4;
          const uint64_t kdesc = in_ring_b(c, S.half) ? bd + (((c - 4 * S.half) * CHUNK_K) >> 4) + in_chunk
                                                        : ad + ((a_index(c, S.half) * CHUNK_K) >> 4) + in_chunk;
          if (kk < Q_TMEM_FEATS / 16) {
            mma_ts_warp(dS, aQ + kk * 8, kdesc, IDESC_S, kk > 0 ? 1u : 0u);
          } else {
            const uint64_t qd = qs_desc + (((c - Q_TMEM_FEATS / 64) * CHUNK_Q) >> 4) + in_chunk;
            mma_ss_warp(dS, qd, kdesc, IDESC_S, 1u);
          }
        }
        mma_commit_warp(bar(B_SFULL));
        mma_commit_warp(bar(B_AEMPTY + as));
        if (++as == AS) { as = 0; aph ^= 1u; }
        if (j == S.n - 1) mma_commit_warp(bar(B_QEMPTY));
        // O += P V: P (64 keys, bf16 pairs) from TMEM over S, V = ring B;
        // keys 0..31 as soon as their P is in TMEM, keys 32..63 after
        if (j == 0) {
          // the previous segment's epilogue must have read O
          if (!(ok = warp_wait(bar(B_OEMPTY), oeph ^ 1u, wctx))) break;
          oeph ^= 1u;
        }
        if (!(ok = warp_wait(bar(B_PHALF), pph, wctx))) break;
        tc_fence_after();
        const uint64_t vd = v_desc0 + ((bs * B_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < BN / 32; ++kk)
          mma_ts_warp(dO, dS + kk * 8, vd + ((kk * 16 * 128) >> 4), IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
        if (!(ok = warp_wait(bar(B_PFULL), pph, wctx))) break;
        pph ^= 1u;
        tc_fence_after();
#pragma unroll
        for (int kk = BN / 32; kk < BN / 16; ++kk)
          mma_ts_warp(dO, dS + kk * 8, vd + ((kk * 16 * 128) >> 4), IDESC_PV, 1u);
        mma_commit_warp(bar(B_BEMPTY + bs));
        if (++bs == BS) { bs = 0; bph ^= 1u; }
      }
      if (!ok) break;
      mma_commit_warp(bar(B_OFULL));
    }
    mma_commit_warp(bar(B_DRAIN));
    mbar_wait_drain(bar(B_DRAIN), 0);
    __syncwarp();
  } else if (warp < 4) {
    // ----------------------------- Q into TMEM, softmax, rescale, epilogue
    const int r = static_cast<int>(warp * 32 + lane);
    const uint32_t lane_addr = (warp * 32u) << 16;
    const float sl2 = p.scale_log2;
    uint32_t sph = 0, ofph = 0, qeph = 0;
    // Q features 0..383 of row r into TMEM (bf16 pairs, column COL_Q + c
    // holds features 2c, 2c+1), once the previous segment's last Q K^T has
    // finished: two rounds of 24 loads of 16 bytes in flight.
    auto load_q = [&](const Segment& s) -> bool {
      if (!warp_wait(bar(B_QEMPTY), qeph ^ 1u, wctx)) return false;
      qeph ^= 1u;
      tc_fence_after();
      const bool live = q_live(p, s, r);
      const uint4* qrow = reinterpret_cast<const uint4*>(q_row(p, s, live ? r : 0));
#pragma unroll 1
      for (int b = 0; b < 2; ++b) {
        uint32_t w[3][32];
#pragma unroll
        for (int i = 0; i < 24; ++i) {
          const uint4 x = live ? qrow[b * 24 + i] : make_uint4(0u, 0u, 0u, 0u);
          w[i >> 3][4 * (i & 7)] = x.x;
          w[i >> 3][4 * (i & 7) + 1] = x.y;
          w[i >> 3][4 * (i & 7) + 2] = x.z;
          w[i >> 3][4 * (i & 7) + 3] = x.w;
        }
#pragma unroll
        for (int t = 0; t < 3; ++t) tmem_st32u(tm + lane_addr + COL_Q + (b * 3 + t) * 32, w[t]);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QTFULL));
      return true;
    };
    Walker walk(p);
    // The next work item with at least one K tile.  A prefill block that
    // sees no key (causal, Nq > Nkv) gets O = 0 and LSE = -inf here.
    auto advance = [&](Segment& s) -> bool {
      while (walk.next(s)) {
        if (s.n > 0) return true;
        if constexpr (kPrefill) {
          if (q_live(p, s, r)) {
            const size_t orow = (static_cast<size_t>(s.qplane) * p.Nq + s.qrow0 + r) * (2 * DVH) + s.half * DVH;
            if (p.o_bf16 != nullptr) {
#pragma unroll 4
              for (int c = 0; c < DVH / 8; ++c) reinterpret_cast<uint4*>(p.o_bf16 + orow)[c] = make_uint4(0u, 0u, 0u, 0u);
            } else {
#pragma unroll 4
              for (int c = 0; c < DVH / 4; ++c) reinterpret_cast<float4*>(p.o + orow)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (s.half == 0 && p.lse != nullptr) p.lse[static_cast<size_t>(s.qplane) * p.Nq + s.qrow0 + r] = -INFINITY;
          }
        }
      }
      return false;
    };
    Segment S, Snext;
    bool have = advance(S);
    bool ok = true;
    if (have) ok = load_q(S);
    while (ok && have) {
      float m_used = -INFINITY, l = 0.f;
      // Last key row r may see: all of them, or up to the causal diagonal
      // (bottom-right alignment); the tile needs the mask when its last key
      // is past the limit of its first row.
      int key_lim = p.Nkv - 1, causal_lim0 = p.Nkv - 1;
      if constexpr (kPrefill) {
        if (p.causal) {
          key_lim = min(S.qrow0 + r + (p.Nkv - p.Nq), p.Nkv - 1);
          causal_lim0 = S.qrow0 + (p.Nkv - p.Nq);
        }
      }
      for (int j = 0; j < S.n; ++j) {
        if (!(ok = warp_wait(bar(B_SFULL), sph, wctx))) break;
        sph ^= 1u;
        tc_fence_after();
        float v[BN];
        tmem_ld64(tm + lane_addr + COL_S, v);
        const int key0 = (S.t0 + j) * BN;
        const bool ragged = key0 + BN - 1 > causal_lim0;
        if (ragged) {
#pragma unroll
          for (int i = 0; i < BN; ++i)
            if (key0 + i > key_lim) v[i] = -INFINITY;
        }
        float mx8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = fmaxf(v[2 * a], v[2 * a + 1]);
#pragma unroll
        for (int i = 8; i < BN / 2; ++i) mx8[i & 7] = fmax3(mx8[i & 7], v[2 * i], v[2 * i + 1]);
        const float mx = fmaxf(fmax3(fmax3(mx8[0], mx8[1], mx8[2]), mx8[3], mx8[4]), fmax3(mx8[5], mx8[6], mx8[7]));
        const float m_new = (mx == -INFINITY) ? -INFINITY : mx * sl2;
        float alpha = 1.f;
        const bool grow = m_new > m_used + kRescaleThreshold;
        if (grow) {
          alpha = ex2(m_used - m_new);
          m_used = m_new;
        }
        l *= alpha;
        // O is stable here: this tile's S was issued after the previous P V.
        if (j >= 1 && __any_sync(kFull, grow)) {
#pragma unroll 1
          for (int c = 0; c < DVH / 32; ++c) {
            float o[32];
            tmem_ld32(tm + lane_addr + COL_O + c * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tm + lane_addr + COL_O + c * 32, o);
          }
        }
        const float base = (m_used == -INFINITY) ? 0.f : m_used;
        // Keys past Nkv are -inf and ex2(-inf) = 0, so the exp2 loop needs no
        // mask; only scale 0 (0 * -inf) needs the visible logits set to 0
        // with a unit factor.
        float csl = sl2;
        if (ragged && sl2 == 0.f) {
#pragma unroll
          for (int i = 0; i < BN; ++i) v[i] = (v[i] == -INFINITY) ? -INFINITY : 0.f;
          csl = 1.f;
        }
        const uint64_t c2 = f2_pack(csl, csl);
        const uint64_t nb2 = f2_pack(-base, -base);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        // P in two halves: keys 0..31 are published first, so the MMA warp
        // starts P V on them while keys 32..63 are computed.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[BN / 4];
#pragma unroll
          for (int i = 0; i < BN / 4; ++i) {
            const int e = h * (BN / 4) + i;
            const uint64_t x = f2_fma(f2_pack(v[2 * e], v[2 * e + 1]), c2, nb2);
            const float p0 = ex2(f2_lo(x));
            const float p1 = ex2(f2_hi(x));
            acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tm + lane_addr + COL_S + h * (BN / 4), pk);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(h == 0 ? B_PHALF : B_PFULL));
        }
        const uint64_t a01 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
        l += f2_lo(a01) + f2_hi(a01);
      }
      if (!ok) break;
      // The next segment's Q first, so that its first Q K^T overlaps this
      // segment's epilogue.
      have = advance(Snext);
      if (have && !(ok = load_q(Snext))) break;
      if (!(ok = warp_wait(bar(B_OFULL), ofph, wctx))) break;
      ofph ^= 1u;
      tc_fence_after();
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const float lse_r = (l > 0.f) ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      if constexpr (kPrefill) {
        // O half of rows qrow0 .. qrow0+127, straight to the output.  O
        // leaves TMEM in the 16x256b shape, so each warp store writes 8 rows
        // x 32 contiguous bytes.
        const size_t ohead = (static_cast<size_t>(S.qplane) * p.Nq) * (2 * DVH) + S.half * DVH;
        const bool bf = p.o_bf16 != nullptr;
#pragma unroll 1
        for (int hl = 0; hl < 2; ++hl) {
          const int ra = static_cast<int>(warp * 32 + hl * 16 + (lane >> 2));   // rows ra and ra + 8 of the tile
          const float ia = __shfl_sync(kFull, inv_l, hl * 16 + (lane >> 2));
          const float ib = __shfl_sync(kFull, inv_l, hl * 16 + (lane >> 2) + 8);
          const bool la = S.qrow0 + ra < p.Nq, lb = S.qrow0 + ra + 8 < p.Nq;
          const size_t oa = ohead + static_cast<size_t>(la ? S.qrow0 + ra : 0) * (2 * DVH) + 2 * (lane & 3);
          const size_t ob = ohead + static_cast<size_t>(lb ? S.qrow0 + ra + 8 : 0) * (2 * DVH) + 2 * (lane & 3);
#pragma unroll 1
          for (int ch = 0; ch < DVH / 64; ++ch) {
            uint32_t rr[32];
            tmem_ld16x256b_x8(tm + ((warp * 32u + hl * 16u) << 16) + COL_O + ch * 64, rr);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float a0 = __uint_as_float(rr[4 * k]) * ia, a1 = __uint_as_float(rr[4 * k + 1]) * ia;
              const float b0 = __uint_as_float(rr[4 * k + 2]) * ib, b1 = __uint_as_float(rr[4 * k + 3]) * ib;
              const size_t c = static_cast<size_t>(ch * 64 + 8 * k);
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
        if (S.half == 0 && p.lse != nullptr && q_live(p, S, r))
          p.lse[static_cast<size_t>(S.qplane) * p.Nq + S.qrow0 + r] = lse_r;
      } else {
        // Partial O, normalised, in a layout where the float4 of row r and
        // columns 4c..4c+3 sits at [slot][c][r]: a warp's 32 rows store 512
        // contiguous bytes at a time.
        const bool live = q_live(p, S, r);
        const size_t slot = static_cast<size_t>(blockIdx.x) * p.max_seg + S.slot;
        float4* opart = reinterpret_cast<float4*>(p.o_part) + slot * (DVH / 4) * BM + r;
#pragma unroll 1
        for (int c = 0; c < DVH / 32; ++c) {
          float o[32];
          tmem_ld32(tm + lane_addr + COL_O + c * 32, o);
          if (live) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              opart[static_cast<size_t>(c * 8 + i) * BM] =
                  make_float4(o[4 * i] * inv_l, o[4 * i + 1] * inv_l, o[4 * i + 2] * inv_l, o[4 * i + 3] * inv_l);
          }
        }
        if (live) p.lse_part[slot * BM + r] = lse_r;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_OEMPTY));
      S = Snext;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

// Combine: one warp per (value half, plane, 32 output rows, 32 output
// columns), one lane per row.  A lane reduces its row's partial LSEs (a few
// per row) and merges its row's 32 columns: float4 reads of the partials
// that are coalesced across the lanes (their rows are adjacent in the partial
// layout), a transpose through shared memory, and one 128-byte store per
// row.  `grid` is the decode kernel's grid size, which fixes where the
// partials are.
constexpr int kCombineWarps = 4;
constexpr int kCombineMaxSlots = 4;   // partials per (half, sequence) handled in registers
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const DecodeParams p, int grid, float* o,
                                                                     uint16_t* o_bf16, float* lse) {
  __shared__ float tile[kCombineWarps][32][33];
  const int wib = static_cast<int>(threadIdx.x >> 5);
  const int wid = blockIdx.x * kCombineWarps + wib;
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int rblocks = (p.group + 31) / 32;
  constexpr int kColBlocks = DVH / 32;
  if (wid >= 2 * p.planes * rblocks * kColBlocks) return;
  const int blk = wid % kColBlocks;
  const int rb = wid / kColBlocks;
  const int half = rb / (p.planes * rblocks);
  const int rest = rb - half * p.planes * rblocks;
  const int plane = rest / rblocks;
  const int r0 = (rest - plane * rblocks) * 32;
  const int r = r0 + lane;
  const bool live = r < p.group;
  const int rr = live ? r : r0;   // dead lanes read a live row and write nothing
  const long long tiles = p.tiles;
  const long long total = 2LL * p.planes * tiles;
  const long long sg = static_cast<long long>(half) * p.planes + plane;
  const long long gs = sg * tiles, ge = gs + tiles - 1;
  const int c_first = static_cast<int>(((gs + 1) * grid + total - 1) / total - 1);
  const int c_last = static_cast<int>(((ge + 1) * grid + total - 1) / total - 1);
  // Partial slot of the i-th CTA whose range meets this (half, plane), or -1.
  auto slot_of = [&](int i) -> long long {
    const int cta = c_first + i;
    const long long b0 = range_begin(total, cta, grid), b1 = range_begin(total, cta + 1, grid);
    if (b1 <= b0) return -1;
    return static_cast<long long>(cta) * p.max_seg + (sg - b0 / tiles);
  };
  const int ns = c_last - c_first + 1;
  float mx = -INFINITY, tot = 0.f;
  float4 acc[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (ns <= kCombineMaxSlots) {
    // Every slot's LSE in one round of loads, then every slot's 32 columns
    // in one round, so the warp waits for memory twice, not once per slot.
    long long sl[kCombineMaxSlots];
    float ls[kCombineMaxSlots];
#pragma unroll
    for (int i = 0; i < kCombineMaxSlots; ++i) sl[i] = (i < ns) ? slot_of(i) : -1;
#pragma unroll
    for (int i = 0; i < kCombineMaxSlots; ++i) ls[i] = (sl[i] >= 0) ? p.lse_part[sl[i] * BM + rr] : -INFINITY;
#pragma unroll
    for (int i = 0; i < kCombineMaxSlots; ++i) mx = fmaxf(mx, ls[i]);
    float4 x[kCombineMaxSlots][8];
#pragma unroll
    for (int i = 0; i < kCombineMaxSlots; ++i) {
      const bool use = ls[i] != -INFINITY;   // also false for a missing slot
      const float4* src = reinterpret_cast<const float4*>(p.o_part) + ((use ? sl[i] : 0) * (DVH / 4) + blk * 8) * BM + rr;
#pragma unroll
      for (int c = 0; c < 8; ++c) x[i][c] = use ? src[static_cast<size_t>(c) * BM] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float w[kCombineMaxSlots];
#pragma unroll
    for (int i = 0; i < kCombineMaxSlots; ++i) {
      w[i] = (ls[i] != -INFINITY) ? expf(ls[i] - mx) : 0.f;
      tot += w[i];
    }
    const float inv = (tot > 0.f) ? 1.f / tot : 0.f;
#pragma unroll
    for (int i = 0; i < kCombineMaxSlots; ++i) {
      const float wi = w[i] * inv;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        acc[c].x += wi * x[i][c].x; acc[c].y += wi * x[i][c].y; acc[c].z += wi * x[i][c].z; acc[c].w += wi * x[i][c].w;
      }
    }
  } else {
    for (int i = 0; i < ns; ++i) {
      const long long s = slot_of(i);
      if (s >= 0) mx = fmaxf(mx, p.lse_part[s * BM + rr]);
    }
    if (mx != -INFINITY) {
      for (int i = 0; i < ns; ++i) {
        const long long s = slot_of(i);
        if (s < 0) continue;
        const float ls = p.lse_part[s * BM + rr];
        if (ls != -INFINITY) tot += expf(ls - mx);
      }
    }
    const float inv = (tot > 0.f) ? 1.f / tot : 0.f;
    if (mx != -INFINITY) {
      for (int i = 0; i < ns; ++i) {
        const long long s = slot_of(i);
        if (s < 0) continue;
        const float ls = p.lse_part[s * BM + rr];
        if (ls == -INFINITY) continue;
        const float w = expf(ls - mx) * inv;
        const float4* src = reinterpret_cast<const float4*>(p.o_part) + (s * (DVH / 4) + blk * 8) * BM + rr;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 x = src[static_cast<size_t>(c) * BM];
          acc[c].x += w * x.x; acc[c].y += w * x.y; acc[c].z += w * x.z; acc[c].w += w * x.w;
        }
      }
    }
  }
  const size_t out_rows = (static_cast<size_t>(plane) * p.group + r0) * (2 * DVH) + half * DVH;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    tile[wib][lane][4 * c] = acc[c].x;
    tile[wib][lane][4 * c + 1] = acc[c].y;
    tile[wib][lane][4 * c + 2] = acc[c].z;
    tile[wib][lane][4 * c + 3] = acc[c].w;
  }
  __syncwarp();
  for (int row = 0; row < 32 && r0 + row < p.group; ++row) {
    const size_t at = out_rows + static_cast<size_t>(row) * (2 * DVH) + blk * 32 + lane;
    if (o != nullptr)
      o[at] = tile[wib][row][lane];
    else
      o_bf16[at] = static_cast<uint16_t>(pack_bf16x2(tile[wib][row][lane], 0.f) & 0xFFFFu);   // round to nearest even
  }
  if (half == 0 && blk == 0 && live && lse != nullptr)
    lse[static_cast<size_t>(plane) * p.group + r] = (tot > 0.f) ? mx + logf(tot) : -INFINITY;
}

}  // namespace

int decode_tiles(int Nkv) { return (Nkv + BN - 1) / BN; }
int decode_key_tile() { return BN; }

int decode_max_segments(int planes, int tiles, int grid) {
  const long long total = 2LL * planes * tiles;
  int mx = 1;
  for (int c = 0; c < grid; ++c) {
    const long long g0 = range_begin(total, c, grid), g1 = range_begin(total, c + 1, grid);
    if (g1 <= g0) continue;
    const int n = static_cast<int>((g1 - 1) / tiles - g0 / tiles + 1);
    if (n > mx) mx = n;
  }
  return mx;
}

cudaError_t launch_decode(const LatentMaps& m, const DecodeParams& p, int grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(latent_kernel<DecodeParams>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  latent_kernel<DecodeParams><<<grid, kThreads, SMEM_BYTES, stream>>>(m.q, m.k5, m.k4, m.k1, p);
  return cudaGetLastError();
}

cudaError_t launch_latent_prefill(const LatentMaps& m, const LatentPrefillParams& p, int num_sms,
                                  cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(latent_kernel<LatentPrefillParams>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  const int grid = min(p.num_units, num_sms);
  if (grid <= 0) return cudaSuccess;
  latent_kernel<LatentPrefillParams><<<grid, kThreads, SMEM_BYTES, stream>>>(m.q, m.k5, m.k4, m.k1, p);
  return cudaGetLastError();
}

cudaError_t launch_combine(const DecodeParams& p, int grid, float* o, uint16_t* o_bf16, float* lse,
                           cudaStream_t stream) {
  const int warps = 2 * p.planes * ((p.group + 31) / 32) * (DVH / 32);
  combine_kernel<<<(warps + kCombineWarps - 1) / kCombineWarps, kCombineWarps * 32, 0, stream>>>(p, grid, o, o_bf16,
                                                                                                    lse);
  return cudaGetLastError();
}

}  // namespace gbattn
