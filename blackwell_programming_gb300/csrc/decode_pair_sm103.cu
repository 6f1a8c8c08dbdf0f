// decode_pair_sm103.cu - the split-KV decode for the latent head-dim shape
// (d_qk = 576, d_v = 512, V = the first 512 features of K) on CTA pairs whose
// two CTAs have different jobs.
//
// The shape is the DeepSeek MLA case of "Distilling a 4.5 hour CUDA talk",
// sections 12-13.  Nq = 1, so the Hq / Hkv query heads that share a KV head
// are the 128 rows (TMEM lanes) of every tile.  A 128 x 512 fp32 O fills all
// 512 columns of one SM's tensor memory, which leaves no room there for the
// scores; so the work of one (sequence, key tile) is split by role across the
// two SMs of a cluster instead of by O columns:
//
//   score CTA: Q (all 576 features, 288 TMEM columns) and two 64-column
//     score buffers in TMEM; S = Q K^T on the tensor core, the online
//     softmax on its four softmax warps, and P (bf16) sent to the value CTA.
//     The two score buffers let the tensor core compute tile j+1 while the
//     softmax works on tile j.
//   value CTA: the whole 128 x 512 fp32 O in TMEM; O += P V with P from
//     shared memory, the rescale of O when a row's reference grows, and the
//     epilogue.
//
// Every score tile is computed once, by one SM, and P crosses the pair in one
// direction only: one bulk copy of 17.5 KB per tile (P in the 128-byte
// swizzled K-major layout the MMA reads, then per row the rescale factor and,
// on a segment's last tile, 1/l and the LSE), which completes a barrier of the
// value CTA.  Nothing the score CTA does waits on the value CTA except the
// flow control of the P ring, so the copy latency is hidden behind the ring's
// depth.
//
// Parallel split ("stream-K" style, "Distilling..." section 5): the
// (sequence, key tile) space is cut into one contiguous equal range per pair.
// Each piece of a sequence that a range holds (normalised O over its keys,
// and its LSE) goes to its own workspace slot -- pair c's piece of sequence b
// to slot c + b, unique because the ranges are increasing -- so no two CTAs
// write the same slot.  The combine kernel then merges the pieces of each row
// with all SMs at once:
//   LSE = log sum_s exp(lse_s),   O = sum_s exp(lse_s - LSE) O_s.
//
// Prefill (Nq > 1, causal or not): a work unit is (batch, query head, block
// of 128 query rows) and covers every K tile the block sees -- all of them,
// or up to the causal diagonal with bottom-right alignment -- so the value
// CTA writes O and the score CTA the LSE directly; the same two roles, Q
// block in the score CTA's TMEM, O in the value CTA's.
//
// Roles (192 threads in both CTAs): warp 5 = TMA producer, warp 4 = MMA issuer
// (whole warp, one elected lane), warps 0-3 = one row per thread (the score
// CTA's softmax and Q, the value CTA's rescale and epilogue).
#include <cmath>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int DQK = 576;
constexpr int DV = 512;
constexpr int BM = 128;                 // rows = query heads of one KV head
constexpr int BN = 64;                  // keys per K tile
constexpr int KCH = DQK / 64;           // 9 chunks of 64 features (128 bytes)
constexpr int GCH = kPairKeyChunks;     // chunks per K granule (one TMA box)
constexpr int GRANS = KCH / GCH;        // granules per K tile
constexpr int QPOS = 2 * GRANS;         // ring positions of a segment's Q: 2 halves of 64 rows x GRANS chunk groups
constexpr int KSLOTS = 7;               // score CTA: K granule ring
constexpr int NSTG = 2;                 // score CTA: P staging buffers
constexpr int VST = 2;                  // value CTA: V stages
constexpr int NP = 5;                   // value CTA: P blocks in flight
constexpr int kThreads = 192;
constexpr int kMmaWarp = 4;
constexpr int kTmaWarp = 5;
constexpr uint32_t kValueRank = 0;
constexpr uint32_t kScoreRank = 1;
constexpr uint32_t kSenderLane = 3;     // score CTA, warp 5: issues the P copies
constexpr uint32_t kQBar = 1;           // named barrier of the score CTA's 128 softmax threads
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kFull = 0xFFFFFFFFu;

constexpr uint32_t CHUNK_K = BN * 128;            // 8 KB: 64 keys x 64 features
constexpr uint32_t GRAN_BYTES = GCH * CHUNK_K;    // 24 KB
constexpr uint32_t V_BYTES = (DV / 64) * CHUNK_K; // 64 KB
constexpr uint32_t P_TILE = BM * 128;             // 16 KB: 128 rows x 64 keys, bf16
constexpr uint32_t HDR_ALPHA = P_TILE;            // float per row: O's rescale factor
constexpr uint32_t HDR_INVL = P_TILE + BM * 4;    // float per row: 1/l on a segment's last tile
constexpr uint32_t HDR_LSE = P_TILE + 2 * BM * 4; // float per row: the segment's LSE, on its last tile
constexpr uint32_t P_BLOCK = P_TILE + 3 * BM * 4; // bytes copied per tile (17.5 KB)
constexpr uint32_t P_STRIDE = 18 * 1024;          // P slot stride, a multiple of 1024

// Barriers sit at the same offsets in both CTAs, so a commit can arrive on
// the peer's barrier by offset and a message names the peer's barrier by
// mapping its own offset.
enum : int {
  B_KFULL = 0,
  B_KEMPTY = B_KFULL + KSLOTS,
  B_SFULL = B_KEMPTY + KSLOTS,
  B_SFREE = B_SFULL + 2,
  B_QFULL = B_SFREE + 2,
  B_PFREE = B_QFULL + 1,       // score CTA: P block s free (the value CTA's P V on it finished)
  B_STGFREE = B_PFREE + NP,    // score CTA: staging buffer's copy has landed
  B_STAGED = B_STGFREE + NSTG, // score CTA: staging buffer written by the softmax warps
  B_SDRAIN = B_STAGED + NSTG,
  B_VFULL = B_SDRAIN + 1,
  B_VEMPTY = B_VFULL + VST,
  B_PFULL = B_VEMPTY + VST,    // value CTA: P block s has landed
  B_CORR = B_PFULL + NP,       // value CTA: O rescaled (or not needed) for the block in s
  B_PVDONE = B_CORR + NP,      // value CTA: P V of the block in s finished
  B_OFULL = B_PVDONE + NP,
  B_OEMPTY = B_OFULL + 1,
  B_VDRAIN = B_OEMPTY + 1,
  NUM_BARS = B_VDRAIN + 1
};
constexpr uint32_t OFF_BAR = 0;
constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;   // TMEM address, abort flag, blocks sent
constexpr uint32_t OFF_DATA = 1024;
// score CTA
constexpr uint32_t OFF_K = OFF_DATA;
constexpr uint32_t OFF_STG = OFF_K + KSLOTS * GRAN_BYTES;
constexpr uint32_t S_END = OFF_STG + NSTG * P_STRIDE;
// value CTA
constexpr uint32_t OFF_V = OFF_DATA;
constexpr uint32_t OFF_P = OFF_V + VST * V_BYTES;
constexpr uint32_t V_END = OFF_P + NP * P_STRIDE;
constexpr uint32_t SMEM_BYTES = (S_END > V_END ? S_END : V_END) + 1024;
static_assert(OFF_MISC + 16 <= OFF_DATA, "barrier area");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(KCH % GCH == 0 && P_STRIDE % 1024 == 0 && P_BLOCK % 16 == 0 && P_BLOCK <= P_STRIDE &&
                  OFF_STG % 1024 == 0 && OFF_P % 1024 == 0,
              "1024-byte aligned swizzled tiles");

// TMEM.  Score CTA: Q features 2i, 2i+1 in column i (0..287), score buffers
// at 384 and 448.  Value CTA: O in columns 0..511.
constexpr uint32_t COL_Q = 0;
constexpr uint32_t COL_S = 384;
constexpr uint32_t COL_O = 0;
constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, 256, false, true);

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(kFull, ok);
}
__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const bool ok = mbar_wait_cluster(bar, parity, w);
  return __all_sync(kFull, ok);
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__host__ __device__ __forceinline__ long long range_begin(long long total, int c, int n) { return total * c / n; }

// One run of K tiles of one sequence for one block of query rows: in decode a
// contiguous piece of a pair's range, in prefill a whole work unit.
struct Segment {
  int plane;   // K plane (batch * Hkv + KV head)
  int qplane;  // Q plane: decode = the K plane (rows = heads), prefill = batch * Hq + head
  int qrow0;   // first query row of the block in its Q plane
  int t0, n;   // first tile, tile count (0: a prefill block that sees no key)
  int slot;    // decode: workspace slot of its piece
};

// Decode: the (sequence, key tile) space cut into one contiguous equal range
// per pair.
struct DecodeWalker {
  long long g, g1, g0;
  int tiles, pair;
  __device__ explicit DecodeWalker(const DecodeParams& p) {
    const long long total = static_cast<long long>(p.planes) * p.tiles;
    pair = static_cast<int>(blockIdx.x >> 1);
    const int pairs = static_cast<int>(gridDim.x >> 1);
    g0 = g = range_begin(total, pair, pairs);
    g1 = range_begin(total, pair + 1, pairs);
    tiles = p.tiles;
  }
  __device__ bool next(Segment& s) {
    if (g >= g1) return false;
    const long long pl = g / tiles;
    s.plane = static_cast<int>(pl);
    s.t0 = static_cast<int>(g - pl * tiles);
    const long long end = min(g1, (pl + 1) * tiles);
    s.n = static_cast<int>(end - g);
    s.slot = pair + s.plane;
    s.qplane = s.plane;
    s.qrow0 = 0;
    g = end;
    return true;
  }
};

// Prefill: unit u = (query block counted from the bottom) * B * Hq + batch *
// Hq + head, so long causal blocks come first and the heads that share a KV
// head run side by side (their K tiles come from L2); the units go to the
// pairs in rounds, every other round reversed (snake), so each pair gets a
// similar mix of long and short blocks.
struct PrefillWalker {
  const LatentPrefillParams& p;
  int it = 0;
  __device__ explicit PrefillWalker(const LatentPrefillParams& prm) : p(prm) {}
  __device__ bool next(Segment& s) {
    const int pairs = static_cast<int>(gridDim.x >> 1), pair = static_cast<int>(blockIdx.x >> 1);
    const int base = it * pairs;
    const int u = (it & 1) ? base + pairs - 1 - pair : base + pair;
    ++it;
    if (u >= p.num_units) return false;
    const int bh_count = p.B * p.Hq;
    const int qb = p.nqb - 1 - u / bh_count;
    const int bh = u - (u / bh_count) * bh_count;
    const int b = bh / p.Hq, h = bh - b * p.Hq;
    s.qplane = bh;
    s.plane = b * p.Hkv + h / (p.Hq / p.Hkv);
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
template <> struct WalkerFor<DecodeParams> { using type = DecodeWalker; };
template <> struct WalkerFor<LatentPrefillParams> { using type = PrefillWalker; };
template <class P> __host__ __device__ constexpr bool is_prefill() { return std::is_same<P, LatentPrefillParams>::value; }

struct Ctx {
  uint32_t sbase, tm, warp, lane, peer;
  WaitCtx w;
  __device__ uint32_t bar(int i) const { return sbase + OFF_BAR + 8u * static_cast<uint32_t>(i); }
};

// ---------------------------------------------------------------- score CTA
// The K ring carries Q too.  Ring positions count slot uses: at each segment
// the sequence's Q takes the next six positions, one box of 64 rows x 3
// chunks each (rows 0-63 then 64-127; rows past the group read as zeros),
// which the softmax warps move into TMEM; then every K tile takes three (its
// granules), which the MMA warp reads.  So a segment's Q is fetched as early
// as the ring's look-ahead allows, like a K tile, and all of it fits in the
// ring at once.
//
// Warp 5: lanes 0..GRANS-1 fill the ring; lane g fills the positions
// congruent to g mod GRANS (positions advance by 6 and 3, so a segment
// starts at a multiple of 3).  Lane kSenderLane sends each staged P block to
// the value CTA, once the block's slot there is free, as one bulk copy that
// completes the slot's barrier (armed by the value CTA).  Returns the number
// of blocks sent (on the sender lane).
template <class P>
__device__ uint32_t score_producer(const Ctx& x, const CUtensorMap* tmQ, const CUtensorMap* tmK, const P& p) {
  using Walker = typename WalkerFor<P>::type;
  const int g = static_cast<int>(x.lane);
  int last = -1;   // the last ring position this lane filled
  uint32_t sent = 0;
  if (x.lane == kSenderLane) {
    const uint32_t pdst0 = mapa_shared(x.sbase + OFF_P, x.peer);
    const uint32_t pfull0 = mapa_shared(x.bar(B_PFULL), x.peer);
    Walker walk(p);
    Segment S;
    bool ok = true;
    int c = 0;
    while (ok && walk.next(S)) {
      for (int j = 0; j < S.n; ++j, ++c) {
        const int sb = c % NSTG, s = c % NP;
        if (!(ok = mbar_wait(x.bar(B_STAGED + sb), (c / NSTG) & 1, x.w))) break;
        if (!(ok = mbar_wait_cluster(x.bar(B_PFREE + s), ((c / NP) & 1) ^ 1u, x.w))) break;
        bulk_copy_to_cluster(pdst0 + static_cast<uint32_t>(s) * P_STRIDE, x.sbase + OFF_STG + sb * P_STRIDE, P_BLOCK,
                             pfull0 + 8u * s);
        ++sent;
      }
    }
  } else if (g < GRANS) {
    if (g == 0) {
      tma_prefetch_desc(tmQ);
      tma_prefetch_desc(tmK);
    }
    // decode: the value CTA reads the first 512 features of K again, from L2;
    // prefill: every head of the KV head and every query block reads K again
    const uint64_t pol = is_prefill<P>() ? l2_policy_evict_last() : l2_policy_evict_normal();
    // claim ring position idx for `bytes`: wait until its slot is free
    auto claim = [&](int idx, uint32_t bytes) -> bool {
      const int slot = idx % KSLOTS;
      if (!mbar_wait(x.bar(B_KEMPTY + slot), ((idx / KSLOTS) & 1) ^ 1u, x.w)) return false;
      mbar_arrive_expect_tx(x.bar(B_KFULL + slot), bytes);
      return true;
    };
    Walker walk(p);
    Segment S;
    bool ok = true;
    int ridx = 0;
    while (ok && walk.next(S)) {
      if (S.n == 0) continue;   // a prefill block that sees no key: the row warps write it
      for (int i = g; i < QPOS; i += GRANS) {
        const int idx = ridx + i;
        if (!(ok = claim(idx, GRAN_BYTES))) break;
        const int slot = idx % KSLOTS;
        tma_load_4d(x.sbase + OFF_K + slot * GRAN_BYTES, tmQ, x.bar(B_KFULL + slot), 0, S.qrow0 + BN * (i / GRANS),
                    GCH * (i % GRANS), S.qplane, pol);
        last = idx;
      }
      if (!ok) break;
      ridx += QPOS;
      for (int j = 0; j < S.n; ++j, ridx += GRANS) {
        const int idx = ridx + g;
        if (!(ok = claim(idx, GRAN_BYTES))) break;
        const int slot = idx % KSLOTS;
        tma_load_4d(x.sbase + OFF_K + slot * GRAN_BYTES, tmK, x.bar(B_KFULL + slot), 0, (S.t0 + j) * BN, GCH * g,
                    S.plane, pol);
        last = idx;
      }
    }
  }
  // Every issued copy must have landed before the CTA may exit: for each
  // slot, wait for the phase of its latest fill by any lane.
  int lst[GRANS];
#pragma unroll
  for (int i = 0; i < GRANS; ++i) lst[i] = __shfl_sync(kFull, last, i);
  if (x.lane == 0) {
    for (int slot = 0; slot < KSLOTS; ++slot) {
      int best = -1;
      for (int i = 0; i < GRANS; ++i)
        for (int idx = lst[i]; idx >= 0 && idx > lst[i] - GRANS * KSLOTS; idx -= GRANS)
          if (idx % KSLOTS == slot) {
            best = max(best, idx);
            break;
          }
      if (best >= 0) mbar_wait_drain(x.bar(B_KFULL + slot), (best / KSLOTS) & 1);
    }
  }
  __syncwarp();
  return sent;
}

// Warp 4: S = Q K^T (36 MMAs of 16 features, A = Q in TMEM) into score
// buffer c & 1, once the softmax has read what the buffer held two tiles ago.
template <class P>
__device__ void score_mma(const Ctx& x, const P& p) {
  using Walker = typename WalkerFor<P>::type;
  const uint64_t kd0 = smem_desc_sw128(x.sbase + OFF_K, 16, 1024);
  Walker walk(p);
  Segment S;
  bool ok = true;
  int c = 0, ridx = 0;
  uint32_t qph = 0;
  while (ok && walk.next(S)) {
    if (S.n == 0) continue;
    ridx += QPOS;   // this segment's Q, which the softmax warps consume
    if (!(ok = warp_wait(x.bar(B_QFULL), qph, x.w))) break;
    qph ^= 1u;
    tc_fence_after();
    for (int j = 0; j < S.n && ok; ++j, ++c, ridx += GRANS) {
      const int b = c & 1;
      if (!(ok = warp_wait(x.bar(B_SFREE + b), ((c >> 1) & 1) ^ 1u, x.w))) break;
      tc_fence_after();
      const uint32_t dS = x.tm + COL_S + static_cast<uint32_t>(b) * BN;
      for (int g = 0; g < GRANS; ++g) {
        const int idx = ridx + g;
        const int slot = idx % KSLOTS;
        if (!(ok = warp_wait(x.bar(B_KFULL + slot), (idx / KSLOTS) & 1, x.w))) break;
        tc_fence_after();
        const uint64_t gd = kd0 + ((slot * GRAN_BYTES) >> 4);
#pragma unroll
        for (int cc = 0; cc < GCH; ++cc) {
          const int kk0 = (g * GCH + cc) * 4;
          uint32_t a[4];
          uint64_t bd[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            a[i] = x.tm + COL_Q + static_cast<uint32_t>(kk0 + i) * 8u;
            bd[i] = gd + ((cc * CHUNK_K) >> 4) + static_cast<uint64_t>(i * 2);
          }
          mma_ts_warp4(dS, a, bd, IDESC_S, kk0 > 0 ? 1u : 0u);
        }
        mma_commit_warp(x.bar(B_KEMPTY + slot));
      }
      if (!ok) break;
      mma_commit_warp(x.bar(B_SFULL + b));
    }
  }
  mma_commit_warp(x.bar(B_SDRAIN));
  mbar_wait_drain(x.bar(B_SDRAIN), 0);
  __syncwarp();
}

// Warps 0-3: Q into TMEM at every segment; per tile the softmax of row r,
// then P and the row's header into a staging buffer, which the sender lane
// copies to the value CTA.  Each warp runs on its own: it waits for the
// staging buffer's previous copy to have landed, writes its 32 rows and
// arrives on the buffer's barrier.
template <class P>
__device__ void score_softmax(const Ctx& x, const P& p) {
  using Walker = typename WalkerFor<P>::type;
  const int r = static_cast<int>(x.warp * 32 + x.lane);
  const uint32_t lane_addr = (x.warp * 32u) << 16;
  const float sl2 = p.scale_log2;
  const uint32_t rsw = static_cast<uint32_t>(r & 7);
  const uint32_t stg0 = x.sbase + OFF_STG;
  Walker walk(p);
  Segment S;
  bool ok = true;
  int c = 0, ridx = 0;
  while (ok && walk.next(S)) {
    bool live = true;
    // The last key row r may see (all of them, or up to the causal diagonal
    // with bottom-right alignment), and the first row's limit: a tile whose
    // last key is past it needs the mask.
    int key_lim = p.Nkv - 1, lim0 = p.Nkv - 1;
    if constexpr (is_prefill<P>()) {
      live = S.qrow0 + r < p.Nq;
      if (p.causal) {
        key_lim = min(S.qrow0 + r + (p.Nkv - p.Nq), p.Nkv - 1);
        lim0 = S.qrow0 + (p.Nkv - p.Nq);
      }
      if (S.n == 0) {   // a block that sees no key
        if (live && p.lse != nullptr) p.lse[static_cast<size_t>(S.qplane) * p.Nq + S.qrow0 + r] = -INFINITY;
        continue;
      }
    }
    // Q row r of this sequence from the ring into TMEM: chunk group cg of row
    // r is box (r / 64) * GRANS + cg, chunk cg * GCH + t at t * 8 KB and row
    // r mod 64.  The previous segment's last score tile has been read, so
    // every Q K^T that used the old Q has finished.  Both boxes of a chunk
    // group go back to the producer once all four warps have read them.
    for (int cg = 0; cg < GRANS; ++cg) {
      const int idx = ridx + (r >> 6) * GRANS + cg;   // warp-uniform
      const int slot = idx % KSLOTS;
      const bool good = warp_wait(x.bar(B_KFULL + slot), (idx / KSLOTS) & 1, x.w);
      if (good) {
#pragma unroll
        for (int t = 0; t < GCH; ++t) {
          const uint32_t src = x.sbase + OFF_K + static_cast<uint32_t>(slot) * GRAN_BYTES + t * CHUNK_K +
                               static_cast<uint32_t>(r & 63) * 128u;
          uint32_t w[32];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            ld_shared_v4(src + ((static_cast<uint32_t>(u) ^ rsw) << 4), w[4 * u], w[4 * u + 1], w[4 * u + 2],
                         w[4 * u + 3]);
          tmem_st32u(x.tm + lane_addr + COL_Q + static_cast<uint32_t>(cg * GCH + t) * 32u, w);
        }
      }
      if (!bar_sync_and(kQBar, 128, good)) {
        ok = false;
        break;
      }
      if (threadIdx.x == 0) {
        mbar_arrive(x.bar(B_KEMPTY + (ridx + cg) % KSLOTS));
        mbar_arrive(x.bar(B_KEMPTY + (ridx + GRANS + cg) % KSLOTS));
      }
    }
    if (!ok) break;
    ridx += QPOS;
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (x.lane == 0) mbar_arrive(x.bar(B_QFULL));
    float R = -INFINITY, l = 0.f;   // the row's reference (log2 units) and sum
    for (int j = 0; j < S.n; ++j, ++c, ridx += GRANS) {
      const int b = c & 1;
      const int sb = c % NSTG;
      float v[BN];
      if (!(ok = warp_wait(x.bar(B_SFULL + b), (c >> 1) & 1, x.w))) break;
      tc_fence_after();
      tmem_ld64(x.tm + lane_addr + COL_S + static_cast<uint32_t>(b) * BN, v);
      tc_fence_before();
      __syncwarp();
      if (x.lane == 0) mbar_arrive(x.bar(B_SFREE + b));
      const int key0 = (S.t0 + j) * BN;
      const bool ragged = key0 + BN - 1 > lim0;
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
      if (m_new > R + kRescaleThreshold) {
        alpha = ex2(R - m_new);
        R = m_new;
      }
      l *= alpha;
      const float base = (R == -INFINITY) ? 0.f : R;
      // Keys past Nkv are -inf and ex2(-inf) = 0; only scale 0 (0 * -inf)
      // needs the visible logits set to 0 with a unit factor.
      float csl = sl2;
      if (ragged && sl2 == 0.f) {
#pragma unroll
        for (int i = 0; i < BN; ++i) v[i] = (v[i] == -INFINITY) ? -INFINITY : 0.f;
        csl = 1.f;
      }
      const uint64_t c2 = f2_pack(csl, csl);
      const uint64_t nb2 = f2_pack(-base, -base);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t pk[BN / 2];
#pragma unroll
      for (int i = 0; i < BN / 2; ++i) {
        const uint64_t e = f2_fma(f2_pack(v[2 * i], v[2 * i + 1]), c2, nb2);
        const float p0 = ex2(f2_lo(e));
        const float p1 = ex2(f2_hi(e));
        acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
        pk[i] = pack_bf16x2(p0, p1);
      }
      const uint64_t a01 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
      l += f2_lo(a01) + f2_hi(a01);
      // The staging buffer is free once its copy two tiles back has landed
      // in the value CTA (which says so on B_STGFREE).
      if (!(ok = warp_wait_cluster(x.bar(B_STGFREE + sb), ((c / NSTG) & 1) ^ 1u, x.w))) break;
      const uint32_t stg = stg0 + static_cast<uint32_t>(sb) * P_STRIDE;
      const uint32_t row = stg + static_cast<uint32_t>(r) * 128u;
#pragma unroll
      for (int u = 0; u < BN / 8; ++u)
        st_shared_v4(row + ((static_cast<uint32_t>(u) ^ rsw) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                     pk[4 * u + 3]);
      st_shared_f32(stg + HDR_ALPHA + 4u * r, alpha);
      if (j == S.n - 1) {
        const float lse_r = l > 0.f ? (R + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        st_shared_f32(stg + HDR_INVL + 4u * r, l > 0.f ? 1.f / l : 0.f);
        st_shared_f32(stg + HDR_LSE + 4u * r, lse_r);
        if constexpr (is_prefill<P>()) {
          if (live && p.lse != nullptr) p.lse[static_cast<size_t>(S.qplane) * p.Nq + S.qrow0 + r] = lse_r;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (x.lane == 0) mbar_arrive(x.bar(B_STAGED + sb));
    }
    if (!ok) break;
  }
}

// ---------------------------------------------------------------- value CTA
// Warp 5, lane 0: the first 512 features of each K tile (V) as one box.
// Lane 1: as each P block lands, tells the score CTA that the staging buffer
// it came from may be refilled (the row warps cannot, as they are busy during
// an epilogue).
template <class P>
__device__ void value_producer(const Ctx& x, const CUtensorMap* tmV, const P& p) {
  using Walker = typename WalkerFor<P>::type;
  if (x.lane == 1) {
    const uint32_t stgfree_peer = mapa_shared(x.bar(B_STGFREE), x.peer);
    Walker walk(p);
    Segment S;
    bool ok = true;
    int c = 0;
    while (ok && walk.next(S)) {
      for (int j = 0; j < S.n; ++j, ++c) {
        if (!(ok = mbar_wait_cluster(x.bar(B_PFULL + c % NP), (c / NP) & 1, x.w))) break;
        mbar_arrive_cluster_relaxed(stgfree_peer + 8u * (c % NSTG));
      }
    }
  } else if (x.lane == 0) {
    tma_prefetch_desc(tmV);
    // decode: the score CTA has read this tile already; prefill: other blocks read it again
    const uint64_t pol = is_prefill<P>() ? l2_policy_evict_last() : l2_policy_evict_first();
    Walker walk(p);
    Segment S;
    bool ok = true;
    int c = 0;
    while (ok && walk.next(S)) {
      for (int j = 0; j < S.n; ++j, ++c) {
        const int v = c % VST;
        if (!(ok = mbar_wait(x.bar(B_VEMPTY + v), ((c / VST) & 1) ^ 1u, x.w))) break;
        mbar_arrive_expect_tx(x.bar(B_VFULL + v), V_BYTES);
        tma_load_4d(x.sbase + OFF_V + v * V_BYTES, tmV, x.bar(B_VFULL + v), 0, (S.t0 + j) * BN, 0, S.plane, pol);
      }
    }
    for (int v = 0; v < VST; ++v) {
      if (c <= v) continue;
      const int last = v + ((c - 1 - v) / VST) * VST;
      mbar_wait_drain(x.bar(B_VFULL + v), (last / VST) & 1);
    }
  }
  __syncwarp();
}

// Warp 4: O += P V, A = P from the block in shared memory (128 rows x 64
// keys), B = V in two 256-column halves, D = O in TMEM.  After each tile it
// frees the V stage, records P V done for the rescale, and frees the P block
// in the score CTA's flow control (a commit that arrives there by offset).
// The row warps read the block's header before they arrive on B_CORR, which
// this warp waits for before the P V, so the commit also covers those reads.
template <class P>
__device__ void value_mma(const Ctx& x, const P& p) {
  using Walker = typename WalkerFor<P>::type;
  const uint64_t pd0 = smem_desc_sw128(x.sbase + OFF_P, 16, 1024);
  const uint64_t vd0 = smem_desc_sw128(x.sbase + OFF_V, CHUNK_K, 1024);
  const uint16_t peer_mask = static_cast<uint16_t>(1u << x.peer);
  Walker walk(p);
  Segment S;
  bool ok = true;
  int c = 0;
  uint32_t oeph = 0;
  while (ok && walk.next(S)) {
    for (int j = 0; j < S.n; ++j, ++c) {
      const int v = c % VST, s = c % NP;
      const uint32_t pph = (c / NP) & 1;
      if (!(ok = warp_wait(x.bar(B_VFULL + v), (c / VST) & 1, x.w))) break;
      if (!(ok = warp_wait_cluster(x.bar(B_PFULL + s), pph, x.w))) break;
      if (!(ok = warp_wait(x.bar(B_CORR + s), pph, x.w))) break;
      if (j == 0) {
        // the previous segment's epilogue must have read O
        if (!(ok = warp_wait(x.bar(B_OEMPTY), oeph ^ 1u, x.w))) break;
        oeph ^= 1u;
      }
      tc_fence_after();
      const uint64_t pd = pd0 + ((static_cast<uint32_t>(s) * P_STRIDE) >> 4);
      const uint64_t vd = vd0 + ((static_cast<uint32_t>(v) * V_BYTES) >> 4);
#pragma unroll
      for (int nh = 0; nh < 2; ++nh) {
        uint64_t a[4], bd[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          a[kk] = pd + static_cast<uint64_t>(kk * 2);
          bd[kk] = vd + ((static_cast<uint32_t>(nh) * 4u * CHUNK_K + static_cast<uint32_t>(kk) * 16u * 128u) >> 4);
        }
        mma_ss_warp4(x.tm + COL_O + static_cast<uint32_t>(nh) * 256u, a, bd, IDESC_PV, j > 0 ? 1u : 0u);
      }
      mma_commit_warp(x.bar(B_VEMPTY + v));
      mma_commit_warp(x.bar(B_PVDONE + s));
      mma_commit_multicast_warp(x.bar(B_PFREE + s), peer_mask);
      if (j == S.n - 1) mma_commit_warp(x.bar(B_OFULL));
    }
  }
  mma_commit_warp(x.bar(B_VDRAIN));
  mbar_wait_drain(x.bar(B_VDRAIN), 0);
  __syncwarp();
}

// Prefill: the block's O rows straight to the output, normalised.  O leaves
// TMEM in the 16x256b shape (lane i holds columns 8k + 2(i mod 4), +1 of rows
// i/4 and i/4 + 8 of a 16-row group), so each warp store writes 8 rows x 32
// contiguous bytes.
__device__ void write_block(const Ctx& x, const LatentPrefillParams& p, const Segment& S, float inv_l) {
  const int lane = static_cast<int>(x.lane);
  const bool bf = p.o == nullptr;
#pragma unroll 1
  for (int hl = 0; hl < 2; ++hl) {
    const int src = hl * 16 + (lane >> 2);   // the lanes that own rows ra and ra + 8 above
    const int ra = static_cast<int>(x.warp) * 32 + src;
    const float iA = __shfl_sync(kFull, inv_l, src), iB = __shfl_sync(kFull, inv_l, src + 8);
    const bool lA = S.qrow0 + ra < p.Nq, lB = S.qrow0 + ra + 8 < p.Nq;
    const size_t base = static_cast<size_t>(S.qplane) * p.Nq + S.qrow0;
    const size_t oA = (base + (lA ? ra : 0)) * DV + 2 * (lane & 3);
    const size_t oB = (base + (lB ? ra + 8 : 0)) * DV + 2 * (lane & 3);
#pragma unroll 1
    for (int ch = 0; ch < DV / 64; ++ch) {
      uint32_t v[32];
      tmem_ld16x256b_x8(x.tm + ((x.warp * 32u + static_cast<uint32_t>(hl) * 16u) << 16) + COL_O + ch * 64, v);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const size_t col = static_cast<size_t>(ch * 64 + 8 * k);
        const float a0 = __uint_as_float(v[4 * k]) * iA, a1 = __uint_as_float(v[4 * k + 1]) * iA;
        const float b0 = __uint_as_float(v[4 * k + 2]) * iB, b1 = __uint_as_float(v[4 * k + 3]) * iB;
        if (bf) {
          if (lA) *reinterpret_cast<uint32_t*>(p.o_bf16 + oA + col) = pack_bf16x2(a0, a1);
          if (lB) *reinterpret_cast<uint32_t*>(p.o_bf16 + oB + col) = pack_bf16x2(b0, b1);
        } else {
          if (lA) *reinterpret_cast<float2*>(p.o + oA + col) = make_float2(a0, a1);
          if (lB) *reinterpret_cast<float2*>(p.o + oB + col) = make_float2(b0, b1);
        }
      }
    }
  }
}

// Warps 0-3: per tile, the row's rescale factor from the block header (O is
// rescaled, after the previous tile's P V, when any row of the warp grew its
// reference); warp 0 then arms the slot's barrier for the block that will
// land there next.  At a segment's end the normalised O goes to the output
// (prefill) or, as a piece with its LSE, to the segment's workspace slot
// (decode).
template <class P>
__device__ void value_rows(const Ctx& x, const P& p) {
  using Walker = typename WalkerFor<P>::type;
  const int r = static_cast<int>(x.warp * 32 + x.lane);
  const uint32_t lane_addr = (x.warp * 32u) << 16;
  Walker walk(p);
  Segment S;
  bool ok = true;
  int c = 0;
  uint32_t ofph = 0;
  while (ok && walk.next(S)) {
    bool live;
    if constexpr (is_prefill<P>()) {
      live = S.qrow0 + r < p.Nq;
      if (S.n == 0) {   // a block that sees no key: O = 0
        if (live) {
          const size_t orow = (static_cast<size_t>(S.qplane) * p.Nq + S.qrow0 + r) * DV;
          if (p.o != nullptr) {
#pragma unroll 4
            for (int k = 0; k < DV / 4; ++k) reinterpret_cast<float4*>(p.o + orow)[k] = make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
#pragma unroll 4
            for (int k = 0; k < DV / 8; ++k) reinterpret_cast<uint4*>(p.o_bf16 + orow)[k] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        continue;
      }
    } else {
      live = r < p.group;
    }
    float inv_l = 0.f, lse_own = -INFINITY;
    for (int j = 0; j < S.n; ++j, ++c) {
      const int s = c % NP;
      if (!(ok = warp_wait_cluster(x.bar(B_PFULL + s), (c / NP) & 1, x.w))) break;
      const uint32_t blk = x.sbase + OFF_P + static_cast<uint32_t>(s) * P_STRIDE;
      const float alpha = ld_shared_f32(blk + HDR_ALPHA + 4u * r);
      if (j == S.n - 1) {
        inv_l = ld_shared_f32(blk + HDR_INVL + 4u * r);
        lse_own = ld_shared_f32(blk + HDR_LSE + 4u * r);
      }
      if (j > 0 && __any_sync(kFull, alpha != 1.f)) {
        // O must hold the previous tile's P V before it is rescaled
        const int cp = c - 1;
        if (!(ok = warp_wait(x.bar(B_PVDONE + cp % NP), (cp / NP) & 1, x.w))) break;
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < DV / 32; ++cc) {
          float o[32];
          tmem_ld32(x.tm + lane_addr + COL_O + cc * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(x.tm + lane_addr + COL_O + cc * 32, o);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (x.lane == 0) {
        mbar_arrive(x.bar(B_CORR + s));
        if (x.warp == 0) mbar_arrive_expect_tx(x.bar(B_PFULL + s), P_BLOCK);
      }
    }
    if (!ok) break;
    if (!(ok = warp_wait(x.bar(B_OFULL), ofph, x.w))) break;
    ofph ^= 1u;
    tc_fence_after();
    if constexpr (is_prefill<P>()) {
      write_block(x, p, S, inv_l);
    } else {
      // Normalised piece, with the float4 of row r and columns 4k..4k+3 at
      // [slot][k][r]: a warp's 32 rows store 512 contiguous bytes at a time.
      float4* opart = reinterpret_cast<float4*>(p.o_part) + static_cast<size_t>(S.slot) * (DV / 4) * BM + r;
  #pragma unroll 1
      for (int cc = 0; cc < DV / 64; ++cc) {
        float o[64];
        tmem_ld64(x.tm + lane_addr + COL_O + cc * 64, o);
        if (live) {
  #pragma unroll
          for (int i = 0; i < 16; ++i)
            opart[static_cast<size_t>(cc * 16 + i) * BM] =
                make_float4(o[4 * i] * inv_l, o[4 * i + 1] * inv_l, o[4 * i + 2] * inv_l, o[4 * i + 3] * inv_l);
        }
      }
      if (live) p.lse_part[static_cast<size_t>(S.slot) * BM + r] = lse_own;
    }
    tc_fence_before();
    __syncwarp();
    if (x.lane == 0) mbar_arrive(x.bar(B_OEMPTY));
  }
}

template <class P>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    latent_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const P p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctx x;
  x.sbase = smem_u32(smem);
  x.warp = warp_id();
  x.lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  x.peer = rank ^ 1u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC + 4);
  volatile uint32_t* sent_count = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC + 8);
  x.w = WaitCtx{abort_flag, p.err};
  // The merge kernel that follows a decode launch may be scheduled now: its
  // blocks wait for this grid to complete before they read anything.
  grid_launch_dependents();

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    *sent_count = 0u;
    for (int s = 0; s < KSLOTS; ++s) {
      mbar_init(x.bar(B_KFULL + s), 1);
      mbar_init(x.bar(B_KEMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(x.bar(B_SFULL + b), 1);
      mbar_init(x.bar(B_SFREE + b), 4);
    }
    mbar_init(x.bar(B_QFULL), 4);
    for (int s = 0; s < NP; ++s) {
      mbar_init(x.bar(B_PFREE + s), 1);   // the value CTA's P V commit
      mbar_init(x.bar(B_PFULL + s), 1);   // armed by the value CTA with the block's bytes
      mbar_init(x.bar(B_CORR + s), 4);
      mbar_init(x.bar(B_PVDONE + s), 1);
    }
    for (int b = 0; b < NSTG; ++b) {
      mbar_init(x.bar(B_STGFREE + b), 1);
      mbar_init(x.bar(B_STAGED + b), 4);
    }
    mbar_init(x.bar(B_SDRAIN), 1);
    for (int v = 0; v < VST; ++v) {
      mbar_init(x.bar(B_VFULL + v), 1);
      mbar_init(x.bar(B_VEMPTY + v), 1);
    }
    mbar_init(x.bar(B_OFULL), 1);
    mbar_init(x.bar(B_OEMPTY), 4);
    mbar_init(x.bar(B_VDRAIN), 1);
    fence_mbar_init();
    // value CTA: the first block of every P slot is expected from the start
    if (rank == kValueRank)
      for (int s = 0; s < NP; ++s) mbar_arrive_expect_tx(x.bar(B_PFULL + s), P_BLOCK);
  }
  if (x.warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync_all();   // both CTAs' barriers exist before any message crosses
  tc_fence_after();
  x.tm = *tmem_slot;

  uint32_t sent = 0;
  if (rank == kScoreRank) {
    if (x.warp == kTmaWarp)
      sent = score_producer(x, &tmQ, &tmK, p);
    else if (x.warp == kMmaWarp)
      score_mma(x, p);
    else
      score_softmax(x, p);
  } else {
    if (x.warp == kTmaWarp)
      value_producer(x, &tmV, p);
    else if (x.warp == kMmaWarp)
      value_mma(x, p);
    else
      value_rows(x, p);
  }

  // Teardown.  After an early stop the value CTA may not have waited for
  // every block the score CTA sent, so it learns the count and waits for
  // them to land before either CTA leaves (a copy must not land in the
  // shared memory of an exited CTA).
  tc_fence_before();
  if (rank == kScoreRank && x.warp == kTmaWarp && x.lane == kSenderLane)
    st_cluster_u32(mapa_shared(x.sbase + OFF_MISC + 8, x.peer), sent);
  cluster_sync_all();
  if (rank == kValueRank && threadIdx.x == 0) {
    const int n = static_cast<int>(*sent_count);
    for (int s = 0; s < NP; ++s) {
      if (n <= s) continue;
      const int last = s + ((n - 1 - s) / NP) * NP;
      mbar_wait_drain(x.bar(B_PFULL + s), (last / NP) & 1);
    }
  }
  cluster_sync_all();
  if (x.warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(x.tm, 512);
  }
}

// Combine: one warp per (sequence, 32 output rows, 32 output columns), one
// lane per row.  A lane reduces its row's piece LSEs and merges its 32
// columns from float4 reads that are coalesced across the lanes, then the
// block is transposed through shared memory into 128-byte row stores.
constexpr int kCombineWarps = 4;
constexpr int kCombineMaxSlots = 4;   // pieces per sequence handled in registers
__global__ void __launch_bounds__(kCombineWarps * 32) combine_pair_kernel(const DecodeParams p, int pairs, float* o,
                                                                          uint16_t* o_bf16, float* lse) {
  __shared__ float tile[kCombineWarps][32][33];
  // launched as a programmatic dependent of the decode grid: its pieces are
  // read only once that grid has completed
  grid_dependency_wait();
  const int wib = static_cast<int>(threadIdx.x >> 5);
  const int wid = blockIdx.x * kCombineWarps + wib;
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int rblocks = (p.group + 31) / 32;
  constexpr int kColBlocks = DV / 32;
  if (wid >= p.planes * rblocks * kColBlocks) return;
  const int blk = wid % kColBlocks;
  const int rb = wid / kColBlocks;
  const int plane = rb / rblocks;
  const int r0 = (rb - plane * rblocks) * 32;
  const int r = r0 + lane;
  const bool live = r < p.group;
  const int rr = live ? r : r0;   // dead lanes read a live row and write nothing
  const long long total = static_cast<long long>(p.planes) * p.tiles;
  const long long gs = static_cast<long long>(plane) * p.tiles, ge = gs + p.tiles - 1;
  // the pairs whose ranges hold the sequence's first and last tiles
  const int c_first = static_cast<int>(((gs + 1) * pairs + total - 1) / total - 1);
  const int c_last = static_cast<int>(((ge + 1) * pairs + total - 1) / total - 1);
  auto slot_of = [&](int i) -> long long {
    const int cta = c_first + i;
    if (range_begin(total, cta + 1, pairs) <= range_begin(total, cta, pairs)) return -1;
    return static_cast<long long>(cta) + plane;
  };
  const int ns = c_last - c_first + 1;
  float mx = -INFINITY, tot = 0.f;
  float4 acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (ns <= kCombineMaxSlots) {
    long long sl[kCombineMaxSlots];
    float ls[kCombineMaxSlots];
#pragma unroll
    for (int i = 0; i < kCombineMaxSlots; ++i) sl[i] = (i < ns) ? slot_of(i) : -1;
#pragma unroll
    for (int i = 0; i < kCombineMaxSlots; ++i) ls[i] = (sl[i] >= 0) ? p.lse_part[sl[i] * BM + rr] : -INFINITY;
#pragma unroll
    for (int i = 0; i < kCombineMaxSlots; ++i) mx = fmaxf(mx, ls[i]);
    // The pieces' columns are loaded in the same round as their LSEs (a
    // piece whose LSE is -inf holds zeros, and its weight is 0).
    float4 xv[kCombineMaxSlots][8];
#pragma unroll
    for (int i = 0; i < kCombineMaxSlots; ++i) {
      const bool use = sl[i] >= 0;
      const float4* src = reinterpret_cast<const float4*>(p.o_part) + ((use ? sl[i] : 0) * (DV / 4) + blk * 8) * BM + rr;
#pragma unroll
      for (int k = 0; k < 8; ++k) xv[i][k] = use ? src[static_cast<size_t>(k) * BM] : make_float4(0.f, 0.f, 0.f, 0.f);
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
      for (int k = 0; k < 8; ++k) {
        acc[k].x += wi * xv[i][k].x; acc[k].y += wi * xv[i][k].y; acc[k].z += wi * xv[i][k].z; acc[k].w += wi * xv[i][k].w;
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
        const float4* src = reinterpret_cast<const float4*>(p.o_part) + (s * (DV / 4) + blk * 8) * BM + rr;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float4 xv = src[static_cast<size_t>(k) * BM];
          acc[k].x += w * xv.x; acc[k].y += w * xv.y; acc[k].z += w * xv.z; acc[k].w += w * xv.w;
        }
      }
    }
  }
  const size_t out_rows = (static_cast<size_t>(plane) * p.group + r0) * DV;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    tile[wib][lane][4 * k] = acc[k].x;
    tile[wib][lane][4 * k + 1] = acc[k].y;
    tile[wib][lane][4 * k + 2] = acc[k].z;
    tile[wib][lane][4 * k + 3] = acc[k].w;
  }
  __syncwarp();
  // Four rows per store: lane l writes columns 4(l mod 8) .. +3 of row l/8.
  const int c4 = 4 * (lane & 7);
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int row = it * 4 + (lane >> 3);
    if (r0 + row >= p.group) continue;
    const float a0 = tile[wib][row][c4], a1 = tile[wib][row][c4 + 1], a2 = tile[wib][row][c4 + 2],
                a3 = tile[wib][row][c4 + 3];
    const size_t at = out_rows + static_cast<size_t>(row) * DV + blk * 32 + c4;
    if (o != nullptr)
      *reinterpret_cast<float4*>(o + at) = make_float4(a0, a1, a2, a3);
    else
      *reinterpret_cast<uint2*>(o_bf16 + at) = make_uint2(pack_bf16x2(a0, a1), pack_bf16x2(a2, a3));
  }
  if (blk == 0 && live && lse != nullptr)
    lse[static_cast<size_t>(plane) * p.group + r] = (tot > 0.f) ? mx + logf(tot) : -INFINITY;
}

}  // namespace

int decode_pair_slots(int planes, int pairs) { return pairs + planes - 1; }

int decode_pair_max_pairs(int num_sms, int* out) {
  // Both instances (decode and prefill) use the same resources.
  cudaError_t e = cudaFuncSetAttribute(latent_pair_kernel<DecodeParams>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return static_cast<int>(e);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2u * static_cast<unsigned>(num_sms / 2), 1u, 1u);
  cfg.blockDim = dim3(kThreads, 1u, 1u);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if ((e = cudaOccupancyMaxActiveClusters(&n, latent_pair_kernel<DecodeParams>, &cfg)) != cudaSuccess)
    return static_cast<int>(e);
  *out = n;
  return 0;
}

template <class P>
cudaError_t launch_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const P& p, int pairs,
                        cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(latent_pair_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  if (pairs <= 0) return cudaSuccess;
  latent_pair_kernel<P><<<2 * pairs, kThreads, SMEM_BYTES, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

cudaError_t launch_decode_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, int pairs, cudaStream_t stream) {
  return launch_pair(tq, tk, tv, p, pairs, stream);
}

cudaError_t launch_latent_prefill_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                       const LatentPrefillParams& p, int pairs, cudaStream_t stream) {
  return launch_pair(tq, tk, tv, p, pairs, stream);
}

cudaError_t launch_combine_pair(const DecodeParams& p, int pairs, float* o, uint16_t* o_bf16, float* lse,
                                cudaStream_t stream) {
  const int warps = p.planes * ((p.group + 31) / 32) * (DV / 32);
  // Programmatic stream serialization: the merge grid is set up while the
  // decode grid runs and starts as soon as that grid has completed.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((warps + kCombineWarps - 1) / kCombineWarps), 1u, 1u);
  cfg.blockDim = dim3(kCombineWarps * 32, 1u, 1u);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_pair_kernel, p, pairs, o, o_bf16, lse);
}

}  // namespace gbattn
