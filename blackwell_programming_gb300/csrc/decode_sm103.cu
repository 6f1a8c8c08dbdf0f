// decode_sm103.cu - split-KV attention decode for the latent head-dim shape
// (d_qk = 576, d_v = 512, V = the first 512 features of K), and the combine
// kernel that merges the splits.
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
// Roles: warp 5 = TMA producer (Q once per segment, K tiles through a ring),
// warp 4 = tcgen05 MMA issuer, warps 0-3 = softmax (one row per thread),
// O rescale and epilogue.
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int DQK = 576;
constexpr int DVH = 256;              // O columns per work item (half of d_v)
constexpr int BM = 128;               // rows = query heads of one KV head
constexpr int BN = 32;                // keys per K tile
constexpr int QCH = DQK / 64;         // 9 chunks of 64 features (128 bytes)
constexpr int KS = 2;                 // K stages
constexpr int kThreads = 192;
constexpr int kMmaWarp = 4;
constexpr int kTmaWarp = 5;
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kFull = 0xFFFFFFFFu;

constexpr uint32_t CHUNK_Q = BM * 128;              // 16 KB
constexpr uint32_t CHUNK_K = BN * 128;              // 4 KB
constexpr uint32_t Q_BYTES = QCH * CHUNK_Q;         // 147456
constexpr uint32_t K_BYTES = QCH * CHUNK_K;         // 36864
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
constexpr uint32_t OFF_BAR = OFF_K + KS * K_BYTES;
constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_KEMPTY = 2 + KS, B_SFULL = 2 + 2 * KS,
              B_PFULL = B_SFULL + 2, B_PVDONE = B_PFULL + 1, B_OFULL = B_PVDONE + 1, B_OEMPTY = B_OFULL + 1,
              B_DRAIN = B_OEMPTY + 1, NUM_BARS = B_DRAIN + 1;
constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t COL_S0 = 0;        // S buffers at columns 0 and 32
constexpr uint32_t COL_O = 256;
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
  int slot;     // partial slot within this CTA
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
    g = end;
    return true;
  }
};

__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + OFF_Q, sK = sbase + OFF_K;
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC + 4);
  const WaitCtx wctx{abort_flag, p.err};
  const uint32_t warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
    }
    mbar_init(bar(B_SFULL + 0), 1);
    mbar_init(bar(B_SFULL + 1), 1);
    mbar_init(bar(B_PFULL), 4);
    mbar_init(bar(B_PVDONE), 1);
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
      tma_prefetch_desc(&tmK);
      const uint64_t pol_k = l2_policy_evict_first();   // each K tile is read by the two halves, then dead
      const uint64_t pol_q = l2_policy_evict_last();
      int ks = 0;
      uint32_t kph = 0, qph = 0;
      int k_last[KS], q_last = -1;
      for (int s = 0; s < KS; ++s) k_last[s] = -1;
      SegmentWalker walk(p);
      Segment S;
      bool ok = true;
      while (ok && walk.next(S)) {
        if (!(ok = mbar_wait(bar(B_QEMPTY), qph ^ 1u, wctx))) break;
        qph ^= 1u;
        mbar_arrive_expect_tx(bar(B_QFULL), Q_BYTES);
        q_last = static_cast<int>(qph ^ 1u);
        for (int kc = 0; kc < QCH; ++kc)
          tma_load_3d(sQ + kc * CHUNK_Q, &tmQ, bar(B_QFULL), kc * 64, 0, S.plane, pol_q);
        for (int j = 0; j < S.n; ++j) {
          if (!(ok = mbar_wait(bar(B_KEMPTY + ks), kph ^ 1u, wctx))) break;
          mbar_arrive_expect_tx(bar(B_KFULL + ks), K_BYTES);
          k_last[ks] = static_cast<int>(kph);
          for (int kc = 0; kc < QCH; ++kc)
            tma_load_3d(sK + ks * K_BYTES + kc * CHUNK_K, &tmK, bar(B_KFULL + ks), kc * 64, (S.t0 + j) * BN,
                        S.plane, pol_k);
          if (++ks == KS) { ks = 0; kph ^= 1u; }
        }
      }
      if (q_last >= 0) mbar_wait_drain(bar(B_QFULL), static_cast<uint32_t>(q_last));
      for (int s = 0; s < KS; ++s)
        if (k_last[s] >= 0) mbar_wait_drain(bar(B_KFULL + s), static_cast<uint32_t>(k_last[s]));
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int ks = 0, prev = 0;
      uint32_t kph = 0, qph = 0, pph = 0, oeph = 0;
      SegmentWalker walk(p);
      Segment S;
      bool ok = true;
      while (ok && walk.next(S)) {
        if (!(ok = mbar_wait(bar(B_OEMPTY), oeph ^ 1u, wctx))) break;
        oeph ^= 1u;
        if (!(ok = mbar_wait(bar(B_QFULL), qph, wctx))) break;
        qph ^= 1u;
        tc_fence_after();
        for (int j = 0; j <= S.n; ++j) {
          if (j < S.n) {
            if (!(ok = mbar_wait(bar(B_KFULL + ks), kph, wctx))) break;
            tc_fence_after();
            const uint32_t kbase = sK + ks * K_BYTES;
            const uint32_t dS = tm + COL_S0 + (j & 1) * BN;
#pragma unroll 4
            for (int kk = 0; kk < DQK / 16; ++kk) {
              const uint32_t off = (kk & 3) * 32;
              mma_ss(dS, smem_desc_sw128(sQ + (kk >> 2) * CHUNK_Q + off, 16, 1024),
                     smem_desc_sw128(kbase + (kk >> 2) * CHUNK_K + off, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar(B_SFULL + (j & 1)));
            if (j == S.n - 1) mma_commit(bar(B_QEMPTY));
          }
          if (j >= 1) {
            if (!(ok = mbar_wait(bar(B_PFULL), pph, wctx))) break;
            pph ^= 1u;
            tc_fence_after();
            // V half = K features [256 * half, 256 * half + 256): chunks 4*half .. 4*half+3
            const uint32_t vbase = sK + prev * K_BYTES + (4 * S.half) * CHUNK_K;
            const uint32_t aP = tm + COL_S0 + ((j - 1) & 1) * BN;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_ts(tm + COL_O, aP + kk * 8, smem_desc_sw128(vbase + kk * 16 * 128, CHUNK_K, 1024), IDESC_PV,
                     (j - 1 > 0 || kk > 0) ? 1u : 0u);
            mma_commit(bar(B_PVDONE));
            mma_commit(bar(B_KEMPTY + prev));
          }
          if (j < S.n) {
            prev = ks;
            if (++ks == KS) { ks = 0; kph ^= 1u; }
          } else {
            mma_commit(bar(B_OFULL));
          }
        }
      }
      mma_commit(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------- softmax, rescale, epilogue
    const int r = static_cast<int>(warp * 32 + lane);
    const uint32_t lane_addr = (warp * 32u) << 16;
    const float sl2 = p.scale_log2;
    uint32_t sph[2] = {0, 0}, pvph = 0, ofph = 0;
    SegmentWalker walk(p);
    Segment S;
    bool ok = true;
    while (ok && walk.next(S)) {
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < S.n; ++j) {
        const int sb = j & 1;
        if (!(ok = warp_wait(bar(B_SFULL + sb), sph[sb], wctx))) break;
        sph[sb] ^= 1u;
        tc_fence_after();
        float v[32];
        tmem_ld32(tm + lane_addr + COL_S0 + sb * BN, v);
        const int key0 = (S.t0 + j) * BN;
        const bool ragged = key0 + BN > p.Nkv;
        if (ragged) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (key0 + i >= p.Nkv) v[i] = -INFINITY;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, v[i]);
        const float m_new = (mx == -INFINITY) ? -INFINITY : mx * sl2;
        float alpha = 1.f;
        const bool grow = m_new > m_used + kRescaleThreshold;
        if (grow) {
          alpha = ex2(m_used - m_new);
          m_used = m_new;
        }
        l *= alpha;
        if (j >= 1) {
          // O is only touched once the previous P.V has finished.
          if (!(ok = warp_wait(bar(B_PVDONE), pvph, wctx))) break;
          pvph ^= 1u;
          tc_fence_after();
          if (__any_sync(kFull, grow)) {
#pragma unroll 1
            for (int c = 0; c < DVH / 32; ++c) {
              float o[32];
              tmem_ld32(tm + lane_addr + COL_O + c * 32, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= alpha;
              tmem_st32(tm + lane_addr + COL_O + c * 32, o);
            }
          }
        }
        const float base = (m_used == -INFINITY) ? 0.f : m_used;
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float p0 = ex2(fmaf(v[2 * i], sl2, -base));
          float p1 = ex2(fmaf(v[2 * i + 1], sl2, -base));
          if (ragged) {
            if (key0 + 2 * i >= p.Nkv) p0 = 0.f;
            if (key0 + 2 * i + 1 >= p.Nkv) p1 = 0.f;
          }
          l += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tm + lane_addr + COL_S0 + sb * BN, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL));
      }
      if (!ok) break;
      if (!(ok = warp_wait(bar(B_OFULL), ofph, wctx))) break;
      ofph ^= 1u;
      // the last P.V of the segment also completed pv_done once
      if (!(ok = warp_wait(bar(B_PVDONE), pvph, wctx))) break;
      pvph ^= 1u;
      tc_fence_after();
      const size_t slot = static_cast<size_t>(blockIdx.x) * p.max_seg + S.slot;
      const bool live = r < p.group;
      float* orow = p.o_part + (slot * BM + r) * DVH;
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < DVH / 32; ++c) {
        float v[32];
        tmem_ld32(tm + lane_addr + COL_O + c * 32, v);
        if (live) {
          float4* dst = reinterpret_cast<float4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(v[4 * i] * inv_l, v[4 * i + 1] * inv_l, v[4 * i + 2] * inv_l, v[4 * i + 3] * inv_l);
        }
      }
      if (live) p.lse_part[slot * BM + r] = (l > 0.f) ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_OEMPTY));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

// One block per (half, plane); thread c owns O column half * 256 + c.  `grid`
// is the decode kernel's grid size, which fixes where the partials are.
__global__ void __launch_bounds__(DVH) combine_kernel(const DecodeParams p, int grid, float* o, float* lse) {
  const int half = blockIdx.x / p.planes;
  const int plane = blockIdx.x - half * p.planes;
  const int c = threadIdx.x;
  const long long tiles = p.tiles;
  const long long total = 2LL * p.planes * tiles;
  const long long sg = static_cast<long long>(half) * p.planes + plane;
  const long long gs = sg * tiles, ge = gs + tiles - 1;
  const int c_first = static_cast<int>(((gs + 1) * grid + total - 1) / total - 1);
  const int c_last = static_cast<int>(((ge + 1) * grid + total - 1) / total - 1);
  for (int r = 0; r < p.group; ++r) {
    float mx = -INFINITY;
    for (int cta = c_first; cta <= c_last; ++cta) {
      const long long b0 = range_begin(total, cta, grid), b1 = range_begin(total, cta + 1, grid);
      if (b1 <= b0) continue;
      const size_t slot = static_cast<size_t>(cta) * p.max_seg + static_cast<size_t>(sg - b0 / tiles);
      mx = fmaxf(mx, p.lse_part[slot * BM + r]);
    }
    float acc = 0.f, tot = 0.f;
    if (mx != -INFINITY) {
      for (int cta = c_first; cta <= c_last; ++cta) {
        const long long b0 = range_begin(total, cta, grid), b1 = range_begin(total, cta + 1, grid);
        if (b1 <= b0) continue;
        const size_t slot = static_cast<size_t>(cta) * p.max_seg + static_cast<size_t>(sg - b0 / tiles);
        const float w = expf(p.lse_part[slot * BM + r] - mx);
        tot += w;
        acc += w * p.o_part[(slot * BM + r) * DVH + c];
      }
    }
    const size_t row = static_cast<size_t>(plane) * p.group + r;
    o[row * (2 * DVH) + half * DVH + c] = (tot > 0.f) ? acc / tot : 0.f;
    if (half == 0 && c == 0 && lse != nullptr) lse[row] = (tot > 0.f) ? mx + logf(tot) : -INFINITY;
  }
}

}  // namespace

int decode_tiles(int Nkv) { return (Nkv + BN - 1) / BN; }

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

cudaError_t launch_decode(const CUtensorMap& tq, const CUtensorMap& tk, const DecodeParams& p, int grid,
                          cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  decode_kernel<<<grid, kThreads, SMEM_BYTES, stream>>>(tq, tk, p);
  return cudaGetLastError();
}

cudaError_t launch_combine(const DecodeParams& p, int grid, float* o, float* lse, cudaStream_t stream) {
  combine_kernel<<<2 * p.planes, DVH, 0, stream>>>(p, grid, o, lse);
  return cudaGetLastError();
}

}  // namespace gbattn
