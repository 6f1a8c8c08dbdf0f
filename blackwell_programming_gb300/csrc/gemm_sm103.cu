// gemm_sm103.cu - C = A B^T in bf16 with fp32 accumulation, for the
// projections that feed and drain the attention forward (the QKV and O
// projections of the decoder chain on "CS149 L11: Programming Specialized
// Hardware", section 6; the matrix-multiply kernel of its section 4 is the
// pages' model: a producer of tiles, a consumer that runs the tensor core, a
// pipeline of stages between them).
//
// A is [M, K] row-major (activations), B is [N, K] row-major (a linear layer's
// weight), C is [M, N] row-major in bf16 or fp32.
//
// How, on sm_103a:
//  * One persistent CTA per SM walks 128 x 256 output tiles in groups of
//    kGroupM row blocks (all column blocks of a group before the next group),
//    so that the A and B tiles a wave of CTAs works on stay in L2.
//  * Warp 5 is the TMA producer: per 64-deep K step it loads a 128 x 64 A box
//    and a 256 x 64 B box (128-byte swizzle) into one of kStages ring stages.
//  * Warp 4 issues tcgen05.mma (M 128, N 256, K 16: four per stage, one elect
//    each group of four) into one of two 256-column TMEM accumulators, so
//    that the epilogue of one tile runs while the next tile accumulates.
//  * Warps 0-3 are the epilogue: each reads its 32 accumulator rows in the
//    16x256b shape (8 rows x 32 bytes per store instruction of the warp),
//    converts and stores C, then hands the accumulator back.
#include "internal.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr int kGroupM = 16;
constexpr int kThreads = 192;
constexpr int kMmaWarp = 4;
constexpr int kTmaWarp = 5;
constexpr uint32_t kFull = 0xFFFFFFFFu;

constexpr uint32_t A_BYTES = BM * BK * 2;   // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;   // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t OFF_BAR = kStages * STAGE_BYTES;
constexpr int B_FULL = 0, B_EMPTY = kStages, B_ACCFULL = 2 * kStages, B_ACCEMPTY = B_ACCFULL + 2,
              B_DRAIN = B_ACCEMPTY + 2, NUM_BARS = B_DRAIN + 1;
constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;   // + slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, false, false);

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(kFull, ok);
}

// Tile t -> (row block, column block): groups of kGroupM row blocks, the row
// block fastest inside a group.
__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& mb, int& nb) {
  const int per_group = kGroupM * p.tiles_n;
  const int g = t / per_group;
  const int first = g * kGroupM;
  const int gsize = min(p.tiles_m - first, kGroupM);
  const int in = t - g * per_group;
  mb = first + in % gsize;
  nb = in / gsize;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC + 4);
  const WaitCtx wctx{abort_flag, p.err};
  const uint32_t warp = warp_id(), lane = lane_id();
  const int kblocks = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(B_ACCFULL + a), 1);
      mbar_init(bar(B_ACCEMPTY + a), 4);
    }
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
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      const uint64_t pol = l2_policy_evict_last();   // tiles are re-read by the other CTAs of a group
      int s = 0;
      uint32_t ph = 0;
      uint32_t filled = 0u, fill_par = 0u;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, p, mb, nb);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!(ok = mbar_wait(bar(B_EMPTY + s), ph ^ 1u, wctx))) break;
          const uint32_t st = sbase + s * STAGE_BYTES;
          mbar_arrive_expect_tx(bar(B_FULL + s), STAGE_BYTES);
          filled |= 1u << s;
          fill_par = (fill_par & ~(1u << s)) | (ph << s);
          tma_load_3d(st, &tmA, bar(B_FULL + s), kb * BK, mb * BM, 0, pol);
          tma_load_3d(st + A_BYTES, &tmB, bar(B_FULL + s), kb * BK, nb * BN, 0, pol);
          if (++s == kStages) { s = 0; ph ^= 1u; }
        }
      }
      // Every issued copy must have landed before the CTA may exit.
      for (int b = 0; b < kStages; ++b)
        if ((filled >> b) & 1u) mbar_wait_drain(bar(B_FULL + b), (fill_par >> b) & 1u);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issuer (whole warp)
    int s = 0;
    uint32_t ph = 0;
    uint32_t aeph = 0u;   // bit a: parity of accumulator a's next "empty" wait
    const uint64_t a_desc0 = smem_desc_sw128(sbase, 16, 1024);
    const uint64_t b_desc0 = smem_desc_sw128(sbase + A_BYTES, 16, 1024);
    bool ok = true;
    int i = 0;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++i) {
      const int a = i & 1;
      // the epilogue has read this accumulator's previous tile
      if (!(ok = warp_wait(bar(B_ACCEMPTY + a), ((aeph >> a) & 1u) ^ 1u, wctx))) break;
      aeph ^= 1u << a;
      tc_fence_after();
      const uint32_t d = tm + a * BN;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!(ok = warp_wait(bar(B_FULL + s), ph, wctx))) break;
        tc_fence_after();
        const uint64_t ad = a_desc0 + ((s * STAGE_BYTES) >> 4);
        const uint64_t bd = b_desc0 + ((s * STAGE_BYTES) >> 4);
        uint64_t da[4], db[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          da[kk] = ad + kk * 2;   // +32 bytes per 16-deep step inside the 128-byte swizzled row
          db[kk] = bd + kk * 2;
        }
        mma_ss_warp4(d, da, db, IDESC, kb > 0 ? 1u : 0u);
        mma_commit_warp(bar(B_EMPTY + s));
        if (++s == kStages) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
      mma_commit_warp(bar(B_ACCFULL + a));
    }
    mma_commit_warp(bar(B_DRAIN));
    mbar_wait_drain(bar(B_DRAIN), 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t quad = warp;   // warps 0-3 own TMEM lanes 32*warp .. +31
    uint32_t afph = 0u;   // bit a: parity of accumulator a's next "full" wait
    bool ok = true;
    int i = 0;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++i) {
      const int a = i & 1;
      int mb, nb;
      tile_coords(t, p, mb, nb);
      if (!(ok = warp_wait(bar(B_ACCFULL + a), (afph >> a) & 1u, wctx))) break;
      afph ^= 1u << a;
      tc_fence_after();
      const int col0 = nb * BN + 2 * static_cast<int>(lane & 3);
#pragma unroll 1
      for (int hl = 0; hl < 2; ++hl) {
        const int ra = mb * BM + static_cast<int>(quad * 32 + hl * 16 + (lane >> 2));   // rows ra and ra + 8
        const bool la = ra < p.M, lb = ra + 8 < p.M;
#pragma unroll 1
        for (int ch = 0; ch < BN / 64; ++ch) {
          uint32_t r[32];
          tmem_ld16x256b_x8(tm + ((quad * 32u + hl * 16u) << 16) + a * BN + ch * 64, r);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int col = col0 + ch * 64 + 8 * k;
            if (col >= p.N) continue;   // N is even, so col + 1 < N too
            const float a0 = __uint_as_float(r[4 * k]), a1 = __uint_as_float(r[4 * k + 1]);
            const float b0 = __uint_as_float(r[4 * k + 2]), b1 = __uint_as_float(r[4 * k + 3]);
            if (p.c_fp32) {
              float* c = static_cast<float*>(p.c);
              if (la) *reinterpret_cast<float2*>(c + static_cast<size_t>(ra) * p.N + col) = make_float2(a0, a1);
              if (lb) *reinterpret_cast<float2*>(c + static_cast<size_t>(ra + 8) * p.N + col) = make_float2(b0, b1);
            } else {
              uint16_t* c = static_cast<uint16_t*>(p.c);
              if (la) *reinterpret_cast<uint32_t*>(c + static_cast<size_t>(ra) * p.N + col) = pack_bf16x2(a0, a1);
              if (lb) *reinterpret_cast<uint32_t*>(c + static_cast<size_t>(ra + 8) * p.N + col) = pack_bf16x2(b0, b1);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ACCEMPTY + a));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

// ------------------------------------------------------------------------
// CTA-pair variant: the two CTAs of a cluster share one 256 x 256 output
// tile.  Each CTA loads its own 128 rows of A and its half (128 rows) of B,
// and the even CTA issues M256 N256 K16 MMAs that read A from each CTA's
// shared memory and B from both halves and write each CTA's 128 rows of the
// accumulator into that CTA's TMEM.  Per CTA and 64-deep step this moves
// 32 KB from L2 for the same 128 x 256 x 64 products that take 48 KB above.
namespace pair {

constexpr int BM = 128;           // rows per CTA (the pair covers 256)
constexpr int BN = 256;           // columns per pair tile
constexpr int BNH = 128;          // rows of B each CTA loads
constexpr int kStages = 6;
constexpr uint32_t A_BYTES = BM * BK * 2;    // 16 KB
constexpr uint32_t B_BYTES = BNH * BK * 2;   // 16 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
// TMA-store epilogue staging: per epilogue warp two 4 KB buffers of 32 rows x
// 128 bytes (a box of 64 bf16 or 32 fp32 columns, 128-byte swizzle).
constexpr uint32_t OUT_WARP_BYTES = 32 * 128;
constexpr uint32_t OFF_OUT = kStages * STAGE_BYTES;
constexpr uint32_t OFF_BAR = OFF_OUT + 4 * 2 * OUT_WARP_BYTES;
constexpr int B_FULL = 0, B_EMPTY = kStages, B_ACCFULL = 2 * kStages, B_ACCEMPTY = B_ACCFULL + 2,
              B_DRAIN = B_ACCEMPTY + 2, NUM_BARS = B_DRAIN + 1;
constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
constexpr uint32_t IDESC = idesc_bf16_f32(2 * BM, BN, false, false);

// Tile t -> (256-row block, column block): groups of p.group_m row blocks,
// all column blocks of a group before the next, the row block fastest inside
// a group (a group's A rows stay in L2 while B's columns stream past them).
__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& mb, int& nb) {
  const int per_group = p.group_m * p.tiles_n;
  const int g = t / per_group;
  const int first = g * p.group_m;
  const int gsize = min(p.tiles_m - first, p.group_m);
  const int in = t - g * per_group;
  mb = first + in % gsize;
  nb = in / gsize;
}

__device__ __forceinline__ bool warp_wait_cl(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const bool ok = mbar_wait_cluster(bar, parity, w);
  return __all_sync(kFull, ok);
}

}  // namespace pair

// TMA_STORE: the epilogue stages each 32-row x 128-byte block of C in shared
// memory and writes it with a TMA store (C's row pitch a multiple of 16
// bytes); otherwise it stores straight from registers.
template <bool TMA_STORE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  // the pair's tile shape and layout (shadowing the single-CTA constants)
  constexpr int BM = pair::BM, BN = pair::BN, BNH = pair::BNH, kStages = pair::kStages;
  constexpr uint32_t A_BYTES = pair::A_BYTES, STAGE_BYTES = pair::STAGE_BYTES, OFF_BAR = pair::OFF_BAR,
                     OFF_MISC = pair::OFF_MISC, IDESC = pair::IDESC;
  constexpr int B_FULL = pair::B_FULL, B_EMPTY = pair::B_EMPTY, B_ACCFULL = pair::B_ACCFULL,
                B_ACCEMPTY = pair::B_ACCEMPTY, B_DRAIN = pair::B_DRAIN;
  using pair::tile_coords;
  using pair::warp_wait_cl;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC + 4);
  const WaitCtx wctx{abort_flag, p.err};
  const uint32_t warp = warp_id(), lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int kblocks = (p.K + BK - 1) / BK;
  const int cid = static_cast<int>(blockIdx.x >> 1), ncl = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(B_ACCFULL + a), 1);
      mbar_init(bar(B_ACCEMPTY + a), 8);   // four epilogue warps of each CTA
    }
    mbar_init(bar(B_DRAIN), 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();   // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tm = *tmem_slot;

  if (warp == kTmaWarp) {
    // ------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      const uint64_t pol = l2_policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = cid; t < p.num_tiles && ok; t += ncl) {
        int mb, nb;
        tile_coords(t, p, mb, nb);
        for (int kb = 0; kb < kblocks; ++kb) {
          // the pair's MMAs have read this stage (in both CTAs)
          if (!(ok = mbar_wait_cluster(bar(B_EMPTY + s), ph ^ 1u, wctx))) break;
          const uint32_t st = sbase + s * STAGE_BYTES;
          const uint32_t full = mapa_shared(bar(B_FULL + s), 0);   // counted on the even CTA's barrier
          if (leader) mbar_arrive_expect_tx(bar(B_FULL + s), 2 * STAGE_BYTES);
          tma_load_3d_pair(st, &tmA, full, kb * BK, mb * 2 * BM + static_cast<int>(rank) * BM, 0, pol);
          tma_load_3d_pair(st + A_BYTES, &tmB, full, kb * BK, nb * BN + static_cast<int>(rank) * BNH, 0, pol);
          if (++s == kStages) { s = 0; ph ^= 1u; }
        }
      }
      // Each stage's last fill lands before its MMAs run, and the MMA warp
      // drains every MMA before the pair's final cluster barrier, so no copy
      // of this CTA is in flight when it exits.
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------- MMA issuer (even CTA only)
    if (leader) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t aeph = 0u;
      const uint64_t a_desc0 = smem_desc_sw128(sbase, 16, 1024);
      const uint64_t b_desc0 = smem_desc_sw128(sbase + A_BYTES, 16, 1024);
      bool ok = true;
      int i = 0;
      for (int t = cid; t < p.num_tiles && ok; t += ncl, ++i) {
        const int a = i & 1;
        if (!(ok = warp_wait_cl(bar(B_ACCEMPTY + a), ((aeph >> a) & 1u) ^ 1u, wctx))) break;
        aeph ^= 1u << a;
        tc_fence_after();
        const uint32_t d = tm + a * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!(ok = warp_wait_cl(bar(B_FULL + s), ph, wctx))) break;
          tc_fence_after();
          const uint64_t ad = a_desc0 + ((s * STAGE_BYTES) >> 4);
          const uint64_t bd = b_desc0 + ((s * STAGE_BYTES) >> 4);
          uint64_t da[4], db[4];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            da[kk] = ad + kk * 2;
            db[kk] = bd + kk * 2;
          }
          mma_pair_ss_warp4(d, da, db, IDESC, kb > 0 ? 1u : 0u);
          mma_commit_pair_both(bar(B_EMPTY + s));
          if (++s == kStages) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        mma_commit_pair_both(bar(B_ACCFULL + a));
      }
      mma_commit_pair_local(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue (both CTAs)
    const uint32_t quad = warp;
    uint32_t afph = 0u;
    bool ok = true;
    int i = 0;
    int nstore = 0;   // TMA stores this warp has issued (lane 0)
    for (int t = cid; t < p.num_tiles && ok; t += ncl, ++i) {
      const int a = i & 1;
      int mb, nb;
      tile_coords(t, p, mb, nb);
      if (!(ok = warp_wait_cl(bar(B_ACCFULL + a), (afph >> a) & 1u, wctx))) break;
      afph ^= 1u << a;
      tc_fence_after();
      const int row0 = mb * 2 * BM + static_cast<int>(rank) * BM;
      if constexpr (TMA_STORE) {
        // Row `lane` of this warp's 32 rows, one 128-byte block of C at a
        // time: TMEM -> registers -> a swizzled staging buffer -> one TMA
        // store of 32 rows.  Two buffers per warp; a buffer is rewritten
        // once the store issued from it two blocks ago has read it.
        const int cols = p.c_fp32 ? 32 : 64;   // columns per 128-byte block
        const uint32_t rsw = lane & 7u;
        const uint32_t stage0 = sbase + pair::OFF_OUT + quad * 2u * pair::OUT_WARP_BYTES;
#pragma unroll 1
        for (int blk = 0; blk < BN / cols; ++blk, ++nstore) {
          const uint32_t buf = stage0 + static_cast<uint32_t>(nstore & 1) * pair::OUT_WARP_BYTES;
          uint32_t w[32];
          if (p.c_fp32) {
            float v[32];
            tmem_ld32(tm + ((quad * 32u) << 16) + a * BN + blk * 32, v);
#pragma unroll
            for (int k = 0; k < 32; ++k) w[k] = __float_as_uint(v[k]);
          } else {
            float v[32], u[32];
            tmem_ld32(tm + ((quad * 32u) << 16) + a * BN + blk * 64, v);
            tmem_ld32(tm + ((quad * 32u) << 16) + a * BN + blk * 64 + 32, u);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              w[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
              w[16 + k] = pack_bf16x2(u[2 * k], u[2 * k + 1]);
            }
          }
          if (nstore >= 2) {
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            st_shared_v4(buf + lane * 128u + ((static_cast<uint32_t>(u) ^ rsw) << 4), w[4 * u], w[4 * u + 1],
                         w[4 * u + 2], w[4 * u + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC, buf, nb * BN + blk * cols, row0 + static_cast<int>(quad) * 32);
            bulk_commit_group();
          }
        }
        // the accumulator is in the staging buffers (or already written)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(bar(B_ACCEMPTY + a), 0));
        continue;
      }
      const int col0 = nb * BN + 2 * static_cast<int>(lane & 3);
#pragma unroll 1
      for (int hl = 0; hl < 2; ++hl) {
        const int ra = row0 + static_cast<int>(quad * 32 + hl * 16 + (lane >> 2));
        const bool la = ra < p.M, lb = ra + 8 < p.M;
#pragma unroll 1
        for (int ch = 0; ch < BN / 64; ++ch) {
          uint32_t r[32];
          tmem_ld16x256b_x8(tm + ((quad * 32u + hl * 16u) << 16) + a * BN + ch * 64, r);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int col = col0 + ch * 64 + 8 * k;
            if (col >= p.N) continue;
            const float a0 = __uint_as_float(r[4 * k]), a1 = __uint_as_float(r[4 * k + 1]);
            const float b0 = __uint_as_float(r[4 * k + 2]), b1 = __uint_as_float(r[4 * k + 3]);
            if (p.c_fp32) {
              float* c = static_cast<float*>(p.c);
              if (la) *reinterpret_cast<float2*>(c + static_cast<size_t>(ra) * p.N + col) = make_float2(a0, a1);
              if (lb) *reinterpret_cast<float2*>(c + static_cast<size_t>(ra + 8) * p.N + col) = make_float2(b0, b1);
            } else {
              uint16_t* c = static_cast<uint16_t*>(p.c);
              if (la) *reinterpret_cast<uint32_t*>(c + static_cast<size_t>(ra) * p.N + col) = pack_bf16x2(a0, a1);
              if (lb) *reinterpret_cast<uint32_t*>(c + static_cast<size_t>(ra + 8) * p.N + col) = pack_bf16x2(b0, b1);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(bar(B_ACCEMPTY + a), 0));
    }
    // every store has written global memory before the CTA exits
    if (TMA_STORE && lane == 0) bulk_wait_group_all();
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync_all();   // no barrier or TMEM of either CTA is touched after this
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tm, 512);
  }
}

}  // namespace

int gemm_tile_rows() { return BM; }
int gemm_tile_cols() { return BN; }
int gemm_tile_depth() { return BK; }

bool gemm_use_pair(int M) { return M > BM; }
int gemm_b_box_rows(bool use_pair) { return use_pair ? pair::BNH : BN; }

cudaError_t launch_gemm_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap* tc,
                             const GemmParams& p, int num_sms, cudaStream_t stream) {
  const int clusters = min(p.num_tiles, num_sms / 2);
  cudaError_t e;
  if (tc != nullptr) {
    if ((e = cudaFuncSetAttribute(gemm_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(pair::SMEM_BYTES))) != cudaSuccess)
      return e;
    if (clusters <= 0) return cudaSuccess;
    gemm_pair_kernel<true><<<2 * clusters, kThreads, pair::SMEM_BYTES, stream>>>(ta, tb, *tc, p);
  } else {
    if ((e = cudaFuncSetAttribute(gemm_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(pair::SMEM_BYTES))) != cudaSuccess)
      return e;
    if (clusters <= 0) return cudaSuccess;
    gemm_pair_kernel<false><<<2 * clusters, kThreads, pair::SMEM_BYTES, stream>>>(ta, tb, ta, p);
  }
  return cudaGetLastError();
}

cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, int num_sms,
                        cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  const int grid = min(p.num_tiles, num_sms);
  if (grid <= 0) return cudaSuccess;
  gemm_kernel<<<grid, kThreads, SMEM_BYTES, stream>>>(ta, tb, p);
  return cudaGetLastError();
}

}  // namespace gbattn
