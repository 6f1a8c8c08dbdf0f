// attn_api.cu - the C ABI declared in include/gbattn.h: argument checks,
// tensor-map (TMA descriptor) encoding, dispatch to the prefill or the
// split-KV decode kernels, and the device error word.
//
// Tensor maps follow the "gl" global-layout idea of "Distilling a 4.5 hour
// CUDA talk", section 10 (a shape-annotated pointer from which the copy
// engine's descriptor is derived, with the swizzle chosen from the tile
// width): every [B, H, N, d] tensor is described as a 3-D box grid
// (d, N, B*H) with 64-feature (128-byte) boxes and the 128-byte swizzle, so a
// tile that runs past N reads zeros instead of the next head's rows.  The
// prefill kernel takes 4-D maps (d, N, H, B), or (d, H, N, B) for the
// token-major [B, N, H, d] layout that a projection GEMM writes, so Q, K and V
// can be read where the QKV GEMM left them.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "gbattn.h"
#include "philox.cuh"
#include "gbgemm.h"
#include "gblayer.h"
#include "internal.h"

namespace gbattn {

// Error bits in [0]; the first timed-out wait's block, warp, barrier and
// parity in [1..4].
__device__ unsigned g_device_error[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};

namespace {

constexpr int kVersion = 100;
constexpr int kDefaultExp2Split = 0;
constexpr int kGemmGroupM = 16;   // row blocks of 256 per raster group of the CTA-pair GEMM
constexpr int kMaxDevices = 64;

thread_local char t_cuda_error[256] = "";

int cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(t_cuda_error, sizeof(t_cuda_error), "%s: %s", where, cudaGetErrorString(e));
  return ATTN_ERR_CUDA;
}

struct DeviceInfo {
  bool ready = false;
  int status = ATTN_OK;
  int num_sms = 0;
  unsigned* err = nullptr;
  // Stream-ordered pool for the split-KV workspace, created by decode_pool()
  // on the first decode call that needs it.  Its release threshold
  // is unlimited, so memory freed at the end of one call is reused by the
  // next instead of being unmapped at every synchronisation and mapped again
  // (which the default pool does, at about 0.1 ms per call for a 40 MB
  // workspace).
  cudaMemPool_t pool = nullptr;
  // Clusters of the CTA-pair decode kernel that fit on the device at once
  // (-1 until first asked).
  int decode_pairs = -1;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3) {
      std::snprintf(t_cuda_error, sizeof(t_cuda_error), "device %d is sm_%d%d; this library is built for sm_103a",
                    dev, major, minor);
      return ATTN_ERR_NO_DEVICE;
    }
    if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_device_error)) != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    d.err = static_cast<unsigned*>(p);
    if (g_encode == nullptr) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
        return cuda_fail(e == cudaSuccess ? cudaErrorNotSupported : e, "cuTensorMapEncodeTiled lookup");
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return ATTN_OK;
}

// The decode workspace pool of the current device, created on first use (only
// attn_fwd's split-KV decode takes workspace from it).
int decode_pool(DeviceInfo* d, cudaMemPool_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_mu);
  if (d->pool == nullptr) {
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if ((e = cudaMemPoolCreate(&pool, &props)) != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
    uint64_t keep = UINT64_MAX;
    if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return cuda_fail(e, "cudaMemPoolSetAttribute");
    }
    d->pool = pool;
  }
  *out = d->pool;
  return ATTN_OK;
}

// 3-D bf16 tensor map (inner features, rows, planes) with a 64 x box_rows x 1
// box and the 128-byte swizzle.
int make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t planes,
             uint64_t row_stride_bytes, uint64_t plane_stride_bytes, uint32_t box_rows) {
  cuuint64_t dims[3] = {inner, rows, planes};
  cuuint64_t strides[2] = {row_stride_bytes, plane_stride_bytes};
  cuuint32_t box[3] = {64u, box_rows, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(t_cuda_error, sizeof(t_cuda_error), "cuTensorMapEncodeTiled failed (CUresult %d)",
                  static_cast<int>(r));
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

// 4-D bf16 tensor map with a 64 x box1 x box2 x 1 box and the 128-byte
// swizzle.  Strides are in bytes, for dimensions 1..3.
int make_map4(CUtensorMap* m, const void* base, const uint64_t dims[4], const uint64_t strides[3], uint32_t box1,
              uint32_t box2) {
  cuuint64_t gd[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t gs[3] = {strides[0], strides[1], strides[2]};
  cuuint32_t box[4] = {64u, box1, box2, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gd, gs, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(t_cuda_error, sizeof(t_cuda_error), "cuTensorMapEncodeTiled (4-D) failed (CUresult %d)",
                  static_cast<int>(r));
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

// C [M, N] (bf16 or fp32) as a 2-D map with boxes of 32 rows x 128 bytes
// and the 128-byte swizzle: the GEMM's TMA-store epilogue.
int make_c_map(CUtensorMap* m, void* c, int M, int N, bool fp32) {
  const uint64_t es = fp32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
  cuuint64_t strides[1] = {es * static_cast<uint64_t>(N)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / es), 32u};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = g_encode(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c, dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(t_cuda_error, sizeof(t_cuda_error), "cuTensorMapEncodeTiled (C) failed (CUresult %d)",
                  static_cast<int>(r));
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

// Map of one prefill operand with H heads of N rows of d features per batch.
// Head-major [B, H, N, d] (ld == 0): dimensions (d, N, H, B), 128-row boxes
// along N.  Token-major (ld > 0 = elements from one token's row to the
// next): element (b, h, i, c) at base + (b * N + i) * ld + h * d + c,
// dimensions (d, H, N, B) so that the strides still grow with the dimension.
int make_prefill_map(CUtensorMap* m, const void* base, int B, int H, int N, int d, long long ld) {
  const uint64_t es = 2;
  if (ld == 0) {
    const uint64_t dims[4] = {static_cast<uint64_t>(d), static_cast<uint64_t>(N), static_cast<uint64_t>(H),
                              static_cast<uint64_t>(B)};
    const uint64_t st[3] = {es * d, es * d * N, es * d * N * H};
    return make_map4(m, base, dims, st, 128, 1);
  }
  const uint64_t dims[4] = {static_cast<uint64_t>(d), static_cast<uint64_t>(H), static_cast<uint64_t>(N),
                            static_cast<uint64_t>(B)};
  const uint64_t st[3] = {es * d, es * static_cast<uint64_t>(ld), es * static_cast<uint64_t>(ld) * N};
  return make_map4(m, base, dims, st, 1, 128);
}

// The latent kernel's maps: Q [q_planes, q_rows, 576] and K [k_planes,
// k_rows, 576] bf16, each seen as (64 features, rows, 9 chunks, planes) with
// the 128-byte chunk stride inside the 1152-byte row stride, so that one box
// of r rows x c chunks is c consecutive chunk images of r rows.
int make_latent_maps(LatentMaps* m, const void* q, uint64_t q_rows, uint64_t q_planes, const void* k, uint64_t k_rows,
                     uint64_t k_planes) {
  const uint64_t row = 576 * 2;
  const uint64_t qd[4] = {64, q_rows, 9, q_planes};
  const uint64_t qs[3] = {row, 128, row * q_rows};
  const uint64_t kd[4] = {64, k_rows, 9, k_planes};
  const uint64_t ks[3] = {row, 128, row * k_rows};
  int st;
  if ((st = make_map4(&m->q, q, qd, qs, kLatentQRows, kLatentQChunks)) != ATTN_OK) return st;
  if ((st = make_map4(&m->k5, k, kd, ks, kLatentKeyRows, 5)) != ATTN_OK) return st;
  if ((st = make_map4(&m->k4, k, kd, ks, kLatentKeyRows, 4)) != ATTN_OK) return st;
  return make_map4(&m->k1, k, kd, ks, kLatentKeyRows, 1);
}

// The CTA-pair decode's maps: Q [planes, group, 576] in boxes of 64 rows x 3
// chunks, and over K [planes, Nkv, 576] the score CTA's boxes of 64 keys x 3
// chunks and the value CTA's of 64 keys x 8 chunks (V).
int make_pair_maps(CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv, const void* q, uint64_t q_rows,
                   uint64_t q_planes, const void* k, uint64_t k_rows, uint64_t planes) {
  const uint64_t row = 576 * 2;
  const uint64_t qd[4] = {64, q_rows, 9, q_planes};
  const uint64_t qs[3] = {row, 128, row * q_rows};
  const uint64_t kd[4] = {64, k_rows, 9, planes};
  const uint64_t ks[3] = {row, 128, row * k_rows};
  int st;
  if ((st = make_map4(tq, q, qd, qs, kLatentKeyRows, kPairKeyChunks)) != ATTN_OK) return st;
  if ((st = make_map4(tk, k, kd, ks, kLatentKeyRows, kPairKeyChunks)) != ATTN_OK) return st;
  return make_map4(tv, k, kd, ks, kLatentKeyRows, kPairValueChunks);
}

// Which kernel runs the latent shape (decode and prefill): the CTA-pair
// kernel (score and value CTAs), or with ATTN_LATENT=single the one-CTA
// kernel that computes the score tile for both O halves (read at every call).
bool latent_use_pair() {
  const char* s = std::getenv("ATTN_LATENT");
  return !(s != nullptr && std::strcmp(s, "single") == 0);
}

// Clusters of the CTA-pair kernel that fit on the device at once (cached).
int latent_pairs(DeviceInfo* dev, int* out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev->decode_pairs < 0) {
    int n = 0;
    const int e = decode_pair_max_pairs(dev->num_sms, &n);
    if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "cudaOccupancyMaxActiveClusters");
    dev->decode_pairs = n;
  }
  if (dev->decode_pairs <= 0) return ATTN_ERR_UNSUPPORTED;
  *out = std::min(dev->decode_pairs, dev->num_sms / 2);
  return ATTN_OK;
}

// Shape of one split-KV decode launch: the kernel, its CTAs (single) or
// clusters (pair), and the workspace its partials need.
struct DecodePlan {
  bool pair = false;
  int grid = 0;          // CTAs (single) or CTA pairs (pair)
  int max_seg = 0;       // single: partial slots per CTA
  size_t rows = 0;       // partial rows (slots x 128)
  int cols = 0;          // partial O columns per row
  size_t floats() const { return rows * static_cast<size_t>(cols + 1); }
};

int plan_decode(DeviceInfo* dev, int planes, int tiles, DecodePlan* out) {
  DecodePlan pl;
  pl.pair = latent_use_pair();
  if (pl.pair) {
    int pairs = 0;
    const int st = latent_pairs(dev, &pairs);
    if (st != ATTN_OK) return st;
    const long long total = static_cast<long long>(planes) * tiles;
    pl.grid = static_cast<int>(std::min<long long>(total, pairs));
    pl.rows = static_cast<size_t>(decode_pair_slots(planes, pl.grid)) * 128;
    pl.cols = 512;
  } else {
    const long long total = 2LL * planes * tiles;
    pl.grid = static_cast<int>(std::min<long long>(total, dev->num_sms));
    pl.max_seg = decode_max_segments(planes, tiles, pl.grid);
    pl.rows = static_cast<size_t>(pl.grid) * pl.max_seg * 128;
    pl.cols = 256;
  }
  *out = pl;
  return ATTN_OK;
}

// The decode kernel and the combine of `pl` on checked arguments; `ws` holds
// pl.floats() floats.
int launch_decode_plan(const DecodePlan& pl, const void* q, const void* k, float* o32, uint16_t* o16, float* lse,
                       int group, int planes, int Nkv, float scale_log2, float* ws, DeviceInfo* dev,
                       cudaStream_t stream) {
  DecodeParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.planes = planes;
  p.group = group;
  p.Nkv = Nkv;
  p.tiles = decode_tiles(Nkv);
  p.max_seg = pl.max_seg;
  p.scale_log2 = scale_log2;
  p.err = dev->err;
  p.o_part = ws;
  p.lse_part = ws + pl.rows * static_cast<size_t>(pl.cols);
  int st;
  cudaError_t e;
  if (pl.pair) {
    CUtensorMap tq, tk, tv;
    if ((st = make_pair_maps(&tq, &tk, &tv, q, group, planes, k, Nkv, planes)) != ATTN_OK) return st;
    if ((e = launch_decode_pair(tq, tk, tv, p, pl.grid, stream)) != cudaSuccess) return cuda_fail(e, "decode launch");
    if ((e = launch_combine_pair(p, pl.grid, o32, o16, lse, stream)) != cudaSuccess)
      return cuda_fail(e, "combine launch");
    return ATTN_OK;
  }
  LatentMaps maps;
  if ((st = make_latent_maps(&maps, q, group, planes, k, Nkv, planes)) != ATTN_OK) return st;
  if ((e = launch_decode(maps, p, pl.grid, stream)) != cudaSuccess) return cuda_fail(e, "decode launch");
  if ((e = launch_combine(p, pl.grid, o32, o16, lse, stream)) != cudaSuccess) return cuda_fail(e, "combine launch");
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool env_flag(const char* name) {
  const char* s = std::getenv(name);
  return s != nullptr && s[0] == '1';
}

// Share of the softmax's exponentials evaluated on the FMA pipe instead of
// the SFU: ATTN_EXP2_SPLIT=4 or 8 puts one pair in four or eight there
// (read at every call); anything else, or unset, keeps them all on the SFU.
int exp2_split() {
  const char* s = std::getenv("ATTN_EXP2_SPLIT");
  if (s == nullptr) return kDefaultExp2Split;
  const int v = std::atoi(s);
  return (v == 4 || v == 8) ? v : 0;
}

// Key-split units for problems under one wave (d = 64): on unless
// ATTN_PREFILL_KVSPLIT=0 (read at every call).
bool prefill_kv_split_enabled() {
  const char* s = std::getenv("ATTN_PREFILL_KVSPLIT");
  return s == nullptr || s[0] != '0';
}

bool check_env() {
  static const bool on = [] {
    const char* s = std::getenv("ATTN_CHECK");
    return s != nullptr && s[0] == '1';
  }();
  return on;
}

int read_device_error(cudaStream_t stream, unsigned* err, int reset) {
  unsigned h[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
  cudaError_t e = cudaMemcpyAsync(h, err, sizeof(h), cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(error word)");
  if (reset) {
    if ((e = cudaMemsetAsync(err, 0, sizeof(h), stream)) != cudaSuccess)
      return cuda_fail(e, "cudaMemsetAsync(error word)");
  }
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (h[0] == 0u) return ATTN_OK;
  std::snprintf(t_cuda_error, sizeof(t_cuda_error),
                "a kernel wait gave up: block %u warp %u barrier at shared offset 0x%x parity %u", h[1], h[2],
                h[3], h[4]);
  return ATTN_ERR_TIMEOUT;
}

}  // namespace
}  // namespace gbattn

using namespace gbattn;

extern "C" {

int attn_version(void) { return kVersion; }

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "kernel wait timed out";
    case ATTN_ERR_NO_DEVICE: return "no sm_103 device";
    case ATTN_ERR_SCRATCH_LIMIT: return "problem needs more than the fixed static scratch";
    default: return "unknown status";
  }
}

const char* attn_last_cuda_error(void) { return t_cuda_error; }

size_t attn_decode_workspace_bytes(int B, int Hkv, int Nkv) {
  if (B <= 0 || Hkv <= 0 || Nkv <= 0) return 0;
  DeviceInfo* d = nullptr;
  if (device_info(&d) != ATTN_OK) return 0;
  DecodePlan pl;
  if (plan_decode(d, B * Hkv, decode_tiles(Nkv), &pl) != ATTN_OK) return 0;
  return pl.floats() * sizeof(float);
}

int attn_check_device(attn_stream_t stream, int reset) {
  DeviceInfo* d = nullptr;
  int st = device_info(&d);
  if (st != ATTN_OK) return st;
  return read_device_error(reinterpret_cast<cudaStream_t>(stream), d->err, reset);
}

}  // extern "C"

namespace {

// Token strides (elements) of Q, K, V and O; all zero = head-major
// [B, H, N, d] for every operand.
struct PrefillLayout {
  long long q_ld, k_ld, v_ld, o_ld;
};

// Dropout of the prefill kernel: 8-bit threshold (0 = none) and seed.
struct Dropout {
  uint32_t t;
  unsigned long long seed;
};

// The prefill kernel (d 64 or 128, d_v == d) on checked arguments.
int run_prefill(const void* q, const void* k, const void* v, float* o32, uint16_t* o16, float* lse, int B, int Hq,
                int Hkv, int Nq, int Nkv, int d, int causal, float scale_log2, const PrefillLayout& lay,
                const Dropout& drop, DeviceInfo* dev, cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  int st;
  if ((st = make_prefill_map(&tq, q, B, Hq, Nq, d, lay.q_ld)) != ATTN_OK) return st;
  if ((st = make_prefill_map(&tk, k, B, Hkv, Nkv, d, lay.k_ld)) != ATTN_OK) return st;
  if ((st = make_prefill_map(&tv, v, B, Hkv, Nkv, d, lay.v_ld)) != ATTN_OK) return st;
  PrefillParams p{};
  p.o = o32;
  p.o_bf16 = o16;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Nq = Nq;
  p.Nkv = Nkv;
  p.d_v = d;
  p.token_major = lay.q_ld != 0 ? 1 : 0;
  if (lay.o_ld == 0) {
    p.o_sr = d;
    p.o_sh = static_cast<long long>(Nq) * d;
    p.o_sb = p.o_sh * Hq;
  } else {
    p.o_sr = lay.o_ld;
    p.o_sh = d;
    p.o_sb = lay.o_ld * Nq;
  }
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale_log2;
  p.seed_lo = static_cast<uint32_t>(drop.seed & 0xFFFFFFFFull);
  p.seed_hi = static_cast<uint32_t>(drop.seed >> 32);
  philox_round_keys(p.seed_lo, p.seed_hi, p.round_keys);
  p.drop_t = drop.t;
  p.drop_scale = static_cast<float>(256.0 / (256.0 - static_cast<double>(drop.t)));
  // Two 128-row tiles per unit (they ping-pong on the tensor core); one when
  // two-tile units would leave SMs idle, so that more SMs share the work.
  p.tiles_per_unit = (static_cast<long long>(B) * Hq * ((Nq + 255) / 256) < dev->num_sms) ? 1 : 2;
  // With one tile per unit the second tile slot would idle: at d = 64 it
  // takes the second half of the unit's key tiles instead (the merge buffer
  // fits beside the d = 64 rings only).
  p.kv_split = (p.tiles_per_unit == 1 && d == 64 && prefill_kv_split_enabled()) ? 1 : 0;
  p.nqb = (Nq + 128 * p.tiles_per_unit - 1) / (128 * p.tiles_per_unit);
  p.nkv_tiles = (Nkv + 127) / 128;
  p.num_units = B * Hq * p.nqb;
  p.exp2_split = exp2_split();
  p.err = dev->err;
  cudaError_t e;
  if ((e = launch_prefill(d, tq, tk, tv, p, dev->num_sms, stream)) != cudaSuccess)
    return cuda_fail(e, "prefill launch");
  return ATTN_OK;
}

// attn_fwd, attn_fwd_bf16out and attn_fwd_dropout: O is written as fp32
// (o32) or bf16 (o16); `drop` is applied by the prefill kernel only.
int attn_fwd_impl(const void* q, const void* k, const void* v, float* o32, uint16_t* o16, float* lse, int B, int Hq,
                  int Hkv, int Nq, int Nkv, int d_qk, int d_v, int causal, float scale, attn_stream_t stream_,
                  const Dropout& drop = Dropout{0u, 0ull}) {
  t_cuda_error[0] = '\0';
  const void* o = o32 != nullptr ? static_cast<const void*>(o32) : static_cast<const void*>(o16);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // ---------------------------------------------------------------- checks
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nkv <= 0 || d_qk <= 0 || d_v <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  const bool v_aliases_k = (v == k) && (d_v < d_qk);
  if (v == k && d_v > d_qk) return ATTN_ERR_INVALID_ARG;
  // sizes must fit the kernels' 32-bit row indexing
  if (static_cast<long long>(B) * Hq * Nq >= (1LL << 31) || static_cast<long long>(B) * Hkv * Nkv >= (1LL << 31))
    return ATTN_ERR_UNSUPPORTED;

  const bool prefill = (d_qk == d_v) && (d_qk == 64 || d_qk == 128);
  const bool latent = (d_qk == 576 && d_v == 512);
  if (!prefill && !latent) return ATTN_ERR_UNSUPPORTED;
  if (drop.t != 0u && !prefill) return ATTN_ERR_UNSUPPORTED;
  if (latent && !v_aliases_k) return ATTN_ERR_UNSUPPORTED;
  // One query per sequence sees every key under the bottom-right causal
  // alignment, so the causal flag changes nothing for the split-KV decode.
  const bool decode = latent && Nq == 1 && Hq / Hkv <= 128;

  DeviceInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != ATTN_OK) return st;

  const float scale_log2 = scale * 1.4426950408889634f;
  cudaError_t e;

  if (prefill) {
    const PrefillLayout lay{0, 0, 0, 0};
    if ((st = run_prefill(q, k, v, o32, o16, lse, B, Hq, Hkv, Nq, Nkv, d_qk, causal, scale_log2, lay, drop, dev,
                          stream)) != ATTN_OK)
      return st;
  } else if (!decode) {
    // latent shape, Nq > 1: the latent kernel in prefill mode
    LatentPrefillParams p{};
    p.q = static_cast<const uint16_t*>(q);
    p.o = o32;
    p.o_bf16 = o16;
    p.lse = lse;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Nq = Nq;
    p.Nkv = Nkv;
    p.causal = causal ? 1 : 0;
    p.tiles = decode_tiles(Nkv);
    p.nqb = (Nq + 127) / 128;
    p.scale_log2 = scale_log2;
    p.err = dev->err;
    if (latent_use_pair()) {
      int pairs = 0;
      if ((st = latent_pairs(dev, &pairs)) != ATTN_OK) return st;
      p.num_units = B * Hq * p.nqb;
      CUtensorMap tq, tk, tv;
      if ((st = make_pair_maps(&tq, &tk, &tv, q, Nq, static_cast<uint64_t>(B) * Hq, k, Nkv,
                               static_cast<uint64_t>(B) * Hkv)) != ATTN_OK)
        return st;
      if ((e = launch_latent_prefill_pair(tq, tk, tv, p, std::min(pairs, p.num_units), stream)) != cudaSuccess)
        return cuda_fail(e, "latent prefill launch");
    } else {
      LatentMaps maps;
      if ((st = make_latent_maps(&maps, q, Nq, static_cast<uint64_t>(B) * Hq, k, Nkv,
                                 static_cast<uint64_t>(B) * Hkv)) != ATTN_OK)
        return st;
      p.num_units = 2 * B * Hq * p.nqb;
      if ((e = launch_latent_prefill(maps, p, dev->num_sms, stream)) != cudaSuccess)
        return cuda_fail(e, "latent prefill launch");
    }
  } else {
    const int group = Hq / Hkv;
    const int planes = B * Hkv;
    DecodePlan pl;
    if ((st = plan_decode(dev, planes, decode_tiles(Nkv), &pl)) != ATTN_OK) return st;
    cudaMemPool_t pool = nullptr;
    if ((st = decode_pool(dev, &pool)) != ATTN_OK) return st;
    void* ws = nullptr;
    if ((e = cudaMallocFromPoolAsync(&ws, pl.floats() * sizeof(float), pool, stream)) != cudaSuccess)
      return cuda_fail(e, "cudaMallocFromPoolAsync(decode workspace)");
    if ((st = launch_decode_plan(pl, q, k, o32, o16, lse, group, planes, Nkv, scale_log2, static_cast<float*>(ws),
                                 dev, stream)) != ATTN_OK) {
      cudaFreeAsync(ws, stream);
      return st;
    }
    if ((e = cudaFreeAsync(ws, stream)) != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(decode workspace)");
  }

  if (check_env()) return read_device_error(stream, dev->err, 0);
  return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, float* o, float* lse, int B, int Hq, int Hkv, int Nq,
             int Nkv, int d_qk, int d_v, int causal, float scale, attn_stream_t stream) {
  return attn_fwd_impl(q, k, v, o, nullptr, lse, B, Hq, Hkv, Nq, Nkv, d_qk, d_v, causal, scale, stream);
}

int gemm_bf16_nt(const void* a, const void* b, void* c, int M, int N, int K, int c_fp32, attn_stream_t stream_) {
  t_cuda_error[0] = '\0';
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (a == nullptr || b == nullptr || c == nullptr) return ATTN_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || K % 8 != 0 || N % 2 != 0) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || !aligned16(c)) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(M) * K >= (1LL << 31) || static_cast<long long>(N) * K >= (1LL << 31) ||
      static_cast<long long>(M) * N >= (1LL << 31))
    return ATTN_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != ATTN_OK) return st;
  CUtensorMap ta, tb;
  const uint64_t rs = static_cast<uint64_t>(K) * 2;
  const bool use_pair = gemm_use_pair(M) && !env_flag("ATTN_GEMM_SINGLE_CTA");
  if ((st = make_map(&ta, a, K, M, 1, rs, rs * M, gemm_tile_rows())) != ATTN_OK) return st;
  if ((st = make_map(&tb, b, K, N, 1, rs, rs * N, gemm_b_box_rows(use_pair))) != ATTN_OK) return st;
  GemmParams p{};
  p.c = c;
  p.M = M;
  p.N = N;
  p.K = K;
  p.c_fp32 = c_fp32 ? 1 : 0;
  const int rows_per_tile = use_pair ? 2 * gemm_tile_rows() : gemm_tile_rows();
  p.tiles_m = (M + rows_per_tile - 1) / rows_per_tile;
  p.tiles_n = (N + gemm_tile_cols() - 1) / gemm_tile_cols();
  p.num_tiles = p.tiles_m * p.tiles_n;
  {
    const char* s = std::getenv("ATTN_GEMM_GROUP_M");
    const int g = s != nullptr ? std::atoi(s) : 0;
    p.group_m = (g >= 1 && g <= 1024) ? g : kGemmGroupM;
  }
  p.err = dev->err;
  // The pair kernel writes C with TMA stores when C's row pitch is a
  // multiple of 16 bytes (ATTN_GEMM_DIRECT_STORE=1 keeps the register stores).
  CUtensorMap tc;
  const CUtensorMap* ptc = nullptr;
  if (use_pair && N % 8 == 0 && !env_flag("ATTN_GEMM_DIRECT_STORE")) {
    if ((st = make_c_map(&tc, c, M, N, c_fp32 != 0)) != ATTN_OK) return st;
    ptc = &tc;
  }
  cudaError_t e;
  if ((e = use_pair ? launch_gemm_pair(ta, tb, ptc, p, dev->num_sms, stream)
                    : launch_gemm(ta, tb, p, dev->num_sms, stream)) != cudaSuccess)
    return cuda_fail(e, "gemm launch");
  if (check_env()) return read_device_error(stream, dev->err, 0);
  return ATTN_OK;
}

int attn_fwd_bf16out(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Nq, int Nkv, int d_qk, int d_v, int causal, float scale, attn_stream_t stream) {
  if (o == nullptr) return ATTN_ERR_INVALID_ARG;
  return attn_fwd_impl(q, k, v, nullptr, static_cast<uint16_t*>(o), lse, B, Hq, Hkv, Nq, Nkv, d_qk, d_v, causal,
                       scale, stream);
}

int attn_fwd_dropout(const void* q, const void* k, const void* v, float* o, float* lse, int B, int Hq, int Hkv,
                     int Nq, int Nkv, int d_qk, int d_v, int causal, float scale, float p_drop,
                     unsigned long long seed, attn_stream_t stream) {
  t_cuda_error[0] = '\0';
  if (!(p_drop >= 0.f && p_drop < 1.f)) return ATTN_ERR_INVALID_ARG;   // also refuses NaN
  const double tf = std::floor(static_cast<double>(p_drop) * 256.0 + 0.5);
  if (tf >= 256.0) return ATTN_ERR_INVALID_ARG;                         // would drop every weight
  if (p_drop > 0.f && tf == 0.0) {
    std::snprintf(t_cuda_error, sizeof(t_cuda_error),
                  "p_drop %g is below the 8-bit resolution (1/512) and would drop nothing", p_drop);
    return ATTN_ERR_INVALID_ARG;
  }
  const Dropout drop{static_cast<uint32_t>(tf), seed};
  return attn_fwd_impl(q, k, v, o, nullptr, lse, B, Hq, Hkv, Nq, Nkv, d_qk, d_v, causal, scale, stream, drop);
}

int attn_fwd_bshd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                  int Nkv, int d, long long q_ld, long long k_ld, long long v_ld, long long o_ld, int o_fp32,
                  int causal, float scale, attn_stream_t stream_) {
  t_cuda_error[0] = '\0';
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nkv <= 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  // each token row holds its heads side by side, in whole 16-byte units
  const long long lds[4] = {q_ld, k_ld, v_ld, o_ld};
  const long long need[4] = {static_cast<long long>(Hq) * d, static_cast<long long>(Hkv) * d,
                             static_cast<long long>(Hkv) * d, static_cast<long long>(Hq) * d};
  for (int i = 0; i < 4; ++i)
    if (lds[i] < need[i] || lds[i] % 8 != 0) return ATTN_ERR_INVALID_ARG;
  // tensor-map strides stay below 2^40 bytes; query rows fit 32-bit indexing
  if (2 * q_ld * B * Nq >= (1LL << 40) || 2 * k_ld * B * Nkv >= (1LL << 40) || 2 * v_ld * B * Nkv >= (1LL << 40))
    return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq * Nq >= (1LL << 31)) return ATTN_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != ATTN_OK) return st;
  const PrefillLayout lay{q_ld, k_ld, v_ld, o_ld};
  float* o32 = o_fp32 ? static_cast<float*>(o) : nullptr;
  uint16_t* o16 = o_fp32 ? nullptr : static_cast<uint16_t*>(o);
  if ((st = run_prefill(q, k, v, o32, o16, lse, B, Hq, Hkv, Nq, Nkv, d, causal, scale * 1.4426950408889634f, lay,
                        Dropout{0u, 0ull}, dev, stream)) != ATTN_OK)
    return st;
  if (check_env()) return read_device_error(stream, dev->err, 0);
  return ATTN_OK;
}

int attn_layer_fwd(const void* x, const void* w_qkv, const void* w_o, void* qkv, void* o, void* y, float* lse, int B,
                   int N, int d_model, int Hq, int Hkv, int d, int causal, float scale, int y_fp32,
                   attn_stream_t stream) {
  t_cuda_error[0] = '\0';
  if (x == nullptr || w_qkv == nullptr || w_o == nullptr || qkv == nullptr || o == nullptr || y == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || N <= 0 || d_model <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  const long long tokens = static_cast<long long>(B) * N;
  const long long nqkv = static_cast<long long>(Hq + 2 * Hkv) * d;
  const long long nq = static_cast<long long>(Hq) * d;
  if (tokens >= (1LL << 31) || nqkv >= (1LL << 31)) return ATTN_ERR_UNSUPPORTED;
  const uint16_t* base = static_cast<const uint16_t*>(qkv);
  int st;
  // QKV = X W_qkv^T: one token per row, the Q heads, then the K heads, then
  // the V heads side by side
  if ((st = gemm_bf16_nt(x, w_qkv, qkv, static_cast<int>(tokens), static_cast<int>(nqkv), d_model, 0, stream)) !=
      ATTN_OK)
    return st;
  // attention straight on the GEMM's output rows; O token-major [B*N, Hq*d]
  if ((st = attn_fwd_bshd(base, base + nq, base + nq + static_cast<long long>(Hkv) * d, o, lse, B, Hq, Hkv, N, N, d,
                          nqkv, nqkv, nqkv, nq, 0, causal, scale, stream)) != ATTN_OK)
    return st;
  // Y = O W_o^T
  return gemm_bf16_nt(o, w_o, y, static_cast<int>(tokens), d_model, static_cast<int>(nq), y_fp32, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// attn_decode_fwd_noalloc: the split-KV decode without any allocation.
//
// Its partial results live in one fixed array in device memory, declared
// here at file scope.  Every GPU that loads this library holds the array
// until the process exits; all calls on a device share it.
namespace gbattn {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(48) << 20;   // 48 MiB
__device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
int noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    float* ptr = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace
}  // namespace gbattn

extern "C" int attn_decode_fwd_noalloc(const void* q, const void* kv, float* o, float* lse, int B, int Hq, int Hkv,
                                       int Nkv, float scale, attn_stream_t stream_) {
  t_cuda_error[0] = '\0';
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (q == nullptr || kv == nullptr || o == nullptr) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nkv <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  if (Hq / Hkv > 128) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hkv * Nkv >= (1LL << 31)) return ATTN_ERR_UNSUPPORTED;

  DeviceInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != ATTN_OK) return st;
  float* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != ATTN_OK) return st;

  const int group = Hq / Hkv;
  const int planes = B * Hkv;
  DecodePlan pl;
  if ((st = plan_decode(dev, planes, decode_tiles(Nkv), &pl)) != ATTN_OK) return st;
  const size_t need = pl.floats() * sizeof(float);
  if (need > kNoAllocScratchBytes) {
    std::snprintf(t_cuda_error, sizeof(t_cuda_error), "needs %zu bytes of scratch, the static array holds %zu", need,
                  kNoAllocScratchBytes);
    return ATTN_ERR_SCRATCH_LIMIT;
  }
  // Every slot the combine kernel reads is written first by the decode
  // kernel in the same call, so nothing needs clearing between calls.
  if ((st = launch_decode_plan(pl, q, kv, o, nullptr, lse, group, planes, Nkv, scale * 1.4426950408889634f, scratch,
                               dev, stream)) != ATTN_OK)
    return st;
  if (check_env()) return read_device_error(stream, dev->err, 0);
  return ATTN_OK;
}
