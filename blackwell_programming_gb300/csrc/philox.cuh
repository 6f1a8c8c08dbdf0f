// philox.cuh - the Philox4x32-10 counter-based generator on the device.
//
// Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2,
// 3" (SC 2011): a 128-bit counter (x, y, z, w) and a 64-bit key (k0, k1);
// each of ten rounds multiplies x and z by two fixed odd 32-bit constants,
// keeps both halves of each 64-bit product, and forms the next counter as
// (hi(z*M1) ^ y ^ k0, lo(z*M1), hi(x*M0) ^ w ^ k1, lo(x*M0)); between rounds
// the key advances by the two Weyl constants.  Every call is independent, so
// a thread draws the bits for any (batch, head, query, key block) directly.
#pragma once

#include <cstdint>

namespace gbattn {

constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

// The key of round r is (k0 + r W0, k1 + r W1) (mod 2^32).
__host__ __device__ inline void philox_round_keys(uint32_t k0, uint32_t k1, uint32_t (&rk)[20]) {
  for (int r = 0; r < 10; ++r) {
    rk[2 * r] = k0;
    rk[2 * r + 1] = k1;
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
}

// The same generator with the round keys given (philox_round_keys): each
// round is two 32 x 32 -> 64-bit multiplies and two three-input XORs.
__device__ __forceinline__ uint4 philox4x32_10_rk(uint4 c, const uint32_t (&rk)[20]) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = static_cast<uint64_t>(kPhiloxM0) * c.x;
    const uint64_t p1 = static_cast<uint64_t>(kPhiloxM1) * c.z;
    c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ rk[2 * r], static_cast<uint32_t>(p1),
                   static_cast<uint32_t>(p0 >> 32) ^ c.w ^ rk[2 * r + 1], static_cast<uint32_t>(p0));
  }
  return c;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    // one 32 x 32 -> 64-bit multiply per product gives both halves
    const uint64_t p0 = static_cast<uint64_t>(kPhiloxM0) * c.x;
    const uint64_t p1 = static_cast<uint64_t>(kPhiloxM1) * c.z;
    c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ k0, static_cast<uint32_t>(p1),
                   static_cast<uint32_t>(p0 >> 32) ^ c.w ^ k1, static_cast<uint32_t>(p0));
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
  return c;
}

}  // namespace gbattn
