// philox.cuh -- Philox4x64-10 on the device.
//
// Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
// (SC'11): each of the 10 rounds multiplies counter words 0 and 2 by fixed
// 64-bit constants, xors the high halves of the 128-bit products with the other
// two words and the round key, and the key advances by two Weyl increments.
// The verify round keys the generator with the caller's seed and counts it by
// (position, lane), so the uniforms of a lane do not depend on how the work is
// split over threads, CTAs or launches.
#pragma once

#include <cstdint>

namespace specv {

struct Philox4x64Out {
  uint64_t w0, w1, w2, w3;
};

__device__ __forceinline__ Philox4x64Out philox4x64_10(uint64_t c0, uint64_t c1, uint64_t c2,
                                                       uint64_t c3, uint64_t k0, uint64_t k1) {
  constexpr uint64_t kMul0 = 0xD2E7470EE14C6C93ull;
  constexpr uint64_t kMul1 = 0xCA5A826395121157ull;
  constexpr uint64_t kWeyl0 = 0x9E3779B97F4A7C15ull;
  constexpr uint64_t kWeyl1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t lo0 = kMul0 * c0, hi0 = __umul64hi(kMul0, c0);
    const uint64_t lo1 = kMul1 * c2, hi1 = __umul64hi(kMul1, c2);
    const uint64_t n0 = hi1 ^ c1 ^ k0;
    const uint64_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += kWeyl0;
    k1 += kWeyl1;
  }
  return {c0, c1, c2, c3};
}

// Top 24 bits of a word as a float in [0, 1); exact in fp32.
__device__ __forceinline__ float philox_uniform24(uint64_t w) {
  return static_cast<float>(static_cast<uint32_t>(w >> 40)) * 5.9604644775390625e-8f;  // 2^-24
}

// Uniforms of (seed, lane, position): .x accepts/rejects the draft at
// `position`, .y drives an inverse-CDF draw made at `position`.
__device__ __forceinline__ float2 round_uniforms(uint64_t seed, uint32_t lane, uint32_t position) {
  const Philox4x64Out o = philox4x64_10(position, lane, 0, 0, seed, 0);
  return make_float2(philox_uniform24(o.w0), philox_uniform24(o.w1));
}

}  // namespace specv
