// Counter-based uniforms for speculative sampling on the device.
//
// Philox4x32 with 10 rounds, from its published definition (Salmon, Moraes,
// Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11): each
// round multiplies counter words 0 and 2 by two fixed odd constants; the next
// counter is (hi(B*x2) ^ x1 ^ k0, lo(B*x2), hi(A*x0) ^ x3 ^ k1, lo(A*x0));
// the key is advanced by two Weyl increments between rounds.
//
// Keying used by the verify walk: key = (seed lo, seed hi), counter =
// (step lo, step hi, node, child); u = (first word >> 8) * 2^-24, which is
// exact in fp32 and fp64.  The residual draw at a node uses child 0xffffffff.
#pragma once

#include <stdint.h>

namespace eagle {

constexpr uint32_t kPhiloxMulA = 0xD2511F53u;
constexpr uint32_t kPhiloxMulB = 0xCD9E8D57u;
constexpr uint32_t kPhiloxWeylA = 0x9E3779B9u;
constexpr uint32_t kPhiloxWeylB = 0xBB67AE85u;
constexpr uint32_t kResidualChild = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t philox_first_word(uint64_t seed, uint64_t step, uint32_t node,
                                                      uint32_t child) {
  uint32_t x0 = static_cast<uint32_t>(step), x1 = static_cast<uint32_t>(step >> 32);
  uint32_t x2 = node, x3 = child;
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += kPhiloxWeylA;
      k1 += kPhiloxWeylB;
    }
    const uint32_t hi_a = __umulhi(kPhiloxMulA, x0), lo_a = kPhiloxMulA * x0;
    const uint32_t hi_b = __umulhi(kPhiloxMulB, x2), lo_b = kPhiloxMulB * x2;
    x0 = hi_b ^ x1 ^ k0;
    x1 = lo_b;
    x2 = hi_a ^ x3 ^ k1;
    x3 = lo_a;
  }
  return x0;
}

__device__ __forceinline__ double philox_uniform(uint64_t seed, uint64_t step, uint32_t node,
                                                 uint32_t child) {
  return static_cast<double>(philox_first_word(seed, step, node, child) >> 8) * 0x1p-24;
}

}  // namespace eagle
