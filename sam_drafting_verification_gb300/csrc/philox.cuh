// philox.cuh -- device Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
// random numbers: as easy as 1, 2, 3", SC'11) and the uniform map used for the
// verification coins.  Written for the device independently of any host copy.
#pragma once

#include <cstdint>

namespace samspec {

struct Philox4 {
  uint32_t x[4];
};

// Ten rounds; the key is advanced by the Weyl constants after every round
// (the advance after the tenth round is never used).
__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                                 uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t a = c0, c = c2;
    const uint32_t lo_a = 0xD2511F53u * a, hi_a = __umulhi(0xD2511F53u, a);
    const uint32_t lo_c = 0xCD9E8D57u * c, hi_c = __umulhi(0xCD9E8D57u, c);
    c0 = hi_c ^ c1 ^ k0;
    c1 = lo_c;
    c2 = hi_a ^ c3 ^ k1;
    c3 = lo_a;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  Philox4 r;
  r.x[0] = c0;
  r.x[1] = c1;
  r.x[2] = c2;
  r.x[3] = c3;
  return r;
}

// ((w >> 9) + 0.5) * 2^-23: a value in (0, 1), exact in binary32.
__device__ __forceinline__ float unit_uniform(uint32_t w) {
  return (static_cast<float>(w >> 9) + 0.5f) * 1.1920928955078125e-07f;
}

// Coins of sequence b at draft position j: word 0 -> accept test, word 1 ->
// resample.  key = (seed lo, seed hi); counter = (j, b, step lo, step hi).
__device__ __forceinline__ void verify_coins(uint64_t seed, uint64_t step, uint32_t b, uint32_t j,
                                             float* u_accept, float* u_resample) {
  const Philox4 r = philox4x32_10(j, b, static_cast<uint32_t>(step),
                                  static_cast<uint32_t>(step >> 32), static_cast<uint32_t>(seed),
                                  static_cast<uint32_t>(seed >> 32));
  *u_accept = unit_uniform(r.x[0]);
  *u_resample = unit_uniform(r.x[1]);
}

}  // namespace samspec
