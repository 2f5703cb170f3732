// verify_common.cuh -- row statistics shared by the verifier's kernels, and
// the element-level arithmetic of the target and draft distributions
// (vLLM PR #65007 Part 2: temperature, exact top-p with 64-bit fixed-point
// masses, the rejection sampler).
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace dspark {

enum TgtMode : int32_t {
  kModeUnset = 0,
  kModeThreshold = 1,  // keep iff kd > kd_thr or (kd == kd_thr and id <= id_thr)
  kModeKeepAll = 2,    // no top-p truncation
  kModeOneHot = 3,     // no value above -inf: p = one-hot at column 0
  kModeGreedy = 4      // only amax_key is meaningful
};

struct TgtStats {
  float m;           // max of the scaled row (NaN read as -inf)
  float D;           // fp32(kept fixed-point mass) * 2^-40
  uint32_t kd_thr;   // ordered bits of the boundary logit
  int32_t id_thr;    // token id of the boundary element
  float p_d;         // p at this row's drafted token (rows k < K), else 0
  int32_t mode;
  unsigned long long amax_key;  // greedy rows: winner key of the raw row
};

struct DrfStats {
  float m;
  float D;
  float q_d;
  int32_t zero;  // no value above -inf: q = 0 everywhere
};

// xt = t / T (IEEE; T = 1 is exact without the division), NaN read as -inf.
__device__ __forceinline__ float scale_logit(float t, float T) {
  const float x = (T == 1.0f) ? t : __fdiv_rn(t, T);
  return (x != x) ? -INFINITY : x;
}


// rint(e * 2^40) for 0 <= e <= 1, round half to even, without a 64-bit
// float-to-integer conversion. v = e * 2^40 is exact in fp32. Below 2^23,
// adding 2^23 rounds v to an integer (nearest even) held in the mantissa
// bits; from 2^23 up, v is an integer: its 24-bit mantissa shifted left.
__device__ __forceinline__ unsigned long long fixed_mass(float e) {
  const float v = __fmul_rn(e, 0x1p40f);
  const uint32_t lo = __float_as_uint(__fadd_rn(v, 8388608.0f)) - 0x4B000000u;
  const uint32_t bits = __float_as_uint(v);
  const uint32_t sh = ((bits >> 23) - 150u) & 63u;
  const unsigned long long hi = static_cast<unsigned long long>((bits & 0x7FFFFFu) | 0x800000u) << sh;
  return v < 8388608.0f ? static_cast<unsigned long long>(lo) : hi;
}

// ordered bits of a non-NaN value (larger value -> larger key)
__device__ __forceinline__ uint32_t kd_of(float x) { return ordered_bits(x); }

// c * 2^32 >= (t_hi:t_lo), all unsigned
__device__ __forceinline__ bool reaches(unsigned long long c, unsigned long long t_hi,
                                        unsigned long long t_lo) {
  const unsigned long long c_hi = c >> 32, c_lo = c << 32;
  return c_hi > t_hi || (c_hi == t_hi && c_lo >= t_lo);
}

// rint(top_p * 2^32) from the fp32 bits (0 for top_p <= 0).
__device__ __forceinline__ unsigned long long topp_scaled(float top_p) {
  const uint32_t pb = __float_as_uint(top_p);
  const int ex = static_cast<int>((pb >> 23) & 0xFFu);
  if (!(top_p > 0.0f) || ex == 0) return 0ull;
  const unsigned long long mant = (pb & 0x7FFFFFu) | 0x800000u;
  const int sh = ex - 127 - 23 + 32;  // top_p * 2^32 = mant * 2^sh
  if (sh >= 0) return mant << sh;
  const int rs = -sh;
  if (rs > 24) return 0ull;
  const unsigned long long q = mant >> rs, rem = mant & ((1ull << rs) - 1ull),
                           half = 1ull << (rs - 1);
  return q + ((rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull);
}

}  // namespace dspark
