// common.cuh -- device helpers shared by the Markov-step and verify kernels:
// the Philox4x32-10 noise generator, the winner key, fixed-point masses,
// mbarrier / bulk-copy wrappers with bounded waits, and the status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dspark.h"
#include "kernels.h"

namespace dspark {

// Noise streams (the header's "draft", "verifier categorical", "accept").
constexpr uint32_t kStreamDraft = 1u << 30;
constexpr uint32_t kStreamTarget = 0u;
constexpr uint32_t kStreamAccept = 1u << 29;

// One unit of exp-mass in the 64-bit fixed point of the top-p select.
constexpr int kFixShift = 40;

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies with the
// round multipliers, a half swap and a key xor; the key advances by the two
// Weyl increments between rounds.
// ---------------------------------------------------------------------------
struct U4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ U4 philox4x32_10(U4 c, uint32_t k0, uint32_t k1) {
  constexpr uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
  constexpr uint32_t kWeyl0 = 0x9E3779B9u, kWeyl1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = kMul0 * c.x, hi0 = __umulhi(kMul0, c.x);
    const uint32_t lo1 = kMul1 * c.z, hi1 = __umulhi(kMul1, c.z);
    U4 n;
    n.x = hi1 ^ c.y ^ k0;
    n.y = lo1;
    n.z = hi0 ^ c.w ^ k1;
    n.w = lo0;
    c = n;
    k0 += kWeyl0;
    k1 += kWeyl1;
  }
  return c;
}

// All four words of the counter block holding `col` (cols 4j..4j+3).
__device__ __forceinline__ U4 noise_block(uint64_t seed, int64_t pos,
                                          uint32_t col, uint32_t stream) {
  const uint64_t upos = static_cast<uint64_t>(pos);
  U4 c{col >> 2, static_cast<uint32_t>(upos), static_cast<uint32_t>(upos >> 32),
       stream};
  return philox4x32_10(c, static_cast<uint32_t>(seed),
                       static_cast<uint32_t>(seed >> 32));
}

__device__ __forceinline__ uint32_t pick_word(const U4& r, uint32_t j) {
  return j == 0 ? r.x : (j == 1 ? r.y : (j == 2 ? r.z : r.w));
}

// u = ((w >> 9) + 1/2) * 2^-23: every step is exact in fp32.
__device__ __forceinline__ float uniform_of(uint32_t w) {
  // 1 + k 2^-23 (k = w >> 9) from its bits, then minus (1 - 2^-24): the
  // exact result (k + 1/2) 2^-23 has at most 24 significant bits, so the one
  // rounding is exact and no integer conversion is needed
  return __fadd_rn(__uint_as_float(0x3F800000u | (w >> 9)), -0x1.fffffep-1f);
}

// ---- packed fp32 pairs (Blackwell f32x2 arithmetic, round to nearest) -------
// Each lane of a pair is one IEEE fp32 operation, so a pair gives the same
// bits as two scalar operations in one instruction.
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// round toward zero: with 2^23 added to a value in [0, 2^23), the sum holds
// the value's integer part in its low mantissa bits
__device__ __forceinline__ unsigned long long f2_add_rz(unsigned long long a,
                                                        unsigned long long b) {
  unsigned long long d;
  asm("add.rz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---- temperature: x = z / T, correctly rounded ------------------------------
// For a column with T in [2^-30, 2^30] and r = rn(1/T) (correctly rounded
// reciprocal), q = rn(z r) is within one ulp of z / T, the residual
// z - q T is exact in one FMA, and rn(q + (z - q T) r) is the correctly
// rounded quotient: Markstein's theorem (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990; also the FMA-division chapter of Muller et al.,
// "Handbook of Floating-Point Arithmetic"). The theorem needs every
// intermediate to stay normal, which |z| in [2^-60, 2^60] and T in
// [2^-30, 2^30] guarantee; other z (zeros, infinities, NaN, tiny or huge
// values) and columns whose T lies outside that range (`slow`) take the IEEE
// division itself. Two columns at a time, in packed pairs; the bits are
// those of z / T either way.
__device__ __forceinline__ bool temp_div_fast_ok(float z) {
  const float a = fabsf(z);
  return a >= 0x1p-60f && a <= 0x1p60f;
}
__device__ __forceinline__ unsigned long long temp_div2(unsigned long long z,
                                                        unsigned long long r,
                                                        unsigned long long neg_t, bool slow) {
  const unsigned long long q = f2_mul(z, r);
  const unsigned long long e = f2_fma(q, neg_t, z);  // z - q T, exact
  unsigned long long x = f2_fma(e, r, q);
  float z0, z1;
  f2_unpack(z, z0, z1);
  const bool bad = slow || !temp_div_fast_ok(z0) || !temp_div_fast_ok(z1);
  if (bad) {  // rare: this lane takes IEEE divisions
    float x0, x1, t0, t1;
    f2_unpack(x, x0, x1);
    f2_unpack(neg_t, t0, t1);
    if (slow || !temp_div_fast_ok(z0)) x0 = __fdiv_rn(z0, -t0);
    if (slow || !temp_div_fast_ok(z1)) x1 = __fdiv_rn(z1, -t1);
    x = f2_pack(x0, x1);
  }
  return x;
}
// T in the range where temp_div2's fast form holds.
__device__ __forceinline__ bool temp_div_t_ok(float T) {
  return T >= 0x1p-30f && T <= 0x1p30f;
}

// lg2.approx.f32: log2 with an absolute error of about 2^-22.6 on the
// mantissa part (plus the rounding of the fp32 result).
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// rcp.approx.ftz.f32: 1/x to about 1 ulp (x normal).
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Standard Gumbel variate g = -ln(-ln u) of the uniform of word w.
// E = -ln u is computed with small relative error on both sides of the
// range: for u > 3/4 from t = 1 - u (exact on the 2^-23 grid) by the series
// -ln(1 - t) = 2 atanh(s), s = t / (2 - t) <= 1/7 (t times an approximate
// reciprocal), to s^9; for u <= 3/4 as
// -ln 2 * lg2(u), where E >= 0.28 keeps the relative error near 4e-7. Then
// g = -ln 2 * lg2(E). The absolute error on g stays below about 1.3e-6 over
// the whole grid (checked against an fp64 evaluation in the tests).
__device__ __forceinline__ float gumbel_of(uint32_t w) {
  // -log u is 2 atanh(t / (2 - t)), t = 1 - u, for u > 3/4 (where log2 of u
  // near 1 would lose the relative accuracy of a small result) and
  // -ln2 * log2(u) below; both are computed and one is selected, so a warp
  // never diverges here
  constexpr float kLn2 = 0.693147180559945309f;
  const float u = uniform_of(w);
  const float t = __fsub_rn(1.0f, u);
  const float sr = __fmul_rn(t, rcp_approx(__fsub_rn(2.0f, t)));
  const float s2 = __fmul_rn(sr, sr);
  float p = __fmaf_rn(s2, 2.0f / 9.0f, 2.0f / 7.0f);  // 2 (1 + s^2/3 + s^4/5 + s^6/7 + s^8/9)
  p = __fmaf_rn(s2, p, 2.0f / 5.0f);
  p = __fmaf_rn(s2, p, 2.0f / 3.0f);
  p = __fmaf_rn(s2, p, 2.0f);
  const float e_near = __fmul_rn(sr, p);
  const float e_far = __fmul_rn(-kLn2, lg2_approx(u));
  const float E = u > 0.75f ? e_near : e_far;
  return __fmul_rn(-kLn2, lg2_approx(E));
}

// E = -ln u of two words at once, the first half of gumbel_of (the same
// operations lane by lane, in packed pairs): an exponential variate.
__device__ __forceinline__ void neglog_u2(uint32_t w0, uint32_t w1, float& E0, float& E1) {
  constexpr float kLn2 = 0.693147180559945309f;
  const unsigned long long one = f2_pack(1.0f, 1.0f), two = f2_pack(2.0f, 2.0f);
  const unsigned long long u = f2_add(f2_pack(__uint_as_float(0x3F800000u | (w0 >> 9)),
                                              __uint_as_float(0x3F800000u | (w1 >> 9))),
                                      f2_pack(-0x1.fffffep-1f, -0x1.fffffep-1f));
  const unsigned long long t = f2_sub(one, u);
  float d0, d1;
  f2_unpack(f2_sub(two, t), d0, d1);
  const unsigned long long sr = f2_mul(t, f2_pack(rcp_approx(d0), rcp_approx(d1)));
  const unsigned long long s2 = f2_mul(sr, sr);
  unsigned long long p = f2_fma(s2, f2_pack(2.0f / 9.0f, 2.0f / 9.0f), f2_pack(2.0f / 7.0f, 2.0f / 7.0f));
  p = f2_fma(s2, p, f2_pack(2.0f / 5.0f, 2.0f / 5.0f));
  p = f2_fma(s2, p, f2_pack(2.0f / 3.0f, 2.0f / 3.0f));
  p = f2_fma(s2, p, two);
  const unsigned long long nl2 = f2_pack(-kLn2, -kLn2);
  float u0, u1, n0, n1, f0, f1;
  f2_unpack(u, u0, u1);
  f2_unpack(f2_mul(sr, p), n0, n1);
  f2_unpack(f2_mul(f2_pack(lg2_approx(u0), lg2_approx(u1)), nl2), f0, f1);
  E0 = u0 > 0.75f ? n0 : f0;
  E1 = u1 > 0.75f ? n1 : f1;
}

// Winner key of a categorical draw in exponential-race form: the Gumbel-max
// argmax of log w + g, g = -log E, is the argmax of w / E (the same order in
// exact arithmetic), taken as w * (1/E). Positive ratios only (w > 0, E > 0):
// the order key of a positive float is its bits with the sign bit set; the
// column breaks ties, lowest first. 0 is below every real key.
__device__ __forceinline__ unsigned long long race_key(float w, float E, uint32_t col) {
  const float ratio = __fmul_rn(w, rcp_approx(E));
  const uint32_t o = w > 0.0f ? (__float_as_uint(ratio) | 0x80000000u) : 0u;
  return o == 0u ? 0ull
                 : (static_cast<unsigned long long>(o) << 32) |
                       static_cast<unsigned long long>(0xFFFFFFFFu - col);
}

// gumbel_of of two words at once: the same operations lane by lane, the
// arithmetic in packed pairs (lg2, rcp and the selection per value).
__device__ __forceinline__ void gumbel_of2(uint32_t w0, uint32_t w1, float& g0, float& g1) {
  constexpr float kLn2 = 0.693147180559945309f;
  const unsigned long long one = f2_pack(1.0f, 1.0f), two = f2_pack(2.0f, 2.0f);
  const unsigned long long u = f2_add(f2_pack(__uint_as_float(0x3F800000u | (w0 >> 9)),
                                              __uint_as_float(0x3F800000u | (w1 >> 9))),
                                      f2_pack(-0x1.fffffep-1f, -0x1.fffffep-1f));
  const unsigned long long t = f2_sub(one, u);
  float d0, d1;
  f2_unpack(f2_sub(two, t), d0, d1);
  const unsigned long long sr = f2_mul(t, f2_pack(rcp_approx(d0), rcp_approx(d1)));
  const unsigned long long s2 = f2_mul(sr, sr);
  unsigned long long p = f2_fma(s2, f2_pack(2.0f / 9.0f, 2.0f / 9.0f), f2_pack(2.0f / 7.0f, 2.0f / 7.0f));
  p = f2_fma(s2, p, f2_pack(2.0f / 5.0f, 2.0f / 5.0f));
  p = f2_fma(s2, p, f2_pack(2.0f / 3.0f, 2.0f / 3.0f));
  p = f2_fma(s2, p, two);
  const unsigned long long nl2 = f2_pack(-kLn2, -kLn2);
  float u0, u1, n0, n1, f0, f1;
  f2_unpack(u, u0, u1);
  f2_unpack(f2_mul(sr, p), n0, n1);
  f2_unpack(f2_mul(f2_pack(lg2_approx(u0), lg2_approx(u1)), nl2), f0, f1);
  const float E0 = u0 > 0.75f ? n0 : f0;
  const float E1 = u1 > 0.75f ? n1 : f1;
  f2_unpack(f2_mul(f2_pack(lg2_approx(E0), lg2_approx(E1)), nl2), g0, g1);
}

// Natural log of a positive, normal x with an absolute error of about 1e-7
// (plus the rounding of the result).
__device__ __forceinline__ float ln_approx(float x) {
  return 0.693147180559945309f * lg2_approx(x);
}

// ---------------------------------------------------------------------------
// Winner key. Larger key = better: NaN above everything, then larger values,
// then lower column index. -0 and +0 map to the same value bits.
// 0 is below every real key ("no candidate").
// ---------------------------------------------------------------------------
// e = exp(x - m): ex2.approx of fp32(x - m) * log2(e), which is exactly 1 at
// the maximum (ex2 of +-0 is 1) and within about 3 ulp elsewhere (the
// oracle's exp is correctly rounded, and the tests bound the effect: accept
// margins and top-p boundaries within 1e-6). -inf gives 0.
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float t) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t));
  return y;
}

// exp(y) = 2^(y log2 e), with y = fp32(x - m) and the product rounded once.
__device__ __forceinline__ float exp_rel(float x, float m) {
  return ex2_approx(__fmul_rn(__fsub_rn(x, m), kLog2e));
}


// The same order key without branches: -0 becomes +0 by adding +0, every
// NaN maps to the largest key.
__device__ __forceinline__ uint32_t ordered_key(float y) {
  const uint32_t b = __float_as_uint(__fadd_rn(y, 0.0f));
  const uint32_t k = b ^ (static_cast<uint32_t>(static_cast<int32_t>(b) >> 31) | 0x80000000u);
  return (y != y) ? 0xFFFFFFFFu : k;
}

__device__ __forceinline__ uint32_t ordered_bits(float y) {
  if (y != y) return 0xFFFFFFFFu;
  uint32_t b = __float_as_uint(y);
  if (b == 0x80000000u) b = 0u;  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ unsigned long long winner_key(float y, uint32_t col) {
  return (static_cast<unsigned long long>(ordered_bits(y)) << 32) |
         static_cast<unsigned long long>(0xFFFFFFFFu - col);
}

__device__ __forceinline__ int32_t key_index(unsigned long long key) {
  return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a,
                                                     unsigned long long b) {
  return a > b ? a : b;
}

__device__ __forceinline__ unsigned long long warp_max64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = umax64(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ unsigned long long warp_sum64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// Element access.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ float load_logit(const void* p, bool bf16, int64_t i) {
  return bf16 ? bf16_bits_to_float(__ldg(static_cast<const unsigned short*>(p) + i))
              : __ldg(static_cast<const float*>(p) + i);
}

// fp32 -> bf16, round to nearest even (NaN stays NaN).
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ---------------------------------------------------------------------------
// Status word: the first error wins.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier and bulk async copies (sm_90+ PTX), all waits bounded.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may sleep up to `hint_ns` for the phase
// to complete instead of returning at once (no spinning on the issue slots
// of the warps that do the work).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t phase,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(phase), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Waits for the phase with parity `phase` to complete. Returns false (and
// records DSPARK_ERR_TIMEOUT) if it has not completed within limit_ns
// nanoseconds of %globaltimer.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t phase,
                                          int32_t* status,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, phase)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    for (int i = 0; i < 8; ++i)
      if (mbar_try_wait_sleep(bar, phase, 2000u)) return true;
    if (globaltimer_ns() - t0 > limit_ns) {
      report(status, DSPARK_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Loads of read-only rows with an L2 eviction priority from `policy` (no L1
// allocation). Not volatile: the compiler may batch them for more loads in
// flight.
__device__ __forceinline__ float4 ld_hint_f4(const float* p, uint64_t policy) {
  float4 v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "l"(p), "l"(policy));
  return v;
}
__device__ __forceinline__ uint2 ld_hint_u2(const void* p, uint64_t policy) {
  uint2 v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
      : "=r"(v.x), "=r"(v.y)
      : "l"(p), "l"(policy));
  return v;
}
__device__ __forceinline__ float ld_hint_f32(const float* p, uint64_t policy) {
  float v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(policy));
  return v;
}
__device__ __forceinline__ uint16_t ld_hint_u16(const uint16_t* p, uint64_t policy) {
  unsigned short v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.u16 %0, [%1], %2;" : "=h"(v) : "l"(p), "l"(policy));
  return v;
}
}  // namespace dspark
