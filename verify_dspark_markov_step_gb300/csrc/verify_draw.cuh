// verify_draw.cuh -- the verifier's categorical draws over a column range:
// the residual max(0, p - q) at the first rejected draft, p at a -1
// placeholder, or the bonus row p_K (vLLM PR #65007 Part 2, "Rejection
// sampling": resample from the normalised residual, bonus token). A draw is
// the Gumbel-max argmax_v log w_v + g_v with g = -log E from the target
// noise stream at the row's position, under the drafter's winner rule
// (largest value, lowest column on ties), compared in its exponential-race
// form w_v / E_v (race_key): the same order without two logarithms.
#pragma once

#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "verify_common.cuh"

namespace dspark {

enum DrawMode : int32_t { kDrawNone = 0, kDrawResidual = 1, kDrawP = 2 };

// What one request's draw needs, gathered once per work item.
struct DrawJob {
  int32_t b;        // request
  int32_t mode;     // DrawMode
  int32_t row;      // k of the row drawn from (K = the bonus row)
  int32_t invalid;  // request is padding or out of range: nothing to draw
  int64_t crow;     // cache row of the request
  int64_t P0;       // position of the first draft token
  uint64_t seed;
  float T;
  int32_t n_acc;    // accepted drafts
  int32_t emit;     // greedy: the token emitted without a draw
  TgtStats ts;      // statistics of target row `row`
  DrfStats ds;      // statistics of draft row `row` (residual draws)
};

// p at column v of a target row from its statistics (invD = 1 / D).
__device__ __forceinline__ float p_at(const TgtStats& ts, float t, float T, float invD, int v) {
  if (ts.mode == kModeOneHot) return v == 0 ? 1.0f : 0.0f;
  const float x = scale_logit(t, T);
  if (ts.mode == kModeThreshold) {
    const uint32_t kd = kd_of(x);
    if (!(kd > ts.kd_thr || (kd == ts.kd_thr && v <= ts.id_thr))) return 0.0f;
  }
  return exp_rel(x, ts.m) * invD;
}

__device__ __forceinline__ float q_at(const DrfStats& ds, float c, float invD) {
  if (ds.zero) return 0.0f;
  const float x = (c != c) ? -INFINITY : c;
  return exp_rel(x, ds.m) * invD;
}

// Four consecutive logits [g, g+4) clipped to [.., c1), fp32 or bf16.
__device__ __forceinline__ void draw_load4(const void* base, bool bf16, int64_t off, int g,
                                           int c1, bool vec, float (&out)[4]) {
  if (vec && g + 3 < c1) {
    if (bf16) {
      const uint2 raw =
          __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + off + g));
      out[0] = __uint_as_float(raw.x << 16);
      out[1] = __uint_as_float(raw.x & 0xFFFF0000u);
      out[2] = __uint_as_float(raw.y << 16);
      out[3] = __uint_as_float(raw.y & 0xFFFF0000u);
    } else {
      const float4 f =
          __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + off + g));
      out[0] = f.x;
      out[1] = f.y;
      out[2] = f.z;
      out[3] = f.w;
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) out[j] = g + j < c1 ? load_logit(base, bf16, off + g + j) : 0.0f;
}

// The common draw, specialised at compile time: a sampled row kept whole or
// cut at a top-p threshold, temperature 1 or not, from p or from the
// residual max(0, p - q) with a nonzero draft row. Straight-line per column;
// the noise of a 4-column block is drawn only if one of its weights is
// positive. Thread t of `nthr` takes the 4-column groups c0 + 4t, c0 + 4t +
// 4 nthr, ...; returns the thread's winner key.
template <bool kResidual, bool kScale, bool kThreshold>
__device__ unsigned long long draw_fast(const VerifyParams& P, const DrawJob& J, int64_t toff,
                                        int64_t coff, int c0, int c1, bool tvec, bool cvec,
                                        int nthr, unsigned int* anypos) {
  const bool tbf = P.target_bf16 != 0, cbf = P.cache_bf16 != 0;
  const TgtStats& ts = J.ts;
  const float invD = 1.0f / ts.D;
  const float invDq = kResidual ? 1.0f / J.ds.D : 0.0f;
  const unsigned long long mm = f2_pack(ts.m, ts.m), mq = f2_pack(J.ds.m, J.ds.m);
  const unsigned long long l2e = f2_pack(kLog2e, kLog2e);
  const unsigned long long invD2 = f2_pack(invD, invD), invDq2 = f2_pack(invDq, invDq);
  const int64_t npos = J.P0 + J.row - 1;
  // running winner of this thread: its columns only grow, so a strict >
  // keeps the lowest column on ties
  uint32_t run_o = 0u, run_c = 0u;
  unsigned int any = 0u;
  // one 4-column group: weights, and the noise only if a weight is positive
  auto group = [&](int g, const float (&t4)[4], const float (&c4)[4]) {
    // p = exp(x - m) / D (and q likewise) two columns at a time in packed
    // pairs: the same fp32 operations as exp_rel and the scalar products
    float x4[4], p4[4], q4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      x4[j] = fmaxf(kScale ? __fdiv_rn(t4[j], J.T) : t4[j], -INFINITY);  // NaN -> -inf
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      float a, b;
      f2_unpack(f2_mul(f2_sub(f2_pack(x4[j], x4[j + 1]), mm), l2e), a, b);
      f2_unpack(f2_mul(f2_pack(ex2_approx(a), ex2_approx(b)), invD2), p4[j], p4[j + 1]);
      if (kResidual) {
        f2_unpack(f2_mul(f2_sub(f2_pack(fmaxf(c4[j], -INFINITY), fmaxf(c4[j + 1], -INFINITY)),
                                mq),
                         l2e),
                  a, b);
        f2_unpack(f2_mul(f2_pack(ex2_approx(a), ex2_approx(b)), invDq2), q4[j], q4[j + 1]);
      }
    }
    float w[4];
    bool need = false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float pv = p4[j];
      if (kThreshold) {
        const uint32_t kd = kd_of(x4[j]);
        const bool keep = kd > ts.kd_thr || (kd == ts.kd_thr && g + j <= ts.id_thr);
        pv = keep ? pv : 0.0f;
      }
      if (kResidual) pv = fmaxf(__fsub_rn(pv, q4[j]), 0.0f);
      w[j] = g + j < c1 ? pv : 0.0f;
      need |= w[j] > 0.0f;
    }
    if (!need) return;
    any = 1u;
    const U4 r = noise_block(J.seed, npos, static_cast<uint32_t>(g), kStreamTarget);
    float E[4];
    neglog_u2(r.x, r.y, E[0], E[1]);
    neglog_u2(r.z, r.w, E[2], E[3]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float ratio = __fmul_rn(w[j], rcp_approx(E[j]));
      const uint32_t o = w[j] > 0.0f ? (__float_as_uint(ratio) | 0x80000000u) : 0u;
      if (o > run_o) {
        run_o = o;
        run_c = static_cast<uint32_t>(g + j);
      }
    }
  };
  // two groups per iteration, both loaded before either is used (a group at
  // or past c1 loads nothing and weighs 0); the thread's columns still come
  // in increasing order
  for (int g = c0 + 4 * static_cast<int>(threadIdx.x); g < c1; g += 8 * nthr) {
    const int g2 = g + 4 * nthr;
    float t4[4], c4[4] = {0.f, 0.f, 0.f, 0.f}, t4b[4], c4b[4] = {0.f, 0.f, 0.f, 0.f};
    draw_load4(P.target, tbf, toff, g, c1, tvec, t4);
    draw_load4(P.target, tbf, toff, g2, c1, tvec, t4b);
    if (kResidual) {
      draw_load4(P.cache, cbf, coff, g, c1, cvec, c4);
      draw_load4(P.cache, cbf, coff, g2, c1, cvec, c4b);
    }
    group(g, t4, c4);
    if (g2 < c1) group(g2, t4b, c4b);
  }
  *anypos = any;
  return run_o == 0u ? 0ull
                     : (static_cast<unsigned long long>(run_o) << 32) |
                           static_cast<unsigned long long>(0xFFFFFFFFu - run_c);
}

// This thread's winner key over columns [c0, c1) (c0 a multiple of 4) of
// the request's draw; *anypos = some weight was positive. `mode` overrides
// J.mode (the all-zero-residual fallback draws from p).
__device__ unsigned long long draw_range(const VerifyParams& P, const DrawJob& J, int mode,
                                         int c0, int c1, int nthr, unsigned int* anypos) {
  const int V = P.V, K = P.K;
  const int64_t toff = (static_cast<int64_t>(J.b) * (K + 1) + J.row) * V;
  const bool residual = mode == kDrawResidual;
  const int64_t coff = residual ? (J.crow * K + J.row) * V : 0;
  const bool tbf = P.target_bf16 != 0, cbf = P.cache_bf16 != 0;
  // 4-element vector loads need 16-byte (fp32) or 8-byte (bf16) aligned rows
  const bool tvec =
      ((reinterpret_cast<uintptr_t>(P.target) + toff * (tbf ? 2 : 4)) & (tbf ? 7u : 15u)) == 0;
  const bool cvec =
      ((reinterpret_cast<uintptr_t>(P.cache) + coff * (cbf ? 2 : 4)) & (cbf ? 7u : 15u)) == 0;
  const TgtStats& ts = J.ts;
  const DrfStats ds = residual ? J.ds : DrfStats{0.f, 1.f, 0.f, 1};
  if (ts.mode != kModeOneHot && !(residual && ds.zero)) {
    const bool scale = J.T != 1.0f;
    const bool thr = ts.mode == kModeThreshold;
#define DSPARK_DRAW(R, S, H) \
  return draw_fast<R, S, H>(P, J, toff, coff, c0, c1, tvec, cvec, nthr, anypos)
    if (residual) {
      if (scale) {
        if (thr) DSPARK_DRAW(true, true, true);
        DSPARK_DRAW(true, true, false);
      }
      if (thr) DSPARK_DRAW(true, false, true);
      DSPARK_DRAW(true, false, false);
    }
    if (scale) {
      if (thr) DSPARK_DRAW(false, true, true);
      DSPARK_DRAW(false, true, false);
    }
    if (thr) DSPARK_DRAW(false, false, true);
    DSPARK_DRAW(false, false, false);
#undef DSPARK_DRAW
  }
  // generic path: one-hot target rows and all-zero draft rows
  const float invD = 1.0f / ts.D;
  const float invDq = ds.zero ? 0.0f : 1.0f / ds.D;
  const int64_t npos = J.P0 + J.row - 1;
  unsigned long long best = 0ull;
  unsigned int any = 0u;
  for (int g = c0 + 4 * static_cast<int>(threadIdx.x); g < c1; g += 4 * nthr) {
    float t4[4], c4[4] = {0.f, 0.f, 0.f, 0.f};
    draw_load4(P.target, tbf, toff, g, c1, tvec, t4);
    if (residual) draw_load4(P.cache, cbf, coff, g, c1, cvec, c4);
    bool need = false;
    float w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float pv = 0.0f;
      if (g + j < c1) {
        pv = p_at(ts, t4[j], J.T, invD, g + j);
        if (residual) {
          const float r = __fsub_rn(pv, q_at(ds, c4[j], invDq));
          pv = r > 0.0f ? r : 0.0f;
        }
      }
      w[j] = pv;
      need |= pv > 0.0f;
    }
    if (!need) continue;
    any = 1u;
    const U4 r = noise_block(J.seed, npos, static_cast<uint32_t>(g), kStreamTarget);
    float E[4];
    neglog_u2(r.x, r.y, E[0], E[1]);
    neglog_u2(r.z, r.w, E[2], E[3]);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      best = umax64(best, race_key(w[j], E[j], static_cast<uint32_t>(g + j)));
  }
  *anypos = any;
  return best;
}

}  // namespace dspark
