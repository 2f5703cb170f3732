// verify.cu -- probabilistic rejection-sampling verification.
//
// Follows vLLM PR #65007 Part 2 ("Temperature and top-p": the smallest prefix
// by logit, then token id, whose probability mass reaches p, plus the row
// max, with masses summed in 64-bit fixed point; "Rejection sampling": accept
// with probability min(1, p/q), resample from the normalised max(0, p - q),
// bonus token) and vLLM PR #63554 (greedy rows compare with the target
// argmax and never read the draft-logits cache).
//
// Two launches:
//   1. verify_rows_kernel (verify_stats.cu), one thread-block cluster per
//      row (B*(K+1) target rows, B*K draft rows): the row max, the
//      fixed-point mass, the exact top-p threshold, and p or q at the drafted
//      token; greedy target rows get their winner key.
//   2. verify_resample_kernel, grid (chunks, B): every CTA replays the
//      accept/reject chain of its request from the row statistics, then draws
//      its column chunk of the one categorical the request needs (residual at
//      the first rejection, or p at a -1 placeholder, or the bonus row); the
//      last CTA of the request reduces the chunk winners and writes the
//      outputs.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "verify_common.cuh"

namespace dspark {

namespace {

constexpr int kResThreads = 256;

// ---------------------------------------------------------------------------
// Kernel 2: chain replay, chunked categorical draw, outputs
// ---------------------------------------------------------------------------
enum DrawMode : int { kDrawNone = 0, kDrawResidual = 1, kDrawP = 2 };

struct ResSmem {
  int mode;       // DrawMode
  int row;        // k of the row drawn from
  int n_acc;      // accepted drafts
  int emit;       // token emitted without a draw (greedy), or -1
  int invalid;    // request is padding / out of range
  int64_t crow;
  float T;
  uint64_t seed;
  int64_t P0;
  int acc[DSPARK_MAX_STEPS];
  int dtok[DSPARK_MAX_STEPS];
  unsigned long long red[kResThreads / 32];
  unsigned int any[kResThreads / 32];
  unsigned int last;
};

// p at column v of a target row from its statistics.
// exp(x - m) of the row statistics (see exp_rel).
__device__ __forceinline__ float exp_rel_fast(float x, float m) { return exp_rel(x, m); }

// p at column v of a target row from its statistics (invD = 1 / D).
__device__ __forceinline__ float p_fast(const TgtStats& ts, float t, float T, float invD, int v) {
  if (ts.mode == kModeOneHot) return v == 0 ? 1.0f : 0.0f;
  const float x = scale_logit(t, T);
  if (ts.mode == kModeThreshold) {
    const uint32_t kd = kd_of(x);
    if (!(kd > ts.kd_thr || (kd == ts.kd_thr && v <= ts.id_thr))) return 0.0f;
  }
  return exp_rel_fast(x, ts.m) * invD;
}

__device__ __forceinline__ float q_fast(const DrfStats& ds, float c, float invD) {
  if (ds.zero) return 0.0f;
  const float x = (c != c) ? -INFINITY : c;
  return exp_rel_fast(x, ds.m) * invD;
}

// Four consecutive logits [g, g+4) clipped to [.., c1), fp32 or bf16.
__device__ __forceinline__ void load4(const void* base, bool bf16, int64_t off, int g, int c1,
                                      bool vec, float (&out)[4]) {
  if (vec && g + 3 < c1) {
    if (bf16) {
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + off + g));
      out[0] = __uint_as_float(raw.x << 16);
      out[1] = __uint_as_float(raw.x & 0xFFFF0000u);
      out[2] = __uint_as_float(raw.y << 16);
      out[3] = __uint_as_float(raw.y & 0xFFFF0000u);
    } else {
      const float4 f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + off + g));
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
// positive, as in the generic path.
template <bool kResidual, bool kScale, bool kThreshold>
__device__ unsigned long long draw_fast(const VerifyParams& P, const TgtStats& ts,
                                        const DrfStats& ds, float T, uint64_t seed,
                                        int64_t npos, int64_t toff, int64_t coff, int c0,
                                        int c1, bool tvec, bool cvec, unsigned int* anypos) {
  const bool tbf = P.target_bf16 != 0, cbf = P.cache_bf16 != 0;
  const float invD = 1.0f / ts.D;
  const float invDq = kResidual ? 1.0f / ds.D : 0.0f;
  const unsigned long long mm = f2_pack(ts.m, ts.m), mq = f2_pack(ds.m, ds.m);
  const unsigned long long l2e = f2_pack(kLog2e, kLog2e);
  const unsigned long long invD2 = f2_pack(invD, invD), invDq2 = f2_pack(invDq, invDq);
  // running winner of this thread: its columns only grow, so a strict >
  // keeps the lowest column on ties
  uint32_t run_o = 0u, run_c = 0u;
  unsigned int any = 0u;
  for (int g = c0 + 4 * threadIdx.x; g < c1; g += 4 * kResThreads) {
    float t4[4], c4[4];
    load4(P.target, tbf, toff, g, c1, tvec, t4);
    if (kResidual) load4(P.cache, cbf, coff, g, c1, cvec, c4);
    // p = exp(x - m) / D (and q likewise) two columns at a time in packed
    // pairs: the same fp32 operations as exp_rel and the scalar products
    float x4[4], p4[4], q4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      x4[j] = fmaxf(kScale ? __fdiv_rn(t4[j], T) : t4[j], -INFINITY);  // NaN -> -inf
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
    if (!need) continue;
    any = 1u;
    const U4 r = noise_block(seed, npos, static_cast<uint32_t>(g), kStreamTarget);
    float gn[4];
    gumbel_of2(r.x, r.y, gn[0], gn[1]);
    gumbel_of2(r.z, r.w, gn[2], gn[3]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float y = __fadd_rn(ln_approx(w[j]), gn[j]);
      const uint32_t o = w[j] > 0.0f ? ordered_key(y) : 0u;
      if (o > run_o) {
        run_o = o;
        run_c = static_cast<uint32_t>(g + j);
      }
    }
  }
  *anypos = any;
  return run_o == 0u ? 0ull
                     : (static_cast<unsigned long long>(run_o) << 32) |
                           static_cast<unsigned long long>(0xFFFFFFFFu - run_c);
}

// Winner key over columns [c0, c1) (c0 a multiple of 4) of the draw for
// this request; *anypos = some residual entry was positive.
__device__ unsigned long long draw_chunk(const VerifyParams& P, const ResSmem& rs,
                                         int c0, int c1, unsigned int* anypos) {
  const int V = P.V, K = P.K, b = blockIdx.y;
  const int k = rs.row;
  const TgtStats ts = *(static_cast<const TgtStats*>(P.tstats) + static_cast<int64_t>(b) * (K + 1) + k);
  const int64_t toff = (static_cast<int64_t>(b) * (K + 1) + k) * V;
  const bool residual = rs.mode == kDrawResidual;
  DrfStats ds{0.f, 1.f, 0.f, 1};
  int64_t coff = 0;
  if (residual) {
    ds = *(static_cast<const DrfStats*>(P.dstats) + static_cast<int64_t>(b) * K + k);
    coff = (rs.crow * K + k) * V;
  }
  const float invD = 1.0f / ts.D;
  const float invDq = ds.zero ? 0.0f : 1.0f / ds.D;
  const bool tbf = P.target_bf16 != 0, cbf = P.cache_bf16 != 0;
  // 4-element vector loads need 16-byte (fp32) or 8-byte (bf16) aligned rows
  const bool tvec = ((reinterpret_cast<uintptr_t>(P.target) + toff * (tbf ? 2 : 4)) & (tbf ? 7u : 15u)) == 0;
  const bool cvec = ((reinterpret_cast<uintptr_t>(P.cache) + coff * (cbf ? 2 : 4)) & (cbf ? 7u : 15u)) == 0;
  const int64_t npos = rs.P0 + k - 1;
  // the chunk's rows come from HBM: start them as bulk L2 prefetches
  if (threadIdx.x == 0) {
    auto pf = [](const void* base, int64_t off, int es, int n) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(static_cast<const unsigned char*>(base) + off * es);
      const uintptr_t a16 = (a + 15) & ~static_cast<uintptr_t>(15);
      const uint32_t bytes = static_cast<uint32_t>(n) * es;
      const uint32_t skip = static_cast<uint32_t>(a16 - a);
      if (bytes > skip + 16)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a16),
                     "r"((bytes - skip) & ~15u) : "memory");
    };
    pf(P.target, toff + c0, tbf ? 2 : 4, c1 - c0);
    if (residual) pf(P.cache, coff + c0, cbf ? 2 : 4, c1 - c0);
  }
  if (ts.mode != kModeOneHot && !(residual && ds.zero)) {
    const bool scale = rs.T != 1.0f;
    const bool thr = ts.mode == kModeThreshold;
#define DSPARK_DRAW(R, S, H)                                                                   \
  return draw_fast<R, S, H>(P, ts, ds, rs.T, rs.seed, npos, toff, coff, c0, c1, tvec, cvec, \
                            anypos)
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
  unsigned long long best = 0ull;
  unsigned int any = 0u;
  for (int g = c0 + 4 * threadIdx.x; g < c1; g += 4 * kResThreads) {
    float t4[4], c4[4] = {0.f, 0.f, 0.f, 0.f};
    load4(P.target, tbf, toff, g, c1, tvec, t4);
    if (residual) load4(P.cache, cbf, coff, g, c1, cvec, c4);
    bool need = false;
    float w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float pv = 0.0f;
      if (g + j < c1) {
        pv = p_fast(ts, t4[j], rs.T, invD, g + j);
        if (residual) {
          const float r = __fsub_rn(pv, q_fast(ds, c4[j], invDq));
          pv = r > 0.0f ? r : 0.0f;
        }
      }
      w[j] = pv;
      need |= pv > 0.0f;
    }
    if (!need) continue;
    any = 1u;
    const U4 r = noise_block(rs.seed, npos, static_cast<uint32_t>(g), kStreamTarget);
    const uint32_t words[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (w[j] > 0.0f) {
        const float y = __fadd_rn(ln_approx(w[j]), gumbel_of(words[j]));
        best = umax64(best, winner_key(y, static_cast<uint32_t>(g + j)));
      }
    }
  }
  *anypos = any;
  return best;
}

__global__ void __launch_bounds__(kResThreads) verify_resample_kernel(VerifyParams P) {
  __shared__ ResSmem rs;
  const int b = blockIdx.y, chunk = blockIdx.x, K = P.K, V = P.V;
  const int tid = threadIdx.x;

  // ---- replay the chain (threads 0..K-1 test one draft each) --------------
  if (tid == 0) {
    rs.mode = kDrawNone;
    rs.row = 0;
    rs.n_acc = 0;
    rs.emit = -1;
    rs.invalid = 0;
    rs.crow = 0;
    const int32_t s = P.rsi[b];
    if (s < 0 || s >= P.S) {
      rs.invalid = 1;
      if (s >= P.S && chunk == 0) report(P.status, DSPARK_ERR_BOUNDS);
    } else {
      rs.T = P.temperature[s];
      rs.seed = P.seeds[s];
      rs.P0 = P.pos[b];
      if (rs.T > 0.0f) {
        if (P.cache == nullptr) {
          rs.invalid = 1;
          if (chunk == 0) report(P.status, DSPARK_ERR_INVALID_ARG);
        } else {
          rs.crow = P.row_map ? P.row_map[s] : s;
          if (rs.crow < 0 || rs.crow >= P.C) {
            rs.invalid = 1;
            if (chunk == 0) report(P.status, DSPARK_ERR_BOUNDS);
          }
        }
      } else {
        rs.T = 0.0f;
      }
    }
  }
  __syncthreads();
  if (!rs.invalid && tid < K) {
    const int k = tid;
    const int32_t d = P.draft[static_cast<int64_t>(b) * K + k];
    int a = 0;  // 1 accept, 0 reject, -1 placeholder, -2 out of range
    if (d == -1) {
      a = -1;
    } else if (d < -1 || d >= V) {
      a = -2;
    } else if (!(rs.T > 0.0f)) {
      const TgtStats ts = *(static_cast<const TgtStats*>(P.tstats) + static_cast<int64_t>(b) * (K + 1) + k);
      a = key_index(ts.amax_key) == d ? 1 : 0;
    } else {
      const TgtStats ts = *(static_cast<const TgtStats*>(P.tstats) + static_cast<int64_t>(b) * (K + 1) + k);
      const DrfStats ds = *(static_cast<const DrfStats*>(P.dstats) + static_cast<int64_t>(b) * K + k);
      const U4 r = noise_block(rs.seed, rs.P0 + k - 1, 0u, kStreamAccept);
      const float u = uniform_of(r.x);
      a = __fmul_rn(u, ds.q_d) < ts.p_d ? 1 : 0;
    }
    rs.acc[k] = a;
    rs.dtok[k] = d;
  }
  __syncthreads();
  if (tid == 0 && !rs.invalid) {
    int k = 0;
    for (; k < K; ++k) {
      const int a = rs.acc[k];
      if (a == -2) {
        rs.invalid = 1;
        if (chunk == 0) report(P.status, DSPARK_ERR_BOUNDS);
        break;
      }
      if (a != 1) break;
    }
    if (!rs.invalid) {
      rs.n_acc = k;
      rs.row = k;  // row of the emitted token (K = bonus)
      if (!(rs.T > 0.0f)) {
        const TgtStats ts = *(static_cast<const TgtStats*>(P.tstats) + static_cast<int64_t>(b) * (K + 1) + k);
        rs.emit = key_index(ts.amax_key);
        rs.mode = kDrawNone;
      } else if (k < K && rs.acc[k] == 0) {
        rs.mode = kDrawResidual;
      } else {
        rs.mode = kDrawP;  // -1 placeholder or bonus
      }
    }
  }
  __syncthreads();

  // ---- this CTA's chunk of the draw -----------------------------------------
  const int nch = P.nchunk;
  int cw = (V + nch - 1) / nch;
  cw = (cw + 3) & ~3;
  const int c0 = chunk * cw, c1 = min(V, c0 + cw);
  unsigned long long key = 0ull;
  unsigned int any = 0u;
  if (!rs.invalid && rs.mode != kDrawNone && c0 < c1) key = draw_chunk(P, rs, c0, c1, &any);
  key = warp_max64(key);
  any = __any_sync(0xFFFFFFFFu, any != 0u) ? 1u : 0u;
  if ((tid & 31) == 0) {
    rs.red[tid >> 5] = key;
    rs.any[tid >> 5] = any;
  }
  __syncthreads();
  if (tid == 0) {
    unsigned long long k2 = 0ull;
    unsigned int a2 = 0u;
    for (int i = 0; i < kResThreads / 32; ++i) {
      k2 = umax64(k2, rs.red[i]);
      a2 |= rs.any[i];
    }
    P.keys[static_cast<int64_t>(b) * nch + chunk] = k2;
    P.anypos[static_cast<int64_t>(b) * nch + chunk] = a2;
    __threadfence();
    const unsigned int ticket = atomicAdd(&P.counters[b], 1u);
    rs.last = ticket == static_cast<unsigned int>(nch) - 1u;
  }
  __syncthreads();
  if (!rs.last) return;
  __threadfence();

  // ---- last CTA of the request: reduce and write the outputs -----------------
  __shared__ int s_tok;
  if (tid == 0) {
    int tok = -1;
    bool need_fallback = false;
    if (!rs.invalid) {
      if (rs.mode == kDrawNone) {
        tok = rs.emit;
      } else {
        unsigned long long m = 0ull;
        unsigned int a = 0u;
        for (int i = 0; i < nch; ++i) {
          m = umax64(m, __ldcg(P.keys + static_cast<int64_t>(b) * nch + i));
          a |= __ldcg(P.anypos + static_cast<int64_t>(b) * nch + i);
        }
        if (rs.mode == kDrawResidual && a == 0u) {
          need_fallback = true;  // r is all zero (fp32 rounding): draw from p
        } else {
          tok = m ? key_index(m) : 0;
        }
      }
    }
    s_tok = need_fallback ? -2 : tok;
    P.counters[b] = 0u;
  }
  __syncthreads();
  if (s_tok == -2) {
    __syncthreads();
    if (tid == 0) rs.mode = kDrawP;
    __syncthreads();
    unsigned int dummy = 0u;
    unsigned long long k3 = draw_chunk(P, rs, 0, V, &dummy);
    k3 = warp_max64(k3);
    if ((tid & 31) == 0) rs.red[tid >> 5] = k3;
    __syncthreads();
    if (tid == 0) {
      unsigned long long m = 0ull;
      for (int i = 0; i < kResThreads / 32; ++i) m = umax64(m, rs.red[i]);
      s_tok = m ? key_index(m) : 0;
    }
    __syncthreads();
  }
  for (int k = tid; k <= K; k += kResThreads) {
    int32_t o = -1;
    if (!rs.invalid) {
      if (k < rs.n_acc)
        o = rs.dtok[k];
      else if (k == rs.n_acc)
        o = s_tok;
    }
    P.out_tokens[static_cast<int64_t>(b) * (K + 1) + k] = o;
  }
  if (tid == 0) P.num_accepted[b] = rs.invalid ? 0 : rs.n_acc;
}

__global__ void noise_kernel(const uint64_t* seed, const int64_t* pos, const uint32_t* col,
                             const uint32_t* stream_word, uint32_t* word, float* u, float* g,
                             int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const U4 r = noise_block(seed[i], pos[i], col[i], stream_word[i]);
    const uint32_t w = pick_word(r, col[i] & 3u);
    if (word) word[i] = w;
    if (u) u[i] = uniform_of(w);
    if (g) g[i] = gumbel_of(w);
  }
}

}  // namespace

size_t verify_tstats_bytes(int B, int K) {
  return static_cast<size_t>(B) * (K + 1) * sizeof(TgtStats);
}
size_t verify_dstats_bytes(int B, int K) {
  return static_cast<size_t>(B) * K * sizeof(DrfStats);
}
int verify_max_chunks(int V) { return (V + 1023) / 1024; }
int verify_chunks(int B, int V, int num_sms) {
  int want = (4 * num_sms + (B > 0 ? B : 1) - 1) / (B > 0 ? B : 1);
  const int mx = verify_max_chunks(V);
  if (want > mx) want = mx;
  if (want < 1) want = 1;
  return want;
}

cudaError_t launch_verify(const VerifyParams& p, int CL, int W, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  cudaError_t err = launch_verify_rows(p, CL, W, stream);
  if (err != cudaSuccess) return err;
  verify_resample_kernel<<<dim3(p.nchunk, p.B), kResThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_noise(const uint64_t* seed, const int64_t* pos, const uint32_t* col,
                         const uint32_t* stream_word, uint32_t* word, float* u, float* g,
                         int64_t n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  int blocks = static_cast<int>((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  noise_kernel<<<blocks, 256, 0, stream>>>(seed, pos, col, stream_word, word, u, g, n);
  return cudaGetLastError();
}

}  // namespace dspark
