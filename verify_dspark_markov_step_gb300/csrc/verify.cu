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
//   1. verify_stats_kernel, one CTA per row (B*(K+1) target rows, B*K draft
//      rows): the row max, the fixed-point mass, the exact top-p threshold
//      (a radix select over the ordered bits of the scaled logits, 12+12+8
//      bits, then over token ids, with histograms of fixed-point mass), and
//      p or q at the drafted token. Greedy target rows get their winner key.
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

namespace dspark {

namespace {

constexpr int kStatThreads = 512;
constexpr int kStatWarps = kStatThreads / 32;
constexpr int kBins = 4096;
constexpr int kResThreads = 256;
constexpr int kUnroll = 4;

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

// ---------------------------------------------------------------------------
// Shared helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float scale_logit(float t, float T) {
  float x = (T == 1.0f) ? t : __fdiv_rn(t, T);
  return (x != x) ? -INFINITY : x;
}

__device__ __forceinline__ float exp_rel(float x, float m) {
  return (x == m) ? 1.0f : expf(__fsub_rn(x, m));
}

// ordered bits of a non-NaN value (larger value -> larger key)
__device__ __forceinline__ uint32_t kd_of(float x) { return ordered_bits(x); }

// c * 2^32 >= (t_hi:t_lo), all unsigned
__device__ __forceinline__ bool reaches(unsigned long long c, unsigned long long t_hi,
                                        unsigned long long t_lo) {
  const unsigned long long c_hi = c >> 32, c_lo = c << 32;
  return c_hi > t_hi || (c_hi == t_hi && c_lo >= t_lo);
}

struct StatSmem {
  unsigned long long mass[kBins];
  unsigned int cnt[kBins];
  unsigned int idmax[kBins];
  unsigned long long red64[kStatWarps];
  float redf[kStatWarps];
  int found_pos;
  unsigned long long found_before;
};

__device__ float block_max_f(float v, StatSmem& sm) {
  v = warp_maxf(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sm.redf[w] = v;
  __syncthreads();
  if (w == 0) {
    float x = l < kStatWarps ? sm.redf[l] : -INFINITY;
    x = warp_maxf(x);
    if (l == 0) sm.redf[0] = x;
  }
  __syncthreads();
  return sm.redf[0];
}

__device__ unsigned long long block_sum_u64(unsigned long long v, StatSmem& sm) {
  v = warp_sum64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sm.red64[w] = v;
  __syncthreads();
  if (w == 0) {
    unsigned long long x = l < kStatWarps ? sm.red64[l] : 0ull;
    x = warp_sum64(x);
    if (l == 0) sm.red64[0] = x;
  }
  __syncthreads();
  return sm.red64[0];
}

__device__ unsigned long long block_max_u64(unsigned long long v, StatSmem& sm) {
  v = warp_max64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sm.red64[w] = v;
  __syncthreads();
  if (w == 0) {
    unsigned long long x = l < kStatWarps ? sm.red64[l] : 0ull;
    x = warp_max64(x);
    if (l == 0) sm.red64[0] = x;
  }
  __syncthreads();
  return sm.red64[0];
}

// Warp-uniform walk over a row: calls fn(v, value, valid) for kUnroll
// elements per lane per iteration; every lane of a warp makes the same calls.
template <bool VEC, bool BF16, class Fn>
__device__ __forceinline__ void row_walk(const void* row, int V, Fn&& fn) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if constexpr (!BF16) {
    const float* r = static_cast<const float*>(row);
    if constexpr (VEC) {
      // each lane loads float4s: 4 consecutive columns per load
      const int n4 = (V + 3) >> 2;
      for (int base = warp * 32; base < n4; base += kStatThreads) {
        const int q = base + lane;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (4 * q + 3 < V) {
          x = __ldg(reinterpret_cast<const float4*>(r) + q);
        } else if (q < n4) {
          x.x = 4 * q < V ? __ldg(r + 4 * q) : 0.f;
          x.y = 4 * q + 1 < V ? __ldg(r + 4 * q + 1) : 0.f;
          x.z = 4 * q + 2 < V ? __ldg(r + 4 * q + 2) : 0.f;
        }
        fn(4 * q, x.x, 4 * q < V);
        fn(4 * q + 1, x.y, 4 * q + 1 < V);
        fn(4 * q + 2, x.z, 4 * q + 2 < V);
        fn(4 * q + 3, x.w, 4 * q + 3 < V);
      }
    } else {
      for (int base = warp * 32 * kUnroll; base < V; base += kStatThreads * kUnroll) {
        float x[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = base + u * 32 + lane;
          x[u] = v < V ? __ldg(r + v) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = base + u * 32 + lane;
          fn(v, x[u], v < V);
        }
      }
    }
  } else {
    const uint16_t* r = static_cast<const uint16_t*>(row);
    if constexpr (VEC) {
      const int n8 = (V + 7) >> 3;
      for (int base = warp * 32; base < n8; base += kStatThreads) {
        const int q = base + lane;
        uint32_t w4[4] = {0u, 0u, 0u, 0u};
        if (8 * q + 7 < V) {
          const uint4 raw = __ldg(reinterpret_cast<const uint4*>(r) + q);
          w4[0] = raw.x;
          w4[1] = raw.y;
          w4[2] = raw.z;
          w4[3] = raw.w;
        } else if (q < n8) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int v = 8 * q + j;
            const uint32_t h = v < V ? __ldg(reinterpret_cast<const unsigned short*>(r) + v) : 0u;
            w4[j >> 1] |= (j & 1) ? (h << 16) : h;
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t h = (j & 1) ? (w4[j >> 1] >> 16) : (w4[j >> 1] & 0xFFFFu);
          fn(8 * q + j, bf16_bits_to_float(static_cast<uint16_t>(h)), 8 * q + j < V);
        }
      }
    } else {
      for (int base = warp * 32 * kUnroll; base < V; base += kStatThreads * kUnroll) {
        float x[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = base + u * 32 + lane;
          x[u] = v < V ? bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(r) + v))
                       : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = base + u * 32 + lane;
          fn(v, x[u], v < V);
        }
      }
    }
  }
}

template <class Fn>
__device__ __forceinline__ void row_walk_any(const void* row, bool bf16, int V, Fn&& fn) {
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  if (bf16) {
    if (vec)
      row_walk<true, true>(row, V, fn);
    else
      row_walk<false, true>(row, V, fn);
  } else {
    if (vec)
      row_walk<true, false>(row, V, fn);
    else
      row_walk<false, false>(row, V, fn);
  }
}

// Adds (mass f, one count, id) to histogram bin `bin`, aggregated over the
// lanes of the warp that share the bin. Called by every lane of the warp;
// lanes with active == false add nothing.
__device__ __forceinline__ void hist_add(StatSmem& sm, bool active, int bin,
                                         unsigned long long f, uint32_t id) {
  unsigned int todo = __ballot_sync(0xFFFFFFFFu, active);
  const int lane = threadIdx.x & 31;
  while (todo) {
    const int leader = __ffs(todo) - 1;
    const int lb = __shfl_sync(0xFFFFFFFFu, bin, leader);
    const bool mine = active && bin == lb;
    const unsigned int peers = __ballot_sync(0xFFFFFFFFu, mine);
    // f <= 2^40: split in two 20-bit halves so 32-bit sums cannot overflow
    const unsigned int hi = __reduce_add_sync(0xFFFFFFFFu, mine ? static_cast<unsigned int>(f >> 20) : 0u);
    const unsigned int lo = __reduce_add_sync(0xFFFFFFFFu, mine ? static_cast<unsigned int>(f & 0xFFFFFu) : 0u);
    const unsigned int idm = __reduce_max_sync(0xFFFFFFFFu, mine ? id : 0u);
    if (lane == leader) {
      atomicAdd(&sm.mass[lb], (static_cast<unsigned long long>(hi) << 20) + lo);
      atomicAdd(&sm.cnt[lb], static_cast<unsigned int>(__popc(peers)));
      atomicMax(&sm.idmax[lb], idm);
    }
    todo &= ~peers;
  }
}

__device__ void hist_clear(StatSmem& sm, int nb) {
  for (int i = threadIdx.x; i < nb; i += kStatThreads) {
    sm.mass[i] = 0ull;
    sm.cnt[i] = 0u;
    sm.idmax[i] = 0u;
  }
}

// Scans the nb bins in scan order (descending bin index if desc) starting
// from mass `above`, and returns the first non-empty bin at which the
// running mass reaches the target; *before = the running mass before it.
// Falls back to the last non-empty bin if none reaches (cannot happen when
// the set holds the boundary).
__device__ int hist_find(StatSmem& sm, int nb, bool desc, unsigned long long above,
                         unsigned long long t_hi, unsigned long long t_lo,
                         unsigned long long* before) {
  const int per = (nb + kStatThreads - 1) / kStatThreads;
  const int p0 = threadIdx.x * per;
  unsigned long long mine = 0ull;
  for (int i = 0; i < per; ++i) {
    const int pos = p0 + i;
    if (pos < nb) mine += sm.mass[desc ? nb - 1 - pos : pos];
  }
  // exclusive block scan of `mine` (u64)
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  unsigned long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  __syncthreads();
  if (lane == 31) sm.red64[w] = incl;
  if (threadIdx.x == 0) {
    sm.found_pos = 0x7FFFFFFF;
    sm.found_before = 0ull;
  }
  __syncthreads();
  unsigned long long warp_off = 0ull;
  for (int i = 0; i < w; ++i) warp_off += sm.red64[i];
  unsigned long long run = above + warp_off + incl - mine;
  int found = 0x7FFFFFFF;
  unsigned long long found_before = 0ull;
  for (int i = 0; i < per; ++i) {
    const int pos = p0 + i;
    if (pos >= nb) break;
    const int bin = desc ? nb - 1 - pos : pos;
    const unsigned long long mb = sm.mass[bin];
    if (sm.cnt[bin] > 0u && reaches(run + mb, t_hi, t_lo)) {
      found = pos;
      found_before = run;
      break;
    }
    run += mb;
  }
  atomicMin(&sm.found_pos, found);
  __syncthreads();
  if (found != 0x7FFFFFFF && found == sm.found_pos) sm.found_before = found_before;
  __syncthreads();
  int pos = sm.found_pos;
  if (pos == 0x7FFFFFFF) {
    // fallback: last non-empty bin in scan order
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long r = above;
      int last = -1;
      unsigned long long last_before = above;
      for (int q = 0; q < nb; ++q) {
        const int bin = desc ? nb - 1 - q : q;
        if (sm.cnt[bin] > 0u) {
          last = q;
          last_before = r;
        }
        r += sm.mass[bin];
      }
      sm.found_pos = last < 0 ? 0 : last;
      sm.found_before = last_before;
    }
    __syncthreads();
    pos = sm.found_pos;
  }
  *before = sm.found_before;
  const int bin = desc ? nb - 1 - pos : pos;
  __syncthreads();
  return bin;
}

// ---------------------------------------------------------------------------
// Kernel 1: per-row statistics
// ---------------------------------------------------------------------------
__device__ void target_row_stats(const VerifyParams& P, StatSmem& sm, int b, int k,
                                 float T, float top_p) {
  const int V = P.V, K = P.K;
  const int64_t roff = (static_cast<int64_t>(b) * (K + 1) + k) * V;
  const void* row = P.target_bf16 ? static_cast<const void*>(static_cast<const uint16_t*>(P.target) + roff)
                                  : static_cast<const void*>(static_cast<const float*>(P.target) + roff);
  const bool bf16 = P.target_bf16 != 0;
  TgtStats* out = static_cast<TgtStats*>(P.tstats) + static_cast<int64_t>(b) * (K + 1) + k;
  const int32_t d = k < K ? P.draft[static_cast<int64_t>(b) * K + k] : -1;

  // pass A: max of the scaled row
  float m = -INFINITY;
  row_walk_any(row, bf16, V, [&](int v, float t, bool valid) {
    if (valid) m = fmaxf(m, scale_logit(t, T));
  });
  m = block_max_f(m, sm);
  if (m == -INFINITY) {
    if (threadIdx.x == 0) {
      TgtStats s;
      s.m = m;
      s.D = 1.0f;
      s.kd_thr = 0u;
      s.id_thr = 0;
      s.p_d = d == 0 ? 1.0f : 0.0f;
      s.mode = kModeOneHot;
      s.amax_key = 0ull;
      *out = s;
    }
    return;
  }
  const bool topp = top_p < 1.0f;

  // pass B: total fixed-point mass (+ first histogram level)
  if (topp) hist_clear(sm, kBins);
  __syncthreads();
  unsigned long long F = 0ull;
  row_walk_any(row, bf16, V, [&](int v, float t, bool valid) {
    const float x = scale_logit(t, T);
    const unsigned long long f = valid ? to_fixed(exp_rel(x, m)) : 0ull;
    F += f;
    if (topp) hist_add(sm, valid, static_cast<int>(kd_of(x) >> 20), f, static_cast<uint32_t>(v));
  });
  F = block_sum_u64(F, sm);

  uint32_t kd_thr = 0u;
  int32_t id_thr = 0;
  unsigned long long Fk = F;
  int32_t mode = kModeKeepAll;
  if (topp) {
    mode = kModeThreshold;
    // P32 = rint(top_p * 2^32) in integer arithmetic on the fp32 bits
    unsigned long long P32 = 0ull;
    {
      const uint32_t pb = __float_as_uint(top_p);
      const int ex = static_cast<int>((pb >> 23) & 0xFFu);
      if (top_p > 0.0f && ex != 0) {
        const unsigned long long mant = (pb & 0x7FFFFFu) | 0x800000u;
        const int sh = ex - 127 - 23 + 32;  // top_p * 2^32 = mant * 2^sh
        if (sh >= 0) {
          P32 = mant << sh;
        } else {
          const int rs = -sh;
          if (rs <= 24) {
            const unsigned long long q = mant >> rs, rem = mant & ((1ull << rs) - 1ull),
                                     half = 1ull << (rs - 1);
            P32 = q + ((rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull);
          }
        }
      }
    }
    // target = P32 * F as 128 bits
    const unsigned long long t_lo = P32 * F;
    const unsigned long long t_hi = __umul64hi(P32, F);
    unsigned long long above = 0ull, before = 0ull;
    // kd stages: bits [31:20] (done in pass B), [19:8], [7:0]
    int bin = hist_find(sm, kBins, true, above, t_hi, t_lo, &before);
    above = before;
    uint32_t prefix = static_cast<uint32_t>(bin);  // fixed high bits of kd
    int fixed_bits = 12;
    bool resolved = false;
    if (sm.cnt[bin] == 1u) {
      id_thr = static_cast<int32_t>(sm.idmax[bin]);
      Fk = above + sm.mass[bin];
      resolved = true;
    }
    const int shifts[2] = {8, 0};
    const int widths[2] = {12, 8};
    for (int st = 0; st < 2 && !resolved; ++st) {
      const int sh = shifts[st], wd = widths[st];
      const int nb = 1 << wd;
      __syncthreads();
      hist_clear(sm, nb);
      __syncthreads();
      const uint32_t pre = prefix;
      const int fb = fixed_bits;
      row_walk_any(row, bf16, V, [&](int v, float t, bool valid) {
        const float x = scale_logit(t, T);
        const uint32_t kd = kd_of(x);
        const bool match = valid && (kd >> (32 - fb)) == pre;
        const unsigned long long f = match ? to_fixed(exp_rel(x, m)) : 0ull;
        hist_add(sm, match, static_cast<int>((kd >> sh) & ((1u << wd) - 1u)), f,
                 static_cast<uint32_t>(v));
      });
      __syncthreads();
      bin = hist_find(sm, nb, true, above, t_hi, t_lo, &before);
      above = before;
      prefix = (prefix << wd) | static_cast<uint32_t>(bin);
      fixed_bits += wd;
      if (sm.cnt[bin] == 1u) {
        id_thr = static_cast<int32_t>(sm.idmax[bin]);
        Fk = above + sm.mass[bin];
        resolved = true;
      }
    }
    if (resolved) {
      // boundary element known by id; its full kd from the element itself
      const float t = load_logit(row, bf16, id_thr);
      kd_thr = kd_of(scale_logit(t, T));
    } else {
      // exact ties at the boundary value: select among them by token id
      kd_thr = prefix;
      const int id_shifts[2] = {12, 0};
      uint32_t id_prefix = 0u;
      int id_fixed = 0;  // number of id bits fixed above bit 24
      for (int st = 0; st < 2 && !resolved; ++st) {
        const int sh = id_shifts[st];
        __syncthreads();
        hist_clear(sm, kBins);
        __syncthreads();
        const uint32_t ip = id_prefix;
        const int ifx = id_fixed;
        row_walk_any(row, bf16, V, [&](int v, float t, bool valid) {
          const float x = scale_logit(t, T);
          const uint32_t id = static_cast<uint32_t>(v);
          const bool match = valid && kd_of(x) == kd_thr &&
                             (ifx == 0 || (id >> (24 - ifx)) == ip);
          const unsigned long long f = match ? to_fixed(exp_rel(x, m)) : 0ull;
          hist_add(sm, match, static_cast<int>((id >> sh) & 0xFFFu), f, id);
        });
        __syncthreads();
        bin = hist_find(sm, kBins, false, above, t_hi, t_lo, &before);
        above = before;
        id_prefix = (id_prefix << 12) | static_cast<uint32_t>(bin);
        id_fixed += 12;
        if (sm.cnt[bin] == 1u || st == 1) {
          id_thr = static_cast<int32_t>(sm.idmax[bin]);
          Fk = above + sm.mass[bin];
          resolved = true;
        }
      }
    }
  }
  const float D = __fmul_rn(__ull2float_rn(Fk), 0x1p-40f);

  if (threadIdx.x == 0) {
    float p_d = 0.0f;
    if (d >= 0 && d < V) {
      const float x = scale_logit(load_logit(row, bf16, d), T);
      const uint32_t kd = kd_of(x);
      const bool keep = mode == kModeKeepAll || kd > kd_thr || (kd == kd_thr && d <= id_thr);
      p_d = keep ? __fdiv_rn(exp_rel(x, m), D) : 0.0f;
    }
    TgtStats s;
    s.m = m;
    s.D = D;
    s.kd_thr = kd_thr;
    s.id_thr = id_thr;
    s.p_d = p_d;
    s.mode = mode;
    s.amax_key = 0ull;
    *out = s;
  }
}

__device__ void target_row_greedy(const VerifyParams& P, StatSmem& sm, int b, int k) {
  const int V = P.V, K = P.K;
  const int64_t roff = (static_cast<int64_t>(b) * (K + 1) + k) * V;
  const void* row = P.target_bf16 ? static_cast<const void*>(static_cast<const uint16_t*>(P.target) + roff)
                                  : static_cast<const void*>(static_cast<const float*>(P.target) + roff);
  unsigned long long best = 0ull;
  row_walk_any(row, P.target_bf16 != 0, V, [&](int v, float t, bool valid) {
    if (valid) best = umax64(best, winner_key(t, static_cast<uint32_t>(v)));
  });
  best = block_max_u64(best, sm);
  if (threadIdx.x == 0) {
    TgtStats s;
    s.m = 0.f;
    s.D = 1.f;
    s.kd_thr = 0u;
    s.id_thr = 0;
    s.p_d = 0.f;
    s.mode = kModeGreedy;
    s.amax_key = best;
    *(static_cast<TgtStats*>(P.tstats) + static_cast<int64_t>(b) * (K + 1) + k) = s;
  }
}

__device__ void draft_row_stats(const VerifyParams& P, StatSmem& sm, int b, int k,
                                int64_t crow) {
  const int V = P.V, K = P.K;
  const int64_t roff = (crow * K + k) * V;
  const void* row = P.cache_bf16 ? static_cast<const void*>(static_cast<const uint16_t*>(P.cache) + roff)
                                 : static_cast<const void*>(static_cast<const float*>(P.cache) + roff);
  const bool bf16 = P.cache_bf16 != 0;
  DrfStats* out = static_cast<DrfStats*>(P.dstats) + static_cast<int64_t>(b) * K + k;
  const int32_t d = P.draft[static_cast<int64_t>(b) * K + k];
  float m = -INFINITY;
  row_walk_any(row, bf16, V, [&](int v, float c, bool valid) {
    if (valid && c == c) m = fmaxf(m, c);
  });
  m = block_max_f(m, sm);
  if (m == -INFINITY) {
    if (threadIdx.x == 0) {
      DrfStats s;
      s.m = m;
      s.D = 1.f;
      s.q_d = 0.f;
      s.zero = 1;
      *out = s;
    }
    return;
  }
  unsigned long long F = 0ull;
  row_walk_any(row, bf16, V, [&](int v, float c, bool valid) {
    const float x = (c != c) ? -INFINITY : c;
    if (valid) F += to_fixed(exp_rel(x, m));
  });
  F = block_sum_u64(F, sm);
  const float D = __fmul_rn(__ull2float_rn(F), 0x1p-40f);
  if (threadIdx.x == 0) {
    float q_d = 0.f;
    if (d >= 0 && d < V) {
      float c = load_logit(row, bf16, d);
      if (c != c) c = -INFINITY;
      q_d = __fdiv_rn(exp_rel(c, m), D);
    }
    DrfStats s;
    s.m = m;
    s.D = D;
    s.q_d = q_d;
    s.zero = 0;
    *out = s;
  }
}

__global__ void __launch_bounds__(kStatThreads, 2) verify_stats_kernel(VerifyParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  StatSmem& sm = *reinterpret_cast<StatSmem*>(smem_raw);
  const int K = P.K;
  const int nT = P.B * (K + 1);
  int b, k;
  bool is_target;
  if (static_cast<int>(blockIdx.x) < nT) {
    b = blockIdx.x / (K + 1);
    k = blockIdx.x % (K + 1);
    is_target = true;
  } else {
    const int r = blockIdx.x - nT;
    b = r / K;
    k = r % K;
    is_target = false;
  }
  const int32_t s = P.rsi[b];
  if (s < 0 || s >= P.S) return;  // padding or out of range (reported later)
  const float T = P.temperature[s];
  const bool greedy = !(T > 0.0f);
  if (is_target) {
    if (greedy)
      target_row_greedy(P, sm, b, k);
    else
      target_row_stats(P, sm, b, k, T, P.top_p[s]);
  } else {
    if (greedy || P.cache == nullptr) return;
    const int64_t crow = P.row_map ? P.row_map[s] : s;
    if (crow < 0 || crow >= P.C) return;
    draft_row_stats(P, sm, b, k, crow);
  }
}

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
__device__ __forceinline__ float p_at(const TgtStats& ts, float t, float T, int v) {
  if (ts.mode == kModeOneHot) return v == 0 ? 1.0f : 0.0f;
  const float x = scale_logit(t, T);
  if (ts.mode == kModeThreshold) {
    const uint32_t kd = kd_of(x);
    if (!(kd > ts.kd_thr || (kd == ts.kd_thr && v <= ts.id_thr))) return 0.0f;
  }
  return __fdiv_rn(exp_rel(x, ts.m), ts.D);
}

__device__ __forceinline__ float q_at(const DrfStats& ds, float c) {
  if (ds.zero) return 0.0f;
  const float x = (c != c) ? -INFINITY : c;
  return __fdiv_rn(exp_rel(x, ds.m), ds.D);
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
  const int64_t npos = rs.P0 + k - 1;
  unsigned long long best = 0ull;
  unsigned int any = 0u;
  for (int g = c0 + 4 * threadIdx.x; g < c1; g += 4 * kResThreads) {
    bool need = false;
    float w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int v = g + j;
      w[j] = 0.f;
      if (v < c1) {
        const float t = load_logit(P.target, P.target_bf16 != 0, toff + v);
        float pv = p_at(ts, t, rs.T, v);
        if (residual) {
          const float c = load_logit(P.cache, P.cache_bf16 != 0, coff + v);
          const float r = __fsub_rn(pv, q_at(ds, c));
          pv = r > 0.0f ? r : 0.0f;
        }
        w[j] = pv;
        need |= pv > 0.0f;
      }
    }
    if (!need) continue;
    any = 1u;
    const U4 r = noise_block(rs.seed, npos, static_cast<uint32_t>(g), kStreamTarget);
    const uint32_t words[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (w[j] > 0.0f) {
        const float y = __fadd_rn(logf(w[j]), gumbel_of(words[j]));
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

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  const int rows = p.B * (p.K + 1) + p.B * p.K;
  const size_t smem = sizeof(StatSmem);
  cudaError_t err = cudaFuncSetAttribute(verify_stats_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  verify_stats_kernel<<<rows, kStatThreads, smem, stream>>>(p);
  err = cudaGetLastError();
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
