// verify_stats.cu -- the verifier (one persistent launch) and the top-k
// candidate selection of the top-k Markov loop.
//
// The verifier follows vLLM PR #65007 Part 2 ("Temperature and top-p" and
// the rejection sampler): per request, the target rows after temperature
// (their maximum, exp-mass and, for a sampled row with top_p < 1, the exact
// keep set -- the smallest prefix by (logit desc, token id asc) whose 64-bit
// fixed-point mass reaches p, plus the row max), the draft rows' maximum and
// exp-mass, the accept/reject chain, and one categorical draw (residual,
// placeholder row or bonus row). Greedy target rows get their winner key.
// How the work is scheduled is described above verify_flat_kernel; the
// top-p select above flat_topp_row_t.
//
// The top-k selection (topk_rows_kernel, at the end of the file) runs one
// thread-block cluster per base-logit row and reduces through distributed
// shared memory; the helpers right below (RowSmem, cluster_reduce,
// cluster_find) serve it.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "verify_common.cuh"
#include "verify_draw.cuh"

namespace cg = cooperative_groups;

namespace dspark {

namespace {

constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowBins = 2048;

struct RowSmem {
  unsigned long long hmass[kRowBins];
  unsigned int hcnt[kRowBins];
  unsigned int hid[kRowBins];
  unsigned long long red64[kRowWarps];
  float redf[kRowWarps];
  // slots read by the other CTAs of the cluster
  int x_pos;
  unsigned long long x_key;
  unsigned long long x_sum;
  unsigned long long x_range;
  unsigned long long x_before;
  unsigned long long x_mass;
  unsigned int x_cnt;
  unsigned int x_id;
  unsigned int x_cmin;  // value-key range of the stage's candidates in this CTA
  unsigned int x_cmax;
  unsigned int x_pref;  // a per-CTA count for a cluster prefix
  unsigned int list_n;  // top-p candidates this CTA appended to its list
  // per-row reductions: one slot per CTA, two alternating sets (a row's slots
  // are rewritten only after the next row's first cluster barrier)
  unsigned long long c_sum[2];   // fixed-point mass
  unsigned int w_u32[kRowWarps];
  unsigned long long w_u64[kRowWarps];
  // block-local scratch
  int found_pos;
  int bcast_i;
  unsigned long long found_before;
  unsigned long long bcast_u;
  float bcast_f;
  int pad_[2];
};

struct Found {
  int bin;
  unsigned long long before;  // running mass before the bin
  unsigned int cnt;
  unsigned long long mass;
  unsigned int id;
  unsigned int kmin, kmax;    // value-key range of all the stage's candidates
};

__device__ unsigned long long block_sum_u64(unsigned long long v, RowSmem& sm) {
  v = warp_sum64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sm.red64[w] = v;
  __syncthreads();
  if (w == 0) {
    unsigned long long x = l < kRowWarps ? sm.red64[l] : 0ull;
    x = warp_sum64(x);
    if (l == 0) sm.red64[0] = x;
  }
  __syncthreads();
  return sm.red64[0];
}

// ---- cluster reductions of one value per thread --------------------------------
// The CTA reduces its warps through shared memory and thread 0 stores the
// result in the CTA's slot of the current set; after one cluster barrier warp
// 0 reads the CL slots of the cluster and broadcasts the result.
template <class T, class Op>
__device__ __forceinline__ T block_reduce(T v, T* wslots, T init, Op op) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  if ((threadIdx.x & 31) == 0) wslots[threadIdx.x >> 5] = v;
  __syncthreads();
  T r = init;
  if (threadIdx.x < 32) {
    r = threadIdx.x < kRowWarps ? wslots[threadIdx.x] : init;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r = op(r, __shfl_xor_sync(0xFFFFFFFFu, r, o));
  }
  return r;  // valid in warp 0
}

template <class T, class Op>
__device__ __forceinline__ T cluster_reduce(cg::cluster_group& cl, RowSmem& sm, T v, T* cslot,
                                            T* bcast, int CL, T init, Op op) {
  v = block_reduce<T>(v, reinterpret_cast<T*>(sizeof(T) == 4 ? static_cast<void*>(sm.w_u32)
                                                             : static_cast<void*>(sm.w_u64)),
                      init, op);
  if (threadIdx.x == 0) *cslot = v;
  cl.sync();
  if (threadIdx.x < 32) {
    T r = static_cast<int>(threadIdx.x) < CL ? *cl.map_shared_rank(cslot, threadIdx.x) : init;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r = op(r, __shfl_xor_sync(0xFFFFFFFFu, r, o));
    if (threadIdx.x == 0) *bcast = r;
  }
  __syncthreads();
  return *bcast;
}

__device__ unsigned long long cluster_sum_u64(cg::cluster_group& cl, RowSmem& sm,
                                              unsigned long long v, int set, int CL) {
  return cluster_reduce<unsigned long long>(
      cl, sm, v, &sm.c_sum[set], &sm.bcast_u, CL, 0ull,
      [](unsigned long long a, unsigned long long b) { return a + b; });
}

// ---- histograms -------------------------------------------------------------
__device__ void hist_clear(RowSmem& sm, int nb) {
  for (int i = threadIdx.x; i < nb; i += kRowThreads) {
    sm.hmass[i] = 0ull;
    sm.hcnt[i] = 0u;
    sm.hid[i] = 0u;
  }
}

// Adds (mass f, one count, id) to bin `bin` with shared-memory atomics (one
// per lane: the bins of a warp's 32 elements rarely collide).
__device__ __forceinline__ void hist_add(RowSmem& sm, bool active, int bin,
                                         unsigned long long f, uint32_t id) {
  if (!active) return;
  atomicAdd(&sm.hmass[bin], f);
  atomicAdd(&sm.hcnt[bin], 1u);
  atomicMax(&sm.hid[bin], id);
}

// Reduces the local histograms over the cluster and finds the first
// non-empty bin, in scan order (descending bin index if desc), at which the
// running mass (starting from `above`) reaches the target (t_hi:t_lo). Each
// thread passes the value-key range [kmin, kmax] of the candidates it saw
// (~0, 0: none); Found carries the range over the cluster. With counted =
// false the histogram holds masses only: a bin qualifies by its mass, and
// the count and id of the result are unknown (cnt reads 0).
__device__ Found cluster_find(cg::cluster_group& cl, RowSmem& sm, int nb, bool desc,
                              unsigned long long above, unsigned long long t_hi,
                              unsigned long long t_lo, int CL, int rank,
                              uint32_t kmin = 0xFFFFFFFFu, uint32_t kmax = 0u,
                              bool counted = true) {
  const int tid = threadIdx.x;
  const int b0 = rank * nb / CL;
  const int w = (rank + 1) * nb / CL - b0;
  __syncthreads();
  {
    const uint32_t lo = block_reduce<uint32_t>(kmin, sm.w_u32, 0xFFFFFFFFu,
                                               [](uint32_t a, uint32_t b) { return min(a, b); });
    if (tid == 0) sm.x_cmin = lo;
    __syncthreads();  // the warp slots are reused below
    const uint32_t hi = block_reduce<uint32_t>(kmax, sm.w_u32, 0u,
                                               [](uint32_t a, uint32_t b) { return max(a, b); });
    if (tid == 0) sm.x_cmax = hi;
    __syncthreads();
  }
  cl.sync();  // every local histogram and candidate range is complete
  // 1. reduce the bins this CTA owns over the cluster, in place: only this
  //    CTA reads any CTA's entries of its own range
  unsigned long long mine = 0ull;
  for (int bi = tid; bi < w; bi += kRowThreads) {
    unsigned long long bm = 0ull;
    unsigned int bc = 0u, bid = 0u;
    for (int r = 0; r < CL; ++r) {
      const RowSmem* o = cl.map_shared_rank(&sm, r);
      bm += o->hmass[b0 + bi];
      bc += o->hcnt[b0 + bi];
      bid = max(bid, o->hid[b0 + bi]);
    }
    sm.hmass[b0 + bi] = bm;
    sm.hcnt[b0 + bi] = bc;
    sm.hid[b0 + bi] = bid;
    mine += bm;
  }
  const unsigned long long range_mass = block_sum_u64(mine, sm);
  if (tid == 0) sm.x_range = range_mass;
  cl.sync();
  // 2. running mass before this CTA's range, in scan order
  if (tid < 32) {
    unsigned long long s = 0ull;
    const int r = tid;
    if (r < CL && (desc ? r > rank : r < rank)) s = *cl.map_shared_rank(&sm.x_range, r);
    s = warp_sum64(s);
    if (tid == 0) sm.bcast_u = s;
  }
  __syncthreads();
  const unsigned long long range_before = above + sm.bcast_u;
  // 3. scan the owned range: thread t takes positions [t*per, t*per+per)
  const int per = (w + kRowThreads - 1) / kRowThreads;
  const int p0 = tid * per;
  unsigned long long tsum = 0ull;
  for (int i = 0; i < per; ++i) {
    const int pos = p0 + i;
    if (pos < w) tsum += sm.hmass[desc ? b0 + w - 1 - pos : b0 + pos];
  }
  const int lane = tid & 31, wp = tid >> 5;
  unsigned long long incl = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long nv = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += nv;
  }
  __syncthreads();
  if (lane == 31) sm.red64[wp] = incl;
  if (tid == 0) sm.found_pos = 0x7FFFFFFF;
  __syncthreads();
  unsigned long long woff = 0ull;
  for (int i = 0; i < wp; ++i) woff += sm.red64[i];
  unsigned long long run = range_before + woff + incl - tsum;
  int found = 0x7FFFFFFF;
  unsigned long long fbefore = 0ull;
  for (int i = 0; i < per; ++i) {
    const int pos = p0 + i;
    if (pos >= w) break;
    const int bin = desc ? b0 + w - 1 - pos : b0 + pos;
    const unsigned long long mb = sm.hmass[bin];
    if ((counted ? sm.hcnt[bin] > 0u : mb > 0ull) && reaches(run + mb, t_hi, t_lo)) {
      found = pos;
      fbefore = run;
      break;
    }
    run += mb;
  }
  atomicMin(&sm.found_pos, found);
  __syncthreads();
  if (found != 0x7FFFFFFF && found == sm.found_pos) {
    const int bin = desc ? b0 + w - 1 - found : b0 + found;
    sm.x_pos = desc ? nb - 1 - bin : bin;  // global scan position
    sm.x_before = fbefore;
    sm.x_cnt = sm.hcnt[bin];
    sm.x_mass = sm.hmass[bin];
    sm.x_id = sm.hid[bin];
  }
  if (tid == 0 && sm.found_pos == 0x7FFFFFFF) sm.x_pos = 0x7FFFFFFF;
  cl.sync();
  // 4. the first qualifying bin over the cluster
  if (tid == 0) {
    int best_r = -1, best_pos = 0x7FFFFFFF;
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    for (int r = 0; r < CL; ++r) {
      const RowSmem* o = cl.map_shared_rank(&sm, r);
      const int p = o->x_pos;
      if (p < best_pos) {
        best_pos = p;
        best_r = r;
      }
      lo = min(lo, o->x_cmin);
      hi = max(hi, o->x_cmax);
    }
    sm.bcast_i = best_r;
    sm.w_u32[0] = lo;
    sm.w_u32[1] = hi;
  }
  __syncthreads();
  Found f;
  const int br = sm.bcast_i;
  if (br < 0) {  // cannot happen: the stage's set always holds the boundary
    f.bin = 0;
    f.before = above;
    f.cnt = 1u;
    f.mass = 0ull;
    f.id = 0u;
  } else {
    const RowSmem* o = cl.map_shared_rank(&sm, br);
    const int pos = o->x_pos;
    f.bin = desc ? nb - 1 - pos : pos;
    f.before = o->x_before;
    f.cnt = o->x_cnt;
    f.mass = o->x_mass;
    f.id = o->x_id;
  }
  f.kmin = sm.w_u32[0];
  f.kmax = sm.w_u32[1];
  cl.sync();  // slots may be rewritten by the next stage
  return f;
}

// Digits of the first two top-p stages: the distance to the maximum in bins
// of 1/64 (the last bin takes everything from 2047/64 on, -inf included),
// then 2048 sub-bins of bin a0. Both are non-decreasing in m - x (fp32
// rounding is monotone and the scalings are exact; for x in bin a0 the
// subtraction of a0 is exact), so bins follow the descending order of x and
// equal values share a bin.
__device__ __forceinline__ int adigit0(float x, float m) {
  return static_cast<int>(fminf(__fmul_rn(__fsub_rn(m, x), 64.0f), 2047.0f));
}
__device__ __forceinline__ int adigit1(float x, float m, int a0) {
  const float t = __fsub_rn(__fmul_rn(__fsub_rn(m, x), 64.0f), static_cast<float>(a0));
  return static_cast<int>(fminf(__fmul_rn(t, 2048.0f), 2047.0f));
}

// Reads of one row's slice [v0, v0 + n) straight from global memory, the
// eviction priority in L2 chosen by the caller (a top-p row's first passes
// keep it for the later ones); `fix` maps a raw value to x (temperature,
// NaN read as -inf). The sweeps read the few elements before the first
// 16-byte (fp32) or 8-byte (bf16) boundary one at a time, then 4 at a time.
struct RowView {
  const float* f;
  const uint16_t* h;
  bool bf16;
  int n;
};

template <int kU, bool kBf16, class Fix, class Body>
__device__ __forceinline__ void row_sweep_t(RowView rv, uint64_t pol, Fix fix, Body body);

// The dtype is decided once per sweep: each instantiation reads one format.
template <int kU = 8, class Fix, class Body>  // kU: 16-byte loads in flight per thread
__device__ __forceinline__ void row_sweep(const RowView& rv, uint64_t pol, Fix fix, Body body) {
  if (rv.bf16)
    row_sweep_t<kU, true>(rv, pol, fix, body);
  else
    row_sweep_t<kU, false>(rv, pol, fix, body);
}

// Elements before the slice's first vector-aligned address (16 bytes for
// fp32, 8 for bf16): a row of an odd-sized vocabulary starts anywhere.
template <bool kBf16>
__device__ __forceinline__ int aligned_head(const RowView& rv) {
  constexpr uintptr_t al = kBf16 ? 8 : 16;
  const uintptr_t a = kBf16 ? reinterpret_cast<uintptr_t>(rv.h) : reinterpret_cast<uintptr_t>(rv.f);
  const int head = static_cast<int>(((al - (a & (al - 1))) & (al - 1)) / (kBf16 ? 2 : 4));
  return head < rv.n ? head : rv.n;
}

template <int kU, bool kBf16, class Fix, class Body>
__device__ __forceinline__ void row_sweep_t(RowView rv, uint64_t pol, Fix fix, Body body) {
  const int tid = threadIdx.x;
  auto ld1 = [&](int i) -> float {
    return kBf16 ? bf16_bits_to_float(ld_hint_u16(rv.h + i, pol)) : ld_hint_f32(rv.f + i, pol);
  };
  auto ld4 = [&](int i, float (&v)[4]) {  // 4 values from aligned element index i
    if constexpr (kBf16) {
      const uint2 w = ld_hint_u2(rv.h + i, pol);
      v[0] = bf16_bits_to_float(static_cast<uint16_t>(w.x & 0xFFFFu));
      v[1] = bf16_bits_to_float(static_cast<uint16_t>(w.x >> 16));
      v[2] = bf16_bits_to_float(static_cast<uint16_t>(w.y & 0xFFFFu));
      v[3] = bf16_bits_to_float(static_cast<uint16_t>(w.y >> 16));
    } else {
      const float4 c = ld_hint_f4(rv.f + i, pol);
      v[0] = c.x;
      v[1] = c.y;
      v[2] = c.z;
      v[3] = c.w;
    }
  };
  // the few elements before the first aligned address, then 4 at a time
  const int head = aligned_head<kBf16>(rv);
  if (tid < head) body(tid, fix(ld1(tid)));
  const int n4 = (rv.n - head) >> 2;
  int i = tid;
  for (; i + (kU - 1) * kRowThreads < n4; i += kU * kRowThreads) {
    float v[kU][4];
#pragma unroll
    for (int u = 0; u < kU; ++u) ld4(head + 4 * (i + u * kRowThreads), v[u]);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int j = head + 4 * (i + u * kRowThreads);
#pragma unroll
      for (int e = 0; e < 4; ++e) body(j + e, fix(v[u][e]));
    }
  }
  for (; i < n4; i += kRowThreads) {
    float v[4];
    ld4(head + 4 * i, v);
#pragma unroll
    for (int e = 0; e < 4; ++e) body(head + 4 * i + e, fix(v[e]));
  }
  for (int t = head + 4 * n4 + tid; t < rv.n; t += kRowThreads) body(t, fix(ld1(t)));
}

// ---- rows kept whole: one pass, a deterministic fp32 online softmax sum -----
// (max m, s = sum of exp(x - m)) of the values a thread saw, in a fixed
// order; two such pairs combine into the pair of their union. The combine is
// commutative (fmaxf, and one fp32 addition of two products), so the
// butterfly reductions below give the same bits in every lane and every run.
__device__ __forceinline__ unsigned long long ms_pack(float m, float s) {
  return (static_cast<unsigned long long>(__float_as_uint(s)) << 32) | __float_as_uint(m);
}
__device__ __forceinline__ float ms_m(unsigned long long v) {
  return __uint_as_float(static_cast<uint32_t>(v));
}
__device__ __forceinline__ float ms_s(unsigned long long v) {
  return __uint_as_float(static_cast<uint32_t>(v >> 32));
}
// exp2 of (a - base) * log2(e) with base = 0 when the maximum is -inf (then
// every term is exp(-inf) = 0 rather than NaN)
__device__ __forceinline__ float ms_base(float m) { return m == -INFINITY ? 0.0f : m; }
__device__ __forceinline__ unsigned long long ms_combine(unsigned long long a,
                                                         unsigned long long b) {
  const float m = fmaxf(ms_m(a), ms_m(b));
  const float base = ms_base(m);
  const float s = __fadd_rn(__fmul_rn(ms_s(a), exp_rel(ms_m(a), base)),
                            __fmul_rn(ms_s(b), exp_rel(ms_m(b), base)));
  return ms_pack(m, s);
}

// One pass over the slice: per thread, chunks of up to kU x 4 values take
// one rescale of the running sum to the chunk's new maximum and one ex2 per
// value. known_m: the row maximum is known (recorded by the Markov loop), so
// no rescale is needed. Returns this thread's (m, s).
// Thread 0 keeps the slice's next pf_window bytes on their way into L2
// (cp.async.bulk.prefetch.L2), so that far more of the slice is in flight
// than the threads' own loads; a window rather than the whole slice keeps
// the bytes in flight over all CTAs well inside L2.
struct L2Window {
  uintptr_t base, end;  // the slice's bytes
  uintptr_t done;       // prefetched up to here
  uint32_t window;
  __device__ L2Window(const void* p, size_t bytes, uint32_t w)
      : base(reinterpret_cast<uintptr_t>(p)), end(reinterpret_cast<uintptr_t>(p) + bytes),
        done(reinterpret_cast<uintptr_t>(p) & ~static_cast<uintptr_t>(15)), window(w) {}
  // the threads have reached byte offset `at` of the slice
  __device__ __forceinline__ void advance(size_t at) {
    if (window == 0u) return;
    uintptr_t want = base + at + window;
    if (want > end) want = end;
    want &= ~static_cast<uintptr_t>(15);
    if (want > done + 4096u || (want == (end & ~static_cast<uintptr_t>(15)) && want > done)) {
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(done),
                   "r"(static_cast<uint32_t>(want - done))
                   : "memory");
      done = want;
    }
  }
};

template <int kU, bool kBf16, class Fix>
__device__ __forceinline__ unsigned long long slice_online_t(const RowView& rv, uint64_t pol,
                                                             Fix fix, bool known, float known_m,
                                                             uint32_t pf_window = 0u) {
  const int tid = threadIdx.x;
  float m = known ? known_m : -INFINITY;
  float s0 = 0.0f, s1 = 0.0f;
  constexpr int kEs = kBf16 ? 2 : 4;
  L2Window pf(kBf16 ? static_cast<const void*>(rv.h) : static_cast<const void*>(rv.f),
              static_cast<size_t>(rv.n) * kEs, tid == 0 ? pf_window : 0u);
  pf.advance(0);
  const unsigned long long l2e = f2_pack(kLog2e, kLog2e);
  // the few elements before the first aligned address, then 4 at a time
  const int head = aligned_head<kBf16>(rv);
  const float* af = rv.f + head;
  const uint16_t* ah = rv.h + head;
  const int an = rv.n - head;
  auto ld1 = [&](int i) -> float {  // element i of the slice
    return kBf16 ? bf16_bits_to_float(ld_hint_u16(rv.h + i, pol)) : ld_hint_f32(rv.f + i, pol);
  };
  auto load4 = [&](int j, float (&v)[4]) {  // aligned vector j
    if constexpr (kBf16) {
      const uint2 w = ld_hint_u2(ah + 4 * j, pol);
      v[0] = bf16_bits_to_float(static_cast<uint16_t>(w.x & 0xFFFFu));
      v[1] = bf16_bits_to_float(static_cast<uint16_t>(w.x >> 16));
      v[2] = bf16_bits_to_float(static_cast<uint16_t>(w.y & 0xFFFFu));
      v[3] = bf16_bits_to_float(static_cast<uint16_t>(w.y >> 16));
    } else {
      const float4 c = ld_hint_f4(af + 4 * j, pol);
      v[0] = c.x;
      v[1] = c.y;
      v[2] = c.z;
      v[3] = c.w;
    }
  };
  // the running sums follow the chunk's maximum; returns the subtraction base
  auto rescale = [&](float cm) -> float {
    if (known) return ms_base(m);
    const float mn = fmaxf(m, cm);
    const float base = ms_base(mn);
    const float f = exp_rel(m, base);  // 1 if the maximum did not move
    s0 = __fmul_rn(s0, f);
    s1 = __fmul_rn(s1, f);
    m = mn;
    return base;
  };
  auto add4 = [&](const float (&v)[4], float base) {
    const unsigned long long bb = f2_pack(base, base);
    float a, b, c, d;
    f2_unpack(f2_mul(f2_sub(f2_pack(v[0], v[1]), bb), l2e), a, b);
    f2_unpack(f2_mul(f2_sub(f2_pack(v[2], v[3]), bb), l2e), c, d);
    s0 = __fadd_rn(s0, ex2_approx(a));
    s1 = __fadd_rn(s1, ex2_approx(b));
    s0 = __fadd_rn(s0, ex2_approx(c));
    s1 = __fadd_rn(s1, ex2_approx(d));
  };
  auto add1 = [&](float x) {
    const float base = rescale(x);  // before s0 is read: rescale updates it
    s0 = __fadd_rn(s0, exp_rel(x, base));
  };
  if (tid < head) add1(fix(ld1(tid)));
  const int n4 = an >> 2;
  int i = tid;
  for (; i + (kU - 1) * kRowThreads < n4; i += kU * kRowThreads) {
    pf.advance(static_cast<size_t>(head) * kEs + static_cast<size_t>(i + kU * kRowThreads) * 4 * kEs);
    float v[kU][4];
#pragma unroll
    for (int u = 0; u < kU; ++u) load4(i + u * kRowThreads, v[u]);
    float cm = -INFINITY;
#pragma unroll
    for (int u = 0; u < kU; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[u][e] = fix(v[u][e]);
        cm = fmaxf(cm, v[u][e]);
      }
    const float base = rescale(cm);
#pragma unroll
    for (int u = 0; u < kU; ++u) add4(v[u], base);
  }
  for (; i < n4; i += kRowThreads) {
    float v[4];
    load4(i, v);
    float cm = -INFINITY;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[e] = fix(v[e]);
      cm = fmaxf(cm, v[e]);
    }
    add4(v, rescale(cm));
  }
  for (int t = head + 4 * n4 + tid; t < rv.n; t += kRowThreads) add1(fix(ld1(t)));
  return ms_pack(m, __fadd_rn(s0, s1));
}

template <class Fix>
__device__ __forceinline__ unsigned long long slice_online(const RowView& rv, uint64_t pol,
                                                           Fix fix, bool known, float known_m,
                                                           uint32_t pf_window = 0u) {
  if (rv.bf16) return slice_online_t<4, true>(rv, pol, fix, known, known_m, pf_window);
  return slice_online_t<4, false>(rv, pol, fix, known, known_m, pf_window);
}

// ---------------------------------------------------------------------------
// Verification in one launch: verify_flat_kernel, persistent CTAs (no
// clusters, four per SM, cooperative so that every CTA is resident) over one
// work queue. Row items come in request order (request b: target rows 0..K,
// then draft rows 0..K-1). A row kept whole (or a greedy row) is cut into
// `nslice` slices, one item per slice: a slice yields a partial (the online
// maximum and exp-sum, or the greedy winner key) and the CTA that finishes a
// row's last slice combines the partials in slice order (the same bits every
// run) into the row's statistics. A sampled target row with a top-p cut is
// one item, done whole by one CTA (flat_topp_row). The CTA that finishes a
// request's last row replays the request's accept chain (one thread per
// draft), writes the request's draw job and publishes `ndraw` draw items:
// column chunks of the one categorical the request needs. A CTA that finds
// the row queue empty takes draw items in publish order (four waves of
// chunks over the CTAs, so that the last requests' draws spread over many CTAs),
// waiting for a request still finishing its rows; the CTA that finishes a
// request's last chunk writes the outputs. (Taking published draws between
// row items was measured slower: requests publish at about the items'
// boundaries, so the draws ran late and delayed the rows claimed before
// them.) Each CTA claims its next row at the start of the current item, so
// the claim's latency hides behind the item's work. Every wait is bounded.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire_gpu(const unsigned int* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---- the flat kernels ------------------------------------------------------
struct RowPart {
  float m;                   // online maximum of the slice
  float s;                   // sum of exp(x - m) over the slice
  unsigned long long key;    // greedy rows: the slice's winner key
};

struct CtlView {
  unsigned int* draw_head;   // next draw item (its own 128-byte line)
  unsigned int* ready_count; // requests published (its own line)
  unsigned int* row_head;    // next row item (its own line)
  unsigned int* rows_done;   // [B] rows finished per request
  unsigned int* draws_done;  // [B] draw chunks finished per request
  unsigned int* ready;       // [B] request + 1, in publish order
  unsigned int* slices_done; // [B * (2K + 1)] slices finished per row
  DrawJob* jobs;             // [B] what each request's draw needs
  static constexpr int kHead = 96;  // words of the three queue lines
  __device__ CtlView(unsigned int* c, int B, int K)
      : draw_head(c), ready_count(c + 32), row_head(c + 64), rows_done(c + kHead),
        draws_done(c + kHead + B),
        ready(c + kHead + 2 * B), slices_done(c + kHead + 3 * B),
        jobs(reinterpret_cast<DrawJob*>(c + jobs_word(B, K))) {}
  static __host__ __device__ size_t jobs_word(int B, int K) {
    return (static_cast<size_t>(kHead) + 3 * static_cast<size_t>(B) +
            static_cast<size_t>(B) * (2 * K + 1) + 3) & ~size_t(3);
  }
};

struct FlatSmem {
  unsigned long long w_u64[kRowWarps];
  int last;          // this CTA finished a row / a request / a draw
  int bcast_i;
  int acc[DSPARK_MAX_STEPS];  // the chain replay's per-draft outcome
  int chunk;         // the draw item taken: its chunk, or -1 (none left)
  DrawJob job;       // the draw item's request
};

// Outcome of draft k of request b (thread k of the CTA that finished the
// request's rows): 1 accepted, 0 rejected, -1 placeholder, -2 out of range.
__device__ int chain_step(const VerifyParams& P, int b, int k, bool greedy, uint64_t seed,
                          int64_t P0) {
  const int K = P.K, V = P.V;
  const int32_t d = P.draft[static_cast<int64_t>(b) * K + k];
  if (d == -1) return -1;
  if (d < -1 || d >= V) return -2;
  const TgtStats* ts = static_cast<const TgtStats*>(P.tstats) + static_cast<int64_t>(b) * (K + 1) + k;
  if (greedy) return key_index(__ldcg(&ts->amax_key)) == d ? 1 : 0;
  const DrfStats* ds = static_cast<const DrfStats*>(P.dstats) + static_cast<int64_t>(b) * K + k;
  const U4 w = noise_block(seed, P0 + k - 1, 0u, kStreamAccept);
  return __fmul_rn(uniform_of(w.x), __ldcg(&ds->q_d)) < __ldcg(&ts->p_d) ? 1 : 0;
}

__device__ __forceinline__ TgtStats ld_tstats(const TgtStats* p) {
  TgtStats t;
  t.m = __ldcg(&p->m);
  t.D = __ldcg(&p->D);
  t.kd_thr = __ldcg(&p->kd_thr);
  t.id_thr = __ldcg(&p->id_thr);
  t.p_d = __ldcg(&p->p_d);
  t.mode = __ldcg(&p->mode);
  t.amax_key = __ldcg(&p->amax_key);
  return t;
}
__device__ __forceinline__ DrfStats ld_dstats(const DrfStats* p) {
  DrfStats d;
  d.m = __ldcg(&p->m);
  d.D = __ldcg(&p->D);
  d.q_d = __ldcg(&p->q_d);
  d.zero = __ldcg(&p->zero);
  return d;
}

// The whole CTA, after it finished a row of request b (that row's
// statistics written): count the row; the request's last row replays the
// accept chain (one thread per draft) and writes the request's draw job.
__device__ void request_row_done(const VerifyParams& P, const CtlView& C, FlatSmem& sm, int b) {
  const int tid = threadIdx.x, K = P.K;
  __syncthreads();  // every thread's part of the row is written
  if (tid == 0) {
    __threadfence();  // the row's statistics before the count
    sm.last = atomicAdd(&C.rows_done[b], 1u) + 1u == static_cast<unsigned int>(2 * K + 1);
    if (sm.last) __threadfence();  // every row's statistics are visible from here on
  }
  __syncthreads();
  if (!sm.last) return;
  const int32_t s = P.rsi[b];
  const bool valid_slot = s >= 0 && s < P.S;
  const float T = valid_slot ? P.temperature[s] : 0.0f;
  const bool greedy = !(T > 0.0f);
  const uint64_t seed = valid_slot ? P.seeds[s] : 0ull;
  const int64_t P0 = P.pos[b];
  if (valid_slot && tid < K) sm.acc[tid] = chain_step(P, b, tid, greedy, seed, P0);
  __syncthreads();
  if (tid == 0) {
    DrawJob J;
    J.b = b;
    J.mode = kDrawNone;
    J.row = 0;
    J.invalid = 0;
    J.crow = 0;
    J.P0 = P0;
    J.seed = seed;
    J.T = T;
    J.n_acc = 0;
    J.emit = -1;
    if (!valid_slot) {
      J.invalid = 1;
      if (s >= P.S) report(P.status, DSPARK_ERR_BOUNDS);
    } else if (!greedy) {
      if (P.cache == nullptr) {
        J.invalid = 1;
        report(P.status, DSPARK_ERR_INVALID_ARG);
      } else {
        J.crow = P.row_map ? P.row_map[s] : s;
        if (J.crow < 0 || J.crow >= P.C) {
          J.invalid = 1;
          report(P.status, DSPARK_ERR_BOUNDS);
        }
      }
    }
    if (!J.invalid) {
      int k = 0;
      bool placeholder = false;
      for (; k < K; ++k) {
        const int a = sm.acc[k];
        if (a == -2) {
          J.invalid = 1;
          report(P.status, DSPARK_ERR_BOUNDS);
          break;
        }
        if (a == -1) placeholder = true;
        if (a != 1) break;
      }
      if (!J.invalid) {
        J.n_acc = k;
        J.row = k;  // the row of the emitted token (K: the bonus row)
        const TgtStats* tst =
            static_cast<const TgtStats*>(P.tstats) + static_cast<int64_t>(b) * (K + 1);
        if (greedy) {
          J.emit = key_index(__ldcg(&tst[k].amax_key));
        } else {
          J.mode = (k < K && !placeholder) ? kDrawResidual : kDrawP;
          J.ts = ld_tstats(tst + k);
          if (J.mode == kDrawResidual)
            J.ds = ld_dstats(static_cast<const DrfStats*>(P.dstats) +
                             static_cast<int64_t>(b) * K + k);
        }
      }
    }
    C.jobs[b] = J;
    __threadfence();  // the job before the request is listed
    const unsigned int slot = atomicAdd(C.ready_count, 1u);
    atomicExch(&C.ready[slot], static_cast<unsigned int>(b + 1));
  }
}

// What a row needs from the flat kernel.
enum FlatRowKind : int {
  kFlatNone = 0,       // nothing to compute (padding, greedy draft row, top-p row done before)
  kFlatGreedy = 1,     // greedy target row: winner key of the raw row
  kFlatOnline = 2,     // max and exp-sum of the row (sampled target row kept whole, draft row)
  kFlatRecorded = 3,   // draft row whose statistics the Markov loop recorded
  kFlatTopp = 4        // sampled target row with a top-p cut: the exact select, whole
};
struct FlatRow {
  int kind;
  int b, k;
  bool is_target;
  bool bf16;
  float T;           // target rows: the temperature (1: none)
  int64_t off;       // element offset of the row in its tensor
  const void* base;
};

__device__ FlatRow classify_row(const VerifyParams& P, int b, int j) {
  const int K = P.K;
  FlatRow r;
  r.kind = kFlatNone;
  r.b = b;
  r.is_target = j <= K;
  r.k = r.is_target ? j : j - K - 1;
  r.bf16 = false;
  r.T = 1.0f;
  r.off = 0;
  r.base = nullptr;
  const int32_t s = P.rsi[b];
  if (s < 0 || s >= P.S) return r;
  const float T = P.temperature[s];
  const bool greedy = !(T > 0.0f);
  if (r.is_target) {
    r.kind = greedy ? kFlatGreedy : (P.top_p[s] < 1.0f ? kFlatTopp : kFlatOnline);
    r.T = greedy ? 1.0f : T;
    r.off = (static_cast<int64_t>(b) * (K + 1) + r.k) * P.V;
    r.base = P.target;
    r.bf16 = P.target_bf16 != 0;
    return r;
  }
  if (greedy || P.cache == nullptr) return r;
  const int64_t crow = P.row_map ? P.row_map[s] : s;
  if (crow < 0 || crow >= P.C) return r;
  r.kind = kFlatOnline;
  if (P.stats_items) {
    const float mrec = __ldcg(&P.draft_stats[static_cast<int64_t>(b) * K + r.k].m);
    if (mrec == mrec) r.kind = kFlatRecorded;
  }
  r.off = (crow * K + r.k) * P.V;
  r.base = P.cache;
  r.bf16 = P.cache_bf16 != 0;
  return r;
}

// Bytes of the L2 prefetch window a slice keeps ahead of its loads.
constexpr uint32_t kSliceWindow = 48u << 10;

// ---- top-p rows inside the flat kernel: one CTA per row ---------------------
// The keep set of a sampled row with top_p < 1 (vLLM PR #65007 Part 2,
// "Temperature and top-p"): the smallest prefix, in the order of larger x
// first and lower token id on ties, whose 2^40 fixed-point mass reaches
// top_p times the row's total F. Two passes over the row find it in the
// common case:
//  1. the maximum m, and a count histogram of the values in bins of 1/128 of
//     a logit unit around an anchor (the largest of 256 values spread over
//     the row); the counts, weighted by exp at the bin centres, estimate
//     where the cumulative mass reaches top_p, and so a window of distance
//     bins (1/64 unit below m, the bins of the exact select) around the
//     boundary;
//  2. the exact F, the exact mass of every element above the window, and a
//     list (token id, x) of the elements inside it.
// The exact mass of each window bin then comes from the list, and the
// boundary bin is the one where the exact running mass first reaches the
// target; its elements are split further from the list alone (stages 1-6
// below). When the estimate missed (the boundary lies outside the window)
// or the list overflowed, the row takes the exact select: a third pass with
// the full distance-bin mass histogram (stage 0), then the stages, sweeping
// the row again if the boundary bin's candidates do not fit in the list.
// Either way the result is the same exact boundary.
struct TopSmem {
  unsigned long long hmass[kRowBins];  // pass 1: the count histogram (kTopFine words)
  unsigned int hcnt[kRowBins];
  unsigned int hid[kRowBins];
  unsigned long long red64[2 * kRowWarps];
  unsigned long long wmass[kRowWarps][8];  // window-bin masses per warp
  unsigned int wcnt[kRowWarps][8];
  unsigned int wlen[kRowWarps];            // entries in each warp's list segment
  unsigned int cand_n;                     // candidates of the boundary bin
  unsigned int red32[2 * kRowWarps];
  float redf[kRowWarps];
  int found_pos;
  int f_bin;
  unsigned long long f_before, f_mass;
  unsigned int f_cnt, f_id, f_kmin, f_kmax;
  unsigned int list_n;
  int fast_ok;
  float bcast_f;
};

// pass-1 histogram: kTopFine bins of 1/128 unit, from kTopFineTop above the
// anchor down (the first and last bins also take everything beyond)
constexpr int kTopFine = 4096;
constexpr float kTopFineTop = 12.0f;
static_assert(kTopFine * sizeof(unsigned int) <= sizeof(unsigned long long) * kRowBins,
              "the pass-1 histogram lives in the stage histogram's words");
// distance bins on each side of the estimated boundary bin kept exact in pass 2
constexpr int kTopWin = 2;
static_assert(2 * kTopWin + 1 <= 8, "window bins per warp slot");
// each warp's share of the CTA's list in pass 2, and the candidates that the
// boundary bin may hold for the sort below
constexpr int kTopSeg = kVerifyListCap / kRowWarps;
constexpr int kTopSort = 1024;
static_assert(kTopSort * sizeof(unsigned long long) <= sizeof(unsigned long long) * kRowBins,
              "the sort keys live in the stage histogram's words");

struct BFound {
  int bin;
  unsigned long long before;  // running mass before the bin
  unsigned long long mass;
  unsigned int cnt, id;
  unsigned int kmin, kmax;    // value-key range of all the stage's candidates
};

__device__ void top_hist_clear(TopSmem& t, int nb) {
  for (int i = threadIdx.x; i < nb; i += kRowThreads) {
    t.hmass[i] = 0ull;
    t.hcnt[i] = 0u;
    t.hid[i] = 0u;
  }
}

// The first bin, in scan order (descending bin index if desc), whose running
// mass from `above` reaches the target (t_hi:t_lo): a bin qualifies if it
// holds an element (counted) or mass (mass-only histogram). Thread t scans a
// run of nb / 256 bins; an exclusive prefix over the block gives each run's
// start. Every thread returns the same result.
__device__ BFound block_find(TopSmem& t, int nb, bool desc, unsigned long long above,
                             unsigned long long t_hi, unsigned long long t_lo, uint32_t kmin,
                             uint32_t kmax, bool counted) {
  const int tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
  __syncthreads();  // the histogram is complete
  // the candidates' value-key range
  {
    uint32_t lo = kmin, hi = kmax;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, o));
    }
    if (lane == 0) {
      t.red32[wp] = lo;
      t.red32[kRowWarps + wp] = hi;
    }
  }
  const int per = nb / kRowThreads;
  const int p0 = tid * per;
  auto bin_at = [&](int pos) { return desc ? nb - 1 - pos : pos; };
  unsigned long long tsum = 0ull;
  for (int i = 0; i < per; ++i) tsum += t.hmass[bin_at(p0 + i)];
  unsigned long long incl = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long nv = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += nv;
  }
  if (lane == 31) t.red64[wp] = incl;
  if (tid == 0) t.found_pos = 0x7FFFFFFF;
  __syncthreads();
  unsigned long long woff = 0ull;
  for (int i = 0; i < wp; ++i) woff += t.red64[i];
  unsigned long long run = above + woff + incl - tsum;
  int found = 0x7FFFFFFF;
  unsigned long long fbefore = 0ull;
  for (int i = 0; i < per; ++i) {
    const int bin = bin_at(p0 + i);
    const unsigned long long mb = t.hmass[bin];
    if ((counted ? t.hcnt[bin] > 0u : mb > 0ull) && reaches(run + mb, t_hi, t_lo)) {
      found = p0 + i;
      fbefore = run;
      break;
    }
    run += mb;
  }
  atomicMin(&t.found_pos, found);
  __syncthreads();
  if (found != 0x7FFFFFFF && found == t.found_pos) {
    const int bin = bin_at(found);
    t.f_bin = bin;
    t.f_before = fbefore;
    t.f_mass = t.hmass[bin];
    t.f_cnt = t.hcnt[bin];
    t.f_id = t.hid[bin];
  }
  if (tid == 0) {
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    for (int i = 0; i < kRowWarps; ++i) {
      lo = min(lo, t.red32[i]);
      hi = max(hi, t.red32[kRowWarps + i]);
    }
    t.f_kmin = lo;
    t.f_kmax = hi;
    if (t.found_pos == 0x7FFFFFFF) {  // cannot happen: the stage's set holds the boundary
      t.f_bin = 0;
      t.f_before = above;
      t.f_mass = 0ull;
      t.f_cnt = 1u;
      t.f_id = 0u;
    }
  }
  __syncthreads();
  BFound f;
  f.bin = t.f_bin;
  f.before = t.f_before;
  f.mass = t.f_mass;
  f.cnt = t.f_cnt;
  f.id = t.f_id;
  f.kmin = t.f_kmin;
  f.kmax = t.f_kmax;
  __syncthreads();  // the slots may be rewritten by the next stage
  return f;
}

// Block sums of two values (every thread gets both).
__device__ void block_sum64x2(TopSmem& t, unsigned long long& a, unsigned long long& b) {
  a = warp_sum64(a);
  b = warp_sum64(b);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    t.red64[threadIdx.x >> 5] = a;
    t.red64[kRowWarps + (threadIdx.x >> 5)] = b;
  }
  __syncthreads();
  a = 0ull;
  b = 0ull;
  for (int i = 0; i < kRowWarps; ++i) {
    a += t.red64[i];
    b += t.red64[kRowWarps + i];
  }
  __syncthreads();
}

__device__ unsigned long long block_sum64(TopSmem& t, unsigned long long v) {
  unsigned long long z = 0ull;
  block_sum64x2(t, v, z);
  return v;
}

__device__ __forceinline__ float warp_maxf(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// x of a raw target value: divided by the temperature (correctly rounded, by
// Markstein's FMA form where it holds, as temp_div2), NaN read as -inf.
template <bool kScale>
struct TempFix {
  float T = 1.0f, r = 1.0f;
  bool slow = false;
  unsigned long long r2 = 0ull, nt2 = 0ull;
  __device__ explicit TempFix(float T_) : T(T_) {
    if constexpr (kScale) {
      r = __frcp_rn(T);
      slow = !temp_div_t_ok(T);
      r2 = f2_pack(r, r);
      nt2 = f2_pack(-T, -T);
    }
  }
  __device__ __forceinline__ float one(float z) const {
    if constexpr (!kScale) {
      return fmaxf(z, -INFINITY);
    } else {
      float x;
      if (slow || !temp_div_fast_ok(z)) {
        x = __fdiv_rn(z, T);
      } else {
        const float q = __fmul_rn(z, r);
        x = __fmaf_rn(__fmaf_rn(q, -T, z), r, q);
      }
      return fmaxf(x, -INFINITY);
    }
  }
  __device__ __forceinline__ void four(const float (&z)[4], float (&x)[4]) const {
    if constexpr (!kScale) {
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = fmaxf(z[e], -INFINITY);
    } else {
      f2_unpack(temp_div2(f2_pack(z[0], z[1]), r2, nt2, slow), x[0], x[1]);
      f2_unpack(temp_div2(f2_pack(z[2], z[3]), r2, nt2, slow), x[2], x[3]);
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = fmaxf(x[e], -INFINITY);
    }
  }
};

// A sweep that hands `body4` the four raw values of each aligned group
// (element index of the first) and `body1` the single values of the
// unaligned head and the ragged tail, each with a flag that says whether the
// values are the row's (false: padding to keep the warp together). Every
// loop runs the same trip count in all 32 lanes of a warp, so a body may use
// full-warp votes. Thread 0 keeps pf_window bytes of the row on their way
// into L2 (L2Window).
template <int kU, bool kBf16, class Body4, class Body1>
__device__ __forceinline__ void row_quads_t(const RowView& rv, uint64_t pol, uint32_t pf_window,
                                            Body4 body4, Body1 body1) {
  const int tid = threadIdx.x, lane = tid & 31;
  constexpr int kEs = kBf16 ? 2 : 4;
  L2Window pf(kBf16 ? static_cast<const void*>(rv.h) : static_cast<const void*>(rv.f),
              static_cast<size_t>(rv.n) * kEs, tid == 0 ? pf_window : 0u);
  pf.advance(0);
  const int head = aligned_head<kBf16>(rv);
  auto ld1 = [&](int i) -> float {
    return kBf16 ? bf16_bits_to_float(ld_hint_u16(rv.h + i, pol)) : ld_hint_f32(rv.f + i, pol);
  };
  auto load4 = [&](int i, float (&v)[4]) {  // 4 values from aligned element index i
    if constexpr (kBf16) {
      const uint2 w = ld_hint_u2(rv.h + i, pol);
      v[0] = bf16_bits_to_float(static_cast<uint16_t>(w.x & 0xFFFFu));
      v[1] = bf16_bits_to_float(static_cast<uint16_t>(w.x >> 16));
      v[2] = bf16_bits_to_float(static_cast<uint16_t>(w.y & 0xFFFFu));
      v[3] = bf16_bits_to_float(static_cast<uint16_t>(w.y >> 16));
    } else {
      const float4 c = ld_hint_f4(rv.f + i, pol);
      v[0] = c.x;
      v[1] = c.y;
      v[2] = c.z;
      v[3] = c.w;
    }
  };
  const int n4 = (rv.n - head) >> 2;
  const int tail0 = head + 4 * n4;  // the ragged tail: fewer than 4 values
  if (tid < 32) {                   // warp 0: the head and the tail, at most 3 values each
    const bool hv = lane < head;
    body1(lane, hv ? ld1(lane) : 0.0f, hv);
    const bool tv = tail0 + lane < rv.n;
    body1(tail0 + lane, tv ? ld1(tail0 + lane) : 0.0f, tv);
  }
  int i = tid;
  const int w0 = tid - lane;  // this warp's first thread: the loops' bounds are the warp's
  for (; w0 + (i - tid) + 31 + (kU - 1) * kRowThreads < n4; i += kU * kRowThreads) {
    pf.advance(static_cast<size_t>(head) * kEs + static_cast<size_t>(i + kU * kRowThreads) * 4 * kEs);
    float v[kU][4];
#pragma unroll
    for (int u = 0; u < kU; ++u) load4(head + 4 * (i + u * kRowThreads), v[u]);
#pragma unroll
    for (int u = 0; u < kU; ++u) body4(head + 4 * (i + u * kRowThreads), v[u], true);
  }
  for (; w0 + (i - tid) < n4; i += kRowThreads) {
    const bool ok = i < n4;
    float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (ok) load4(head + 4 * i, v);
    body4(head + 4 * i, v, ok);
  }
}

// The pass-2 sums of one thread. The mass f = rint(e 2^40) of an element
// is taken in two exact fp32 pieces, h = floor(e 2^20) and l = rint of the
// rest times 2^20 (f = h 2^20 + l, ties to even as rint), each read from
// the mantissa of a sum with 2^23; the 32-bit sums of their bit patterns
// are folded into 64-bit totals every kFold elements, before they could
// wrap (kFold (2^20 + 1) < 2^31).
struct MassSums {
  static constexpr uint32_t kBias = 0x4B000000u;  // bits of 2^23
  static constexpr uint32_t kFold = 1024u;
  unsigned long long F = 0ull, A = 0ull;  // all elements; elements above the window
  uint32_t h = 0u, l = 0u, n = 0u, ha = 0u, la = 0u, na = 0u;
  __device__ __forceinline__ void add(uint32_t hb, uint32_t lb, bool above) {
    h += hb;
    l += lb;
    ++n;
    if (above) {
      ha += hb;
      la += lb;
      ++na;
    }
  }
  __device__ __forceinline__ void fold() {
    F += (static_cast<unsigned long long>(h - n * kBias) << 20) +
         static_cast<unsigned long long>(l - n * kBias);
    A += (static_cast<unsigned long long>(ha - na * kBias) << 20) +
         static_cast<unsigned long long>(la - na * kBias);
    h = l = n = ha = la = na = 0u;
  }
};

// Appends to a warp's own list segment: every lane of the warp calls it
// with the same `n` (entries so far, kept in a register); no atomics.
__device__ __forceinline__ void seg_append(uint2* seg, unsigned int& n, bool want, uint32_t id,
                                           float x) {
  const unsigned int bal = __ballot_sync(0xFFFFFFFFu, want);
  const int lane = threadIdx.x & 31;
  if (want) {
    const unsigned int at = n + static_cast<unsigned int>(__popc(bal & ((1u << lane) - 1u)));
    if (at < static_cast<unsigned int>(kTopSeg)) seg[at] = make_uint2(id, __float_as_uint(x));
  }
  n += static_cast<unsigned int>(__popc(bal));
}

// x from its order key (ordered_bits, x not NaN)
__device__ __forceinline__ float x_of_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// The boundary element among the boundary bin's nc candidates (order keys
// in key[0, nc): value key << 32 | ~id): a bitonic sort into descending key
// order (x descending, id ascending) with E keys per thread in registers --
// exchanges between threads of a warp by shuffles, between warps through
// shared memory -- then running masses in that order from `above`; the
// element where the running mass first reaches the target writes its id,
// mass and the mass before it to t.f_id, t.f_mass, t.f_before.
template <int E>
__device__ void topp_sort_find(TopSmem& t, unsigned long long* key, unsigned int nc, float m,
                               unsigned long long above, unsigned long long t_hi,
                               unsigned long long t_lo) {
  constexpr unsigned int np = kRowThreads * E;
  const unsigned int tid = threadIdx.x, lane = tid & 31u, wp = tid >> 5;
  unsigned long long k[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const unsigned int i = tid * E + e;
    k[e] = i < nc ? key[i] : 0ull;  // 0 sorts last
  }
  for (unsigned int ks = 2; ks <= np; ks <<= 1) {
    for (unsigned int jj = ks >> 1; jj > 0; jj >>= 1) {
      if (jj < static_cast<unsigned int>(E)) {  // both keys in this thread
        // (the partner's register index must be a constant: jj is 1 or 2)
        auto local = [&](auto J) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            constexpr int kJ = decltype(J)::value;
            const int p = e ^ kJ;
            if (p > e) {
              const bool desc = ((tid * E + e) & ks) == 0u;
              const unsigned long long a = k[e], b = k[p];
              const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
              k[e] = desc ? hi : lo;
              k[p] = desc ? lo : hi;
            }
          }
        };
        if constexpr (E >= 2) {
          if (jj == 1u) local(std::integral_constant<int, 1>{});
        }
        if constexpr (E >= 4) {
          if (jj == 2u) local(std::integral_constant<int, 2>{});
        }
      } else {
        unsigned long long other[E];
        if (jj < 32u * E) {  // the partner is in this warp
#pragma unroll
          for (int e = 0; e < E; ++e) other[e] = __shfl_xor_sync(0xFFFFFFFFu, k[e], jj / E);
        } else {             // in another warp
          __syncthreads();   // the last readers of key[] are done
#pragma unroll
          for (int e = 0; e < E; ++e) key[tid * E + e] = k[e];
          __syncthreads();
#pragma unroll
          for (int e = 0; e < E; ++e) other[e] = key[(tid * E + e) ^ jj];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const unsigned int i = tid * E + e;
          const bool keep_max = (((i & ks) == 0u) == ((i & jj) == 0u));
          const unsigned long long a = k[e], b = other[e];
          k[e] = keep_max ? (a > b ? a : b) : (a > b ? b : a);
        }
      }
    }
  }
  unsigned long long fm[E];
  unsigned long long mine = 0ull;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    fm[e] = tid * E + e < nc ? fixed_mass(exp_rel(x_of_key(static_cast<uint32_t>(k[e] >> 32)), m))
                             : 0ull;
    mine += fm[e];
  }
  unsigned long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long nv = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= static_cast<unsigned int>(o)) incl += nv;
  }
  __syncthreads();  // t.red64 is free
  if (lane == 31u) t.red64[wp] = incl;
  __syncthreads();
  unsigned long long run = above + incl - mine;
  for (unsigned int i = 0; i < wp; ++i) run += t.red64[i];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (fm[e] > 0ull && !reaches(run, t_hi, t_lo) && reaches(run + fm[e], t_hi, t_lo)) {
      t.f_id = 0xFFFFFFFFu - static_cast<uint32_t>(k[e]);
      t.f_mass = fm[e];
      t.f_before = run;
    }
    run += fm[e];
  }
}

// ---- bf16 rows at temperature 1: the exact top-p from a value histogram -------
// A bf16 row holds at most 2^16 distinct values. Set apart the few values of
// magnitude below 2^-10 (listed one by one) and every other value is one bin
// of a histogram keyed by its order key with the small-magnitude keys removed
// (the compact key): each bin holds one value, so the fixed-point mass of a
// bin is its count times that value's mass, exactly. Every value whose mass is
// not 0 (x > m - 28.5) lies within 4096 compact keys below m, so pass 1 (HBM)
// takes the maximum and counts the values into 4096 bins below a top set
// from the anchor; F, the boundary value and the number r of its columns kept
// follow from the bins; pass 2 (L2) finds the r-th column holding the boundary
// value, in column order. A row whose maximum is above the bins, whose values
// below the bins could carry mass, or whose boundary lies among more listed
// small values than the sort takes is left to the general select.
constexpr uint32_t kOkNegBig = 0x457Fu;   // order key of -2^-10
constexpr uint32_t kOkPosBig = 0xBA80u;   // order key of +2^-10
constexpr uint32_t kTinyKeys = kOkPosBig - kOkNegBig - 1u;
constexpr uint32_t kCkMax = 0xFF80u - kTinyKeys;  // compact key of +inf
constexpr int kValBins = 4096;

// order key of bf16 bits (not NaN): larger value, larger key
__device__ __forceinline__ uint32_t bf16_okey(uint32_t b) {
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}
__device__ __forceinline__ uint32_t ckey_of_okey(uint32_t ok) {
  return ok <= kOkNegBig ? ok : ok - kTinyKeys;
}
__device__ __forceinline__ uint32_t bits_of_ckey(uint32_t ck) {
  const uint32_t ok = ck <= kOkNegBig ? ck : ck + kTinyKeys;
  return (ok & 0x8000u) ? (ok & 0x7FFFu) : (~ok & 0xFFFFu);
}

// Returns true when it wrote the row's statistics; false leaves the row to
// the general select (nothing written).
__device__ bool topp_bf16_exact(const VerifyParams& P, const FlatRow& R, TopSmem& t) {
  const int tid = threadIdx.x, lane = tid & 31, wp = tid >> 5, K = P.K, V = P.V;
  const uint16_t* h = static_cast<const uint16_t*>(R.base) + R.off;
  RowView rv;
  rv.bf16 = true;
  rv.f = nullptr;
  rv.h = h;
  rv.n = V;
  unsigned int* cnt = reinterpret_cast<unsigned int*>(t.hmass);  // kValBins words
  uint2* tiny = P.cand + static_cast<size_t>(blockIdx.x) * kVerifyListCap;
  const uint64_t pol_keep = policy_evict_last();
  const uint64_t pol_last = policy_evict_first();

  // ---- the anchor, and the bins' top: 512 compact keys above it ------------------
  uint32_t top;
  {
    const int at = static_cast<int>((static_cast<long long>(tid) * V) / kRowThreads);
    const uint32_t b = h[at];
    uint32_t ok = (b & 0x7FFFu) > 0x7F80u ? 0u : bf16_okey(b);
    ok = __reduce_max_sync(0xFFFFFFFFu, ok);
    for (int i = tid; i < kValBins; i += kRowThreads) cnt[i] = 0u;
    if (lane == 0) t.red32[wp] = ok;
    if (tid == 0) {
      t.list_n = 0u;
      t.fast_ok = 0;  // set: a value above the bins
    }
    __syncthreads();
    uint32_t aok = 0u;
    for (int i = 0; i < kRowWarps; ++i) aok = max(aok, t.red32[i]);
    const uint32_t ca = aok >= kOkPosBig ? ckey_of_okey(aok) : (aok <= kOkNegBig ? aok : kOkNegBig + 1u);
    top = min(ca + 512u, kCkMax);
  }
  const uint32_t bottom = top >= static_cast<uint32_t>(kValBins - 1) ? top - (kValBins - 1) : 0u;

  // ---- pass 1 (HBM): the maximum, the value counts, the small values -------------
  uint32_t mok = 0u;  // the largest order key (0: no value but NaN)
  auto count1 = [&](int j, float z) {
    const uint32_t b = __float_as_uint(z) >> 16;  // the bf16 bits
    const uint32_t mag = b & 0x7FFFu;
    if (mag > 0x7F80u) return;  // NaN
    const uint32_t ok = bf16_okey(b);
    mok = max(mok, ok);
    if (mag < 0x3A80u) {  // |x| < 2^-10: listed
      const unsigned int at = atomicAdd(&t.list_n, 1u);
      if (at < static_cast<unsigned int>(kVerifyListCap)) tiny[at] = make_uint2(static_cast<uint32_t>(j), b);
      return;
    }
    const uint32_t ck = ckey_of_okey(ok);
    if (ck > top) {
      t.fast_ok = 1;
    } else if (ck >= bottom) {
      atomicAdd(&cnt[top - ck], 1u);
    }
  };
  row_quads_t<4, true>(
      rv, pol_keep, kSliceWindow,
      [&](int j, const float (&z)[4], bool ok) {
        if (!ok) return;
#pragma unroll
        for (int e = 0; e < 4; ++e) count1(j + e, z[e]);
      },
      [&](int j, float z, bool ok) {
        if (ok) count1(j, z);
      });
  mok = __reduce_max_sync(0xFFFFFFFFu, mok);
  if (lane == 0) t.red32[kRowWarps + wp] = mok;
  __syncthreads();
  mok = 0u;
  for (int i = 0; i < kRowWarps; ++i) mok = max(mok, t.red32[kRowWarps + i]);
  const unsigned int ntiny = t.list_n;
  const int32_t d = R.k < K ? P.draft[static_cast<int64_t>(R.b) * K + R.k] : -1;
  TgtStats* ts = static_cast<TgtStats*>(P.tstats) + static_cast<int64_t>(R.b) * (K + 1) + R.k;
  if (mok <= 0x007Fu) {  // no value above -inf: p is one-hot at column 0
    if (tid == 0) {
      ts->m = -INFINITY;
      ts->D = 1.0f;
      ts->kd_thr = 0u;
      ts->id_thr = 0;
      ts->p_d = d == 0 ? 1.0f : 0.0f;
      ts->mode = kModeOneHot;
      ts->amax_key = 0ull;
    }
    return true;
  }
  const uint32_t mbits = (mok & 0x8000u) ? (mok & 0x7FFFu) : (~mok & 0xFFFFu);
  const float m = __uint_as_float(mbits << 16);
  // left to the general select: a maximum of +inf or of magnitude below 2^-10,
  // a value above the bins, an overfull list of small values, or values below
  // the bins that could carry mass
  if (!(m < INFINITY) || (mbits & 0x7FFFu) < 0x3A80u || t.fast_ok != 0 ||
      ntiny > static_cast<unsigned int>(kVerifyListCap))
    return false;
  if (bottom > 0x007Fu &&
      fixed_mass(exp_rel(__uint_as_float(bits_of_ckey(bottom - 1u) << 16), m)) != 0ull)
    return false;

  // ---- F, and the boundary: bins in descending value order, the small values
  // after the bin of +2^-10 (the last positive one) --------------------------------
  constexpr int per = kValBins / kRowThreads;
  const int j0 = tid * per;
  const int bp = static_cast<int>(top) - static_cast<int>(kOkNegBig + 1u);  // bin of +2^-10
  unsigned long long tiny_mass = 0ull;
  for (unsigned int q = tid; q < ntiny; q += kRowThreads) {
    const uint2 e = __ldcg(tiny + q);
    tiny_mass += fixed_mass(exp_rel(__uint_as_float(e.y << 16), m));
  }
  unsigned long long mine = 0ull;
#pragma unroll 4
  for (int q = 0; q < per; ++q) {
    const unsigned int c = cnt[j0 + q];
    if (c != 0u) {
      const float x = __uint_as_float(bits_of_ckey(top - static_cast<uint32_t>(j0 + q)) << 16);
      mine += static_cast<unsigned long long>(c) * fixed_mass(exp_rel(x, m));
    }
  }
  unsigned long long T = tiny_mass;
  block_sum64x2(t, mine, T);  // every thread: the bins' total (mine) and the small values'
  // (bp past the last bin: the small values lie below the bins, and the
  // check above made their mass 0; bp below 0: m < 0 and there are none)
  const bool tiny_in = bp >= 0 && bp < kValBins;
  const unsigned long long Fb = mine;
  const unsigned long long F = Fb + (tiny_in ? T : 0ull);
  const unsigned long long P32 = topp_scaled(P.top_p[P.rsi[R.b]]);
  const unsigned long long t_lo = P32 * F, t_hi = __umul64hi(P32, F);
  // this thread's run of bins (the small values' mass with the run holding bp)
  unsigned long long tsum = 0ull;
  for (int q = 0; q < per; ++q) {
    const unsigned int c = cnt[j0 + q];
    if (c != 0u) {
      const float x = __uint_as_float(bits_of_ckey(top - static_cast<uint32_t>(j0 + q)) << 16);
      tsum += static_cast<unsigned long long>(c) * fixed_mass(exp_rel(x, m));
    }
    if (tiny_in && j0 + q == bp) tsum += T;
  }
  unsigned long long incl = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long nv = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += nv;
  }
  if (lane == 31) t.red64[wp] = incl;
  if (tid == 0) t.found_pos = -1;
  __syncthreads();
  unsigned long long run = incl - tsum;
  for (int i = 0; i < wp; ++i) run += t.red64[i];
  for (int q = 0; q < per; ++q) {
    const int b = j0 + q;
    const unsigned int c = cnt[b];
    if (c != 0u) {
      const float x = __uint_as_float(bits_of_ckey(top - static_cast<uint32_t>(b)) << 16);
      const unsigned long long mb = static_cast<unsigned long long>(c) * fixed_mass(exp_rel(x, m));
      if (mb > 0ull && !reaches(run, t_hi, t_lo) && reaches(run + mb, t_hi, t_lo)) {
        t.found_pos = b;
        t.f_before = run;
      }
      run += mb;
    }
    if (tiny_in && b == bp) {
      if (T > 0ull && !reaches(run, t_hi, t_lo) && reaches(run + T, t_hi, t_lo)) {
        t.found_pos = kValBins;  // among the small values
        t.f_before = run;
      }
      run += T;
    }
  }
  __syncthreads();
  const int fb = t.found_pos;
  const unsigned long long before = t.f_before;
  __syncthreads();
  if (fb < 0) return false;  // cannot happen: the target is at most F
  uint32_t id_thr, vbits;
  unsigned long long kept;
  if (fb == kValBins) {
    // ---- the boundary among the small values: sort them (value desc, id asc) -----
    if (ntiny > static_cast<unsigned int>(kTopSort)) return false;
    unsigned long long* key = reinterpret_cast<unsigned long long*>(t.hmass);
    for (unsigned int q = tid; q < ntiny; q += kRowThreads) {
      const uint2 e = __ldcg(tiny + q);
      key[q] = (static_cast<unsigned long long>(kd_of(__uint_as_float(e.y << 16))) << 32) |
               static_cast<unsigned long long>(0xFFFFFFFFu - e.x);
    }
    unsigned int np = kRowThreads;
    while (np < ntiny) np <<= 1;
    if (tid == 0) {
      t.f_id = 0u;
      t.f_mass = 0ull;
      t.f_before = before;
    }
    __syncthreads();
    if (np == kRowThreads) topp_sort_find<1>(t, key, ntiny, m, before, t_hi, t_lo);
    else if (np == 2 * kRowThreads) topp_sort_find<2>(t, key, ntiny, m, before, t_hi, t_lo);
    else topp_sort_find<4>(t, key, ntiny, m, before, t_hi, t_lo);
    __syncthreads();
    id_thr = t.f_id;
    kept = t.f_before + t.f_mass;
    vbits = h[id_thr];
  } else {
    // ---- the boundary value: r of its columns are kept, the first r in column
    // order; pass 2 (L2) counts its columns per run of 2^sh columns ------------------
    vbits = bits_of_ckey(top - static_cast<uint32_t>(fb));
    const unsigned long long fv = fixed_mass(exp_rel(__uint_as_float(vbits << 16), m));
    const unsigned int c = cnt[fb];
    // r: the fewest columns with before + r fv reaching the target (1 <= r <= c)
    unsigned int lo_r = 1u, hi_r = c;
    while (lo_r < hi_r) {
      const unsigned int mid = (lo_r + hi_r) >> 1;
      if (reaches(before + static_cast<unsigned long long>(mid) * fv, t_hi, t_lo)) hi_r = mid;
      else lo_r = mid + 1u;
    }
    const unsigned int r = lo_r;
    kept = before + static_cast<unsigned long long>(r) * fv;
    int sh = 7;
    while ((static_cast<long long>(V) >> sh) >= kRowBins) ++sh;
    unsigned int* runs = t.hcnt;  // kRowBins words
    __syncthreads();              // cnt (in hmass) is read; runs are cleared next
    for (int i = tid; i < kRowBins; i += kRowThreads) runs[i] = 0u;
    __syncthreads();
    row_quads_t<4, true>(
        rv, pol_last, kSliceWindow,
        [&](int j, const float (&z)[4], bool ok) {
          if (!ok) return;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if ((__float_as_uint(z[e]) >> 16) == vbits) atomicAdd(&runs[(j + e) >> sh], 1u);
        },
        [&](int j, float z, bool ok) {
          if (ok && (__float_as_uint(z) >> 16) == vbits) atomicAdd(&runs[j >> sh], 1u);
        });
    __syncthreads();
    // the run holding the r-th column: a prefix over the runs (8 per thread)
    constexpr int rper = kRowBins / kRowThreads;
    unsigned int rs = 0u;
    for (int q = 0; q < rper; ++q) rs += runs[tid * rper + q];
    unsigned int rin = rs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned int nv = __shfl_up_sync(0xFFFFFFFFu, rin, o);
      if (lane >= o) rin += nv;
    }
    if (lane == 31) t.red32[wp] = rin;
    if (tid == 0) t.found_pos = -1;
    __syncthreads();
    unsigned int racc = rin - rs;
    for (int i = 0; i < wp; ++i) racc += t.red32[i];
    for (int q = 0; q < rper; ++q) {
      const unsigned int cq = runs[tid * rper + q];
      if (racc < r && racc + cq >= r) {
        t.found_pos = tid * rper + q;
        t.f_cnt = r - racc;  // the r-th overall is this run's (r - racc)-th
      }
      racc += cq;
    }
    __syncthreads();
    const int run_id = t.found_pos;
    const unsigned int nth = t.f_cnt;
    if (run_id < 0) return false;  // cannot happen: the value has c >= r columns
    // warp 0 walks the run's columns in order
    if (wp == 0) {
      const int c0 = run_id << sh, c1 = min(V, (run_id + 1) << sh);
      unsigned int seen = 0u;
      int found = -1;
      for (int b0 = c0; b0 < c1 && found < 0; b0 += 32) {
        const int j = b0 + lane;
        const bool hit = j < c1 && static_cast<uint32_t>(h[j]) == vbits;
        const unsigned int bal = __ballot_sync(0xFFFFFFFFu, hit);
        const unsigned int k = nth - seen;  // 1-based within this chunk
        if (static_cast<unsigned int>(__popc(bal)) >= k) {
          // the k-th set bit of bal
          unsigned int bb = bal;
          for (unsigned int i = 1u; i < k; ++i) bb &= bb - 1u;
          found = b0 + __ffs(bb) - 1;
        }
        seen += static_cast<unsigned int>(__popc(bal));
      }
      if (lane == 0) t.f_id = static_cast<uint32_t>(found < 0 ? 0 : found);
    }
    __syncthreads();
    id_thr = t.f_id;
  }
  if (tid == 0) {
    const float D = __fmul_rn(__ull2float_rn(kept), 0x1p-40f);
    const uint32_t kd_thr = kd_of(__uint_as_float(vbits << 16));
    const bool has_d = d >= 0 && d < V;
    const float x = has_d ? fmaxf(__uint_as_float(static_cast<uint32_t>(h[d]) << 16), -INFINITY) : 0.0f;
    const uint32_t kd = kd_of(x);
    const bool keep = kd > kd_thr || (kd == kd_thr && d <= static_cast<int32_t>(id_thr));
    ts->p_d = has_d && keep ? __fdiv_rn(exp_rel(x, m), D) : 0.0f;
    ts->m = m;
    ts->D = D;
    ts->kd_thr = kd_thr;
    ts->id_thr = static_cast<int32_t>(id_thr);
    ts->mode = kModeThreshold;
    ts->amax_key = 0ull;
  }
  return true;
}

template <bool kBf16, bool kScale>
__device__ void flat_topp_row_t(const VerifyParams& P, const FlatRow& R, TopSmem& t) {
  if constexpr (kBf16 && !kScale) {
    if (topp_bf16_exact(P, R, t)) return;
    __syncthreads();  // the general select reuses the shared memory
  }
  const int tid = threadIdx.x, lane = tid & 31, wp = tid >> 5, K = P.K, V = P.V;
  const TempFix<kScale> fx(R.T);
  auto fix = [&](float c) { return fx.one(c); };
  RowView rv;
  rv.bf16 = kBf16;
  rv.f = static_cast<const float*>(R.base) + R.off;
  rv.h = static_cast<const uint16_t*>(R.base) + R.off;
  rv.n = V;
  const uint64_t pol_keep = policy_evict_last();   // read again by a later pass
  const uint64_t pol_last = policy_evict_first();  // the last full pass
  const int32_t d = R.k < K ? P.draft[static_cast<int64_t>(R.b) * K + R.k] : -1;
  TgtStats* ts = static_cast<TgtStats*>(P.tstats) + static_cast<int64_t>(R.b) * (K + 1) + R.k;
  auto raw_at = [&](int v) -> float {
    return kBf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(R.base)[R.off + v])
                 : static_cast<const float*>(R.base)[R.off + v];
  };
  uint2* list = P.cand + static_cast<size_t>(blockIdx.x) * kVerifyListCap;
  unsigned int* fine = reinterpret_cast<unsigned int*>(t.hmass);

  // ---- the anchor: the largest of 256 values spread over the row ----------------
  float anchor;
  {
    const int at = static_cast<int>((static_cast<long long>(tid) * V) / kRowThreads);
    const float v = warp_maxf(fix(raw_at(at)));
    for (int i = tid; i < kTopFine; i += kRowThreads) fine[i] = 0u;
    if (lane == 0) t.red32[wp] = __float_as_uint(v);
    __syncthreads();
    anchor = -INFINITY;
    for (int i = 0; i < kRowWarps; ++i) anchor = fmaxf(anchor, __uint_as_float(t.red32[i]));
    if (!(anchor > -INFINITY && anchor < INFINITY)) anchor = 0.0f;  // any anchor is valid
  }
  // ---- pass 1 (HBM): the maximum and the count histogram ------------------------
  // With a temperature in the range where the division is monotone and
  // finite (T in [2^-30, 2^30]) the pass reads z itself: the correctly
  // rounded z / T is non-decreasing in z, so the maximum of x is the
  // quotient of the maximum of z (NaN read as -inf on both sides), and the
  // histogram, an estimate only, bins z times an approximate 128 / T.
  const bool by_z = kScale && temp_div_t_ok(R.T);
  const float c128 = __fmul_rn(__fadd_rn(anchor, kTopFineTop), 128.0f);
  const float s128 = by_z ? __fmul_rn(128.0f, __frcp_rn(R.T)) : 128.0f;
  float mx = -INFINITY;
  auto count1 = [&](float y) {
    // bin = floor((anchor + top - x) 128), clamped to the histogram; v >= 0
    // keeps the sum with 2^23 in [2^23, inf] and so the index in range
    const float v = fmaxf(__fmaf_rn(y, -s128, c128), 0.0f);
    const int b = static_cast<int>(__float_as_uint(__fadd_rz(v, 8388608.0f)) - MassSums::kBias);
    atomicAdd(&fine[min(b, kTopFine - 1)], 1u);
  };
  row_quads_t<4, kBf16>(
      rv, pol_keep, kSliceWindow,
      [&](int, const float (&z)[4], bool ok) {
        if (!ok) return;
        float x[4];
        if (by_z) {
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] = fmaxf(z[e], -INFINITY);
        } else {
          fx.four(z, x);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          mx = fmaxf(mx, x[e]);
          count1(x[e]);
        }
      },
      [&](int, float z, bool ok) {
        if (!ok) return;
        const float x = by_z ? fmaxf(z, -INFINITY) : fix(z);
        mx = fmaxf(mx, x);
        count1(x);
      });
  mx = warp_maxf(mx);
  if (by_z) mx = fix(mx);
  if (lane == 0) t.red32[kRowWarps + wp] = __float_as_uint(mx);
  if (tid == 0) {
    t.found_pos = 0x7FFFFFFF;
    t.cand_n = 0u;
  }
  __syncthreads();  // the histogram is complete
  float m = -INFINITY;
  for (int i = 0; i < kRowWarps; ++i) m = fmaxf(m, __uint_as_float(t.red32[kRowWarps + i]));
  if (m == -INFINITY) {  // no value above -inf: p is one-hot at column 0
    if (tid == 0) {
      ts->m = m;
      ts->D = 1.0f;
      ts->kd_thr = 0u;
      ts->id_thr = 0;
      ts->p_d = d == 0 ? 1.0f : 0.0f;
      ts->mode = kModeOneHot;
      ts->amax_key = 0ull;
    }
    return;
  }
  const int32_t s = P.rsi[R.b];
  const unsigned long long P32 = topp_scaled(P.top_p[s]);

  // ---- the estimated boundary and its window of distance bins -------------------
  // (every branch below depends on shared values only: uniform over the CTA)
  bool fast = m < INFINITY;
  int lo = 0, hi = -1;
  if (fast) {
    constexpr int per = kTopFine / kRowThreads;
    const int j0 = tid * per;
    const float top = __fadd_rn(anchor, kTopFineTop);
    auto centre = [&](int j) { return __fsub_rn(top, (static_cast<float>(j) + 0.5f) * 0.0078125f); };
    float est[per];
    float sum = 0.0f;
#pragma unroll
    for (int q = 0; q < per; ++q) {
      const unsigned int c = fine[j0 + q];
      est[q] = c ? __fmul_rn(static_cast<float>(c), exp_rel(fminf(centre(j0 + q), m), m)) : 0.0f;
      sum += est[q];
    }
    float incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float nv = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += nv;
    }
    if (lane == 31) t.redf[wp] = incl;
    __syncthreads();
    float total = 0.0f, woff = 0.0f;
    for (int i = 0; i < kRowWarps; ++i) {
      total += t.redf[i];
      if (i < wp) woff += t.redf[i];
    }
    const float target = __fmul_rn(P.top_p[s], total);
    float run = woff + incl - sum;
    int found = 0x7FFFFFFF;
    for (int q = 0; q < per; ++q) {
      run += est[q];
      if (fine[j0 + q] != 0u && run >= target) {
        found = j0 + q;
        break;
      }
    }
    atomicMin(&t.found_pos, found);
    __syncthreads();
    const int jf = t.found_pos;
    fast = jf != 0x7FFFFFFF;
    if (fast) {
      const float cj = fminf(centre(jf), m);
      const int g = static_cast<int>(fminf(__fmul_rn(__fsub_rn(m, cj), 64.0f), 2047.0f));
      lo = max(g - kTopWin, 0);
      hi = min(g + kTopWin, kRowBins - 1);
    }
  }

  // ---- pass 2 (L2): exact F, the exact mass above the window, the window's list -
  // An element's distance bin is trunc((m - x) 64) (adigit0); with
  // d = x - m (one rounding, d = -(m - x) exactly) the bin is below lo when
  // d > -lo / 64 and at most hi when d > -(hi + 1) / 64: the scalings by
  // powers of two are exact, so the tests on d decide exactly as the bins.
  unsigned long long F = 0ull, above = 0ull;
  int a0 = 0;
  uint2* seg = list + wp * kTopSeg;
  unsigned int seg_n = 0u;
  if (fast) {
    MassSums ms;
    const unsigned long long mm = f2_pack(m, m), l2e = f2_pack(kLog2e, kLog2e);
    const unsigned long long p20 = f2_pack(0x1p20f, 0x1p20f), c23 = f2_pack(8388608.0f, 8388608.0f);
    const float d_lo = -static_cast<float>(lo) * 0.015625f;
    const float d_hi = hi == kRowBins - 1 ? -INFINITY : -static_cast<float>(hi + 1) * 0.015625f;
    // two elements: their masses into the sums; returns the in-window bits
    auto pair = [&](float x0, float x1, bool ok) -> uint32_t {
      const unsigned long long dd = f2_sub(f2_pack(x0, x1), mm);
      float t0, t1, d0, d1;
      f2_unpack(f2_mul(dd, l2e), t0, t1);
      f2_unpack(dd, d0, d1);
      const unsigned long long a = f2_mul(f2_pack(ex2_approx(t0), ex2_approx(t1)), p20);
      const unsigned long long hb = f2_add_rz(a, c23);
      const unsigned long long lb = f2_fma(f2_sub(a, f2_sub(hb, c23)), p20, c23);
      if (ok) {
        ms.add(static_cast<uint32_t>(hb), static_cast<uint32_t>(lb), d0 > d_lo);
        ms.add(static_cast<uint32_t>(hb >> 32), static_cast<uint32_t>(lb >> 32), d1 > d_lo);
      }
      return ok ? ((d0 <= d_lo && d0 > d_hi ? 1u : 0u) | (d1 <= d_lo && d1 > d_hi ? 2u : 0u)) : 0u;
    };
    row_quads_t<4, kBf16>(
        rv, pol_last, kSliceWindow,
        [&](int j, const float (&z)[4], bool ok) {
          float x[4];
          fx.four(z, x);
          const uint32_t w = pair(x[0], x[1], ok) | (pair(x[2], x[3], ok) << 2);
          if (__any_sync(0xFFFFFFFFu, w != 0u)) {
#pragma unroll
            for (int e = 0; e < 4; ++e) seg_append(seg, seg_n, (w >> e) & 1u, j + e, x[e]);
          }
          if (ms.n >= MassSums::kFold - 4u) ms.fold();
        },
        [&](int j, float z, bool ok) {
          const float x = fix(z);
          const float dd = __fsub_rn(x, m);
          const float a = __fmul_rn(ex2_approx(__fmul_rn(dd, kLog2e)), 0x1p20f);
          const float hb = __fadd_rz(a, 8388608.0f);
          const float lb = __fmaf_rn(__fsub_rn(a, __fsub_rn(hb, 8388608.0f)), 0x1p20f, 8388608.0f);
          if (ok) ms.add(__float_as_uint(hb), __float_as_uint(lb), dd > d_lo);
          seg_append(seg, seg_n, ok && dd <= d_lo && dd > d_hi, j, x);
          if (ms.n >= MassSums::kFold - 4u) ms.fold();
        });
    ms.fold();
    F = ms.F;
    above = ms.A;
    if (lane == 0) t.wlen[wp] = seg_n;
    block_sum64x2(t, F, above);  // synchronises: every segment is complete
    for (int w = 0; w < kRowWarps; ++w) fast = fast && t.wlen[w] <= static_cast<unsigned int>(kTopSeg);
  }
  const unsigned long long t_lo = P32 * F, t_hi = __umul64hi(P32, F);
  BFound f;
  f.cnt = 0u;
  if (fast) {
    // the exact mass and count of each window bin, each warp from its own
    // segment; then warp 0 finds the bin where the exact running mass from
    // `above` first reaches the target
    constexpr int kW = 2 * kTopWin + 1;
    unsigned long long mw[kW];
    unsigned int cw[kW];
#pragma unroll
    for (int q = 0; q < kW; ++q) {
      mw[q] = 0ull;
      cw[q] = 0u;
    }
    unsigned int bad = 0u;
    for (unsigned int j = lane; j < seg_n; j += 32) {
      const float x = __uint_as_float(__ldcg(seg + j).y);
      const int q = adigit0(x, m) - lo;
      bad |= static_cast<uint32_t>(q) > static_cast<uint32_t>(hi - lo) ? 1u : 0u;
      const unsigned long long fm = fixed_mass(exp_rel(x, m));
#pragma unroll
      for (int k = 0; k < kW; ++k) {
        mw[k] += q == k ? fm : 0ull;
        cw[k] += q == k ? 1u : 0u;
      }
    }
#pragma unroll
    for (int k = 0; k < kW; ++k) {
      mw[k] = warp_sum64(mw[k]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cw[k] += __shfl_xor_sync(0xFFFFFFFFu, cw[k], o);
    }
    bad = __reduce_or_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < kW; ++k) {
        t.wmass[wp][k] = mw[k];
        t.wcnt[wp][k] = cw[k] | (bad << 31);
      }
    }
    __syncthreads();
    if (wp == 0) {
      unsigned long long mb = 0ull;
      unsigned int cb = 0u, bd = 0u;
      if (lane <= hi - lo) {
        for (int w = 0; w < kRowWarps; ++w) {
          mb += t.wmass[w][lane];
          cb += t.wcnt[w][lane] & 0x7FFFFFFFu;
          bd |= t.wcnt[w][lane] >> 31;
        }
      }
      unsigned long long incl = mb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long nv = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += nv;
      }
      const unsigned long long run = above + incl - mb;
      const unsigned int hit =
          __ballot_sync(0xFFFFFFFFu, lane <= hi - lo && mb > 0ull && reaches(run + mb, t_hi, t_lo));
      // no bin reaches (the boundary lies below the window), the mass above
      // the window already reaches (it lies above), a listed element outside
      // the window, or more candidates than the sort takes: the exact select
      const int qf = hit ? __ffs(hit) - 1 : 0;
      const unsigned int cf = __shfl_sync(0xFFFFFFFFu, cb, qf);
      const bool ok = hit != 0u && !__any_sync(0xFFFFFFFFu, bd != 0u) &&
                      !reaches(above, t_hi, t_lo) && cf <= static_cast<unsigned int>(kTopSort);
      if (lane == qf) {
        t.f_bin = lo + qf;
        t.f_before = run;
        t.f_cnt = cb;
      }
      if (lane == 0) t.fast_ok = ok ? 1 : 0;
    }
    __syncthreads();
    fast = t.fast_ok != 0;
    a0 = t.f_bin;
    above = t.f_before;
  }
  if (fast) {
    // ---- the boundary bin's candidates, sorted: x descending, id ascending ----
    unsigned long long* key = reinterpret_cast<unsigned long long*>(t.hmass);
    const unsigned int nc = t.f_cnt;
    unsigned int np = kRowThreads;
    while (np < nc) np <<= 1;
    for (unsigned int j0 = 0; j0 < seg_n; j0 += 32) {  // the same trip count in every lane
      const unsigned int j = j0 + static_cast<unsigned int>(lane);
      bool in = false;
      uint2 e = make_uint2(0u, 0u);
      if (j < seg_n) {
        e = __ldcg(seg + j);
        in = adigit0(__uint_as_float(e.y), m) == a0;
      }
      const unsigned int bal = __ballot_sync(0xFFFFFFFFu, in);
      if (bal == 0u) continue;
      unsigned int base = 0u;
      if (lane == 0) base = atomicAdd(&t.cand_n, static_cast<unsigned int>(__popc(bal)));
      base = __shfl_sync(0xFFFFFFFFu, base, 0);
      if (in) {
        const unsigned int at = base + static_cast<unsigned int>(__popc(bal & ((1u << lane) - 1u)));
        if (at < static_cast<unsigned int>(kTopSort))
          key[at] = (static_cast<unsigned long long>(kd_of(__uint_as_float(e.y))) << 32) |
                    static_cast<unsigned long long>(0xFFFFFFFFu - e.x);
      }
    }
    if (tid == 0) {  // found below; a valid token id whatever happens
      t.f_id = 0u;
      t.f_mass = 0ull;
      t.f_before = above;
    }
    __syncthreads();
    if (np == kRowThreads) topp_sort_find<1>(t, key, nc, m, above, t_hi, t_lo);
    else if (np == 2 * kRowThreads) topp_sort_find<2>(t, key, nc, m, above, t_hi, t_lo);
    else topp_sort_find<4>(t, key, nc, m, above, t_hi, t_lo);
    __syncthreads();
    f.id = t.f_id;
    f.mass = t.f_mass;
    above = t.f_before;
    f.cnt = 1u;
  }

  // ---- otherwise the exact select: pass 2' (L2), the stage-0 histogram ----------
  unsigned int list_len = 0xFFFFFFFFu;  // not built yet
  unsigned long long tt_lo = t_lo, tt_hi = t_hi;
  if (!fast) {
    top_hist_clear(t, kRowBins);
    __syncthreads();
    unsigned long long Fx = 0ull;
    row_sweep_t<4, kBf16>(rv, pol_keep, fix, [&](int, float x) {
      const unsigned long long fm = fixed_mass(exp_rel(x, m));
      Fx += fm;
      atomicAdd(&t.hmass[adigit0(x, m)], fm);
    });
    F = block_sum64(t, Fx);
    tt_lo = P32 * F;
    tt_hi = __umul64hi(P32, F);
    // stage 0: distance bins, ascending (mass only: stage 1 always runs)
    f = block_find(t, kRowBins, false, 0ull, tt_hi, tt_lo, 0xFFFFFFFFu, 0u, false);
    f.cnt = 0u;
    above = f.before;
    a0 = f.bin;
  }
  int a1 = -1;
  int kd_len = 0, id_len = 0;
  uint32_t kd_pre = 0u, id_pre = 0u;
  for (int stage = 1; f.cnt != 1u && stage <= 6; ++stage) {
    const int c_a1 = a1, c_kl = kd_len, c_il = id_len;
    const uint32_t c_kp = kd_pre, c_ip = id_pre;
    auto match = [=](float x, uint32_t kd, uint32_t id) {
      if (adigit0(x, m) != a0) return false;
      if (c_a1 >= 0 && adigit1(x, m, a0) != c_a1) return false;
      if (c_kl > 0 && (kd >> (32 - c_kl)) != c_kp) return false;
      if (c_il > 0 && (id >> (22 - c_il)) != c_ip) return false;
      return true;
    };
    auto digit = [=](float x, uint32_t kd, uint32_t id) -> int {
      switch (stage) {
        case 1: return adigit1(x, m, a0);
        case 2: return static_cast<int>(kd >> 21);
        case 3: return static_cast<int>((kd >> 10) & 0x7FFu);
        case 4: return static_cast<int>(kd & 0x3FFu);
        case 5: return static_cast<int>((id >> 11) & 0x7FFu);
        default: return static_cast<int>(id & 0x7FFu);
      }
    };
    const int nb = stage == 4 ? 1024 : kRowBins;
    const bool desc = stage >= 2 && stage <= 4;  // larger kd first; distance and id ascending
    top_hist_clear(t, nb);
    if (stage == 1 && tid == 0) t.list_n = 0u;
    __syncthreads();
    uint32_t cmin = 0xFFFFFFFFu, cmax = 0u;  // value-key range of the candidates
    auto visit = [&](uint32_t id, float x, bool append) {
      const uint32_t kd = kd_of(x);
      if (match(x, kd, id)) {
        const int bin = digit(x, kd, id);
        atomicAdd(&t.hmass[bin], fixed_mass(exp_rel(x, m)));
        atomicAdd(&t.hcnt[bin], 1u);
        atomicMax(&t.hid[bin], id);
        cmin = min(cmin, kd);
        cmax = max(cmax, kd);
        if (append) {
          const unsigned int at = atomicAdd(&t.list_n, 1u);
          if (at < static_cast<unsigned int>(kVerifyListCap)) list[at] = make_uint2(id, __float_as_uint(x));
        }
      }
    };
    const bool from_list = list_len <= static_cast<unsigned int>(kVerifyListCap);
    if (from_list) {
      for (unsigned int j = tid; j < list_len; j += kRowThreads) {
        const uint2 e = __ldcg(list + j);
        visit(e.x, __uint_as_float(e.y), false);
      }
    } else {
      const bool append = stage == 1;
      row_sweep_t<4, kBf16>(rv, stage == 1 ? pol_last : pol_keep, fix,
                            [&](int i, float x) { visit(static_cast<uint32_t>(i), x, append); });
    }
    f = block_find(t, nb, desc, above, tt_hi, tt_lo, cmin, cmax, true);
    if (stage == 1) list_len = t.list_n;  // complete: block_find synchronised the CTA
    above = f.before;
    const uint32_t bin = static_cast<uint32_t>(f.bin);
    if (stage == 1) {
      a1 = f.bin;
    } else if (stage <= 4) {
      kd_pre = (kd_pre << (stage == 4 ? 10 : 11)) | bin;
      kd_len += stage == 4 ? 10 : 11;
    } else {
      id_pre = (id_pre << 11) | bin;
      id_len += 11;
    }
    // every candidate of this stage had one value (ties, e.g. in a bf16
    // row), so the boundary bin does too: go on with the token-id stages
    if (stage < 5 && f.cnt > 1u && f.kmin == f.kmax) {
      kd_pre = f.kmin;
      kd_len = 32;
      stage = 4;
    }
  }
  // f is the one-element bin at the boundary: its token, mass and logit
  if (tid == 0) {
    const int32_t id_thr = static_cast<int32_t>(f.id);
    const unsigned long long Fk = above + f.mass;
    const uint32_t kd_thr = kd_of(fix(raw_at(id_thr)));
    const float D = __fmul_rn(__ull2float_rn(Fk), 0x1p-40f);
    const bool has_d = d >= 0 && d < V;
    const float x = has_d ? fix(raw_at(d)) : 0.0f;
    const uint32_t kd = kd_of(x);
    const bool keep = kd > kd_thr || (kd == kd_thr && d <= id_thr);
    ts->p_d = has_d && keep ? __fdiv_rn(exp_rel(x, m), D) : 0.0f;
    ts->m = m;
    ts->D = D;
    ts->kd_thr = kd_thr;
    ts->id_thr = id_thr;
    ts->mode = kModeThreshold;
    ts->amax_key = 0ull;
  }
}

// Out of line: the select's registers and code stay out of the kernel's
// common path (slices, draws), which runs at the kernel's register limit.
__device__ __noinline__ void flat_topp_row(const VerifyParams& P, const FlatRow& R, TopSmem& t) {
  const bool scale = R.T != 1.0f;
  if (R.bf16) {
    if (scale) flat_topp_row_t<true, true>(P, R, t);
    else flat_topp_row_t<true, false>(P, R, t);
  } else {
    if (scale) flat_topp_row_t<false, true>(P, R, t);
    else flat_topp_row_t<false, false>(P, R, t);
  }
}


// One slice of a row: this CTA's partial in P.parts.
__device__ void flat_slice(const VerifyParams& P, const FlatRow& R, int s, FlatSmem& sm) {
  const int V = P.V;
  int sw = (V + P.nslice - 1) / P.nslice;
  sw = (sw + 7) & ~7;
  const int v0 = min(V, s * sw), v1 = min(V, v0 + sw);
  RowView rv;
  rv.bf16 = R.bf16;
  rv.f = static_cast<const float*>(R.base) + R.off + v0;
  rv.h = static_cast<const uint16_t*>(R.base) + R.off + v0;
  rv.n = v1 - v0;
  // normal priority: a residual draw soon reads the rows of the request's
  // first rejection again
  const uint64_t pol = policy_evict_normal();
  RowPart part;
  part.m = -INFINITY;
  part.s = 0.0f;
  part.key = 0ull;
  if (R.kind == kFlatGreedy) {
    unsigned long long key = 0ull;
    row_sweep(rv, pol, [](float c) { return c; }, [&](int i, float t) {
      key = umax64(key, winner_key(t, static_cast<uint32_t>(v0 + i)));
    });
    part.key = block_reduce<unsigned long long>(
        key, sm.w_u64, 0ull, [](unsigned long long a, unsigned long long b) { return a > b ? a : b; });
  } else {
    unsigned long long ms;
    if (R.T != 1.0f) {
      const float T = R.T;
      ms = slice_online(rv, pol, [T](float c) { return fmaxf(__fdiv_rn(c, T), -INFINITY); }, false,
                        0.0f, kSliceWindow);
    } else {
      ms = slice_online(rv, pol, [](float c) { return fmaxf(c, -INFINITY); }, false, 0.0f,
                        kSliceWindow);
    }
    ms = block_reduce<unsigned long long>(ms, sm.w_u64, ms_pack(-INFINITY, 0.0f),
                                          [](unsigned long long a, unsigned long long b) {
                                            return ms_combine(a, b);
                                          });
    part.m = ms_m(ms);
    part.s = ms_s(ms);
  }
  if (threadIdx.x == 0) {
    const int row = R.is_target ? R.b * (P.K + 1) + R.k : P.B * (P.K + 1) + R.b * P.K + R.k;
    reinterpret_cast<RowPart*>(P.parts)[static_cast<int64_t>(row) * P.nslice + s] = part;
  }
}

// Warp 0, after every slice of the row is done: the row's statistics from
// its partials (lane i holds slice i; a butterfly of commutative combines,
// the same bits every run).
__device__ void flat_finish_row(const VerifyParams& P, const FlatRow& R) {
  const int K = P.K, V = P.V, lane = threadIdx.x & 31;
  const int row = R.is_target ? R.b * (K + 1) + R.k : P.B * (K + 1) + R.b * K + R.k;
  const RowPart* parts = reinterpret_cast<const RowPart*>(P.parts) + static_cast<int64_t>(row) * P.nslice;
  const int32_t d = R.k < K ? P.draft[static_cast<int64_t>(R.b) * K + R.k] : -1;
  const bool has_d = d >= 0 && d < V;
  if (R.kind == kFlatGreedy) {
    unsigned long long key = lane < P.nslice ? __ldcg(&parts[lane].key) : 0ull;
    key = warp_max64(key);
    if (lane == 0) {
      TgtStats* ts = static_cast<TgtStats*>(P.tstats) + static_cast<int64_t>(R.b) * (K + 1) + R.k;
      ts->m = 0.f;
      ts->D = 1.f;
      ts->kd_thr = 0u;
      ts->id_thr = 0;
      ts->p_d = 0.f;
      ts->mode = kModeGreedy;
      ts->amax_key = key;
    }
    return;
  }
  float m = -INFINITY, s = 0.0f;
  if (R.kind == kFlatRecorded) {
    const dspark_row_stats* st = P.draft_stats + static_cast<int64_t>(R.b) * K + R.k;
    m = __ldcg(&st->m);
    const unsigned long long mass =
        __ldcg(reinterpret_cast<const unsigned long long*>(&st->mass));
    s = __fmul_rn(__ull2float_rn(mass), 0x1p-40f);
  } else {
    unsigned long long ms = lane < P.nslice ? ms_pack(__ldcg(&parts[lane].m), __ldcg(&parts[lane].s))
                                            : ms_pack(-INFINITY, 0.0f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ms = ms_combine(ms, __shfl_xor_sync(0xFFFFFFFFu, ms, o));
    m = ms_m(ms);
    s = ms_s(ms);
  }
  if (lane != 0) return;
  // the value at the drafted token, as the row's distribution reads it
  float x = -INFINITY;
  if (has_d) {
    const int64_t o = R.off + d;
    const float c = R.bf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(R.base)[o])
                           : static_cast<const float*>(R.base)[o];
    x = R.is_target ? scale_logit(c, R.T) : fmaxf(c, -INFINITY);
  }
  if (R.is_target) {
    TgtStats* ts = static_cast<TgtStats*>(P.tstats) + static_cast<int64_t>(R.b) * (K + 1) + R.k;
    ts->kd_thr = 0u;
    ts->id_thr = 0;
    ts->amax_key = 0ull;
    if (m == -INFINITY) {  // no value above -inf: p is one-hot at column 0
      ts->m = m;
      ts->D = 1.0f;
      ts->p_d = d == 0 ? 1.0f : 0.0f;
      ts->mode = kModeOneHot;
    } else {
      ts->m = m;
      ts->D = s;
      ts->p_d = has_d ? __fdiv_rn(exp_rel(x, m), s) : 0.0f;
      ts->mode = kModeKeepAll;
    }
  } else {
    DrfStats* ds = static_cast<DrfStats*>(P.dstats) + static_cast<int64_t>(R.b) * K + R.k;
    if (m == -INFINITY) {  // no value above -inf: q = 0
      ds->m = m;
      ds->D = 1.0f;
      ds->q_d = 0.0f;
      ds->zero = 1;
    } else {
      ds->m = m;
      ds->D = s;
      ds->q_d = has_d ? __fdiv_rn(exp_rel(x, m), s) : 0.0f;
      ds->zero = 0;
    }
  }
}

struct FlatShared {
  FlatSmem f;
  TopSmem t;         // top-p rows
};

// One row item r = (request, row, slice).
__device__ void flat_row_item(const VerifyParams& P, const CtlView& C, FlatSmem& sm, TopSmem& t,
                              int r) {
  const int per_req = 2 * P.K + 1;
  const int s = r % P.nslice;
  const int rr = r / P.nslice;
  const int b = rr / per_req, j = rr % per_req;
  const FlatRow R = classify_row(P, b, j);
  bool row_complete;
  if (R.kind == kFlatGreedy || R.kind == kFlatOnline) {
    flat_slice(P, R, s, sm);
    if (threadIdx.x == 0) {
      __threadfence();  // the partial before the count
      const int row = R.is_target ? b * (P.K + 1) + R.k : P.B * (P.K + 1) + b * P.K + R.k;
      sm.last = atomicAdd(&C.slices_done[row], 1u) + 1u == static_cast<unsigned int>(P.nslice);
      if (sm.last) __threadfence();
    }
    __syncthreads();
    row_complete = sm.last != 0;
    if (row_complete && threadIdx.x < 32) flat_finish_row(P, R);
  } else if (R.kind == kFlatTopp) {
    // the whole row, by the CTA holding its first slice
    row_complete = s == 0;
    if (row_complete) flat_topp_row(P, R, t);
  } else {
    // nothing to read (or the recorded statistics): the first slice does it
    row_complete = s == 0;
    if (row_complete && R.kind == kFlatRecorded && threadIdx.x < 32) flat_finish_row(P, R);
  }
  if (row_complete) request_row_done(P, C, sm, b);
}

// One draw item: chunk `chunk` of request J.b's categorical; the CTA that
// finishes the request's last chunk writes its outputs.
__device__ void flat_draw_chunk(const VerifyParams& P, const CtlView& C, FlatSmem& sm,
                                const DrawJob& J, int chunk) {
  const int tid = threadIdx.x;
  const int b = J.b, nsub = P.ndraw, K = P.K, V = P.V;
  int cw = (V + nsub - 1) / nsub;
  cw = (cw + 3) & ~3;
  const int c0 = chunk * cw, c1 = min(V, c0 + cw);
  auto umax = [](unsigned long long a, unsigned long long b2) { return a > b2 ? a : b2; };
  unsigned long long key = 0ull;
  unsigned int any = 0u;
  if (!J.invalid && J.mode != kDrawNone && c0 < c1)
    key = draw_range(P, J, J.mode, c0, c1, kRowThreads, &any);
  key = block_reduce<unsigned long long>(key, sm.w_u64, 0ull, umax);
  __syncthreads();
  const unsigned int anyb = __syncthreads_or(any != 0u) ? 1u : 0u;
  if (tid == 0) {
    P.keys[static_cast<int64_t>(b) * P.kstride + chunk] = key;
    P.anypos[static_cast<int64_t>(b) * P.kstride + chunk] = anyb;
    __threadfence();
    sm.last = atomicAdd(&C.draws_done[b], 1u) == static_cast<unsigned int>(nsub) - 1u;
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  // ---- the request's last chunk: reduce (warp 0, chunks in parallel) --------
  if (tid < 32) {
    unsigned long long m = 0ull;
    unsigned int a = 0u;
    for (int i = tid; i < nsub; i += 32) {
      m = umax64(m, __ldcg(P.keys + static_cast<int64_t>(b) * P.kstride + i));
      a |= __ldcg(P.anypos + static_cast<int64_t>(b) * P.kstride + i);
    }
    m = warp_max64(m);
    a = __any_sync(0xFFFFFFFFu, a != 0u) ? 1u : 0u;
    if (tid == 0) {
      int tok = -1;
      if (!J.invalid) {
        if (J.mode == kDrawNone)
          tok = J.emit;
        else if (J.mode == kDrawResidual && a == 0u)
          tok = -2;  // r is all zero (fp32 rounding): draw from p
        else
          tok = m ? key_index(m) : 0;
      }
      sm.bcast_i = tok;
    }
  }
  __syncthreads();
  int tok = sm.bcast_i;
  if (tok == -2) {
    unsigned int dummy = 0u;
    unsigned long long k3 = draw_range(P, J, kDrawP, 0, V, kRowThreads, &dummy);
    __syncthreads();
    k3 = block_reduce<unsigned long long>(k3, sm.w_u64, 0ull, umax);
    if (tid == 0) sm.bcast_i = k3 ? key_index(k3) : 0;
    __syncthreads();
    tok = sm.bcast_i;
  }
  for (int k = tid; k <= K; k += kRowThreads) {
    int32_t o = -1;
    if (!J.invalid) {
      if (k < J.n_acc)
        o = P.draft[static_cast<int64_t>(b) * K + k];
      else if (k == J.n_acc)
        o = tok;
    }
    P.out_tokens[static_cast<int64_t>(b) * (K + 1) + k] = o;
  }
  if (tid == 0) P.num_accepted[b] = J.invalid ? 0 : J.n_acc;
}

// Thread 0: the next draw item (sm.chunk = -1 when none is left). Items are
// taken in publish order; item h is chunk h % ndraw of the request listed in
// slot h / ndraw, which may still be finishing its rows (bounded wait).
__device__ void take_draw(const VerifyParams& P, const CtlView& C, FlatSmem& sm) {
  sm.chunk = -1;
  const unsigned int n_draw = static_cast<unsigned int>(P.B) * P.ndraw;
  const unsigned int h = atomicAdd(C.draw_head, 1u);
  if (h >= n_draw) return;
  const unsigned int slot = h / P.ndraw;
  unsigned int b1 = ld_acquire_gpu(&C.ready[slot]);
  if (b1 == 0u) {
    const unsigned long long t0 = globaltimer_ns();
    unsigned int nap = 64u;
    do {
      __nanosleep(nap);
      if (nap < 512u) nap <<= 1;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        report(P.status, DSPARK_ERR_TIMEOUT);
        return;
      }
      b1 = ld_acquire_gpu(&C.ready[slot]);
    } while (b1 == 0u);
  }
  // the publisher's job, 8-byte words loaded independently
  const unsigned long long* src = reinterpret_cast<const unsigned long long*>(&C.jobs[b1 - 1u]);
  unsigned long long* dst = reinterpret_cast<unsigned long long*>(&sm.job);
#pragma unroll
  for (int i = 0; i < static_cast<int>(sizeof(DrawJob) / 8); ++i) dst[i] = __ldcg(src + i);
  sm.chunk = static_cast<int>(h % P.ndraw);
}

// Row statistics of every row, the requests' accept chains, and the draws.
// The rows: each CTA claims the next row item (request order, a row's
// slices in turn) with an atomic counter, the claim of its next item issued
// when it starts the current one, so the claim's latency hides behind the
// item's work; then each CTA takes draw items of the requests published so
// far.
__global__ void __launch_bounds__(kRowThreads, 4) verify_flat_kernel(VerifyParams P) {
  __shared__ FlatShared shared;
  FlatSmem& sm = shared.f;
  const CtlView C(P.ctl, P.B, P.K);
  const unsigned int n_items = static_cast<unsigned int>(P.B) * (2 * P.K + 1) * P.nslice;
  if (threadIdx.x == 0) sm.chunk = static_cast<int>(atomicAdd(C.row_head, 1u));
  __syncthreads();
  for (;;) {
    const unsigned int r = static_cast<unsigned int>(sm.chunk);
    if (r >= n_items) break;
    unsigned int next = 0u;
    if (threadIdx.x == 0) next = atomicAdd(C.row_head, 1u);  // used after this item
    __syncthreads();  // every thread has read r
    flat_row_item(P, C, sm, shared.t, static_cast<int>(r));
    __syncthreads();  // sm is reused by the next item
    if (threadIdx.x == 0) sm.chunk = static_cast<int>(next);
    __syncthreads();
  }
  for (;;) {
    if (threadIdx.x == 0) take_draw(P, C, sm);
    __syncthreads();
    if (sm.chunk < 0) break;
    flat_draw_chunk(P, C, sm, sm.job, sm.chunk);
    __syncthreads();  // sm.job is rewritten by the next take
  }
}

// ---------------------------------------------------------------------------
// Top-k candidates of the base-logit rows for the top-k Markov loop (the
// "DSparkSpeculator" page, _sample_sequential_topk): per (request, draft
// step) the k largest base logits by (value descending, token id
// ascending), NaN above every number, -0 equal to +0. A radix select with a
// unit mass per element over the order key (11 + 11 + 10 bits, its first
// stage counted during the pass that reads the row from HBM) and then the
// token id: the boundary is the k-th element of that order. The cluster also
// fills the step's cache row with -inf (the loop writes the candidates'
// values).

// Exclusive prefix over the cluster's ranks of one per-CTA count, and the
// total (one cluster barrier; every CTA must call it).
__device__ void cluster_prefix(cg::cluster_group& cl, RowSmem& sm, unsigned int v, int CL,
                               int rank, unsigned int* before, unsigned int* total) {
  if (threadIdx.x == 0) sm.x_pref = v;
  cl.sync();
  if (threadIdx.x < 32) {
    const int r = threadIdx.x;
    unsigned int x = r < CL ? *cl.map_shared_rank(&sm.x_pref, r) : 0u;
    unsigned int lower = r < rank ? x : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
      lower += __shfl_xor_sync(0xFFFFFFFFu, lower, o);
    }
    if (threadIdx.x == 0) {
      sm.w_u32[0] = lower;
      sm.w_u32[1] = x;
    }
  }
  __syncthreads();
  *before = sm.w_u32[0];
  *total = sm.w_u32[1];
  cl.sync();  // the slots may be rewritten by the next call
}

// cluster_prefix for three counts at once (one exchange, two cluster barriers).
__device__ void cluster_prefix3(cg::cluster_group& cl, RowSmem& sm, const unsigned int (&v)[3],
                                int CL, int rank, unsigned int (&before)[3],
                                unsigned int (&total)[3]) {
  if (threadIdx.x == 0) {
    sm.x_pref = v[0];
    sm.x_cmin = v[1];
    sm.x_cmax = v[2];
  }
  cl.sync();
  if (threadIdx.x < 32) {
    const int r = threadIdx.x;
    unsigned int x[3] = {0u, 0u, 0u};
    if (r < CL) {
      x[0] = *cl.map_shared_rank(&sm.x_pref, r);
      x[1] = *cl.map_shared_rank(&sm.x_cmin, r);
      x[2] = *cl.map_shared_rank(&sm.x_cmax, r);
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      unsigned int lower = r < rank ? x[j] : 0u;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        x[j] += __shfl_xor_sync(0xFFFFFFFFu, x[j], o);
        lower += __shfl_xor_sync(0xFFFFFFFFu, lower, o);
      }
      if (threadIdx.x == 0) {
        sm.w_u32[2 * j] = lower;
        sm.w_u32[2 * j + 1] = x[j];
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    before[j] = sm.w_u32[2 * j];
    total[j] = sm.w_u32[2 * j + 1];
  }
  cl.sync();  // the slots may be rewritten by the next call
}

// Exclusive prefix of a per-thread count over the block, and the block total.
__device__ unsigned int block_prefix(RowSmem& sm, unsigned int v, unsigned int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  unsigned int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  __syncthreads();
  if (lane == 31) sm.w_u32[w] = incl;
  __syncthreads();
  unsigned int before_w = 0u, tot = 0u;
  for (int i = 0; i < kRowWarps; ++i) {
    const unsigned int x = sm.w_u32[i];
    if (i < w) before_w += x;
    tot += x;
  }
  *total = tot;
  __syncthreads();  // w_u32 may be reused right after
  return before_w + incl - v;
}

__device__ void topk_row(const TopkParams& P, int W, int row_id, cg::cluster_group& cl, int CL,
                         int rank, RowSmem& sm, int& jrow) {
  const int tid = threadIdx.x;
  const int K = P.K, V = P.V;
  const int b = row_id / K, i = row_id % K;
  const int32_t s = P.rsi[b];
  if (s < 0) return;
  if (s >= P.S) {
    if (rank == 0 && tid == 0) report(P.status, DSPARK_ERR_BOUNDS);
    return;
  }
  const int set = jrow & 1;
  ++jrow;
  const int v0 = rank * W;
  const int n = max(0, min(W, V - v0));
  const int64_t off = (static_cast<int64_t>(b) * K + i) * V;
  RowView rv;
  rv.bf16 = P.base_bf16 != 0;
  rv.f = static_cast<const float*>(P.base) + off + v0;
  rv.h = static_cast<const uint16_t*>(P.base) + off + v0;
  rv.n = n;
  const uint64_t pol = policy_evict_last();
  int32_t* cidx = P.cand_idx + static_cast<int64_t>(row_id) * P.k;
  float* cval = P.cand_val + static_cast<int64_t>(row_id) * P.k;
  auto ident = [](float c) { return c; };

  // the cache row starts as -inf: the loop stores only the candidates
  if (P.cache != nullptr) {
    const int64_t row = P.row_map ? P.row_map[s] : s;
    if (row >= 0 && row < P.C) {
      const int64_t co = (row * K + i) * V + v0;
      if (P.cache_bf16) {
        uint16_t* c = static_cast<uint16_t*>(P.cache) + co;
        for (int j = tid; j < n; j += kRowThreads) c[j] = 0xFF80u;  // bf16 -inf
      } else {
        float* c = static_cast<float*>(P.cache) + co;
        for (int j = tid; j < n; j += kRowThreads) c[j] = -INFINITY;
      }
    }
  }
  const int k_eff = P.k < V ? P.k : V;
  if (k_eff == V) {  // every column is a candidate
    row_sweep(rv, pol, ident, [&](int j, float x) {
      cidx[v0 + j] = v0 + j;
      cval[v0 + j] = x;
    });
    return;
  }

  // ---- pass 1 (HBM): the NaN count and a count histogram of the numbers by
  // the top 11 bits of their order key (sign, exponent, two mantissa bits),
  // one shared atomic per element: the first radix stage needs no maximum
  hist_clear(sm, kRowBins);
  __syncthreads();
  unsigned long long nan_loc = 0ull;
  row_sweep(rv, pol, ident, [&](int, float x) {
    if (x != x)
      nan_loc += 1ull;
    else
      atomicAdd(&sm.hcnt[kd_of(x) >> 21], 1u);
  });
  const unsigned long long nan_tot = cluster_sum_u64(cl, sm, nan_loc, set, CL);

  if (nan_tot >= static_cast<unsigned long long>(k_eff)) {
    // the candidates are the first k NaN columns: warp 0 walks the slice in
    // order and takes this CTA's share of them
    unsigned int before, total;
    const unsigned int mine = static_cast<unsigned int>(block_sum_u64(nan_loc, sm));
    cluster_prefix(cl, sm, mine, CL, rank, &before, &total);
    if (tid < 32 && before < static_cast<unsigned int>(k_eff)) {
      unsigned int pos = before;
      for (int c0 = 0; c0 < n && pos < static_cast<unsigned int>(k_eff); c0 += 32) {
        const int j = c0 + tid;
        float x = 0.0f;
        if (j < n) x = rv.bf16 ? bf16_bits_to_float(rv.h[j]) : rv.f[j];
        const bool isn = j < n && x != x;
        const unsigned int bal = __ballot_sync(0xFFFFFFFFu, isn);
        const unsigned int at = pos + __popc(bal & ((1u << tid) - 1u));
        if (isn && at < static_cast<unsigned int>(k_eff)) {
          cidx[at] = v0 + j;
          cval[at] = x;
        }
        pos += __popc(bal);
      }
    }
    return;
  }

  // ---- the top (k - NaNs) numbers: radix select with unit masses -------------
  const unsigned long long need = static_cast<unsigned long long>(k_eff) - nan_tot;
  // reach: count * 2^32 >= need * 2^32, as the 128-bit target (t_hi:t_lo)
  const unsigned long long t_hi = 0ull, t_lo = need << 32;
  // the first stage's histogram is pass 1's (counts only: the mass of a bin
  // is its count, and the bin's token id is found by a later stage)
  __syncthreads();
  for (int q = tid; q < kRowBins; q += kRowThreads) sm.hmass[q] = sm.hcnt[q];
  Found f = cluster_find(cl, sm, kRowBins, true, 0ull, t_hi, t_lo, CL, rank);
  // ---- one sweep: the values above the boundary bin (and the NaNs) are
  // candidates whatever the rest, the boundary bin's values are listed by
  // their order keys; the cluster's rank 0 sorts those keys (x descending,
  // id ascending) and takes the top ones. Lists longer than the shared
  // memory holds take the radix stages below instead.
  {
    constexpr unsigned int kCap = kRowBins;  // entries per list (16 KB each)
    const uint32_t b_star = static_cast<uint32_t>(f.bin);
    const unsigned int need_b = static_cast<unsigned int>(need - f.before);
    int2* alist = reinterpret_cast<int2*>(sm.hmass);                  // (id, value bits)
    unsigned long long* blist = reinterpret_cast<unsigned long long*>(sm.hcnt);  // order keys
    static_assert(sizeof(unsigned int) * 2 * kRowBins >= sizeof(unsigned long long) * kRowBins,
                  "the boundary list lives in hcnt and hid");
    __syncthreads();  // the histograms are read
    if (tid == 0) {
      sm.x_pref = 0u;
      sm.list_n = 0u;
    }
    __syncthreads();
    row_sweep<4>(rv, pol, ident, [&](int j, float x) {
      const uint32_t id = static_cast<uint32_t>(v0 + j);
      const uint32_t kd = kd_of(x);
      const uint32_t dg = kd >> 21;
      if (x != x || dg > b_star) {
        const unsigned int at = atomicAdd(&sm.x_pref, 1u);
        if (at < kCap) alist[at] = make_int2(static_cast<int>(id), __float_as_int(x));
      } else if (dg == b_star) {
        const unsigned int at = atomicAdd(&sm.list_n, 1u);
        if (at < kCap)
          blist[at] = (static_cast<unsigned long long>(kd) << 32) |
                      static_cast<unsigned long long>(0xFFFFFFFFu - id);
      }
    });
    __syncthreads();
    const unsigned int na = sm.x_pref, nbl = sm.list_n;
    const unsigned int counts[3] = {na, nbl, (na > kCap || nbl > kCap) ? 1u : 0u};
    unsigned int cb[3], ct[3];
    cluster_prefix3(cl, sm, counts, CL, rank, cb, ct);
    const unsigned int a_before = cb[0], a_total = ct[0], b_total = ct[1], ovf_total = ct[2];
    if (ovf_total == 0u && b_total <= kCap && b_total >= need_b) {
      for (unsigned int q = tid; q < na; q += kRowThreads) {
        const unsigned int at = a_before + q;
        if (at < static_cast<unsigned int>(k_eff)) {
          cidx[at] = alist[q].x;
          cval[at] = __int_as_float(alist[q].y);
        }
      }
      if (rank == 0) {  // the other ranks' boundary lists after this CTA's own
        unsigned int at = nbl;
        for (int r = 1; r < CL; ++r) {
          const unsigned int nr = *cl.map_shared_rank(&sm.list_n, r);
          const unsigned long long* src = cl.map_shared_rank(blist, r);
          for (unsigned int q = tid; q < nr; q += kRowThreads) blist[at + q] = src[q];
          at += nr;
        }
      }
      cl.sync();  // rank 0 has read the other ranks' lists
      if (rank == 0) {
        // the top need_b keys of the boundary bin: a count histogram of the
        // next 11 key bits over the list finds the sub-bin where they end;
        // every key above it is taken, the sub-bin's keys are sorted
        unsigned int* cnt = reinterpret_cast<unsigned int*>(sm.hmass);  // 2048 words
        for (int q = tid; q < kRowBins; q += kRowThreads) cnt[q] = 0u;
        if (tid == 0) {
          sm.x_pref = 0u;     // keys taken so far
          sm.found_pos = -1;  // the boundary sub-bin
        }
        __syncthreads();
        auto sub = [](unsigned long long key) {
          return static_cast<int>((static_cast<uint32_t>(key >> 32) >> 10) & 0x7FFu);
        };
        for (unsigned int q = tid; q < b_total; q += kRowThreads) atomicAdd(&cnt[sub(blist[q])], 1u);
        __syncthreads();
        // thread t holds sub-bins 2047 - 8t .. 2040 - 8t (descending); an
        // exclusive prefix over the block gives the count above each run
        constexpr int per = kRowBins / kRowThreads;
        unsigned int run[per], tsum = 0u;
#pragma unroll
        for (int i = 0; i < per; ++i) {
          run[i] = cnt[kRowBins - 1 - (tid * per + i)];
          tsum += run[i];
        }
        unsigned int all_keys;
        const unsigned int before = block_prefix(sm, tsum, &all_keys);
        unsigned int acc = before;
#pragma unroll
        for (int i = 0; i < per; ++i) {
          if (acc < need_b && acc + run[i] >= need_b) {
            sm.found_pos = kRowBins - 1 - (tid * per + i);
            sm.found_before = acc;
          }
          acc += run[i];
        }
        __syncthreads();
        const int sb = sm.found_pos;
        const unsigned int taken_above = static_cast<unsigned int>(sm.found_before);
        const unsigned int rest = need_b - taken_above;  // from sub-bin sb
        // keys above the sub-bin: all taken (order inside does not matter)
        for (unsigned int q = tid; q < b_total; q += kRowThreads) {
          const unsigned long long key = blist[q];
          if (sub(key) > sb) {
            const unsigned int at = a_total + atomicAdd(&sm.x_pref, 1u);
            const int32_t id = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
            if (at < static_cast<unsigned int>(k_eff)) {
              cidx[at] = id;
              cval[at] = rv.bf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(P.base)[off + id])
                                 : static_cast<const float*>(P.base)[off + id];
            }
          }
        }
        __syncthreads();
        // the sub-bin's keys, moved to the front of the list (cnt[sb] of them)
        // and sorted descending; the first `rest` are taken
        const unsigned int nsb = cnt[sb];
        unsigned long long* keys2 = reinterpret_cast<unsigned long long*>(sm.hmass);
        __syncthreads();  // cnt is read
        if (tid == 0) sm.list_n = 0u;
        __syncthreads();
        for (unsigned int q = tid; q < b_total; q += kRowThreads) {
          const unsigned long long key = blist[q];
          if (sub(key) == sb) keys2[atomicAdd(&sm.list_n, 1u)] = key;
        }
        unsigned int np = 1u;
        while (np < nsb) np <<= 1;
        __syncthreads();
        for (unsigned int q = nsb + tid; q < np; q += kRowThreads) keys2[q] = 0ull;  // last
        __syncthreads();
        for (unsigned int ks = 2; ks <= np; ks <<= 1) {
          for (unsigned int jj = ks >> 1; jj > 0; jj >>= 1) {
            for (unsigned int q = tid; q < np; q += kRowThreads) {
              const unsigned int r2 = q ^ jj;
              if (r2 > q) {
                const unsigned long long x0 = keys2[q], x1 = keys2[r2];
                if (((q & ks) == 0u) ? (x0 < x1) : (x0 > x1)) {
                  keys2[q] = x1;
                  keys2[r2] = x0;
                }
              }
            }
            __syncthreads();
          }
        }
        for (unsigned int q = tid; q < rest; q += kRowThreads) {
          const unsigned int at = a_total + taken_above + q;
          if (at < static_cast<unsigned int>(k_eff)) {
            const int32_t id = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(keys2[q]));
            cidx[at] = id;
            cval[at] = rv.bf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(P.base)[off + id])
                               : static_cast<const float*>(P.base)[off + id];
          }
        }
      }
      return;
    }
    // the histograms were overwritten: count pass 1's bins again for the stages
    hist_clear(sm, kRowBins);
    __syncthreads();
    row_sweep(rv, pol, ident, [&](int, float x) {
      if (x == x) atomicAdd(&sm.hcnt[kd_of(x) >> 21], 1u);
    });
    __syncthreads();
    for (int q = tid; q < kRowBins; q += kRowThreads) sm.hmass[q] = sm.hcnt[q];
    f = cluster_find(cl, sm, kRowBins, true, 0ull, t_hi, t_lo, CL, rank);
  }
  unsigned long long above = f.before;
  int kd_len = 11, id_len = 0;
  uint32_t kd_pre = static_cast<uint32_t>(f.bin), id_pre = 0u;
  // then kd bits [20:10] and [9:0], token id bits [21:11] and [10:0], while
  // the boundary bin holds more than one element (at least once, for its id)
  for (int stage = 3; (stage == 3 || f.cnt != 1u) && stage <= 6; ++stage) {
    const int c_kl = kd_len, c_il = id_len;
    const uint32_t c_kp = kd_pre, c_ip = id_pre;
    auto match = [=](float x, uint32_t kd, uint32_t id) {
      if (x != x || (kd >> (32 - c_kl)) != c_kp) return false;
      if (c_il > 0 && (id >> (22 - c_il)) != c_ip) return false;
      return true;
    };
    auto digit = [=](uint32_t kd, uint32_t id) -> int {
      switch (stage) {
        case 3: return static_cast<int>((kd >> 10) & 0x7FFu);
        case 4: return static_cast<int>(kd & 0x3FFu);
        case 5: return static_cast<int>((id >> 11) & 0x7FFu);
        default: return static_cast<int>(id & 0x7FFu);
      }
    };
    const int nb = stage == 4 ? 1024 : kRowBins;
    const bool desc = stage <= 4;  // larger kd first; token ids ascending
    hist_clear(sm, nb);
    __syncthreads();
    row_sweep<4>(rv, pol, ident, [&](int j, float x) {
      const uint32_t kd = kd_of(x);
      const uint32_t id = static_cast<uint32_t>(v0 + j);
      if (match(x, kd, id)) hist_add(sm, true, digit(kd, id), 1ull, id);
    });
    f = cluster_find(cl, sm, nb, desc, above, t_hi, t_lo, CL, rank);
    above = f.before;
    const uint32_t bin = static_cast<uint32_t>(f.bin);
    if (stage <= 4) {
      kd_pre = (kd_pre << (stage == 4 ? 10 : 11)) | bin;
      kd_len += stage == 4 ? 10 : 11;
    } else {
      id_pre = (id_pre << 11) | bin;
      id_len += 11;
    }
  }
  const int32_t id_thr = static_cast<int32_t>(f.id);
  const float xb = rv.bf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(P.base)[off + id_thr])
                           : static_cast<const float*>(P.base)[off + id_thr];
  const uint32_t kd_thr = kd_of(xb);
  auto is_cand = [=](float x, int id) {
    if (x != x) return true;
    const uint32_t kd = kd_of(x);
    return kd > kd_thr || (kd == kd_thr && id <= id_thr);
  };
  // ---- compaction: this CTA's candidates after the lower ranks' -------------
  if (k_eff <= kRowBins) {
    // one sweep: append to a shared list (the order inside a CTA does not
    // matter to the loop), then copy it after the lower ranks' lists
    int2* list = reinterpret_cast<int2*>(sm.hmass);  // kRowBins (id, value bits) pairs
    if (tid == 0) sm.x_pref = 0u;
    __syncthreads();
    row_sweep<4>(rv, pol, ident, [&](int j, float x) {
      if (is_cand(x, v0 + j)) {
        const unsigned int at = atomicAdd(&sm.x_pref, 1u);
        if (at < static_cast<unsigned int>(kRowBins)) list[at] = make_int2(v0 + j, __float_as_int(x));
      }
    });
    __syncthreads();
    const unsigned int mine = sm.x_pref;
    unsigned int before, total;
    cluster_prefix(cl, sm, mine, CL, rank, &before, &total);
    for (unsigned int q = tid; q < mine; q += kRowThreads) {
      const unsigned int at = before + q;
      if (at < static_cast<unsigned int>(k_eff)) {
        cidx[at] = list[q].x;
        cval[at] = __int_as_float(list[q].y);
      }
    }
    return;
  }
  unsigned int cnt = 0u;
  row_sweep<4>(rv, pol, ident, [&](int j, float x) { cnt += is_cand(x, v0 + j) ? 1u : 0u; });
  unsigned int blk_total;
  const unsigned int tpos = block_prefix(sm, cnt, &blk_total);
  unsigned int before, total;
  cluster_prefix(cl, sm, blk_total, CL, rank, &before, &total);
  unsigned int at = before + tpos;
  row_sweep<4>(rv, pol, ident, [&](int j, float x) {
    if (is_cand(x, v0 + j) && at < static_cast<unsigned int>(k_eff)) {
      cidx[at] = v0 + j;
      cval[at] = x;
      ++at;
    }
  });
}

__global__ void __launch_bounds__(kRowThreads, 4) topk_rows_kernel(TopkParams P, int W, int nrows) {
  cg::cluster_group cl = cg::this_cluster();
  const int CL = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int cid = blockIdx.x / CL;
  const int nclusters = gridDim.x / CL;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  RowSmem& sm = *reinterpret_cast<RowSmem*>(smem_raw);
  int jrow = 0;
  for (int row = cid; row < nrows; row += nclusters) topk_row(P, W, row, cl, CL, rank, sm, jrow);
  cl.sync();  // no CTA exits while another may still read its shared memory
}

}  // namespace

size_t verify_rows_smem_bytes(int W) {
  (void)W;
  return (sizeof(RowSmem) + 15) & ~size_t(15);
}

// Cluster size and slice width for vocabulary V and element size es (the
// larger of the target and cache dtypes): the smallest cluster whose slices
// are at most 128 KB (32768 fp32 or 65536 bf16 values per CTA).
bool verify_rows_plan(int V, int es, int* CL, int* W) {
  const int candidates[] = {1, 2, 4, 8, 16};
  const int max_w = (128 * 1024) / (es > 0 ? es : 4);
  for (int cl : candidates) {
    int w = (V + cl - 1) / cl;
    w = (w + 7) & ~7;
    if (w <= max_w || cl == 16) {
      *CL = cl;
      *W = w;
      return true;
    }
  }
  return false;
}

size_t verify_ctl_bytes(int B, int K) {
  return CtlView::jobs_word(B, K) * sizeof(unsigned int) + static_cast<size_t>(B) * sizeof(DrawJob);
}

// Enough slices that about 1024 row items fill the GPU's CTAs, none shorter
// than 2048 values, at most 32.
int verify_nslice(int B, int K, int V) {
  const int rows = B * (2 * K + 1);
  if (rows <= 0) return 1;
  int n = (1024 + rows - 1) / rows;
  const int by_len = V / 2048;
  if (n > by_len) n = by_len;
  if (n > 32) n = 32;
  return n < 1 ? 1 : n;
}

size_t verify_parts_bytes(int B, int K, int V) {
  return static_cast<size_t>(B) * (2 * K + 1) * verify_nslice(B, K, V) * sizeof(RowPart);
}

cudaError_t launch_verify(const VerifyParams& p0, cudaStream_t stream) {
  if (p0.B == 0) return cudaSuccess;
  VerifyParams p = p0;
  // ---- every row, the chains, the draws: persistent CTAs ----------------------
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_flat_kernel, kRowThreads, 0) !=
          cudaSuccess ||
      per_sm < 1) {
    (void)cudaGetLastError();
    sms = 1;
    per_sm = 1;
  }
  const int ctas = sms * per_sm;
  // draw chunks per request: about four waves of CTAs over the batch (the
  // last requests' draws then spread over many CTAs), none shorter than 1024
  // columns
  int nd = (4 * ctas + p.B - 1) / p.B;
  if (nd > p.kstride) nd = p.kstride;
  if (nd < 1) nd = 1;
  p.ndraw = nd;
  // cooperative: every CTA is resident at once, which a CTA waiting for a
  // request that other CTAs are still finishing relies on
  cudaLaunchConfig_t fc = {};
  fc.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  fc.blockDim = dim3(kRowThreads, 1, 1);
  fc.dynamicSmemBytes = 0;
  fc.stream = stream;
  cudaLaunchAttribute fa[1];
  fa[0].id = cudaLaunchAttributeCooperative;
  fa[0].val.cooperative = 1;
  fc.attrs = fa;
  fc.numAttrs = 1;
  return cudaLaunchKernelEx(&fc, verify_flat_kernel, p);
}

cudaError_t launch_topk_rows(const TopkParams& p, int CL, int W, cudaStream_t stream) {
  const int rows = p.B * p.K;
  if (rows == 0) return cudaSuccess;
  const size_t smem = verify_rows_smem_bytes(W);
  cudaError_t err = cudaFuncSetAttribute(topk_rows_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  if (CL > 8) {
    err = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                               1);
    if (err != cudaSuccess) return err;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kRowThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(CL);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(rows * CL), 1, 1);
  int max_clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&max_clusters, topk_rows_kernel, &cfg) != cudaSuccess ||
      max_clusters < 1) {
    (void)cudaGetLastError();
    max_clusters = 1;
  }
  const size_t row_bytes = static_cast<size_t>(p.V) * (p.base_bf16 ? 2 : 4);
  const int l2_rows = static_cast<int>((80ull << 20) / (row_bytes > 0 ? row_bytes : 1));
  int nclusters = rows < max_clusters ? rows : max_clusters;
  if (l2_rows >= 1 && nclusters > l2_rows) nclusters = l2_rows;
  if (nclusters < 1) nclusters = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters * CL), 1, 1);
  return cudaLaunchKernelEx(&cfg, topk_rows_kernel, p, W, rows);
}

}  // namespace dspark
