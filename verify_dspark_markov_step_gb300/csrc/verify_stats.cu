// verify_stats.cu -- per-row statistics of the verifier, one thread-block
// cluster per row.
//
// vLLM PR #65007 Part 2 ("Temperature and top-p"): the target row after
// temperature, its maximum and total exp-mass in 64-bit fixed point, and the
// exact top-p keep set -- the smallest prefix by (logit desc, token id asc)
// whose mass reaches p, plus the row max. Draft rows (the cache) get their
// maximum and fixed-point mass. Greedy target rows get their winner key.
//
// A row is split over the CL CTAs of a cluster (CL up to 16, slices of at
// most 32768 values). Each CTA starts its slice as one bulk L2 prefetch,
// reads it once for the maximum with an L2 evict-last hint, and the later
// passes (fixed-point mass, the radix stages of the top-p select) read it
// again from L2; with nothing held in shared memory but histograms, four CTAs
// share an SM and many rows are in flight (odd clusters take their rows in
// reverse order, so one-pass draft rows and two-pass target rows overlap).
// Reductions across the cluster go through distributed shared memory:
// scalars by each CTA reading the others' slots, histograms by each CTA
// reducing its own range of bins over the cluster, in place.
//
// Top-p select: a radix select in (logit descending, token id ascending)
// order with histograms of fixed-point mass; each stage finds the first bin at
// which the running mass reaches P32 * F / 2^32 and the next stage splits
// that bin, until the bin holds one element. The first two stages bin by the
// distance to the row maximum (2048 bins of 1/64 over [0, 32), counted during
// the mass pass, then 2048 sub-bins of the chosen bin, whose elements are
// also copied to a per-CTA candidate list that the later stages read instead
// of the slice); then come the ordered bits kd of the logit (11 + 11 + 10
// bits, skipped once a stage's candidates all share one value) and, for
// exact ties, the token id (11 + 11 bits).
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "verify_common.cuh"

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
  float x_max;
  int x_fail;
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
  unsigned int c_max[2];         // ordered bits of the CTA maximum (~0: failed)
  unsigned long long c_sum[2];   // fixed-point mass
  unsigned long long c_key[2];   // greedy winner key
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
__device__ __forceinline__ float from_ordered(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

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

// Maximum over the cluster; *any_fail = some CTA passed fail = true.
__device__ float cluster_max_f(cg::cluster_group& cl, RowSmem& sm, float v, bool fail, int set,
                               int CL, bool* any_fail) {
  const unsigned int mine = fail ? 0xFFFFFFFFu : ordered_bits(v);
  const unsigned int o = cluster_reduce<unsigned int>(
      cl, sm, mine, &sm.c_max[set], reinterpret_cast<unsigned int*>(&sm.bcast_i), CL, 0u,
      [](unsigned int a, unsigned int b) { return a > b ? a : b; });
  *any_fail = o == 0xFFFFFFFFu;  // a real maximum is never NaN here (NaN reads as -inf)
  return from_ordered(o);
}

__device__ unsigned long long cluster_sum_u64(cg::cluster_group& cl, RowSmem& sm,
                                              unsigned long long v, int set, int CL) {
  return cluster_reduce<unsigned long long>(
      cl, sm, v, &sm.c_sum[set], &sm.bcast_u, CL, 0ull,
      [](unsigned long long a, unsigned long long b) { return a + b; });
}

__device__ unsigned long long cluster_max_u64(cg::cluster_group& cl, RowSmem& sm,
                                              unsigned long long v, int set, int CL) {
  return cluster_reduce<unsigned long long>(
      cl, sm, v, &sm.c_key[set], &sm.bcast_u, CL, 0ull,
      [](unsigned long long a, unsigned long long b) { return a > b ? a : b; });
}

// ---- histograms -------------------------------------------------------------
__device__ void hist_clear(RowSmem& sm, int nb) {
  for (int i = threadIdx.x; i < nb; i += kRowThreads) {
    sm.hmass[i] = 0ull;
    sm.hcnt[i] = 0u;
    sm.hid[i] = 0u;
  }
}

// Adds mass f alone to bin `bin` (the first top-p stage, over every element
// of the row: its counts are not needed).
__device__ __forceinline__ void hist_add_mass(RowSmem& sm, int bin, unsigned long long f) {
  atomicAdd(&sm.hmass[bin], f);
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

// Reads of one row's slice [v0, v0 + n) straight from global memory. The
// first pass brings the slice from HBM (L2 evict-last: every later pass of
// the row reads it again from L2); `fix` maps a raw value to x (temperature,
// NaN read as -inf). `vec` = the slice start is 16-byte aligned (fp32) or
// 8-byte aligned (bf16), so it can be read 4 values at a time.
struct RowView {
  const float* f;
  const uint16_t* h;
  bool bf16;
  bool vec;
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

template <int kU, bool kBf16, class Fix, class Body>
__device__ __forceinline__ void row_sweep_t(RowView rv, uint64_t pol, Fix fix, Body body) {
  rv.bf16 = kBf16;  // a compile-time constant from here on
  const int tid = threadIdx.x;
  int done = 0;
  if (rv.vec) {
    const int n4 = rv.n >> 2;
    int i = tid;
    for (; i + (kU - 1) * kRowThreads < n4; i += kU * kRowThreads) {
      float v[kU][4];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = i + u * kRowThreads;
        if (rv.bf16) {
          const uint2 w = ld_hint_u2(rv.h + 4 * j, pol);
          v[u][0] = bf16_bits_to_float(static_cast<uint16_t>(w.x & 0xFFFFu));
          v[u][1] = bf16_bits_to_float(static_cast<uint16_t>(w.x >> 16));
          v[u][2] = bf16_bits_to_float(static_cast<uint16_t>(w.y & 0xFFFFu));
          v[u][3] = bf16_bits_to_float(static_cast<uint16_t>(w.y >> 16));
        } else {
          const float4 c = ld_hint_f4(rv.f + 4 * j, pol);
          v[u][0] = c.x;
          v[u][1] = c.y;
          v[u][2] = c.z;
          v[u][3] = c.w;
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = 4 * (i + u * kRowThreads);
#pragma unroll
        for (int e = 0; e < 4; ++e) body(j + e, fix(v[u][e]));
      }
    }
    for (; i < n4; i += kRowThreads) {
      float v[4];
      if (rv.bf16) {
        const uint2 w = ld_hint_u2(rv.h + 4 * i, pol);
        v[0] = bf16_bits_to_float(static_cast<uint16_t>(w.x & 0xFFFFu));
        v[1] = bf16_bits_to_float(static_cast<uint16_t>(w.x >> 16));
        v[2] = bf16_bits_to_float(static_cast<uint16_t>(w.y & 0xFFFFu));
        v[3] = bf16_bits_to_float(static_cast<uint16_t>(w.y >> 16));
      } else {
        const float4 c = ld_hint_f4(rv.f + 4 * i, pol);
        v[0] = c.x;
        v[1] = c.y;
        v[2] = c.z;
        v[3] = c.w;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) body(4 * i + e, fix(v[e]));
    }
    done = 4 * n4;
  }
  for (int i = done + tid; i < rv.n; i += kRowThreads) {
    const float c =
        rv.bf16 ? bf16_bits_to_float(ld_hint_u16(rv.h + i, pol)) : ld_hint_f32(rv.f + i, pol);
    body(i, fix(c));
  }
}

// As row_sweep, with the values of each aligned group of four handed to
// quad(x[4]) together (for packed pair arithmetic) and the rest to single(x).
template <int kU, bool kBf16, class Fix, class Quad, class Single>
__device__ __forceinline__ void row_sweep_quads_t(RowView rv, uint64_t pol, Fix fix, Quad quad,
                                                  Single single) {
  const int tid = threadIdx.x;
  auto load4 = [&](int j, float (&v)[4]) {
    if constexpr (kBf16) {
      const uint2 w = ld_hint_u2(rv.h + 4 * j, pol);
      v[0] = bf16_bits_to_float(static_cast<uint16_t>(w.x & 0xFFFFu));
      v[1] = bf16_bits_to_float(static_cast<uint16_t>(w.x >> 16));
      v[2] = bf16_bits_to_float(static_cast<uint16_t>(w.y & 0xFFFFu));
      v[3] = bf16_bits_to_float(static_cast<uint16_t>(w.y >> 16));
    } else {
      const float4 c = ld_hint_f4(rv.f + 4 * j, pol);
      v[0] = c.x;
      v[1] = c.y;
      v[2] = c.z;
      v[3] = c.w;
    }
  };
  int done = 0;
  if (rv.vec) {
    const int n4 = rv.n >> 2;
    int i = tid;
    for (; i + (kU - 1) * kRowThreads < n4; i += kU * kRowThreads) {
      float v[kU][4];
#pragma unroll
      for (int u = 0; u < kU; ++u) load4(i + u * kRowThreads, v[u]);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[u][e] = fix(v[u][e]);
        quad(v[u]);
      }
    }
    for (; i < n4; i += kRowThreads) {
      float v[4];
      load4(i, v);
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = fix(v[e]);
      quad(v);
    }
    done = 4 * n4;
  }
  for (int i = done + tid; i < rv.n; i += kRowThreads) {
    const float c = kBf16 ? bf16_bits_to_float(ld_hint_u16(rv.h + i, pol))
                          : ld_hint_f32(rv.f + i, pol);
    single(fix(c));
  }
}

// Fixed-point mass of the slice relative to m: exp(x - m) per value, four at
// a time in packed pairs.
template <class Fix>
__device__ __forceinline__ unsigned long long slice_mass(const RowView& rv, uint64_t pol, Fix fix,
                                                         float m) {
  MassAcc acc;
  const unsigned long long mm = f2_pack(m, m);
  const unsigned long long l2e = f2_pack(kLog2e, kLog2e);
  auto quad = [&](const float (&x)[4]) {
    float a, b, c, d;
    f2_unpack(f2_mul(f2_sub(f2_pack(x[0], x[1]), mm), l2e), a, b);
    f2_unpack(f2_mul(f2_sub(f2_pack(x[2], x[3]), mm), l2e), c, d);
    acc.add2(f2_pack(ex2_approx(a), ex2_approx(b)));
    acc.add2(f2_pack(ex2_approx(c), ex2_approx(d)));
  };
  auto single = [&](float x) { acc.add(exp_rel(x, m)); };
  if (rv.bf16)
    row_sweep_quads_t<8, true>(rv, pol, fix, quad, single);
  else
    row_sweep_quads_t<8, false>(rv, pol, fix, quad, single);
  return acc.total();
}

// One row: statistics written to P.tstats / P.dstats. Every CTA of the
// cluster runs the same sequence of cluster barriers (all decisions depend on
// the row or on cluster-reduced values only).
__device__ void process_row(const VerifyParams& P, int W, int row_id, cg::cluster_group& cl,
                            int CL, int rank, RowSmem& sm, int& jrow) {
  const int tid = threadIdx.x;
  const int K = P.K, V = P.V;
  const int nT = P.B * (K + 1);
  int b, k;
  bool is_target;
  if (row_id < nT) {
    b = row_id / (K + 1);
    k = row_id % (K + 1);
    is_target = true;
  } else {
    const int r = row_id - nT;
    b = r / K;
    k = r % K;
    is_target = false;
  }
  const int32_t s = P.rsi[b];
  if (s < 0 || s >= P.S) return;
  const float T = P.temperature[s];
  const bool greedy = !(T > 0.0f);
  int64_t crow = 0;
  if (!is_target) {
    if (greedy || P.cache == nullptr) return;
    crow = P.row_map ? P.row_map[s] : s;
    if (crow < 0 || crow >= P.C) return;
  }
  const int set = jrow & 1;
  ++jrow;
  const int v0 = rank * W;
  const int n = max(0, min(W, V - v0));
  int64_t off;
  bool bf16;
  if (is_target) {
    off = (static_cast<int64_t>(b) * (K + 1) + k) * V;
    bf16 = P.target_bf16 != 0;
  } else {
    off = (crow * K + k) * V;
    bf16 = P.cache_bf16 != 0;
  }
  const void* base = is_target ? P.target : P.cache;
  RowView rv;
  rv.bf16 = bf16;
  rv.f = static_cast<const float*>(base) + off + v0;
  rv.h = static_cast<const uint16_t*>(base) + off + v0;
  rv.vec = bf16 ? (reinterpret_cast<uintptr_t>(rv.h) & 7u) == 0
                : (reinterpret_cast<uintptr_t>(rv.f) & 15u) == 0;
  rv.n = n;
  // the slice's first read comes from HBM: start it as one bulk L2 prefetch,
  // so that the whole slice is in flight at once
  if (tid == 0) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(bf16 ? static_cast<const void*>(rv.h)
                                                         : static_cast<const void*>(rv.f));
    const uintptr_t a16 = (a + 15) & ~static_cast<uintptr_t>(15);
    const uint32_t bytes = static_cast<uint32_t>(n) * (bf16 ? 2u : 4u);
    const uint32_t skip = static_cast<uint32_t>(a16 - a);
    if (bytes > skip + 16) {
      const uint32_t len = (bytes - skip) & ~15u;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a16), "r"(len) : "memory");
    }
  }
  const int32_t d = k < K ? P.draft[static_cast<int64_t>(b) * K + k] : -1;
  TgtStats* ts = static_cast<TgtStats*>(P.tstats) + static_cast<int64_t>(b) * (K + 1) + k;
  DrfStats* ds = static_cast<DrfStats*>(P.dstats) + static_cast<int64_t>(b) * K + (k < K ? k : 0);
  const uint64_t pol_keep = policy_evict_last();
  const uint64_t pol_last_use = policy_evict_first();
  // one element of the row by token id (any CTA may read any element)
  auto raw_at = [&](int v) -> float {
    const int64_t o = off + v;
    return bf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(base)[o])
                : static_cast<const float*>(base)[o];
  };

  // ---- greedy target row: winner key of the raw row ----------------------------
  if (is_target && greedy) {
    unsigned long long key = 0ull;
    row_sweep(rv, pol_last_use, [](float c) { return c; }, [&](int i, float t) {
      key = umax64(key, winner_key(t, static_cast<uint32_t>(v0 + i)));
    });
    key = cluster_max_u64(cl, sm, key, set, CL);
    if (rank == 0 && tid == 0) {
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

  // x: the target row after temperature, the draft row as stored; NaN reads
  // as -inf. The passes are instantiated for scaled and unscaled rows, so an
  // unscaled row never evaluates a division.
  const bool topp = is_target && P.top_p[s] < 1.0f;
  auto passes = [&](auto prescale) {
    auto fix = [=](float c) -> float {
      return fmaxf(prescale(c), -INFINITY);  // fmaxf returns the other operand for NaN
    };

    // ---- pass 1 (HBM): maximum (fmaxf skips NaN, as if it were -inf) ---------------
    // A draft row whose maximum the Markov loop recorded skips this pass and
    // is read once, by pass 2 (every CTA of the cluster decides alike).
    const float m_rec = (!is_target && P.draft_stats != nullptr)
                            ? P.draft_stats[static_cast<int64_t>(b) * K + k].m
                            : __int_as_float(0x7FC00000);
    float m;
    if (m_rec == m_rec) {  // recorded (NaN: not recorded)
      m = m_rec;
    } else {
      float lmax = -INFINITY;
      row_sweep(rv, pol_keep, prescale, [&](int, float x) { lmax = fmaxf(lmax, x); });
      bool any_fail = false;
      m = cluster_max_f(cl, sm, lmax, false, set, CL, &any_fail);
    }
    if (m == -INFINITY) {
      if (rank == 0 && tid == 0) {
        if (is_target) {
          ts->m = m;
          ts->D = 1.0f;
          ts->kd_thr = 0u;
          ts->id_thr = 0;
          ts->p_d = d == 0 ? 1.0f : 0.0f;
          ts->mode = kModeOneHot;
          ts->amax_key = 0ull;
        } else {
          ds->m = m;
          ds->D = 1.0f;
          ds->q_d = 0.0f;
          ds->zero = 1;
        }
      }
      return;
    }

    // ---- pass 2 (L2): fixed-point mass (+ first top-p histogram) -----------------
    if (topp) hist_clear(sm, kRowBins);
    __syncthreads();
    unsigned long long F = 0ull;
    if (topp) {
      row_sweep<4>(rv, pol_keep, fix, [&](int, float x) {
        const unsigned long long f = fixed_mass(exp_rel(x, m));
        F += f;
        hist_add_mass(sm, adigit0(x, m), f);
      });
    } else {
      F = slice_mass(rv, pol_last_use, fix, m);
    }
    F = cluster_sum_u64(cl, sm, F, set, CL);

    uint32_t kd_thr = 0u;
    int32_t id_thr = 0;
    unsigned long long Fk = F;
    int32_t mode = kModeKeepAll;
    if (topp) {
      mode = kModeThreshold;
      const unsigned long long P32 = topp_scaled(P.top_p[s]);
      const unsigned long long t_lo = P32 * F;
      const unsigned long long t_hi = __umul64hi(P32, F);
      // stage 0 (its histogram was built in pass 2): distance bins, ascending
      // (a mass-only histogram: the bin's count is unknown, so stage 1 always runs)
      Found f = cluster_find(cl, sm, kRowBins, false, 0ull, t_hi, t_lo, CL, rank, 0xFFFFFFFFu,
                             0u, false);
      f.cnt = 0u;
      unsigned long long above = f.before;
      const int a0 = f.bin;
      int a1 = -1;
      int kd_len = 0, id_len = 0;
      uint32_t kd_pre = 0u, id_pre = 0u;
      // Stages 1..6 split the boundary bin until it holds one element: the
      // distance sub-bins, kd bits [31:21], [20:10], [9:0], id bits [21:11],
      // [10:0]. After the last id stage the bin is a single token. Once the
      // bin holds a single value, the value stages left are skipped.
      // Stage 1 also copies its candidates (the elements of bin a0) to this
      // CTA's list; the later stages read the list instead of the slice
      // unless it overflowed.
      uint2* list = P.cand + static_cast<size_t>(blockIdx.x) * kVerifyListCap;
      unsigned int list_len = 0xFFFFFFFFu;  // not built yet
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
        hist_clear(sm, nb);
        if (stage == 1 && tid == 0) sm.list_n = 0u;
        __syncthreads();
        uint32_t cmin = 0xFFFFFFFFu, cmax = 0u;  // value-key range of the candidates
        auto visit = [&](uint32_t id, float x, bool append) {
          const uint32_t kd = kd_of(x);
          if (match(x, kd, id)) {
            hist_add(sm, true, digit(x, kd, id), fixed_mass(exp_rel(x, m)), id);
            cmin = min(cmin, kd);
            cmax = max(cmax, kd);
            if (append) {
              const unsigned int at = atomicAdd(&sm.list_n, 1u);
              if (at < static_cast<unsigned int>(kVerifyListCap))
                list[at] = make_uint2(id, __float_as_uint(x));
            }
          }
        };
        if (list_len <= static_cast<unsigned int>(kVerifyListCap)) {
          for (unsigned int j = tid; j < list_len; j += kRowThreads) {
            const uint2 e = __ldcg(list + j);
            visit(e.x, __uint_as_float(e.y), false);
          }
        } else {
          const bool append = stage == 1;
          row_sweep<4>(rv, pol_keep, fix, [&](int i, float x) {
            visit(static_cast<uint32_t>(v0 + i), x, append);
          });
        }
        f = cluster_find(cl, sm, nb, desc, above, t_hi, t_lo, CL, rank, cmin, cmax);
        if (stage == 1) list_len = sm.list_n;  // complete: cluster_find synchronised the CTA
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
        // row), so the boundary bin does too: the value stages cannot split
        // it, go on with the token-id stages
        if (stage < 5 && f.cnt > 1u && f.kmin == f.kmax) {
          kd_pre = f.kmin;
          kd_len = 32;
          stage = 4;
        }
      }
      // f is the one-element bin at the boundary: its token, mass and logit
      id_thr = static_cast<int32_t>(f.id);
      Fk = above + f.mass;
      kd_thr = kd_of(fix(raw_at(id_thr)));
    }
    const float D = __fmul_rn(__ull2float_rn(Fk), 0x1p-40f);

    // ---- outputs (rank 0): p or q at the drafted token, the row statistics --------
    if (rank == 0 && tid == 0) {
      const bool has_d = d >= 0 && d < V;
      const float x = has_d ? fix(raw_at(d)) : 0.0f;
      if (is_target) {
        const uint32_t kd = kd_of(x);
        const bool keep = mode == kModeKeepAll || kd > kd_thr || (kd == kd_thr && d <= id_thr);
        ts->p_d = has_d && keep ? __fdiv_rn(exp_rel(x, m), D) : 0.0f;
        ts->m = m;
        ts->D = D;
        ts->kd_thr = kd_thr;
        ts->id_thr = id_thr;
        ts->mode = mode;
        ts->amax_key = 0ull;
      } else {
        ds->q_d = has_d ? __fdiv_rn(exp_rel(x, m), D) : 0.0f;
        ds->m = m;
        ds->D = D;
        ds->zero = 0;
      }
    }
  };
  if (is_target && T != 1.0f)
    passes([T](float c) { return __fdiv_rn(c, T); });
  else
    passes([](float c) { return c; });
}

// ---------------------------------------------------------------------------
// Persistent clusters: cluster c handles rows c, c + nclusters, ...
__global__ void __launch_bounds__(kRowThreads, 4) verify_rows_kernel(VerifyParams P, int W,
                                                                     int nrows) {
  cg::cluster_group cl = cg::this_cluster();
  const int CL = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int cid = blockIdx.x / CL;
  const int nclusters = gridDim.x / CL;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  RowSmem& sm = *reinterpret_cast<RowSmem*>(smem_raw);
  // the draw kernel that follows counts its finished chunks per request here
  if (blockIdx.x == 0)
    for (int b = threadIdx.x; b < P.B; b += kRowThreads) P.counters[b] = 0u;
  int jrow = 0;
  // odd clusters walk their rows backward: about half the clusters stream a
  // draft row (one pass) while the others are on a target row (two passes)
  const int nmine = nrows > cid ? (nrows - cid + nclusters - 1) / nclusters : 0;
  const int first = (cid & 1) ? cid + (nmine - 1) * nclusters : cid;
  const int stride = (cid & 1) ? -nclusters : nclusters;
  for (int row = first; row >= cid && row < nrows; row += stride)
    process_row(P, W, row, cl, CL, rank, sm, jrow);
  cl.sync();  // no CTA exits while another may still read its shared memory
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
  rv.vec = rv.bf16 ? (reinterpret_cast<uintptr_t>(rv.h) & 7u) == 0
                   : (reinterpret_cast<uintptr_t>(rv.f) & 15u) == 0;
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

cudaError_t launch_verify_rows(const VerifyParams& p, int CL, int W, cudaStream_t stream) {
  const int rows = p.B * (p.K + 1) + p.B * p.K;
  const size_t smem = verify_rows_smem_bytes(W);
  cudaError_t err = cudaFuncSetAttribute(verify_rows_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  if (CL > 8) {
    err = cudaFuncSetAttribute(verify_rows_kernel,
                               cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
  // As many clusters as fit on the GPU at once, each looping over rows, but
  // no more rows in flight than about 80 MB of L2 holds: every pass after
  // the first reads the row again from L2.
  cfg.gridDim = dim3(static_cast<unsigned>(rows * CL), 1, 1);
  int max_clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&max_clusters, verify_rows_kernel, &cfg) != cudaSuccess ||
      max_clusters < 1) {
    (void)cudaGetLastError();
    max_clusters = 1;
  }
  const size_t row_bytes = static_cast<size_t>(p.V) * (p.target_bf16 ? 2 : 4);
  const int l2_rows = static_cast<int>((80ull << 20) / (row_bytes > 0 ? row_bytes : 1));
  int nclusters = rows < max_clusters ? rows : max_clusters;
  if (l2_rows >= 1 && nclusters > l2_rows) nclusters = l2_rows;
  if (nclusters * CL > kVerifyMaxCtas) nclusters = kVerifyMaxCtas / CL;  // one list per CTA
  if (nclusters < 1) nclusters = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters * CL), 1, 1);
  return cudaLaunchKernelEx(&cfg, verify_rows_kernel, p, W, rows);
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
