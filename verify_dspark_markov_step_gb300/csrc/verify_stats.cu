// verify_stats.cu -- per-row statistics of the verifier, one thread-block
// cluster per row.
//
// vLLM PR #65007 Part 2 ("Temperature and top-p"): the target row after
// temperature, its maximum and total exp-mass in 64-bit fixed point, and the
// exact top-p keep set -- the smallest prefix by (logit desc, token id asc)
// whose mass reaches p, plus the row max. Draft rows (the cache) get their
// maximum and fixed-point mass. Greedy target rows get their winner key.
//
// A row is split over the CL CTAs of a cluster (CL up to 16). Each CTA reads
// its slice from HBM exactly once into shared memory and every later pass
// (fixed-point mass, the radix stages of the top-p select) runs on the
// shared-memory copy. Reductions across the cluster go through distributed
// shared memory: scalars by each CTA reading the others' slots, histograms
// by each CTA reducing its own range of bins over the cluster.
//
// Top-p select: a radix select on the ordered bits kd of the scaled logits,
// most significant first (11 + 11 + 10 bits), with histograms of fixed-point
// mass; each stage finds the first bin (in descending kd order) at which the
// running mass reaches P32 * F / 2^32. Exact ties at the boundary value are
// resolved by two more stages on the token id (ascending, 11 + 11 bits).
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "verify_common.cuh"

namespace cg = cooperative_groups;

namespace dspark {

namespace {

constexpr int kRowThreads = 512;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowBins = 2048;
constexpr size_t kRowSmemLimit = 227u * 1024u;

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
// running mass (starting from `above`) reaches the target (t_hi:t_lo).
__device__ Found cluster_find(cg::cluster_group& cl, RowSmem& sm, int nb, bool desc,
                              unsigned long long above, unsigned long long t_hi,
                              unsigned long long t_lo, int CL, int rank) {
  const int tid = threadIdx.x;
  const int b0 = rank * nb / CL;
  const int w = (rank + 1) * nb / CL - b0;
  __syncthreads();
  cl.sync();  // every local histogram is complete
  // 1. reduce the bins this CTA owns over the cluster
  constexpr int kPer = kRowBins / kRowThreads;  // at most 4 owned bins per thread
  unsigned long long rm[kPer];
  unsigned int rc[kPer], ri[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    rm[j] = 0ull;
    rc[j] = 0u;
    ri[j] = 0u;
    const int bi = tid + j * kRowThreads;
    if (bi < w) {
      for (int r = 0; r < CL; ++r) {
        RowSmem* o = cl.map_shared_rank(&sm, r);
        rm[j] += o->hmass[b0 + bi];
        rc[j] += o->hcnt[b0 + bi];
        ri[j] = max(ri[j], o->hid[b0 + bi]);
      }
    }
  }
  cl.sync();  // every remote read is done; owned bins may be overwritten
  unsigned long long mine = 0ull;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int bi = tid + j * kRowThreads;
    if (bi < w) {
      sm.hmass[b0 + bi] = rm[j];
      sm.hcnt[b0 + bi] = rc[j];
      sm.hid[b0 + bi] = ri[j];
      mine += rm[j];
    }
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
    if (sm.hcnt[bin] > 0u && reaches(run + mb, t_hi, t_lo)) {
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
    for (int r = 0; r < CL; ++r) {
      const int p = cl.map_shared_rank(&sm, r)->x_pos;
      if (p < best_pos) {
        best_pos = p;
        best_r = r;
      }
    }
    sm.bcast_i = best_r;
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
  cl.sync();  // slots may be rewritten by the next stage
  return f;
}

// One local histogram pass over the shared-memory slice: elements whose kd
// and id pass `match` add their fixed-point mass to bin digit(kd, id).
template <class Val, class Match, class Digit>
__device__ void hist_pass(RowSmem& sm, Val xval, int n, int v0, float m, int nb, Match match,
                          Digit digit) {
  hist_clear(sm, nb);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  for (int base = threadIdx.x & ~31; base < n; base += kRowThreads) {
    const int i = base + lane;
    const bool valid = i < n;
    const float x = valid ? xval(i) : -INFINITY;
    const uint32_t kd = kd_of(x);
    const uint32_t id = static_cast<uint32_t>(v0 + i);
    const bool act = valid && match(kd, id);
    const unsigned long long f = act ? fixed_mass(exp_rel(x, m)) : 0ull;
    hist_add(sm, act, act ? digit(kd, id) : 0, f, id);
  }
}

// Loads the slice [v0, v0 + n) of a row into shared memory: one bulk copy of
// the 16-byte-aligned body (issued by thread 0, completion on `bar`), plain
// loads for a ragged tail or an unaligned row. fp32 rows land as fp32, bf16
// rows as bf16 bit patterns. Returns false if the bounded wait ran out.
__device__ bool slice_fetch(const void* row, bool bf16, int v0, int n, void* dst, uint64_t* bar,
                            uint32_t& phase, int32_t* status) {
  const int es = bf16 ? 2 : 4;
  const unsigned char* src = static_cast<const unsigned char*>(row) + static_cast<size_t>(v0) * es;
  const bool aligned = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  const int body = aligned ? ((n * es) & ~15) / es : 0;  // elements moved by the bulk copy
  if (body > 0 && threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(body * es));
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(static_cast<uint32_t>(body * es)), "r"(smem_addr(bar))
        : "memory");
  }
  for (int j = body + threadIdx.x; j < n; j += kRowThreads) {
    if (bf16)
      static_cast<uint16_t*>(dst)[j] = __ldg(reinterpret_cast<const unsigned short*>(src) + j);
    else
      static_cast<float*>(dst)[j] = __ldg(reinterpret_cast<const float*>(src) + j);
  }
  bool ok = true;
  if (body > 0) {
    ok = mbar_wait(bar, phase, status);
    phase ^= 1u;
  }
  if (body < n) __syncthreads();  // the plain-loaded tail is visible to every thread
  return ok;
}

// One row: statistics written to P.tstats / P.dstats. Every CTA of the
// cluster runs the same sequence of cluster barriers (all decisions depend on
// the row or on cluster-reduced values only).
__device__ void process_row(const VerifyParams& P, int W, int row_id, cg::cluster_group& cl,
                            int CL, int rank, RowSmem& sm, float* xs, uint64_t* bar,
                            uint32_t& phase, int& jrow) {
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
  const void* row;
  bool bf16;
  if (is_target) {
    const int64_t off = (static_cast<int64_t>(b) * (K + 1) + k) * V;
    bf16 = P.target_bf16 != 0;
    row = bf16 ? static_cast<const void*>(static_cast<const uint16_t*>(P.target) + off)
               : static_cast<const void*>(static_cast<const float*>(P.target) + off);
  } else {
    const int64_t off = (crow * K + k) * V;
    bf16 = P.cache_bf16 != 0;
    row = bf16 ? static_cast<const void*>(static_cast<const uint16_t*>(P.cache) + off)
               : static_cast<const void*>(static_cast<const float*>(P.cache) + off);
  }
  const int32_t d = k < K ? P.draft[static_cast<int64_t>(b) * K + k] : -1;
  TgtStats* ts = static_cast<TgtStats*>(P.tstats) + static_cast<int64_t>(b) * (K + 1) + k;
  DrfStats* ds = static_cast<DrfStats*>(P.dstats) + static_cast<int64_t>(b) * K + (k < K ? k : 0);
  const uint16_t* xh = reinterpret_cast<const uint16_t*>(xs);

  // ---- the slice into shared memory --------------------------------------------
  fence_proxy_async_smem();
  const bool fetched = slice_fetch(row, bf16, v0, n, xs, bar, phase, P.status);

  // ---- greedy target row: winner key of the raw row ----------------------------
  if (is_target && greedy) {
    unsigned long long key = 0ull;
    for (int i = tid; i < n; i += kRowThreads) {
      const float t = bf16 ? bf16_bits_to_float(xh[i]) : xs[i];
      key = umax64(key, winner_key(t, static_cast<uint32_t>(v0 + i)));
    }
    key = cluster_max_u64(cl, sm, fetched ? key : 0ull, set, CL);
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

  // ---- pass 1: scale in place (fp32) and maximum -----------------------------------
  // bf16 slices stay as bit patterns; the passes widen them on the fly.
  float lmax = -INFINITY;
  if (bf16) {
    for (int i = tid; i < n; i += kRowThreads) {
      const float c = bf16_bits_to_float(xh[i]);
      lmax = fmaxf(lmax, is_target ? scale_logit(c, T) : ((c != c) ? -INFINITY : c));
    }
  } else {
    auto fix = [&](float c) { return is_target ? scale_logit(c, T) : ((c != c) ? -INFINITY : c); };
    const int n4 = n >> 2;
    float4* xs4 = reinterpret_cast<float4*>(xs);
    for (int i = tid; i < n4; i += kRowThreads) {
      const float4 c = xs4[i];
      const float4 x = make_float4(fix(c.x), fix(c.y), fix(c.z), fix(c.w));
      if (__float_as_uint(x.x) != __float_as_uint(c.x) || __float_as_uint(x.y) != __float_as_uint(c.y) ||
          __float_as_uint(x.z) != __float_as_uint(c.z) || __float_as_uint(x.w) != __float_as_uint(c.w))
        xs4[i] = x;
      lmax = fmaxf(lmax, fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)));
    }
    for (int i = 4 * n4 + tid; i < n; i += kRowThreads) {
      const float c = xs[i];
      const float x = fix(c);
      if (__float_as_uint(x) != __float_as_uint(c)) xs[i] = x;
      lmax = fmaxf(lmax, x);
    }
  }
  // a timed-out copy drops the row for the whole cluster (status is set)
  bool any_fail = false;
  const float m = cluster_max_f(cl, sm, lmax, !fetched, set, CL, &any_fail);
  if (any_fail) return;
  auto xval = [&](int i) -> float {
    if (!bf16) return xs[i];
    const float c = bf16_bits_to_float(xh[i]);
    return is_target ? scale_logit(c, T) : ((c != c) ? -INFINITY : c);
  };
  // The drafted token's value, read now: after this row's last cluster
  // barrier the CTA's threads may already be loading the next row's slice.
  const bool own_d = tid == 0 && d >= v0 && d < v0 + n;
  const float xd = own_d ? xval(d - v0) : 0.0f;
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

  // ---- pass 2: fixed-point mass (+ first top-p histogram) -------------------------
  const bool topp = is_target && P.top_p[s] < 1.0f;
  if (topp) hist_clear(sm, kRowBins);
  __syncthreads();
  unsigned long long F = 0ull;
  if (topp) {
    const int lane = tid & 31;
    for (int base = tid & ~31; base < n; base += kRowThreads) {
      const int i = base + lane;
      const bool valid = i < n;
      const float x = valid ? xval(i) : -INFINITY;
      const unsigned long long f = valid ? fixed_mass(exp_rel(x, m)) : 0ull;
      F += f;
      hist_add(sm, valid, static_cast<int>(kd_of(x) >> 21), f, static_cast<uint32_t>(v0 + i));
    }
  } else if (!bf16) {
    const int n4 = n >> 2;
    for (int i = tid; i < n4; i += kRowThreads) {
      const float4 x4 = reinterpret_cast<const float4*>(xs)[i];
      F += fixed_mass(exp_rel(x4.x, m)) + fixed_mass(exp_rel(x4.y, m)) +
           fixed_mass(exp_rel(x4.z, m)) + fixed_mass(exp_rel(x4.w, m));
    }
    for (int i = 4 * n4 + tid; i < n; i += kRowThreads) F += fixed_mass(exp_rel(xs[i], m));
  } else {
    for (int i = tid; i < n; i += kRowThreads) F += fixed_mass(exp_rel(xval(i), m));
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
    bool resolved = false;
    // kd stage 0: bits [31:21]
    Found f = cluster_find(cl, sm, kRowBins, true, 0ull, t_hi, t_lo, CL, rank);
    unsigned long long above = f.before;
    uint32_t pre = static_cast<uint32_t>(f.bin);
    if (f.cnt == 1u) {
      id_thr = static_cast<int32_t>(f.id);
      Fk = above + f.mass;
      resolved = true;
    }
    if (!resolved) {  // kd stage 1: bits [20:10]
      const uint32_t p0 = pre;
      hist_pass(sm, xval, n, v0, m, kRowBins, [=](uint32_t kd, uint32_t) { return (kd >> 21) == p0; },
                [](uint32_t kd, uint32_t) { return static_cast<int>((kd >> 10) & 0x7FFu); });
      f = cluster_find(cl, sm, kRowBins, true, above, t_hi, t_lo, CL, rank);
      above = f.before;
      pre = (pre << 11) | static_cast<uint32_t>(f.bin);
      if (f.cnt == 1u) {
        id_thr = static_cast<int32_t>(f.id);
        Fk = above + f.mass;
        resolved = true;
      }
    }
    if (!resolved) {  // kd stage 2: bits [9:0]
      const uint32_t p1 = pre;
      hist_pass(sm, xval, n, v0, m, 1024, [=](uint32_t kd, uint32_t) { return (kd >> 10) == p1; },
                [](uint32_t kd, uint32_t) { return static_cast<int>(kd & 0x3FFu); });
      f = cluster_find(cl, sm, 1024, true, above, t_hi, t_lo, CL, rank);
      above = f.before;
      pre = (pre << 10) | static_cast<uint32_t>(f.bin);
      if (f.cnt == 1u) {
        id_thr = static_cast<int32_t>(f.id);
        Fk = above + f.mass;
        resolved = true;
      }
    }
    if (resolved) {
      // full kd of the boundary element, read from the CTA that holds it
      if (tid == 0) {
        const int owner = id_thr / W;
        const int li = id_thr - owner * W;
        float xb;
        if (bf16) {
          const float c = bf16_bits_to_float(
              *cl.map_shared_rank(const_cast<uint16_t*>(xh) + li, owner));
          xb = scale_logit(c, T);
        } else {
          xb = *cl.map_shared_rank(xs + li, owner);
        }
        sm.bcast_i = static_cast<int>(kd_of(xb));
      }
      cl.sync();  // the owner keeps its slice until this remote read is done
      kd_thr = static_cast<uint32_t>(sm.bcast_i);
    } else {
      // exact ties at the boundary value: token id ascending, 11 + 11 bits
      kd_thr = pre;
      const uint32_t kt = kd_thr;
      hist_pass(sm, xval, n, v0, m, kRowBins, [=](uint32_t kd, uint32_t) { return kd == kt; },
                [](uint32_t, uint32_t id) { return static_cast<int>((id >> 11) & 0x7FFu); });
      f = cluster_find(cl, sm, kRowBins, false, above, t_hi, t_lo, CL, rank);
      above = f.before;
      if (f.cnt == 1u) {
        id_thr = static_cast<int32_t>(f.id);
        Fk = above + f.mass;
      } else {
        const uint32_t ip = static_cast<uint32_t>(f.bin);
        hist_pass(sm, xval, n, v0, m, kRowBins,
                  [=](uint32_t kd, uint32_t id) { return kd == kt && (id >> 11) == ip; },
                  [](uint32_t, uint32_t id) { return static_cast<int>(id & 0x7FFu); });
        f = cluster_find(cl, sm, kRowBins, false, above, t_hi, t_lo, CL, rank);
        above = f.before;
        id_thr = static_cast<int32_t>(f.id);
        Fk = above + f.mass;
      }
    }
  }
  const float D = __fmul_rn(__ull2float_rn(Fk), 0x1p-40f);

  // ---- outputs: p or q at the drafted token (its owner), the rest (rank 0) ---------
  if (own_d) {
    const float x = xd;
    if (is_target) {
      const uint32_t kd = kd_of(x);
      const bool keep = mode == kModeKeepAll || kd > kd_thr || (kd == kd_thr && d <= id_thr);
      ts->p_d = keep ? __fdiv_rn(exp_rel(x, m), D) : 0.0f;
    } else {
      ds->q_d = __fdiv_rn(exp_rel(x, m), D);
    }
  }
  if (rank == 0 && tid == 0) {
    if (is_target) {
      ts->m = m;
      ts->D = D;
      ts->kd_thr = kd_thr;
      ts->id_thr = id_thr;
      ts->mode = mode;
      ts->amax_key = 0ull;
      if (!(d >= 0 && d < V)) ts->p_d = 0.0f;
    } else {
      ds->m = m;
      ds->D = D;
      ds->zero = 0;
      if (!(d >= 0 && d < V)) ds->q_d = 0.0f;
    }
  }
  // A CTA may start its next slice copy now: its own threads are past every
  // read of this slice (the last cluster barrier), and the other CTAs read a
  // remote slice only inside the top-p stages, which end with a barrier.
}

// ---------------------------------------------------------------------------
// Persistent clusters: cluster c handles rows c, c + nclusters, ...
__global__ void __launch_bounds__(kRowThreads, 2) verify_rows_kernel(VerifyParams P, int W,
                                                                     int nrows) {
  cg::cluster_group cl = cg::this_cluster();
  const int CL = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int cid = blockIdx.x / CL;
  const int nclusters = gridDim.x / CL;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  RowSmem& sm = *reinterpret_cast<RowSmem*>(smem_raw);
  float* xs = reinterpret_cast<float*>(smem_raw + ((sizeof(RowSmem) + 15) & ~size_t(15)));
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  cl.sync();  // barriers initialised in every CTA before any row starts
  uint32_t phase = 0;
  int jrow = 0;
  for (int row = cid; row < nrows; row += nclusters)
    process_row(P, W, row, cl, CL, rank, sm, xs, &bar, phase, jrow);
  cl.sync();  // no CTA exits while another may still touch its shared memory
}

}  // namespace

size_t verify_rows_smem_bytes(int W) {
  return ((sizeof(RowSmem) + 15) & ~size_t(15)) + static_cast<size_t>(W) * sizeof(float);
}

// Cluster size and slice width for vocabulary V: slices small enough for two
// CTAs per SM (at most 100 KB of shared memory), and among those cluster
// sizes the one that keeps the most CTAs resident (the GPU places a cluster
// inside one GPC, so 16-CTA clusters can leave SMs idle).
bool verify_rows_plan(int V, int* CL, int* W) {
  int best_cl = 0, best_w = 0, best_ctas = -1;
  const int candidates[] = {16, 14, 12, 10, 8, 6, 4, 2, 1};
  for (int cl : candidates) {
    int w = (V + cl - 1) / cl;
    w = (w + 7) & ~7;
    const size_t smem = verify_rows_smem_bytes(w);
    if (smem > 100u * 1024u && cl < 16) break;  // smaller clusters only get larger slices
    if (smem > kRowSmemLimit) continue;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kRowThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.gridDim = dim3(static_cast<unsigned>(cl * 64), 1, 1);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaFuncSetAttribute(verify_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        (cl > 8 && cudaFuncSetAttribute(verify_rows_kernel,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                       cudaSuccess) ||
        cudaOccupancyMaxActiveClusters(&clusters, verify_rows_kernel, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      clusters = 0;
    }
    if (clusters * cl > best_ctas) {
      best_ctas = clusters * cl;
      best_cl = cl;
      best_w = w;
    }
  }
  if (best_ctas <= 0) return false;
  *CL = best_cl;
  *W = best_w;
  return true;
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
  // as many clusters as fit on the GPU at once, each looping over rows
  cfg.gridDim = dim3(static_cast<unsigned>(rows * CL), 1, 1);
  int max_clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&max_clusters, verify_rows_kernel, &cfg) != cudaSuccess ||
      max_clusters < 1) {
    (void)cudaGetLastError();
    max_clusters = 1;
  }
  const int nclusters = rows < max_clusters ? rows : max_clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters * CL), 1, 1);
  return cudaLaunchKernelEx(&cfg, verify_rows_kernel, p, W, rows);
}

}  // namespace dspark
