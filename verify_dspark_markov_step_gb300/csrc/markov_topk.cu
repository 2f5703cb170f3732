// markov_topk.cu -- the top-k variant of the K-step Markov loop.
//
// The "DSparkSpeculator" page, _sample_sequential_topk: the Markov head is
// applied only to the top-k base-logit candidates of each draft step (chosen
// once, for every step, from the base logits); every other column of the
// step's logits is -inf, and the dense sampler (temperature, Gumbel noise,
// winner rule, draft-logits cache) then runs on that truncated row.
//
// Two launches: topk_rows_kernel (verify_stats.cu) selects the candidates of
// every (request, step) row and fills the cache rows with -inf; this file's
// kernel then runs the K steps of each request on a cluster of 8 CTAs that
// split its candidates. The bias of a candidate is the dot product of its
// markov_w2 row (gathered by 8 lanes, 16-byte loads, all in flight at once)
// with the Markov embedding: the projection shrinks from the whole
// vocabulary to k rows per request and step. The step's winner is reduced
// across the cluster through distributed shared memory.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace dspark {

namespace {

constexpr int kTopkThreads = 256;
constexpr int kTopkCluster = 8;  // CTAs per request
constexpr int kLanesPerCand = 8;

__global__ void __launch_bounds__(kTopkThreads) markov_topk_loop_kernel(TopkParams P) {
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank());
  extern __shared__ float s_e[];  // [R] the step's Markov embedding, fp32
  __shared__ unsigned long long s_warp[kTopkThreads / 32];
  __shared__ unsigned long long s_slot[2];  // this CTA's best key, per step parity
  const int b = blockIdx.x / kTopkCluster, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int K = P.K, V = P.V, R = P.R;
  const int k = P.k < V ? P.k : V;
  const int kc = (k + kTopkCluster - 1) / kTopkCluster;  // candidates of this CTA
  const int j0 = rank * kc, j1 = min(k, j0 + kc);

  // ---- per-request state (every CTA of the cluster decides alike) -----------
  const int32_t s = P.rsi[b];
  bool active = s >= 0 && s < P.S;
  int64_t crow = -1;
  if (active && P.cache != nullptr) {
    crow = P.row_map ? P.row_map[s] : s;
    if (crow < 0 || crow >= P.C) active = false;
  }
  int32_t prev = active ? P.anchor[b] : -1;
  if (active && !(prev >= 0 && prev < V)) active = false;
  if (!active) {
    if (rank == 0 && tid == 0 && s >= 0) report(P.status, DSPARK_ERR_BOUNDS);
    if (rank == 0)
      for (int i = tid; i < K; i += kTopkThreads)
        P.out_tokens[static_cast<int64_t>(b) * K + i] = -1;
    return;  // the whole cluster leaves: no cluster barrier follows
  }
  const float T = P.temperature[s];
  const bool scaled = T > 0.f && T != 1.f;  // x = z / T (IEEE); T = 1 and greedy: x = z
  const float gs = T > 0.f ? 1.f : 0.f;      // greedy: no noise
  const float tdiv = scaled ? T : 1.f;
  const unsigned long long r2 = f2_pack(__frcp_rn(tdiv), __frcp_rn(tdiv));
  const unsigned long long nt2 = f2_pack(-tdiv, -tdiv);
  const bool tslow = !temp_div_t_ok(tdiv);
  const uint64_t seed = P.seeds[s];
  const int64_t p0 = P.pos[b];
  const uint32_t neg_inf_key = ordered_key(-INFINITY);
  const int nq = R / 64;  // 16-byte chunks of a w2 row per lane (R / 8 chunks over 8 lanes)
  const int sub = lane / kLanesPerCand, sl = lane % kLanesPerCand;

  const uint32_t wbytes = static_cast<uint32_t>(R) * 2;  // one markov_w2 row
  for (int i = 0; i < K; ++i) {
    // the next step's candidates are already known: bring their markov_w2
    // rows into L2 while this step runs
    if (i + 1 < K) {
      const int32_t* nidx = P.cand_idx + (static_cast<int64_t>(b) * K + i + 1) * P.k;
      for (int j = j0 + tid; j < j1; j += kTopkThreads) {
        const uint16_t* row = P.w2 + static_cast<int64_t>(nidx[j]) * R;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(row), "r"(wbytes)
                     : "memory");
      }
    }
    for (int r = tid; r < R; r += kTopkThreads)
      s_e[r] = bf16_bits_to_float(P.w1[static_cast<int64_t>(prev) * R + r]);
    __syncthreads();
    const int64_t row_id = static_cast<int64_t>(b) * K + i;
    const int32_t* cidx = P.cand_idx + row_id * P.k;
    const float* cval = P.cand_val + row_id * P.k;
    unsigned long long best = 0ull;
    // 8 lanes per candidate, 4 candidates per warp and pass
    for (int jb = j0 + warp * 4; jb < j1; jb += (kTopkThreads / 32) * 4) {
      const int j = jb + sub;
      const bool has = j < j1;
      const int32_t v = has ? cidx[j] : 0;
      const uint4* wrow = reinterpret_cast<const uint4*>(P.w2 + static_cast<int64_t>(v) * R);
      uint4 u[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < nq && has) u[q] = __ldg(wrow + sl + q * kLanesPerCand);
      float acc = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (q < nq && has) {
          const float* e = s_e + (sl + q * kLanesPerCand) * 8;
          acc = fmaf(__uint_as_float(u[q].x << 16), e[0], acc);
          acc = fmaf(__uint_as_float(u[q].x & 0xFFFF0000u), e[1], acc);
          acc = fmaf(__uint_as_float(u[q].y << 16), e[2], acc);
          acc = fmaf(__uint_as_float(u[q].y & 0xFFFF0000u), e[3], acc);
          acc = fmaf(__uint_as_float(u[q].z << 16), e[4], acc);
          acc = fmaf(__uint_as_float(u[q].z & 0xFFFF0000u), e[5], acc);
          acc = fmaf(__uint_as_float(u[q].w << 16), e[6], acc);
          acc = fmaf(__uint_as_float(u[q].w & 0xFFFF0000u), e[7], acc);
        }
      }
      // sum over the candidate's 8 lanes
#pragma unroll
      for (int o = kLanesPerCand / 2; o > 0; o >>= 1)
        acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
      // (every lane computes z and x; lane 0 of a candidate's group keeps them)
      const float z = __fadd_rn(has ? cval[j] : 0.f, acc);
      float x, x_unused;
      f2_unpack(temp_div2(f2_pack(z, z), r2, nt2, tslow), x, x_unused);
      if (has && sl == 0) {
        const U4 blk = noise_block(seed, p0 + i - 1, static_cast<uint32_t>(v), kStreamDraft);
        const float y =
            __fmaf_rn(gumbel_of(pick_word(blk, static_cast<uint32_t>(v) & 3u)), gs, x);
        if (crow >= 0) {
          const int64_t co = (crow * K + i) * V + v;
          if (P.cache_bf16)
            static_cast<uint16_t*>(P.cache)[co] = float_to_bf16_bits(x);
          else
            static_cast<float*>(P.cache)[co] = x;
        }
        const uint32_t vkey = 0xFFFFFFFFu - static_cast<uint32_t>(v);
        best = umax64(best, (static_cast<unsigned long long>(ordered_key(y)) << 32) | vkey);
      }
    }
    best = warp_max64(best);
    if (lane == 0) s_warp[warp] = best;
    __syncthreads();
    if (tid == 0) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kTopkThreads / 32; ++w) m = umax64(m, s_warp[w]);
      s_slot[i & 1] = m;
    }
    cl.sync();  // every CTA's best of this step is in its slot
    if (tid < 32) {
      unsigned long long m =
          lane < kTopkCluster ? *cl.map_shared_rank(&s_slot[i & 1], lane) : 0ull;
      m = warp_max64(m);
      if (lane == 0) s_warp[0] = m;
    }
    __syncthreads();
    const unsigned long long m = s_warp[0];
    // every candidate -inf: the whole row is -inf and its first column wins
    const int32_t tok = static_cast<uint32_t>(m >> 32) == neg_inf_key ? 0 : key_index(m);
    if (rank == 0 && tid == 0) P.out_tokens[row_id] = tok;
    prev = tok;
    __syncthreads();  // s_warp and s_e are rewritten by the next step
  }
  cl.sync();  // no CTA exits while another may still read its slots
}

}  // namespace

cudaError_t launch_markov_topk_loop(const TopkParams& p, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B * kTopkCluster), 1, 1);
  cfg.blockDim = dim3(kTopkThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(p.R) * sizeof(float);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kTopkCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, markov_topk_loop_kernel, p);
}

}  // namespace dspark
