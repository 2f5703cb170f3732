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
// kernel then runs the K steps of each request in one CTA. The bias of a
// candidate is the dot product of its markov_w2 row (gathered, 16-byte loads)
// with the Markov embedding, one candidate per thread: the projection shrinks
// from the whole vocabulary to k rows per request and step.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kTopkThreads = 256;

__global__ void __launch_bounds__(kTopkThreads) markov_topk_loop_kernel(TopkParams P) {
  extern __shared__ float s_e[];  // [R] the step's Markov embedding, fp32
  __shared__ unsigned long long s_best[kTopkThreads / 32];
  __shared__ int32_t s_tok;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int K = P.K, V = P.V, R = P.R;
  const int k = P.k < V ? P.k : V;

  // ---- per-request state (every thread reads the same values) --------------
  const int32_t s = P.rsi[b];
  bool active = s >= 0 && s < P.S;
  int64_t crow = -1;
  if (active && P.cache != nullptr) {
    crow = P.row_map ? P.row_map[s] : s;
    if (crow < 0 || crow >= P.C) {
      if (tid == 0) report(P.status, DSPARK_ERR_BOUNDS);
      active = false;
    }
  }
  int32_t prev = active ? P.anchor[b] : -1;
  if (active && !(prev >= 0 && prev < V)) {
    if (tid == 0) report(P.status, DSPARK_ERR_BOUNDS);
    active = false;
  }
  if (s >= P.S && tid == 0) report(P.status, DSPARK_ERR_BOUNDS);
  if (!active) {
    for (int i = tid; i < K; i += kTopkThreads) P.out_tokens[static_cast<int64_t>(b) * K + i] = -1;
    return;
  }
  const float T = P.temperature[s];
  const float xs = T > 0.f ? __frcp_rn(T) : 1.f;  // greedy: x = z
  const float gs = T > 0.f ? 1.f : 0.f;           // greedy: no noise
  const uint64_t seed = P.seeds[s];
  const int64_t p0 = P.pos[b];
  const uint32_t neg_inf_key = ordered_key(-INFINITY);

  for (int i = 0; i < K; ++i) {
    for (int r = tid; r < R; r += kTopkThreads)
      s_e[r] = bf16_bits_to_float(P.w1[static_cast<int64_t>(prev) * R + r]);
    __syncthreads();
    const int64_t row_id = static_cast<int64_t>(b) * K + i;
    const int32_t* cidx = P.cand_idx + row_id * P.k;
    const float* cval = P.cand_val + row_id * P.k;
    unsigned long long best = 0ull;
    for (int j = tid; j < k; j += kTopkThreads) {
      const int32_t v = cidx[j];
      // bias = markov_w2[v, :] . e, fp32 accumulation over 8-wide chunks
      const uint4* wrow = reinterpret_cast<const uint4*>(P.w2 + static_cast<int64_t>(v) * R);
      float acc = 0.f;
      for (int q = 0; q < R / 8; ++q) {
        const uint4 u = __ldg(wrow + q);
        const float* e = s_e + q * 8;
        acc = fmaf(__uint_as_float(u.x << 16), e[0], acc);
        acc = fmaf(__uint_as_float(u.x & 0xFFFF0000u), e[1], acc);
        acc = fmaf(__uint_as_float(u.y << 16), e[2], acc);
        acc = fmaf(__uint_as_float(u.y & 0xFFFF0000u), e[3], acc);
        acc = fmaf(__uint_as_float(u.z << 16), e[4], acc);
        acc = fmaf(__uint_as_float(u.z & 0xFFFF0000u), e[5], acc);
        acc = fmaf(__uint_as_float(u.w << 16), e[6], acc);
        acc = fmaf(__uint_as_float(u.w & 0xFFFF0000u), e[7], acc);
      }
      const float z = __fadd_rn(cval[j], acc);
      const float x = __fmul_rn(z, xs);
      const U4 blk = noise_block(seed, p0 + i - 1, static_cast<uint32_t>(v), kStreamDraft);
      const float y = __fmaf_rn(gumbel_of(pick_word(blk, static_cast<uint32_t>(v) & 3u)), gs, x);
      if (crow >= 0) {
        const int64_t co = (crow * K + i) * V + v;
        if (P.cache_bf16)
          static_cast<uint16_t*>(P.cache)[co] = float_to_bf16_bits(x);
        else
          static_cast<float*>(P.cache)[co] = x;
      }
      best = umax64(best, (static_cast<unsigned long long>(ordered_key(y)) << 32) |
                              static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(v)));
    }
    best = warp_max64(best);
    if ((tid & 31) == 0) s_best[tid >> 5] = best;
    __syncthreads();
    if (tid == 0) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kTopkThreads / 32; ++w) m = umax64(m, s_best[w]);
      // every candidate -inf: the whole row is -inf and its first column wins
      const int32_t tok = static_cast<uint32_t>(m >> 32) == neg_inf_key ? 0 : key_index(m);
      P.out_tokens[row_id] = tok;
      s_tok = tok;
    }
    __syncthreads();
    prev = s_tok;
  }
}

}  // namespace

cudaError_t launch_markov_topk_loop(const TopkParams& p, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  markov_topk_loop_kernel<<<p.B, kTopkThreads, static_cast<size_t>(p.R) * sizeof(float), stream>>>(
      p);
  return cudaGetLastError();
}

}  // namespace dspark
