// markov_step.cu -- one step of the drafter's sequential Markov loop, fused.
//
// Follows the "DSparkSpeculator" API page (_sample_markov_chain,
// _sample_logits) and vLLM PR #65007 Part 1 (per-step list, items 1-4):
// Markov embedding of the previous token, the markov_w2 bias projection, the
// bias add, temperature, Gumbel noise keyed by (seed, position - 1, column),
// the block-argmax winner rule, and the draft-logits cache store -- in one
// kernel per step, plus a last-CTA reduction of the per-CTA winners.
//
// This file holds the CUDA-core variant: every CTA streams whole 64-row
// tiles of markov_w2 (contiguous 64*R*2 bytes) into shared memory with 1-D
// bulk copies (two stages), computes the bias of its 64 columns for every
// request from the tile, and runs the epilogue (bias add, temperature,
// noise, winner key, cache store) straight from registers.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kTileV = 64;      // vocabulary rows per tile
constexpr int kThreads = 128;   // 2 threads per row: each owns half of R
constexpr int kStages = 2;

struct ReqInfo {
  float temperature;   // > 0 sampled, else greedy
  int32_t valid;       // 0 = padding or out of range
  int32_t prev;
  int32_t pad_;
  uint64_t seed;
  int64_t noise_pos;   // P0 + step - 1
  int64_t cache_off;   // element offset of cache[row, step, 0], or -1
};

// Dynamic shared memory layout (all offsets 16-byte aligned):
//   [stages][kTileV][R] bf16   w2 tiles
//   [B][R] bf16                Markov embeddings e[b] = w1[prev_b]
//   [B] ReqInfo
//   [B] u64                    running winner key of this CTA
//   2 x u64                    mbarriers
struct SmemLayout {
  size_t w2, e, info, best, bars, total;
  __host__ __device__ SmemLayout(int B, int R) {
    w2 = 0;
    e = w2 + static_cast<size_t>(kStages) * kTileV * R * 2;
    info = e + ((static_cast<size_t>(B) * R * 2 + 15) & ~size_t(15));
    best = info + static_cast<size_t>(B) * sizeof(ReqInfo);
    bars = best + static_cast<size_t>(B) * 8;
    total = bars + kStages * 8;
  }
};

template <int NCH>  // R = 64 * NCH; each thread covers R/2 = 32*NCH elements
__global__ void __launch_bounds__(kThreads)
markov_step_simt_kernel(MarkovStepParams P) {
  constexpr int R = 64 * NCH;
  constexpr int CH_HALF = 4 * NCH;  // 16-byte chunks per half row
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout L(P.B, R);
  uint16_t* w2s = reinterpret_cast<uint16_t*>(smem + L.w2);
  uint16_t* es = reinterpret_cast<uint16_t*>(smem + L.e);
  ReqInfo* info = reinterpret_cast<ReqInfo*>(smem + L.info);
  unsigned long long* best = reinterpret_cast<unsigned long long*>(smem + L.best);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);

  const int tid = threadIdx.x;
  const int B = P.B, V = P.V, K = P.K, step = P.step;

  // ---- prologue: per-request state and Markov embeddings ------------------
  for (int b = tid; b < B; b += kThreads) {
    ReqInfo ri;
    const int32_t s = P.rsi[b];
    ri.valid = 0;
    ri.prev = -1;
    ri.temperature = 0.f;
    ri.seed = 0;
    ri.noise_pos = 0;
    ri.cache_off = -1;
    ri.pad_ = 0;
    if (s >= 0) {
      if (s >= P.S) {
        report(P.status, DSPARK_ERR_BOUNDS);
      } else {
        const int32_t prev =
            step == 0 ? P.anchor[b] : P.out_tokens[static_cast<int64_t>(b) * K + step - 1];
        bool ok = prev >= 0 && prev < V;
        if (!ok) report(P.status, DSPARK_ERR_BOUNDS);
        int64_t off = -1;
        if (ok && P.cache != nullptr) {
          const int64_t row = P.row_map ? P.row_map[s] : s;
          if (row < 0 || row >= P.C) {
            report(P.status, DSPARK_ERR_BOUNDS);
            ok = false;
          } else {
            off = (row * K + step) * static_cast<int64_t>(V);
          }
        }
        if (ok) {
          ri.valid = 1;
          ri.prev = prev;
          ri.temperature = P.temperature[s];
          ri.seed = P.seeds[s];
          ri.noise_pos = P.pos[b] + step - 1;
          ri.cache_off = off;
        }
      }
    }
    info[b] = ri;
    best[b] = 0ull;
  }
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], 1);
    fence_mbar_init();
  }
  __syncthreads();
  {
    const int chunks_per_row = R / 8;
    const int total = B * chunks_per_row;
    for (int c = tid; c < total; c += kThreads) {
      const int b = c / chunks_per_row, j = c % chunks_per_row;
      const int prev = info[b].valid ? info[b].prev : 0;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(P.w1 + static_cast<int64_t>(prev) * R) + j);
      reinterpret_cast<uint4*>(es + static_cast<int64_t>(b) * R)[j] = v;
    }
  }

  // ---- tile loop -------------------------------------------------------------
  const int num_tiles = (V + kTileV - 1) / kTileV;
  const int G = gridDim.x;
  const uint64_t pol_w2 = policy_evict_last();
  auto issue = [&](int local_k) {
    const int t = blockIdx.x + local_k * G;
    if (t >= num_tiles) return;
    const int stage = local_k % kStages;
    const int v0 = t * kTileV;
    const int rows = min(kTileV, V - v0);
    const uint32_t bytes = static_cast<uint32_t>(rows) * R * 2;
    mbar_arrive_expect_tx(&bars[stage], bytes);
    bulk_g2s(w2s + static_cast<size_t>(stage) * kTileV * R,
             P.w2 + static_cast<int64_t>(v0) * R, bytes, &bars[stage], pol_w2);
  };
  if (tid == 0) {
    for (int k = 0; k < kStages; ++k) issue(k);
  }
  __syncthreads();

  const int col = tid >> 1;  // row of the tile owned by this thread pair
  const int half = tid & 1;
  const bool base_bf16 = P.base_bf16 != 0;
  const bool cache_bf16 = P.cache_bf16 != 0;
  int fail_k = -1;

  for (int k = 0;; ++k) {
    const int t = blockIdx.x + k * G;
    if (t >= num_tiles) break;
    const int stage = k % kStages;
    const uint32_t phase = (k / kStages) & 1u;
    const bool ok = mbar_wait(&bars[stage], phase, P.status);
    if (__syncthreads_or(!ok)) {
      fail_k = k;
      break;
    }
    const int v0 = t * kTileV;
    const int v = v0 + col;
    const bool in_range = v < V;
    const uint16_t* wrow = w2s + (static_cast<size_t>(stage) * kTileV + col) * R;

    // Load this thread's half row of w2 into registers as fp32 pairs.
    float wf[CH_HALF * 8];
#pragma unroll
    for (int j = 0; j < CH_HALF; ++j) {
      // rotate the chunk order by the row so that 8 consecutive threads hit
      // 8 different bank groups; the two halves are offset by 4 chunks
      const int cj = (j + col + 4 * half) % CH_HALF + half * CH_HALF;
      const uint4 raw = reinterpret_cast<const uint4*>(wrow)[cj];
      const uint32_t r4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        wf[j * 8 + 2 * q] = __uint_as_float(r4[q] << 16);
        wf[j * 8 + 2 * q + 1] = __uint_as_float(r4[q] & 0xFFFF0000u);
      }
    }

    for (int b = 0; b < B; ++b) {
      const uint16_t* erow = es + static_cast<size_t>(b) * R;
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < CH_HALF; ++j) {
        const int cj = (j + col + 4 * half) % CH_HALF + half * CH_HALF;
        const uint4 raw = reinterpret_cast<const uint4*>(erow)[cj];
        const uint32_t r4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc = fmaf(wf[j * 8 + 2 * q], __uint_as_float(r4[q] << 16), acc);
          acc = fmaf(wf[j * 8 + 2 * q + 1], __uint_as_float(r4[q] & 0xFFFF0000u), acc);
        }
      }
      acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
      const ReqInfo ri = info[b];
      uint32_t ord = 0u;
      // the pair's two threads share the row; the even one runs the epilogue
      if (half == 0 && in_range && ri.valid) {
        const int64_t boff = (static_cast<int64_t>(b) * K + step) * V + v;
        const float base = load_logit(P.base, base_bf16, boff);
        const float z = __fadd_rn(base, acc);
        float x = z, y = z;
        if (ri.temperature > 0.f) {
          x = ri.temperature == 1.0f ? z : __fdiv_rn(z, ri.temperature);
          const U4 r = noise_block(ri.seed, ri.noise_pos, static_cast<uint32_t>(v),
                                   kStreamDraft);
          y = __fadd_rn(x, gumbel_of(pick_word(r, static_cast<uint32_t>(v) & 3u)));
        }
        if (ri.cache_off >= 0) {
          if (cache_bf16)
            static_cast<uint16_t*>(P.cache)[ri.cache_off + v] = float_to_bf16_bits(x);
          else
            static_cast<float*>(P.cache)[ri.cache_off + v] = x;
        }
        ord = ordered_bits(y);  // every real value maps above 0
      }
      // winner over the warp's rows: largest value, then lowest column
      const uint32_t omax = __reduce_max_sync(0xFFFFFFFFu, ord);
      const uint32_t cand = (ord == omax && ord != 0u) ? static_cast<uint32_t>(v) : 0xFFFFFFFFu;
      const uint32_t vmin = __reduce_min_sync(0xFFFFFFFFu, cand);
      if ((tid & 31) == 0 && omax != 0u)
        atomicMax(&best[b], (static_cast<unsigned long long>(omax) << 32) | (0xFFFFFFFFu - vmin));
    }
    __syncthreads();  // every thread is done reading this stage
    if (tid == 0) {
      fence_proxy_async_smem();
      issue(k + kStages);
    }
  }

  if (fail_k >= 0 && tid == 0) {
    // A bounded wait ran out: before exiting, wait (bounded again) for the
    // copies this CTA still has in flight so none lands after it is gone.
    for (int k2 = fail_k; k2 < fail_k + kStages; ++k2) {
      if (blockIdx.x + k2 * G >= num_tiles) break;
      (void)mbar_wait(&bars[k2 % kStages], (k2 / kStages) & 1u, P.status);
    }
  }

  // ---- publish this CTA's winners; the last CTA reduces ----------------------
  __syncthreads();
  for (int b = tid; b < B; b += kThreads)
    P.partials[static_cast<int64_t>(b) * G + blockIdx.x] = best[b];
  __threadfence();
  __syncthreads();
  __shared__ unsigned int s_last;
  if (tid == 0) {
    const unsigned int ticket = atomicAdd(P.counter, 1u);
    s_last = (ticket == static_cast<unsigned int>(G) - 1u);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int b = tid; b < B; b += kThreads) {
    unsigned long long m = 0ull;
    const unsigned long long* row = P.partials + static_cast<int64_t>(b) * G;
    for (int g = 0; g < G; ++g) m = umax64(m, __ldcg(row + g));
    const int32_t tok = (info[b].valid && m != 0ull) ? key_index(m) : -1;
    P.out_tokens[static_cast<int64_t>(b) * K + step] = tok;
  }
  if (tid == 0) *P.counter = 0u;
}

}  // namespace

size_t markov_simt_smem_bytes(int B, int R) { return SmemLayout(B, R).total; }

int markov_simt_grid(int B, int V, int R, int num_sms) {
  const size_t smem = markov_simt_smem_bytes(B, R);
  int per_sm = static_cast<int>((227u * 1024u) / (smem + 1024));
  if (per_sm < 1) per_sm = 1;
  if (per_sm > 4) per_sm = 4;
  const int tiles = (V + kTileV - 1) / kTileV;
  const int g = per_sm * num_sms;
  return tiles < g ? tiles : g;
}

int markov_simt_max_grid(int V) { return (V + kTileV - 1) / kTileV; }

cudaError_t launch_markov_step_simt(const MarkovStepParams& p, int grid,
                                    cudaStream_t stream) {
  const size_t smem = markov_simt_smem_bytes(p.B, p.R);
  const int nch = p.R / 64;
  cudaError_t err = cudaSuccess;
  switch (nch) {
#define DSPARK_CASE(N)                                                          \
  case N:                                                                       \
    err = cudaFuncSetAttribute(markov_step_simt_kernel<N>,                      \
                               cudaFuncAttributeMaxDynamicSharedMemorySize,     \
                               static_cast<int>(smem));                         \
    if (err != cudaSuccess) return err;                                         \
    markov_step_simt_kernel<N><<<grid, kThreads, smem, stream>>>(p);            \
    break;
    DSPARK_CASE(1)
    DSPARK_CASE(2)
    DSPARK_CASE(3)
    DSPARK_CASE(4)
    DSPARK_CASE(5)
    DSPARK_CASE(6)
    DSPARK_CASE(7)
    DSPARK_CASE(8)
#undef DSPARK_CASE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace dspark
