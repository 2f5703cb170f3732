// kernels.h -- launch interface between the C-ABI layer (api.cu) and the
// kernels (markov_tc.cu, verify_stats.cu, verify.cu). Internal to the library.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

// The K-step Markov loop.
struct MarkovStepParams {
  const void* base;
  int base_bf16;
  const uint16_t* w1;
  const uint16_t* w2;
  const int32_t* anchor;
  const int32_t* rsi;
  const int64_t* pos;
  const float* temperature;
  const uint64_t* seeds;
  void* cache;
  int cache_bf16;
  const int32_t* row_map;
  int32_t* out_tokens;
  int B, K, V, R, S, C;
  unsigned long long* keys;      // [K][B] winner key of each step and request (zeroed)
  dspark_row_stats* draft_stats; // [B][K] statistics of the cache rows written, or null (zeroed)
  unsigned int* counter;         // grid-barrier arrivals (zeroed before the launch)
  int32_t* status;
};

// Tensor-core variant (markov_tc.cu).
struct MarkovTcPlan {
  int Npad;            // batch padded to a multiple of 16 (UMMA N)
  int stages;          // shared-memory ring stages of 16 KB (markov_w2)
  int acc_buffers;     // TMEM accumulator buffers (2-4)
  int base_slots;      // staged base tiles (0: base read directly)
  unsigned tmem_cols;  // TMEM columns allocated
  unsigned base_stage_bytes;  // bytes of one staged base tile
  size_t smem;         // dynamic shared memory bytes
};
bool markov_tc_plan(int B, int R, int base_elem_bytes, bool base_tma_ok, MarkovTcPlan* plan);
int markov_tc_make_tmap(void* tmap_out /* 128-byte CUtensorMap */, const void* w2, int V, int R);
int markov_tc_make_base_tmap(void* tmap_out, const void* base, bool bf16, int B, int K, int V);
int markov_tc_grid(int V, int num_sms);
// All K steps in one cooperative launch of `grid` CTAs (at most one per SM).
cudaError_t launch_markov_loop_tc(const MarkovStepParams& p, const void* tmap, const void* bmap,
                                  const MarkovTcPlan& plan, int grid, cudaStream_t stream);

// Top-k variant of the Markov loop: candidate selection (verify_stats.cu)
// and the loop over the candidates (markov_topk.cu).
struct TopkParams {
  const void* base;
  int base_bf16;
  const uint16_t* w1;
  const uint16_t* w2;
  const int32_t* anchor;
  const int32_t* rsi;
  const int64_t* pos;
  const float* temperature;
  const uint64_t* seeds;
  void* cache;
  int cache_bf16;
  const int32_t* row_map;
  int32_t* out_tokens;
  int B, K, V, R, S, C, k;
  int32_t* cand_idx;  // [B*K][k] candidate token ids
  float* cand_val;    // [B*K][k] their base logits
  int32_t* status;
};
cudaError_t launch_topk_rows(const TopkParams& p, int CL, int W, cudaStream_t stream);
cudaError_t launch_markov_topk_loop(const TopkParams& p, cudaStream_t stream);

// Verification (verify.cu).
struct VerifyParams {
  const int32_t* draft;
  const void* cache;
  int cache_bf16;
  const int32_t* row_map;
  const dspark_row_stats* draft_stats;  // [B][K] from the Markov loop, or null
  const void* target;
  int target_bf16;
  const int32_t* rsi;
  const int64_t* pos;
  const float* temperature;
  const float* top_p;
  const uint64_t* seeds;
  int32_t* out_tokens;
  int32_t* num_accepted;
  int B, K, V, S, C;
  void* tstats;                  // [B][K+1] target-row statistics
  void* dstats;                  // [B][K] draft-row statistics
  unsigned long long* keys;      // [B][nchunk] chunk winner keys
  unsigned int* anypos;          // [B][nchunk] residual had a positive entry
  unsigned int* counters;        // [B] finished chunks (self-resetting)
  uint2* cand;                   // [kVerifyMaxCtas][kVerifyListCap] top-p candidates (id, x bits)
  int nchunk;
  int32_t* status;
};

// Row-statistics CTAs that keep a top-p candidate list in the workspace, and
// the list's capacity per CTA (a longer candidate set is swept instead).
constexpr int kVerifyMaxCtas = 1024;
constexpr int kVerifyListCap = 512;

size_t verify_tstats_bytes(int B, int K);
size_t verify_dstats_bytes(int B, int K);
int verify_max_chunks(int V);
int verify_chunks(int B, int V, int num_sms);
size_t verify_rows_smem_bytes(int W);
bool verify_rows_plan(int V, int es, int* CL, int* W);
cudaError_t launch_verify_rows(const VerifyParams& p, int CL, int W, cudaStream_t stream);
cudaError_t launch_verify(const VerifyParams& p, int CL, int W, cudaStream_t stream);

// Noise generator on its own (api.cu / verify.cu).
cudaError_t launch_noise(const uint64_t* seed, const int64_t* pos,
                         const uint32_t* col, const uint32_t* stream_word,
                         uint32_t* word, float* u, float* g, int64_t n,
                         cudaStream_t stream);

}  // namespace dspark
