// kernels.h -- launch interface between the C-ABI layer (api.cu) and the
// kernels (markov_tc.cu, verify_stats.cu, verify.cu). Internal to the library.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

// Upper bound of any spin on an mbarrier or flag, in nanoseconds of
// %globaltimer (about 2 s, like the pages' exchange timeout).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

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
  // Bounded waits: each mbarrier wait and the grid barrier give up after
  // wait_limit_ns; the grid barrier waits for barrier_extra arrivals more
  // than the grid makes (0 except in the bounded-wait test hook).
  unsigned long long wait_limit_ns;
  unsigned int barrier_extra;
};

// Host-side argument checks of dspark_markov_sample other than the workspace
// (sizes, dtypes, markov_rank, null pointers, alignment), in its order.
dspark_status markov_sample_args(const void* base_logits, dspark_dtype base_dtype,
                                 const uint16_t* markov_w1, const uint16_t* markov_w2,
                                 const int32_t* anchor_tokens, const int32_t* req_state_idx,
                                 const int64_t* positions, const float* temperature,
                                 const uint64_t* seeds, const void* cache,
                                 dspark_dtype cache_dtype, const int32_t* out_tokens, int B,
                                 int K, int V, int R, int S, int C);

// The Markov loop records draft-row statistics (maximum and exp-mass) for
// batches up to this size (8 request columns per epilogue warp, whose
// running sums fit in registers); above it the statistics read "not
// recorded" and the verifier reads the rows.
constexpr int kRowStatsMaxBatch = 32;

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
  unsigned long long* keys;      // [B][kstride] winner key of each draw sub-chunk
  unsigned int* anypos;          // [B][kstride] the sub-chunk had a positive weight
  unsigned int* ctl;             // per-request and per-row progress, draw jobs
  uint2* cand;                   // [kVerifyMaxCtas][kVerifyListCap] top-p candidates (id, x bits)
  void* parts;                   // [B * (2K + 1)][nslice] per-slice row partials
  int nslice;                    // slices per row in the flat kernel
  int kstride;                   // chunk slots per request in keys / anypos
  int ndraw;                     // draw chunks per request (set at launch)
  int stats_items;               // draft_stats hold the loop's recorded statistics:
                                 // a request's draft rows are one item, not read
  int32_t* status;
};

// VerifyParams::ctl: the draw queue's two words (on lines of their own), per
// request the rows finished, the draw chunks finished and the publish list,
// per row the slices finished (32-bit words, zeroed before each call's
// kernel), then one draw job per request (verify_draw.cuh).
size_t verify_ctl_bytes(int B, int K);
// Slices per row of the flat verification kernel, and the bytes of their
// partials.
int verify_nslice(int B, int K, int V);
size_t verify_parts_bytes(int B, int K, int V);

// Row-statistics CTAs that keep a top-p candidate list in the workspace, and
// the list's capacity per CTA (a longer candidate set is swept instead).
constexpr int kVerifyMaxCtas = 1024;
constexpr int kVerifyListCap = 8192;

size_t verify_tstats_bytes(int B, int K);
size_t verify_dstats_bytes(int B, int K);
int verify_max_chunks(int V);
size_t verify_rows_smem_bytes(int W);
bool verify_rows_plan(int V, int es, int* CL, int* W);
// The whole verification in one persistent launch (row statistics, the
// accept chains, the draws, the outputs).
cudaError_t launch_verify(const VerifyParams& p, cudaStream_t stream);

// The drafter's temperature division on its own (a test hook; verify.cu).
cudaError_t launch_temperature_divide(const float* z, const float* T, float* x, int64_t n,
                                      cudaStream_t stream);

// Noise generator on its own (api.cu / verify.cu).
cudaError_t launch_noise(const uint64_t* seed, const int64_t* pos,
                         const uint32_t* col, const uint32_t* stream_word,
                         uint32_t* word, float* u, float* g, int64_t n,
                         cudaStream_t stream);

}  // namespace dspark
