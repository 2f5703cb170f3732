// api.cu -- the C ABI declared in include/dspark.h: host-side argument
// checks, workspace carving and kernel launches. No allocation, no host
// synchronisation, no state kept between calls.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dspark.h"
#include "dspark_testing.h"
#include "kernels.h"

namespace {

constexpr size_t kAlign = 256;


size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtype(int d) { return d == DSPARK_F32 || d == DSPARK_BF16; }

int num_sms_of_current_device(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  return 0;
}

// The arrival counter and the [K][B] winner keys sit back to back, so that
// one memset clears both.
struct MarkovWs {
  size_t counter, keys, cleared, total;
  MarkovWs(int B, int K) {
    counter = 0;
    keys = 8;
    cleared = keys + static_cast<size_t>(K) * B * sizeof(unsigned long long);
    total = align_up(cleared);
  }
};

struct VerifyWs {
  size_t ctl, parts, tstats, dstats, keys, anypos, cand, total;
  VerifyWs(int B, int K, int V) {
    const int mc = dspark::verify_max_chunks(V);
    ctl = 0;
    parts = align_up(ctl + dspark::verify_ctl_bytes(B, K));
    tstats = align_up(parts + dspark::verify_parts_bytes(B, K, V));
    dstats = align_up(tstats + dspark::verify_tstats_bytes(B, K));
    keys = align_up(dstats + dspark::verify_dstats_bytes(B, K));
    anypos = align_up(keys + static_cast<size_t>(B) * mc * sizeof(unsigned long long));
    cand = align_up(anypos + static_cast<size_t>(B) * mc * sizeof(unsigned int));
    total = align_up(cand + static_cast<size_t>(dspark::kVerifyMaxCtas) *
                                dspark::kVerifyListCap * sizeof(uint2));
  }
};

bool sizes_ok(int B, int K, int V, int S) {
  return B >= 0 && B <= DSPARK_MAX_BATCH && K >= 1 && K <= DSPARK_MAX_STEPS && V >= 1 &&
         V < DSPARK_MAX_VOCAB && S >= 1;
}

}  // namespace

extern "C" {

size_t dspark_markov_workspace_bytes(int B, int K, int V, int R) {
  (void)V;
  (void)R;
  if (B < 0 || K < 1) return 0;
  return MarkovWs(B, K).total;
}

}  // extern "C"

namespace dspark {

dspark_status markov_sample_args(const void* base_logits, dspark_dtype base_dtype,
                                 const uint16_t* markov_w1, const uint16_t* markov_w2,
                                 const int32_t* anchor_tokens, const int32_t* req_state_idx,
                                 const int64_t* positions, const float* temperature,
                                 const uint64_t* seeds, const void* cache,
                                 dspark_dtype cache_dtype, const int32_t* out_tokens, int B,
                                 int K, int V, int R, int S, int C) {
  if (!sizes_ok(B, K, V, S) || R < 1) return DSPARK_ERR_INVALID_ARG;
  if (!valid_dtype(base_dtype) || !valid_dtype(cache_dtype)) return DSPARK_ERR_INVALID_ARG;
  if (R % 64 != 0 || R > 512) return DSPARK_ERR_UNSUPPORTED;
  if (B == 0) return DSPARK_OK;
  if (!base_logits || !markov_w1 || !markov_w2 || !anchor_tokens || !req_state_idx ||
      !positions || !temperature || !seeds || !out_tokens)
    return DSPARK_ERR_INVALID_ARG;
  if (cache && C < 1) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(base_logits) || !aligned16(markov_w1) || !aligned16(markov_w2) ||
      (cache && !aligned16(cache)))
    return DSPARK_ERR_ALIGNMENT;
  return DSPARK_OK;
}

}  // namespace dspark

namespace {

// dspark_markov_sample with the bounded waits' limit and the grid barrier's
// extra arrivals as parameters (see dspark_testing_markov_wait_limit).
dspark_status markov_sample_run(
    const void* base_logits, dspark_dtype base_dtype, const uint16_t* markov_w1,
    const uint16_t* markov_w2, const int32_t* anchor_tokens, const int32_t* req_state_idx,
    const int64_t* positions, const float* temperature, const uint64_t* seeds, void* cache,
    dspark_dtype cache_dtype, const int32_t* cache_row_map, int32_t* out_tokens,
    dspark_row_stats* draft_stats, int B, int K, int V, int R, int S, int C, void* workspace,
    size_t workspace_bytes, int32_t* status, dspark_stream_t stream,
    unsigned long long wait_limit_ns, unsigned int barrier_extra) {
  const dspark_status args = dspark::markov_sample_args(
      base_logits, base_dtype, markov_w1, markov_w2, anchor_tokens, req_state_idx, positions,
      temperature, seeds, cache, cache_dtype, out_tokens, B, K, V, R, S, C);
  if (args != DSPARK_OK || B == 0) return args;
  const MarkovWs ws(B, K);
  if (!workspace || workspace_bytes < ws.total || !aligned16(workspace))
    return DSPARK_ERR_WORKSPACE;
  int sms = 0;
  if (num_sms_of_current_device(&sms) != 0) return DSPARK_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned char* w = static_cast<unsigned char*>(workspace);
  dspark::MarkovStepParams p;
  p.base = base_logits;
  p.base_bf16 = base_dtype == DSPARK_BF16;
  p.w1 = markov_w1;
  p.w2 = markov_w2;
  p.anchor = anchor_tokens;
  p.rsi = req_state_idx;
  p.pos = positions;
  p.temperature = temperature;
  p.seeds = seeds;
  p.cache = cache;
  p.cache_bf16 = cache_dtype == DSPARK_BF16;
  p.row_map = cache_row_map;
  p.out_tokens = out_tokens;
  p.B = B;
  p.K = K;
  p.V = V;
  p.R = R;
  p.S = S;
  p.C = C;
  p.keys = reinterpret_cast<unsigned long long*>(w + ws.keys);
  p.counter = reinterpret_cast<unsigned int*>(w + ws.counter);
  p.status = status;
  p.draft_stats = cache != nullptr ? draft_stats : nullptr;
  p.wait_limit_ns = wait_limit_ns;
  p.barrier_extra = barrier_extra;
  if (cudaMemsetAsync(w, 0, ws.cleared, st) != cudaSuccess) return DSPARK_ERR_CUDA;
  // the statistics' mass and order-key fields accumulate from zero
  if (p.draft_stats != nullptr &&
      cudaMemsetAsync(p.draft_stats, 0, static_cast<size_t>(B) * K * sizeof(dspark_row_stats),
                      st) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  dspark::MarkovTcPlan plan;
  alignas(64) unsigned char tmap[128];
  alignas(64) unsigned char bmap[128] = {};
  const int es = base_dtype == DSPARK_BF16 ? 2 : 4;
  // TMA can stage the base logits when their rows are 16-byte multiples
  const bool base_tma = (static_cast<size_t>(V) * es) % 16 == 0;
  if (!dspark::markov_tc_plan(B, R, es, base_tma, &plan)) return DSPARK_ERR_UNSUPPORTED;
  if (dspark::markov_tc_make_tmap(tmap, markov_w2, V, R) != 0) return DSPARK_ERR_CUDA;
  if (plan.base_stage_bytes != 0 &&
      dspark::markov_tc_make_base_tmap(bmap, base_logits, es == 2, B, K, V) != 0 &&
      !dspark::markov_tc_plan(B, R, es, false, &plan))
    return DSPARK_ERR_UNSUPPORTED;
  const int grid = dspark::markov_tc_grid(V, sms);
  if (dspark::launch_markov_loop_tc(p, tmap, bmap, plan, grid, st) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

// The shortest and longest wait limits the test hook accepts.
constexpr unsigned long long kTestLimitMinNs = 100000ull;      // 0.1 ms
constexpr unsigned long long kTestLimitMaxNs = dspark::kWaitLimitNs;

}  // namespace

extern "C" {

dspark_status dspark_markov_sample(
    const void* base_logits, dspark_dtype base_dtype, const uint16_t* markov_w1,
    const uint16_t* markov_w2, const int32_t* anchor_tokens, const int32_t* req_state_idx,
    const int64_t* positions, const float* temperature, const uint64_t* seeds, void* cache,
    dspark_dtype cache_dtype, const int32_t* cache_row_map, int32_t* out_tokens,
    dspark_row_stats* draft_stats, int B, int K, int V, int R, int S, int C, void* workspace,
    size_t workspace_bytes, int32_t* status, dspark_stream_t stream) {
  return markov_sample_run(base_logits, base_dtype, markov_w1, markov_w2, anchor_tokens,
                           req_state_idx, positions, temperature, seeds, cache, cache_dtype,
                           cache_row_map, out_tokens, draft_stats, B, K, V, R, S, C, workspace,
                           workspace_bytes, status, stream, dspark::kWaitLimitNs, 0u);
}

dspark_status dspark_testing_markov_wait_limit(
    const void* base_logits, dspark_dtype base_dtype, const uint16_t* markov_w1,
    const uint16_t* markov_w2, const int32_t* anchor_tokens, const int32_t* req_state_idx,
    const int64_t* positions, const float* temperature, const uint64_t* seeds, void* cache,
    dspark_dtype cache_dtype, const int32_t* cache_row_map, int32_t* out_tokens, int B, int K,
    int V, int R, int S, int C, void* workspace, size_t workspace_bytes, int32_t* status,
    dspark_stream_t stream, uint64_t wait_limit_ns, uint32_t barrier_extra) {
  if (wait_limit_ns < kTestLimitMinNs || wait_limit_ns > kTestLimitMaxNs || barrier_extra > 1u)
    return DSPARK_ERR_INVALID_ARG;
  return markov_sample_run(base_logits, base_dtype, markov_w1, markov_w2, anchor_tokens,
                           req_state_idx, positions, temperature, seeds, cache, cache_dtype,
                           cache_row_map, out_tokens, nullptr, B, K, V, R, S, C, workspace,
                           workspace_bytes, status, stream, wait_limit_ns, barrier_extra);
}

size_t dspark_markov_topk_workspace_bytes(int B, int K, int V, int R, int topk) {
  (void)V;
  (void)R;
  if (B < 0 || K < 1 || topk < 1) return 0;
  const size_t list = align_up(static_cast<size_t>(B) * K * topk * sizeof(int32_t));
  return 2 * list;
}

dspark_status dspark_markov_sample_topk(
    const void* base_logits, dspark_dtype base_dtype, const uint16_t* markov_w1,
    const uint16_t* markov_w2, const int32_t* anchor_tokens, const int32_t* req_state_idx,
    const int64_t* positions, const float* temperature, const uint64_t* seeds, void* cache,
    dspark_dtype cache_dtype, const int32_t* cache_row_map, int32_t* out_tokens, int topk, int B,
    int K, int V, int R, int S, int C, void* workspace, size_t workspace_bytes, int32_t* status,
    dspark_stream_t stream) {
  if (!sizes_ok(B, K, V, S) || R < 1 || topk < 1) return DSPARK_ERR_INVALID_ARG;
  if (!valid_dtype(base_dtype) || !valid_dtype(cache_dtype)) return DSPARK_ERR_INVALID_ARG;
  if (R % 64 != 0 || R > 512 || topk > 65536) return DSPARK_ERR_UNSUPPORTED;
  if (B == 0) return DSPARK_OK;
  if (!base_logits || !markov_w1 || !markov_w2 || !anchor_tokens || !req_state_idx ||
      !positions || !temperature || !seeds || !out_tokens)
    return DSPARK_ERR_INVALID_ARG;
  if (cache && C < 1) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(base_logits) || !aligned16(markov_w1) || !aligned16(markov_w2) ||
      (cache && !aligned16(cache)))
    return DSPARK_ERR_ALIGNMENT;
  const size_t need = dspark_markov_topk_workspace_bytes(B, K, V, R, topk);
  if (!workspace || workspace_bytes < need || !aligned16(workspace))
    return DSPARK_ERR_WORKSPACE;
  int cluster = 0, slice = 0;
  if (!dspark::verify_rows_plan(V, base_dtype == DSPARK_BF16 ? 2 : 4, &cluster, &slice))
    return DSPARK_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned char* w = static_cast<unsigned char*>(workspace);
  dspark::TopkParams p;
  p.base = base_logits;
  p.base_bf16 = base_dtype == DSPARK_BF16;
  p.w1 = markov_w1;
  p.w2 = markov_w2;
  p.anchor = anchor_tokens;
  p.rsi = req_state_idx;
  p.pos = positions;
  p.temperature = temperature;
  p.seeds = seeds;
  p.cache = cache;
  p.cache_bf16 = cache_dtype == DSPARK_BF16;
  p.row_map = cache_row_map;
  p.out_tokens = out_tokens;
  p.B = B;
  p.K = K;
  p.V = V;
  p.R = R;
  p.S = S;
  p.C = C;
  p.k = topk;
  p.cand_idx = reinterpret_cast<int32_t*>(w);
  p.cand_val = reinterpret_cast<float*>(w + need / 2);
  p.status = status;
  if (dspark::launch_topk_rows(p, cluster, slice, st) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (dspark::launch_markov_topk_loop(p, st) != cudaSuccess) return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

size_t dspark_verify_workspace_bytes(int B, int K, int V) {
  if (B < 0 || K < 1 || V < 1) return 0;
  return VerifyWs(B, K, V).total;
}

dspark_status dspark_rejection_sample(
    const int32_t* draft_tokens, const void* draft_cache, dspark_dtype cache_dtype,
    const int32_t* cache_row_map, const dspark_row_stats* draft_stats, const void* target_logits,
    dspark_dtype target_dtype,
    const int32_t* req_state_idx, const int64_t* positions, const float* temperature,
    const float* top_p, const uint64_t* seeds, int32_t* out_tokens, int32_t* num_accepted,
    int B, int K, int V, int S, int C, void* workspace, size_t workspace_bytes,
    int32_t* status, dspark_stream_t stream) {
  if (!sizes_ok(B, K, V, S)) return DSPARK_ERR_INVALID_ARG;
  if (!valid_dtype(cache_dtype) || !valid_dtype(target_dtype)) return DSPARK_ERR_INVALID_ARG;
  if (B == 0) return DSPARK_OK;
  if (!draft_tokens || !target_logits || !req_state_idx || !positions || !temperature ||
      !top_p || !seeds || !out_tokens || !num_accepted)
    return DSPARK_ERR_INVALID_ARG;
  if (draft_cache && C < 1) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(target_logits) || (draft_cache && !aligned16(draft_cache)))
    return DSPARK_ERR_ALIGNMENT;
  const VerifyWs ws(B, K, V);
  if (!workspace || workspace_bytes < ws.total || !aligned16(workspace))
    return DSPARK_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned char* w = static_cast<unsigned char*>(workspace);
  dspark::VerifyParams p;
  p.draft = draft_tokens;
  p.cache = draft_cache;
  p.cache_bf16 = cache_dtype == DSPARK_BF16;
  p.row_map = cache_row_map;
  p.draft_stats = draft_stats;
  p.target = target_logits;
  p.target_bf16 = target_dtype == DSPARK_BF16;
  p.rsi = req_state_idx;
  p.pos = positions;
  p.temperature = temperature;
  p.top_p = top_p;
  p.seeds = seeds;
  p.out_tokens = out_tokens;
  p.num_accepted = num_accepted;
  p.B = B;
  p.K = K;
  p.V = V;
  p.S = S;
  p.C = C;
  p.ctl = reinterpret_cast<unsigned int*>(w + ws.ctl);
  p.parts = w + ws.parts;
  p.nslice = dspark::verify_nslice(B, K, V);
  p.tstats = w + ws.tstats;
  p.dstats = w + ws.dstats;
  p.keys = reinterpret_cast<unsigned long long*>(w + ws.keys);
  p.anypos = reinterpret_cast<unsigned int*>(w + ws.anypos);
  p.cand = reinterpret_cast<uint2*>(w + ws.cand);
  p.kstride = dspark::verify_max_chunks(V);
  p.stats_items = draft_stats != nullptr && B <= dspark::kRowStatsMaxBatch;
  p.ndraw = 1;  // chosen at launch from the grid
  p.status = status;
  // the progress counters start from zero
  if (cudaMemsetAsync(w + ws.ctl, 0, dspark::verify_ctl_bytes(B, K), st) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (dspark::launch_verify(p, st) != cudaSuccess) return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

dspark_status dspark_noise(const uint64_t* seed, const int64_t* pos, const uint32_t* col,
                           const uint32_t* stream, uint32_t* word, float* u, float* g,
                           int64_t n, dspark_stream_t stream_handle) {
  if (n < 0) return DSPARK_ERR_INVALID_ARG;
  if (n == 0) return DSPARK_OK;
  if (!seed || !pos || !col || !stream) return DSPARK_ERR_INVALID_ARG;
  if (dspark::launch_noise(seed, pos, col, stream, word, u, g, n,
                           reinterpret_cast<cudaStream_t>(stream_handle)) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

dspark_status dspark_testing_temperature_divide(const float* z, const float* T, float* x,
                                                int64_t n, dspark_stream_t stream) {
  if (n < 0) return DSPARK_ERR_INVALID_ARG;
  if (n == 0) return DSPARK_OK;
  if (!z || !T || !x) return DSPARK_ERR_INVALID_ARG;
  if (dspark::launch_temperature_divide(z, T, x, n, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

const char* dspark_status_string(int status) {
  switch (status) {
    case DSPARK_OK:
      return "ok";
    case DSPARK_ERR_INVALID_ARG:
      return "invalid argument";
    case DSPARK_ERR_UNSUPPORTED:
      return "unsupported configuration";
    case DSPARK_ERR_CUDA:
      return "CUDA error";
    case DSPARK_ERR_TIMEOUT:
      return "device wait timed out";
    case DSPARK_ERR_BOUNDS:
      return "token, slot or cache row out of range";
    case DSPARK_ERR_WORKSPACE:
      return "workspace missing or too small";
    case DSPARK_ERR_ALIGNMENT:
      return "pointer not 16-byte aligned";
    case DSPARK_ERR_SCRATCH_LIMIT:
      return "sizes need more scratch than the library's fixed array";
    default:
      return "unknown status";
  }
}

int dspark_version(void) { return 100; }

}  // extern "C"
