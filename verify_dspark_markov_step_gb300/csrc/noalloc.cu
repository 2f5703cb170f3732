// noalloc.cu -- dspark_markov_sample_static: the Markov sampling loop for
// callers that may not allocate device memory (an engine plug-in that is
// handed all of its memory, a latency-bound loop that cannot afford
// cudaMalloc, a host with no CUDA allocator). Its scratch is a fixed array
// in the library's device image instead of a caller-supplied workspace; the
// work itself is dspark_markov_sample's, unchanged.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dspark.h"
#include "kernels.h"

// The scratch: one per GPU that loads the library, alive until the process
// exits. Host code must not hand this name to a kernel: on the host it only
// stands for the symbol, and its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_markov_scratch[DSPARK_STATIC_SCRATCH_BYTES];

extern "C" dspark_status dspark_markov_sample_static(
    const void* base_logits, dspark_dtype base_dtype, const uint16_t* markov_w1,
    const uint16_t* markov_w2, const int32_t* anchor_tokens, const int32_t* req_state_idx,
    const int64_t* positions, const float* temperature, const uint64_t* seeds, void* cache,
    dspark_dtype cache_dtype, const int32_t* cache_row_map, int32_t* out_tokens,
    dspark_row_stats* draft_stats, int B, int K, int V, int R, int S, int C, int32_t* status,
    dspark_stream_t stream) {
  // the argument checks of dspark_markov_sample, in its order, come first;
  // then the scratch limit; both before anything touches the device
  const dspark_status args = dspark::markov_sample_args(
      base_logits, base_dtype, markov_w1, markov_w2, anchor_tokens, req_state_idx, positions,
      temperature, seeds, cache, cache_dtype, out_tokens, B, K, V, R, S, C);
  if (args != DSPARK_OK || B == 0) return args;
  if (dspark_markov_workspace_bytes(B, K, V, R) > DSPARK_STATIC_SCRATCH_BYTES)
    return DSPARK_ERR_SCRATCH_LIMIT;
  // The array's address on the current device, looked up on every call (a
  // host-side table lookup once the module is loaded): a cached address would
  // go stale if the device were reset and the module loaded again elsewhere.
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, g_markov_scratch) != cudaSuccess || scratch == nullptr)
    return DSPARK_ERR_CUDA;
  // dspark_markov_sample clears the arrival counter on `stream` itself and
  // writes every other scratch word before reading it, so what an earlier
  // call left in the array does not matter.
  return dspark_markov_sample(base_logits, base_dtype, markov_w1, markov_w2, anchor_tokens,
                              req_state_idx, positions, temperature, seeds, cache, cache_dtype,
                              cache_row_map, out_tokens, draft_stats, B, K, V, R, S, C, scratch,
                              DSPARK_STATIC_SCRATCH_BYTES, status, stream);
}
