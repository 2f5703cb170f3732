/*
 * dspark_testing.h -- a test hook of the dspark library, outside the API
 * that include/dspark.h describes. The pages have no counterpart: it exists so
 * that a test can make the Markov loop's bounded waits run out on purpose and
 * check that the library then reports the failure instead of hanging.
 */
#ifndef DSPARK_TESTING_H_
#define DSPARK_TESTING_H_

#include "dspark.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------------
 * dspark_testing_markov_wait_limit -- dspark_markov_sample (without the
 * draft_stats output) with two knobs of its bounded waits:
 *   wait_limit_ns  how long every wait of the launch (each mbarrier wait of
 *                  its warps, and the grid barrier between draft steps) may
 *                  take before it gives up, in [1e5, 2e9] ns;
 *                  dspark_markov_sample uses 2e9 (2 s).
 *   barrier_extra  0 or 1: arrivals the grid barrier waits for beyond the
 *                  ones the grid makes. With 1 the barrier after the first
 *                  draft step can never complete, so every CTA's wait runs
 *                  out after wait_limit_ns.
 * A wait that runs out stores DSPARK_ERR_TIMEOUT into *status (if it was 0);
 * the CTA then stops issuing work, lets every copy and tensor-core operation
 * it started complete, frees its tensor memory and exits, so the launch ends
 * within a few wait limits and leaves the device usable. out_tokens and the
 * cache are then unspecified; the workspace needs nothing before the next
 * call. Other arguments, their checks and their errors are those of
 * dspark_markov_sample; a limit outside the range or barrier_extra > 1 gives
 * DSPARK_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------ */
dspark_status dspark_testing_markov_wait_limit(
    const void* base_logits, dspark_dtype base_dtype,
    const uint16_t* markov_w1, const uint16_t* markov_w2,
    const int32_t* anchor_tokens, const int32_t* req_state_idx,
    const int64_t* positions, const float* temperature, const uint64_t* seeds,
    void* cache, dspark_dtype cache_dtype, const int32_t* cache_row_map,
    int32_t* out_tokens, int B, int K, int V, int R, int S, int C,
    void* workspace, size_t workspace_bytes, int32_t* status,
    dspark_stream_t stream, uint64_t wait_limit_ns, uint32_t barrier_extra);

/* ------------------------------------------------------------------------
 * dspark_testing_temperature_divide -- the Markov loop's temperature step on
 * its own, for checking it against IEEE division: for i < n,
 * x[i] = z[i] / T[i] computed exactly as the loop's epilogue computes it
 * (an FMA-corrected product with the correctly rounded reciprocal of T where
 * every intermediate stays normal, else the IEEE division), which must be
 * the correctly rounded quotient. T[i] > 0. Device arrays; returns
 * DSPARK_ERR_INVALID_ARG for n < 0 or a null pointer (n > 0).
 * ------------------------------------------------------------------------ */
dspark_status dspark_testing_temperature_divide(const float* z, const float* T, float* x,
                                                int64_t n, dspark_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_TESTING_H_ */
