/*
 * dspark.h -- C ABI of the DSpark Markov drafting step and rejection-sampling
 * verifier for one NVIDIA GB300 (sm_103a).
 *
 * The operations follow these pages (cited by title and section):
 *   - "DSparkSpeculator" API page (vllm/v1/worker/gpu/spec_decode/dspark/
 *     speculator.py): _sample_markov_chain (the K sequential steps: Markov
 *     embedding of the previous token, Markov bias, bias add, sampling) and
 *     _sample_logits (gumbel_sample with temperature, per-request seeds, the
 *     position before the sampled token, the draft-logits cache and its row
 *     mapping).
 *   - vLLM PR #65007 "vocab-parallel DSpark Markov sampling", Part 1 (per-step
 *     list: Gumbel-noised argmax over 1024-column blocks, the first NaN block
 *     wins, otherwise the first maximum) and Part 2 (temperature, exact top-p
 *     by logit then token id with 64-bit fixed-point masses, and the
 *     rejection sampler).
 *   - vLLM PR #63554 "batch-sharded draft logits cache" (cache rows addressed
 *     through a row mapping; greedy rows never read the cache).
 *
 * Conventions shared by every entry point
 *   Memory.  Every pointer argument is DEVICE memory owned by the caller,
 *            except `status`, which may also be pinned (mapped) host memory.
 *            The library allocates nothing and keeps no state between calls;
 *            scratch space is the caller's `workspace` (one entry point,
 *            dspark_markov_sample_static, uses a fixed array inside the
 *            library instead: see there).
 *   Layout.  Row-major and contiguous. fp32 tensors are IEEE binary32; bf16
 *            tensors are passed as uint16 bit patterns.
 *   Streams. All work is enqueued on `stream` (a cudaStream_t; NULL = the
 *            legacy default stream). Calls return before the work finishes.
 *            Two calls in flight at once must not share a workspace.
 *   Errors.  Argument errors (null pointers, sizes, dtypes, alignment, a
 *            workspace that is too small) are detected on the host before
 *            anything is launched: a negative dspark_status is returned and
 *            nothing runs. A failed launch returns DSPARK_ERR_CUDA. Errors
 *            found on the device (a token, slot or cache row out of range; a
 *            bounded wait that ran out) never fault: the kernel stores the
 *            first error code into *status (if `status` is not NULL, with an
 *            atomic compare-and-swap from 0) and the affected request is
 *            treated as padding. The caller reads *status after the stream
 *            has been synchronised; it should be 0 before the call.
 *   Noise.   Random draws use the Philox4x32-10 counter-based generator
 *            (Salmon, Moraes, Dror, Shaw, SC'11): key = (seed low word, seed
 *            high word), counter = (column / 4, position low word, position
 *            high word, stream), output word = column mod 4; u = ((w >> 9) +
 *            1/2) * 2^-23; Gumbel g = -log(-log u). Streams: 2^30 for draft
 *            noise (the pages' draft-noise salt), 0 for the verifier's
 *            categorical draws, 2^29 for its accept uniforms.
 */
#ifndef DSPARK_H_
#define DSPARK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* dspark_stream_t;

typedef enum {
  DSPARK_F32 = 0,  /* IEEE binary32                     */
  DSPARK_BF16 = 1  /* bfloat16, passed as uint16 bits    */
} dspark_dtype;

typedef enum {
  DSPARK_OK = 0,
  DSPARK_ERR_INVALID_ARG = -1, /* null pointer, bad size or dtype          */
  DSPARK_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. R % 64)  */
  DSPARK_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed     */
  DSPARK_ERR_TIMEOUT = -4,     /* device: a bounded wait ran out           */
  DSPARK_ERR_BOUNDS = -5,      /* device: token, slot or row out of range  */
  DSPARK_ERR_WORKSPACE = -6,   /* workspace null or smaller than required  */
  DSPARK_ERR_ALIGNMENT = -7,   /* a pointer is not 16-byte aligned         */
  DSPARK_ERR_SCRATCH_LIMIT = -8 /* sizes need more scratch than the fixed
                                   array of dspark_markov_sample_static    */
} dspark_status;

/* Statistics of one draft-logits cache row (one request, one draft step),
 * recorded by dspark_markov_sample while it writes the row:
 *   m     the maximum of the row's stored values (NaN read as -inf; for a
 *         bf16 cache the stored bf16 value); exact, whatever order it is
 *         taken in. NaN: not recorded.
 *   mass  the row's exp-mass sum_v exp(x_v - m) in 64-bit fixed point
 *         (2^40 per unit): each CTA of the loop sums its part of the row in
 *         fp32 (a fixed order) and adds it, rescaled to m and rounded to an
 *         integer, with an integer atomic, so the total does not depend on
 *         the order of the additions. 0 for a row with no value above -inf.
 * dspark_rejection_sample uses them in place of reading the row. */
typedef struct {
  float m;
  uint32_t scratch;  /* used by dspark_markov_sample while it runs */
  uint64_t mass;
} dspark_row_stats;

/* Limits checked on the host. */
#define DSPARK_MAX_VOCAB (1 << 22)  /* token ids fit 22 bits; V * 2^40 < 2^63 */
#define DSPARK_MAX_BATCH 256
#define DSPARK_MAX_STEPS 16

/* ------------------------------------------------------------------------
 * dspark_markov_sample -- the drafter's K-step Markov sampling loop.
 * (DSparkSpeculator page, _sample_markov_chain / _sample_logits; PR #65007
 *  Part 1, per-step list.)
 *
 * For every request b with slot s = req_state_idx[b] >= 0, starting from
 * prev = anchor_tokens[b], for i = 0..K-1:
 *   e      = markov_w1[prev, :]                        (Markov embedding)
 *   bias_v = sum_r markov_w2[v, r] * e[r]              (fp32 accumulation)
 *   z_v    = base_logits[b, i, v] + bias_v             (fp32)
 *   T = temperature[s] > 0:  x_v = z_v / T (IEEE division, correctly
 *       rounded; T = 1 leaves z_v as it is), y_v = x_v + g_v with g the
 *       Gumbel noise of (seeds[s], positions[b] + i - 1, v, draft stream)
 *   otherwise (greedy):      x_v = y_v = z_v
 *   out_tokens[b, i] = lowest-index NaN of y if any, else the lowest index of
 *       max(y) (the "first NaN block, else first maximum" rule over
 *       1024-column blocks, which does not depend on the blocking);
 *   cache[row, i, :] = x (fp32, or bf16 rounded to nearest even), row =
 *       cache_row_map ? cache_row_map[s] : s;
 *   prev = out_tokens[b, i].
 * Requests with req_state_idx[b] < 0 are padding: out_tokens[b, :] = -1 and
 * nothing else is read or written for them.
 *
 * Arguments
 *   base_logits   [B, K, V] base_dtype (fp32 or bf16)
 *   markov_w1     [V, R] bf16    Markov embedding table (indexed by token)
 *   markov_w2     [V, R] bf16    Markov bias projection
 *   anchor_tokens [B] int32      first `prev` of each request, in [0, V)
 *   req_state_idx [B] int32      slot in [0, S), or < 0 for padding
 *   positions     [B] int64      position P0 of each request's first draft token
 *   temperature   [S] fp32       per slot; <= 0 (or NaN) = greedy
 *   seeds         [S] uint64     per slot
 *   cache         [C, K, V] cache_dtype, or NULL for no cache write
 *   cache_row_map [S] int32 in [0, C), or NULL for row = slot
 *   out_tokens    [B, K] int32   (written)
 *   draft_stats   [B, K] dspark_row_stats, or NULL: if given (and cache is
 *                 not NULL), the maximum and exp-mass of every cache row the
 *                 call writes, so that dspark_rejection_sample need not read
 *                 the row (padding requests: zero; B > 32: m = NaN, "not
 *                 recorded"). No counterpart in the pages: the loop has every
 *                 value of the row at hand.
 *   B in [0, 256], K in [1, 16], V in [1, 2^22), R a multiple of 64 up to
 *   512, S >= 1, C >= 1 if cache != NULL.
 *   workspace     device scratch of at least dspark_markov_workspace_bytes()
 *                 bytes, 256-byte aligned. Its contents need no
 *                 initialisation; the call leaves it ready for the next call.
 *   status        see the conventions above; may be NULL.
 * Alignment: base_logits, markov_w2 and cache must be 16-byte aligned.
 * ------------------------------------------------------------------------ */
size_t dspark_markov_workspace_bytes(int B, int K, int V, int R);

dspark_status dspark_markov_sample(
    const void* base_logits, dspark_dtype base_dtype,
    const uint16_t* markov_w1, const uint16_t* markov_w2,
    const int32_t* anchor_tokens, const int32_t* req_state_idx,
    const int64_t* positions, const float* temperature, const uint64_t* seeds,
    void* cache, dspark_dtype cache_dtype, const int32_t* cache_row_map,
    int32_t* out_tokens, dspark_row_stats* draft_stats, int B, int K, int V,
    int R, int S, int C, void* workspace, size_t workspace_bytes,
    int32_t* status, dspark_stream_t stream);

/* ------------------------------------------------------------------------
 * dspark_markov_sample_topk -- the top-k variant of the Markov loop.
 * ("DSparkSpeculator" page, _sample_sequential_topk.)
 *
 * As dspark_markov_sample, except that for each request and draft step i the
 * Markov bias is applied only to the `topk` candidates of that step -- the
 * topk largest base_logits[b, i, :] by value, ties to the lower token id,
 * NaN above every number, -0 equal to +0 (topk >= V: every column) -- and
 * every other column of z is -inf:
 *   z_v = base_logits[b, i, v] + bias_v   for the candidates, -inf otherwise;
 * temperature, Gumbel noise, the winner rule and the cache store are then the
 * dense ones (so cache[row, i, :] is -inf outside the candidates, and
 * dspark_rejection_sample consumes the truncated distribution unchanged).
 * Only the candidates' markov_w2 rows are read.
 *
 * Arguments as for dspark_markov_sample, plus
 *   topk          candidates per request and step, in [1, 65536]
 *   workspace     at least dspark_markov_topk_workspace_bytes() bytes,
 *                 256-byte aligned (the candidate lists); no initialisation.
 * Alignment: base_logits, markov_w2 and cache must be 16-byte aligned.
 * ------------------------------------------------------------------------ */
size_t dspark_markov_topk_workspace_bytes(int B, int K, int V, int R, int topk);

dspark_status dspark_markov_sample_topk(
    const void* base_logits, dspark_dtype base_dtype,
    const uint16_t* markov_w1, const uint16_t* markov_w2,
    const int32_t* anchor_tokens, const int32_t* req_state_idx,
    const int64_t* positions, const float* temperature, const uint64_t* seeds,
    void* cache, dspark_dtype cache_dtype, const int32_t* cache_row_map,
    int32_t* out_tokens, int topk, int B, int K, int V, int R, int S, int C,
    void* workspace, size_t workspace_bytes, int32_t* status,
    dspark_stream_t stream);

/* ------------------------------------------------------------------------
 * dspark_markov_sample_static -- dspark_markov_sample without a workspace
 * argument: the same computation, arguments and results, with the scratch
 * kept in a fixed device array compiled into the library. The pages describe
 * no such variant; it exists for callers that may not allocate device memory
 * at all: a plug-in run by an inference engine that hands out every byte of
 * device memory itself, a real-time decode loop that must not take the
 * latency and implicit synchronisation of cudaMalloc, or a foreign-language
 * host that can pass pointers but has no CUDA allocator of its own. This call
 * makes no cudaMalloc or cudaFree and calls no allocating library.
 *
 * Limit.    The array holds DSPARK_STATIC_SCRATCH_BYTES bytes; every GPU that
 *           loads the library holds it until the process exits. A call whose
 *           dspark_markov_workspace_bytes(B, K, V, R) exceeds that is rejected
 *           on the host with DSPARK_ERR_SCRATCH_LIMIT before anything runs.
 *           32 KiB holds B * K <= 4095: every batch up to 256 requests with up
 *           to 15 draft steps, or up to 255 requests with 16.
 * Checks.   The argument checks of dspark_markov_sample come first, in its
 *           order and with its codes; the scratch limit after them.
 * Set-up.   Every call looks up the array's address on the current device
 *           (cudaGetSymbolAddress, with that device current; a failure
 *           returns DSPARK_ERR_CUDA), so a device reset that reloads the
 *           library's module elsewhere leaves no stale address behind. The
 *           first call on a device may load the module: make it before any
 *           stream capture begins.
 * Sharing.  Every call on a device uses the same array, which keeps what the
 *           last call left there. The part that must start at zero (the
 *           kernel's arrival counter) is cleared on `stream` by each call;
 *           the rest is written before it is read. Calls whose work overlaps
 *           on the GPU (other streams, other host threads) race on the array
 *           and give wrong tokens: order them on one stream or with events.
 * ------------------------------------------------------------------------ */
#define DSPARK_STATIC_SCRATCH_BYTES (32u << 10)

dspark_status dspark_markov_sample_static(
    const void* base_logits, dspark_dtype base_dtype,
    const uint16_t* markov_w1, const uint16_t* markov_w2,
    const int32_t* anchor_tokens, const int32_t* req_state_idx,
    const int64_t* positions, const float* temperature, const uint64_t* seeds,
    void* cache, dspark_dtype cache_dtype, const int32_t* cache_row_map,
    int32_t* out_tokens, dspark_row_stats* draft_stats, int B, int K, int V,
    int R, int S, int C, int32_t* status, dspark_stream_t stream);

/* ------------------------------------------------------------------------
 * dspark_rejection_sample -- probabilistic rejection-sampling verification.
 * (PR #65007 Part 2: temperature, exact top-p, the rejection sampler;
 *  PR #63554: greedy rows compare with the target argmax.)
 *
 * For every request b with slot s >= 0, T = temperature[s]:
 *   target row k (k = 0..K): xt = target[b,k,:] / T, NaN read as -inf;
 *     m = max xt; e_v = exp(xt_v - m) (fp32); f_v = rint(e_v * 2^40) (uint64);
 *     if top_p[s] < 1 keep the shortest prefix of the (xt desc, id asc) order
 *     with (sum of f over the prefix) * 2^32 >= rint(top_p * 2^32) * (sum of
 *     all f), and D = fp32(sum of kept f) * 2^-40; else keep all, and D =
 *     the fp32 sum of e_v in a fixed order (per-slice running sums, each
 *     rescaled to the slice maximum as it grows, combined in slice order:
 *     one pass over the row, the same bits every run; it differs from
 *     fp32(sum of f) * 2^-40 by fp32 rounding only). p_v = e_v / D on the
 *     kept set, 0 elsewhere. A row with no value above -inf is one-hot at 0.
 *   draft row k (k < K): q = exp(c_v - m) / D of c = cache[row, k, :] with
 *     no temperature and no top-p (the cache holds scaled logits), D the
 *     fp32 sum as for a target row kept whole (or, with draft_stats, from the
 *     recorded fixed-point mass); a row with no value above -inf gives q = 0.
 *   for k = 0..K-1, d = draft_tokens[b, k]:
 *     d = -1: emit a draw from p_k and stop;
 *     u = uniform(seeds[s], positions[b] + k - 1, column 0, accept stream);
 *     accept iff fp32(u * q_k(d)) < p_k(d)  (probability min(1, p/q));
 *     on reject emit the Gumbel-max draw (target stream, same position) from
 *     r = max(0, p_k - q_k) (from p_k if r is all zero) and stop.
 *   all K accepted: emit a draw from p_K (position positions[b] + K - 1).
 *   A "draw from w" is argmax_v fp32(log w_v) + g_v, same winner rule as
 *   the drafter.
 *   Greedy slots (T <= 0 or NaN): accept d iff d equals the winner of the
 *   raw target row k; emit that winner on mismatch or d = -1; the bonus is
 *   the winner of row K. The cache is not read.
 * Outputs: out_tokens[b, :] = the accepted drafts, then the one emitted
 * token, then -1; num_accepted[b] = number of accepted drafts. Padding
 * requests (slot < 0) get all -1 and 0.
 *
 * Arguments
 *   draft_tokens  [B, K] int32 in [0, V) or -1
 *   draft_cache   [C, K, V] cache_dtype (may be NULL if every slot is greedy)
 *   cache_row_map [S] int32 or NULL (row = slot)
 *   draft_stats   [B, K] dspark_row_stats or NULL: the statistics that
 *                 dspark_markov_sample recorded for these cache rows; a draft
 *                 row with recorded statistics (m not NaN) is then not read
 *                 for its distribution: q = exp(x - m) / (fp32(mass) 2^-40),
 *                 and only the row a residual draw needs is read. They must
 *                 describe the cache passed here.
 *   target_logits [B, K+1, V] target_dtype
 *   req_state_idx [B], positions [B], temperature [S], top_p [S] fp32,
 *   seeds [S] as for dspark_markov_sample
 *   out_tokens    [B, K+1] int32, num_accepted [B] int32 (written)
 *   workspace     at least dspark_verify_workspace_bytes() bytes (per-row
 *                 and per-request statistics plus a fixed 64 MB area of
 *                 top-p candidate lists); no initial contents required
 * Alignment: draft_cache and target_logits must be 16-byte aligned.
 * ------------------------------------------------------------------------ */
size_t dspark_verify_workspace_bytes(int B, int K, int V);

dspark_status dspark_rejection_sample(
    const int32_t* draft_tokens, const void* draft_cache,
    dspark_dtype cache_dtype, const int32_t* cache_row_map,
    const dspark_row_stats* draft_stats, const void* target_logits,
    dspark_dtype target_dtype,
    const int32_t* req_state_idx, const int64_t* positions,
    const float* temperature, const float* top_p, const uint64_t* seeds,
    int32_t* out_tokens, int32_t* num_accepted, int B, int K, int V, int S,
    int C, void* workspace, size_t workspace_bytes, int32_t* status,
    dspark_stream_t stream);

/* ------------------------------------------------------------------------
 * dspark_noise -- the device noise generator on its own, for checking it
 * against other implementations: for i < n, word[i] = Philox output of
 * (seed[i], pos[i], col[i], stream[i]) as described above, u[i] its uniform
 * and g[i] its Gumbel variate. Any of word, u, g may be NULL. Device arrays.
 * ------------------------------------------------------------------------ */
dspark_status dspark_noise(const uint64_t* seed, const int64_t* pos,
                           const uint32_t* col, const uint32_t* stream,
                           uint32_t* word, float* u, float* g, int64_t n,
                           dspark_stream_t stream_handle);

/* Human-readable name of a status code (static storage; never NULL). */
const char* dspark_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int dspark_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H_ */
