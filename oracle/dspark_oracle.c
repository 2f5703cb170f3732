/*
 * dspark_oracle.c -- plain, slow, single-threaded CPU oracle for the DSpark
 * Markov drafting step and the probabilistic rejection-sampling verifier.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load this file. The product path never calls it, and it
 * shares no code, header, table or constant generator with the CUDA library.
 *
 * Sources (web pages, cited by title and section):
 *   [DSP]  "DSparkSpeculator" API page (vllm/v1/worker/gpu/spec_decode/dspark/
 *          speculator.py): _sample_markov_chain, _sample_logits.
 *   [TPM]  vLLM PR #65007 "vocab-parallel DSpark Markov sampling",
 *          Part 1 (per-step list, items 1-4) and Part 2 (top-p and the
 *          rejection sampler).
 *   [BSH]  vLLM PR #63554 "batch-sharded draft logits cache" (row mapping,
 *          greedy rows never read cached draft logits).
 *   [PHX]  J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel random numbers:
 *          as easy as 1, 2, 3", SC'11 -- the Philox4x32-10 generator.
 *
 * Where the pages leave a step open this file takes one reading; each reading
 * is marked READING and is the same one the CUDA library implements.
 *
 * Arithmetic precision: IEEE binary32 with round-to-nearest-even wherever the
 * method's own arithmetic is fp32 (bias add, temperature division, noise add,
 * ratio test); fp64 where the oracle evaluates a transcendental (log, exp) or a
 * dot product, rounded once to fp32. Compile with -ffp-contract=off so that no
 * a*b+c is fused.
 *
 * Parity pins: see tests/test_oracle_pins.py (Philox against a library
 * Philox, chi-square of Gumbel-max against softmax, brute-force top-p, the
 * Sum(min(p,q)) acceptance identity, chi-square of the verifier's first token
 * against the target distribution, argmax tie and NaN rules).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Requests are independent, so the batch entry points can run them on
 * several host threads: built with -fopenmp the two batch loops below are
 * OpenMP loops over requests (one request per thread at a time, each thread
 * with its own scratch); built without it they are plain loops. Nothing
 * inside a request changes. */
#ifdef _OPENMP
#include <omp.h>
#define ORC_OMP(x) _Pragma(#x)
#else
#define ORC_OMP(x)
#endif

/* ------------------------------------------------------------------------ */
/* Error codes of this oracle (its own; unrelated to the library's).         */
/* ------------------------------------------------------------------------ */
#define ORC_OK 0
#define ORC_EINVAL 1   /* bad size or pointer                          */
#define ORC_EBOUNDS 2  /* token, slot or cache row out of range         */
#define ORC_ENOMEM 3

/* Noise streams. [DSP] _sample_logits passes is_drafting=True; gumbel.py
 * salts draft noise with _DRAFT_NOISE_SALT = 1 << 30 ([TPM] review thread on
 * module constants). READING: the verifier's own draws use two other stream
 * words, 0 for categorical draws from target-side distributions and 1 << 29
 * for the accept uniforms. */
#define ORC_STREAM_DRAFT (1u << 30)
#define ORC_STREAM_TARGET 0u
#define ORC_STREAM_ACCEPT (1u << 29)

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 [PHX]: a 4x32-bit counter, a 2x32-bit key, 10 rounds. Each   */
/* round multiplies counter words 0 and 2 by the two round multipliers,      */
/* swaps the halves and xors in the key; the key is bumped by the two Weyl    */
/* constants between rounds.                                                 */
/* ------------------------------------------------------------------------ */
static void philox4x32_10(const uint32_t ctr_in[4], uint32_t k0, uint32_t k1,
                          uint32_t out[4]) {
  const uint32_t mult0 = 0xD2511F53u, mult1 = 0xCD9E8D57u;
  const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
  uint32_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
  for (int round = 0; round < 10; round++) {
    if (round > 0) {
      k0 += weyl0;
      k1 += weyl1;
    }
    uint64_t prod0 = (uint64_t)mult0 * (uint64_t)x0;
    uint64_t prod1 = (uint64_t)mult1 * (uint64_t)x2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t y0 = hi1 ^ x1 ^ k0;
    uint32_t y1 = lo1;
    uint32_t y2 = hi0 ^ x3 ^ k1;
    uint32_t y3 = lo0;
    x0 = y0;
    x1 = y1;
    x2 = y2;
    x3 = y3;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

/* READING (the pages name the noise keys -- request seed, position P-1,
 * column, draft salt -- but no generator): key = (seed low word, seed high
 * word); counter = (column / 4, position low word, position high word,
 * stream); the column's word is output (column mod 4). */
static uint32_t noise_word(uint64_t seed, int64_t pos, uint32_t col,
                           uint32_t stream) {
  uint64_t upos = (uint64_t)pos;
  uint32_t ctr[4] = {col >> 2, (uint32_t)upos, (uint32_t)(upos >> 32), stream};
  uint32_t out[4];
  philox4x32_10(ctr, (uint32_t)seed, (uint32_t)(seed >> 32), out);
  return out[col & 3u];
}

/* READING: u = (top 23 bits + 1/2) * 2^-23, an exact fp32 value in (0, 1). */
static float uniform_from_word(uint32_t w) {
  double u = ((double)(w >> 9) + 0.5) * 0x1p-23;
  return (float)u; /* exact: at most 24 significant bits */
}

/* Standard Gumbel variate g = -log(-log u), evaluated in fp64 and rounded
 * once to fp32. */
static float gumbel_from_uniform(float u) {
  double g = -log(-log((double)u));
  return (float)g;
}

static float bf16_to_f32(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, 4);
  return f;
}

/* fp32 -> bf16, round to nearest even; NaN stays NaN (quiet, sign kept). */
static uint16_t f32_to_bf16(float f) {
  uint32_t bits;
  memcpy(&bits, &f, 4);
  if (isnan(f)) return (uint16_t)((bits >> 16) | 0x0040u);
  uint32_t lsb = (bits >> 16) & 1u;
  bits += 0x7FFFu + lsb;
  return (uint16_t)(bits >> 16);
}

static float load_elem(const void* p, int is_bf16, int64_t idx) {
  if (is_bf16) return bf16_to_f32(((const uint16_t*)p)[idx]);
  return ((const float*)p)[idx];
}

/* ------------------------------------------------------------------------ */
/* The block-argmax rule ([TPM] Part 1, item 4: the first NaN block wins,     */
/* otherwise the first maximum; blocks are 1024 columns and the in-block     */
/* argmax keeps the lowest index). Over contiguous blocks scanned in order   */
/* this is the same as: the lowest-index NaN if any, else the lowest index    */
/* holding the maximum. -0 and +0 compare equal. The block form is written   */
/* out literally here; the pin tests compare it with the flat form.          */
/* ------------------------------------------------------------------------ */
#define ORC_BLOCK 1024

typedef struct {
  int64_t idx;   /* winning column                                         */
  double gap;    /* winner minus the best other value; +inf if NaN wins     */
} orc_winner;

static orc_winner block_argmax(const float* y, int64_t n) {
  orc_winner w;
  w.idx = 0;
  w.gap = INFINITY;
  if (n <= 0) {
    w.idx = -1;
    return w;
  }
  /* Per block: (is_nan, max value, index of its first occurrence). */
  int64_t best_blk_idx = -1;
  int best_is_nan = 0;
  float best_val = 0.0f;
  for (int64_t b0 = 0; b0 < n; b0 += ORC_BLOCK) {
    int64_t b1 = b0 + ORC_BLOCK < n ? b0 + ORC_BLOCK : n;
    int blk_nan = 0;
    int64_t blk_idx = b0;
    float blk_val = y[b0];
    if (isnan(blk_val)) blk_nan = 1;
    for (int64_t v = b0 + 1; v < b1 && !blk_nan; v++) {
      if (isnan(y[v])) {
        blk_nan = 1;
        blk_idx = v;
        blk_val = y[v];
      } else if (y[v] > blk_val) {
        blk_val = y[v];
        blk_idx = v;
      }
    }
    if (best_blk_idx < 0) {
      best_blk_idx = blk_idx;
      best_is_nan = blk_nan;
      best_val = blk_val;
    } else if (!best_is_nan) {
      if (blk_nan || blk_val > best_val) {
        best_blk_idx = blk_idx;
        best_is_nan = blk_nan;
        best_val = blk_val;
      }
    }
  }
  w.idx = best_blk_idx;
  if (best_is_nan) {
    w.gap = INFINITY;
    return w;
  }
  double second = -INFINITY;
  int have_second = 0;
  for (int64_t v = 0; v < n; v++) {
    if (v == w.idx) continue;
    if (!have_second || (double)y[v] > second) {
      second = (double)y[v];
      have_second = 1;
    }
  }
  if (!have_second)
    w.gap = INFINITY;
  else if (second == (double)best_val)
    w.gap = 0.0; /* a tie, including two infinities of one sign */
  else
    w.gap = (double)best_val - second;
  return w;
}

/* ======================================================================== */
/* Part 1: the K-step Markov drafting loop ([DSP] _sample_markov_chain).     */
/* ======================================================================== */

/* One Markov step for one request: bias from the previous token, bias add,
 * temperature, Gumbel noise, block argmax. Writes the temperature-scaled
 * logits x to x_out[V] (what the draft-logits cache stores).
 *
 *   e_r    = markov_w1[prev, r]                         (markov_embed)
 *   bias_v = fp32( sum_r fp64(w2[v,r]) * fp64(e_r) )     (markov_bias)
 *   z_v    = fp32(base_v + bias_v)                      (base_logits[:, i] + bias)
 *   T > 0: x_v = fp32(z_v / T), y_v = fp32(x_v + g_v),  g from the DRAFT stream
 *          at position P - 1 ([DSP] _sample_logits: "keys a draw by the
 *          position before the sampled token")
 *   T = 0: x_v = z_v, y_v = z_v (greedy)
 *   token  = block_argmax(y)
 *
 * READING: the bias stays fp32 (no bf16 round trip); the dot product is an
 * exact-as-possible fp64 sum rounded once. READING: the cache holds x, the
 * temperature-scaled biased logits, i.e. the logits of the distribution the
 * draft was sampled from ([TPM] Part 2: the verifier works on "processed
 * logits"). */
static int markov_step_one(const void* base_row, int base_bf16,
                           const uint16_t* w1, const uint16_t* w2, int32_t prev,
                           float temperature, uint64_t seed, int64_t noise_pos,
                           int V, int R, const unsigned char* cand, float* x_out,
                           float* y_scratch, double* e_scratch, int32_t* tok_out,
                           double* gap_out) {
  if (prev < 0 || prev >= V) return ORC_EBOUNDS;
  for (int r = 0; r < R; r++)
    e_scratch[r] = (double)bf16_to_f32(w1[(int64_t)prev * R + r]);
  const int sampled = temperature > 0.0f;
  for (int64_t v = 0; v < V; v++) {
    float z;
    if (cand && !cand[v]) {
      /* top-k variant: a column outside the candidates is -inf */
      z = -INFINITY;
    } else {
      double acc = 0.0;
      const uint16_t* wrow = w2 + v * (int64_t)R;
      for (int r = 0; r < R; r++) acc += (double)bf16_to_f32(wrow[r]) * e_scratch[r];
      float bias = (float)acc;
      z = load_elem(base_row, base_bf16, v) + bias;
    }
    float x, y;
    if (sampled) {
      x = z / temperature;
      float g = gumbel_from_uniform(
          uniform_from_word(noise_word(seed, noise_pos, (uint32_t)v, ORC_STREAM_DRAFT)));
      y = x + g;
    } else {
      x = z;
      y = z;
    }
    x_out[v] = x;
    y_scratch[v] = y;
  }
  orc_winner w = block_argmax(y_scratch, V);
  *tok_out = (int32_t)w.idx;
  if (gap_out) *gap_out = w.gap;
  return ORC_OK;
}

/* Top-k candidates of one base-logit row ([DSP] _sample_sequential_topk:
 * "Apply the sequential Markov head only to top-k base-logit candidates",
 * chosen once per draft position from the base logits). READING: the k
 * largest by value, ties broken by the lower token id, -0 equal to +0, NaN
 * above every number (the ranking of a descending torch sort); k >= V keeps
 * every column. mask[v] = 1 for the candidates. */
typedef struct {
  uint32_t key;
  int64_t idx;
} orc_rank;

static uint32_t rank_key(float x) {
  if (x != x) return 0xFFFFFFFFu;
  if (x == 0.0f) x = 0.0f; /* -0 -> +0 */
  uint32_t b;
  memcpy(&b, &x, 4);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

static int rank_cmp(const void* a, const void* b) {
  const orc_rank* p = (const orc_rank*)a;
  const orc_rank* q = (const orc_rank*)b;
  if (p->key != q->key) return p->key > q->key ? -1 : 1; /* value descending */
  return p->idx < q->idx ? -1 : (p->idx > q->idx ? 1 : 0); /* id ascending */
}

static int topk_mask(const void* base_row, int base_bf16, int64_t V, int64_t k,
                     unsigned char* mask) {
  orc_rank* r = (orc_rank*)malloc(sizeof(orc_rank) * (size_t)V);
  if (!r) return ORC_ENOMEM;
  for (int64_t v = 0; v < V; v++) {
    r[v].key = rank_key(load_elem(base_row, base_bf16, v));
    r[v].idx = v;
  }
  qsort(r, (size_t)V, sizeof(orc_rank), rank_cmp);
  for (int64_t v = 0; v < V; v++) mask[v] = 0;
  for (int64_t j = 0; j < V && j < k; j++) mask[r[j].idx] = 1;
  free(r);
  return ORC_OK;
}

/* The whole K-step loop for a batch.
 *
 * base      [B,K,V] fp32 or bf16 (base_bf16)
 * w1, w2    [V,R] bf16 bit patterns
 * anchor    [B]   first `prev` of each request ([DSP] _sample_sequential:
 *                 the input id at query offset 0)
 * rsi       [B]   request-state slot; < 0 marks a padding request, which is
 *                 inert (no cache write, tokens -1) -- READING of [DSP]
 *                 _sample_sequential_sharded's "empty slots are inert"
 * pos       [B]   position P0 of the first draft token; step i samples the
 *                 token at P0 + i with noise keyed at P0 + i - 1 (READING)
 * temperature, seeds [S] per slot
 * cache     [C,K,V] fp32 or bf16 (cache_bf16) or NULL; row = row_map[s] if
 *                 row_map else s ([BSH] shard_row / row_mapping)
 * forced    [B,K] or NULL: if given, step i+1 takes forced[b,i] as prev
 *                 instead of the token it sampled (teacher forcing, used by
 *                 the parity tests after a counted near-tie)
 * tokens    [B,K] out
 * gaps      [B,K] out or NULL: top-two gap of the noised values per step
 */
/* One request of the batch loop (scratch: x[V], y[V], e[R], cand[V] or
 * NULL). */
static int markov_request(int b, const void* base, int base_bf16, const uint16_t* w1,
                          const uint16_t* w2, const int32_t* anchor, const int32_t* rsi,
                          const int64_t* pos, const float* temperature,
                          const uint64_t* seeds, void* cache, int cache_bf16,
                          const int32_t* row_map, const int32_t* forced, int32_t* tokens,
                          double* gaps, int K, int V, int R, int S, int C, int topk,
                          float* x, float* y, double* e, unsigned char* cand) {
  int32_t s = rsi[b];
  if (s < 0) {
    for (int i = 0; i < K; i++) {
      tokens[(int64_t)b * K + i] = -1;
      if (gaps) gaps[(int64_t)b * K + i] = INFINITY;
    }
    return ORC_OK;
  }
  if (s >= S) return ORC_EBOUNDS;
  int64_t row = row_map ? (int64_t)row_map[s] : (int64_t)s;
  if (cache && (row < 0 || row >= C)) return ORC_EBOUNDS;
  int32_t prev = anchor[b];
  for (int i = 0; i < K; i++) {
    const int64_t base_off = ((int64_t)b * K + i) * V;
    const void* base_row =
        base_bf16 ? (const void*)((const uint16_t*)base + base_off)
                  : (const void*)((const float*)base + base_off);
    int32_t tok;
    double gap;
    int rc;
    if (topk > 0) {
      rc = topk_mask(base_row, base_bf16, V, topk, cand);
      if (rc != ORC_OK) return rc;
    }
    rc = markov_step_one(base_row, base_bf16, w1, w2, prev, temperature[s], seeds[s],
                         pos[b] + i - 1, V, R, topk > 0 ? cand : NULL, x, y, e, &tok, &gap);
    if (rc != ORC_OK) return rc;
    tokens[(int64_t)b * K + i] = tok;
    if (gaps) gaps[(int64_t)b * K + i] = gap;
    if (cache) {
      const int64_t off = (row * K + i) * (int64_t)V;
      for (int64_t v = 0; v < V; v++) {
        if (cache_bf16)
          ((uint16_t*)cache)[off + v] = f32_to_bf16(x[v]);
        else
          ((float*)cache)[off + v] = x[v];
      }
    }
    prev = forced ? forced[(int64_t)b * K + i] : tok;
  }
  return ORC_OK;
}

static int markov_sample_impl(const void* base, int base_bf16, const uint16_t* w1,
                              const uint16_t* w2, const int32_t* anchor,
                              const int32_t* rsi, const int64_t* pos,
                              const float* temperature, const uint64_t* seeds,
                              void* cache, int cache_bf16, const int32_t* row_map,
                              const int32_t* forced, int32_t* tokens, double* gaps,
                              int B, int K, int V, int R, int S, int C, int topk) {
  if (B < 0 || K <= 0 || V <= 0 || R <= 0 || S <= 0 || topk < 0) return ORC_EINVAL;
  if (!base || !w1 || !w2 || !anchor || !rsi || !pos || !temperature || !seeds ||
      !tokens)
    return ORC_EINVAL;
  int rc = ORC_OK;
  ORC_OMP(omp parallel)
  {
    float* x = (float*)malloc(sizeof(float) * (size_t)V);
    float* y = (float*)malloc(sizeof(float) * (size_t)V);
    double* e = (double*)malloc(sizeof(double) * (size_t)R);
    unsigned char* cand = topk > 0 ? (unsigned char*)malloc((size_t)V) : NULL;
    const int have = x && y && e && (topk == 0 || cand);
    ORC_OMP(omp for schedule(dynamic, 1))
    for (int b = 0; b < B; b++) {
      const int r = have ? markov_request(b, base, base_bf16, w1, w2, anchor, rsi, pos,
                                          temperature, seeds, cache, cache_bf16, row_map,
                                          forced, tokens, gaps, K, V, R, S, C, topk, x, y, e,
                                          cand)
                         : ORC_ENOMEM;
      if (r != ORC_OK) {
        ORC_OMP(omp critical(orc_rc))
        if (rc == ORC_OK) rc = r;
      }
    }
    free(x);
    free(y);
    free(e);
    free(cand);
  }
  return rc;
}

int orc_markov_sample(const void* base, int base_bf16, const uint16_t* w1,
                      const uint16_t* w2, const int32_t* anchor,
                      const int32_t* rsi, const int64_t* pos,
                      const float* temperature, const uint64_t* seeds,
                      void* cache, int cache_bf16, const int32_t* row_map,
                      const int32_t* forced, int32_t* tokens, double* gaps,
                      int B, int K, int V, int R, int S, int C) {
  return markov_sample_impl(base, base_bf16, w1, w2, anchor, rsi, pos, temperature,
                            seeds, cache, cache_bf16, row_map, forced, tokens, gaps,
                            B, K, V, R, S, C, 0);
}

/* The top-k variant of the loop ([DSP] _sample_sequential_topk): per request
 * and draft step, the Markov bias is applied to the top-k base-logit
 * candidates of that step and every other column is -inf; sampling, the
 * winner rule and the cache store are then the dense ones. topk >= 1. */
int orc_markov_sample_topk(const void* base, int base_bf16, const uint16_t* w1,
                           const uint16_t* w2, const int32_t* anchor,
                           const int32_t* rsi, const int64_t* pos,
                           const float* temperature, const uint64_t* seeds,
                           void* cache, int cache_bf16, const int32_t* row_map,
                           const int32_t* forced, int32_t* tokens, double* gaps,
                           int B, int K, int V, int R, int S, int C, int topk) {
  if (topk < 1) return ORC_EINVAL;
  return markov_sample_impl(base, base_bf16, w1, w2, anchor, rsi, pos, temperature,
                            seeds, cache, cache_bf16, row_map, forced, tokens, gaps,
                            B, K, V, R, S, C, topk);
}

/* One step of one request with an explicit `prev` (for sampled checks at full
 * size): writes x[V], the token and the top-two gap. */
int orc_markov_step(const void* base_row, int base_bf16, const uint16_t* w1,
                    const uint16_t* w2, int32_t prev, float temperature,
                    uint64_t seed, int64_t noise_pos, int V, int R,
                    float* x_out, int32_t* tok_out, double* gap_out) {
  if (!base_row || !w1 || !w2 || !x_out || !tok_out || V <= 0 || R <= 0)
    return ORC_EINVAL;
  float* y = (float*)malloc(sizeof(float) * (size_t)V);
  double* e = (double*)malloc(sizeof(double) * (size_t)R);
  if (!y || !e) {
    free(y);
    free(e);
    return ORC_ENOMEM;
  }
  int rc = markov_step_one(base_row, base_bf16, w1, w2, prev, temperature, seed,
                           noise_pos, V, R, NULL, x_out, y, e, tok_out, gap_out);
  free(y);
  free(e);
  return rc;
}

/* ======================================================================== */
/* Part 2: the rejection-sampling verifier.                                   */
/* ======================================================================== */

/* READING of "masses are summed in 64-bit fixed point" ([TPM] Part 2,
 * temperature and top-p): one unit of exp-mass is 2^40; V * 2^40 < 2^63 for
 * every vocabulary below 2^23. */
#define ORC_FIX_SHIFT 40
#define ORC_MAX_VOCAB (1 << 23)

static uint64_t to_fixed(float e) {
  double scaled = (double)e * 0x1p40; /* exact */
  return (uint64_t)nearbyint(scaled); /* round half to even */
}

/* Sort key for the top-p order: logit descending, then token id ascending. */
typedef struct {
  float val;
  int32_t id;
} orc_kv;

static int kv_cmp(const void* a, const void* b) {
  const orc_kv* x = (const orc_kv*)a;
  const orc_kv* y = (const orc_kv*)b;
  if (x->val > y->val) return -1;
  if (x->val < y->val) return 1;
  return (x->id > y->id) - (x->id < y->id);
}

/* Target distribution of one row after temperature and exact top-p.
 *
 *   xt_v = fp32(t_v / T); NaN is read as -inf (READING)
 *   m    = max_v xt_v
 *   no value above -inf: p = one-hot at column 0 (READING: the first-maximum
 *          rule applied to an all -inf row)
 *   e_v  = 1 if xt_v == m else fp32(exp(fp32(xt_v - m)))   [exp in fp64]
 *   f_v  = rint(e_v * 2^40)  (uint64), F = sum_v f_v
 *   top_p < 1: keep = the shortest prefix of the (xt desc, id asc) order whose
 *          fixed-point mass S satisfies S * 2^32 >= P32 * F, P32 =
 *          rint(top_p * 2^32) (128-bit compare); never empty, so the row max
 *          is always kept ([TPM] Part 2: "the smallest prefix (by logit, then
 *          token id) whose probability mass reaches p, plus the row max")
 *   Fk   = sum over keep of f_v; D = fp32(Fk) * 2^-40
 *   p_v  = fp32(e_v / D) on keep, else 0
 *
 * Outputs: p[V], keep[V] (0/1), *F_total, *F_kept, *boundary_slack =
 * min(|S_{n-1}/F - p|, |S_n/F - p|) for the kept count n (the margin by which
 * the top-p boundary was decided; +inf when top-p does not apply). */
static int target_probs_impl(const void* row, int is_bf16, int V,
                             float temperature, float top_p, float* p,
                             uint8_t* keep, uint64_t* F_total,
                             uint64_t* F_kept, double* boundary_slack,
                             float* e_scratch, orc_kv* kv_scratch) {
  float m = -INFINITY;
  for (int64_t v = 0; v < V; v++) {
    float t = load_elem(row, is_bf16, v);
    float xt = t / temperature;
    if (isnan(xt)) xt = -INFINITY;
    e_scratch[v] = xt; /* holds xt for now */
    if (xt > m) m = xt;
  }
  if (boundary_slack) *boundary_slack = INFINITY;
  if (m == -INFINITY) {
    for (int64_t v = 0; v < V; v++) {
      p[v] = v == 0 ? 1.0f : 0.0f;
      keep[v] = v == 0;
    }
    if (F_total) *F_total = (uint64_t)1 << ORC_FIX_SHIFT;
    if (F_kept) *F_kept = (uint64_t)1 << ORC_FIX_SHIFT;
    return ORC_OK;
  }
  uint64_t F = 0;
  for (int64_t v = 0; v < V; v++) {
    float xt = e_scratch[v];
    kv_scratch[v].val = xt;
    kv_scratch[v].id = (int32_t)v;
    float e;
    if (xt == m) {
      e = 1.0f;
    } else {
      float d = xt - m;
      e = (float)exp((double)d);
    }
    e_scratch[v] = e;
    F += to_fixed(e);
  }
  for (int64_t v = 0; v < V; v++) keep[v] = 1;
  uint64_t Fk = F;
  if (top_p < 1.0f) {
    double p_scaled = nearbyint((double)top_p * 0x1p32);
    uint64_t P32 = p_scaled <= 0.0 ? 0u : (uint64_t)p_scaled;
    qsort(kv_scratch, (size_t)V, sizeof(orc_kv), kv_cmp);
    unsigned __int128 target = (unsigned __int128)P32 * (unsigned __int128)F;
    uint64_t S = 0;
    int64_t n = 0;
    for (; n < V; n++) {
      S += to_fixed(e_scratch[kv_scratch[n].id]);
      if ((((unsigned __int128)S) << 32) >= target) {
        n++;
        break;
      }
    }
    if (n > V) n = V;
    for (int64_t v = 0; v < V; v++) keep[v] = 0;
    for (int64_t j = 0; j < n; j++) keep[kv_scratch[j].id] = 1;
    Fk = S;
    if (boundary_slack) {
      double pd = (double)top_p;
      double s_n = (double)S / (double)F;
      double s_prev =
          (double)(S - to_fixed(e_scratch[kv_scratch[n - 1].id])) / (double)F;
      double a = fabs(s_n - pd), b2 = fabs(s_prev - pd);
      *boundary_slack = a < b2 ? a : b2;
    }
  }
  float D = (float)Fk * 0x1p-40f;
  for (int64_t v = 0; v < V; v++) p[v] = keep[v] ? e_scratch[v] / D : 0.0f;
  if (F_total) *F_total = F;
  if (F_kept) *F_kept = Fk;
  return ORC_OK;
}

/* Draft distribution q = softmax of one cached draft row (the cache already
 * holds temperature-scaled logits, so no temperature here; READING). Same
 * fixed-point normalisation as the target, no top-p (READING: q is the
 * distribution the draft token was drawn from). NaN reads as -inf; a row
 * with no value above -inf gives q = 0 everywhere (READING). */
static int draft_probs_impl(const void* row, int is_bf16, int V, float* q) {
  float m = -INFINITY;
  for (int64_t v = 0; v < V; v++) {
    float c = load_elem(row, is_bf16, v);
    if (isnan(c)) c = -INFINITY;
    q[v] = c;
    if (c > m) m = c;
  }
  if (m == -INFINITY) {
    for (int64_t v = 0; v < V; v++) q[v] = 0.0f;
    return ORC_OK;
  }
  uint64_t F = 0;
  for (int64_t v = 0; v < V; v++) {
    float c = q[v];
    float e = c == m ? 1.0f : (float)exp((double)(c - m));
    q[v] = e;
    F += to_fixed(e);
  }
  float D = (float)F * 0x1p-40f;
  for (int64_t v = 0; v < V; v++) q[v] = q[v] / D;
  return ORC_OK;
}

/* Categorical draw by Gumbel-max (READING: the pages name "residual-mass and
 * resample kernels" but no method): argmax_v fp32(fp32(log w_v) + g_v) with
 * g from the TARGET stream at the given noise position, under the same
 * block-argmax rule as the drafter. log is evaluated in fp64 and rounded. */
static orc_winner categorical_draw(const float* w, int V, uint64_t seed,
                                   int64_t noise_pos, float* y_scratch) {
  for (int64_t v = 0; v < V; v++) {
    float lw = w[v] > 0.0f ? (float)log((double)w[v]) : -INFINITY;
    float g = gumbel_from_uniform(
        uniform_from_word(noise_word(seed, noise_pos, (uint32_t)v, ORC_STREAM_TARGET)));
    y_scratch[v] = lw + g;
  }
  return block_argmax(y_scratch, V);
}

/* The verifier for a batch.
 *
 * draft   [B,K]     drafted tokens; -1 marks "no draft from here on"
 * cache   [C,K,V]   draft-logits cache (fp32 or bf16), rows via row_map
 * target  [B,K+1,V] target logits (fp32 or bf16)
 * rsi, pos, temperature, top_p, seeds as in the drafter
 * out     [B,K+1]   accepted drafts, then one recovered or bonus token; -1 after
 * num_acc [B]       number of accepted drafts
 * margins [B,K]     or NULL: |u - p/q| of each ratio test actually made
 *                   (+inf when q = 0 or greedy; NaN where no test was made)
 * gaps    [B]       or NULL: top-two gap of the draw that produced the last
 *                   emitted token (recovered, bonus, or greedy argmax)
 * slack   [B,K+1]   or NULL: top-p boundary slack of each target row whose
 *                   distribution was used (+inf if top-p did not apply, NaN
 *                   if the row was not used)
 *
 * Per request with slot s >= 0, T = temperature[s]:
 *  sampled (T > 0), for k = 0..K-1:
 *    d = draft[b,k]; d = -1: emit a draw from p_k (READING) and stop.
 *    u = uniform(seed, P0+k-1, column 0, ACCEPT stream)
 *    accept iff fp32(u * q_k(d)) < p_k(d): probability min(1, p/q).
 *    reject: emit a Gumbel-max draw from r = max(0, p_k - q_k) (fp32), TARGET
 *    stream at P0+k-1; if r is all zero, draw from p_k instead (READING).
 *  all K accepted: emit the bonus, a draw from p_K at P0+K-1.
 *  greedy (T <= 0 or NaN): accept iff d == block_argmax(target row k); on
 *    mismatch (or d = -1) emit that argmax; bonus = argmax of row K. The draft
 *    cache is never read ([BSH] notes: "verification compares against the
 *    target argmax and never reads cached draft logits").
 *  padding (s < 0): all -1, num_acc 0, nothing read. */
/* One request of the verifier (scratch: p, q, r, e [V], keep [V], kv [V]). */
static int verify_request(int b, const int32_t* draft, const void* cache, int cache_bf16,
                          const int32_t* row_map, const void* target, int target_bf16,
                          const int32_t* rsi, const int64_t* pos, const float* temperature,
                          const float* top_p, const uint64_t* seeds, int32_t* out,
                          int32_t* num_acc, double* margins, double* gaps, double* slack,
                          int K, int V, int S, int C, float* p, float* q, float* r, float* e,
                          uint8_t* keep, orc_kv* kv) {
  const int64_t K1 = (int64_t)K + 1;
  for (int64_t k = 0; k < K1; k++) out[b * K1 + k] = -1;
  num_acc[b] = 0;
  if (margins)
    for (int k = 0; k < K; k++) margins[(int64_t)b * K + k] = NAN;
  if (gaps) gaps[b] = INFINITY;
  if (slack)
    for (int64_t k = 0; k < K1; k++) slack[b * K1 + k] = NAN;
  const int32_t s = rsi[b];
  if (s < 0) return ORC_OK;
  if (s >= S) return ORC_EBOUNDS;
  const float T = temperature[s];
  const int greedy = !(T > 0.0f);
  const uint64_t seed = seeds[s];
  const int64_t P0 = pos[b];
  int64_t crow = 0;
  if (!greedy) {
    if (!cache) return ORC_EINVAL;
    crow = row_map ? (int64_t)row_map[s] : (int64_t)s;
    if (crow < 0 || crow >= C) return ORC_EBOUNDS;
  }
  int done = 0;
  int32_t n_acc = 0;
  for (int64_t k = 0; k < K && !done; k++) {
    const int32_t d = draft[(int64_t)b * K + k];
    if (d < -1 || d >= V) return ORC_EBOUNDS;
    const int64_t toff = ((int64_t)b * K1 + k) * V;
    const void* trow = target_bf16
                           ? (const void*)((const uint16_t*)target + toff)
                           : (const void*)((const float*)target + toff);
    if (greedy) {
      for (int64_t v = 0; v < V; v++) r[v] = load_elem(trow, target_bf16, v);
      orc_winner w = block_argmax(r, V);
      if (margins) margins[(int64_t)b * K + k] = INFINITY;
      if (d >= 0 && d == (int32_t)w.idx) {
        out[(int64_t)b * K1 + k] = d;
        n_acc++;
      } else {
        out[(int64_t)b * K1 + k] = (int32_t)w.idx;
        if (gaps) gaps[b] = w.gap;
        done = 1;
      }
      continue;
    }
    double sl;
    target_probs_impl(trow, target_bf16, V, T, top_p[s], p, keep, NULL, NULL,
                      &sl, e, kv);
    if (slack) slack[b * K1 + k] = sl;
    if (d == -1) {
      orc_winner w = categorical_draw(p, V, seed, P0 + k - 1, r);
      out[(int64_t)b * K1 + k] = (int32_t)w.idx;
      if (gaps) gaps[b] = w.gap;
      done = 1;
      break;
    }
    const int64_t coff = (crow * K + k) * (int64_t)V;
    const void* qrow = cache_bf16 ? (const void*)((const uint16_t*)cache + coff)
                                  : (const void*)((const float*)cache + coff);
    draft_probs_impl(qrow, cache_bf16, V, q);
    const float u = uniform_from_word(
        noise_word(seed, P0 + k - 1, 0u, ORC_STREAM_ACCEPT));
    const float pd = p[d], qd = q[d];
    const float uq = u * qd;
    if (margins) {
      margins[(int64_t)b * K + k] =
          qd > 0.0f ? fabs((double)u - (double)pd / (double)qd) : INFINITY;
    }
    if (uq < pd) {
      out[(int64_t)b * K1 + k] = d;
      n_acc++;
      continue;
    }
    int any_pos = 0;
    for (int64_t v = 0; v < V; v++) {
      float diff = p[v] - q[v];
      r[v] = diff > 0.0f ? diff : 0.0f;
      if (r[v] > 0.0f) any_pos = 1;
    }
    orc_winner w = categorical_draw(any_pos ? r : p, V, seed, P0 + k - 1, e);
    out[(int64_t)b * K1 + k] = (int32_t)w.idx;
    if (gaps) gaps[b] = w.gap;
    done = 1;
  }
  if (!done) {
    const int64_t toff = ((int64_t)b * K1 + K) * V;
    const void* trow = target_bf16
                           ? (const void*)((const uint16_t*)target + toff)
                           : (const void*)((const float*)target + toff);
    orc_winner w;
    if (greedy) {
      for (int64_t v = 0; v < V; v++) r[v] = load_elem(trow, target_bf16, v);
      w = block_argmax(r, V);
    } else {
      double sl;
      target_probs_impl(trow, target_bf16, V, T, top_p[s], p, keep, NULL,
                        NULL, &sl, e, kv);
      if (slack) slack[b * K1 + K] = sl;
      w = categorical_draw(p, V, seed, P0 + K - 1, r);
    }
    out[(int64_t)b * K1 + K] = (int32_t)w.idx;
    if (gaps) gaps[b] = w.gap;
  }
  num_acc[b] = n_acc;
  return ORC_OK;
}

int orc_rejection_sample(const int32_t* draft, const void* cache,
                         int cache_bf16, const int32_t* row_map,
                         const void* target, int target_bf16,
                         const int32_t* rsi, const int64_t* pos,
                         const float* temperature, const float* top_p,
                         const uint64_t* seeds, int32_t* out, int32_t* num_acc,
                         double* margins, double* gaps, double* slack, int B,
                         int K, int V, int S, int C) {
  if (B < 0 || K <= 0 || V <= 0 || V > ORC_MAX_VOCAB || S <= 0) return ORC_EINVAL;
  if (!draft || !target || !rsi || !pos || !temperature || !top_p || !seeds ||
      !out || !num_acc)
    return ORC_EINVAL;
  int rc = ORC_OK;
  ORC_OMP(omp parallel)
  {
    float* p = (float*)malloc(sizeof(float) * (size_t)V);
    float* q = (float*)malloc(sizeof(float) * (size_t)V);
    float* r = (float*)malloc(sizeof(float) * (size_t)V);
    float* e = (float*)malloc(sizeof(float) * (size_t)V);
    uint8_t* keep = (uint8_t*)malloc((size_t)V);
    orc_kv* kv = (orc_kv*)malloc(sizeof(orc_kv) * (size_t)V);
    const int have = p && q && r && e && keep && kv;
    ORC_OMP(omp for schedule(dynamic, 1))
    for (int b = 0; b < B; b++) {
      const int rr = have ? verify_request(b, draft, cache, cache_bf16, row_map, target,
                                           target_bf16, rsi, pos, temperature, top_p, seeds,
                                           out, num_acc, margins, gaps, slack, K, V, S, C, p,
                                           q, r, e, keep, kv)
                          : ORC_ENOMEM;
      if (rr != ORC_OK) {
        ORC_OMP(omp critical(orc_rc))
        if (rc == ORC_OK) rc = rr;
      }
    }
    free(p);
    free(q);
    free(r);
    free(e);
    free(keep);
    free(kv);
  }
  return rc;
}

/* Host threads the batch entry points use: n > 0 sets it (OpenMP build);
 * returns the count now in force (1 in the plain build). */
int orc_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Row-level and noise entry points, for the pin tests.                      */
/* ------------------------------------------------------------------------ */

int orc_philox_batch(int64_t n, const uint32_t* key, const uint32_t* ctr,
                     uint32_t* out) {
  if (n < 0 || (n > 0 && (!key || !ctr || !out))) return ORC_EINVAL;
  for (int64_t i = 0; i < n; i++)
    philox4x32_10(ctr + 4 * i, key[2 * i], key[2 * i + 1], out + 4 * i);
  return ORC_OK;
}

int orc_noise_batch(int64_t n, const uint64_t* seed, const int64_t* pos,
                    const uint32_t* col, const uint32_t* stream, uint32_t* word,
                    float* u, float* g) {
  if (n < 0 || (n > 0 && (!seed || !pos || !col || !stream))) return ORC_EINVAL;
  for (int64_t i = 0; i < n; i++) {
    uint32_t w = noise_word(seed[i], pos[i], col[i], stream[i]);
    float uu = uniform_from_word(w);
    if (word) word[i] = w;
    if (u) u[i] = uu;
    if (g) g[i] = gumbel_from_uniform(uu);
  }
  return ORC_OK;
}

int orc_block_argmax(const float* y, int64_t n, int64_t* idx, double* gap) {
  if (n <= 0 || !y || !idx) return ORC_EINVAL;
  orc_winner w = block_argmax(y, n);
  *idx = w.idx;
  if (gap) *gap = w.gap;
  return ORC_OK;
}

int orc_target_probs(const void* row, int is_bf16, int V, float temperature,
                     float top_p, float* p, uint8_t* keep, uint64_t* F_total,
                     uint64_t* F_kept, double* boundary_slack) {
  if (!row || !p || !keep || V <= 0 || V > ORC_MAX_VOCAB || !(temperature > 0.0f))
    return ORC_EINVAL;
  float* e = (float*)malloc(sizeof(float) * (size_t)V);
  orc_kv* kv = (orc_kv*)malloc(sizeof(orc_kv) * (size_t)V);
  if (!e || !kv) {
    free(e);
    free(kv);
    return ORC_ENOMEM;
  }
  int rc = target_probs_impl(row, is_bf16, V, temperature, top_p, p, keep,
                             F_total, F_kept, boundary_slack, e, kv);
  free(e);
  free(kv);
  return rc;
}

int orc_draft_probs(const void* row, int is_bf16, int V, float* q) {
  if (!row || !q || V <= 0 || V > ORC_MAX_VOCAB) return ORC_EINVAL;
  return draft_probs_impl(row, is_bf16, V, q);
}

int orc_categorical(const float* w, int V, uint64_t seed, int64_t noise_pos,
                    int64_t* idx, double* gap) {
  if (!w || !idx || V <= 0) return ORC_EINVAL;
  float* y = (float*)malloc(sizeof(float) * (size_t)V);
  if (!y) return ORC_ENOMEM;
  orc_winner win = categorical_draw(w, V, seed, noise_pos, y);
  free(y);
  *idx = win.idx;
  if (gap) *gap = win.gap;
  return ORC_OK;
}
