// markov_tc.cu -- one Markov step on the 5th-generation tensor cores.
//
// The "DSparkSpeculator" page's _sample_markov_chain / _sample_logits and
// vLLM PR #65007 Part 1 (per-step list): Markov embedding of the previous
// token, the markov_w2 bias projection, bias add, temperature, Gumbel noise
// keyed by (seed, position - 1, column), the block-argmax winner rule and the
// draft-logits cache store, fused into one kernel per step.
//
// The bias projection [B, R] x [R, V] runs on the tensor cores for every
// batch size: the step is bound by streaming markov_w2 and by the epilogue's
// ALU work, and the MMA takes the B * R multiply-adds per column off the
// epilogue warps (for small B the padding of N to 16 costs nothing).
// markov_w2 rows are the M side of a tcgen05 MMA
// (M = 128 vocabulary rows per tile, K = markov_rank), the Markov embeddings
// of the batch are the N side (N = batch padded to a multiple of 16), and the
// fp32 accumulator lives in tensor memory.
//
// Persistent, warp-specialised CTA (one per SM):
//   warp 0      TMA producer: 128x64 bf16 boxes of markov_w2 (128-byte
//               swizzle) into a ring of shared-memory stages, L2 evict-last;
//               and, per tile, the tile's base logits of every request (a
//               128 x 1 x B box of the [B, K, V] tensor) into one of two slots
//   warp 1      TMEM allocation; one thread issues the MMAs (4 per 64-wide K
//               chunk) into one of two accumulator buffers and commits
//   warps 2-17  epilogue: warp (q, sub) owns TMEM lane quarter q (32 rows of
//               each tile) and a fixed set of CPW batch columns. Per chunk of
//               4 columns: tcgen05.ld, bias add, temperature (x = z * (1/T),
//               within 1.5 ulp of z / T), Gumbel noise (one Philox block per
//               lane quad, shared by a 4x4 butterfly transpose), cache store,
//               and the running winner of each
//               column -- per lane in registers across tiles when CPW <= 16,
//               else reduced per tile with redux.sync.
// The per-CTA winners go to the workspace; the last CTA to finish reduces
// them per request and writes the step's tokens.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace dspark {

namespace {

constexpr int kM = 128;                 // vocabulary rows per tile (UMMA M)
constexpr int kStageBytes = kM * 128;   // one 64-element K chunk of a tile
constexpr int kEpiWarps = 16;           // four per TMEM lane quarter
constexpr int kThreadsTc = 64 + 32 * kEpiWarps;
constexpr int kMaxStages = 12;
constexpr size_t kSmemLimit = 227u * 1024u;

// Per-request data of one step, structure of arrays (Npad entries each).
struct TcLayout {
  size_t a, e, bases, temp, seed, npos, boff, coff, best, bars, slot, flags, total;
  // base_stage: bytes of one staged base tile (0 = base logits read directly)
  __host__ __device__ TcLayout(int Npad, int NK, int ns, size_t base_stage) {
    a = 0;
    e = a + static_cast<size_t>(ns) * kStageBytes;
    bases = e + static_cast<size_t>(NK) * Npad * 128;
    temp = bases + 2 * ((base_stage + 1023) & ~size_t(1023));
    seed = temp + static_cast<size_t>(Npad) * 4;
    npos = seed + static_cast<size_t>(Npad) * 8;
    boff = npos + static_cast<size_t>(Npad) * 8;
    coff = boff + static_cast<size_t>(Npad) * 8;
    best = coff + static_cast<size_t>(Npad) * 8;
    bars = best + static_cast<size_t>(Npad) * 8;
    slot = bars + static_cast<size_t>(2 * ns + 7) * 8;
    flags = slot + 8;
    total = flags + 8 + kMaxStages * 4 + 1024;  // + slack to align the base to 1024 B
  }
};

// Lanes 4j..4j+3 each hold the four Philox words of request b0 + (lane & 3)
// for the same 4-column block (a 4x4 matrix, one row per lane). A two-round
// butterfly transposes it: afterwards w[r] = word (lane & 3) of request
// b0 + r, i.e. the noise of this lane's own column for request b0 + r.
__device__ __forceinline__ void quad_transpose(uint32_t (&w)[4]) {
  const uint32_t c = threadIdx.x & 3u;
  // round 1 (lanes c, c^2): the upper lane takes the lower lane's words 2,3
  {
    const bool up = (c & 2u) != 0u;
    const uint32_t s0 = up ? w[0] : w[2];
    const uint32_t s1 = up ? w[1] : w[3];
    const uint32_t r0 = __shfl_xor_sync(0xFFFFFFFFu, s0, 2);
    const uint32_t r1 = __shfl_xor_sync(0xFFFFFFFFu, s1, 2);
    if (up) {
      w[0] = r0;
      w[1] = r1;
    } else {
      w[2] = r0;
      w[3] = r1;
    }
  }
  // round 2 (lanes c, c^1)
  {
    const bool odd = (c & 1u) != 0u;
    const uint32_t s0 = odd ? w[0] : w[1];
    const uint32_t s1 = odd ? w[2] : w[3];
    const uint32_t r0 = __shfl_xor_sync(0xFFFFFFFFu, s0, 1);
    const uint32_t r1 = __shfl_xor_sync(0xFFFFFFFFu, s1, 1);
    if (odd) {
      w[0] = r0;
      w[2] = r1;
    } else {
      w[1] = r0;
      w[3] = r1;
    }
  }
}

// Winner over the warp's lanes of (ord, v): largest ord, then lowest v.
__device__ __forceinline__ unsigned long long warp_winner(uint32_t ord, uint32_t v) {
  const uint32_t omax = __reduce_max_sync(0xFFFFFFFFu, ord);
  const uint32_t cand = (ord == omax && ord != 0u) ? v : 0xFFFFFFFFu;
  const uint32_t vmin = __reduce_min_sync(0xFFFFFFFFu, cand);
  return omax == 0u ? 0ull
                    : (static_cast<unsigned long long>(omax) << 32) | (0xFFFFFFFFu - vmin);
}

template <int CPW>  // batch columns per epilogue warp (Npad / 4)
__global__ void __launch_bounds__(kThreadsTc, 1)
markov_step_tc_kernel(const __grid_constant__ CUtensorMap tmap_w2,
                      const __grid_constant__ CUtensorMap tmap_base, MarkovStepParams P, int Npad,
                      int ns, uint32_t tmem_cols, uint32_t base_stage_bytes) {
  constexpr bool kRegWinners = CPW <= 16;
  const int R = P.R;
  const int NK = R / 64;
  const bool tma_base = base_stage_bytes != 0u;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const TcLayout L(Npad, NK, ns, base_stage_bytes);
  unsigned char* a_base = smem + L.a;
  unsigned char* e_base = smem + L.e;
  unsigned char* base_s = smem + L.bases;  // two staged base tiles [B][128]
  const size_t base_stride = (static_cast<size_t>(base_stage_bytes) + 1023) & ~size_t(1023);
  float* s_temp = reinterpret_cast<float*>(smem + L.temp);      // 1/T (0: greedy)
  uint64_t* s_seed = reinterpret_cast<uint64_t*>(smem + L.seed);
  int64_t* s_npos = reinterpret_cast<int64_t*>(smem + L.npos);
  int64_t* s_boff = reinterpret_cast<int64_t*>(smem + L.boff);   // -1: inert column
  int64_t* s_coff = reinterpret_cast<int64_t*>(smem + L.coff);   // -1: no cache store
  int32_t* s_prev = reinterpret_cast<int32_t*>(smem + L.coff);   // prologue only (aliases coff)
  unsigned long long* best = reinterpret_cast<unsigned long long*>(smem + L.best);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + ns;
  uint64_t* acc_full = empty + ns;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* base_full = drain + 1;     // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.slot);
  int* fail_flag = reinterpret_cast<int*>(smem + L.flags);
  uint32_t* issued = reinterpret_cast<uint32_t*>(smem + L.flags + 8);  // last parity per stage

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = P.B, V = P.V, K = P.K, step = P.step;
  const int G = gridDim.x;
  const int tiles = (V + kM - 1) / kM;

  // ---- prologue: per-request data (thread n < Npad owns column n) ------------
  int32_t my_prev = -1;
  int64_t my_coff = -1;
  if (tid < Npad) {
    const int n = tid;
    float temp = 0.f;
    uint64_t seed = 0;
    int64_t npos = 0, boff = -1, coff = -1;
    int32_t prev = -1;
    const int32_t s = n < B ? P.rsi[n] : -1;
    if (s >= 0) {
      if (s >= P.S) {
        report(P.status, DSPARK_ERR_BOUNDS);
      } else {
        const int32_t pv =
            step == 0 ? P.anchor[n] : P.out_tokens[static_cast<int64_t>(n) * K + step - 1];
        bool ok = pv >= 0 && pv < V;
        if (!ok) report(P.status, DSPARK_ERR_BOUNDS);
        if (ok && P.cache != nullptr) {
          const int64_t row = P.row_map ? P.row_map[s] : s;
          if (row < 0 || row >= P.C) {
            report(P.status, DSPARK_ERR_BOUNDS);
            ok = false;
          } else {
            coff = (row * K + step) * static_cast<int64_t>(V);
          }
        }
        if (ok) {
          prev = pv;
          temp = P.temperature[s];
          seed = P.seeds[s];
          npos = P.pos[n] + step - 1;
          boff = (static_cast<int64_t>(n) * K + step) * V;
        } else {
          coff = -1;
        }
      }
    }
    s_temp[n] = temp > 0.f ? __frcp_rn(temp) : 0.f;  // 1/T; 0 marks a greedy column
    s_seed[n] = seed;
    s_npos[n] = npos;
    s_boff[n] = boff;
    s_prev[n] = prev;
    best[n] = 0ull;
    my_prev = prev;
    my_coff = coff;
  }
  (void)my_prev;
  if (tid == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&acc_full[0], 1);
    mbar_init(&acc_full[1], 1);
    mbar_init(&acc_empty[0], kEpiWarps);
    mbar_init(&acc_empty[1], kEpiWarps);
    mbar_init(drain, 1);
    mbar_init(&base_full[0], 1);
    mbar_init(&base_full[1], 1);
    for (int i = 0; i < kMaxStages; ++i) issued[i] = 0xFFFFFFFFu;
    *fail_flag = 0;
    fence_mbar_init();
    tc::prefetch_tensormap(&tmap_w2);
    if (tma_base) tc::prefetch_tensormap(&tmap_base);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, tmem_cols);
    tc::tmem_relinquish();
  }
  __syncthreads();

  // Markov embeddings e[n] = w1[prev_n] as the N-side operand, K-major,
  // 128-byte swizzle: chunk c of row n of K-chunk kc at n*128 + (c ^ (n%8))*16.
  {
    const int per_row = NK * 8;
    const int total = Npad * per_row;
    for (int c = tid; c < total; c += kThreadsTc) {
      const int n = c / per_row, rem = c % per_row;
      const int kc = rem >> 3, cc = rem & 7;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      const int32_t pv = s_prev[n];
      if (pv >= 0)
        val = __ldg(reinterpret_cast<const uint4*>(P.w1 + static_cast<int64_t>(pv) * R + kc * 64) +
                    cc);
      *reinterpret_cast<uint4*>(e_base + static_cast<size_t>(kc) * Npad * 128 + n * 128 +
                                ((cc ^ (n & 7)) << 4)) = val;
    }
  }
  __syncthreads();
  if (tid < Npad) s_coff[tid] = my_coff;  // s_prev (same storage) is no longer read
  fence_proxy_async_smem();
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer -----------------------------------------------------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      const uint64_t pol_stream = policy_evict_first();
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      uint32_t base_par[2] = {0xFFFFFFFFu, 0xFFFFFFFFu};  // parity of the last copy per slot
      for (int i = 0; ok; ++i) {
        const int t = blockIdx.x + i * G;
        if (t >= tiles) break;
        if (tma_base) {
          // base slot i&1 is free once the epilogue released tile i-2
          const int bs = i & 1;
          if (!mbar_wait(&acc_empty[bs], ((i >> 1) & 1) ^ 1u, P.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&base_full[bs], base_stage_bytes);
          tc::tma_load_3d(base_s + bs * base_stride, &tmap_base, t * kM, step, 0, &base_full[bs],
                          pol_stream);
          base_par[bs] = (i >> 1) & 1;
        }
        for (int kc = 0; kc < NK; ++kc) {
          if (!mbar_wait(&empty[stage], ph ^ 1u, P.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], kStageBytes);
          tc::tma_load_2d(a_base + static_cast<size_t>(stage) * kStageBytes, &tmap_w2, kc * 64,
                          t * kM, &full[stage], pol);
          issued[stage] = ph;
          if (++stage == ns) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) atomicExch(fail_flag, 1);
      // every copy this CTA issued has landed before the CTA may exit
      for (int s2 = 0; s2 < ns; ++s2)
        if (issued[s2] != 0xFFFFFFFFu) (void)mbar_wait(&full[s2], issued[s2], P.status);
      for (int bs = 0; bs < 2; ++bs)
        if (base_par[bs] != 0xFFFFFFFFu) (void)mbar_wait(&base_full[bs], base_par[bs], P.status);
    }
  } else if (warp == 1) {
    // ---- MMA issuer -------------------------------------------------------------
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(kM, Npad);
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int t = blockIdx.x + i * G;
        if (t >= tiles) break;
        const int ab = i & 1;
        const uint32_t aph = (i >> 1) & 1;
        if (!mbar_wait(&acc_empty[ab], aph ^ 1u, P.status)) {
          ok = false;
          break;
        }
        tc::fence_after_thread_sync();
        const uint32_t d = tmem + static_cast<uint32_t>(ab * Npad);
        for (int kc = 0; kc < NK; ++kc) {
          if (!mbar_wait(&full[stage], ph, P.status)) {
            ok = false;
            break;
          }
          tc::fence_after_thread_sync();
          const uint32_t a0 = smem_addr(a_base + static_cast<size_t>(stage) * kStageBytes);
          const uint32_t b0 = smem_addr(e_base + static_cast<size_t>(kc) * Npad * 128);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc::mma_bf16(d, tc::sw128_kmajor_desc(a0 + j * 32), tc::sw128_kmajor_desc(b0 + j * 32),
                         idesc, (kc | j) != 0 ? 1u : 0u);
          tc::mma_commit(&empty[stage]);
          if (++stage == ns) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc::mma_commit(&acc_full[ab]);
      }
      if (!ok) atomicExch(fail_flag, 1);
      // every MMA this thread issued has completed before TMEM is freed
      tc::mma_commit(drain);
      (void)mbar_wait(drain, 0u, P.status);
    }
  } else {
    // ---- epilogue -------------------------------------------------------------
    const int q = warp & 3;          // TMEM lane quarter: rows 32q..32q+31 of a tile
    const int sub = (warp - 2) >> 2;
    const int c_begin = sub * CPW;   // batch columns [c_begin, c_begin + CPW)
    const int c_live = min(CPW, B - c_begin);  // columns below B (may be <= 0)
    const bool base_bf16 = P.base_bf16 != 0;
    const bool cache_bf16 = P.cache_bf16 != 0;
    const float* base_f = static_cast<const float*>(P.base);
    const uint16_t* base_h = static_cast<const uint16_t*>(P.base);
    float* cache_f = static_cast<float*>(P.cache);
    uint16_t* cache_h = static_cast<uint16_t*>(P.cache);
    uint32_t run_ord[kRegWinners ? CPW : 1];
    uint32_t run_v[kRegWinners ? CPW : 1];
#pragma unroll
    for (int j = 0; j < (kRegWinners ? CPW : 1); ++j) {
      run_ord[j] = 0u;
      run_v[j] = 0xFFFFFFFFu;
    }
    auto load_base = [&](int cb, int v, bool in_range, float (&bv)[4]) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int64_t bo = s_boff[cb + jj];  // warp-uniform
        bv[jj] = 0.f;
        if (bo >= 0 && in_range)
          bv[jj] = base_bf16 ? bf16_bits_to_float(__ldg(base_h + bo + v)) : __ldg(base_f + bo + v);
      }
    };
    // staged tile: element (b, row r) of slot ab at b * 128 + r
    auto smem_base = [&](int ab, int cb, int r, float (&bv)[4]) {
      const unsigned char* sb = base_s + ab * base_stride;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int b = cb + jj;
        bv[jj] = b < B ? (base_bf16 ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(sb)[b * kM + r])
                                    : reinterpret_cast<const float*>(sb)[b * kM + r])
                       : 0.f;
      }
    };
    for (int i = 0;; ++i) {
      const int t = blockIdx.x + i * G;
      if (t >= tiles) break;
      const int ab = i & 1;
      const uint32_t aph = (i >> 1) & 1;
      const int v = t * kM + q * 32 + lane;
      const bool in_range = v < V;
      // base logits of the first chunk, issued before the accumulator wait
      float bnext[4];
      if (!tma_base && c_live > 0) load_base(c_begin, v, in_range, bnext);
      if (!mbar_wait(&acc_full[ab], aph, P.status)) {
        atomicExch(fail_flag, 1);
        break;
      }
      if (tma_base && !mbar_wait(&base_full[ab], aph, P.status)) {
        atomicExch(fail_flag, 1);
        break;
      }
      tc::fence_after_thread_sync();
      if (tma_base && c_live > 0) smem_base(ab, c_begin, q * 32 + lane, bnext);
#pragma unroll
      for (int c = 0; c < CPW; c += 4) {
        if (c >= c_live) break;
        const int cb = c_begin + c;
        const float bv[4] = {bnext[0], bnext[1], bnext[2], bnext[3]};
        if (c + 4 < c_live) {
          if (tma_base)
            smem_base(ab, cb + 4, q * 32 + lane, bnext);
          else
            load_base(cb + 4, v, in_range, bnext);
        }
        uint32_t acc[4];
        tc::tmem_ld4(tmem + (static_cast<uint32_t>(q * 32) << 16) +
                         static_cast<uint32_t>(ab * Npad + cb),
                     acc);
        // Philox block of this lane quad's 4 columns, for request cb+(lane&3),
        // transposed so that nw[r] is this lane's noise for request cb+r
        const int bq = cb + (lane & 3);
        const U4 r = noise_block(s_seed[bq], s_npos[bq], static_cast<uint32_t>(v), kStreamDraft);
        uint32_t nw[4] = {r.x, r.y, r.z, r.w};
        quad_transpose(nw);
        const float4 ti4 = *reinterpret_cast<const float4*>(s_temp + cb);
        const float tinv[4] = {ti4.x, ti4.y, ti4.z, ti4.w};
        tc::tmem_wait_ld();
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
          if (jb >= c_live - c) break;  // warp-uniform
          const int b = cb + jb;
          const int64_t co = s_coff[b];  // warp-uniform
          uint32_t ord = 0u;
          if (s_boff[b] >= 0) {  // warp-uniform: a live request
            const float z = __fadd_rn(bv[jb], __uint_as_float(acc[jb]));
            float x = z, y = z;
            if (tinv[jb] > 0.f) {  // warp-uniform: sampled (x = z * (1/T))
              x = __fmul_rn(z, tinv[jb]);
              y = __fadd_rn(x, gumbel_of(nw[jb]));
            }
            if (co >= 0 && in_range) {
              if (cache_bf16)
                cache_h[co + v] = float_to_bf16_bits(x);
              else
                cache_f[co + v] = x;
            }
            ord = in_range ? ordered_bits(y) : 0u;  // every real value maps above 0
          }
          if constexpr (kRegWinners) {
            // rows of a lane only grow across tiles: a strict > keeps the
            // lowest row on ties
            if (ord > run_ord[c + jb]) {
              run_ord[c + jb] = ord;
              run_v[c + jb] = static_cast<uint32_t>(v);
            }
          } else {
            const unsigned long long key = warp_winner(ord, static_cast<uint32_t>(v));
            if (lane == 0 && key != 0ull) atomicMax(&best[b], key);
          }
        }
      }
      tc::fence_before_thread_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
    if constexpr (kRegWinners) {
#pragma unroll
      for (int j = 0; j < CPW; ++j) {
        if (j < c_live) {
          const unsigned long long key = warp_winner(run_ord[j], run_v[j]);
          if (lane == 0 && key != 0ull) atomicMax(&best[c_begin + j], key);
        }
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc::fence_after_thread_sync();
    tc::tmem_dealloc(tmem, tmem_cols);
  }

  // ---- publish this CTA's winners; the last CTA reduces -----------------------
  for (int b = tid; b < B; b += kThreadsTc)
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
  for (int b = tid; b < B; b += kThreadsTc) {
    unsigned long long m = 0ull;
    const unsigned long long* row = P.partials + static_cast<int64_t>(b) * G;
    for (int g2 = 0; g2 < G; ++g2) m = umax64(m, __ldcg(row + g2));
    const int32_t tok = (s_boff[b] >= 0 && m != 0ull) ? key_index(m) : -1;
    P.out_tokens[static_cast<int64_t>(b) * K + step] = tok;
  }
  if (tid == 0) *P.counter = 0u;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <int CPW>
cudaError_t launch_tc_cpw(const MarkovStepParams& p, const CUtensorMap& map,
                          const CUtensorMap& bmap, const MarkovTcPlan& plan, int grid,
                          cudaStream_t stream) {
  cudaError_t err = cudaFuncSetAttribute(markov_step_tc_kernel<CPW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(plan.smem));
  if (err != cudaSuccess) return err;
  markov_step_tc_kernel<CPW><<<grid, kThreadsTc, plan.smem, stream>>>(
      map, bmap, p, plan.Npad, plan.stages, plan.tmem_cols, plan.base_stage_bytes);
  return cudaGetLastError();
}

}  // namespace

bool markov_tc_plan(int B, int R, int base_elem_bytes, bool base_tma_ok, MarkovTcPlan* plan) {
  if (R % 64 != 0 || R > 512 || B < 1 || B > 256) return false;
  const int NK = R / 64;
  int Npad = (B + 15) & ~15;
  if (Npad < 16) Npad = 16;
  // stage the base logits through TMA when it leaves at least 4 w2 stages
  size_t bstage = base_tma_ok ? static_cast<size_t>(kM) * B * base_elem_bytes : 0;
  int ns = kMaxStages;
  while (ns >= 4 && TcLayout(Npad, NK, ns, bstage).total > kSmemLimit) --ns;
  if (TcLayout(Npad, NK, ns, bstage).total > kSmemLimit) {
    bstage = 0;
    ns = kMaxStages;
    while (ns >= 2 && TcLayout(Npad, NK, ns, 0).total > kSmemLimit) --ns;
  }
  if (ns < 2) return false;
  plan->base_stage_bytes = static_cast<unsigned>(bstage);
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(2 * Npad)) cols <<= 1;
  if (cols > 512) return false;
  plan->Npad = Npad;
  plan->stages = ns;
  plan->tmem_cols = cols;
  plan->smem = TcLayout(Npad, NK, ns, bstage).total;
  return true;
}

int markov_tc_make_tmap(void* tmap_out, const void* w2, int V, int R) {
  static_assert(sizeof(CUtensorMap) == 128, "CUtensorMap is 128 bytes");
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return -1;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(R), static_cast<cuuint64_t>(V)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(R) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kM)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = reinterpret_cast<EncodeTiledFn>(fn)(
      static_cast<CUtensorMap*>(tmap_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
      const_cast<void*>(w2), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -2;
}

int markov_tc_make_base_tmap(void* tmap_out, const void* base, bool bf16, int B, int K, int V) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return -1;
  const cuuint64_t es = bf16 ? 2 : 4;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(K),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(V) * es,
                                 static_cast<cuuint64_t>(V) * K * es};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kM), 1, static_cast<cuuint32_t>(B)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = reinterpret_cast<EncodeTiledFn>(fn)(
      static_cast<CUtensorMap*>(tmap_out),
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
      const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -2;
}

int markov_tc_max_grid(int V) { return (V + kM - 1) / kM; }

int markov_tc_grid(int V, int num_sms) {
  const int tiles = (V + kM - 1) / kM;
  return tiles < num_sms ? tiles : num_sms;
}

cudaError_t launch_markov_step_tc(const MarkovStepParams& p, const void* tmap, const void* bmap,
                                  const MarkovTcPlan& plan, int grid, cudaStream_t stream) {
  const CUtensorMap& map = *static_cast<const CUtensorMap*>(tmap);
  const CUtensorMap& bm = *static_cast<const CUtensorMap*>(bmap);
  const int cpw = plan.Npad / 4;
  if (cpw <= 4) return launch_tc_cpw<4>(p, map, bm, plan, grid, stream);
  if (cpw <= 8) return launch_tc_cpw<8>(p, map, bm, plan, grid, stream);
  if (cpw <= 16) return launch_tc_cpw<16>(p, map, bm, plan, grid, stream);
  return launch_tc_cpw<64>(p, map, bm, plan, grid, stream);
}

}  // namespace dspark
