// markov_tc.cu -- the K-step Markov sampling loop on the 5th-generation
// tensor cores, all K steps in one persistent, cooperative launch.
//
// The "DSparkSpeculator" page's _sample_markov_chain / _sample_logits and
// vLLM PR #65007 Part 1 (per-step list): Markov embedding of the previous
// token, the markov_w2 bias projection, bias add, temperature, Gumbel noise
// keyed by (seed, position - 1, column), the block-argmax winner rule and the
// draft-logits cache store, fused; the steps are chained on the device.
//
// The bias projection [B, R] x [R, V] runs on the tensor cores for every
// batch size: each step is bound by streaming markov_w2 and the logits and by
// the epilogue's ALU work, and the MMA takes the B * R multiply-adds per
// column off the epilogue warps (for small B the padding of N to 16 costs
// nothing). markov_w2 rows are the M side of a tcgen05 MMA (M = 128
// vocabulary rows per tile, K = markov_rank), the Markov embeddings of the
// batch are the N side (N = batch padded to a multiple of 16), and the fp32
// accumulator lives in tensor memory.
//
// One CTA per SM, warp-specialised; the CTAs sweep the vocabulary tiles once
// per step, forward on even steps and backward on odd ones (the tiles a step
// ends on, still in L2, start the next), and the pipeline runs across step
// boundaries:
//   warp 0      TMA producer of markov_w2: 128x64 bf16 boxes (128-byte
//               swizzle) into a ring of up to 12 shared-memory stages, L2
//               evict-last, as far ahead as the ring allows (into the next
//               step while the current one is being finished).
//   warp 18     TMA producer of the base logits: per tile, the tile's logits
//               of every request for that step (a 128 x 1 x B box of the
//               [B, K, V] tensor) into one of up to 8 slots, L2 evict-first;
//               for large batches the epilogue reads them from global memory.
//   warp 1      TMEM allocation; one thread issues the MMAs (4 per 64-wide K
//               chunk) into one of 2-4 accumulator buffers and commits; it
//               waits for the step's Markov embeddings before its first tile.
//   warps 2-17  epilogue: warp (q, sub) owns TMEM lane quarter q (32 rows of
//               each tile) and a fixed set of CPW batch columns. Per group of
//               4 columns: one tcgen05.ld and one Philox block (a lane quad
//               shares its 4 blocks by a 4x4 butterfly transpose); per pair of
//               columns, in packed fp32 pairs: Gumbel noise, bias add and
//               noise add; temperature x = z / T correctly rounded (an FMA
//               correction of z * rn(1/T)), compiled into a second version of
//               the tile loop that only warps holding a column with T other
//               than 1 run (T = 1 and greedy columns keep x = z); per column:
//               cache store and the running winner -- per lane in registers
//               across tiles when CPW <= 16, else reduced per tile with
//               redux.sync.
// At the end of a step each CTA folds its winners into the step's global
// winner keys (64-bit atomicMax), then a grid barrier (an arrival counter,
// bounded wait) lets every CTA read the step's tokens, gather the next Markov
// embeddings w1[token] into shared memory and release the MMA warp.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cfloat>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace dspark {

namespace {

constexpr int kM = 128;                 // vocabulary rows per tile (UMMA M)
constexpr int kStageBytes = kM * 128;   // one 64-element K chunk of a tile
constexpr int kEpiWarps = 16;           // four per TMEM lane quarter (warps 2..17)
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kBaseWarp = 2 + kEpiWarps;  // TMA producer of the base logits
constexpr int kThreadsTc = 32 * (kBaseWarp + 1);
constexpr int kMaxStages = 12;
constexpr int kMaxAcc = 4;              // accumulator buffers in TMEM
constexpr int kMaxBaseSlots = 8;        // staged base tiles
constexpr size_t kSmemLimit = 227u * 1024u;

struct TcCfg {
  int Npad;                   // batch padded to a multiple of 16 (UMMA N)
  int ns;                     // markov_w2 ring stages of 16 KB
  int na;                     // accumulator buffers (na * Npad TMEM columns)
  int nb;                     // staged base tiles (0: base logits read directly)
  uint32_t tmem_cols;
  uint32_t base_stage_bytes;  // bytes of one staged base tile
};

__host__ __device__ inline size_t base_slot_stride(size_t base_stage) {
  return (base_stage + 1023) & ~size_t(1023);
}

// Shared-memory layout (offsets from a 1024-byte aligned base).
struct TcLayout {
  size_t a, e, bases, xs, gs, rcp, seed, npos, bptr, cptr, cb0, prev, act, best, wkey, wx, ws,
      cm, cs, bars, slot, flags, total;
  __host__ __device__ TcLayout(int Npad, int NK, int ns, int nb, size_t base_stage) {
    a = 0;                                                       // markov_w2 ring
    e = a + static_cast<size_t>(ns) * kStageBytes;               // Markov embeddings
    bases = e + static_cast<size_t>(NK) * Npad * 128;            // staged base tiles
    xs = bases + static_cast<size_t>(nb) * base_slot_stride(base_stage);
    gs = xs + static_cast<size_t>(Npad) * 4;
    rcp = gs + static_cast<size_t>(Npad) * 4;
    seed = rcp + static_cast<size_t>(Npad) * 4;                  // per request:
    npos = seed + static_cast<size_t>(Npad) * 8;                 //   noise position
    bptr = npos + static_cast<size_t>(Npad) * 8;                 //   base row of the step
    cptr = bptr + static_cast<size_t>(Npad) * 8;                 //   cache row of the step
    cb0 = cptr + static_cast<size_t>(Npad) * 8;                  //   cache row of step 0
    prev = cb0 + static_cast<size_t>(Npad) * 8;                  //   token feeding the step
    act = prev + static_cast<size_t>(Npad) * 4;
    best = act + static_cast<size_t>(Npad) * 4;
    wkey = best + static_cast<size_t>(Npad) * 8;                 // per lane quarter: winner key,
    wx = wkey + static_cast<size_t>(4 * Npad) * 8;               //   cache-row maximum key,
    ws = wx + static_cast<size_t>(4 * Npad) * 4;                 //   its exp-sum
    cm = ws + static_cast<size_t>(4 * Npad) * 4;                 // per request: the CTA's
    cs = cm + static_cast<size_t>(Npad) * 4;                     //   row maximum key, exp-sum
    bars = cs + static_cast<size_t>(Npad) * 4;
    slot = bars + static_cast<size_t>(2 * kMaxStages + 2 * kMaxAcc + 2 * kMaxBaseSlots + 2) * 8;
    flags = slot + 8;
    total = flags + 16 + 1024;  // + slack to align the base to 1024 B
  }
};

// Lanes 4j..4j+3 each hold the four Philox words of request b0 + (lane & 3)
// for the same 4-column block (a 4x4 matrix, one row per lane). A two-round
// butterfly transposes it: afterwards w[r] = word (lane & 3) of request
// b0 + r, i.e. the noise of this lane's own column for request b0 + r.
__device__ __forceinline__ void quad_transpose(uint32_t* w) {
  const uint32_t c = threadIdx.x & 3u;
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

__device__ __forceinline__ void epi_bar() {  // the epilogue warps only
  asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const unsigned int* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Stores without a branch: the predicate travels into the instruction.
__device__ __forceinline__ void st_pred(float* p, float v, bool pred) {
  asm volatile("{ .reg .pred q; setp.ne.u32 q, %2, 0; @q st.global.f32 [%0], %1; }" ::"l"(p),
               "f"(v), "r"(static_cast<uint32_t>(pred))
               : "memory");
}
__device__ __forceinline__ void st_pred_bits(uint16_t* p, uint16_t h, bool pred) {
  asm volatile("{ .reg .pred q; setp.ne.u32 q, %2, 0; @q st.global.u16 [%0], %1; }" ::"l"(p),
               "h"(h), "r"(static_cast<uint32_t>(pred))
               : "memory");
}
// The value of an order key (0, the empty key, reads as -inf).
__device__ __forceinline__ float key_to_float(uint32_t k) {
  if (k == 0u) return -INFINITY;
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Loads without a branch: 0 where the predicate is false.
__device__ __forceinline__ float ld_pred(const float* p, bool pred) {
  float v;
  asm volatile("{ .reg .pred q; setp.ne.u32 q, %2, 0; mov.f32 %0, 0f00000000; @q ld.global.nc.f32 %0, [%1]; }"
               : "=f"(v)
               : "l"(p), "r"(static_cast<uint32_t>(pred)));
  return v;
}
__device__ __forceinline__ float ld_pred(const uint16_t* p, bool pred) {
  unsigned short h;
  asm volatile("{ .reg .pred q; setp.ne.u32 q, %2, 0; mov.u16 %0, 0; @q ld.global.nc.u16 %0, [%1]; }"
               : "=h"(h)
               : "l"(p), "r"(static_cast<uint32_t>(pred)));
  return bf16_bits_to_float(h);
}

// A CTA's share of the vocabulary tiles: n_full whole tiles blockIdx.x + j * G
// and, when the tile count is not a multiple of the grid, possibly one
// remainder tile tx of which it takes half the request columns (half_id 0:
// the first two epilogue column groups, 1: the last two); two CTAs share
// each remainder tile, so no CTA has a whole tile more than another.
struct TileShare {
  int n_loc, n_full, tx, half_id;
  __device__ TileShare(int tiles, int G, bool split) {
    const int bx = static_cast<int>(blockIdx.x);
    const int nb = tiles / G, rem = tiles - nb * G;
    if (split && rem > 0 && 2 * rem <= G) {
      n_full = nb;
      const bool has = bx < 2 * rem;
      n_loc = nb + (has ? 1 : 0);
      tx = has ? nb * G + (bx < rem ? bx : bx - rem) : -1;
      half_id = bx < rem ? 0 : 1;
    } else {
      n_full = n_loc = nb + (bx < rem ? 1 : 0);
      tx = -1;
      half_id = 0;
    }
  }
};

// Position of loop iteration g = step * n_loc + il of a CTA: its j-th tile
// with j rising on even steps and falling on odd ones (so a step starts on
// the tile the previous one ended on, still in L2), and the slot/parity of a
// ring of n buffers, advanced without integer division.
struct TileIter {
  int step, il, t, n_loc, n_full, tx, G;
  bool half;  // the remainder tile: this CTA takes half its columns
  __device__ TileIter(const TileShare& sh, int G_)
      : step(0), il(0), n_loc(sh.n_loc), n_full(sh.n_full), tx(sh.tx), G(G_) {
    locate();
  }
  __device__ __forceinline__ void locate() {
    const int j = (step & 1) ? n_loc - 1 - il : il;
    half = j >= n_full;
    t = half ? tx : static_cast<int>(blockIdx.x) + j * G;
  }
  __device__ __forceinline__ bool first() const { return il == 0; }
  __device__ __forceinline__ bool last() const { return il == n_loc - 1; }
  __device__ __forceinline__ void next() {
    if (++il == n_loc) {
      il = 0;
      ++step;
    }
    locate();
  }
};
struct RingPos {
  int slot, n;
  uint32_t phase;
  __device__ explicit RingPos(int n_) : slot(0), n(n_), phase(0u) {}
  __device__ __forceinline__ void next() {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

template <int GW>
__device__ __forceinline__ void tmem_load_group(uint32_t taddr, uint32_t (&r)[GW]) {
  if constexpr (GW == 8) {
    tc::tmem_ld8(taddr, r);
  } else {
    tc::tmem_ld4(taddr, r);
  }
}

// CPW: batch columns per epilogue warp; kStats: record each cache row's
// maximum and exp-mass (a separate instantiation, so that a loop without
// them carries none of their registers or instructions)
template <int CPW, bool kBaseBf16, bool kCacheBf16, bool kStats>
__global__ void __launch_bounds__(kThreadsTc, 1)
markov_loop_tc_kernel(const __grid_constant__ CUtensorMap tmap_w2,
                      const __grid_constant__ CUtensorMap tmap_base, MarkovStepParams P,
                      TcCfg cfg) {
  constexpr bool kRegWinners = CPW <= 16;
  constexpr int GW = 4;  // columns per TMEM load and Philox group
  const int Npad = cfg.Npad, ns = cfg.ns, na = cfg.na, nb = cfg.nb;
  const int R = P.R;
  const int NK = R / 64;
  const bool tma_base = nb != 0;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const TcLayout L(Npad, NK, ns, nb, cfg.base_stage_bytes);
  unsigned char* a_base = smem + L.a;
  unsigned char* e_base = smem + L.e;
  unsigned char* base_s = smem + L.bases;  // nb staged base tiles [B][128]
  const size_t base_stride = base_slot_stride(cfg.base_stage_bytes);
  float* s_xs = reinterpret_cast<float*>(smem + L.xs);  // x = z / xs: T, or 1 (T = 1, greedy)
  float* s_gs = reinterpret_cast<float*>(smem + L.gs);  // y = x + gs * g: 1, or 0 (greedy)
  float* s_rcp = reinterpret_cast<float*>(smem + L.rcp);  // rn(1 / xs)
  uint64_t* s_seed = reinterpret_cast<uint64_t*>(smem + L.seed);
  int64_t* s_npos = reinterpret_cast<int64_t*>(smem + L.npos);      // P0 + step - 1
  const unsigned char** s_bptr = reinterpret_cast<const unsigned char**>(smem + L.bptr);
  unsigned char** s_cptr = reinterpret_cast<unsigned char**>(smem + L.cptr);  // null: no store
  unsigned char** s_cb0 = reinterpret_cast<unsigned char**>(smem + L.cb0);
  // cache-row statistics are recorded by the register-winner epilogue (up to
  // kRowStatsMaxBatch requests); wider batches report them unknown (NaN)
  static_assert(!kStats || 4 * CPW <= kRowStatsMaxBatch, "row statistics batch limit");
  constexpr bool kRowStats = kStats;
  const bool want_stats = kStats && P.draft_stats != nullptr;
  int32_t* s_prev = reinterpret_cast<int32_t*>(smem + L.prev);
  int32_t* s_act = reinterpret_cast<int32_t*>(smem + L.act);        // request live
  unsigned long long* best = reinterpret_cast<unsigned long long*>(smem + L.best);
  // register-winner epilogue: one winner per (TMEM lane quarter, request)
  unsigned long long* s_wkey = reinterpret_cast<unsigned long long*>(smem + L.wkey);
  uint32_t* s_wx = reinterpret_cast<uint32_t*>(smem + L.wx);
  float* s_ws = reinterpret_cast<float*>(smem + L.ws);
  uint32_t* s_cm = reinterpret_cast<uint32_t*>(smem + L.cm);
  float* s_cs = reinterpret_cast<float*>(smem + L.cs);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kMaxStages;
  uint64_t* acc_full = empty + kMaxStages;
  uint64_t* acc_empty = acc_full + kMaxAcc;
  uint64_t* bfull = acc_empty + kMaxAcc;
  uint64_t* bempty = bfull + kMaxBaseSlots;
  uint64_t* drain = bempty + kMaxBaseSlots;
  uint64_t* e_ready = drain + 1;  // one phase per step
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.slot);
  volatile int* fail_flag = reinterpret_cast<volatile int*>(smem + L.flags);
  volatile int* stop_word = fail_flag + 1;  // the epilogue's decision at a step end

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = P.B, V = P.V, K = P.K;
  const int G = gridDim.x;
  const int tiles = (V + kM - 1) / kM;
  // remainder tiles are split by request columns when the last two column
  // groups hold live requests
  const TileShare share(tiles, G, B > 2 * CPW);
  const int n_loc = share.n_loc;  // tiles of this CTA
  const int n_iter = n_loc * K;   // (step, tile) pairs, step-major
  using BaseT = typename std::conditional<kBaseBf16, uint16_t, float>::type;
  using CacheT = typename std::conditional<kCacheBf16, uint16_t, float>::type;
  constexpr int bes = sizeof(BaseT);
  constexpr int ces = sizeof(CacheT);

  // ---- prologue: per-request state (thread n < Npad owns column n) -----------
  if (tid < Npad) {
    const int n = tid;
    float tdiv = 1.f, gscale = 0.f;
    uint64_t seed = 0;
    int64_t npos = 0;
    const unsigned char* bp = nullptr;
    unsigned char* cp = nullptr;
    int32_t prev = -1;
    const int32_t s = n < B ? P.rsi[n] : -1;
    if (s >= 0) {
      if (s >= P.S) {
        report(P.status, DSPARK_ERR_BOUNDS);
      } else {
        const int32_t pv = P.anchor[n];
        bool ok = pv >= 0 && pv < V;
        if (!ok) report(P.status, DSPARK_ERR_BOUNDS);
        int64_t row = -1;
        if (ok && P.cache != nullptr) {
          row = P.row_map ? P.row_map[s] : s;
          if (row < 0 || row >= P.C) {
            report(P.status, DSPARK_ERR_BOUNDS);
            ok = false;
          }
        }
        if (ok) {
          const float T = P.temperature[s];
          if (T > 0.f) {  // sampled; a greedy column keeps x = z and no noise
            tdiv = T;
            gscale = 1.f;
          }
          seed = P.seeds[s];
          npos = P.pos[n] - 1;
          bp = static_cast<const unsigned char*>(P.base) +
               static_cast<int64_t>(n) * K * V * bes;
          if (row >= 0)
            cp = static_cast<unsigned char*>(P.cache) + row * K * static_cast<int64_t>(V) * ces;
          prev = pv;
        }
      }
    }
    s_xs[n] = tdiv;
    s_rcp[n] = __frcp_rn(tdiv);
    s_gs[n] = gscale;
    s_seed[n] = seed;
    s_npos[n] = npos;
    s_bptr[n] = bp;
    s_cptr[n] = cp;
    s_cb0[n] = cp;
    s_prev[n] = prev;
    s_act[n] = prev >= 0;
    best[n] = 0ull;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) s_wkey[qq * Npad + n] = 0ull;
  }
  if (tid == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < na; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps);
    }
    for (int i = 0; i < nb; ++i) {
      mbar_init(&bfull[i], 1);
      mbar_init(&bempty[i], kEpiWarps);
    }
    mbar_init(drain, 1);
    mbar_init(e_ready, 1);
    *fail_flag = 0;
    *stop_word = 0;
    fence_mbar_init();
    tc::prefetch_tensormap(&tmap_w2);
    if (tma_base) tc::prefetch_tensormap(&tmap_base);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, cfg.tmem_cols);
    tc::tmem_relinquish();
  }
  __syncthreads();

  // Markov embeddings e[n] = w1[prev_n] as the N-side operand, K-major,
  // 128-byte swizzle: chunk c of row n of K-chunk kc at n*128 + (c ^ (n%8))*16.
  auto gather_e = [&](int t0, int nt) {
    const int per_row = NK * 8;
    const int total = Npad * per_row;
    for (int c = t0; c < total; c += nt) {
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
    fence_proxy_async_smem();  // generic writes -> visible to the tensor core
  };
  gather_e(tid, kThreadsTc);
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  if (tid == 0) mbar_arrive(e_ready);  // step 0's embeddings are in place
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer of markov_w2: as far ahead as the ring allows ------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      uint32_t issued[kMaxStages];  // parity of the last copy per stage
#pragma unroll
      for (int i = 0; i < kMaxStages; ++i) issued[i] = 0xFFFFFFFFu;
      TileIter it(share, G);
      for (int g = 0; g < n_iter && ok; ++g, it.next()) {
        if (*fail_flag) break;
        const int t = it.t;
        for (int kc = 0; kc < NK; ++kc) {
          if (!mbar_wait(&empty[stage], ph ^ 1u, P.status, P.wait_limit_ns)) {
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
      if (!ok) *fail_flag = 1;
      // every copy this CTA issued has landed before the CTA may exit
      for (int s2 = 0; s2 < ns; ++s2)
        if (issued[s2] != 0xFFFFFFFFu) (void)mbar_wait(&full[s2], issued[s2], P.status, P.wait_limit_ns);
    }
  } else if (warp == kBaseWarp) {
    // ---- TMA producer of the base logits: one [B] x 128 box per tile ------------
    if (lane == 0 && tma_base) {
      const uint64_t pol_stream = policy_evict_first();
      uint32_t last[kMaxBaseSlots];
#pragma unroll
      for (int i = 0; i < kMaxBaseSlots; ++i) last[i] = 0xFFFFFFFFu;
      TileIter it(share, G);
      RingPos br(nb);
      for (int g = 0; g < n_iter; ++g, it.next(), br.next()) {
        if (*fail_flag) break;
        const int step = it.step;
        const int t = it.t;
        const int bs = br.slot;
        const uint32_t bph = br.phase;
        if (!mbar_wait(&bempty[bs], bph ^ 1u, P.status, P.wait_limit_ns)) {
          *fail_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&bfull[bs], cfg.base_stage_bytes);
        tc::tma_load_3d(base_s + bs * base_stride, &tmap_base, t * kM, step, 0, &bfull[bs],
                        pol_stream);
        last[bs] = bph;
      }
      for (int bs = 0; bs < nb; ++bs)
        if (last[bs] != 0xFFFFFFFFu) (void)mbar_wait(&bfull[bs], last[bs], P.status, P.wait_limit_ns);
    }
  } else if (warp == 1) {
    // ---- MMA issuer -------------------------------------------------------------
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(kM, Npad);
      const uint64_t a_desc0 = tc::sw128_kmajor_desc(smem_addr(a_base));
      const uint64_t b_desc0 = tc::sw128_kmajor_desc(smem_addr(e_base));
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      TileIter it(share, G);
      RingPos ar(na);
      for (int g = 0; g < n_iter && ok; ++g, it.next(), ar.next()) {
        if (*fail_flag) break;
        if (it.first()) {  // first tile of a step: wait for its embeddings
          if (!mbar_wait(e_ready, static_cast<uint32_t>(it.step) & 1u, P.status, P.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc::fence_after_thread_sync();
        }
        const int ab = ar.slot;
        if (!mbar_wait(&acc_empty[ab], ar.phase ^ 1u, P.status, P.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc::fence_after_thread_sync();
        const uint32_t d = tmem + static_cast<uint32_t>(ab * Npad);
        for (int kc = 0; kc < NK; ++kc) {
          if (!mbar_wait(&full[stage], ph, P.status, P.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc::fence_after_thread_sync();
          // the descriptor's address field is (address >> 4): a 32-byte K
          // step adds 2, a stage or a K chunk its byte offset >> 4
          const uint64_t ad = a_desc0 + static_cast<uint32_t>((stage * kStageBytes) >> 4);
          const uint64_t bd = b_desc0 + static_cast<uint32_t>((kc * Npad * 128) >> 4);
          tc::mma_bf16(d, ad, bd, idesc, kc != 0 ? 1u : 0u);
#pragma unroll
          for (int j = 1; j < 4; ++j) tc::mma_bf16(d, ad + 2 * j, bd + 2 * j, idesc, 1u);
          tc::mma_commit(&empty[stage]);
          if (++stage == ns) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc::mma_commit(&acc_full[ab]);
      }
      if (!ok) *fail_flag = 1;
      // every MMA this thread issued has completed before TMEM is freed
      tc::mma_commit(drain);
      (void)mbar_wait(drain, 0u, P.status, P.wait_limit_ns);
    }
  } else {
    // ---- epilogue (warps 2..17) -----------------------------------------------
    const int etid = tid - 64;       // 0..511 among the epilogue threads
    const int q = warp & 3;          // TMEM lane quarter: rows 32q..32q+31 of a tile
    const int sub = (warp - 2) >> 2;
    const int c_begin = sub * CPW;   // batch columns [c_begin, c_begin + CPW)
    const int c_live = min(CPW, B - c_begin);  // columns below B (may be <= 0)
    const int r = q * 32 + lane;     // this lane's row of a tile
    float run_xm[kRegWinners ? CPW : 1];  // running maximum of the stored values
    float run_s[kRowStats ? CPW : 1];     // their sum of exp(x - run_xm), fp32
    uint32_t run_ord[kRegWinners ? CPW : 1];
    uint32_t run_v[kRegWinners ? CPW : 1];
#pragma unroll
    for (int j = 0; j < (kRegWinners ? CPW : 1); ++j) {
      run_ord[j] = 0u;
      run_v[j] = 0xFFFFFFFFu;
      run_xm[j] = -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < (kRowStats ? CPW : 1); ++j) run_s[j] = 0.0f;
    const unsigned long long l2e2 = f2_pack(kLog2e, kLog2e);
    // base logits straight from global memory (no staged tile)
    auto load_direct = [&](int cb, int v, bool in_range, float (&bv)[GW]) {
#pragma unroll
      for (int j = 0; j < GW; ++j) {
        const BaseT* bp = reinterpret_cast<const BaseT*>(s_bptr[cb + j]);  // null: not live
        bv[j] = ld_pred(bp + v, bp != nullptr && in_range);
      }
    };
    // Philox blocks of this lane quad's 4 columns for the requests of group
    // [cb, cb + GW): block h for request cb + 4h + (lane & 3), transposed so
    // that nw[4h + i] is this lane's noise for request cb + 4h + i
    auto noise_group = [&](int cb, int v, uint32_t (&nw)[GW]) {
#pragma unroll
      for (int h = 0; h < GW / 4; ++h) {
        const int bq = cb + 4 * h + (lane & 3);
        const U4 blk = noise_block(s_seed[bq], s_npos[bq], static_cast<uint32_t>(v),
                                   kStreamDraft);
        nw[4 * h + 0] = blk.x;
        nw[4 * h + 1] = blk.y;
        nw[4 * h + 2] = blk.z;
        nw[4 * h + 3] = blk.w;
        quad_transpose(nw + 4 * h);
      }
    };
    // this warp's columns: does any divide by a temperature other than 1,
    // and does any such temperature lie outside the fast division's range
    bool wdiv = false, wslow = false;
    for (int j = 0; j < CPW; ++j) {
      const float T = s_xs[c_begin + j];
      wdiv |= T != 1.f;
      wslow |= T != 1.f && !temp_div_t_ok(T);
    }
    bool skip = false;  // set after a failed wait: the warp then only walks the loop
    TileIter it(share, G);
    RingPos ar(na), br(tma_base ? nb : 1);
    for (int g = 0; g < n_iter; ++g, it.next(), ar.next(), br.next()) {
      const int step = it.step;
      const int t = it.t;
      const int ab = ar.slot;
      const uint32_t aph = ar.phase;
      const int bs = br.slot;
      const uint32_t bph = br.phase;
      const int v = t * kM + r;
      const bool in_range = v < V;
      // live columns of this warp in this tile: none in the other half of a
      // shared remainder tile
      const int c_tile = (it.half && (sub >> 1) != share.half_id) ? 0 : c_live;
      float bnext[GW];
      if (!skip && !tma_base && c_tile > 0) {
        load_direct(c_begin, v, in_range, bnext);
        // the next tile's base rows of this warp's columns into L2 (one
        // 32-row line per column), so that its direct loads hit L2
        if (!it.last()) {
          TileIter nx = it;
          nx.next();
          const int vn = nx.t * kM + q * 32;
          if (vn < V) {
            for (int l = lane; l < c_live; l += 32) {
              const unsigned char* bp = s_bptr[c_begin + l];
              if (bp != nullptr)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(
                    bp + static_cast<size_t>(vn) * sizeof(BaseT)));
            }
          }
        }
      }
      // the noise of this tile's first column group does not depend on the
      // step's tokens: with one group per warp (small batches) draw it before
      // waiting for the accumulator (at a step's first tile the wait covers
      // the embedding gather and the MMA chain); wider warps draw it in turn
      constexpr bool kPreNoise = CPW <= GW;
      float gpre[GW];
      if (kPreNoise && !skip && c_tile > 0) {
        uint32_t nw0[GW];
        noise_group(c_begin, v, nw0);
#pragma unroll
        for (int j = 0; j < GW; j += 2) gumbel_of2(nw0[j], nw0[j + 1], gpre[j], gpre[j + 1]);
      }
      if (!skip) {
        bool ok = mbar_wait(&acc_full[ab], aph, P.status, P.wait_limit_ns);
        if (ok && tma_base) ok = mbar_wait(&bfull[bs], bph, P.status, P.wait_limit_ns);
        if (!ok) {
          *fail_flag = 1;
          skip = true;
        }
      }
      // One tile; kRev = the step walks its tiles backward (ties then go to
      // the later, lower row); kDiv = some column divides by T != 1.
      auto tile = [&](auto rev_tag, auto div_tag) {
        constexpr bool kRev = decltype(rev_tag)::value;
        constexpr bool kDiv = decltype(div_tag)::value;
        static_cast<void>(kRev);  // only the register winners depend on the order
        const unsigned char* sb = base_s + bs * base_stride;
#pragma unroll
        for (int c = 0; c < CPW; c += GW) {
          if (c >= c_tile) break;  // warp-uniform
          const int cb = c_begin + c;
          uint32_t acc[GW];
          tmem_load_group<GW>(tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                  static_cast<uint32_t>(ab * Npad + cb),
                              acc);
          float bv[GW];
          if (tma_base) {
            // rows of padding columns (b >= B) read row B - 1: their results are unused
#pragma unroll
            for (int j = 0; j < GW; ++j) {
              const int bb = min(cb + j, B - 1);
              const BaseT raw = reinterpret_cast<const BaseT*>(sb)[bb * kM + r];
              if constexpr (kBaseBf16)
                bv[j] = bf16_bits_to_float(raw);
              else
                bv[j] = raw;
            }
          } else {
#pragma unroll
            for (int j = 0; j < GW; ++j) bv[j] = bnext[j];
            if (c + GW < c_tile) load_direct(cb + GW, v, in_range, bnext);
          }
          float gv[GW];
          if (kPreNoise && c == 0) {
#pragma unroll
            for (int j = 0; j < GW; ++j) gv[j] = gpre[j];
          } else {
            uint32_t nw[GW];
            noise_group(cb, v, nw);
#pragma unroll
            for (int j = 0; j < GW; j += 2) gumbel_of2(nw[j], nw[j + 1], gv[j], gv[j + 1]);
          }
          float gsc[GW];
#pragma unroll
          for (int h = 0; h < GW / 4; ++h) {
            const float4 g4 = *reinterpret_cast<const float4*>(s_gs + cb + 4 * h);
            gsc[4 * h + 0] = g4.x;
            gsc[4 * h + 1] = g4.y;
            gsc[4 * h + 2] = g4.z;
            gsc[4 * h + 3] = g4.w;
          }
          // z = base + bias, x = z / T (T = 1 and greedy: z), y = x + g
          // (greedy: x), two columns at a time in packed fp32 pairs (fewer
          // instructions and registers); padding columns (b >= B) compute
          // values that are neither stored nor folded into a token
          tc::tmem_wait_ld();
          float xv[GW], yv[GW];
          float tq[GW], rq[GW];
          if constexpr (kDiv) {
#pragma unroll
            for (int h = 0; h < GW / 4; ++h) {
              const float4 t4 = *reinterpret_cast<const float4*>(s_xs + cb + 4 * h);
              const float4 r4 = *reinterpret_cast<const float4*>(s_rcp + cb + 4 * h);
              tq[4 * h + 0] = -t4.x;
              tq[4 * h + 1] = -t4.y;
              tq[4 * h + 2] = -t4.z;
              tq[4 * h + 3] = -t4.w;
              rq[4 * h + 0] = r4.x;
              rq[4 * h + 1] = r4.y;
              rq[4 * h + 2] = r4.z;
              rq[4 * h + 3] = r4.w;
            }
          }
#pragma unroll
          for (int j = 0; j < GW; j += 2) {
            unsigned long long x = f2_add(f2_pack(bv[j], bv[j + 1]),
                                          f2_pack(__uint_as_float(acc[j]),
                                                  __uint_as_float(acc[j + 1])));
            // x = z / T (T = 1 and greedy columns: z / 1 = z)
            if constexpr (kDiv)
              x = temp_div2(x, f2_pack(rq[j], rq[j + 1]), f2_pack(tq[j], tq[j + 1]), wslow);
            const unsigned long long y =
                f2_fma(f2_pack(gv[j], gv[j + 1]), f2_pack(gsc[j], gsc[j + 1]), x);
            f2_unpack(x, xv[j], xv[j + 1]);
            f2_unpack(y, yv[j], yv[j + 1]);
          }
#pragma unroll
          for (int j = 0; j < GW; ++j) {
            const int b = cb + j;
            const float x = xv[j];
            const float y = yv[j];
            CacheT* cp = reinterpret_cast<CacheT*>(s_cptr[b]);      // null: no store
            float xr;  // the value as stored (a bf16 cache rounds it)
            if constexpr (kCacheBf16) {
              const uint16_t h = float_to_bf16_bits(x);
              st_pred_bits(cp + v, h, cp != nullptr && in_range);
              xr = bf16_bits_to_float(h);
            } else {
              st_pred(cp + v, x, cp != nullptr && in_range);
              xr = x;
            }
            // the stored value, NaN and rows past V read as -inf
            xr = in_range ? fmaxf(xr, -INFINITY) : -INFINITY;
            if constexpr (kRowStats) {
              // running maximum and exp-sum of the cache row's values this
              // lane stores: both terms rescaled to the new maximum (the
              // base is finite even for an all -inf start, so every exp of
              // -inf is 0, never NaN)
              const float nm = fmaxf(run_xm[c + j], xr);
              const float base = fmaxf(nm, -FLT_MAX);
              float ea, eb;
              f2_unpack(f2_mul(f2_sub(f2_pack(run_xm[c + j], xr), f2_pack(base, base)), l2e2),
                        ea, eb);
              run_s[c + j] = __fmaf_rn(run_s[c + j], ex2_approx(ea), ex2_approx(eb));
              run_xm[c + j] = nm;
            }
            const uint32_t ord = in_range ? ordered_key(y) : 0u;  // real values map above 0
            if constexpr (kRegWinners) {
              // a lane's rows grow (shrink) across a forward (backward)
              // step: > (>=) keeps the lowest row on ties
              if (kRev ? ord >= run_ord[c + j] : ord > run_ord[c + j]) {
                run_ord[c + j] = ord;
                run_v[c + j] = static_cast<uint32_t>(v);
              }
            } else {
              // the warp's winner into its lane quarter's slot of the
              // column: the warp alone writes it (no atomic)
              const unsigned long long key = warp_winner(ord, static_cast<uint32_t>(v));
              if (lane == 0) {
                unsigned long long* sl = &s_wkey[q * Npad + b];
                if (key > *sl) *sl = key;
              }
            }
          }
        }
      };
      if (!skip) {
        tc::fence_after_thread_sync();
        if (wdiv) {
          if (kRegWinners && (step & 1))
            tile(std::true_type{}, std::true_type{});
          else
            tile(std::false_type{}, std::true_type{});
        } else {
          if (kRegWinners && (step & 1))
            tile(std::true_type{}, std::false_type{});
          else
            tile(std::false_type{}, std::false_type{});
        }
        tc::fence_before_thread_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&acc_empty[ab]);
          if (tma_base) mbar_arrive(&bempty[bs]);
        }
      }
      if (!it.last()) continue;

      // ---- end of a step: fold winners, grid barrier, tokens, next embeddings ----
      if constexpr (kRegWinners) {
        // the warp's winner per request column into this lane quarter's slot
        // (plain stores, independent reductions)
        uint32_t om[CPW], vm[CPW], xm[CPW];
#pragma unroll
        for (int j = 0; j < CPW; ++j) om[j] = __reduce_max_sync(0xFFFFFFFFu, run_ord[j]);
#pragma unroll
        for (int j = 0; j < CPW; ++j)
          vm[j] = __reduce_min_sync(0xFFFFFFFFu, (run_ord[j] == om[j] && om[j] != 0u)
                                                     ? run_v[j]
                                                     : 0xFFFFFFFFu);
#pragma unroll
        for (int j = 0; j < CPW; ++j)
          xm[j] = want_stats ? __reduce_max_sync(0xFFFFFFFFu, ordered_key(run_xm[j])) : 0u;
        // the warp's exp-sum of each column, rescaled to the warp's maximum
        // (a butterfly of fp32 additions: lane 0's result is the same bits
        // every run)
        float xs_w[CPW];
#pragma unroll
        for (int j = 0; j < CPW; ++j) {
          float t = 0.0f;
          if constexpr (kRowStats) {
            if (want_stats) {
            const float mw = fmaxf(key_to_float(xm[j]), -FLT_MAX);
            t = __fmul_rn(run_s[j], exp_rel(run_xm[j], mw));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t = __fadd_rn(t, __shfl_xor_sync(0xFFFFFFFFu, t, o));
            }
          }
          xs_w[j] = t;
        }
        if (lane == 0 && !skip) {
#pragma unroll
          for (int j = 0; j < CPW; ++j) {
            if (j < c_live) {
              s_wkey[q * Npad + c_begin + j] =
                  om[j] == 0u ? 0ull
                              : (static_cast<unsigned long long>(om[j]) << 32) |
                                    (0xFFFFFFFFu - vm[j]);
              if constexpr (kRowStats) {
                s_wx[q * Npad + c_begin + j] = xm[j];
                s_ws[q * Npad + c_begin + j] = xs_w[j];
              }
            }
          }
        }
#pragma unroll
        for (int j = 0; j < CPW; ++j) {
          run_ord[j] = 0u;
          run_v[j] = 0xFFFFFFFFu;
          run_xm[j] = -INFINITY;
          if constexpr (kRowStats) run_s[j] = 0.0f;
        }
      }
      epi_bar();
      const bool last = step + 1 == K;
      unsigned long long* keys = P.keys + static_cast<size_t>(step) * B;
      for (int b = etid; b < B; b += kEpiThreads) {
        unsigned long long k;
        uint32_t xk;
        if constexpr (kRegWinners) {
          k = umax64(umax64(s_wkey[b], s_wkey[Npad + b]),
                     umax64(s_wkey[2 * Npad + b], s_wkey[3 * Npad + b]));
          xk = kRowStats ? max(max(s_wx[b], s_wx[Npad + b]),
                               max(s_wx[2 * Npad + b], s_wx[3 * Npad + b]))
                         : 0u;
        } else {
          k = umax64(umax64(s_wkey[b], s_wkey[Npad + b]),
                     umax64(s_wkey[2 * Npad + b], s_wkey[3 * Npad + b]));
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) s_wkey[qq * Npad + b] = 0ull;
          xk = 0u;
        }
        if (k != 0ull) atomicMax(keys + b, k);
        // the cache row's maximum, as an order key in the scratch word; the
        // CTA's exp-sum of the row, rescaled to the CTA's maximum (lane
        // quarters in a fixed order), kept for after the barrier
        if (want_stats && s_cb0[b] != nullptr) {
          atomicMax(&P.draft_stats[static_cast<int64_t>(b) * K + step].scratch, xk);
          const float mc = fmaxf(key_to_float(xk), -FLT_MAX);
          float sc = 0.0f;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq)
            sc = __fadd_rn(sc, __fmul_rn(s_ws[qq * Npad + b],
                                         exp_rel(key_to_float(s_wx[qq * Npad + b]), mc)));
          s_cm[b] = xk;
          s_cs[b] = sc;
        }
      }
      epi_bar();
      if (etid == 0) {
        // one decision for all epilogue warps: stop at the first failure
        int stop = *fail_flag;
        if (!stop) {
          __threadfence();  // the block's key updates before its arrival
          atomicAdd(P.counter, 1u);
        }
        // the last step's tokens are needed by CTA 0 alone; its row
        // maxima (for the exp-sums) by every CTA
        if (!stop && (!last || blockIdx.x == 0 || want_stats)) {
          const unsigned int target =
              static_cast<unsigned int>(step + 1) * static_cast<unsigned int>(G) +
              P.barrier_extra;
          const unsigned long long t0 = globaltimer_ns();
          while (ld_acquire_u32(P.counter) < target) {
            __nanosleep(32);
            if (globaltimer_ns() - t0 > P.wait_limit_ns) {
              report(P.status, DSPARK_ERR_TIMEOUT);
              *fail_flag = 1;
              stop = 1;
              break;
            }
          }
          __threadfence();
        }
        *stop_word = stop;
      }
      epi_bar();
      if (*stop_word) break;  // uniform over the epilogue
      if (want_stats) {
        // every CTA has folded its maxima: add this CTA's exp-sum of each
        // row, rescaled to the row's maximum, in fixed point (2^40 per
        // unit); integer additions, so the total is the same in any order
        for (int b = etid; b < B; b += kEpiThreads) {
          if (s_cb0[b] == nullptr) continue;
          dspark_row_stats* st = &P.draft_stats[static_cast<int64_t>(b) * K + step];
          const float mg = fmaxf(key_to_float(__ldcg(&st->scratch)), -FLT_MAX);
          const float part =
              __fmul_rn(__fmul_rn(s_cs[b], exp_rel(key_to_float(s_cm[b]), mg)), 0x1p40f);
          const unsigned long long f = __float2ull_rn(part);
          if (f != 0ull) atomicAdd(reinterpret_cast<unsigned long long*>(&st->mass), f);
        }
      }
      if (last && blockIdx.x != 0) break;  // uniform over the epilogue
      for (int b = etid; b < Npad; b += kEpiThreads) {
        int32_t tok = -1;
        if (b < B && s_act[b]) {
          const unsigned long long m = __ldcg(keys + b);
          if (m != 0ull) tok = key_index(m);
        }
        if (blockIdx.x == 0 && b < B) {
          P.out_tokens[static_cast<int64_t>(b) * K + step] = tok;
          if (P.draft_stats != nullptr && s_cb0[b] != nullptr) {  // the row's maximum
            dspark_row_stats* st = &P.draft_stats[static_cast<int64_t>(b) * K + step];
            st->m = want_stats ? key_to_float(__ldcg(&st->scratch)) : __int_as_float(0x7FC00000);
          }
        }
        s_prev[b] = tok;
        s_act[b] = tok >= 0;
        if (!last) {  // advance the per-request state to the next step
          s_npos[b] += 1;
          if (tok >= 0) {
            if (s_bptr[b] != nullptr) s_bptr[b] += static_cast<int64_t>(V) * bes;
            if (s_cptr[b] != nullptr) s_cptr[b] += static_cast<int64_t>(V) * ces;
          } else {
            s_bptr[b] = nullptr;
            s_cptr[b] = nullptr;
          }
        }
      }
      if (!last) {
        epi_bar();
        gather_e(etid, kEpiThreads);
        tc::fence_before_thread_sync();
        epi_bar();
        if (etid == 0) mbar_arrive(e_ready);  // the MMA warp may start the next step
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc::fence_after_thread_sync();
    tc::tmem_dealloc(tmem, cfg.tmem_cols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <int CPW, bool kBaseBf16, bool kCacheBf16, bool kStats>
cudaError_t launch_tc_cpw(const MarkovStepParams& p, const CUtensorMap& map,
                          const CUtensorMap& bmap, const MarkovTcPlan& plan, int grid,
                          cudaStream_t stream) {
  cudaError_t err = cudaFuncSetAttribute(markov_loop_tc_kernel<CPW, kBaseBf16, kCacheBf16, kStats>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(plan.smem));
  if (err != cudaSuccess) return err;
  TcCfg cfg;
  cfg.Npad = plan.Npad;
  cfg.ns = plan.stages;
  cfg.na = plan.acc_buffers;
  cfg.nb = plan.base_slots;
  cfg.tmem_cols = plan.tmem_cols;
  cfg.base_stage_bytes = plan.base_stage_bytes;
  // cooperative: every CTA is resident at once, which the grid barrier
  // between steps relies on
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  lc.blockDim = dim3(kThreadsTc, 1, 1);
  lc.dynamicSmemBytes = plan.smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, markov_loop_tc_kernel<CPW, kBaseBf16, kCacheBf16, kStats>, map,
                            bmap, p,
                            cfg);
}

template <int CPW, bool kStats>
cudaError_t launch_tc_dtypes(const MarkovStepParams& p, const CUtensorMap& map,
                             const CUtensorMap& bmap, const MarkovTcPlan& plan, int grid,
                             cudaStream_t stream) {
  if (p.base_bf16) {
    return p.cache_bf16 ? launch_tc_cpw<CPW, true, true, kStats>(p, map, bmap, plan, grid, stream)
                        : launch_tc_cpw<CPW, true, false, kStats>(p, map, bmap, plan, grid, stream);
  }
  return p.cache_bf16 ? launch_tc_cpw<CPW, false, true, kStats>(p, map, bmap, plan, grid, stream)
                      : launch_tc_cpw<CPW, false, false, kStats>(p, map, bmap, plan, grid, stream);
}

}  // namespace

bool markov_tc_plan(int B, int R, int base_elem_bytes, bool base_tma_ok, MarkovTcPlan* plan) {
  if (R % 64 != 0 || R > 512 || B < 1 || B > 256) return false;
  const int NK = R / 64;
  int Npad = (B + 15) & ~15;
  if (Npad < 16) Npad = 16;
  int na = 512 / Npad;  // accumulator buffers: as many as TMEM holds, up to 4
  if (na > kMaxAcc) na = kMaxAcc;
  if (na < 2) return false;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(na * Npad)) cols <<= 1;
  if (cols > 512) return false;
  auto max_stages = [&](int nb, size_t bstage) {
    int ns = kMaxStages;
    while (ns > 0 && TcLayout(Npad, NK, ns, nb, bstage).total > kSmemLimit) --ns;
    return ns;
  };
  // Stage the base logits through TMA when that leaves a deep markov_w2 ring:
  // the most base slots that keep 8 ring stages, else that keep 4.
  int ns = 0, nb = 0;
  size_t bstage = 0;
  if (base_tma_ok) {
    const size_t bt = static_cast<size_t>(kM) * B * base_elem_bytes;
    const int slot_choices[] = {8, 6, 4, 3, 2};
    const int min_stages[] = {8, 4};
    for (int min_ns : min_stages) {
      for (int cand : slot_choices) {
        const int s = max_stages(cand, bt);
        if (s >= min_ns) {
          ns = s;
          nb = cand;
          break;
        }
      }
      if (nb != 0) break;
    }
    if (nb != 0) bstage = bt;
  }
  if (nb == 0) {
    ns = max_stages(0, 0);
    if (ns < 2) return false;
  }
  plan->Npad = Npad;
  plan->stages = ns;
  plan->acc_buffers = na;
  plan->base_slots = nb;
  plan->base_stage_bytes = static_cast<unsigned>(bstage);
  plan->tmem_cols = cols;
  plan->smem = TcLayout(Npad, NK, ns, nb, bstage).total;
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

int markov_tc_grid(int V, int num_sms) {
  const int tiles = (V + kM - 1) / kM;
  return tiles < num_sms ? tiles : num_sms;
}

cudaError_t launch_markov_loop_tc(const MarkovStepParams& p, const void* tmap, const void* bmap,
                                  const MarkovTcPlan& plan, int grid, cudaStream_t stream) {
  const CUtensorMap& map = *static_cast<const CUtensorMap*>(tmap);
  const CUtensorMap& bm = *static_cast<const CUtensorMap*>(bmap);
  const int cpw = plan.Npad / 4;
  // row statistics: asked for, and a batch the register epilogue records
  const bool stats = p.draft_stats != nullptr && cpw <= kRowStatsMaxBatch / 4;
  if (cpw <= 4)
    return stats ? launch_tc_dtypes<4, true>(p, map, bm, plan, grid, stream)
                 : launch_tc_dtypes<4, false>(p, map, bm, plan, grid, stream);
  if (cpw <= 8)
    return stats ? launch_tc_dtypes<8, true>(p, map, bm, plan, grid, stream)
                 : launch_tc_dtypes<8, false>(p, map, bm, plan, grid, stream);
  if (cpw <= 16) return launch_tc_dtypes<16, false>(p, map, bm, plan, grid, stream);
  if (cpw <= 32) return launch_tc_dtypes<32, false>(p, map, bm, plan, grid, stream);
  return launch_tc_dtypes<64, false>(p, map, bm, plan, grid, stream);
}

}  // namespace dspark

