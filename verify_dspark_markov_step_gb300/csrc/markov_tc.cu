// markov_tc.cu -- one Markov step on the 5th-generation tensor cores.
//
// Same operation as markov_step.cu (the "DSparkSpeculator" page's
// _sample_markov_chain / _sample_logits; vLLM PR #65007 Part 1, per-step
// list), for batches where the bias projection [B, R] x [R, V] is a real
// dense contraction. markov_w2 rows are the M side of a tcgen05 MMA
// (M = 128 vocabulary rows per tile, K = markov_rank), the Markov embeddings
// of the batch are the N side (N = batch padded to a multiple of 16), and the
// fp32 accumulator lives in tensor memory.
//
// Persistent, warp-specialised CTA (one per SM):
//   warp 0      TMA producer: 128x64 bf16 boxes of markov_w2 (128-byte
//               swizzle) into a ring of shared-memory stages, L2 evict-last
//   warp 1      TMEM allocation; one thread issues the MMAs (4 per 64-wide K
//               chunk) into one of two accumulator buffers and commits
//   warps 2-17  epilogue: tcgen05.ld of the accumulator rows of their TMEM
//               lane quarter, bias add, temperature, Gumbel noise (one
//               Philox block per 4 columns, shared across a lane quad by a
//               4x4 shuffle transpose), cache store, and the winner of
//               each request over the warp's rows by two redux.sync
//               reductions (max of the ordered value bits, then min index),
//               kept per lane across tiles
// The per-CTA winners are reduced by the last CTA, as in markov_step.cu.
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

struct ReqInfoTc {
  float temperature;
  int32_t valid;
  int32_t prev;
  int32_t pad_;
  uint64_t seed;
  int64_t noise_pos;
  int64_t cache_off;
};

struct TcLayout {
  size_t a, e, info, best, bars, slot, flags, total;
  __host__ __device__ TcLayout(int B, int Npad, int NK, int ns) {
    a = 0;
    e = a + static_cast<size_t>(ns) * kStageBytes;
    info = e + static_cast<size_t>(NK) * Npad * 128;
    best = info + static_cast<size_t>(B) * sizeof(ReqInfoTc);
    bars = (best + static_cast<size_t>(Npad) * 8 + 7) & ~size_t(7);
    slot = bars + static_cast<size_t>(2 * ns + 5) * 8;
    flags = slot + 8;
    total = flags + 8 + kMaxStages * 4 + 1024;  // + slack to align the base to 1024 B
  }
};

__device__ __forceinline__ uint32_t sel4(const uint32_t (&w)[4], uint32_t i) {
  return i == 0 ? w[0] : (i == 1 ? w[1] : (i == 2 ? w[2] : w[3]));
}

// Lanes 4j..4j+3 each hold the four Philox words of request b0 + (lane & 3)
// for the same 4-column block. Afterwards out[r] = word (lane & 3) of
// request b0 + r, i.e. the noise of this lane's own column for request b0+r.
__device__ __forceinline__ void quad_transpose(const uint32_t (&w)[4], uint32_t (&out)[4]) {
  const uint32_t c = threadIdx.x & 3u;
  const int quad = static_cast<int>(threadIdx.x & 31u) & ~3;
#pragma unroll
  for (uint32_t r = 0; r < 4; ++r) {
    const uint32_t src = (c + r) & 3u;
    const uint32_t send = (c - r) & 3u;
    const uint32_t v = __shfl_sync(0xFFFFFFFFu, sel4(w, send), quad + static_cast<int>(src));
    out[0] = src == 0 ? v : out[0];
    out[1] = src == 1 ? v : out[1];
    out[2] = src == 2 ? v : out[2];
    out[3] = src == 3 ? v : out[3];
  }
}

template <int NK>  // markov_rank R = 64 * NK
__global__ void __launch_bounds__(kThreadsTc, 1)
markov_step_tc_kernel(const __grid_constant__ CUtensorMap tmap_w2, MarkovStepParams P, int Npad,
                      int ns, uint32_t tmem_cols) {
  constexpr int R = 64 * NK;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const TcLayout L(P.B, Npad, NK, ns);
  unsigned char* a_base = smem + L.a;
  unsigned char* e_base = smem + L.e;
  ReqInfoTc* info = reinterpret_cast<ReqInfoTc*>(smem + L.info);
  unsigned long long* best = reinterpret_cast<unsigned long long*>(smem + L.best);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + ns;
  uint64_t* acc_full = empty + ns;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.slot);
  int* fail_flag = reinterpret_cast<int*>(smem + L.flags);
  uint32_t* issued = reinterpret_cast<uint32_t*>(smem + L.flags + 8);  // last parity per stage

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = P.B, V = P.V, K = P.K, step = P.step;
  const int G = gridDim.x;
  const int tiles = (V + kM - 1) / kM;

  // ---- prologue ---------------------------------------------------------------
  for (int b = tid; b < B; b += kThreadsTc) {
    ReqInfoTc ri;
    ri.valid = 0;
    ri.prev = 0;
    ri.temperature = 0.f;
    ri.seed = 0;
    ri.noise_pos = 0;
    ri.cache_off = -1;
    ri.pad_ = 0;
    const int32_t s = P.rsi[b];
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
  }
  for (int n = tid; n < Npad; n += kThreadsTc) best[n] = 0ull;
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
    for (int i = 0; i < kMaxStages; ++i) issued[i] = 0xFFFFFFFFu;
    *fail_flag = 0;
    fence_mbar_init();
    tc::prefetch_tensormap(&tmap_w2);
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
      if (n < B && info[n].valid)
        val = __ldg(reinterpret_cast<const uint4*>(P.w1 + static_cast<int64_t>(info[n].prev) * R +
                                                   kc * 64) + cc);
      *reinterpret_cast<uint4*>(e_base + static_cast<size_t>(kc) * Npad * 128 + n * 128 +
                                ((cc ^ (n & 7)) << 4)) = val;
    }
  }
  fence_proxy_async_smem();
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer -----------------------------------------------------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int t = blockIdx.x + i * G;
        if (t >= tiles) break;
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
    // Warp (q, sub) owns TMEM lane quarter q (rows 32q..32q+31 of a tile) and
    // the batch columns [sub * Npad/4, (sub + 1) * Npad/4), in chunks of 4.
    const int q = warp & 3;
    const int sub = (warp - 2) >> 2;
    const int cols = Npad >> 2;                 // a multiple of 4, at most 64
    const int c_begin = sub * cols, c_end = c_begin + cols;
    const bool base_bf16 = P.base_bf16 != 0;
    const bool cache_bf16 = P.cache_bf16 != 0;
    // running winner of column c_begin + 32*j + lane, j = 0, 1
    unsigned long long run0 = 0ull, run1 = 0ull;
    for (int i = 0;; ++i) {
      const int t = blockIdx.x + i * G;
      if (t >= tiles) break;
      const int ab = i & 1;
      const uint32_t aph = (i >> 1) & 1;
      if (!mbar_wait(&acc_full[ab], aph, P.status)) {
        atomicExch(fail_flag, 1);
        break;
      }
      tc::fence_after_thread_sync();
      const int v = t * kM + q * 32 + lane;
      const bool in_range = v < V;
      // base logits of the next chunk are loaded before the current chunk is
      // processed
      float bnext[4];
      auto load_base = [&](int cb, float (&bv)[4]) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int b = cb + jj;
          bv[jj] = 0.f;
          if (b < B && in_range && info[b].valid)
            bv[jj] = load_logit(P.base, base_bf16, (static_cast<int64_t>(b) * K + step) * V + v);
        }
      };
      load_base(c_begin, bnext);
      for (int cb = c_begin; cb < c_end; cb += 4) {
        if (cb >= B) break;
        float bv[4] = {bnext[0], bnext[1], bnext[2], bnext[3]};
        if (cb + 4 < c_end && cb + 4 < B) load_base(cb + 4, bnext);
        uint32_t acc[4];
        tc::tmem_ld4(tmem + (static_cast<uint32_t>(q * 32) << 16) +
                         static_cast<uint32_t>(ab * Npad + cb),
                     acc);
        // Philox block of this lane quad's 4 columns, for request cb+(lane&3)
        const int bq = cb + (lane & 3);
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (bq < B) {
          const U4 r = noise_block(info[bq].seed, info[bq].noise_pos, static_cast<uint32_t>(v),
                                   kStreamDraft);
          w[0] = r.x;
          w[1] = r.y;
          w[2] = r.z;
          w[3] = r.w;
        }
        uint32_t nw[4] = {0u, 0u, 0u, 0u};
        quad_transpose(w, nw);
        tc::tmem_wait_ld();
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
          const int b = cb + jb;
          if (b >= B) break;
          const ReqInfoTc& ri = info[b];
          uint32_t ord = 0u;
          if (ri.valid && in_range) {
            const float z = __fadd_rn(bv[jb], __uint_as_float(acc[jb]));
            float x = z, y = z;
            if (ri.temperature > 0.f) {
              x = ri.temperature == 1.0f ? z : __fdiv_rn(z, ri.temperature);
              y = __fadd_rn(x, gumbel_of(nw[jb]));
            }
            if (ri.cache_off >= 0) {
              if (cache_bf16)
                static_cast<uint16_t*>(P.cache)[ri.cache_off + v] = float_to_bf16_bits(x);
              else
                static_cast<float*>(P.cache)[ri.cache_off + v] = x;
            }
            ord = ordered_bits(y);  // every real value maps above 0
          }
          // winner of this column over the warp's 32 rows: largest value,
          // then lowest row
          const uint32_t omax = __reduce_max_sync(0xFFFFFFFFu, ord);
          const uint32_t cand = (ord == omax && ord != 0u) ? static_cast<uint32_t>(v) : 0xFFFFFFFFu;
          const uint32_t vmin = __reduce_min_sync(0xFFFFFFFFu, cand);
          if (omax != 0u) {
            const unsigned long long key =
                (static_cast<unsigned long long>(omax) << 32) | (0xFFFFFFFFu - vmin);
            const int slot = b - c_begin;
            if ((slot & 31) == lane) {
              if (slot < 32)
                run0 = umax64(run0, key);
              else
                run1 = umax64(run1, key);
            }
          }
        }
      }
      tc::fence_before_thread_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
    if (lane < cols && c_begin + lane < B && run0) atomicMax(&best[c_begin + lane], run0);
    if (lane + 32 < cols && c_begin + lane + 32 < B && run1)
      atomicMax(&best[c_begin + lane + 32], run1);
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
    const int32_t tok = (info[b].valid && m != 0ull) ? key_index(m) : -1;
    P.out_tokens[static_cast<int64_t>(b) * K + step] = tok;
  }
  if (tid == 0) *P.counter = 0u;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

bool markov_tc_plan(int B, int R, MarkovTcPlan* plan) {
  if (R % 64 != 0 || R > 512 || B < 1 || B > 256) return false;
  const int NK = R / 64;
  int Npad = (B + 15) & ~15;
  if (Npad < 16) Npad = 16;
  int ns = kMaxStages;
  while (ns >= 2 && TcLayout(B, Npad, NK, ns).total > kSmemLimit) --ns;
  if (ns < 2) return false;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(2 * Npad)) cols <<= 1;
  if (cols > 512) return false;
  plan->Npad = Npad;
  plan->stages = ns;
  plan->tmem_cols = cols;
  plan->smem = TcLayout(B, Npad, NK, ns).total;
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

int markov_tc_grid(int V, int num_sms) {
  const int tiles = (V + kM - 1) / kM;
  return tiles < num_sms ? tiles : num_sms;
}

cudaError_t launch_markov_step_tc(const MarkovStepParams& p, const void* tmap,
                                  const MarkovTcPlan& plan, int grid, cudaStream_t stream) {
  const CUtensorMap& map = *static_cast<const CUtensorMap*>(tmap);
  const int nk = p.R / 64;
  cudaError_t err = cudaSuccess;
  switch (nk) {
#define DSPARK_TC_CASE(N)                                                                  \
  case N:                                                                                  \
    err = cudaFuncSetAttribute(markov_step_tc_kernel<N>,                                   \
                               cudaFuncAttributeMaxDynamicSharedMemorySize,                \
                               static_cast<int>(plan.smem));                               \
    if (err != cudaSuccess) return err;                                                    \
    markov_step_tc_kernel<N><<<grid, kThreadsTc, plan.smem, stream>>>(map, p, plan.Npad,   \
                                                                      plan.stages,         \
                                                                      plan.tmem_cols);     \
    break;
    DSPARK_TC_CASE(1)
    DSPARK_TC_CASE(2)
    DSPARK_TC_CASE(3)
    DSPARK_TC_CASE(4)
    DSPARK_TC_CASE(5)
    DSPARK_TC_CASE(6)
    DSPARK_TC_CASE(7)
    DSPARK_TC_CASE(8)
#undef DSPARK_TC_CASE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace dspark
