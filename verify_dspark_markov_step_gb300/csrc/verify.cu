// verify.cu -- the verifier's helpers outside the main kernel: workspace
// sizes, and the device noise generator and temperature division exposed on
// their own so that tests can check them against other implementations.
//
// The verification itself (vLLM PR #65007 Part 2: temperature, exact top-p,
// the rejection sampler with residual resampling and the bonus token) is one
// persistent kernel in verify_stats.cu, its draws in verify_draw.cuh.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "verify_common.cuh"

namespace dspark {

namespace {

__global__ void noise_kernel(const uint64_t* seed, const int64_t* pos, const uint32_t* col,
                             const uint32_t* stream_word, uint32_t* word, float* u, float* g,
                             int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const U4 r = noise_block(seed[i], pos[i], col[i], stream_word[i]);
    const uint32_t w = pick_word(r, col[i] & 3u);
    if (word) word[i] = w;
    if (u) u[i] = uniform_of(w);
    if (g) g[i] = gumbel_of(w);
  }
}

// The drafter's temperature step (temp_div2) on independent (z, T) pairs.
__global__ void temperature_divide_kernel(const float* z, const float* T, float* x, int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float t = T[i];
    float x0, x1;
    f2_unpack(temp_div2(f2_pack(z[i], z[i]), f2_pack(__frcp_rn(t), __frcp_rn(t)),
                        f2_pack(-t, -t), !temp_div_t_ok(t)),
              x0, x1);
    x[i] = x0;
  }
}

}  // namespace

cudaError_t launch_temperature_divide(const float* z, const float* T, float* x, int64_t n,
                                      cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  int blocks = static_cast<int>((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  temperature_divide_kernel<<<blocks, 256, 0, stream>>>(z, T, x, n);
  return cudaGetLastError();
}

size_t verify_tstats_bytes(int B, int K) {
  return static_cast<size_t>(B) * (K + 1) * sizeof(TgtStats);
}
size_t verify_dstats_bytes(int B, int K) {
  return static_cast<size_t>(B) * K * sizeof(DrfStats);
}
int verify_max_chunks(int V) { return (V + 1023) / 1024; }
cudaError_t launch_noise(const uint64_t* seed, const int64_t* pos, const uint32_t* col,
                         const uint32_t* stream_word, uint32_t* word, float* u, float* g,
                         int64_t n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  int blocks = static_cast<int>((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  noise_kernel<<<blocks, 256, 0, stream>>>(seed, pos, col, stream_word, word, u, g, n);
  return cudaGetLastError();
}

}  // namespace dspark
