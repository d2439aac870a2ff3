// The two softmax passes of the unfused comparison path.
//
// The online-softmax proposal page ("[WebGPU] Proposal: Add an option to use
// online softmax instead of naive softmax", §三) describes the naive softmax
// as two dispatches, each a full read of the score matrix from global memory:
// the first finds each row's maximum and exp-sum, the second writes the
// normalised probabilities.  "Transformer算子生态深度分析" ch.2 §2.3 gives the
// three steps (max, sum of exp(s - max), divide); §2.5 explains why keeping
// S and A in device memory is the bottleneck.  These kernels do exactly that,
// one CTA per score row, so that the fused kernel has an honest baseline.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.h"

namespace attn {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float block_reduce(float x, bool is_max, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float y = __shfl_xor_sync(0xffffffffu, x, o);
    x = is_max ? fmaxf(x, y) : x + y;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red[] may still be read by a previous reduction
  if (lane == 0) red[warp] = x;
  __syncthreads();
  x = red[lane < kThreads / 32 ? lane : 0];
  if (lane >= kThreads / 32) x = is_max ? -INFINITY : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float y = __shfl_xor_sync(0xffffffffu, x, o);
    x = is_max ? fmaxf(x, y) : x + y;
  }
  return x;
}

// pass 1: m = max_j s_j, l = sum_j exp(s_j - m)
__global__ void __launch_bounds__(kThreads) row_stats_kernel(const float* __restrict__ s, float* m_out,
                                                             float* l_out, int n, long long ld) {
  __shared__ float red[kThreads / 32];
  const float* row = s + blockIdx.x * ld;
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < n; j += kThreads) mx = fmaxf(mx, row[j]);
  mx = block_reduce(mx, true, red);
  float sum = 0.f;
  for (int j = threadIdx.x; j < n; j += kThreads) sum += expf(row[j] - mx);
  sum = block_reduce(sum, false, red);
  if (threadIdx.x == 0) {
    m_out[blockIdx.x] = mx;
    l_out[blockIdx.x] = sum;
  }
}

// pass 2: p_j = exp(s_j - m) / l, stored in the 16-bit input type
template <bool BF16>
__global__ void __launch_bounds__(kThreads) normalise_kernel(const float* __restrict__ s, void* p,
                                                             const float* m_in, const float* l_in,
                                                             float* lse, int n, long long ld) {
  const float* row = s + blockIdx.x * ld;
  const float mx = m_in[blockIdx.x], inv = 1.f / l_in[blockIdx.x];
  if (BF16) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p) + blockIdx.x * ld;
    for (int j = threadIdx.x; j < n; j += kThreads) out[j] = __float2bfloat16_rn(expf(row[j] - mx) * inv);
  } else {
    __half* out = static_cast<__half*>(p) + blockIdx.x * ld;
    for (int j = threadIdx.x; j < n; j += kThreads) out[j] = __float2half_rn(expf(row[j] - mx) * inv);
  }
  if (lse && threadIdx.x == 0) lse[blockIdx.x] = mx + logf(l_in[blockIdx.x]);
}

}  // namespace

cudaError_t launch_naive_softmax(const NaiveSoftmaxLaunch& a, cudaStream_t st) {
  if (a.rows < 1 || a.rows > 0x7fffffffLL) return cudaErrorInvalidValue;
  const unsigned grid = static_cast<unsigned>(a.rows);
  row_stats_kernel<<<grid, kThreads, 0, st>>>(a.s, a.m, a.l, a.n, a.ld);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.bf16)
    normalise_kernel<true><<<grid, kThreads, 0, st>>>(a.s, a.p, a.m, a.l, a.lse, a.n, a.ld);
  else
    normalise_kernel<false><<<grid, kThreads, 0, st>>>(a.s, a.p, a.m, a.l, a.lse, a.n, a.ld);
  return cudaGetLastError();
}

}  // namespace attn
