// fp32 -> fp16 / bf16 conversion of Q, K and V for attn_fwd_mixed.
//
// "WebGPU 算子优化：QKV 内存合并与 FlashAttention 分块计算",
// §浏览器端落地的关键参数与监控, runs the score products in 16-bit with
// fp32 softmax statistics and a 16-bit output.  attn_fwd_mixed accepts fp32
// Q, K, V and rounds them to the 16-bit type once, here, before the fused
// kernel: the fused kernel loads each K/V tile once per query block, so a
// conversion inside it would repeat the work for every block of the head.
//
// HBM-bound: each element is read once (4 bytes) and written once (2 bytes).
// One thread converts 8 consecutive elements per step (two 16-byte loads,
// one 16-byte store); blockIdx.y selects the tensor.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.h"

namespace attn {
namespace {

template <bool BF16>
__device__ __forceinline__ uint32_t cvt2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

template <bool BF16>
__global__ void __launch_bounds__(256) convert3_kernel(const float* __restrict__ q, const float* __restrict__ k,
                                                       const float* __restrict__ v, uint16_t* __restrict__ out,
                                                       long long n8, long long out_stride) {
  const float* src = blockIdx.y == 0 ? q : (blockIdx.y == 1 ? k : v);
  uint16_t* dst = out + blockIdx.y * out_stride;
  const float4* s4 = reinterpret_cast<const float4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (long long g = blockIdx.x * 256LL + threadIdx.x; g < n8; g += 256LL * gridDim.x) {
    const float4 a = __ldcs(s4 + 2 * g), b = __ldcs(s4 + 2 * g + 1);  // read once: streaming
    d4[g] = make_uint4(cvt2<BF16>(a.x, a.y), cvt2<BF16>(a.z, a.w), cvt2<BF16>(b.x, b.y), cvt2<BF16>(b.z, b.w));
  }
}

}  // namespace

cudaError_t launch_convert3(const ConvertLaunch& a, cudaStream_t st) {
  if (a.n % 8 != 0 || a.n <= 0) return cudaErrorInvalidValue;
  const long long n8 = a.n / 8;
  const long long want = (n8 + 255) / 256;
  const long long cap = static_cast<long long>(a.num_sms > 0 ? a.num_sms : 1) * 8;  // 8 blocks of 256 per SM
  const dim3 grid(static_cast<unsigned>(want < cap ? want : cap), 3);
  if (a.bf16)
    convert3_kernel<true><<<grid, 256, 0, st>>>(a.q, a.k, a.v, a.out, n8, a.out_stride);
  else
    convert3_kernel<false><<<grid, 256, 0, st>>>(a.q, a.k, a.v, a.out, n8, a.out_stride);
  return cudaGetLastError();
}

}  // namespace attn
