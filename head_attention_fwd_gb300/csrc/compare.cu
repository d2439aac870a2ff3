// Device-side max |a - b| for the numeric-agreement guard (attn_compare):
// the online-softmax proposal page ("[WebGPU] Proposal: Add an option to use
// online softmax instead of naive softmax", §六) requires the online and the
// naive kernels to agree within a tolerance.

#include <string.h>

#include <atomic>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.h"

namespace attn {
namespace {

// Result words: each call takes the next one in turn, so that up to
// kSlots calls in flight at once (on different streams or host threads)
// accumulate into different words.  A word holds the bits of the running
// maximum (non-negative floats order like their bits; a NaN difference is
// recorded as +inf).
constexpr unsigned kSlots = 64;
__device__ unsigned g_max_bits[kSlots];
std::atomic<unsigned> g_next_slot{0};

__device__ __forceinline__ float load_as_float(const void* p, long long i, int dtype) {
  if (dtype == 1) return __half2float(static_cast<const __half*>(p)[i]);
  if (dtype == 2) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  return static_cast<const float*>(p)[i];
}

__global__ void clear_kernel(unsigned slot) { g_max_bits[slot] = 0u; }

__global__ void __launch_bounds__(256) max_abs_diff_kernel(const void* a, const void* b, long long n,
                                                           int dtype, unsigned slot) {
  float m = 0.f;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n; i += 256LL * gridDim.x) {
    const float d = fabsf(load_as_float(a, i, dtype) - load_as_float(b, i, dtype));
    m = (d == d) ? fmaxf(m, d) : INFINITY;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(&g_max_bits[slot], __float_as_uint(m));
}

}  // namespace

cudaError_t launch_max_abs_diff(const void* a, const void* b, long long n, int dtype, float* host_max,
                                cudaStream_t st) {
  const unsigned slot = g_next_slot.fetch_add(1u) % kSlots;
  clear_kernel<<<1, 1, 0, st>>>(slot);
  const long long blocks = (n + 255) / 256;
  max_abs_diff_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(a, b, n, dtype,
                                                                                             slot);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  unsigned bits = 0;
  if ((e = cudaMemcpyFromSymbolAsync(&bits, g_max_bits, sizeof bits, slot * sizeof(unsigned),
                                     cudaMemcpyDeviceToHost, st)) !=
      cudaSuccess)
    return e;
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return e;
  float f;
  memcpy(&f, &bits, sizeof f);
  *host_max = f;
  return cudaSuccess;
}

}  // namespace attn
