// fp32 attention forward on the CUDA cores (exact fp32 FMA, no tensor cores:
// TF32 would not hold a 1e-4 error bound).
//
// Same online-softmax recurrence as the tensor-core kernel
// ("Transformer算子生态深度分析" ch.2 §2.6), with a block of 32 keys: each warp
// owns one query row; lane l scores key l of the current block, the block
// max and exp-sum are combined with warp shuffles, and the running output
// (features split over the lanes) is rescaled by exp(m_old - m) before the
// block's p·V is added.  K and V blocks are staged in shared memory once per
// CTA and shared by its 8 warps (8 query rows of one head).

#include "common.h"

namespace attn {
namespace {

constexpr int kWarps = 8;
constexpr int kKeys = 32;        // keys per block (one per lane)
constexpr int kMaxD = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Params {
  const float *q, *k, *v;
  float* o;
  float* lse;
  long long sb, sh, ss;
  int H, S, d, n_qblk;
  float c;  // scale · log2(e)
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// MAXD: the largest head dimension of the instance (64, 128 or 256), which
// sizes the per-thread load buffers and output accumulators.
template <int MAXD>
__global__ void __launch_bounds__(kWarps * 32) simt_fwd_kernel(const Params p) {
  constexpr int kPerLaneD = MAXD / 32;
  constexpr int kLoadsD = kKeys * MAXD / (kWarps * 32);  // block elements per thread, at most
  extern __shared__ float sm[];
  const int dp = p.d + 1;                 // padded row: lane-per-key reads hit distinct banks
  float* sk = sm;                         // [kKeys][dp]
  float* sv = sm + kKeys * dp;            // [kKeys][dp]
  float* sq = sv + kKeys * dp;            // [kWarps][d]
  float* sp = sq + kWarps * p.d;          // [kWarps][kKeys]: each warp's probabilities of the block

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qblk = blockIdx.x % p.n_qblk;
  const int bh = blockIdx.x / p.n_qblk;
  const int b = bh / p.H, hh = bh % p.H;
  const int row = qblk * kWarps + warp;
  const bool active = row < p.S;
  const long long base = b * p.sb + hh * p.sh;

  float* q_s = sq + warp * p.d;
  float* p_s = sp + warp * kKeys;
  for (int e = lane; e < p.d; e += 32) q_s[e] = active ? p.q[base + row * p.ss + e] : 0.f;

  // K and V blocks are loaded one block ahead into registers, so that their
  // memory latency overlaps the previous block's arithmetic.
  float kr[kLoadsD], vr[kLoadsD];
  auto load_block = [&](int j0) {
    const int nk = min(kKeys, p.S - j0);
#pragma unroll
    for (int u = 0; u < kLoadsD; ++u) {
      const int i = threadIdx.x + u * kWarps * 32;
      const int r = i / p.d, e = i - r * p.d;
      const bool in = i < kKeys * p.d && r < nk;
      kr[u] = in ? __ldg(p.k + base + (j0 + r) * p.ss + e) : 0.f;
      vr[u] = in ? __ldg(p.v + base + (j0 + r) * p.ss + e) : 0.f;
    }
  };
  load_block(0);

  float m = -INFINITY, l = 0.f;
  float acc[kPerLaneD];
#pragma unroll
  for (int t = 0; t < kPerLaneD; ++t) acc[t] = 0.f;

  for (int j0 = 0; j0 < p.S; j0 += kKeys) {
    __syncthreads();  // previous block fully consumed (and q_s written)
    const int nk = min(kKeys, p.S - j0);
#pragma unroll
    for (int u = 0; u < kLoadsD; ++u) {
      const int i = threadIdx.x + u * kWarps * 32;
      if (i < kKeys * p.d) {
        const int r = i / p.d, e = i - r * p.d;
        sk[r * dp + e] = kr[u];
        sv[r * dp + e] = vr[u];
      }
    }
    __syncthreads();
    if (j0 + kKeys < p.S) load_block(j0 + kKeys);
    // score of key (j0 + lane), in log2 units: four independent fp32 FMA
    // chains over the features, then their sum
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    const float* kl = sk + lane * dp;
    int e = 0;
    for (; e + 4 <= p.d; e += 4) {
      s0 = fmaf(q_s[e], kl[e], s0);
      s1 = fmaf(q_s[e + 1], kl[e + 1], s1);
      s2 = fmaf(q_s[e + 2], kl[e + 2], s2);
      s3 = fmaf(q_s[e + 3], kl[e + 3], s3);
    }
    for (; e < p.d; ++e) s0 = fmaf(q_s[e], kl[e], s0);
    float s = (s0 + s1) + (s2 + s3);
    s = lane < nk ? s * p.c : -INFINITY;
    const float m_new = fmaxf(m, warp_max(s));
    const float alpha = exp2f(m - m_new);  // 0 while m = -inf
    const float pj = exp2f(s - m_new);     // 0 for the missing keys
    l = l * alpha + warp_sum(pj);
    m = m_new;
#pragma unroll
    for (int t = 0; t < kPerLaneD; ++t) acc[t] *= alpha;
    // O += p·V_block: p broadcast from shared memory, lane = feature
    p_s[lane] = pj;
    __syncwarp();
#pragma unroll 4
    for (int kk = 0; kk < nk; ++kk) {
      const float pk = p_s[kk];
#pragma unroll
      for (int t = 0; t < kPerLaneD; ++t) {
        const int ee = lane + 32 * t;
        if (ee < p.d) acc[t] = fmaf(pk, sv[kk * dp + ee], acc[t]);
      }
    }
    __syncwarp();  // p_s is rewritten by the next block
  }
  if (!active) return;
  const float inv = 1.f / l;
#pragma unroll
  for (int t = 0; t < kPerLaneD; ++t) {
    const int e = lane + 32 * t;
    if (e < p.d) p.o[base + row * p.ss + e] = acc[t] * inv;
  }
  if (p.lse && lane == 0)
    p.lse[(static_cast<long long>(b) * p.H + hh) * p.S + row] = (m + log2f(l)) * kLn2;
}

}  // namespace

cudaError_t launch_simt_fwd(const SimtLaunch& a, cudaStream_t st) {
  if (a.d < 1 || a.d > kMaxD) return cudaErrorInvalidValue;
  Params p;
  p.q = a.q;
  p.k = a.k;
  p.v = a.v;
  p.o = a.o;
  p.lse = a.lse;
  p.sb = a.sb;
  p.sh = a.sh;
  p.ss = a.ss;
  p.H = a.H;
  p.S = a.S;
  p.d = a.d;
  p.n_qblk = (a.S + kWarps - 1) / kWarps;
  p.c = a.scale * kLog2e;
  const size_t smem = sizeof(float) * (2 * kKeys * (a.d + 1) + kWarps * a.d + kWarps * kKeys);
  auto kern = a.d <= 64 ? simt_fwd_kernel<64> : (a.d <= 128 ? simt_fwd_kernel<128> : simt_fwd_kernel<256>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(a.B) * a.H * p.n_qblk;
  kern<<<static_cast<unsigned>(grid), kWarps * 32, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
