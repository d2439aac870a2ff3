// Fused multi-head attention forward for sm_103a (GB300).
//
// Computes O = softmax(scale · Q·K^T) · V tile by tile with the online
// softmax of "Transformer算子生态深度分析" ch.2 §2.6: per key tile the row
// maximum and exp-sum are merged into running statistics and the partial
// output is rescaled by exp(m_old - m), so the S×S scores never leave the SM
// ("WebGPU 算子优化：QKV 内存合并与 FlashAttention 分块计算",
// §FlashAttention 分块计算原理与浏览器适配, gives the same merge rule).
//
// GB300 mapping (one CTA per SM, 10 warps, 192 KB shared memory at d = 128):
//   * a CTA owns two 128-row Q tiles of one (batch, head) -- "ping-pong":
//     while one tile's softmax runs on the CUDA cores, the tensor cores work
//     on the other tile;
//   * warp 8: TMA producer.  Q tiles once, then K and V tiles of 128 keys
//     through a STAGES-deep ring of 128-byte-swizzled shared-memory buffers;
//   * warp 9: tcgen05 issuer.  S_t = Q_t·K_j^T into tensor memory (fp32),
//     then O_t += P_t·V_j with P_t read straight from tensor memory;
//   * warps 0-3 / 4-7: softmax of Q tile 0 / 1, one thread per query row
//     (tensor-memory lane = row), so the row max and row sum are
//     thread-local.  exp is 2^x on the SFU with scale·log2(e) folded into
//     one FFMA.  The running max is only moved when the tile max exceeds it
//     by more than 2^8 (a factor of 256 in p, safe in fp16 and bf16); the
//     result is exact either way because O and l always share the same
//     reference, and the O rescale in tensor memory is skipped otherwise.
//   * tensor memory: S0 | S1 | O0 | O1 (128 + 128 + d + d of 512 columns);
//     P_t (16-bit, two per column) overwrites the first 64 columns of S_t.
// Every wait is bounded: a pipeline stall records a code in the device
// status word and the CTA winds down instead of hanging.

#include "common.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Cfg {
  static constexpr int BM = 128;   // rows per Q tile (= tensor-memory lanes)
  static constexpr int NQ = 2;     // Q tiles per CTA
  static constexpr int BN = 128;   // keys per K/V tile
  static constexpr int NCH = D / 64;                       // 128-byte chunks per row
  static constexpr int STAGES = (D == 64) ? 4 : 2;
  static constexpr uint32_t CHUNK = 128u * 128u;           // 128 rows x 128 bytes
  static constexpr uint32_t TILE = CHUNK * NCH;            // 128 rows x D x 2 bytes
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + NQ * TILE;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + STAGES * TILE;
  // barriers: q_full, k_full[ST], k_empty[ST], v_full[ST], v_empty[ST], s_full[2], p_ready[2], drain
  static constexpr int NBAR = 1 + 4 * STAGES + 4 + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM = OFF_MISC + 16 + 1024;   // + slack for 1024-byte alignment
  static constexpr int THREADS = 320;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = 256;

  __host__ __device__ static constexpr int bar_q() { return 0; }
  __host__ __device__ static constexpr int bar_kfull(int s) { return 1 + s; }
  __host__ __device__ static constexpr int bar_kempty(int s) { return 1 + STAGES + s; }
  __host__ __device__ static constexpr int bar_vfull(int s) { return 1 + 2 * STAGES + s; }
  __host__ __device__ static constexpr int bar_vempty(int s) { return 1 + 3 * STAGES + s; }
  __host__ __device__ static constexpr int bar_sfull(int t) { return 1 + 4 * STAGES + t; }
  __host__ __device__ static constexpr int bar_pready(int t) { return 3 + 4 * STAGES + t; }
  __host__ __device__ static constexpr int bar_drain() { return 5 + 4 * STAGES; }
};
static_assert(Cfg<128>::SMEM <= 227 * 1024, "shared memory budget");
static_assert(Cfg<64>::SMEM <= 227 * 1024, "shared memory budget");

struct Params {
  void* o;
  float* lse;
  long long o_sb, o_sh, o_ss;
  int H, S, n_qblk, hs_swap;
  float c;  // scale · log2(e)
  unsigned* status;
  long long limit;
};

__device__ __forceinline__ uint32_t code_of(uint32_t role, int j) {
  return (KID_FLASH << 24) | (role << 16) | (static_cast<uint32_t>(j) & 0xffffu);
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

template <int D, bool BF16>
__global__ void __launch_bounds__(320, 1)
    flash_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;  // 128-byte swizzle wants 1024-byte aligned tiles
  uint8_t* smem = smem_raw + (sb - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };

  const uint32_t warp = warp_id(), lane = lane_id();
  const int qblk = static_cast<int>(blockIdx.x) % p.n_qblk;
  const int bh = static_cast<int>(blockIdx.x) / p.n_qblk;
  const int b = bh / p.H, hh = bh % p.H;
  const int q0 = qblk * (C::NQ * C::BM);
  const int n_kv = (p.S + C::BN - 1) / C::BN;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::bar_q()), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::bar_kfull(s)), 1);
      mbar_init(bar(C::bar_kempty(s)), 1);
      mbar_init(bar(C::bar_vfull(s)), 1);
      mbar_init(bar(C::bar_vempty(s)), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::bar_sfull(t)), 1);
      mbar_init(bar(C::bar_pready(t)), 128);
    }
    mbar_init(bar(C::bar_drain()), 1);
    // A CTA that starts after another one gave up does no work.
    *abort_flag = (*reinterpret_cast<volatile unsigned*>(p.status) != 0u) ? 1 : 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.status, p.limit};
  const bool skip = *abort_flag != 0;

  // Coordinates (feature, row) -> tensor-map coordinates.
  auto tma4 = [&](uint32_t dst, const CUtensorMap* m, uint32_t mbar, int e, int s) {
    if (p.hs_swap)
      tma_load_4d(dst, m, mbar, e, hh, s, b);
    else
      tma_load_4d(dst, m, mbar, e, s, hh, b);
  };

  if (skip) {
    // nothing
  } else if (warp == 8) {
    // ------------------------------------------------------ TMA producer ----
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      mbar_expect_tx(bar(C::bar_q()), C::NQ * C::TILE);
      for (int t = 0; t < C::NQ; ++t)
        for (int c = 0; c < C::NCH; ++c)
          tma4(sb + C::OFF_Q + t * C::TILE + c * C::CHUNK, &tq, bar(C::bar_q()), c * 64,
               q0 + t * C::BM);
    }
    int issued_k = 0, issued_v = 0;
    bool ok = true;
    for (int j = 0; j < n_kv && ok; ++j) {
      const int s = j % C::STAGES, u = j / C::STAGES;
      if (u > 0) ok = mbar_wait_warp(bar(C::bar_kempty(s)), (u - 1) & 1, wc, code_of(ROLE_LOAD, j));
      if (!ok) break;
      if (lane == 0) {
        mbar_expect_tx(bar(C::bar_kfull(s)), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma4(sb + C::OFF_K + s * C::TILE + c * C::CHUNK, &tk, bar(C::bar_kfull(s)), c * 64,
               j * C::BN);
      }
      issued_k = j + 1;
      if (u > 0) ok = mbar_wait_warp(bar(C::bar_vempty(s)), (u - 1) & 1, wc, code_of(ROLE_LOAD, j));
      if (!ok) break;
      if (lane == 0) {
        mbar_expect_tx(bar(C::bar_vfull(s)), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma4(sb + C::OFF_V + s * C::TILE + c * C::CHUNK, &tv, bar(C::bar_vfull(s)), c * 64,
               j * C::BN);
      }
      issued_v = j + 1;
    }
    if (!ok) {
      // Let the copies already in flight land before the CTA can exit.
      const WaitCtx drain{abort_flag, p.status, p.limit};
      for (int j = issued_k - C::STAGES < 0 ? 0 : issued_k - C::STAGES; j < issued_k; ++j)
        mbar_wait_slow(bar(C::bar_kfull(j % C::STAGES)), (j / C::STAGES) & 1, drain, 0, false);
      for (int j = issued_v - C::STAGES < 0 ? 0 : issued_v - C::STAGES; j < issued_v; ++j)
        mbar_wait_slow(bar(C::bar_vfull(j % C::STAGES)), (j / C::STAGES) & 1, drain, 0, false);
      mbar_wait_slow(bar(C::bar_q()), 0, drain, 0, false);
    }
  } else if (warp == 9) {
    // --------------------------------------------------- tcgen05 issuer ----
    constexpr uint32_t id_qk = idesc_f16(128, C::BN, BF16, false, false);
    constexpr uint32_t id_pv = idesc_f16(128, D, BF16, false, true);
    auto qk = [&](int t, int s) {  // S_t = Q_t · K_s^T   (K-major A and B)
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
          const uint64_t a = sdesc_sw128(sb + C::OFF_Q + t * C::TILE + off, 16, 1024);
          const uint64_t bd = sdesc_sw128(sb + C::OFF_K + s * C::TILE + off, 16, 1024);
          mma_ss(tmem + t * 128, a, bd, id_qk, kk > 0 ? 1u : 0u);
        }
      }
    };
    auto pv = [&](int t, int s, bool acc) {  // O_t (+)= P_t · V_s   (P in TMEM, V MN-major)
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          const uint64_t bd = sdesc_sw128(sb + C::OFF_V + s * C::TILE + kk * 2048, C::CHUNK, 1024);
          mma_ts(tmem + C::COL_O + t * D, tmem + t * 128 + kk * 8, bd, id_pv,
                 (acc || kk > 0) ? 1u : 0u);
        }
      }
    };
    auto commit = [&](int i) {
      if (lane == 0) mma_commit(bar(i));
    };
    bool ok = mbar_wait_warp(bar(C::bar_q()), 0, wc, code_of(ROLE_MMA, 0)) &&
              mbar_wait_warp(bar(C::bar_kfull(0)), 0, wc, code_of(ROLE_MMA, 0));
    if (ok) {
      tc_fence_after();
      qk(0, 0);
      commit(C::bar_sfull(0));
      qk(1, 0);
      commit(C::bar_sfull(1));
      commit(C::bar_kempty(0));
    }
    for (int j = 0; j < n_kv && ok; ++j) {
      const int s = j % C::STAGES, u = j / C::STAGES;
      const bool more = j + 1 < n_kv;
      const int s1 = (j + 1) % C::STAGES, u1 = (j + 1) / C::STAGES;
      ok = mbar_wait_warp(bar(C::bar_vfull(s)), u & 1, wc, code_of(ROLE_MMA, j)) &&
           mbar_wait_warp(bar(C::bar_pready(0)), j & 1, wc, code_of(ROLE_MMA, j));
      if (!ok) break;
      tc_fence_after();
      pv(0, s, j > 0);
      if (more) {
        ok = mbar_wait_warp(bar(C::bar_kfull(s1)), u1 & 1, wc, code_of(ROLE_MMA, j));
        if (!ok) break;
        tc_fence_after();
        qk(0, s1);
      }
      commit(C::bar_sfull(0));  // S_0 of the next tile ready, or the final O_0
      ok = mbar_wait_warp(bar(C::bar_pready(1)), j & 1, wc, code_of(ROLE_MMA, j));
      if (!ok) break;
      tc_fence_after();
      pv(1, s, j > 0);
      commit(C::bar_vempty(s));
      if (more) {
        qk(1, s1);
        commit(C::bar_sfull(1));
        commit(C::bar_kempty(s1));
      } else {
        commit(C::bar_sfull(1));
      }
    }
    if (!ok) {
      // Wait for the MMAs already issued before tensor memory is released.
      commit(C::bar_drain());
      const WaitCtx drain{abort_flag, p.status, p.limit};
      mbar_wait_slow(bar(C::bar_drain()), 0, drain, 0, false);
    }
  } else {
    // ------------------------------------------------ softmax warps 0-7 ----
    const int t = static_cast<int>(warp) >> 2;   // Q tile
    const uint32_t wq = warp & 3u;               // tensor-memory sub-partition
    const uint32_t lane_off = (wq * 32u) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + C::COL_O + t * D;
    const float c = p.c;
    float m_ref = -INFINITY;  // running max (log2 units) that P and O are referenced to
    float l = 0.f;            // running sum of p
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      ok = mbar_wait_warp(bar(C::bar_sfull(t)), j & 1, wc, code_of(ROLE_SOFTMAX, j));
      if (!ok) break;
      tc_fence_after();
      uint32_t r[4][32];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, r[q]);
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld_wait(r[q]);
      const int valid = p.S - j * C::BN;
      if (valid < C::BN) {  // ragged key tail: these columns do not exist
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (q * 32 + i >= valid) r[q][i] = f2u(-INFINITY);
      }
      float mx0 = u2f(r[0][0]), mx1 = u2f(r[1][0]);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        mx0 = fmaxf(mx0, fmaxf(u2f(r[0][i]), u2f(r[2][i])));
        mx1 = fmaxf(mx1, fmaxf(u2f(r[1][i]), u2f(r[3][i])));
      }
      const float m_blk = fmaxf(mx0, mx1) * c;
      const float m_new = (m_blk > m_ref + kRescaleThreshold) ? m_blk : m_ref;
      const float alpha = ex2(m_ref - m_new);  // 0 on the first tile, 1 when unchanged
      l *= alpha;
      if (j > 0 && __any_sync(0xffffffffu, m_new != m_ref)) {
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
          tmem_st32(tO + cc * 32, o);
        }
      }
      m_ref = m_new;
      const float nm = -m_ref;
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const float a0 = ex2(fmaf(u2f(r[q][2 * i]), c, nm));
          const float a1 = ex2(fmaf(u2f(r[q][2 * i + 1]), c, nm));
          const float a2 = ex2(fmaf(u2f(r[q][2 * i + 2]), c, nm));
          const float a3 = ex2(fmaf(u2f(r[q][2 * i + 3]), c, nm));
          s0 += a0;
          s1 += a1;
          s2 += a2;
          s3 += a3;
          pk[i] = pack2<BF16>(a0, a1);
          pk[i + 1] = pack2<BF16>(a2, a3);
        }
        tmem_st16(tS + q * 16, pk);  // P columns [16q, 16q+16) hold keys [32q, 32q+32)
      }
      tmem_st_wait();
      l += (s0 + s1) + (s2 + s3);
      tc_fence_before();
      mbar_arrive(bar(C::bar_pready(t)));
    }
    if (ok) ok = mbar_wait_warp(bar(C::bar_sfull(t)), n_kv & 1, wc, code_of(ROLE_EPILOGUE, n_kv));
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l;
      const int row = q0 + t * C::BM + static_cast<int>(wq * 32 + lane);
      const bool in = row < p.S;
      using Elem = uint16_t;
      Elem* out = static_cast<Elem*>(p.o) + b * p.o_sb + hh * p.o_sh +
                  static_cast<long long>(in ? row : 0) * p.o_ss;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        tmem_ld_wait(o);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(u2f(o[2 * i]) * inv, u2f(o[2 * i + 1]) * inv);
        if (in) {
          uint4* dst = reinterpret_cast<uint4*>(out + cc * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
      }
      if (in && p.lse)
        p.lse[(static_cast<long long>(b) * p.H + hh) * p.S + row] = (m_ref + log2f(l)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool BF16>
cudaError_t launch_impl(const FlashLaunch& a, cudaStream_t st) {
  using C = Cfg<D>;
  auto kern = flash_fwd_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  Params p;
  p.o = a.o;
  p.lse = a.lse;
  p.o_sb = a.o_sb;
  p.o_sh = a.o_sh;
  p.o_ss = a.o_ss;
  p.H = a.H;
  p.S = a.S;
  p.n_qblk = (a.S + C::NQ * C::BM - 1) / (C::NQ * C::BM);
  p.hs_swap = a.hs_swap;
  p.c = a.scale * kLog2e;
  p.status = a.status;
  p.limit = a.limit;
  const long long grid = static_cast<long long>(a.B) * a.H * p.n_qblk;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, st>>>(a.tq, a.tk, a.tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_flash_fwd(const FlashLaunch& a, cudaStream_t st) {
  if (a.d == 64) return a.bf16 ? launch_impl<64, true>(a, st) : launch_impl<64, false>(a, st);
  if (a.d == 128) return a.bf16 ? launch_impl<128, true>(a, st) : launch_impl<128, false>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace attn
