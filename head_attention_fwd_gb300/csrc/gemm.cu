// Batched tensor-core GEMM for sm_103a: C[z] = alpha · A[z] · B[z].
//
// Used for the fused QKV projection X·W_qkv ("Transformer算子生态深度分析"
// ch.2 §2.1: one product with the concatenated [D, 3D] weight) and for the
// two products of the unfused comparison path (S = Q·K^T and O = P·V, same
// chapter §2.2 and §2.4).
//
// One 128 x BN output tile per CTA, 6 warps, two CTAs per SM:
//   warp 0     TMA producer: A (128 x 64, K-major) and B tiles through a
//              3-stage ring of 128-byte-swizzled shared-memory buffers;
//   warp 1     tcgen05 issuer, fp32 accumulator of 128 lanes x BN columns
//              in tensor memory;
//   warps 2-5  epilogue: tensor memory -> registers -> alpha, convert ->
//              global (one thread per output row).
// B is either K-major ([N, K], e.g. K of S = Q·K^T) or MN-major ([K, N],
// e.g. W_qkv or V) -- the tensor cores read both directly.

#include "common.h"
#include "ptx.cuh"

namespace attn {
namespace {

template <int BN, bool BK>
struct GCfg {
  static constexpr int BM = 128, BKE = 64, STAGES = 3;
  static constexpr uint32_t A_BYTES = BM * 128;        // 128 rows x 64 elements x 2 B
  static constexpr uint32_t B_BYTES = BN * 128;        // BN x 64 x 2 B (either major)
  static constexpr uint32_t B_CHUNK = 64 * 128;        // MN-major: 64 k-rows x 64 n
  static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
  static constexpr uint32_t OFF_BAR = STAGES * STAGE;
  static constexpr int NBAR = 2 * STAGES + 2;          // full[], empty[], acc_full, drain
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
  __host__ __device__ static constexpr int bar_full(int s) { return s; }
  __host__ __device__ static constexpr int bar_empty(int s) { return STAGES + s; }
  __host__ __device__ static constexpr int bar_acc() { return 2 * STAGES; }
  __host__ __device__ static constexpr int bar_drain() { return 2 * STAGES + 1; }
};

struct Params {
  void* c;
  int c_type;
  long long ldc, c_s1, c_s2;
  int M, N, K, Z1;
  int n_mblk, n_nblk;
  int a_swap, b_swap;  // tensor-map dims (inner, Z1, rows, Z2) instead of (inner, rows, Z1, Z2)
  float alpha;
  unsigned* status;
  long long limit;
};

__device__ __forceinline__ uint32_t gcode(uint32_t role, int j) {
  return (KID_GEMM << 24) | (role << 16) | (static_cast<uint32_t>(j) & 0xffffu);
}

template <int BN, bool BKMAJOR, bool BF16>
__global__ void __launch_bounds__(192, 2)
    gemm_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                const Params p) {
  using C = GCfg<BN, BKMAJOR>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sb - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };

  const uint32_t warp = warp_id(), lane = lane_id();
  const int nb = static_cast<int>(blockIdx.x) % p.n_nblk;
  const int mb = (static_cast<int>(blockIdx.x) / p.n_nblk) % p.n_mblk;
  const int z = static_cast<int>(blockIdx.x) / (p.n_nblk * p.n_mblk);
  const int z1 = z % p.Z1, z2 = z / p.Z1;
  const int m0 = mb * C::BM, n0 = nb * BN;
  const int nk = (p.K + C::BKE - 1) / C::BKE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::bar_full(s)), 1);
      mbar_init(bar(C::bar_empty(s)), 1);
    }
    mbar_init(bar(C::bar_acc()), 1);
    mbar_init(bar(C::bar_drain()), 1);
    *abort_flag = (*reinterpret_cast<volatile unsigned*>(p.status) != 0u) ? 1 : 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);
  const WaitCtx wc{abort_flag, p.status, p.limit};
  const bool skip = *abort_flag != 0;

  auto load = [&](uint32_t dst, const CUtensorMap* m, uint32_t mbar, int inner, int row, int swap) {
    if (swap)
      tma_load_4d(dst, m, mbar, inner, z1, row, z2);
    else
      tma_load_4d(dst, m, mbar, inner, row, z1, z2);
  };

  if (skip) {
  } else if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&ta);
      prefetch_tmap(&tb);
    }
    int issued = 0;
    bool ok = true;
    for (int kt = 0; kt < nk; ++kt) {
      const int s = kt % C::STAGES, u = kt / C::STAGES;
      if (u > 0) ok = mbar_wait_warp(bar(C::bar_empty(s)), (u - 1) & 1, wc, gcode(ROLE_LOAD, kt));
      if (!ok) break;
      if (lane == 0) {
        const uint32_t st = sb + s * C::STAGE;
        mbar_expect_tx(bar(C::bar_full(s)), C::STAGE);
        load(st, &ta, bar(C::bar_full(s)), kt * C::BKE, m0, p.a_swap);
        if constexpr (BKMAJOR) {
          load(st + C::A_BYTES, &tb, bar(C::bar_full(s)), kt * C::BKE, n0, p.b_swap);
        } else {
#pragma unroll
          for (int c = 0; c < BN / 64; ++c)
            load(st + C::A_BYTES + c * C::B_CHUNK, &tb, bar(C::bar_full(s)), n0 + c * 64,
                 kt * C::BKE, p.b_swap);
        }
      }
      issued = kt + 1;
    }
    if (!ok) {
      const WaitCtx drain{abort_flag, p.status, p.limit};
      for (int kt = issued - C::STAGES < 0 ? 0 : issued - C::STAGES; kt < issued; ++kt)
        mbar_wait_slow(bar(C::bar_full(kt % C::STAGES)), (kt / C::STAGES) & 1, drain, 0, false);
    }
  } else if (warp == 1) {
    // The whole warp runs the issue loop; elect.sync inside the helpers picks
    // the lane that issues, so the descriptors stay warp-uniform.
    constexpr uint32_t idesc = idesc_f16(128, BN, BF16, false, !BKMAJOR);
    const uint64_t da = sdesc_sw128(sb, 16, 1024);
    const uint64_t db = BKMAJOR ? sdesc_sw128(sb + C::A_BYTES, 16, 1024)
                                : sdesc_sw128(sb + C::A_BYTES, C::B_CHUNK, 1024);
    bool ok = true;
    for (int kt = 0; kt < nk; ++kt) {
      const int s = kt % C::STAGES, u = kt / C::STAGES;
      ok = mbar_wait_warp(bar(C::bar_full(s)), u & 1, wc, gcode(ROLE_MMA, kt));
      if (!ok) break;
      tc_fence_after();
      const uint32_t st16 = (s * C::STAGE) >> 4;  // stage offset in descriptor address units
#pragma unroll
      for (int kk = 0; kk < C::BKE / 16; ++kk) {
        const uint32_t ka = (kk * 32) >> 4, kb = (BKMAJOR ? kk * 32 : kk * 2048) >> 4;
        mma_ss_elect(tmem, da + st16 + ka, db + st16 + kb, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit_elect(bar(C::bar_empty(s)));
    }
    mma_commit_elect(bar(ok ? C::bar_acc() : C::bar_drain()));
    if (!ok) mbar_wait_slow(bar(C::bar_drain()), 0, wc, 0, false);
  } else {
    // -------------------------------------------------------- epilogue ----
    const uint32_t wq = warp & 3u;
    if (mbar_wait_warp(bar(C::bar_acc()), 0, wc, gcode(ROLE_EPILOGUE, 0))) {
      tc_fence_after();
      const int row = m0 + static_cast<int>(wq * 32 + lane);
      const bool in = row < p.M;
      const long long off = z2 * p.c_s2 + z1 * p.c_s1 + static_cast<long long>(in ? row : 0) * p.ldc;
#pragma unroll 1
      for (int cc = 0; cc < BN / 32; ++cc) {
        uint32_t r[32];
        tmem_ld32(tmem + ((wq * 32u) << 16) + cc * 32, r);
        tmem_ld_wait(r);
        const int col0 = n0 + cc * 32;
        if (!in || col0 >= p.N) continue;
        const int nvalid = min(32, p.N - col0);
        if (p.c_type == 0) {
          float* dst = static_cast<float*>(p.c) + off + col0;
          const bool vec = nvalid == 32 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
          if (vec) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(dst + i) =
                  make_float4(__uint_as_float(r[i]) * p.alpha, __uint_as_float(r[i + 1]) * p.alpha,
                              __uint_as_float(r[i + 2]) * p.alpha, __uint_as_float(r[i + 3]) * p.alpha);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < nvalid) dst[i] = __uint_as_float(r[i]) * p.alpha;
          }
        } else {
          uint16_t* dst = static_cast<uint16_t*>(p.c) + off + col0;
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack2<BF16>(__uint_as_float(r[2 * i]) * p.alpha,
                                __uint_as_float(r[2 * i + 1]) * p.alpha);
          const bool vec = nvalid == 32 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
          if (vec) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              reinterpret_cast<uint4*>(dst)[v4] =
                  make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < nvalid) dst[i] = static_cast<uint16_t>(pk[i >> 1] >> ((i & 1) * 16));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int BN, bool BKMAJOR, bool BF16>
cudaError_t launch_impl(const GemmLaunch& a, cudaStream_t st) {
  using C = GCfg<BN, BKMAJOR>;
  auto kern = gemm_kernel<BN, BKMAJOR, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  Params p;
  p.c = a.c;
  p.c_type = a.c_type;
  p.ldc = a.ldc;
  p.c_s1 = a.c_s1;
  p.c_s2 = a.c_s2;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.Z1 = a.Z1;
  p.n_mblk = (a.M + C::BM - 1) / C::BM;
  p.n_nblk = (a.N + BN - 1) / BN;
  p.a_swap = a.a_swap;
  p.b_swap = a.b_swap;
  p.alpha = a.alpha;
  p.status = a.status;
  p.limit = a.limit;
  const long long grid = static_cast<long long>(p.n_mblk) * p.n_nblk * a.Z1 * a.Z2;
  kern<<<static_cast<unsigned>(grid), 192, C::SMEM, st>>>(a.ta, a.tb, p);
  return cudaGetLastError();
}

template <bool BF16>
cudaError_t dispatch(const GemmLaunch& a, cudaStream_t st) {
  if (a.bn == 64) return a.b_kmajor ? launch_impl<64, true, BF16>(a, st) : launch_impl<64, false, BF16>(a, st);
  if (a.bn == 128)
    return a.b_kmajor ? launch_impl<128, true, BF16>(a, st) : launch_impl<128, false, BF16>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemm(const GemmLaunch& a, cudaStream_t st) {
  return a.bf16 ? dispatch<true>(a, st) : dispatch<false>(a, st);
}

}  // namespace attn
