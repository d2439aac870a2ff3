// Batched tensor-core GEMM for sm_103a: C[z] = alpha · A[z] · B[z].
//
// Used for the fused QKV projection X·W_qkv ("Transformer算子生态深度分析"
// ch.2 §2.1: one product with the concatenated [D, 3D] weight) and for the
// two products of the unfused comparison path (S = Q·K^T and O = P·V, same
// chapter §2.2 and §2.4).
//
// Persistent: one CTA per SM walks the BM x BN output tiles (tile index
// blockIdx.x, + gridDim.x, ...), 10 warps:
//   warp 0     TMA producer: A (BM x 64, K-major) and B tiles through a
//              STAGES-deep ring of 128-byte-swizzled shared-memory buffers,
//              continuing across tiles;
//   warp 1     tcgen05 issuer into fp32 accumulators in tensor memory.  With
//              BM = 128 there are two (128 lanes x BN columns each),
//              alternating per tile.  With BM = 256 (the projection: two
//              M = 128 products per k-step sharing each B stage, a third
//              less operand traffic per flop) one accumulator of 512 columns;
//   warps 2-9  epilogue: accumulator -> registers -> alpha, convert -> a
//              per-warp shared-memory staging area -> global as whole
//              128-byte row segments (one thread per output row; the two
//              warps of a tensor-memory lane quarter split the columns, or
//              with BM = 256 the two row halves), while the issuer already
//              fills the other accumulator with the next tile (BM = 128).
// B is either K-major ([N, K], e.g. K of S = Q·K^T) or MN-major ([K, N],
// e.g. W_qkv or V) -- the tensor cores read both directly.

#include "common.h"
#include "ptx.cuh"

namespace attn {
namespace {

// MB = 2: a tile of 256 rows as two M = 128 products sharing each B stage
// (one third less operand traffic per flop than two 128-row tiles).
template <int BN, bool BK, int MB>
struct GCfg {
  static constexpr int BM = 128 * MB, BKE = 64;
  static constexpr int STAGES = MB == 2 ? 3 : (BN == 256 ? 4 : (BN == 128 ? 5 : 6));
  static constexpr uint32_t A_HALF = 128 * 128;        // 128 rows x 64 elements x 2 B
  static constexpr uint32_t A_BYTES = MB * A_HALF;
  static constexpr uint32_t B_BYTES = BN * 128;        // BN x 64 x 2 B (either major)
  static constexpr uint32_t B_CHUNK = 64 * 128;        // MN-major: 64 k-rows x 64 n
  static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
  static constexpr uint32_t OFF_BAR = STAGES * STAGE;
  // full[], empty[], acc_full[2], acc_empty[2], drain
  static constexpr int NBAR = 2 * STAGES + 5;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  // epilogue staging: per epilogue warp 32 rows x 128 bytes
  static constexpr uint32_t OFF_EPI = (OFF_MISC + 16 + 127) & ~127u;
  static constexpr uint32_t EPI_WARP = 32 * 128;
  static constexpr uint32_t SMEM = OFF_EPI + 8 * EPI_WARP + 1024;
  static constexpr int ACCS = MB * BN * 2 <= 512 ? 2 : 1;  // accumulator sets (tiles in flight)
  static constexpr uint32_t ACC_COLS = MB * BN;
  static constexpr uint32_t TMEM_COLS = ACCS * ACC_COLS;
  __host__ __device__ static constexpr int bar_full(int s) { return s; }
  __host__ __device__ static constexpr int bar_empty(int s) { return STAGES + s; }
  __host__ __device__ static constexpr int bar_accfull(int a) { return 2 * STAGES + a; }
  __host__ __device__ static constexpr int bar_accempty(int a) { return 2 * STAGES + 2 + a; }
  __host__ __device__ static constexpr int bar_drain() { return 2 * STAGES + 4; }
};
static_assert(GCfg<256, false, 1>::SMEM <= 227 * 1024, "shared memory budget");
static_assert(GCfg<256, false, 2>::SMEM <= 227 * 1024, "shared memory budget");
static_assert(GCfg<128, false, 1>::SMEM <= 227 * 1024, "shared memory budget");
static_assert(GCfg<64, false, 1>::SMEM <= 227 * 1024, "shared memory budget");
static_assert(GCfg<256, false, 2>::TMEM_COLS == 512, "tensor memory budget");

struct Params {
  void* c;
  int c_type;
  long long ldc, c_s1, c_s2;
  int M, N, K, Z1;
  int n_mblk, n_nblk, n_tiles;
  int a_swap, b_swap;  // tensor-map dims (inner, Z1, rows, Z2) instead of (inner, rows, Z1, Z2)
  float alpha;
  unsigned* status;
  long long limit;
};

__device__ __forceinline__ uint32_t gcode(uint32_t role, int j) {
  return (KID_GEMM << 24) | (role << 16) | (static_cast<uint32_t>(j) & 0xffffu);
}

template <int BN, bool BKMAJOR, bool BF16, int MB>
__global__ void __launch_bounds__(320, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                const Params p) {
  using C = GCfg<BN, BKMAJOR, MB>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sb - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };

  const uint32_t warp = warp_id(), lane = lane_id();
  const int nk = (p.K + C::BKE - 1) / C::BKE;
  // tile index -> (z, m block, n block), n fastest
  auto tile_coords = [&](int tile, int& z, int& mb, int& nb) {
    nb = tile % p.n_nblk;
    mb = (tile / p.n_nblk) % p.n_mblk;
    z = tile / (p.n_nblk * p.n_mblk);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::bar_full(s)), 1);
      mbar_init(bar(C::bar_empty(s)), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(C::bar_accfull(a)), 1);
      mbar_init(bar(C::bar_accempty(a)), 8);  // one arrival per epilogue warp
    }
    mbar_init(bar(C::bar_drain()), 1);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  // Launched as a programmatic dependent: the set-up above overlaps the
  // previous grid's tail, global memory is touched only after it completed.
  griddep_wait();
  if (threadIdx.x == 0) {
    *abort_flag = (*reinterpret_cast<volatile unsigned*>(p.status) != 0u) ? 1 : 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();  // e.g. the attention kernel that reads this product
  const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);
  const WaitCtx wc{abort_flag, p.status, p.limit};
  const bool skip = *abort_flag != 0;

  if (skip) {
  } else if (warp == 0) {
    // ------------------------------------------------------ TMA producer ----
    if (lane == 0) {
      prefetch_tmap(&ta);
      prefetch_tmap(&tb);
    }
    int g = 0;  // k-steps issued so far (all tiles)
    bool ok = true;
    for (int tile = blockIdx.x; tile < p.n_tiles && ok; tile += gridDim.x) {
      int z, mb, nb;
      tile_coords(tile, z, mb, nb);
      const int z1 = z % p.Z1, z2 = z / p.Z1;
      auto load = [&](uint32_t dst, const CUtensorMap* m, uint32_t mbar, int inner, int row, int swap) {
        if (swap)
          tma_load_4d(dst, m, mbar, inner, z1, row, z2);
        else
          tma_load_4d(dst, m, mbar, inner, row, z1, z2);
      };
      for (int kt = 0; kt < nk; ++kt, ++g) {
        const int s = g % C::STAGES, u = g / C::STAGES;
        if (u > 0 && !(ok = mbar_wait_warp(bar(C::bar_empty(s)), (u - 1) & 1, wc, gcode(ROLE_LOAD, g))))
          break;
        if (lane == 0) {
          const uint32_t st = sb + s * C::STAGE;
          mbar_expect_tx(bar(C::bar_full(s)), C::STAGE);
#pragma unroll
          for (int h = 0; h < MB; ++h)
            load(st + h * C::A_HALF, &ta, bar(C::bar_full(s)), kt * C::BKE, mb * C::BM + h * 128, p.a_swap);
          if constexpr (BKMAJOR) {
            load(st + C::A_BYTES, &tb, bar(C::bar_full(s)), kt * C::BKE, nb * BN, p.b_swap);
          } else {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              load(st + C::A_BYTES + c * C::B_CHUNK, &tb, bar(C::bar_full(s)), nb * BN + c * 64,
                   kt * C::BKE, p.b_swap);
          }
        }
      }
    }
    if (!ok) {  // let the copies in flight land before the CTA can exit
      for (int q = g - C::STAGES < 0 ? 0 : g - C::STAGES; q < g; ++q)
        mbar_wait_slow(bar(C::bar_full(q % C::STAGES)), (q / C::STAGES) & 1, wc, 0, false);
    }
  } else if (warp == 1) {
    // ------------------------------------------------- tcgen05 issuer ----
    // The whole warp runs the issue loop; elect.sync inside the helpers picks
    // the lane that issues, so the descriptors stay warp-uniform.
    constexpr uint32_t idesc = idesc_f16(128, BN, BF16, false, !BKMAJOR);
    const uint64_t da = sdesc_sw128(sb, 16, 1024);
    const uint64_t db = BKMAJOR ? sdesc_sw128(sb + C::A_BYTES, 16, 1024)
                                : sdesc_sw128(sb + C::A_BYTES, C::B_CHUNK, 1024);
    int g = 0, i = 0;  // k-steps consumed, tiles done by this CTA
    bool ok = true;
    for (int tile = blockIdx.x; tile < p.n_tiles && ok; tile += gridDim.x, ++i) {
      const int a = i % C::ACCS;
      if (i >= C::ACCS && !(ok = mbar_wait_warp(bar(C::bar_accempty(a)), ((i / C::ACCS) - 1) & 1, wc,
                                               gcode(ROLE_MMA, i))))
        break;
      tc_fence_after();
      const uint32_t acc = tmem + a * C::ACC_COLS;
      for (int kt = 0; kt < nk; ++kt, ++g) {
        const int s = g % C::STAGES, u = g / C::STAGES;
        if (!(ok = mbar_wait_warp(bar(C::bar_full(s)), u & 1, wc, gcode(ROLE_MMA, g)))) break;
        tc_fence_after();
        const uint32_t st16 = (s * C::STAGE) >> 4;  // stage offset in descriptor address units
#pragma unroll
        for (int kk = 0; kk < C::BKE / 16; ++kk) {
          const uint32_t ka = (kk * 32) >> 4, kb = (BKMAJOR ? kk * 32 : kk * 2048) >> 4;
#pragma unroll
          for (int h = 0; h < MB; ++h)  // rows 128h.. of the tile into accumulator columns h·BN..
            mma_ss_elect(acc + h * BN, da + st16 + ((h * C::A_HALF) >> 4) + ka, db + st16 + kb, idesc,
                         (kt > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit_elect(bar(C::bar_empty(s)));
      }
      if (ok) mma_commit_elect(bar(C::bar_accfull(a)));
    }
    if (!ok) {
      mma_commit_elect(bar(C::bar_drain()));
      mbar_wait_slow(bar(C::bar_drain()), 0, wc, 0, false);
    }
  } else {
    // -------------------------------------------------------- epilogue ----
    // Each thread holds one output row of its warp's 32; the rows go out
    // through a per-warp staging area so that every global store instruction
    // writes whole 128-byte row segments (8 lanes per row, 4 rows) instead of
    // 32 scattered 16-byte pieces.  16-byte unit u of staged row r sits at
    // (u ^ (r & 7)) so that neither side has bank conflicts.
    const uint32_t wq = warp & 3u;               // tensor-memory lane quarter
    // The two warps of a lane quarter split the tile: by columns (MB = 1) or
    // by its two 128-row halves (MB = 2).
    const int half = (static_cast<int>(warp) - 2) >> 2;
    uint8_t* stage = smem + C::OFF_EPI + (warp - 2u) * C::EPI_WARP;
    const int esz = p.c_type == 0 ? 4 : 2;       // output element bytes
    const long long ev = 16 / esz;               // elements per 16 bytes
    const bool vec_ok = (reinterpret_cast<uintptr_t>(p.c) & 15u) == 0 && p.ldc % ev == 0 &&
                        p.c_s1 % ev == 0 && p.c_s2 % ev == 0;
    // Stages this thread's 8 16-byte units (one 128-byte row segment), then
    // writes the warp's 32 segments to rows row0.. with coalesced stores.
    auto flush = [&](const uint4 (&u16)[8], int row0, long long base, int col0) {
      __syncwarp();  // the previous segment's reads are done
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint4*>(stage + lane * 128 + ((u ^ (lane & 7)) << 4)) = u16[u];
      __syncwarp();
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int rr = it * 4 + static_cast<int>(lane >> 3), u = static_cast<int>(lane & 7);
        const uint4 v = *reinterpret_cast<const uint4*>(stage + rr * 128 + ((u ^ (rr & 7)) << 4));
        if (row0 + rr < p.M) {
          uint8_t* dst = static_cast<uint8_t*>(p.c) +
                         (base + static_cast<long long>(row0 + rr) * p.ldc + col0) * esz + u * 16;
          *reinterpret_cast<uint4*>(dst) = v;
        }
      }
    };
    int i = 0;
    for (int tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x, ++i) {
      const int a = i % C::ACCS;
      if (!mbar_wait_warp(bar(C::bar_accfull(a)), (i / C::ACCS) & 1, wc, gcode(ROLE_EPILOGUE, i))) break;
      tc_fence_after();
      int z, mb, nb;
      tile_coords(tile, z, mb, nb);
      const int z1 = z % p.Z1, z2 = z / p.Z1;
      const int row0 = mb * C::BM + (MB == 2 ? half * 128 : 0) + static_cast<int>(wq * 32);
      const int row = row0 + static_cast<int>(lane);
      const bool in = row < p.M;
      const long long base = z2 * p.c_s2 + z1 * p.c_s1;
      const long long off = base + static_cast<long long>(in ? row : 0) * p.ldc;
      const uint32_t acc = tmem + ((wq * 32u) << 16) + a * C::ACC_COLS + (MB == 2 ? half * BN : 0);
      // 128-byte row segments: 32 fp32 or 64 16-bit columns
      const int seg_cols = p.c_type == 0 ? 32 : 64;
      const int c_lo = MB == 2 ? 0 : half * (BN / 2), c_hi = MB == 2 ? BN : (half + 1) * (BN / 2);
#pragma unroll 1
      for (int c0 = c_lo; c0 < c_hi; c0 += seg_cols) {
        const int col0 = nb * BN + c0;
        if (col0 >= p.N) break;
        const bool fast = vec_ok && col0 + seg_cols <= p.N;
        uint32_t r[32];
        tmem_ld32(acc + c0, r);
        tmem_ld_wait(r);
        if (p.c_type == 0) {
          if (fast) {
            uint4 u16[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
              u16[u] = make_uint4(__float_as_uint(__uint_as_float(r[4 * u]) * p.alpha), __float_as_uint(__uint_as_float(r[4 * u + 1]) * p.alpha),
                                  __float_as_uint(__uint_as_float(r[4 * u + 2]) * p.alpha), __float_as_uint(__uint_as_float(r[4 * u + 3]) * p.alpha));
            flush(u16, row0, base, col0);
          } else if (in) {
            float* dst = static_cast<float*>(p.c) + off + col0;
            const int nvalid = min(32, p.N - col0);
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (k < nvalid) dst[k] = __uint_as_float(r[k]) * p.alpha;
          }
        } else {
          uint32_t pk[32];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            pk[k] = pack2<BF16>(__uint_as_float(r[2 * k]) * p.alpha, __uint_as_float(r[2 * k + 1]) * p.alpha);
          const bool second = col0 + 32 < p.N;  // columns [col0 + 32, col0 + 64) exist
          if (second) {
            tmem_ld32(acc + c0 + 32, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int k = 0; k < 16; ++k)
              pk[16 + k] = pack2<BF16>(__uint_as_float(r[2 * k]) * p.alpha, __uint_as_float(r[2 * k + 1]) * p.alpha);
          }
          if (fast) {
            uint4 u16[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) u16[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            flush(u16, row0, base, col0);
          } else if (in) {
            uint16_t* dst = static_cast<uint16_t*>(p.c) + off + col0;
            const int nvalid = min(64, p.N - col0);
#pragma unroll
            for (int k = 0; k < 64; ++k)
              if (k < nvalid) dst[k] = static_cast<uint16_t>(pk[k >> 1] >> ((k & 1) * 16));
          }
        }
      }
      // this accumulator may be overwritten by the tile after next
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::bar_accempty(a)));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      n = v;
    else
      n = 148;
  }
  return n;
}

template <int BN, bool BKMAJOR, bool BF16, int MB = 1>
cudaError_t launch_impl(const GemmLaunch& a, cudaStream_t st) {
  using C = GCfg<BN, BKMAJOR, MB>;
  auto kern = gemm_kernel<BN, BKMAJOR, BF16, MB>;
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
  const long long tiles = static_cast<long long>(p.n_mblk) * p.n_nblk * a.Z1 * a.Z2;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  p.n_tiles = static_cast<int>(tiles);
  p.a_swap = a.a_swap;
  p.b_swap = a.b_swap;
  p.alpha = a.alpha;
  p.status = a.status;
  p.limit = a.limit;
  const int grid = static_cast<int>(tiles < num_sms() ? tiles : num_sms());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(320);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t le = cudaLaunchKernelEx(&cfg, kern, a.ta, a.tb, p);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

template <bool BF16>
cudaError_t dispatch(const GemmLaunch& a, cudaStream_t st) {
  if (a.bn == 64) return a.b_kmajor ? launch_impl<64, true, BF16>(a, st) : launch_impl<64, false, BF16>(a, st);
  if (a.bn == 128)
    return a.b_kmajor ? launch_impl<128, true, BF16>(a, st) : launch_impl<128, false, BF16>(a, st);
  if (a.bn == 256 && a.mb == 2 && !a.b_kmajor) return launch_impl<256, false, BF16, 2>(a, st);
  if (a.bn == 256)
    return a.b_kmajor ? launch_impl<256, true, BF16>(a, st) : launch_impl<256, false, BF16>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemm(const GemmLaunch& a, cudaStream_t st) {
  return a.bf16 ? dispatch<true>(a, st) : dispatch<false>(a, st);
}

}  // namespace attn
