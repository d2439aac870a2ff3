// Fused multi-head attention forward for sm_103a (GB300).
//
// Computes O = softmax(scale · Q·K^T) · V tile by tile with the online
// softmax of "Transformer算子生态深度分析" ch.2 §2.6: per key tile the row
// maximum and exp-sum are merged into running statistics and the partial
// output is rescaled by exp(m_old - m), so the S×S scores never leave the SM
// ("WebGPU 算子优化：QKV 内存合并与 FlashAttention 分块计算",
// §FlashAttention 分块计算原理与浏览器适配, gives the same merge rule).
//
// GB300 mapping (one CTA per SM, 11 warps, up to 192 KB shared memory):
//   * a CTA owns two 128-row Q tiles of one (batch, head) -- "ping-pong":
//     while one tile's softmax runs on the CUDA cores, the tensor cores work
//     on the other tile;
//   * warp 8: TMA producer.  Q tiles once, then K and V tiles of 128 keys
//     through a STAGES-deep ring of 128-byte-swizzled shared-memory buffers;
//   * tcgen05 issue: S_t = Q_t·K_j^T into tensor memory (fp32), then
//     O_t += P_t·V_j with P_t read straight from tensor memory.  At d = 64
//     warps 9 / 10 issue for Q tile 0 / 1, so the two tiles' pipelines are
//     independent and share only the K/V ring; at d = 128 (tensor-bound)
//     warp 9 issues both tiles in alternation;
//   * warps 0-3 / 4-7: softmax of Q tile 0 / 1, one thread per query row
//     (tensor-memory lane = row), so the row max and row sum are
//     thread-local.  exp is 2^x on the SFU with scale·log2(e) folded into
//     one packed FFMA; sums use packed fp32 adds and the max 3-input max.
//     The running max only moves when the tile max exceeds it by more than
//     2^8 (a factor of 256 in p, safe in fp16 and bf16); the result is exact
//     either way because O and l always share the same reference.  So after
//     the first tile the exponentials are computed against the current
//     reference while the tile max is tracked in the same pass (S stays in
//     registers and is released at once); only when some row's max moved by
//     more than 2^8 does the warp recompute P and rescale O in tensor memory.
//   * tensor memory, d = 64:  S0 | S1 | O0 | O1 | P0 | P1 (128+128+64+64+64+64)
//     P has its own columns, so the next Q·K^T can be issued as soon as the
//     softmax has read S, while it is still computing exponentials;
//     d = 128: S0 | S1 | O0 | O1 (128+128+128+128); P overwrites the first
//     64 columns of S, so the next Q·K^T waits for the P·V that reads it.
//   * each issuer warp issues from a converged warp (elect.sync picks the
//     lane), so descriptors stay warp-uniform.
// Every wait is bounded: a pipeline stall records a code in the device
// status word and the CTA winds down instead of hanging.

#include "common.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr bool kExpToken = true;           // d = 64: softmax warpgroups alternate on the exp pass

template <int D>
struct Cfg {
  static constexpr int BM = 128;   // rows per Q tile (= tensor-memory lanes)
  static constexpr int NQ = 2;     // Q tiles per CTA
  static constexpr int BN = 128;   // keys per K/V tile
  static constexpr int NCH = D / 64;                       // 128-byte chunks per row
  static constexpr int STAGES = (D == 64) ? 4 : 2;
  static constexpr bool SEP_P = (D == 64);                 // P in its own tensor-memory columns
  static constexpr int ISSUERS = SEP_P ? 2 : 1;            // MMA issuer warps
  static constexpr uint32_t CHUNK = 128u * 128u;           // 128 rows x 128 bytes
  static constexpr uint32_t TILE = CHUNK * NCH;            // 128 rows x D x 2 bytes
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + NQ * TILE;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + STAGES * TILE;
  // barriers: q_full, k_full[ST], k_empty[ST], v_full[ST], v_empty[ST], s_full[2], p_ready[2],
  //           s_consumed[2], o_ready[2], drain[2], exp_token[2]
  static constexpr int NBAR = 1 + 4 * STAGES + 8 + 2 + 2;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM = OFF_MISC + 16 + 1024;   // + slack for 1024-byte alignment
  static constexpr int THREADS = 352;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0;                     // + 128 t
  static constexpr uint32_t COL_O = 256;                   // + D t
  static constexpr uint32_t COL_P = SEP_P ? 256 + 2 * D : 0;  // + 64 t (SEP_P) / + 128 t

  __host__ __device__ static constexpr int bar_q() { return 0; }
  __host__ __device__ static constexpr int bar_kfull(int s) { return 1 + s; }
  __host__ __device__ static constexpr int bar_kempty(int s) { return 1 + STAGES + s; }
  __host__ __device__ static constexpr int bar_vfull(int s) { return 1 + 2 * STAGES + s; }
  __host__ __device__ static constexpr int bar_vempty(int s) { return 1 + 3 * STAGES + s; }
  __host__ __device__ static constexpr int bar_sfull(int t) { return 1 + 4 * STAGES + t; }
  __host__ __device__ static constexpr int bar_pready(int t) { return 3 + 4 * STAGES + t; }
  __host__ __device__ static constexpr int bar_sconsumed(int t) { return 5 + 4 * STAGES + t; }
  __host__ __device__ static constexpr int bar_oready(int t) { return 7 + 4 * STAGES + t; }
  __host__ __device__ static constexpr int bar_drain(int t) { return 9 + 4 * STAGES + t; }
  __host__ __device__ static constexpr int bar_token(int t) { return 11 + 4 * STAGES + t; }
  __host__ __device__ static constexpr uint32_t col_p(int t) { return COL_P + (SEP_P ? 64u : 128u) * t; }
};
static_assert(Cfg<128>::SMEM <= 227 * 1024, "shared memory budget");
static_assert(Cfg<64>::SMEM <= 227 * 1024, "shared memory budget");
static_assert(Cfg<64>::COL_P + 128 <= 512, "tensor memory budget");

struct Params {
  void* o;
  float* lse;
  long long o_sb, o_sg, o_sh, o_ss;  // O: batch, head group (grouped only), head, position
  int H, S, n_qblk;
  int hs_swap;                         // layouts 0/1: tensor-map dims (d, H, S, B) instead of (d, S, H, B)
  int hg, G;                           // grouped layout: heads per group, groups per batch
  float c;  // scale · log2(e)
  unsigned* status;
  long long limit;
};

__device__ __forceinline__ uint32_t code_of(uint32_t role, int j) {
  return (KID_FLASH << 24) | (role << 16) | (static_cast<uint32_t>(j) & 0xffffu);
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

template <int D, bool BF16, bool GROUPED>
__global__ void __launch_bounds__(352, 1)
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
      mbar_init(bar(C::bar_kempty(s)), C::ISSUERS);  // one commit per issuer
      mbar_init(bar(C::bar_vfull(s)), 1);
      mbar_init(bar(C::bar_vempty(s)), C::ISSUERS);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::bar_sfull(t)), 1);
      mbar_init(bar(C::bar_pready(t)), 128);
      mbar_init(bar(C::bar_sconsumed(t)), 128);
      mbar_init(bar(C::bar_oready(t)), 1);
      mbar_init(bar(C::bar_drain(t)), 1);
      mbar_init(bar(C::bar_token(t)), 128);
    }
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
  const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);
  const WaitCtx wc{abort_flag, p.status, p.limit};
  const bool skip = *abort_flag != 0;


  if (skip) {
    // nothing
  } else if (warp == 8) {
    // ------------------------------------------------------ TMA producer ----
    // (feature, position) -> tensor-map coordinates.  Layouts 0/1: maps
    // (d, S, H, B) or (d, H, S, B); grouped: (d, head within group, S,
    // group and batch).
    auto tma4 = [&](uint32_t dst, const CUtensorMap* m, uint32_t mbar, int e, int s) {
      if constexpr (GROUPED)
        tma_load_4d(dst, m, mbar, e, hh % p.hg, s, b * p.G + hh / p.hg);
      else if (p.hs_swap)
        tma_load_4d(dst, m, mbar, e, hh, s, b);
      else
        tma_load_4d(dst, m, mbar, e, s, hh, b);
    };
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
      for (int j = issued_k - C::STAGES < 0 ? 0 : issued_k - C::STAGES; j < issued_k; ++j)
        mbar_wait_slow(bar(C::bar_kfull(j % C::STAGES)), (j / C::STAGES) & 1, wc, 0, false);
      for (int j = issued_v - C::STAGES < 0 ? 0 : issued_v - C::STAGES; j < issued_v; ++j)
        mbar_wait_slow(bar(C::bar_vfull(j % C::STAGES)), (j / C::STAGES) & 1, wc, 0, false);
      mbar_wait_slow(bar(C::bar_q()), 0, wc, 0, false);
    }
  } else if (warp == 9 || (C::ISSUERS == 2 && warp == 10)) {
    // ------------------------------------------------ tcgen05 issuer(s) ----
    // The whole warp runs this code; elect.sync inside the issue helpers
    // picks the lane that issues each MMA and commit.
    constexpr uint32_t id_qk = idesc_f16(128, C::BN, BF16, false, false);
    constexpr uint32_t id_pv = idesc_f16(128, D, BF16, false, true);
    const int t_own = static_cast<int>(warp) - 9;  // the tile this warp issues for (two issuers)
    const uint64_t dk = sdesc_sw128(sb + C::OFF_K, 16, 1024);
    const uint64_t dv = sdesc_sw128(sb + C::OFF_V, C::CHUNK, 1024);
    auto qk = [&](int t, int s) {  // S_t = Q_t · K_s^T   (K-major A and B; address field += bytes/16)
      const uint64_t dq = sdesc_sw128(sb + C::OFF_Q + t * C::TILE, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
        mma_ss_elect(tmem + C::COL_S + t * 128, dq + off, dk + ((s * C::TILE) >> 4) + off, id_qk,
                     kk > 0 ? 1u : 0u);
      }
    };
    auto pv = [&](int t, int s, bool acc) {  // O_t (+)= P_t · V_s   (P in TMEM, V MN-major)
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk)
        mma_ts_elect(tmem + C::COL_O + t * D, tmem + C::col_p(t) + kk * 8,
                     dv + ((s * C::TILE + kk * 2048) >> 4), id_pv, (acc || kk > 0) ? 1u : 0u);
    };
    auto commit = [&](int i) { mma_commit_elect(bar(i)); };
    auto wait = [&](int i, int parity, int j) {
      return mbar_wait_warp(bar(i), parity, wc, code_of(ROLE_MMA, j));
    };
    bool ok = wait(C::bar_q(), 0, 0) && wait(C::bar_kfull(0), 0, 0);
    if constexpr (C::ISSUERS == 2) {
      // One pipeline per Q tile t: S_t(j+1) as soon as the softmax has read S_t(j).
      const int t = t_own;
      if (ok) {
        tc_fence_after();
        qk(t, 0);
        commit(C::bar_sfull(t));
        commit(C::bar_kempty(0));
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        const int s = j % C::STAGES, u = j / C::STAGES;
        const int s1 = (j + 1) % C::STAGES, u1 = (j + 1) / C::STAGES;
        if (j + 1 < n_kv) {
          if (!(ok = wait(C::bar_sconsumed(t), j & 1, j) && wait(C::bar_kfull(s1), u1 & 1, j))) break;
          tc_fence_after();
          qk(t, s1);
          commit(C::bar_sfull(t));
          commit(C::bar_kempty(s1));
        }
        if (!(ok = wait(C::bar_vfull(s), u & 1, j) && wait(C::bar_pready(t), j & 1, j))) break;
        tc_fence_after();
        pv(t, s, j > 0);
        commit(C::bar_oready(t));
        commit(C::bar_vempty(s));
      }
      if (!ok) {
        // Wait for the MMAs already issued before tensor memory is released.
        commit(C::bar_drain(t));
        mbar_wait_slow(bar(C::bar_drain(t)), 0, wc, 0, false);
      }
    } else {
      // One issuer, tiles in alternation; P overwrites S, so the next S_t is
      // issued after the P·V that reads P_t.
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
        if (!(ok = wait(C::bar_vfull(s), u & 1, j) && wait(C::bar_pready(0), j & 1, j))) break;
        tc_fence_after();
        pv(0, s, j > 0);
        if (more) {
          if (!(ok = wait(C::bar_kfull(s1), u1 & 1, j))) break;
          tc_fence_after();
          qk(0, s1);
        }
        commit(C::bar_sfull(0));  // S_0 of the next tile ready, or the final O_0
        if (!(ok = wait(C::bar_pready(1), j & 1, j))) break;
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
        commit(C::bar_drain(0));
        mbar_wait_slow(bar(C::bar_drain(0)), 0, wc, 0, false);
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------ softmax warps 0-7 ----
    const int t = static_cast<int>(warp) >> 2;   // Q tile
    const uint32_t wq = warp & 3u;               // tensor-memory sub-partition
    const uint32_t lane_off = (wq * 32u) << 16;
    const uint32_t tS = tmem + lane_off + C::COL_S + t * 128;
    const uint32_t tO = tmem + lane_off + C::COL_O + t * D;
    const uint32_t tP = tmem + lane_off + C::col_p(t);
    const float c = p.c;
    const uint64_t c2 = pk64(c, c);
    float m_ref = -INFINITY;  // running max (log2 units) that P and O are referenced to
    float l = 0.f;            // running sum of p
    bool ok = true;
    auto wait = [&](int i, int parity, int j) {
      return mbar_wait_warp(bar(i), parity, wc, code_of(ROLE_SOFTMAX, j));
    };
    uint32_t r[4][32];  // this thread's row of S_t (kept intact for a possible second pass)
    // p = 2^(s·c - m_ref) for the 128 keys, packed to 16-bit and stored to P_t
    // chunk by chunk; returns the sum of p and, in mx, the raw row max.
    auto exps_store = [&](float& mx) -> float {
      const uint64_t nm2 = pk64(-m_ref, -m_ref);
      uint64_t acc[4] = {0, 0, 0, 0};
      float mxc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float s0 = u2f(r[q][2 * i]), s1 = u2f(r[q][2 * i + 1]);
          mxc[i & 3] = max3(mxc[i & 3], s0, s1);
          float y0, y1;
          up64(ffma2(pk64(s0, s1), c2, nm2), y0, y1);
          const float e0 = ex2(y0), e1 = ex2(y1);
          acc[i & 3] = fadd2(acc[i & 3], pk64(e0, e1));
          pk[i] = pack2<BF16>(e0, e1);
        }
        tmem_st16(tP + q * 16, pk);  // P columns [16q, 16q+16) hold keys [32q, 32q+32)
      }
      mx = max3(mxc[0], mxc[1], fmaxf(mxc[2], mxc[3]));
      float a0, a1, a2, a3, a4, a5, a6, a7;
      up64(acc[0], a0, a1);
      up64(acc[1], a2, a3);
      up64(acc[2], a4, a5);
      up64(acc[3], a6, a7);
      return ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
    };
    if constexpr (C::SEP_P) {
    // d = 64: S_t is released to the next Q·K^T as soon as it is in
    // registers; the row max of the tile fixes the reference before any
    // exponential is taken, P is packed in place of S and stored at the end.
    // The two tiles' softmax warpgroups take turns on the exponential pass
    // (a token passed through an mbarrier), so that one runs it alone on the
    // special-function units while the other loads S, reduces and stores P.
    for (int j = 0; j < n_kv; ++j) {
      if (!(ok = wait(C::bar_sfull(t), j & 1, j))) break;
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, r[q]);
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld_wait(r[q]);
      tc_fence_before();
      mbar_arrive(bar(C::bar_sconsumed(t)));  // S_t may now be overwritten
      const int valid = p.S - j * C::BN;
      if (valid < C::BN) {  // ragged key tail: these columns do not exist
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (q * 32 + i >= valid) r[q][i] = f2u(-INFINITY);
      }
      float mxc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mxc[k] = u2f(r[k >> 1][(k & 1) * 16]);
#pragma unroll
      for (int i = 0; i < 16; i += 2)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mxc[k] = max3(mxc[k], u2f(r[k >> 1][(k & 1) * 16 + i]), u2f(r[k >> 1][(k & 1) * 16 + i + 1]));
      const float m_blk =
          max3(max3(mxc[0], mxc[1], mxc[2]), max3(mxc[3], mxc[4], mxc[5]), fmaxf(mxc[6], mxc[7])) * c;
      const bool move = m_blk > m_ref + kRescaleThreshold;  // always on the first tile
      const bool any_move = __any_sync(0xffffffffu, move);
      float alpha = 1.f;
      if (any_move) {  // warp-uniform; rare after the first tile
        const float m_new = move ? m_blk : m_ref;
        alpha = ex2(m_ref - m_new);
        l *= alpha;
        m_ref = m_new;
      }
      if (kExpToken && (t == 1 || j > 0)) {
        // tile 1 follows tile 0 of the same key block, tile 0 follows tile 1 of the previous one
        if (!(ok = wait(C::bar_token(t), (t == 1 ? j : j - 1) & 1, j))) break;
      }
      {
        const uint64_t nm2 = pk64(-m_ref, -m_ref);
        uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float y0, y1;
            up64(ffma2(pk64(u2f(r[q][2 * i]), u2f(r[q][2 * i + 1])), c2, nm2), y0, y1);
            const float e0 = ex2(y0), e1 = ex2(y1);
            acc[i & 3] = fadd2(acc[i & 3], pk64(e0, e1));
            r[q][i] = pack2<BF16>(e0, e1);  // r[q][i] is no longer needed as S
          }
        }
        if (kExpToken) mbar_arrive(bar(C::bar_token(1 - t)));
        float a0, a1, a2, a3, a4, a5, a6, a7;
        up64(acc[0], a0, a1);
        up64(acc[1], a2, a3);
        up64(acc[2], a4, a5);
        up64(acc[3], a6, a7);
        l += ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
      }
      if (j > 0) {  // P_t and O_t are free once the previous P·V has completed
        if (!(ok = wait(C::bar_oready(t), (j - 1) & 1, j))) break;
        tc_fence_after();
        if (any_move) {
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
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t(&pk)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&r[q][0]);
        tmem_st16(tP + q * 16, pk);  // P columns [16q, 16q+16) hold keys [32q, 32q+32)
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::bar_pready(t)));
    }
    } else {
    for (int j = 0; j < n_kv; ++j) {
      if (!(ok = wait(C::bar_sfull(t), j & 1, j))) break;
      tc_fence_after();
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
      if (j == 0) {  // empty history: the reference is this tile's max
        float mxc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int i = 0; i < 16; ++i)
            mxc[i & 3] = max3(mxc[i & 3], u2f(r[q][2 * i]), u2f(r[q][2 * i + 1]));
        m_ref = max3(mxc[0], mxc[1], fmaxf(mxc[2], mxc[3])) * c;
      }
      // One pass against the current reference, tracking the row max.
      float mx;
      float sum = exps_store(mx);
      const float m_blk = mx * c;
      const bool move = m_blk > m_ref + kRescaleThreshold;
      if (__any_sync(0xffffffffu, move)) {  // rare: recompute P, rescale O (warp-uniform)
        const float m_new = move ? m_blk : m_ref;
        const float alpha = ex2(m_ref - m_new);
        l *= alpha;
        m_ref = m_new;
        tmem_st_wait();
        sum = exps_store(mx);
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
      l += sum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::bar_pready(t)));
    }
    }
    if (ok) {
      if constexpr (C::SEP_P)
        ok = wait(C::bar_oready(t), (n_kv - 1) & 1, n_kv);
      else
        ok = wait(C::bar_sfull(t), n_kv & 1, n_kv);
    }
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l;
      const int row = q0 + t * C::BM + static_cast<int>(wq * 32 + lane);
      const bool in = row < p.S;
      using Elem = uint16_t;
      const long long head_off = GROUPED ? (hh / p.hg) * p.o_sg + (hh % p.hg) * p.o_sh
                                         : static_cast<long long>(hh) * p.o_sh;
      Elem* out = static_cast<Elem*>(p.o) + b * p.o_sb + head_off +
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

template <int D, bool BF16, bool GROUPED>
cudaError_t launch_impl(const FlashLaunch& a, cudaStream_t st) {
  using C = Cfg<D>;
  auto kern = flash_fwd_kernel<D, BF16, GROUPED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  Params p;
  p.o = a.o;
  p.lse = a.lse;
  p.o_sb = a.o_sb;
  p.o_sg = a.o_sg;
  p.o_sh = a.o_sh;
  p.o_ss = a.o_ss;
  p.H = a.H;
  p.S = a.S;
  p.n_qblk = (a.S + C::NQ * C::BM - 1) / (C::NQ * C::BM);
  p.hs_swap = a.hs_swap;
  p.hg = a.hg;
  p.G = a.H / a.hg;
  p.c = a.scale * kLog2e;
  p.status = a.status;
  p.limit = a.limit;
  const long long grid = static_cast<long long>(a.B) * a.H * p.n_qblk;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, st>>>(a.tq, a.tk, a.tv, p);
  return cudaGetLastError();
}

}  // namespace

template <bool G>
cudaError_t launch_g(const FlashLaunch& a, cudaStream_t st) {
  if (a.d == 64) return a.bf16 ? launch_impl<64, true, G>(a, st) : launch_impl<64, false, G>(a, st);
  if (a.d == 128) return a.bf16 ? launch_impl<128, true, G>(a, st) : launch_impl<128, false, G>(a, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_flash_fwd(const FlashLaunch& a, cudaStream_t st) {
  return a.grouped ? launch_g<true>(a, st) : launch_g<false>(a, st);
}

}  // namespace attn
