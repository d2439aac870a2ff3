// Fused QKV projection + attention in one kernel, for sm_103a (GB300).
//
// "Transformer算子生态深度分析" ch.2 §2.7 (算子层面的优化要点) names the fusion
// of the QKV projection with the attention that follows it, so that the
// projected Q, K, V go straight into the attention instead of making a round
// trip through memory; §2.1 (QKV投影) defines the projection with the fused
// [D, 3D] weight (columns [0, D) give Q, [D, 2D) K, [2D, 3D) V, head-major).
// The attention itself is the online softmax of §2.6, as in flash_fwd.cu.
//
// Scope: d = 64 and S <= 512 -- one head's Q, K and V for the whole sequence
// then fit in shared memory (192 KB) and their fp32 accumulators in tensor
// memory.  That is the short-sequence, BERT-like regime in which the
// projection dominates; longer sequences use the two-launch qkv_proj_attn.
//
// One CTA per (batch, head), 12 warps:
//   warp 8     TMA producer;
//   warp 9     tcgen05 issuer;
//   warps 0-7  epilogue / softmax: warpgroup t owns query block t of the
//              current pair, one thread per row (tensor-memory lane);
//   warps 10-11 spare.
// Phase Q   Q = X_b · W_q,h for all S rows: one N = 64 MMA per 16-wide k-step
//           and 128-row block, each k-chunk of X loaded once for all blocks
//           and the weight chunk shared by them; the epilogue warps round the
//           accumulators to the 16-bit type into shared memory, in the
//           128-byte-swizzled layout that TMA would have produced (the A
//           operand of Q·K^T).
// Phase KV  [K | V] = X_b · [W_k,h | W_v,h]: one N = 128 MMA per k-step and
//           block (K in the accumulator's first 64 columns, V in the next 64),
//           rounded into shared memory the same way (K: B operand of Q·K^T,
//           V: B operand of P·V, both row-major by key).
// Attention for each pair of 128-row query blocks against the shared-memory
//           K and V: the tensor cores compute one block's products while the
//           softmax warps of the other run.  The output rows leave through
//           the pair's Q tiles (free once its Q·K^T products are done) as
//           whole 128-byte row segments.
// Tensor memory: phase Q block r in columns 64r..; phase KV block r in
// columns 128r..; attention S0 | S1 | O0 | O1 | P0 | P1 (128+128+64+64+64+64).
// Shared memory: Q tiles | K tiles | V tiles (64 KB each); the projection
// ring (two stages of 80 KB) overlaps the K and V tiles, which are written
// only once every load has been consumed.
// Every wait is bounded; a stall records a code in the device status word and
// the CTA winds down instead of hanging.

#include "common.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kThresholdF = 8.0f;  // lazy rescale: move the reference when the max grows by > 2^8

struct FCfg {
  static constexpr int MAXT = 4;                         // 128-row blocks (S <= 512)
  static constexpr uint32_t TILE = 128 * 128;            // 128 rows x 64 elements x 2 bytes
  static constexpr uint32_t WCH = 64 * 128;              // weight chunk: 64 k-rows x 64 columns
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = MAXT * TILE;
  static constexpr uint32_t OFF_V = 2 * MAXT * TILE;
  static constexpr uint32_t OFF_R = MAXT * TILE;         // projection ring (overlaps K, V)
  static constexpr uint32_t STAGE = MAXT * TILE + 2 * WCH;  // X tiles of every block + one or two weight chunks
  static constexpr uint32_t OFF_BAR = OFF_R + 2 * STAGE;
  static constexpr int NBAR = 26;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 384;
  static constexpr uint32_t COL_O = 256, COL_P = 384;
  // barriers
  __host__ __device__ static constexpr int full(int s) { return s; }
  __host__ __device__ static constexpr int empty(int s) { return 2 + s; }
  static constexpr int QACC = 4, QREADY = 5, KVACC = 6, KVREADY = 7, QFREE = 8, DRAIN = 9;
  __host__ __device__ static constexpr int sfull(int t) { return 10 + t; }
  __host__ __device__ static constexpr int sconsumed(int t) { return 12 + t; }
  __host__ __device__ static constexpr int pready(int t) { return 14 + t; }
  __host__ __device__ static constexpr int oready(int t) { return 16 + t; }
  __host__ __device__ static constexpr int ofree(int t) { return 18 + t; }
  // attention only: K and V tile j landed (the Q tiles of pair pr use full(pr))
  __host__ __device__ static constexpr int kvfull(int j) { return 20 + j; }
  // output rows of query block t of the current pair staged in shared memory
  __host__ __device__ static constexpr int ostaged(int t) { return 24 + t; }
};
static_assert(FCfg::OFF_R + 2 * FCfg::STAGE <= FCfg::OFF_BAR && FCfg::OFF_V + FCfg::MAXT * FCfg::TILE <= FCfg::OFF_BAR,
              "buffers inside the shared-memory budget");
static_assert(FCfg::SMEM <= 227 * 1024, "shared memory budget");

struct FParams {
  float* lse;              // [B, H, S] fp32 or null
  int o_swap;              // output map dims (d, H, S, B) instead of (d, S, H, B)
  int S, H, D;             // sequence length, heads, model width (projection: H * 64)
  int nkc;                 // projection: D / 64 k-chunks
  int hs_swap;             // attention only: maps (d, H, S, B) instead of (d, S, H, B)
  float c;                 // softmax scale * log2(e)
  unsigned* status;
  long long limit;
};

__device__ __forceinline__ uint32_t fcode(uint32_t role, uint32_t j) {
  return (KID_FUSED << 24) | (role << 16) | (j & 0xffffu);
}

// 64 fp32 values of one row -> 16-bit -> row r of a 128-byte-swizzled tile
// (16-byte unit u of row r at u ^ (r mod 8), the TMA SWIZZLE_128B layout).
template <bool BF16>
__device__ __forceinline__ void store_row_swizzled(uint8_t* tile, int r, const uint32_t (&a)[32],
                                                   const uint32_t (&b)[32]) {
  uint32_t pk[32];
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[16 + i] = pack2<BF16>(__uint_as_float(b[2 * i]), __uint_as_float(b[2 * i + 1]));
  uint8_t* row = tile + r * 128;
#pragma unroll
  for (int u = 0; u < 8; ++u)
    *reinterpret_cast<uint4*>(row + ((u ^ (r & 7)) << 4)) =
        make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
}

// PROJ: the projection phases run first (t0 = X, t1 = W_qkv).  Otherwise the
// kernel is the attention alone on Q, K, V that already exist (t0, t1, t2,
// 4-d maps (d, S, H, B) or (d, H, S, B)): they are loaded straight into the
// same resident tiles.
template <bool BF16, bool PROJ>
__global__ void __launch_bounds__(384, 1)
    fused_qkv_attn_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw,
                          const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                          const __grid_constant__ FParams p) {
  using C = FCfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sb - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };

  const uint32_t warp = warp_id(), lane = lane_id();
  const int b = static_cast<int>(blockIdx.x) / p.H, hh = static_cast<int>(blockIdx.x) % p.H;
  const int nt = (p.S + 127) / 128;        // 128-row blocks (= key tiles)
  const int npair = (nt + 1) / 2;          // pairs of query blocks

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::full(s)), 1);
      mbar_init(bar(C::empty(s)), 1);
    }
    mbar_init(bar(C::QACC), 1);
    mbar_init(bar(C::QREADY), 256);
    mbar_init(bar(C::KVACC), 1);
    mbar_init(bar(C::KVREADY), 256);
    mbar_init(bar(C::QFREE), 1);
    mbar_init(bar(C::DRAIN), 1);
    for (int j = 0; j < C::MAXT; ++j) mbar_init(bar(C::kvfull(j)), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::sfull(t)), 1);
      mbar_init(bar(C::sconsumed(t)), 128);
      mbar_init(bar(C::pready(t)), 128);
      mbar_init(bar(C::oready(t)), 1);
      mbar_init(bar(C::ofree(t)), 128);
      mbar_init(bar(C::ostaged(t)), 128);
    }
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  griddep_wait();
  if (threadIdx.x == 0) {
    *abort_flag = (*reinterpret_cast<volatile unsigned*>(p.status) != 0u) ? 1 : 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);
  const WaitCtx wc{abort_flag, p.status, p.limit};
  const bool skip = *abort_flag != 0;

  if (skip) {
  } else if (warp == 8) {
    // ------------------------------------------------------ TMA producer ----
    // Ring stage s at OFF_R + s·STAGE: the X tiles of every block for one
    // k-chunk, then the weight chunk(s): W_q (phase Q) or W_k, W_v (phase KV).
    if (lane == 0) {
      prefetch_tmap(&tx);
      prefetch_tmap(&tw);
      if (!PROJ) prefetch_tmap(&tv);
    }
    bool ok = true;
    int g = 0;  // ring loads issued (both phases)
    if constexpr (!PROJ) {
      // The first pair's Q tiles, then K and V tile by tile, then the second
      // pair's Q tiles (rows past S read as zeros), each group on its own
      // barrier so that the attention starts once its first tiles are in.
      if (lane == 0) {
        auto load = [&](uint32_t dst, const CUtensorMap* m, uint32_t mbar, int row) {
          if (p.hs_swap)
            tma_load_4d(dst, m, mbar, 0, hh, row, b);
          else
            tma_load_4d(dst, m, mbar, 0, row, hh, b);
        };
        auto load_q = [&](int pr) {
          mbar_expect_tx(bar(C::full(pr)), 2 * C::TILE);
          for (int qb = 2 * pr; qb < 2 * pr + 2; ++qb)
            load(sb + C::OFF_Q + qb * C::TILE, &tx, bar(C::full(pr)), qb * 128);
        };
        load_q(0);
        for (int j = 0; j < nt; ++j) {
          mbar_expect_tx(bar(C::kvfull(j)), 2 * C::TILE);
          load(sb + C::OFF_K + j * C::TILE, &tw, bar(C::kvfull(j)), j * 128);
          load(sb + C::OFF_V + j * C::TILE, &tv, bar(C::kvfull(j)), j * 128);
        }
        if (npair > 1) load_q(1);
      }
      // Every copy lands before the CTA can exit, even if another role gives up.
      for (int pr = 0; pr < npair; ++pr) mbar_wait_slow(bar(C::full(pr)), 0, wc, 0, false);
      for (int j = 0; j < nt; ++j) mbar_wait_slow(bar(C::kvfull(j)), 0, wc, 0, false);
    }
    for (int ph = 0; PROJ && ph < 2 && ok; ++ph) {
      for (int kc = 0; kc < p.nkc; ++kc, ++g) {
        const int s = g & 1, u = g >> 1;
        if (u > 0 && !(ok = mbar_wait_warp(bar(C::empty(s)), (u - 1) & 1, wc, fcode(ROLE_LOAD, g)))) break;
        if (lane == 0) {
          const uint32_t st = sb + C::OFF_R + s * C::STAGE;
          mbar_expect_tx(bar(C::full(s)), nt * C::TILE + (ph == 0 ? 1 : 2) * C::WCH);
          for (int r = 0; r < nt; ++r) tma_load_3d(st + r * C::TILE, &tx, bar(C::full(s)), kc * 64, r * 128, b);
          if (ph == 0) {
            tma_load_2d(st + C::MAXT * C::TILE, &tw, bar(C::full(s)), hh * 64, kc * 64);
          } else {
            tma_load_2d(st + C::MAXT * C::TILE, &tw, bar(C::full(s)), p.D + hh * 64, kc * 64);
            tma_load_2d(st + C::MAXT * C::TILE + C::WCH, &tw, bar(C::full(s)), 2 * p.D + hh * 64, kc * 64);
          }
        }
      }
    }
    if (!ok) {  // let the copies in flight land before the CTA can exit
      for (int q = g - 2 < 0 ? 0 : g - 2; q < g; ++q)
        mbar_wait_slow(bar(C::full(q & 1)), (q >> 1) & 1, wc, 0, false);
    }
  } else if (warp == 9) {
    // ------------------------------------------------- tcgen05 issuer ----
    constexpr uint32_t id_q = idesc_f16(128, 64, BF16, false, true);     // X · W_q
    constexpr uint32_t id_kv = idesc_f16(128, 128, BF16, false, true);   // X · [W_k | W_v]
    constexpr uint32_t id_qk = idesc_f16(128, 128, BF16, false, false);  // Q · K^T
    constexpr uint32_t id_pv = idesc_f16(128, 64, BF16, false, true);    // P · V
    auto wait = [&](int i, uint32_t parity, uint32_t j) {
      return mbar_wait_warp(bar(i), parity, wc, fcode(ROLE_MMA, j));
    };
    auto commit = [&](int i) { mma_commit_elect(bar(i)); };
    bool ok = true;
    int g = 0;
    for (int ph = 0; PROJ && ph < 2 && ok; ++ph) {
      // Phase KV overwrites the Q accumulators: only once they are in shared memory.
      if (ph == 1 && !(ok = wait(C::QREADY, 0, 0))) break;
      for (int kc = 0; kc < p.nkc; ++kc, ++g) {
        const int s = g & 1;
        if (!(ok = wait(C::full(s), (g >> 1) & 1, g))) break;
        tc_fence_after();
        const uint32_t st = sb + C::OFF_R + s * C::STAGE;
        const uint64_t dw = sdesc_sw128(st + C::MAXT * C::TILE, C::WCH, 1024);
        for (int r = 0; r < nt; ++r) {
          const uint64_t dx = sdesc_sw128(st + r * C::TILE, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss_elect(tmem + r * (ph == 0 ? 64 : 128), dx + ((kk * 32) >> 4), dw + ((kk * 2048) >> 4),
                         ph == 0 ? id_q : id_kv, (kc > 0 || kk > 0) ? 1u : 0u);
        }
        commit(C::empty(s));
      }
      if (ok) commit(ph == 0 ? C::QACC : C::KVACC);
    }
    if (PROJ && ok) ok = wait(C::KVREADY, 0, 0);
    auto qk = [&](int t, int qb, int j) {  // S_t = Q_qb · K_j^T
      const uint64_t dq = sdesc_sw128(sb + C::OFF_Q + qb * C::TILE, 16, 1024);
      const uint64_t dk = sdesc_sw128(sb + C::OFF_K + j * C::TILE, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ss_elect(tmem + t * 128, dq + ((kk * 32) >> 4), dk + ((kk * 32) >> 4), id_qk, kk > 0 ? 1u : 0u);
    };
    auto pv = [&](int t, int j) {  // O_t (+)= P_t · V_j
      const uint64_t dv = sdesc_sw128(sb + C::OFF_V + j * C::TILE, C::TILE, 1024);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts_elect(tmem + C::COL_O + t * 64, tmem + C::COL_P + t * 64 + kk * 8, dv + ((kk * 2048) >> 4), id_pv,
                     (j > 0 || kk > 0) ? 1u : 0u);
    };
    uint32_t n = 0;  // key tiles of both blocks done (attention barrier phases)
    for (int pr = 0; pr < npair && ok; ++pr) {
      if (!PROJ && !(ok = wait(C::full(pr), 0, pr) && wait(C::kvfull(0), 0, 0))) break;
      tc_fence_after();
      qk(0, 2 * pr, 0);
      commit(C::sfull(0));
      qk(1, 2 * pr + 1, 0);
      commit(C::sfull(1));
      for (int j = 0; j < nt && ok; ++j, ++n) {
        for (int t = 0; t < 2; ++t) {
          if (!(ok = wait(C::sconsumed(t), n & 1, n))) break;
          if (j + 1 < nt) {
            if (!PROJ && t == 0 && !(ok = wait(C::kvfull(j + 1), 0, j + 1))) break;
            tc_fence_after();
            qk(t, 2 * pr + t, j + 1);
            commit(C::sfull(t));
          }
        }
        if (!ok) break;
        if (j + 1 == nt) commit(C::QFREE);  // the pair's Q tiles are free once these products are done
        for (int t = 0; t < 2; ++t) {
          if (!(ok = wait(C::pready(t), n & 1, n))) break;
          if (j == 0 && pr > 0 && !(ok = wait(C::ofree(t), (pr - 1) & 1, n))) break;
          tc_fence_after();
          pv(t, j);
          commit(C::oready(t));
        }
      }
    }
    if (!ok) {
      commit(C::DRAIN);
      mbar_wait_slow(bar(C::DRAIN), 0, wc, 0, false);
    }
  } else if (warp < 8) {
    // -------------------------------------- epilogue / softmax warps 0-7 ----
    const int t = static_cast<int>(warp) >> 2;
    const uint32_t wq = warp & 3u;
    const int r = static_cast<int>(wq * 32u + lane);  // row within a 128-row block
    const uint32_t lane_off = (wq * 32u) << 16;
    auto wait = [&](int i, uint32_t parity, uint32_t j) {
      return mbar_wait_warp(bar(i), parity, wc, fcode(ROLE_SOFTMAX, j));
    };
    // Phase Q epilogue: warpgroup t rounds blocks t and t + 2 (a block past the
    // sequence that a pair still needs gets zeros).
    bool ok = !PROJ || wait(C::QACC, 0, 0);
    if (PROJ && ok) {
      tc_fence_after();
      for (int qb = t; qb < 2 * npair; qb += 2) {
        uint32_t a[32], c[32];
        if (qb < nt) {
          tmem_ld32(tmem + lane_off + qb * 64, a);
          tmem_ld32(tmem + lane_off + qb * 64 + 32, c);
          tmem_ld_wait(a);
          tmem_ld_wait(c);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = c[i] = 0u;
        }
        store_row_swizzled<BF16>(smem + C::OFF_Q + qb * C::TILE, r, a, c);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::QREADY));
      ok = wait(C::KVACC, 0, 0);
    }
    if (PROJ && ok) {
      // Phase KV epilogue: row r of every block, K (t = 0) or V (t = 1) half.
      tc_fence_after();
      uint8_t* dst = smem + (t == 0 ? C::OFF_K : C::OFF_V);
      for (int rb = 0; rb < nt; ++rb) {
        uint32_t a[32], c[32];
        tmem_ld32(tmem + lane_off + rb * 128 + t * 64, a);
        tmem_ld32(tmem + lane_off + rb * 128 + t * 64 + 32, c);
        tmem_ld_wait(a);
        tmem_ld_wait(c);
        store_row_swizzled<BF16>(dst + rb * C::TILE, r, a, c);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::KVREADY));
    }
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + C::COL_O + t * 64;
    const uint32_t tP = tmem + lane_off + C::COL_P + t * 64;
    const float cs = p.c;
    const uint64_t c2 = pk64(cs, cs);
    uint32_t n = 0;
    uint32_t s_row[4][32];
    for (int pr = 0; pr < npair && ok; ++pr) {
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j, ++n) {
        if (!(ok = wait(C::sfull(t), n & 1, n))) break;
        tc_fence_after();
        float mq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32_max(tS + q * 32, s_row[q], mq[q]);
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld_wait(s_row[q], mq[q]);
        tc_fence_before();
        mbar_arrive(bar(C::sconsumed(t)));
        const int valid = p.S - j * 128;
        if (valid < 128) {  // keys past S do not exist
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (q * 32 + i >= valid) s_row[q][i] = __float_as_uint(-INFINITY);
              mx = fmaxf(mx, __uint_as_float(s_row[q][i]));
            }
            mq[q] = mx;
          }
        }
        const float m_blk = max3(mq[0], mq[1], fmaxf(mq[2], mq[3])) * cs;
        const bool move = m_blk > m_ref + kThresholdF;  // always on the first key tile
        const bool any_move = __any_sync(0xffffffffu, move);
        float alpha = 1.f;
        if (any_move) {
          const float m_new = move ? m_blk : m_ref;
          alpha = ex2(m_ref - m_new);
          l *= alpha;
          m_ref = m_new;
        }
        {
          const uint64_t nm2 = pk64(-m_ref, -m_ref);
          uint64_t acc[2] = {0, 0};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float y0, y1;
              up64(ffma2(pk64(__uint_as_float(s_row[q][2 * i]), __uint_as_float(s_row[q][2 * i + 1])), c2, nm2),
                   y0, y1);
              const float e0 = ex2(y0), e1 = ex2(y1);
              acc[i & 1] = fadd2(acc[i & 1], pk64(e0, e1));
              s_row[q][i] = pack2<BF16>(e0, e1);
            }
          }
          float a0, a1, a2, a3;
          up64(acc[0], a0, a1);
          up64(acc[1], a2, a3);
          l += (a0 + a1) + (a2 + a3);
        }
        // P_t and O_t are free once the previous P·V of this block has completed.
        if (n > 0) {
          if (!(ok = wait(C::oready(t), (n - 1) & 1, n))) break;
          tc_fence_after();
          if (j > 0 && any_move) {
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
              uint32_t o[32];
              tmem_ld32(tO + cc * 32, o);
              tmem_ld_wait(o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(tO + cc * 32, o);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t(&pk)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&s_row[q][0]);
          tmem_st16(tP + q * 16, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::pready(t)));
      }
      if (!ok) break;
      // Output rows of block 2·pr + t: O / l -> 16-bit, written into that
      // block's Q tile (free once the pair's Q·K^T products are done) in the
      // 128-byte-swizzled layout, then stored by one TMA bulk copy while the
      // warps go on with the next pair.
      if (!(ok = wait(C::oready(t), (n - 1) & 1, n))) break;
      tc_fence_after();
      const float inv = 1.f / l;
      uint32_t o0[32], o1[32];
      tmem_ld32(tO, o0);
      tmem_ld32(tO + 32, o1);
      tmem_ld_wait(o0);
      tmem_ld_wait(o1);
      tc_fence_before();
      mbar_arrive(bar(C::ofree(t)));
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        o0[i] = __float_as_uint(__uint_as_float(o0[i]) * inv);
        o1[i] = __float_as_uint(__uint_as_float(o1[i]) * inv);
      }
      const int blk = 2 * pr + t;
      const int my_row = blk * 128 + r;
      if (p.lse && my_row < p.S)
        p.lse[(static_cast<long long>(b) * p.H + hh) * p.S + my_row] = (m_ref + log2f(l)) * 0.6931471805599453f;
      if (!(ok = wait(C::QFREE, pr & 1, n))) break;  // the pair's Q·K^T products no longer read its Q tiles
      store_row_swizzled<BF16>(smem + C::OFF_Q + blk * C::TILE, r, o0, o1);
      fence_proxy_async_smem();
      mbar_arrive(bar(C::ostaged(t)));
      // The warpgroup's first warp waits (bounded, warp-uniform) for the
      // block's 128 rows; one of its threads stores them.
      if (wq == 0 && !(ok = wait(C::ostaged(t), pr & 1, pr))) break;
      if (r == 0 && blk * 128 < p.S) {
        if (p.o_swap)
          tma_store_4d(&to, sb + C::OFF_Q + blk * C::TILE, 0, hh, blk * 128, b);
        else
          tma_store_4d(&to, sb + C::OFF_Q + blk * C::TILE, 0, blk * 128, hh, b);
        bulk_commit();
      }
    }
    if (r == 0) bulk_wait_all();  // the output copies complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool BF16, bool PROJ>
cudaError_t launch_fused_t(const FusedLaunch& a, cudaStream_t st) {
  auto kern = fused_qkv_attn_kernel<BF16, PROJ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FCfg::SMEM);
  if (e != cudaSuccess) return e;
  FParams p{};
  p.lse = a.lse;
  p.o_swap = a.o_swap;
  p.S = a.S;
  p.H = a.H;
  p.D = a.D;
  p.nkc = a.D / 64;
  p.hs_swap = a.hs_swap;
  p.c = a.scale * kLog2eF;
  p.status = a.status;
  p.limit = a.limit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B * a.H));
  cfg.blockDim = dim3(FCfg::THREADS);
  cfg.dynamicSmemBytes = FCfg::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a.t0, a.t1, a.t2, a.to, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fused_qkv_attn(const FusedLaunch& a, cudaStream_t st) {
  if (a.S < 1 || a.S > 512 || a.H < 1 || a.B < 1 || static_cast<long long>(a.B) * a.H > 0x7fffffffLL)
    return cudaErrorInvalidValue;
  if (a.project)
    return a.bf16 ? launch_fused_t<true, true>(a, st) : launch_fused_t<false, true>(a, st);
  return a.bf16 ? launch_fused_t<true, false>(a, st) : launch_fused_t<false, false>(a, st);
}

}  // namespace attn
