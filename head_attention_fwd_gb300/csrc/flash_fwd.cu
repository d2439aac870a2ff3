// Fused multi-head attention forward for sm_103a (GB300).
//
// Computes O = softmax(scale · Q·K^T) · V tile by tile with the online
// softmax of "Transformer算子生态深度分析" ch.2 §2.6: per key tile the row
// maximum and exp-sum are merged into running statistics and the partial
// output is rescaled by exp(m_old - m), so the S×S scores never leave the SM
// ("WebGPU 算子优化：QKV 内存合并与 FlashAttention 分块计算",
// §FlashAttention 分块计算原理与浏览器适配, gives the same merge rule).
//
// GB300 mapping (at most one CTA per SM, 11 warps, 192 KB of shared memory):
//   * work item = one (batch, head) and two 128-row Q tiles -- "ping-pong":
//     while one tile's softmax runs on the CUDA cores, the tensor cores work
//     on the other tile;
//   * each CTA walks a list of segments: an item and a run of its key tiles
//     (see Mode).  d = 128: one item per CTA.  d = 64: a persistent grid
//     deals whole items round-robin (item i on CTA i mod grid); given a
//     scratch buffer, the last one to two waves of items are instead cut
//     into equal runs of key tiles, [g·U/grid, (g+1)·U/grid) for CTA g, so
//     that every SM ends at the same time.  A cut item's later pieces leave
//     their (m, l, unnormalised O) in the scratch; the CTA holding the piece
//     that starts at key 0 merges them into its own with the same
//     rescale-and-add rule that merges key tiles;
//   * launched as a programmatic dependent: barrier set-up, tensor-memory
//     allocation and an L2 prefetch of the first tiles overlap the previous
//     grid; global memory is read only after griddepcontrol.wait;
//   * warp 8: TMA producer.  Q tiles once per segment (at d = 64 into one of
//     two buffers, so the next item's Q arrives during this one), then K and
//     V tiles of 128 keys through a STAGES-deep ring of 128-byte-swizzled
//     shared-memory buffers that runs on across segments;
//   * tcgen05 issue: S_t = Q_t·K_j^T into tensor memory (fp32), then
//     O_t += P_t·V_j with P_t read straight from tensor memory.  At d = 64
//     warps 9 / 10 issue for Q tile 0 / 1, so the two tiles' pipelines are
//     independent and share only the K/V ring; at d = 128 (tensor-bound)
//     warp 9 issues both tiles in alternation;
//   * warps 0-3 / 4-7: softmax of Q tile 0 / 1, one thread per query row
//     (tensor-memory lane = row), so the row max and row sum are
//     thread-local.  S is read with tcgen05.ld.red (sm_103a), which hands
//     back each 32-column chunk's maximum with the data, so the tile max
//     costs three max operations instead of a pass over the row.  exp is
//     2^x on the SFU with scale·log2(e) folded into one packed FFMA; sums use
//     packed fp32 adds.  The running max only moves when the tile max exceeds
//     it by more than 2^8 (a factor of 256 in p, safe in fp16 and bf16); the
//     result is exact either way because O and l always share the same
//     reference.  When some row's max does move (rare after the first tile),
//     the warp rescales O in tensor memory before it writes P;
//   * tensor memory, d = 64:  S0 | S1 | O0 | O1 | P0 | P1 (128+128+64+64+64+64)
//     P has its own columns, so the next Q·K^T can be issued as soon as the
//     softmax has read S, while it is still computing exponentials;
//     d = 128: S0 | S1 | O0 | O1 (128+128+128+128); P overwrites the first
//     64 columns of S, so the next Q·K^T waits for the P·V that reads it.
//     O_t of the next segment is started only after the softmax warps have
//     read this segment's O_t (barrier o_free);
//   * each issuer warp issues from a converged warp (elect.sync picks the
//     lane), so descriptors stay warp-uniform.
// Every wait is bounded: a pipeline stall records a code in the device
// status word and the CTA winds down instead of hanging.

#include <stdlib.h>
#include <string.h>

#include "common.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr bool kExpToken = true;           // d = 64: softmax warpgroups alternate on the exp pass
constexpr int kItemRows = 256;             // query rows per work item (two Q tiles)

template <int D>
struct Cfg {
  static constexpr int BM = 128;   // rows per Q tile (= tensor-memory lanes)
  static constexpr int NQ = 2;     // Q tiles per item
  static constexpr int BN = 128;   // keys per K/V tile
  static constexpr int NCH = D / 64;                       // 128-byte chunks per row
  static constexpr int STAGES = (D == 64) ? 4 : 2;
  static constexpr int NQB = (D == 64) ? 2 : 1;            // Q buffer sets
  static constexpr bool SEP_P = (D == 64);                 // P in its own tensor-memory columns
  static constexpr int ISSUERS = SEP_P ? 2 : 1;            // MMA issuer warps
  static constexpr uint32_t CHUNK = 128u * 128u;           // 128 rows x 128 bytes
  static constexpr uint32_t TILE = CHUNK * NCH;            // 128 rows x D x 2 bytes
  static constexpr uint32_t QSET = NQ * TILE;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + NQB * QSET;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + STAGES * TILE;
  // barriers: q_full[NQB], q_empty[NQB], k_full[ST], k_empty[ST], v_full[ST], v_empty[ST],
  //           then per Q tile: s_full, p_ready, s_consumed, o_ready, drain, exp_token, o_free
  static constexpr int NBAR = 2 * NQB + 4 * STAGES + 14;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t OFF_WORK = OFF_MISC + 16;     // CtaWork
  static constexpr uint32_t SMEM = OFF_WORK + 32 + 1024;   // + slack for 1024-byte alignment
  static constexpr int THREADS = 352;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0;                     // + 128 t
  static constexpr uint32_t COL_O = 256;                   // + D t
  static constexpr uint32_t COL_P = SEP_P ? 256 + 2 * D : 0;  // + 64 t (SEP_P) / + 128 t

  static constexpr int KB = 2 * NQB;
  static constexpr int TB = KB + 4 * STAGES;
  __host__ __device__ static constexpr int bar_qfull(int b) { return b; }
  __host__ __device__ static constexpr int bar_qempty(int b) { return NQB + b; }
  __host__ __device__ static constexpr int bar_kfull(int s) { return KB + s; }
  __host__ __device__ static constexpr int bar_kempty(int s) { return KB + STAGES + s; }
  __host__ __device__ static constexpr int bar_vfull(int s) { return KB + 2 * STAGES + s; }
  __host__ __device__ static constexpr int bar_vempty(int s) { return KB + 3 * STAGES + s; }
  __host__ __device__ static constexpr int bar_sfull(int t) { return TB + t; }
  __host__ __device__ static constexpr int bar_pready(int t) { return TB + 2 + t; }
  __host__ __device__ static constexpr int bar_sconsumed(int t) { return TB + 4 + t; }
  __host__ __device__ static constexpr int bar_oready(int t) { return TB + 6 + t; }
  __host__ __device__ static constexpr int bar_drain(int t) { return TB + 8 + t; }
  __host__ __device__ static constexpr int bar_token(int t) { return TB + 10 + t; }
  __host__ __device__ static constexpr int bar_ofree(int t) { return TB + 12 + t; }
  __host__ __device__ static constexpr uint32_t col_p(int t) { return COL_P + (SEP_P ? 64u : 128u) * t; }
};
static_assert(Cfg<128>::SMEM <= 227 * 1024, "shared memory budget");
static_assert(Cfg<64>::SMEM <= 227 * 1024, "shared memory budget");
static_assert(Cfg<64>::COL_P + 128 <= 512, "tensor memory budget");
static_assert(Cfg<64>::NQ * Cfg<64>::BM == kItemRows && Cfg<128>::NQ * Cfg<128>::BM == kItemRows,
              "item rows");

struct Params {
  void* o;
  float* lse;
  long long o_sb, o_sg, o_sh, o_ss;  // O: batch, head group (grouped only), head, position
  int H, S, n_qblk, n_kv;
  int hs_swap;                         // layouts 0/1: tensor-map dims (d, H, S, B) instead of (d, S, H, B)
  int hg, G;                           // grouped layout: heads per group, groups per batch
  float c;  // scale · log2(e)
  unsigned* status;
  long long limit;
  // work list (see FlashPlan)
  int grid;
  long long dp_end;          // items [0, dp_end) whole, round-robin
  long long sk_units;        // key tiles of items [dp_end, ...), cut into runs
  long long cut[kMaxCutGrid + 1];      // CTA g: cut units [cut[g], cut[g+1])
  unsigned short g_last[kMaxCutGrid];  // see CtaWork
  // pieces of cut items: slot g belongs to CTA g (at most one piece per CTA)
  unsigned long long* flags;  // [grid][8]: tag once warp w's rows of slot g are written
  float2* ml;                 // [grid][256]: (m, l) of each row, m in log2 units
  float* opart;               // [grid][256][D]: O before division by l
  unsigned long long tag;     // unique per launch
};

// Kernel parameters (the three tensor maps and Params) must fit the 4 KB
// parameter space of a launch.
static_assert(3 * sizeof(CUtensorMap) + sizeof(Params) <= 4096, "kernel parameter space");

// One segment of a CTA's work list.
enum SegKind : int {
  SEG_WHOLE = 0,  // all key tiles of the item: normalise and store
  SEG_FIRST = 1,  // key tiles [0, je) of a cut item: merge the later pieces, then store
  SEG_PIECE = 2   // key tiles [jb, je), jb > 0, of a cut item: leave (m, l, O) in the scratch
};
struct Seg {
  long long item;
  int jb, je, kind;
};

// The work list of one CTA, set up once by thread 0 in shared memory: n_dp
// whole items (blockIdx.x + k·grid), then the key-tile run [u0, u1) of the
// cut items, which starts inside item it0 = u0 / n_kv.
struct CtaWork {
  long long u0, u1, it0;
  int n_dp;
  int g_last;  // the CTA holding the last piece of the item this CTA's run ends in
};

__device__ __forceinline__ void cta_work_init(const Params& p, CtaWork* cw) {
  const long long g = blockIdx.x;
  cw->n_dp = p.dp_end > g ? static_cast<int>((p.dp_end - g + p.grid - 1) / p.grid) : 0;
  if (p.sk_units > 0) {
    cw->u0 = p.cut[g];
    cw->u1 = p.cut[g + 1];
    // A run that ends inside an item (a SEG_FIRST segment, or a piece that is
    // not the item's last) leaves the rest to the CTAs up to g_last: the one
    // whose run holds the item's last key tile.
    cw->g_last = p.g_last[g];
  } else {
    cw->u0 = cw->u1 = 0;
    cw->g_last = static_cast<int>(g);
  }
  cw->it0 = cw->u0 / p.n_kv;
}

__device__ __forceinline__ long long lds_s64(uint32_t a) {
  long long v;
  asm volatile("ld.volatile.shared.s64 %0, [%1];" : "=l"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ int lds_s32(uint32_t a) {
  int v;
  asm volatile("ld.volatile.shared.s32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// Kernel modes: one whole item per CTA (the grid covers the items), a
// persistent grid dealing whole items round-robin, or a persistent grid that
// also cuts the last waves' items along the key axis.
enum Mode : int { MODE_ONE = 0, MODE_PERSIST = 1, MODE_SPLIT = 2 };

// Segment k of this CTA's list (false past its end).  Every role of the CTA
// walks the same list; the per-CTA constants (a CtaWork at shared address
// cw) are re-read at each segment so that they hold no registers during one.
// In MODE_ONE the list is the single item blockIdx.x with constant bounds,
// so the segment loops reduce to the plain loop over the item's key tiles.
template <int MODE>
__device__ __forceinline__ bool seg_at(const Params& p, uint32_t cw, int k, Seg& s) {
  if constexpr (MODE == MODE_ONE) {
    s.item = blockIdx.x, s.jb = 0, s.je = p.n_kv, s.kind = SEG_WHOLE;
    return k == 0;
  }
  const int n_dp = lds_s32(cw + offsetof(CtaWork, n_dp));
  if (k < n_dp) {
    s.item = static_cast<long long>(blockIdx.x) + static_cast<long long>(k) * p.grid;
    s.jb = 0, s.je = p.n_kv, s.kind = SEG_WHOLE;
    return true;
  }
  if constexpr (MODE != MODE_SPLIT) return false;
  const int kk = k - n_dp;
  const long long it = lds_s64(cw + offsetof(CtaWork, it0)) + kk;
  const long long us = kk == 0 ? lds_s64(cw + offsetof(CtaWork, u0)) : it * p.n_kv;
  const long long u1 = lds_s64(cw + offsetof(CtaWork, u1));
  if (us >= u1) return false;
  s.item = p.dp_end + it;
  s.jb = static_cast<int>(us - it * p.n_kv);
  s.je = (u1 - us < p.n_kv - s.jb) ? s.jb + static_cast<int>(u1 - us) : p.n_kv;
  s.kind = s.jb > 0 ? SEG_PIECE : (s.je < p.n_kv ? SEG_FIRST : SEG_WHOLE);
  return true;
}

struct ItemPos {
  int b, hh, q0;
};
// Item index -> (batch, head, first query row).  Item counts fit in 31 bits
// (checked on the host), so 32-bit arithmetic suffices.
__device__ __forceinline__ ItemPos item_pos(const Params& p, long long item) {
  const uint32_t it = static_cast<uint32_t>(item);
  const uint32_t bh = it / static_cast<uint32_t>(p.n_qblk);
  const uint32_t qblk = it - bh * static_cast<uint32_t>(p.n_qblk);
  const uint32_t b = bh / static_cast<uint32_t>(p.H);
  return {static_cast<int>(b), static_cast<int>(bh - b * static_cast<uint32_t>(p.H)),
          static_cast<int>(qblk) * kItemRows};
}

__device__ __forceinline__ uint32_t code_of(uint32_t role, uint32_t j) {
  return (KID_FLASH << 24) | (role << 16) | (j & 0xffffu);
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

// MODE (see Mode): only MODE_SPLIT carries the piece / merge code.
template <int D, bool BF16, bool GROUPED, int MODE>
__global__ void __launch_bounds__(352, 1)
    flash_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const __grid_constant__ Params p) {
  using C = Cfg<D>;
  constexpr bool SPLIT = MODE == MODE_SPLIT;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;  // 128-byte swizzle wants 1024-byte aligned tiles
  uint8_t* smem = smem_raw + (sb - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  CtaWork* work = reinterpret_cast<CtaWork*>(smem + C::OFF_WORK);
  const uint32_t cw = sb + C::OFF_WORK;
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };

  const uint32_t warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    for (int b = 0; b < C::NQB; ++b) {
      mbar_init(bar(C::bar_qfull(b)), 1);
      mbar_init(bar(C::bar_qempty(b)), C::ISSUERS);  // one commit per issuer
    }
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::bar_kfull(s)), 1);
      mbar_init(bar(C::bar_kempty(s)), C::ISSUERS);
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
      mbar_init(bar(C::bar_ofree(t)), 128);
    }
    if constexpr (MODE != MODE_ONE) cta_work_init(p, work);
    // Start pulling this CTA's first Q tiles and key/value tiles into L2 while
    // the previous grid finishes: a prefetch delivers nothing to the SM, and
    // L2 is where global memory is coherent, so it cannot see stale data.
    Seg s0;
    if (seg_at<MODE>(p, smem_u32(work), 0, s0)) {
      const ItemPos ip = item_pos(p, s0.item);
      auto pf = [&](const CUtensorMap* m, int e, int s) {
        if constexpr (GROUPED)
          tma_prefetch_4d(m, e, ip.hh % p.hg, s, ip.b * p.G + ip.hh / p.hg);
        else if (p.hs_swap)
          tma_prefetch_4d(m, e, ip.hh, s, ip.b);
        else
          tma_prefetch_4d(m, e, s, ip.hh, ip.b);
      };
      for (int c = 0; c < C::NCH; ++c) {
        for (int tt = 0; tt < C::NQ; ++tt) pf(&tq, c * 64, ip.q0 + tt * C::BM);
        for (int j = s0.jb; j < s0.je && j < s0.jb + C::STAGES; ++j) {
          pf(&tk, c * 64, j * C::BN);
          pf(&tv, c * 64, j * C::BN);
        }
      }
    }
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  // The set-up above overlaps the previous grid's tail; global memory is
  // touched only after it has completed.
  griddep_wait();
  if (threadIdx.x == 0) {
    // A CTA that starts after another one gave up does no work.
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
    // nothing
  } else if (warp >= 8) {
    if (warp == 8) {
    // ------------------------------------------------------ TMA producer ----
    // (feature, position) of item (b, hh) -> tensor-map coordinates.
    // Layouts 0/1: maps (d, S, H, B) or (d, H, S, B); grouped: (d, head
    // within group, S, group and batch).
    auto tma4 = [&](uint32_t dst, const CUtensorMap* m, uint32_t mbar, int e, int s, const ItemPos& ip) {
      if constexpr (GROUPED)
        tma_load_4d(dst, m, mbar, e, ip.hh % p.hg, s, ip.b * p.G + ip.hh / p.hg);
      else if (p.hs_swap)
        tma_load_4d(dst, m, mbar, e, ip.hh, s, ip.b);
      else
        tma_load_4d(dst, m, mbar, e, s, ip.hh, ip.b);
    };
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
    }
    Seg sg;
    uint32_t it = 0, issued_k = 0, issued_v = 0;  // key tiles, counted over all segments
    int kq = 0;                                   // segments (Q loads) issued
    bool ok = true;
    while (ok && seg_at<MODE>(p, cw, kq, sg)) {
      const ItemPos ip = item_pos(p, sg.item);
      const int qs = kq % C::NQB;
      if (kq >= C::NQB)
        ok = mbar_wait_warp(bar(C::bar_qempty(qs)), ((kq / C::NQB) - 1) & 1, wc, code_of(ROLE_LOAD, it));
      if (!ok) break;
      if (lane == 0) {
        mbar_expect_tx(bar(C::bar_qfull(qs)), C::QSET);
        for (int t = 0; t < C::NQ; ++t)
          for (int c = 0; c < C::NCH; ++c)
            tma4(sb + C::OFF_Q + qs * C::QSET + t * C::TILE + c * C::CHUNK, &tq, bar(C::bar_qfull(qs)),
                 c * 64, ip.q0 + t * C::BM, ip);
      }
      ++kq;
      for (int j = sg.jb; j < sg.je; ++j, ++it) {
        const uint32_t s = it % C::STAGES, u = it / C::STAGES;
        if (u > 0) ok = mbar_wait_warp(bar(C::bar_kempty(s)), (u - 1) & 1, wc, code_of(ROLE_LOAD, it));
        if (!ok) break;
        if (lane == 0) {
          mbar_expect_tx(bar(C::bar_kfull(s)), C::TILE);
          for (int c = 0; c < C::NCH; ++c)
            tma4(sb + C::OFF_K + s * C::TILE + c * C::CHUNK, &tk, bar(C::bar_kfull(s)), c * 64,
                 j * C::BN, ip);
        }
        issued_k = it + 1;
        if (u > 0) ok = mbar_wait_warp(bar(C::bar_vempty(s)), (u - 1) & 1, wc, code_of(ROLE_LOAD, it));
        if (!ok) break;
        if (lane == 0) {
          mbar_expect_tx(bar(C::bar_vfull(s)), C::TILE);
          for (int c = 0; c < C::NCH; ++c)
            tma4(sb + C::OFF_V + s * C::TILE + c * C::CHUNK, &tv, bar(C::bar_vfull(s)), c * 64,
                 j * C::BN, ip);
        }
        issued_v = it + 1;
      }
    }
    if (!ok) {
      // Let the copies already in flight land before the CTA can exit.
      for (uint32_t x = issued_k > C::STAGES ? issued_k - C::STAGES : 0; x < issued_k; ++x)
        mbar_wait_slow(bar(C::bar_kfull(x % C::STAGES)), (x / C::STAGES) & 1, wc, 0, false);
      for (uint32_t x = issued_v > C::STAGES ? issued_v - C::STAGES : 0; x < issued_v; ++x)
        mbar_wait_slow(bar(C::bar_vfull(x % C::STAGES)), (x / C::STAGES) & 1, wc, 0, false);
      for (int x = kq > C::NQB ? kq - C::NQB : 0; x < kq; ++x)
        mbar_wait_slow(bar(C::bar_qfull(x % C::NQB)), (x / C::NQB) & 1, wc, 0, false);
    }
    } else if (warp == 9 || (C::ISSUERS == 2 && warp == 10)) {
    // ------------------------------------------------ tcgen05 issuer(s) ----
    // The whole warp runs this code; elect.sync inside the issue helpers
    // picks the lane that issues each MMA and commit.
    constexpr uint32_t id_qk = idesc_f16(128, C::BN, BF16, false, false);
    constexpr uint32_t id_pv = idesc_f16(128, D, BF16, false, true);
    const uint64_t dk = sdesc_sw128(sb + C::OFF_K, 16, 1024);
    const uint64_t dv = sdesc_sw128(sb + C::OFF_V, C::CHUNK, 1024);
    auto qk = [&](int t, int qs, uint32_t s) {  // S_t = Q_t · K_s^T (K-major A and B; address += bytes/16)
      const uint64_t dq = sdesc_sw128(sb + C::OFF_Q + qs * C::QSET + t * C::TILE, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
        mma_ss_elect(tmem + C::COL_S + t * 128, dq + off, dk + ((s * C::TILE) >> 4) + off, id_qk,
                     kk > 0 ? 1u : 0u);
      }
    };
    auto pv = [&](int t, uint32_t s, bool acc) {  // O_t (+)= P_t · V_s   (P in TMEM, V MN-major)
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk)
        mma_ts_elect(tmem + C::COL_O + t * D, tmem + C::col_p(t) + kk * 8,
                     dv + ((s * C::TILE + kk * 2048) >> 4), id_pv, (acc || kk > 0) ? 1u : 0u);
    };
    auto commit = [&](int i) { mma_commit_elect(bar(i)); };
    auto wait = [&](int i, uint32_t parity, uint32_t j) {
      return mbar_wait_warp(bar(i), parity, wc, code_of(ROLE_MMA, j));
    };
    bool ok = true;
    if constexpr (C::ISSUERS == 2) {
      // One pipeline per Q tile t: S_t of the next key tile (of this
      // segment or the next one) as soon as the softmax has read S_t.
      const int t = static_cast<int>(warp) - 9;
      Seg ga, gp;  // Q·K^T runs one key tile ahead of P·V
      int ka = 0;
      bool has_a = seg_at<MODE>(p, cw, ka, ga);
      int ja = ga.jb;
      uint32_t nq = 0, np = 0;
      auto issue_qk = [&]() -> bool {
        const int qs = ka % C::NQB;
        if (ja == ga.jb && !wait(C::bar_qfull(qs), (ka / C::NQB) & 1, nq)) return false;
        const uint32_t s = nq % C::STAGES;
        if (!wait(C::bar_kfull(s), (nq / C::STAGES) & 1, nq)) return false;
        tc_fence_after();
        qk(t, qs, s);
        commit(C::bar_sfull(t));
        commit(C::bar_kempty(s));
        if (ja + 1 == ga.je) commit(C::bar_qempty(qs));  // last use of this Q buffer
        ++nq;
        if (++ja == ga.je) {
          has_a = seg_at<MODE>(p, cw, ++ka, ga);
          ja = ga.jb;
        }
        return true;
      };
      if (has_a) ok = issue_qk();
      for (int kp = 0; ok && seg_at<MODE>(p, cw, kp, gp); ++kp) {
        for (int j = gp.jb; j < gp.je; ++j, ++np) {
          if (has_a && !(ok = wait(C::bar_sconsumed(t), np & 1, np) && issue_qk())) break;
          const uint32_t s = np % C::STAGES;
          if (!(ok = wait(C::bar_vfull(s), (np / C::STAGES) & 1, np) && wait(C::bar_pready(t), np & 1, np)))
            break;
          if (j == gp.jb && kp > 0 && !(ok = wait(C::bar_ofree(t), (kp - 1) & 1, np))) break;
          tc_fence_after();
          pv(t, s, j > gp.jb);
          commit(C::bar_oready(t));
          commit(C::bar_vempty(s));
        }
      }
      if (!ok) {
        // Wait for the MMAs already issued before tensor memory is released.
        commit(C::bar_drain(t));
        mbar_wait_slow(bar(C::bar_drain(t)), 0, wc, 0, false);
      }
    } else {
      // One issuer, tiles in alternation; P overwrites S, so the next S_t is
      // issued after the P·V that reads P_t.  s_full(t) completes once per
      // key tile; the segment's final O_t is signalled on o_ready(t), so that
      // the next segment's first S_t never lands on the same barrier before
      // the softmax warps have seen the final O_t.
      Seg gp;
      uint32_t np = 0;
      for (int kp = 0; ok && seg_at<MODE>(p, cw, kp, gp); ++kp) {
        const int qs = kp % C::NQB;
        const uint32_t s0 = np % C::STAGES;
        if (!(ok = wait(C::bar_qfull(qs), (kp / C::NQB) & 1, np) &&
                   wait(C::bar_kfull(s0), (np / C::STAGES) & 1, np)))
          break;
        tc_fence_after();
        qk(0, qs, s0);
        commit(C::bar_sfull(0));
        qk(1, qs, s0);
        commit(C::bar_sfull(1));
        commit(C::bar_kempty(s0));
        if (gp.je - gp.jb == 1) commit(C::bar_qempty(qs));
        for (int j = gp.jb; j < gp.je; ++j, ++np) {
          const uint32_t s = np % C::STAGES;
          const bool more = j + 1 < gp.je;
          const uint32_t s1 = (np + 1) % C::STAGES, u1 = (np + 1) / C::STAGES;
          if (!(ok = wait(C::bar_vfull(s), (np / C::STAGES) & 1, np) && wait(C::bar_pready(0), np & 1, np)))
            break;
          if (j == gp.jb && kp > 0 && !(ok = wait(C::bar_ofree(0), (kp - 1) & 1, np))) break;
          tc_fence_after();
          pv(0, s, j > gp.jb);
          if (more) {
            if (!(ok = wait(C::bar_kfull(s1), u1 & 1, np))) break;
            tc_fence_after();
            qk(0, qs, s1);
            commit(C::bar_sfull(0));  // S_0 of the next tile ready
          } else {
            commit(C::bar_oready(0));  // the final O_0
          }
          if (!(ok = wait(C::bar_pready(1), np & 1, np))) break;
          if (j == gp.jb && kp > 0 && !(ok = wait(C::bar_ofree(1), (kp - 1) & 1, np))) break;
          tc_fence_after();
          pv(1, s, j > gp.jb);
          commit(C::bar_vempty(s));
          if (more) {
            qk(1, qs, s1);
            commit(C::bar_sfull(1));
            commit(C::bar_kempty(s1));
            if (j + 2 == gp.je) commit(C::bar_qempty(qs));
          } else {
            commit(C::bar_oready(1));
          }
        }
      }
      if (!ok) {
        commit(C::bar_drain(0));
        mbar_wait_slow(bar(C::bar_drain(0)), 0, wc, 0, false);
      }
    }
    }
  } else {
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
    auto wait = [&](int i, uint32_t parity, uint32_t j) {
      return mbar_wait_warp(bar(i), parity, wc, code_of(ROLE_SOFTMAX, j));
    };
    uint32_t r[4][32];  // this thread's row of S_t
    // Ragged key tail: the columns from `valid` on do not exist.  They are set
    // to -inf and the chunk maxima that the loads returned are taken again.
    auto ragged_tail_max = [&](int valid, float (&mq)[4]) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (q * 32 + i >= valid) r[q][i] = f2u(-INFINITY);
          mx = fmaxf(mx, u2f(r[q][i]));
        }
        mq[q] = mx;
      }
    };
    // p = 2^(s·c - m_ref) for the 128 keys, packed to 16-bit and stored to P_t
    // chunk by chunk; returns the sum of p.
    auto exps_store = [&]() -> float {
      const uint64_t nm2 = pk64(-m_ref, -m_ref);
      uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float s0 = u2f(r[q][2 * i]), s1 = u2f(r[q][2 * i + 1]);
          float y0, y1;
          up64(ffma2(pk64(s0, s1), c2, nm2), y0, y1);
          const float e0 = ex2(y0), e1 = ex2(y1);
          acc[i & 3] = fadd2(acc[i & 3], pk64(e0, e1));
          pk[i] = pack2<BF16>(e0, e1);
        }
        tmem_st16(tP + q * 16, pk);  // P columns [16q, 16q+16) hold keys [32q, 32q+32)
      }
      float a0, a1, a2, a3, a4, a5, a6, a7;
      up64(acc[0], a0, a1);
      up64(acc[1], a2, a3);
      up64(acc[2], a4, a5);
      up64(acc[3], a6, a7);
      return ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
    };

    // Output of one segment: its own O_t (tensor memory), m_ref and l, merged
    // with the later pieces of a cut item; normalised, rounded and stored.
    // A later piece instead leaves its unnormalised state in the scratch.
    // Statistics of a segment's output: its own (m_ref, l), merged for a
    // SEG_FIRST segment with those of the later pieces (waited for here).
    struct Merge {
      int g_last;      // pieces are held by CTAs blockIdx.x+1 .. g_last
      float m_new, a_own, L;
    };
    auto merge_stats = [&](const Seg& sg, Merge& mg) -> bool {
      const int rr = static_cast<int>(warp * 32 + lane);
      mg.g_last = static_cast<int>(blockIdx.x);
      mg.m_new = m_ref, mg.a_own = 1.f, mg.L = l;
      if (!SPLIT || sg.kind != SEG_FIRST) return true;
      mg.g_last = lds_s32(cw + offsetof(CtaWork, g_last));
      for (int g = static_cast<int>(blockIdx.x) + 1; g <= mg.g_last; ++g)
        if (!flag_wait_warp(p.flags + static_cast<long long>(g) * 8 + warp, p.tag, wc,
                            code_of(ROLE_EPILOGUE, static_cast<uint32_t>(g))))
          return false;
      for (int g = static_cast<int>(blockIdx.x) + 1; g <= mg.g_last; ++g) {
        // Pull the piece's row into L1 while the last P·V runs: the merge's
        // loads below then hit L1 instead of waiting on L2 twice.  (The tag's
        // acquire above orders them after the piece's stores.)
        const float* src = p.opart + (static_cast<long long>(g) * kItemRows + rr) * D;
#pragma unroll
        for (int c = 0; c < D; c += 32) asm volatile("prefetch.global.L1 [%0];" ::"l"(src + c));
      }
      for (int g = static_cast<int>(blockIdx.x) + 1; g <= mg.g_last; ++g)
        mg.m_new = fmaxf(mg.m_new, __ldcg(p.ml + static_cast<long long>(g) * kItemRows + rr).x);
      mg.a_own = ex2(m_ref - mg.m_new);
      mg.L = mg.a_own * l;
      for (int g = static_cast<int>(blockIdx.x) + 1; g <= mg.g_last; ++g) {
        const float2 q = __ldcg(p.ml + static_cast<long long>(g) * kItemRows + rr);
        mg.L += ex2(q.x - mg.m_new) * q.y;
      }
      return true;
    };

    // O_t may be overwritten by the next segment's first P·V once this
    // thread's last tensor-memory read of it has completed.
    auto release_o = [&]() {
      tc_fence_before();
      mbar_arrive(bar(C::bar_ofree(t)));
    };
    // A piece's ready-flag: its stores, then a release of this warp's tag.
    // Issued after the next segment's first key tile (or at the end), when
    // the stores have long drained, so that the fence costs nothing.
    bool piece_pending = false;
    auto publish_piece = [&]() {
      __threadfence();
      __syncwarp();
      if (lane == 0) st_release_u64(p.flags + static_cast<long long>(blockIdx.x) * 8 + warp, p.tag);
      piece_pending = false;
    };

    auto epilogue = [&](const Seg& sg, const Merge& mg) -> bool {
      const ItemPos ip = item_pos(p, sg.item);
      const int rr = static_cast<int>(warp * 32 + lane);  // this thread's row within the item
      if (SPLIT && sg.kind == SEG_PIECE) {
        const long long slot = static_cast<long long>(blockIdx.x) * kItemRows + rr;
        float4* dst = reinterpret_cast<float4*>(p.opart + slot * D);
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          tmem_ld_wait(o);
          if (cc == D / 32 - 1) release_o();
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            __stcg(dst + cc * 8 + v4,
                   make_float4(u2f(o[4 * v4]), u2f(o[4 * v4 + 1]), u2f(o[4 * v4 + 2]), u2f(o[4 * v4 + 3])));
        }
        __stcg(p.ml + slot, make_float2(m_ref, l));
        piece_pending = true;
        return true;
      }
      // SEG_WHOLE, or SEG_FIRST merging the pieces held by CTAs blockIdx.x+1 .. mg.g_last
      const float inv = 1.f / mg.L;
      const int row = ip.q0 + rr;
      const bool in = row < p.S;
      using Elem = uint16_t;
      const long long head_off = GROUPED ? (ip.hh / p.hg) * p.o_sg + (ip.hh % p.hg) * p.o_sh
                                         : static_cast<long long>(ip.hh) * p.o_sh;
      Elem* out = static_cast<Elem*>(p.o) + ip.b * p.o_sb + head_off +
                  static_cast<long long>(in ? row : 0) * p.o_ss;
      if (SPLIT && sg.kind == SEG_FIRST) {
        // 32 columns per pass: own O from tensor memory, then every piece's
        // 32 values (from L1, see merge_stats) with all 8 loads in flight.
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          tmem_ld_wait(o);
          if (cc == D / 32 - 1) release_o();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * mg.a_own);
#pragma unroll 1
          for (int g = static_cast<int>(blockIdx.x) + 1; g <= mg.g_last; ++g) {
            const long long slot = static_cast<long long>(g) * kItemRows + rr;
            const float4* src = reinterpret_cast<const float4*>(p.opart + slot * D) + cc * 8;
            float4 x[8];
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4) x[v4] = __ldca(src + v4);  // prefetched into L1
            const float wg = ex2(__ldcg(p.ml + slot).x - mg.m_new);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4) {
              o[4 * v4] = f2u(fmaf(wg, x[v4].x, u2f(o[4 * v4])));
              o[4 * v4 + 1] = f2u(fmaf(wg, x[v4].y, u2f(o[4 * v4 + 1])));
              o[4 * v4 + 2] = f2u(fmaf(wg, x[v4].z, u2f(o[4 * v4 + 2])));
              o[4 * v4 + 3] = f2u(fmaf(wg, x[v4].w, u2f(o[4 * v4 + 3])));
            }
          }
          if (in) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(u2f(o[2 * i]) * inv, u2f(o[2 * i + 1]) * inv);
            uint4* dst = reinterpret_cast<uint4*>(out + cc * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
      } else {
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          tmem_ld_wait(o);
          if (cc == D / 32 - 1) release_o();
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
      }
      if (in && p.lse)
        p.lse[(static_cast<long long>(ip.b) * p.H + ip.hh) * p.S + row] = (mg.m_new + log2f(mg.L)) * kLn2;
      return true;
    };

    Seg sg;
    uint32_t n0 = 0;  // key tiles of the earlier segments
    for (int kseg = 0; ok && seg_at<MODE>(p, cw, kseg, sg); ++kseg) {
      // Key tile j of this segment is tile n = n0 + (j - jb) of the CTA (its
      // barrier phase).  With one item per CTA, jb = n0 = 0 and je = n_kv are
      // constants and the loop is the plain loop over the item's key tiles.
      const int jb = sg.jb, je = sg.je;
      m_ref = -INFINITY;
      l = 0.f;
      if constexpr (C::SEP_P) {
      // d = 64: S_t is released to the next Q·K^T as soon as it is in
      // registers; the row max of the tile fixes the reference before any
      // exponential is taken, P is packed in place of S and stored at the end.
      // The two tiles' softmax warpgroups take turns on the exponential pass
      // (a token passed through an mbarrier), so that one runs it alone on the
      // special-function units while the other loads S, reduces and stores P.
      for (int j = jb; j < je; ++j) {
        const uint32_t n = n0 + static_cast<uint32_t>(j - jb);
        if (!(ok = wait(C::bar_sfull(t), n & 1, n))) break;
        tc_fence_after();
        float mq[4];  // the loads' own row maxima, one per 32-column chunk
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32_max(tS + q * 32, r[q], mq[q]);
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld_wait(r[q], mq[q]);
        tc_fence_before();
        mbar_arrive(bar(C::bar_sconsumed(t)));  // S_t may now be overwritten
        const int valid = p.S - j * C::BN;
        if (valid < C::BN) ragged_tail_max(valid, mq);
        const float m_blk = max3(mq[0], mq[1], fmaxf(mq[2], mq[3])) * c;
        const bool move = m_blk > m_ref + kRescaleThreshold;  // always on a segment's first tile
        const bool any_move = __any_sync(0xffffffffu, move);
        float alpha = 1.f;
        if (any_move) {  // warp-uniform; rare after the first tile
          const float m_new = move ? m_blk : m_ref;
          alpha = ex2(m_ref - m_new);
          l *= alpha;
          m_ref = m_new;
        }
        if (kExpToken && (t == 1 || n > 0)) {
          // tile 1 follows tile 0 of the same key tile, tile 0 follows tile 1 of the previous one
          if (!(ok = wait(C::bar_token(t), (t == 1 ? n : n - 1) & 1, n))) break;
        }
        {
          const uint64_t nm2 = pk64(-m_ref, -m_ref);
          uint64_t acc[2] = {0, 0};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float y0, y1;
              up64(ffma2(pk64(u2f(r[q][2 * i]), u2f(r[q][2 * i + 1])), c2, nm2), y0, y1);
              const float e0 = ex2(y0), e1 = ex2(y1);
              acc[i & 1] = fadd2(acc[i & 1], pk64(e0, e1));
              r[q][i] = pack2<BF16>(e0, e1);  // r[q][i] is no longer needed as S
            }
          }
          if (kExpToken) mbar_arrive(bar(C::bar_token(1 - t)));
          float a0, a1, a2, a3;
          up64(acc[0], a0, a1);
          up64(acc[1], a2, a3);
          l += (a0 + a1) + (a2 + a3);
        }
        if (j > jb) {  // P_t and O_t are free once the previous P·V has completed
          if (!(ok = wait(C::bar_oready(t), (n - 1) & 1, n))) break;
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
        if (SPLIT && piece_pending) publish_piece();
      }
      } else {
      for (int j = jb; j < je; ++j) {
        const uint32_t n = n0 + static_cast<uint32_t>(j - jb);
        if (!(ok = wait(C::bar_sfull(t), n & 1, n))) break;
        tc_fence_after();
        float mq[4];  // the loads' own row maxima, one per 32-column chunk
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32_max(tS + q * 32, r[q], mq[q]);
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld_wait(r[q], mq[q]);
        const int valid = p.S - j * C::BN;
        if (valid < C::BN) ragged_tail_max(valid, mq);
        const float m_blk = max3(mq[0], mq[1], fmaxf(mq[2], mq[3])) * c;
        if (j == jb) {  // empty history: the reference is this tile's max
          m_ref = m_blk;
        } else {
          // The tile max is known before any exponential: move the reference
          // (rare) and rescale O first.  O_t already holds the previous
          // P·V, which the issuer committed before this S_t.
          const bool move = m_blk > m_ref + kRescaleThreshold;
          if (__any_sync(0xffffffffu, move)) {  // warp-uniform
            const float m_new = move ? m_blk : m_ref;
            const float alpha = ex2(m_ref - m_new);
            l *= alpha;
            m_ref = m_new;
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
        l += exps_store();
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::bar_pready(t)));
        if (SPLIT && piece_pending) publish_piece();
      }
      }
      if (!ok) break;
      const uint32_t n = n0 + static_cast<uint32_t>(je - jb);  // tiles done, this segment's included
      n0 = n;
      // The merge statistics need only (m, l): gather them while the last P·V runs.
      seg_at<MODE>(p, cw, kseg, sg);  // re-read: nothing of it stays live through the segment
      Merge mg;
      if (!(ok = merge_stats(sg, mg))) break;
      if constexpr (C::SEP_P)
        ok = wait(C::bar_oready(t), (n - 1) & 1, n);  // the segment's last P·V (once per key tile)
      else
        ok = wait(C::bar_oready(t), kseg & 1, n);  // the segment's final O_t (once per segment)
      if (!ok) break;
      tc_fence_after();
      if (!(ok = epilogue(sg, mg))) break;
    }
    if (SPLIT && ok && piece_pending) publish_piece();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool BF16, bool GROUPED, int MODE>
cudaError_t launch_impl(const FlashLaunch& a, const FlashPlan& plan, cudaStream_t st) {
  using C = Cfg<D>;
  auto kern = flash_fwd_kernel<D, BF16, GROUPED, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  Params p{};
  p.o = a.o;
  p.lse = a.lse;
  p.o_sb = a.o_sb;
  p.o_sg = a.o_sg;
  p.o_sh = a.o_sh;
  p.o_ss = a.o_ss;
  p.H = a.H;
  p.S = a.S;
  p.n_qblk = plan.n_qblk;
  p.n_kv = plan.n_kv;
  p.hs_swap = a.hs_swap;
  p.hg = a.hg;
  p.G = a.H / a.hg;
  p.c = a.scale * kLog2e;
  p.status = a.status;
  p.limit = a.limit;
  p.grid = plan.grid;
  p.dp_end = plan.dp_end;
  p.sk_units = plan.sk_units;
  if (plan.sk_units > 0) {
    memcpy(p.cut, plan.cut, sizeof(long long) * (plan.grid + 1));
    memcpy(p.g_last, plan.g_last, sizeof(unsigned short) * plan.grid);
  }
  p.flags = nullptr;
  p.ml = nullptr;
  p.opart = nullptr;
  p.tag = a.tag;
  if (plan.sk_units > 0) {
    uint8_t* ws = static_cast<uint8_t*>(a.scratch);
    const FlashScratch fs = flash_scratch_layout(D, plan.grid);
    p.flags = reinterpret_cast<unsigned long long*>(ws + fs.off_flags);
    p.ml = reinterpret_cast<float2*>(ws + fs.off_ml);
    p.opart = reinterpret_cast<float*>(ws + fs.off_opart);
    if (a.clear_flags) {
      e = cudaMemsetAsync(p.flags, 0, fs.flag_bytes, st);
      if (e != cudaSuccess) return e;
    }
  }
  // Launched as a programmatic dependent of the previous work in the stream:
  // the kernel waits (griddepcontrol.wait) before its first global access.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.grid));
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a.tq, a.tk, a.tv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, bool G, int MODE>
cudaError_t launch_m(const FlashLaunch& a, const FlashPlan& plan, cudaStream_t st) {
  return a.bf16 ? launch_impl<D, true, G, MODE>(a, plan, st) : launch_impl<D, false, G, MODE>(a, plan, st);
}

}  // namespace

FlashScratch flash_scratch_layout(int d, int grid) {
  auto r256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  FlashScratch s;
  s.flag_bytes = static_cast<size_t>(grid) * 8 * sizeof(unsigned long long);
  s.off_flags = 0;
  s.off_ml = r256(s.flag_bytes);
  s.off_opart = s.off_ml + r256(static_cast<size_t>(grid) * kItemRows * sizeof(float2));
  s.total = s.off_opart + static_cast<size_t>(grid) * kItemRows * d * sizeof(float);
  return s;
}

// Whether cutting the last waves is expected to pay at d = 64.  Each extra
// segment costs about 1.5 key-tile steps (Q load, pipeline restart, epilogue)
// and a cut item's piece and merge about 3.5 more, so the cut must save at
// least 8 steps per CTA, and items shorter than 16 key tiles never gain
// (measured: B8 h12 S512 ran 14 % slower cut).  ATTN_SPLIT=force cuts
// whenever the item count leaves a partial wave (used by the tests to cover
// the cut path at small sizes); ATTN_SPLIT=never does not cut.
static bool cut_pays(long long items, int n_kv, long long sms) {
  const char* env = getenv("ATTN_SPLIT");
  if (env && strcmp(env, "force") == 0) return true;
  if (env && strcmp(env, "never") == 0) return false;
  if (n_kv < 16) return false;
  const long long grid = items * n_kv < sms ? items * n_kv : sms;
  const long long steps_cut = (items * n_kv + grid - 1) / grid;
  const long long steps_whole = (items + sms - 1) / sms * n_kv;
  return steps_cut + 8 < steps_whole;
}

namespace {

// Equal runs of the cut units, CTA g taking [g·U/grid, (g+1)·U/grid), and
// for each CTA the CTA whose run holds the last key tile of the item its own
// run ends in (the merge of a cut item waits for the CTAs up to that one).
// Runs balanced by a per-segment cost estimate were tried: no gain on the
// bench workload, and slower where an item is longer than a run, because a
// key-0 part then waits for a long piece that ends with its own run.
void equal_runs(FlashPlan& pl) {
  const long long units = pl.sk_units;
  for (int g = 0; g <= pl.grid; ++g) pl.cut[g] = g * units / pl.grid;
  int h = 0;
  for (int g = 0; g < pl.grid; ++g) {
    pl.g_last[g] = static_cast<unsigned short>(g);
    if (pl.cut[g + 1] <= pl.cut[g]) continue;
    const long long last_unit = ((pl.cut[g + 1] - 1) / pl.n_kv + 1) * pl.n_kv - 1;
    if (h < g) h = g;
    while (pl.cut[h + 1] <= last_unit) ++h;
    pl.g_last[g] = static_cast<unsigned short>(h);
  }
}

}  // namespace

FlashPlan plan_flash(int B, int H, int S, int d, int num_sms, bool split) {
  FlashPlan pl{};
  pl.n_qblk = (S + kItemRows - 1) / kItemRows;
  pl.n_kv = (S + 127) / 128;
  const long long items = static_cast<long long>(B) * H * pl.n_qblk;
  const long long sms = num_sms > 0 ? num_sms : 1;
  pl.dp_end = items;
  pl.sk_units = 0;
  if (d != 64) {
    // d = 128: one item per CTA (measured faster per key tile than the
    // persistent loop nest, and the last wave gains little from cutting)
    pl.mode = MODE_ONE;
    pl.grid = static_cast<int>(items);
  } else if (!split || items % sms == 0 || !cut_pays(items, pl.n_kv, sms)) {
    // whole items, round-robin over at most one CTA per SM
    pl.mode = MODE_PERSIST;
    pl.grid = static_cast<int>(items < sms ? items : sms);
  } else {
    // whole items for all but the last one to two waves; those are cut into
    // equal runs of key tiles over every CTA
    pl.mode = MODE_SPLIT;
    const long long units_all = items * pl.n_kv;
    long long grid = units_all < sms ? units_all : sms;
    if (grid > kMaxCutGrid) grid = kMaxCutGrid;
    pl.grid = static_cast<int>(grid);
    const long long waves = items / pl.grid;
    pl.dp_end = (waves > 0 ? waves - 1 : 0) * pl.grid;
    pl.sk_units = (items - pl.dp_end) * pl.n_kv;
    equal_runs(pl);
  }
  return pl;
}

cudaError_t launch_flash_fwd(const FlashLaunch& a, const FlashPlan& plan, cudaStream_t st) {
  if (a.d != 64 && a.d != 128) return cudaErrorInvalidValue;
  // The head-group layout has no scratch entry point: never cut.
  if (a.grouped && plan.mode == MODE_SPLIT) return cudaErrorInvalidValue;
  switch (plan.mode) {
    case MODE_ONE:  // planned for d = 128 only
      if (a.d != 128) return cudaErrorInvalidValue;
      return a.grouped ? launch_m<128, true, MODE_ONE>(a, plan, st) : launch_m<128, false, MODE_ONE>(a, plan, st);
    case MODE_PERSIST:
      // Whole items run on the cut-capable instance (with no cut units it
      // deals items round-robin like MODE_PERSIST): its register allocation
      // measured 0.7-1.5 % faster per key tile.  The head-group layout keeps
      // the MODE_PERSIST instance.
      if (a.d != 64) return cudaErrorInvalidValue;
      return a.grouped ? launch_m<64, true, MODE_PERSIST>(a, plan, st) : launch_m<64, false, MODE_SPLIT>(a, plan, st);
    case MODE_SPLIT:
      if (a.d != 64) return cudaErrorInvalidValue;
      return launch_m<64, false, MODE_SPLIT>(a, plan, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
