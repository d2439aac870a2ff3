// Host-side interfaces between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// Tensor maps of the attention kernel.  Layouts 0/1: dims (d, S, H, B)
// (contiguous [B,H,S,d], hs_swap = 0) or (d, H, S, B) (head-interleaved
// [B,S,H,d], hs_swap = 1), so that byte strides grow with the dimension.
// Grouped layout [B,H/hg,S,hg,d]: dims (d, hg, S, (H/hg)·B) -- feature, head
// within the group, position, then group and batch merged.

struct FlashLaunch {
  CUtensorMap tq, tk, tv;       // 4-d maps, box = 64 features x 128 positions
  void* o;                      // output, element strides below (feature stride 1)
  float* lse;                   // [B,H,S] fp32 or null
  long long o_sb, o_sg, o_sh, o_ss;  // batch, head group (grouped only), head, position
  int B, H, S, d;
  bool grouped;
  int hs_swap;                  // layouts 0/1
  int hg;                       // grouped: heads per group (divides H)
  bool bf16;
  float scale;                  // softmax scale (already resolved)
  unsigned* status;             // device status word
  long long limit;              // clock cycles per wait before giving up
  void* scratch;                // pieces of cut items (plan.sk_units > 0), flash_scratch_layout bytes
  unsigned long long tag;       // unique per launch: marks this launch's pieces as written
  bool clear_flags;             // zero the piece flags first (needed when the launch can be replayed)
};

// CTAs a cut plan may use: their run bounds travel in the kernel parameters.
constexpr int kMaxCutGrid = 256;

// Work list of the persistent attention kernel.  An item is one (batch, head)
// and 256 query rows; items [0, dp_end) run whole, item i on CTA i % grid;
// the sk_units key tiles of the remaining items are cut into equal
// contiguous runs, CTA g taking units [cut[g], cut[g+1]).
struct FlashPlan {
  int mode;                     // 0: one item per CTA; 1: persistent, whole items; 2: persistent + cut
  int grid;
  int n_qblk, n_kv;             // items per (batch, head); key tiles per item
  long long dp_end;
  long long sk_units;           // 0: no item is cut, no scratch is used
  long long cut[kMaxCutGrid + 1];          // run bounds (mode 2)
  unsigned short g_last[kMaxCutGrid];      // CTA holding the last key tile of the item CTA g's run ends in
};
// split = false: whole items only.  split = true: cut the last one to two
// waves (only when the item count is not a multiple of num_sms).  The mode
// also depends on the head dimension d.
FlashPlan plan_flash(int B, int H, int S, int d, int num_sms, bool split);

// Scratch of a plan with cut items: per CTA 8 flags, then (m, l) and the
// unnormalised O of 256 rows.
struct FlashScratch {
  size_t off_flags, flag_bytes, off_ml, off_opart, total;
};
FlashScratch flash_scratch_layout(int d, int grid);

cudaError_t launch_flash_fwd(const FlashLaunch& a, const FlashPlan& plan, cudaStream_t st);

// Resident-tile attention for d = 64, S <= 512 (fused.cu): one CTA per
// (batch, head) holds the head's Q, K, V tiles in shared memory.
// project = true: the single-kernel QKV projection + attention; t0: X
//   [B, S, D] as a 3-d map (D, S, B), box 64 x 128 x 1; t1: W_qkv [D, 3D] as a
//   2-d map (3D, D), box 64 x 64.
// project = false: attention on existing Q, K, V; t0, t1, t2: the 4-d maps of
//   make_map (box 64 x 128 rows), hs_swap as there.
// to: the output O as a 4-d map of the same form (o_swap like hs_swap).
// All 128-byte swizzled.  lse [B, H, S] or null.
struct FusedLaunch {
  CUtensorMap t0, t1, t2, to;
  bool project;
  float* lse;
  int o_swap;
  int B, S, H, D;
  int hs_swap;
  bool bf16;
  float scale;
  unsigned* status;
  long long limit;
};
cudaError_t launch_fused_qkv_attn(const FusedLaunch& a, cudaStream_t st);

struct SimtLaunch {
  const float *q, *k, *v;
  float* o;
  float* lse;
  long long sb, sh, ss;         // element strides shared by q, k, v, o
  int B, H, S, d;
  float scale;
};
cudaError_t launch_simt_fwd(const SimtLaunch& a, cudaStream_t st);

// Batched tensor-core GEMM   C[z] = alpha · A[z] · op(B[z])
//   A: [M, K] K-major (4-d map: K, M, Z1, Z2; box 64 x 128)
//   B: b_kmajor ? [N, K] (map: K, N, Z1, Z2; box 64 x BN)
//              : [K, N] (map: N, K, Z1, Z2; box 64 x 64)
//   z in [0, Z1·Z2): operand coordinates (z % Z1, z / Z1)
//   C element (z, m, n) at c + (z / Z1)·c_s2 + (z % Z1)·c_s1 + m·ldc + n
struct GemmLaunch {
  CUtensorMap ta, tb;
  void* c;
  int c_type;                   // 0 = fp32, 1 = fp16, 2 = bf16
  long long ldc, c_s1, c_s2;
  int M, N, K, Z1, Z2;
  int bn;                       // 64, 128 or 256: output columns per tile
  int mb = 1;                   // 2: 256-row tiles (bn = 256, MN-major B only), 1: 128-row tiles
  bool b_kmajor;
  int a_swap, b_swap;           // 1: map dims are (inner, Z1, rows, Z2) instead of (inner, rows, Z1, Z2)
  bool bf16;                    // operand type
  float alpha;
  unsigned* status;
  long long limit;
};
cudaError_t launch_gemm(const GemmLaunch& a, cudaStream_t st);

// fp32 -> 16-bit copies of Q, K, V (attn_fwd_mixed): out[i·out_stride + j] =
// round_to_nearest(src_i[j]) for the three tensors, n elements each (n % 8 == 0,
// all pointers 16-byte aligned).
struct ConvertLaunch {
  const float *q, *k, *v;
  uint16_t* out;
  long long n, out_stride;      // elements per tensor; element offset between the outputs
  bool bf16;
  int num_sms;
};
cudaError_t launch_convert3(const ConvertLaunch& a, cudaStream_t st);

// Naive softmax passes over an fp32 score matrix [rows, n] (row stride ld):
//   pass 1: stats[r] = (max_j S[r,j], sum_j exp(S[r,j] - max))
//   pass 2: P[r,j] = exp(S[r,j] - m_r) / l_r  (16-bit), and lse[...] if asked
struct NaiveSoftmaxLaunch {
  const float* s;               // row stride ld (fp32 elements)
  void* p;                      // dtype of the attention
  float* m;                     // [rows]
  float* l;                     // [rows]
  float* lse;                   // [B,H,S] or null (rows are ordered (b, h, i))
  long long rows;
  int n;
  long long ld;                 // row stride of s and p, in elements
  bool bf16;
};
cudaError_t launch_naive_softmax(const NaiveSoftmaxLaunch& a, cudaStream_t st);

// max |a - b| over n elements of two device buffers (dtype as attn.h);
// synchronises the stream and writes the result to *host_max.  Each call
// accumulates into its own one of 64 statically declared device words, taken
// in turn, so calls in flight at the same time do not share a result.
// Argument checks of the fused QKV projection + attention entry points
// (pointers, dtype, shape, 16-byte alignment, output overlapping an input);
// ATTN_OK or a negative ATTN_E_* code.  Makes no CUDA call.
int validate_qkv_proj(const void* x, const void* w_qkv, const void* o, int B, int S, int D, int h, int dtype);

cudaError_t launch_max_abs_diff(const void* a, const void* b, long long n, int dtype,
                                float* host_max, cudaStream_t st);

}  // namespace attn
