// Attention oracle: plain, slow, fp64 CPU implementation of the multi-head
// attention forward.  TEST INFRASTRUCTURE ONLY -- it is used by the tests,
// by the smoke check and by the benchmark's CPU-baseline leg, never by the
// product path, and it shares no code with the CUDA library.
//
// Sources (page title, section):
//   [T2]  "Transformer算子生态深度分析", chapter 2 "自注意力机制算子"
//         §2.1 QKV投影 (fused [D,3D] projection, split into heads)
//         §2.2 注意力分数计算 (S = Q·K^T / sqrt(D_k))
//         §2.3 Softmax (three-step stable softmax: max, sum of exp, divide)
//         §2.4 加权求和 (O = A·V)
//         §2.6 FlashAttention (online merge of per-block max and exp-sum)
//   [W1]  "WebGPU 算子优化：QKV 内存合并与 FlashAttention 分块计算"
//         §QKV 矩阵的内存合并模式选择 (contiguous / head-interleaved layouts)
//         §FlashAttention 分块计算原理与浏览器适配 (m_new / l_new merge rule)
//   [P2]  "[WebGPU] Proposal: Add an option to use online softmax instead of
//         naive softmax", §四 (per-element running max / running sum)
//
// What it computes is the plain definition: for every query row it
// materialises the whole score row in fp64, applies the three-step softmax
// and multiplies by V.  The online (blocked) recurrence is present only so
// that the tests can check it against the three-step softmax.
//
// Input elements are read from the exact bytes given to the GPU (fp32, fp16,
// bf16 or fp64) and widened to double by the decoders below, which follow
// the IEEE-754 binary16 and the bfloat16 bit layouts.
//
// Parity pins for every function live in tests/test_oracle.py.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

enum ElemType { ET_F64 = 0, ET_F32 = 1, ET_F16 = 2, ET_BF16 = 3 };

// IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double decode_f16(uint16_t bits) {
  const int sign = (bits >> 15) & 1;
  const int expo = (bits >> 10) & 0x1f;
  const int frac = bits & 0x3ff;
  double mag;
  if (expo == 0) {
    mag = std::ldexp(static_cast<double>(frac), -24);           // subnormal: frac * 2^-14 * 2^-10
  } else if (expo == 31) {
    mag = frac ? std::numeric_limits<double>::quiet_NaN()
               : std::numeric_limits<double>::infinity();
  } else {
    mag = std::ldexp(1.0 + frac / 1024.0, expo - 15);
  }
  return sign ? -mag : mag;
}

// bfloat16 is the upper half of an IEEE-754 binary32.
double decode_bf16(uint16_t bits) {
  const uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

double load_elem(const void* base, int et, int64_t idx) {
  switch (et) {
    case ET_F64: return static_cast<const double*>(base)[idx];
    case ET_F32: return static_cast<double>(static_cast<const float*>(base)[idx]);
    case ET_F16: return decode_f16(static_cast<const uint16_t*>(base)[idx]);
    case ET_BF16: return decode_bf16(static_cast<const uint16_t*>(base)[idx]);
  }
  return std::numeric_limits<double>::quiet_NaN();
}

// A 4-d tensor (batch, head, position, feature) with the feature index
// contiguous and element strides for the other three.
struct View {
  const void* p;
  int et;
  int64_t sb, sh, ss;
  double at(int64_t b, int64_t h, int64_t s, int64_t e) const {
    return load_elem(p, et, b * sb + h * sh + s * ss + e);
  }
};

// Strides of the two layouts of [W1] §QKV 矩阵的内存合并模式选择:
//   layout 0, contiguous:        [B, H, S, d]
//   layout 1, head-interleaved:  [B, S, H, d]   (row stride rs >= H*d)
void layout_strides(int layout, int64_t H, int64_t S, int64_t d, int64_t rs,
                    int64_t* sb, int64_t* sh, int64_t* ss) {
  if (layout == 0) {
    *ss = d;
    *sh = S * d;
    *sb = H * S * d;
  } else {
    *sh = d;
    *ss = rs;
    *sb = S * rs;
  }
}

// The third layout of the same section ("split", head groups): the heads
// form groups of hg; each group's data is stored contiguously, positions
// first, the group's heads interleaved within a position:
//   [B, H/hg, S, hg, d].
// Element (b, h, s, e) sits at
//   b*H*S*d + (h / hg)*S*hg*d + s*hg*d + (h % hg)*d + e.
int64_t grouped_index(int64_t H, int64_t S, int64_t d, int64_t hg, int64_t b, int64_t h, int64_t s,
                      int64_t e) {
  return b * H * S * d + (h / hg) * S * hg * d + s * hg * d + (h % hg) * d + e;
}

// [T2] §2.3: the three-step numerically stable softmax of one row.
//   step 1  m = max_i s_i
//   step 2  d = sum_i exp(s_i - m)
//   step 3  a_i = exp(s_i - m) / d
void softmax_three_step(const double* s, int64_t n, double* a, double* m_out, double* d_out) {
  double m = -std::numeric_limits<double>::infinity();
  for (int64_t i = 0; i < n; ++i) m = std::max(m, s[i]);
  double d = 0.0;
  for (int64_t i = 0; i < n; ++i) d += std::exp(s[i] - m);
  for (int64_t i = 0; i < n; ++i) a[i] = std::exp(s[i] - m) / d;
  if (m_out) *m_out = m;
  if (d_out) *d_out = d;
}

// One query row of attention, by the definition of [T2] §2.2-§2.4.
// Writes o_row[0..d) and the natural-log log-sum-exp of the scaled scores.
void attention_row(const View& Q, const View& K, const View& V, int64_t b, int64_t h,
                   int64_t i, int64_t Skv, int64_t d, double scale, double* score,
                   double* prob, double* o_row, double* lse) {
  // [T2] §2.2: scores of query i against every key, scaled by `scale`.
  for (int64_t j = 0; j < Skv; ++j) {
    double dot = 0.0;
    for (int64_t e = 0; e < d; ++e) dot += Q.at(b, h, i, e) * K.at(b, h, j, e);
    score[j] = dot * scale;
  }
  // [T2] §2.3: softmax along the key axis.
  double m = 0.0, l = 0.0;
  softmax_three_step(score, Skv, prob, &m, &l);
  // [T2] §2.4: O = A·V for this row.
  for (int64_t e = 0; e < d; ++e) o_row[e] = 0.0;
  for (int64_t j = 0; j < Skv; ++j) {
    const double a = prob[j];
    for (int64_t e = 0; e < d; ++e) o_row[e] += a * V.at(b, h, j, e);
  }
  if (lse) *lse = m + std::log(l);
}

int resolve_threads(int nthreads) {
  if (nthreads > 0) return nthreads;
  const unsigned hc = std::thread::hardware_concurrency();
  return hc ? static_cast<int>(hc) : 1;
}

// Runs fn(r) for r in [0, n) on `nthreads` threads, in contiguous chunks so
// that every row is computed by exactly one thread in a fixed order.
template <class Fn>
void parallel_rows(int64_t n, int nthreads, Fn fn) {
  const int T = static_cast<int>(std::min<int64_t>(resolve_threads(nthreads), std::max<int64_t>(n, 1)));
  if (T <= 1) {
    for (int64_t r = 0; r < n; ++r) fn(r);
    return;
  }
  std::vector<std::thread> pool;
  pool.reserve(T);
  const int64_t chunk = (n + T - 1) / T;
  for (int t = 0; t < T; ++t) {
    const int64_t lo = t * chunk, hi = std::min<int64_t>(n, lo + chunk);
    if (lo >= hi) break;
    pool.emplace_back([=]() {
      for (int64_t r = lo; r < hi; ++r) fn(r);
    });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Number of worker threads a call with `nthreads` will use.
int oracle_threads(int nthreads) { return resolve_threads(nthreads); }

// Widens n elements of type `et` to double (exposed so the tests can pin the
// decoders against independent conversions).
int oracle_decode(const void* src, int et, int64_t n, double* dst) {
  if (!src || !dst || n < 0 || et < 0 || et > 3) return -1;
  for (int64_t i = 0; i < n; ++i) dst[i] = load_elem(src, et, i);
  return 0;
}

// [T2] §2.3 three-step softmax of a single vector.
int oracle_softmax(const double* s, int64_t n, double* p, double* m_out, double* d_out) {
  if (!s || !p || n < 1) return -1;
  softmax_three_step(s, n, p, m_out, d_out);
  return 0;
}

// Online softmax of a single vector processed in blocks of `block` elements.
// For each block: its own max m_blk and exp-sum d_blk = sum exp(s - m_blk)
// ([T2] §2.6); then the running statistics are merged by
//   m = max(m_old, m_blk)
//   d = d_old * exp(m_old - m) + d_blk * exp(m_blk - m)
// ([T2] §2.6 core formula; [W1] §FlashAttention, m_new / l_new).  With
// block == 1 this is the per-element recurrence of [P2] §四.  The running
// (m, d) after each block is written to m_trace / d_trace (may be null).
// The probabilities are produced at the end from the final (m, d).
int oracle_online_softmax(const double* s, int64_t n, int64_t block, double* p,
                          double* m_trace, double* d_trace, double* m_out, double* d_out) {
  if (!s || !p || n < 1 || block < 1) return -1;
  double m = -std::numeric_limits<double>::infinity();
  double d = 0.0;
  int64_t t = 0;
  for (int64_t lo = 0; lo < n; lo += block, ++t) {
    const int64_t hi = std::min(n, lo + block);
    double m_blk = -std::numeric_limits<double>::infinity();
    for (int64_t i = lo; i < hi; ++i) m_blk = std::max(m_blk, s[i]);
    double d_blk = 0.0;
    for (int64_t i = lo; i < hi; ++i) d_blk += std::exp(s[i] - m_blk);
    const double m_new = std::max(m, m_blk);
    // exp(m_old - m_new) with m_old = -inf is 0: an empty history contributes nothing.
    const double f_old = (m == -std::numeric_limits<double>::infinity()) ? 0.0 : std::exp(m - m_new);
    d = d * f_old + d_blk * std::exp(m_blk - m_new);
    m = m_new;
    if (m_trace) m_trace[t] = m;
    if (d_trace) d_trace[t] = d;
  }
  for (int64_t i = 0; i < n; ++i) p[i] = std::exp(s[i] - m) / d;
  if (m_out) *m_out = m;
  if (d_out) *d_out = d;
  return 0;
}

// Full attention forward O = softmax(scale · Q·K^T) · V for every (b, h, i).
// q, k, v, o share `layout` (0 = [B,H,S,d], 1 = [B,S,H,d] with row stride H*d);
// q, k, v are of element type `et`, o and lse are fp64; lse is [B,H,S] and
// may be null.  Returns 0, or -1 on a bad argument.
int oracle_attention(const void* q, const void* k, const void* v, int et, int64_t B,
                     int64_t H, int64_t S, int64_t d, int layout, double scale, double* o,
                     double* lse, int nthreads) {
  if (!q || !k || !v || !o || B < 1 || H < 1 || S < 1 || d < 1 || (layout != 0 && layout != 1) ||
      et < 0 || et > 3)
    return -1;
  int64_t sb, sh, ss;
  layout_strides(layout, H, S, d, H * d, &sb, &sh, &ss);
  const View Q{q, et, sb, sh, ss}, K{k, et, sb, sh, ss}, V{v, et, sb, sh, ss};
  parallel_rows(B * H * S, nthreads, [&](int64_t r) {
    thread_local std::vector<double> score, prob;
    score.resize(S);
    prob.resize(S);
    const int64_t b = r / (H * S), h = (r / S) % H, i = r % S;
    attention_row(Q, K, V, b, h, i, S, d, scale, score.data(), prob.data(),
                  o + b * sb + h * sh + i * ss, lse ? lse + r : nullptr);
  });
  return 0;
}

// The same computation for a chosen set of query rows only.  rows[t] is the
// flat index (b*H + h)*S + i; o_rows is [nrows, d], lse_rows is [nrows]
// (may be null).  Used for sampled checks at sizes where the full oracle
// would take too long.
int oracle_attention_rows(const void* q, const void* k, const void* v, int et, int64_t B,
                          int64_t H, int64_t S, int64_t d, int layout, double scale,
                          const int64_t* rows, int64_t nrows, double* o_rows, double* lse_rows,
                          int nthreads) {
  if (!q || !k || !v || !rows || !o_rows || B < 1 || H < 1 || S < 1 || d < 1 ||
      (layout != 0 && layout != 1) || et < 0 || et > 3 || nrows < 0)
    return -1;
  for (int64_t t = 0; t < nrows; ++t)
    if (rows[t] < 0 || rows[t] >= B * H * S) return -1;
  int64_t sb, sh, ss;
  layout_strides(layout, H, S, d, H * d, &sb, &sh, &ss);
  const View Q{q, et, sb, sh, ss}, K{k, et, sb, sh, ss}, V{v, et, sb, sh, ss};
  parallel_rows(nrows, nthreads, [&](int64_t t) {
    thread_local std::vector<double> score, prob;
    score.resize(S);
    prob.resize(S);
    const int64_t r = rows[t];
    const int64_t b = r / (H * S), h = (r / S) % H, i = r % S;
    attention_row(Q, K, V, b, h, i, S, d, scale, score.data(), prob.data(), o_rows + t * d,
                  lse_rows ? lse_rows + t : nullptr);
  });
  return 0;
}

// [T2] §2.1 fused projection: one product with the concatenated weight
// W_qkv [D, 3D] (columns ordered Q | K | V), giving qkv [B, S, 3D] in fp64.
// x is [B, S, D], both of element type `et`.
int oracle_qkv_projection(const void* x, const void* w, int et, int64_t B, int64_t S, int64_t D,
                          double* qkv, int nthreads) {
  if (!x || !w || !qkv || B < 1 || S < 1 || D < 1 || et < 0 || et > 3) return -1;
  const int64_t N = 3 * D;
  std::vector<double> wd(static_cast<size_t>(D * N));  // W widened to double once
  for (int64_t i = 0; i < D * N; ++i) wd[i] = load_elem(w, et, i);
  parallel_rows(B * S, nthreads, [&](int64_t r) {
    double* out = qkv + r * N;
    for (int64_t c = 0; c < N; ++c) out[c] = 0.0;
    for (int64_t kk = 0; kk < D; ++kk) {
      const double xv = load_elem(x, et, r * D + kk);
      const double* wrow = wd.data() + kk * N;
      for (int64_t c = 0; c < N; ++c) out[c] += xv * wrow[c];
    }
  });
  return 0;
}

// [T2] §2.1 split into heads: column c of the [B, S, 3D] projection belongs
// to tensor c / D (0 = Q, 1 = K, 2 = V), head (c % D) / d, feature c % d.
// Each of q, k, v receives [B, S, H, d] (head-interleaved, layout 1).
int oracle_split_heads(const double* qkv, int64_t B, int64_t S, int64_t D, int64_t H, double* q,
                       double* k, double* v) {
  if (!qkv || !q || !k || !v || B < 1 || S < 1 || H < 1 || D < H || D % H) return -1;
  const int64_t d = D / H;
  double* dst[3] = {q, k, v};
  for (int64_t r = 0; r < B * S; ++r)
    for (int64_t c = 0; c < 3 * D; ++c) {
      const int64_t which = c / D, head = (c % D) / d, e = c % d;
      dst[which][(r * H + head) * d + e] = qkv[r * 3 * D + c];
    }
  return 0;
}

// Fused projection followed by attention ([T2] §2.1 then §2.2-§2.4):
// x [B,S,D], w [D,3D] of type `et`; o is [B,S,H,d] fp64 (head-interleaved);
// lse [B,H,S] may be null.  The projection is kept in fp64 (not rounded).
int oracle_qkv_proj_attention(const void* x, const void* w, int et, int64_t B, int64_t S,
                              int64_t D, int64_t H, double scale, double* o, double* lse,
                              int nthreads) {
  if (!x || !w || !o || B < 1 || S < 1 || H < 1 || D < H || D % H) return -1;
  std::vector<double> qkv(static_cast<size_t>(B * S * 3 * D));
  if (oracle_qkv_projection(x, w, et, B, S, D, qkv.data(), nthreads)) return -1;
  const int64_t d = D / H;
  std::vector<double> q(B * S * D), k(B * S * D), v(B * S * D);
  oracle_split_heads(qkv.data(), B, S, D, H, q.data(), k.data(), v.data());
  return oracle_attention(q.data(), k.data(), v.data(), ET_F64, B, H, S, d, 1, scale, o, lse,
                          nthreads);
}

// Attention over the grouped layout: q, k, v, o are [B, H/hg, S, hg, d]
// (see grouped_index), lse is [B, H, S].  Same arithmetic as
// oracle_attention; only the addressing differs.
int oracle_attention_grouped(const void* q, const void* k, const void* v, int et, int64_t B,
                             int64_t H, int64_t S, int64_t d, int64_t hg, double scale, double* o,
                             double* lse, int nthreads) {
  if (!q || !k || !v || !o || B < 1 || H < 1 || S < 1 || d < 1 || hg < 1 || H % hg || et < 0 ||
      et > 3)
    return -1;
  parallel_rows(B * H * S, nthreads, [&](int64_t r) {
    thread_local std::vector<double> score, prob;
    score.resize(S);
    prob.resize(S);
    const int64_t b = r / (H * S), h = (r / S) % H, i = r % S;
    for (int64_t j = 0; j < S; ++j) {
      double dot = 0.0;
      for (int64_t e = 0; e < d; ++e)
        dot += load_elem(q, et, grouped_index(H, S, d, hg, b, h, i, e)) *
               load_elem(k, et, grouped_index(H, S, d, hg, b, h, j, e));
      score[j] = dot * scale;
    }
    double m = 0.0, l = 0.0;
    softmax_three_step(score.data(), S, prob.data(), &m, &l);
    for (int64_t e = 0; e < d; ++e) {
      double acc = 0.0;
      for (int64_t j = 0; j < S; ++j) acc += prob[j] * load_elem(v, et, grouped_index(H, S, d, hg, b, h, j, e));
      o[grouped_index(H, S, d, hg, b, h, i, e)] = acc;
    }
    if (lse) lse[r] = m + std::log(l);
  });
  return 0;
}

}  // extern "C"
