// C ABI of libattn_gb300.so (declared in include/attn.h): argument
// validation, TMA tensor-map encoding, kernel selection and launch.
//
// Every argument is checked before the first CUDA call, so an invalid call
// returns a negative ATTN_E_* code without touching the device.

#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#include <atomic>
#include <chrono>
#include <mutex>

#include "attn.h"
#include "common.h"
#include "ptx.cuh"

namespace {

// One status word per device; kernels record a pipeline timeout here.
__device__ unsigned g_status;

constexpr int kMaxDevices = 64;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  bool ready = false;
  int rc = ATTN_OK;
  unsigned* status = nullptr;
  int num_sms = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

int elt_bytes(int dtype) { return dtype == ATTN_F32 ? 4 : 2; }

// Resolves the per-device state of the current device: sm_103 check, address
// of the status word and the driver's tensor-map encoder.
int device_setup(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_E_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    st.ready = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        major != 10 || minor != 3 ||
        cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        st.num_sms < 1) {
      st.rc = ATTN_E_DEVICE;
    } else if (cudaGetSymbolAddress(reinterpret_cast<void**>(&st.status), g_status) != cudaSuccess) {
      st.rc = ATTN_E_DEVICE;
    } else if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        st.rc = ATTN_E_DEVICE;
      else
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  *out = &st;
  return st.rc;
}

// Clock cycles a pipeline wait may take before the kernel gives up
// (default 4e9, about two seconds at GB300 clocks; ATTN_WAIT_LIMIT_CYCLES overrides).
long long wait_limit() {
  static long long v = [] {
    const char* s = getenv("ATTN_WAIT_LIMIT_CYCLES");
    long long x = s ? atoll(s) : 0;
    return x > 0 ? x : 4000000000LL;
  }();
  return v;
}

// A tag no earlier launch of this process used (and, seeded from the clock
// and the process id, unlikely to be one another process left in memory).
// The pieces of cut items are marked as written with it.
unsigned long long next_tag() {
  static std::atomic<unsigned long long> ctr{
      static_cast<unsigned long long>(std::chrono::steady_clock::now().time_since_epoch().count()) ^
      (static_cast<unsigned long long>(getpid()) << 40)};
  unsigned long long z = ctr.fetch_add(0x9e3779b97f4a7c15ULL) + 0x9e3779b97f4a7c15ULL;  // splitmix64
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return (z ^ (z >> 31)) | 1ULL;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// 4-d tensor map over a [B, H, S, d] problem in either layout.  `rs` is the
// row stride in elements (distance between consecutive positions s of one
// head in layout 1; ignored in layout 0).  Box: 64 features x box_rows rows.
int make_map(CUtensorMap* m, const void* base, int dtype, int layout, long long B, long long H,
             long long S, long long d, long long rs, int box_rows, int* hs_swap) {
  const cuuint64_t e = static_cast<cuuint64_t>(elt_bytes(dtype));
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
  if (layout == ATTN_LAYOUT_BHSD) {  // dims (d, S, H, B)
    dims[0] = d, dims[1] = S, dims[2] = H, dims[3] = B;
    strides[0] = d * e, strides[1] = S * d * e, strides[2] = H * S * d * e;
    box[0] = 64, box[1] = box_rows, box[2] = 1, box[3] = 1;
    *hs_swap = 0;
  } else {  // dims (d, H, S, B)
    dims[0] = d, dims[1] = H, dims[2] = S, dims[3] = B;
    strides[0] = d * e, strides[1] = rs * e, strides[2] = S * rs * e;
    box[0] = 64, box[1] = 1, box[2] = box_rows, box[3] = 1;
    *hs_swap = 1;
  }
  const CUtensorMapDataType dt =
      dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = g_encode(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_E_DEVICE;
}

// Plain row-major matrices [Z2][Z1][rows][cols] with row stride ld (elements)
// as a 4-d map (cols, rows, Z1, Z2); box 64 x box_rows.
int make_matrix_map(CUtensorMap* m, const void* base, int dtype, long long Z1, long long Z2,
                    long long rows, long long cols, long long ld, int box_rows) {
  const cuuint64_t e = static_cast<cuuint64_t>(elt_bytes(dtype));
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(Z1), static_cast<cuuint64_t>(Z2)};
  cuuint64_t strides[3] = {ld * e, rows * ld * e, Z1 * rows * ld * e};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1}, estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt =
      dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = g_encode(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_E_DEVICE;
}

// Tensor map of the attention kernel over one of Q, K, V: dims
// (d, hg, S, (H/hg)·B) with element strides sh (head within the group), ss
// (position) and sg (group; the batch stride must equal (H/hg)·sg).
int make_flash_map(CUtensorMap* m, const void* base, int dtype, long long B, long long H, long long S,
                   long long d, long long hg, long long sh, long long ss, long long sg) {
  const cuuint64_t e = static_cast<cuuint64_t>(elt_bytes(dtype));
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hg),
                        static_cast<cuuint64_t>(S), static_cast<cuuint64_t>((H / hg) * B)};
  cuuint64_t strides[3] = {sh * e, ss * e, sg * e};
  cuuint32_t box[4] = {64, 1, 128, 1}, estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt =
      dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = g_encode(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_E_DEVICE;
}

int to_rc(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : static_cast<int>(e); }

// One warp waits on an mbarrier that nothing will ever arrive on, with the
// same bounded wait the pipeline kernels use; it must give up after `limit`
// cycles, record the code in the status word and return.
__global__ void selftest_wait_kernel(unsigned* status, long long limit) {
  __shared__ __align__(8) uint64_t mbar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    attn::mbar_init(attn::smem_u32(&mbar), 1);
    abort_flag = 0;
    attn::fence_mbar_init();
  }
  __syncthreads();
  const attn::WaitCtx wc{&abort_flag, status, limit};
  const uint32_t code = (attn::KID_SELFTEST << 24) | (attn::ROLE_LOAD << 16);
  attn::mbar_wait_warp(attn::smem_u32(&mbar), 0, wc, code);
}

// Checks shared by attn_fwd and attn_fwd_naive.  Makes no CUDA call.
int validate_attn(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  int B, int h, int S, int d, int layout, int dtype) {
  if (!q || !k || !v || !o) return ATTN_E_NULL;
  if (layout != ATTN_LAYOUT_BHSD && layout != ATTN_LAYOUT_BSHD) return ATTN_E_LAYOUT;
  if (dtype != ATTN_F32 && dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_E_DTYPE;
  if (B < 1 || h < 1 || S < 1 || d < 1) return ATTN_E_SHAPE;
  if (dtype == ATTN_F32 ? d > 256 : (d != 64 && d != 128)) return ATTN_E_SHAPE;
  const long long elems = static_cast<long long>(B) * h * S * d;
  if (elems > (1LL << 40)) return ATTN_E_SHAPE;
  const long long ctas = static_cast<long long>(B) * h * ((S + 255) / 256);
  if (ctas > 0x7fffffffLL || static_cast<long long>(B) * h * ((S + 7) / 8) > 0x7fffffffLL)
    return ATTN_E_SHAPE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      (lse && !aligned(lse, 4)))
    return ATTN_E_ALIGN;
  const size_t bytes = static_cast<size_t>(elems) * elt_bytes(dtype);
  if (overlap(o, bytes, q, bytes) || overlap(o, bytes, k, bytes) || overlap(o, bytes, v, bytes))
    return ATTN_E_ALIAS;
  if (lse) {
    const size_t lb = static_cast<size_t>(B) * h * S * sizeof(float);
    if (overlap(lse, lb, q, bytes) || overlap(lse, lb, k, bytes) || overlap(lse, lb, v, bytes) ||
        overlap(lse, lb, o, bytes))
      return ATTN_E_ALIAS;
  }
  return ATTN_OK;
}

void o_strides(int layout, long long H, long long S, long long d, long long rs, long long* sb,
               long long* sh, long long* ss) {
  if (layout == ATTN_LAYOUT_BHSD) {
    *ss = d, *sh = S * d, *sb = H * S * d;
  } else {
    *sh = d, *ss = rs, *sb = S * rs;
  }
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Whether a 16-bit problem runs on the resident-tile kernel (fused.cu,
// attention only): d = 64 and S <= 512, where each (batch, head) fits in
// shared memory and the streaming kernel's per-item start and drain dominate
// its few key tiles.  The resident kernel runs one CTA per (batch, head) and
// its pairs of 128-row blocks one after the other; the streaming kernel spreads
// the pairs (its items) over the SMs.  Resident is taken when its waves times
// pairs per head do not exceed the streaming kernel's waves of items
// (measured on GB300: B8 h12 S512 14.2 against 16.2 us, B8 h16 S512 14.3
// against 15.2, B4 h16 S256 5.9 against 6.7; the rule sends B16 h12 S512,
// 27.2 against 22.8, and B2 h16 S384, 11.2 against 7.7, to the streaming
// kernel).  ATTN_RESIDENT=never sends every problem to the streaming kernel
// and ATTN_RESIDENT=force every d = 64, S <= 512 one to the resident kernel
// (the tests cover both kernels on the same shapes).
bool resident_pays(int B, int h, int S, int d, int sms) {
  if (d != 64 || S > 512 || sms < 1) return false;
  const char* env = getenv("ATTN_RESIDENT");
  if (env && strcmp(env, "never") == 0) return false;
  if (env && strcmp(env, "force") == 0) return true;
  const long long heads = static_cast<long long>(B) * h;
  const long long pairs = ((S + 127) / 128 + 1) / 2;
  return (heads + sms - 1) / sms * pairs <= (heads * pairs + sms - 1) / sms;
}

// Flash launch on tensors of a [B,H,S,d] problem; inputs and output may have
// different row strides (rs_in, rs_out: layout 1 only).  Layout
// ATTN_LAYOUT_GROUPED takes hg heads per group ([B,H/hg,S,hg,d]).
// With `scratch` (at least flash_scratch_layout(d, grid).total bytes for the
// plan's grid) the last waves of items may be cut along the key axis.
int run_flash(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h, int S,
              int d, float scale, int layout, long long hg, int dtype, long long rs_in,
              long long rs_out, const DeviceState* ds, cudaStream_t st, void* scratch = nullptr,
              size_t scratch_bytes = 0) {
  if (layout != ATTN_LAYOUT_GROUPED && resident_pays(B, h, S, d, ds->num_sms)) {
    // d = 64, S <= 512: one CTA per (batch, head) with the head's Q, K, V
    // resident in shared memory (no per-item pipeline start and drain).
    attn::FusedLaunch r;
    int hs = 0;
    int rc2 = make_map(&r.t0, q, dtype, layout, B, h, S, d, rs_in, 128, &hs);
    if (!rc2) rc2 = make_map(&r.t1, k, dtype, layout, B, h, S, d, rs_in, 128, &hs);
    if (!rc2) rc2 = make_map(&r.t2, v, dtype, layout, B, h, S, d, rs_in, 128, &hs);
    if (!rc2) rc2 = make_map(&r.to, o, dtype, layout, B, h, S, d, rs_out, 128, &r.o_swap);
    if (rc2) return rc2;
    r.project = false;
    r.lse = lse;
    r.B = B, r.S = S, r.H = h, r.D = h * d;
    r.hs_swap = hs;
    r.bf16 = dtype == ATTN_BF16;
    r.scale = scale;
    r.status = ds->status;
    r.limit = wait_limit();
    (void)scratch;
    (void)scratch_bytes;
    return to_rc(attn::launch_fused_qkv_attn(r, st));
  }
  attn::FlashLaunch a;
  int rc = ATTN_OK;
  a.grouped = layout == ATTN_LAYOUT_GROUPED;
  a.hs_swap = 0;
  a.hg = 1;
  if (a.grouped) {
    const long long sh = d, ss = hg * d, sg = S * hg * d;
    rc = make_flash_map(&a.tq, q, dtype, B, h, S, d, hg, sh, ss, sg);
    if (!rc) rc = make_flash_map(&a.tk, k, dtype, B, h, S, d, hg, sh, ss, sg);
    if (!rc) rc = make_flash_map(&a.tv, v, dtype, B, h, S, d, hg, sh, ss, sg);
    a.o_sb = static_cast<long long>(h) * S * d, a.o_sg = sg, a.o_sh = sh, a.o_ss = ss;
    a.hg = static_cast<int>(hg);
  } else {
    rc = make_map(&a.tq, q, dtype, layout, B, h, S, d, rs_in, 128, &a.hs_swap);
    if (!rc) rc = make_map(&a.tk, k, dtype, layout, B, h, S, d, rs_in, 128, &a.hs_swap);
    if (!rc) rc = make_map(&a.tv, v, dtype, layout, B, h, S, d, rs_in, 128, &a.hs_swap);
    o_strides(layout, h, S, d, rs_out, &a.o_sb, &a.o_sh, &a.o_ss);
    a.o_sg = 0;
  }
  if (rc) return rc;
  a.o = o;
  a.lse = lse;
  a.B = B, a.H = h, a.S = S, a.d = d;
  a.bf16 = dtype == ATTN_BF16;
  a.scale = scale;
  a.status = ds->status;
  a.limit = wait_limit();
  a.scratch = nullptr;
  a.tag = 0;
  a.clear_flags = false;
  attn::FlashPlan plan = attn::plan_flash(B, h, S, d, ds->num_sms, scratch != nullptr);
  if (plan.sk_units > 0) {
    if (scratch_bytes < attn::flash_scratch_layout(d, plan.grid).total) return ATTN_E_WORKSPACE;
    a.scratch = scratch;
    a.tag = next_tag();
    // A captured launch replays with the same tag: its flags must start clear.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return to_rc(e);
    a.clear_flags = cs != cudaStreamCaptureStatusNone;
  }
  return to_rc(attn::launch_flash_fwd(a, plan, st));
}

}  // namespace

extern "C" {

int attn_abi_version(void) { return 1; }

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h, int S,
             int d, float scale, int layout, int dtype, void* stream) {
  int rc = validate_attn(q, k, v, o, lse, B, h, S, d, layout, dtype);
  if (rc) return rc;
  DeviceState* ds = nullptr;
  if ((rc = device_setup(&ds))) return rc;
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(d));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == ATTN_F32) {
    attn::SimtLaunch a;
    a.q = static_cast<const float*>(q);
    a.k = static_cast<const float*>(k);
    a.v = static_cast<const float*>(v);
    a.o = static_cast<float*>(o);
    a.lse = lse;
    o_strides(layout, h, S, d, static_cast<long long>(h) * d, &a.sb, &a.sh, &a.ss);
    a.B = B, a.H = h, a.S = S, a.d = d;
    a.scale = sc;
    return to_rc(attn::launch_simt_fwd(a, st));
  }
  const long long rs = static_cast<long long>(h) * d;
  return run_flash(q, k, v, o, lse, B, h, S, d, sc, layout, 1, dtype, rs, rs, ds, st);
}

int attn_flash_schedule(int B, int h, int S, int d, int num_sms, int split, int* mode, int* grid,
                        long long* dp_end, long long* sk_units, long long* cut, int* g_last) {
  if (B < 1 || h < 1 || S < 1 || num_sms < 1 || (d != 64 && d != 128)) return ATTN_E_SHAPE;
  const attn::FlashPlan plan = attn::plan_flash(B, h, S, d, num_sms, split != 0);
  if (mode) *mode = plan.mode;
  if (grid) *grid = plan.grid;
  if (dp_end) *dp_end = plan.dp_end;
  if (sk_units) *sk_units = plan.sk_units;
  if (plan.sk_units > 0) {
    for (int g = 0; cut && g <= plan.grid; ++g) cut[g] = plan.cut[g];
    for (int g = 0; g_last && g < plan.grid; ++g) g_last[g] = plan.g_last[g];
  }
  return 0;
}

size_t attn_fwd_ws_bytes(int B, int h, int S, int d, int dtype) {
  if (B < 1 || h < 1 || S < 1 || (dtype != ATTN_F16 && dtype != ATTN_BF16) || (d != 64 && d != 128))
    return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return 0;
  const attn::FlashPlan plan = attn::plan_flash(B, h, S, d, sms, true);
  return plan.sk_units > 0 ? attn::flash_scratch_layout(d, plan.grid).total : 0;
}

int attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                int S, int d, float scale, int layout, int dtype, void* workspace, size_t ws_bytes,
                void* stream) {
  int rc = validate_attn(q, k, v, o, lse, B, h, S, d, layout, dtype);
  if (rc) return rc;
  if (dtype == ATTN_F32 || (!workspace && ws_bytes == 0))
    return attn_fwd(q, k, v, o, lse, B, h, S, d, scale, layout, dtype, stream);
  if (!workspace || !aligned(workspace, 256)) return ATTN_E_WORKSPACE;
  const size_t bytes = static_cast<size_t>(B) * h * S * d * 2;
  if (overlap(workspace, ws_bytes, q, bytes) || overlap(workspace, ws_bytes, k, bytes) ||
      overlap(workspace, ws_bytes, v, bytes) || overlap(workspace, ws_bytes, o, bytes) ||
      (lse && overlap(workspace, ws_bytes, lse, static_cast<size_t>(B) * h * S * 4)))
    return ATTN_E_ALIAS;
  DeviceState* ds = nullptr;
  if ((rc = device_setup(&ds))) return rc;
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(d));
  const long long rs = static_cast<long long>(h) * d;
  return run_flash(q, k, v, o, lse, B, h, S, d, sc, layout, 1, dtype, rs, rs, ds,
                   static_cast<cudaStream_t>(stream), workspace, ws_bytes);
}

size_t attn_fwd_mixed_workspace_bytes(int B, int h, int S, int d, int out_dtype) {
  if (B < 1 || h < 1 || S < 1 || (out_dtype != ATTN_F16 && out_dtype != ATTN_BF16) || (d != 64 && d != 128))
    return 0;
  const long long n = static_cast<long long>(B) * h * S * d;
  if (n > (1LL << 40)) return 0;
  return 3 * round256(static_cast<size_t>(n) * 2) + attn_fwd_ws_bytes(B, h, S, d, out_dtype);
}

int attn_fwd_mixed(const float* q, const float* k, const float* v, void* o, float* lse, int B, int h,
                   int S, int d, float scale, int layout, int out_dtype, void* workspace, size_t ws_bytes,
                   void* stream) {
  if (!q || !k || !v || !o) return ATTN_E_NULL;
  if (layout != ATTN_LAYOUT_BHSD && layout != ATTN_LAYOUT_BSHD) return ATTN_E_LAYOUT;
  if (out_dtype != ATTN_F16 && out_dtype != ATTN_BF16) return ATTN_E_DTYPE;
  if (B < 1 || h < 1 || S < 1 || (d != 64 && d != 128)) return ATTN_E_SHAPE;
  const long long n = static_cast<long long>(B) * h * S * d;
  if (n > (1LL << 40) || static_cast<long long>(B) * h * ((S + 255) / 256) > 0x7fffffffLL) return ATTN_E_SHAPE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || (lse && !aligned(lse, 4)))
    return ATTN_E_ALIGN;
  const size_t in_b = static_cast<size_t>(n) * 4, out_b = static_cast<size_t>(n) * 2;
  const size_t lse_b = static_cast<size_t>(B) * h * S * 4;
  if (overlap(o, out_b, q, in_b) || overlap(o, out_b, k, in_b) || overlap(o, out_b, v, in_b) ||
      (lse && (overlap(lse, lse_b, q, in_b) || overlap(lse, lse_b, k, in_b) || overlap(lse, lse_b, v, in_b) ||
               overlap(lse, lse_b, o, out_b))))
    return ATTN_E_ALIAS;
  const size_t conv = 3 * round256(out_b);
  if (!workspace || !aligned(workspace, 256) || ws_bytes < conv) return ATTN_E_WORKSPACE;
  if (overlap(workspace, ws_bytes, q, in_b) || overlap(workspace, ws_bytes, k, in_b) ||
      overlap(workspace, ws_bytes, v, in_b) || overlap(workspace, ws_bytes, o, out_b) ||
      (lse && overlap(workspace, ws_bytes, lse, lse_b)))
    return ATTN_E_ALIAS;
  DeviceState* ds = nullptr;
  int rc = device_setup(&ds);
  if (rc) return rc;
  // Scratch beyond the three copies, if any, must hold the whole cut-wave
  // scratch: checked before the first launch.
  const size_t rest = ws_bytes - conv;
  if (rest > 0) {
    const attn::FlashPlan plan = attn::plan_flash(B, h, S, d, ds->num_sms, true);
    if (plan.sk_units > 0 && rest < attn::flash_scratch_layout(d, plan.grid).total) return ATTN_E_WORKSPACE;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  attn::ConvertLaunch cv;
  cv.q = q, cv.k = k, cv.v = v;
  cv.out = reinterpret_cast<uint16_t*>(ws);
  cv.n = n;
  cv.out_stride = static_cast<long long>(round256(out_b) / 2);
  cv.bf16 = out_dtype == ATTN_BF16;
  cv.num_sms = ds->num_sms;
  if ((rc = to_rc(attn::launch_convert3(cv, st)))) return rc;
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(d));
  const long long rs = static_cast<long long>(h) * d;
  return run_flash(ws, ws + round256(out_b), ws + 2 * round256(out_b), o, lse, B, h, S, d, sc, layout, 1,
                   out_dtype, rs, rs, ds, st, rest > 0 ? ws + conv : nullptr, rest);
}

int attn_fwd_grouped(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                     int S, int d, int heads_per_group, float scale, int dtype, void* stream) {
  int rc = validate_attn(q, k, v, o, lse, B, h, S, d, ATTN_LAYOUT_BHSD, dtype);
  if (rc) return rc;
  if (dtype == ATTN_F32) return ATTN_E_DTYPE;
  if (heads_per_group < 1 || h % heads_per_group) return ATTN_E_SHAPE;
  DeviceState* ds = nullptr;
  if ((rc = device_setup(&ds))) return rc;
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(d));
  const long long rs = static_cast<long long>(h) * d;
  return run_flash(q, k, v, o, lse, B, h, S, d, sc, ATTN_LAYOUT_GROUPED, heads_per_group, dtype, rs,
                   rs, ds, static_cast<cudaStream_t>(stream));
}

size_t attn_fwd_naive_workspace_bytes(int B, int h, int S, int dtype) {
  if (B < 1 || h < 1 || S < 1 || (dtype != ATTN_F16 && dtype != ATTN_BF16)) return 0;
  const size_t rows = static_cast<size_t>(B) * h * S;
  const size_t sp = (static_cast<size_t>(S) + 7) & ~static_cast<size_t>(7);
  return round256(rows * sp * 4) + round256(rows * sp * 2) + 2 * round256(rows * 4);
}

int attn_fwd_naive(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                   int S, int d, float scale, int layout, int dtype, void* workspace,
                   size_t ws_bytes, void* stream) {
  int rc = validate_attn(q, k, v, o, lse, B, h, S, d, layout, dtype);
  if (rc) return rc;
  if (dtype == ATTN_F32) return ATTN_E_DTYPE;
  const size_t need = attn_fwd_naive_workspace_bytes(B, h, S, dtype);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256)) return ATTN_E_WORKSPACE;
  const size_t bytes = static_cast<size_t>(B) * h * S * d * 2;
  if (overlap(workspace, need, q, bytes) || overlap(workspace, need, k, bytes) ||
      overlap(workspace, need, v, bytes) || overlap(workspace, need, o, bytes) ||
      (lse && overlap(workspace, need, lse, static_cast<size_t>(B) * h * S * 4)))
    return ATTN_E_ALIAS;
  DeviceState* ds = nullptr;
  if ((rc = device_setup(&ds))) return rc;
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(d));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long rows = static_cast<long long>(B) * h * S;
  const long long sp = (static_cast<long long>(S) + 7) & ~7LL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* s_mat = reinterpret_cast<float*>(ws);
  void* p_mat = ws + round256(rows * sp * 4);
  float* m_vec = reinterpret_cast<float*>(ws + round256(rows * sp * 4) + round256(rows * sp * 2));
  float* l_vec = m_vec + round256(rows * 4) / 4;
  const long long rs = static_cast<long long>(h) * d;

  // 1. S = scale · Q·K^T  (fp32, [B,H,S,sp])
  attn::GemmLaunch g1;
  int swap = 0;
  const int bn1 = S >= 256 ? 256 : 128;  // key block of the S tile (the K map's box height)
  rc = make_map(&g1.ta, q, dtype, layout, B, h, S, d, rs, 128, &swap);
  if (!rc) rc = make_map(&g1.tb, k, dtype, layout, B, h, S, d, rs, bn1, &swap);
  if (rc) return rc;
  g1.c = s_mat;
  g1.c_type = 0;
  g1.ldc = sp;
  g1.c_s1 = S * sp;
  g1.c_s2 = static_cast<long long>(h) * S * sp;
  g1.M = S, g1.N = S, g1.K = d, g1.Z1 = h, g1.Z2 = B;
  g1.bn = bn1;
  g1.b_kmajor = true;
  g1.a_swap = g1.b_swap = swap;
  g1.bf16 = dtype == ATTN_BF16;
  g1.alpha = sc;
  g1.status = ds->status;
  g1.limit = wait_limit();
  if ((rc = to_rc(attn::launch_gemm(g1, st)))) return rc;

  // 2.-3. row statistics, then P = exp(S - m) / l
  attn::NaiveSoftmaxLaunch sm;
  sm.s = s_mat;
  sm.p = p_mat;
  sm.m = m_vec;
  sm.l = l_vec;
  sm.lse = lse;
  sm.rows = rows;
  sm.n = S;
  sm.ld = sp;
  sm.bf16 = dtype == ATTN_BF16;
  if ((rc = to_rc(attn::launch_naive_softmax(sm, st)))) return rc;

  // 4. O = P·V
  attn::GemmLaunch g2;
  rc = make_matrix_map(&g2.ta, p_mat, dtype, h, B, S, S, sp, 128);
  if (!rc) rc = make_map(&g2.tb, v, dtype, layout, B, h, S, d, rs, 64, &swap);
  if (rc) return rc;
  g2.c = o;
  g2.c_type = dtype;
  o_strides(layout, h, S, d, rs, &g2.c_s2, &g2.c_s1, &g2.ldc);
  g2.M = S, g2.N = d, g2.K = S, g2.Z1 = h, g2.Z2 = B;
  g2.bn = d;
  g2.b_kmajor = false;
  g2.a_swap = 0;
  g2.b_swap = swap;
  g2.bf16 = dtype == ATTN_BF16;
  g2.alpha = 1.f;
  g2.status = ds->status;
  g2.limit = wait_limit();
  return to_rc(attn::launch_gemm(g2, st));
}

size_t qkv_proj_attn_workspace_bytes(int B, int S, int D, int dtype) {
  if (B < 1 || S < 1 || D < 1 || (dtype != ATTN_F16 && dtype != ATTN_BF16)) return 0;
  return round256(static_cast<size_t>(B) * S * 3 * D * 2);
}

}  // extern "C"

namespace attn {

int validate_qkv_proj(const void* x, const void* w_qkv, const void* o, int B, int S, int D, int h,
                      int dtype) {
  if (!x || !w_qkv || !o) return ATTN_E_NULL;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_E_DTYPE;
  if (B < 1 || S < 1 || h < 1 || D < 1 || D % h) return ATTN_E_SHAPE;
  const int d = D / h;
  if (d != 64 && d != 128) return ATTN_E_SHAPE;
  const long long rows = static_cast<long long>(B) * S;
  if (rows > 0x7fffffffLL || rows * 3 * D > (1LL << 40) ||
      static_cast<long long>(B) * h * ((S + 255) / 256) > 0x7fffffffLL ||
      ((rows + 127) / 128) * ((3LL * D + 127) / 128) > 0x7fffffffLL)
    return ATTN_E_SHAPE;
  if (!aligned(x, 16) || !aligned(w_qkv, 16) || !aligned(o, 16)) return ATTN_E_ALIGN;
  const size_t xb = static_cast<size_t>(rows) * D * 2, wb = static_cast<size_t>(D) * 3 * D * 2;
  if (overlap(o, xb, x, xb) || overlap(o, xb, w_qkv, wb)) return ATTN_E_ALIAS;
  return ATTN_OK;
}

}  // namespace attn

extern "C" {

int qkv_proj_attn(const void* x, const void* w_qkv, void* o, int B, int S, int D, int h, int dtype,
                  void* workspace, size_t ws_bytes, void* stream) {
  int rc = attn::validate_qkv_proj(x, w_qkv, o, B, S, D, h, dtype);
  if (rc) return rc;
  const int d = D / h;
  const long long rows = static_cast<long long>(B) * S;
  const size_t need = qkv_proj_attn_workspace_bytes(B, S, D, dtype);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256)) return ATTN_E_WORKSPACE;
  const size_t xb = static_cast<size_t>(rows) * D * 2, wb = static_cast<size_t>(D) * 3 * D * 2;
  if (overlap(o, xb, workspace, need) || overlap(workspace, need, x, xb) || overlap(workspace, need, w_qkv, wb))
    return ATTN_E_ALIAS;
  DeviceState* ds = nullptr;
  if ((rc = device_setup(&ds))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // 1. QKV = X · W_qkv  -> workspace [B·S, 3D]
  attn::GemmLaunch g;
  rc = make_matrix_map(&g.ta, x, dtype, 1, 1, rows, D, D, 128);
  if (!rc) rc = make_matrix_map(&g.tb, w_qkv, dtype, 1, 1, D, 3LL * D, 3LL * D, 64);
  if (rc) return rc;
  g.c = workspace;
  g.c_type = dtype;
  g.ldc = 3LL * D;
  g.c_s1 = g.c_s2 = 0;
  g.M = static_cast<int>(rows), g.N = 3 * D, g.K = D, g.Z1 = 1, g.Z2 = 1;
  g.bn = (3 * D) % 256 == 0 ? 256 : 128;
  g.mb = g.bn == 256 ? 2 : 1;  // 256-row tiles: one third less operand traffic per flop
  g.b_kmajor = false;
  g.a_swap = g.b_swap = 0;
  g.bf16 = dtype == ATTN_BF16;
  g.alpha = 1.f;
  g.status = ds->status;
  g.limit = wait_limit();
  if ((rc = to_rc(attn::launch_gemm(g, st)))) return rc;

  // 2. attention on the projection in place: Q, K, V are the three column
  //    blocks of each row, i.e. head-interleaved with row stride 3D.
  const uint8_t* base = static_cast<const uint8_t*>(workspace);
  return run_flash(base, base + static_cast<size_t>(D) * 2, base + static_cast<size_t>(2 * D) * 2, o,
                   nullptr, B, h, S, d, 1.0f / sqrtf(static_cast<float>(d)), ATTN_LAYOUT_BSHD, 1,
                   dtype, 3LL * D, D, ds, st);
}

int qkv_proj_attn_fused(const void* x, const void* w_qkv, void* o, int B, int S, int D, int h, int dtype,
                        void* stream) {
  int rc = attn::validate_qkv_proj(x, w_qkv, o, B, S, D, h, dtype);
  if (rc) return rc;
  if (D / h != 64 || S > 512) return ATTN_E_SHAPE;
  DeviceState* ds = nullptr;
  if ((rc = device_setup(&ds))) return rc;
  attn::FusedLaunch a;
  const cuuint64_t e = 2;
  const CUtensorMapDataType dt =
      dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  {  // X [B, S, D]: dims (D, S, B), box 64 x 128 x 1
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * e, static_cast<cuuint64_t>(S) * D * e};
    cuuint32_t box[3] = {64, 128, 1}, estr[3] = {1, 1, 1};
    if (g_encode(&a.t0, dt, 3, const_cast<void*>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return ATTN_E_DEVICE;
  }
  {  // W_qkv [D, 3D]: dims (3D, D), box 64 x 64
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(3LL * D), static_cast<cuuint64_t>(D)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(3LL * D) * e};
    cuuint32_t box[2] = {64, 64}, estr[2] = {1, 1};
    if (g_encode(&a.t1, dt, 2, const_cast<void*>(w_qkv), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return ATTN_E_DEVICE;
  }
  a.t2 = a.t1;  // unused by the projection form
  // O [B, S, h, 64]: the head-interleaved layout with row stride D
  if ((rc = make_map(&a.to, o, dtype, ATTN_LAYOUT_BSHD, B, h, S, 64, D, 128, &a.o_swap))) return rc;
  a.project = true;
  a.lse = nullptr;
  a.B = B, a.S = S, a.H = h, a.D = D;
  a.hs_swap = 0;
  a.bf16 = dtype == ATTN_BF16;
  a.scale = 1.0f / sqrtf(64.0f);
  a.status = ds->status;
  a.limit = wait_limit();
  return to_rc(attn::launch_fused_qkv_attn(a, static_cast<cudaStream_t>(stream)));
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_E_NULL: return "ATTN_E_NULL: a required pointer is NULL";
    case ATTN_E_SHAPE: return "ATTN_E_SHAPE: unsupported or inconsistent sizes";
    case ATTN_E_ALIGN: return "ATTN_E_ALIGN: tensor pointer not 16-byte aligned";
    case ATTN_E_LAYOUT: return "ATTN_E_LAYOUT: unknown layout";
    case ATTN_E_DTYPE: return "ATTN_E_DTYPE: unknown or unsupported dtype";
    case ATTN_E_WORKSPACE: return "ATTN_E_WORKSPACE: workspace missing, misaligned or too small";
    case ATTN_E_ALIAS: return "ATTN_E_ALIAS: output overlaps an input or the workspace";
    case ATTN_E_DEVICE: return "ATTN_E_DEVICE: no usable sm_103 device or driver entry point";
    case ATTN_E_TIMEOUT: return "ATTN_E_TIMEOUT: a kernel pipeline wait exceeded its limit";
    case ATTN_E_MISMATCH: return "ATTN_E_MISMATCH: the two outputs differ by more than atol";
    case ATTN_E_SCRATCH_LIMIT:
      return "ATTN_E_SCRATCH_LIMIT: problem exceeds the fixed scratch of qkv_proj_attn_noalloc";
    default: break;
  }
  if (status > 0) return cudaGetErrorString(static_cast<cudaError_t>(status));
  return "unknown attn status";
}

int attn_select_kernel(int option_enabled, int seq_len, int threshold) {
  const int thr = threshold > 0 ? threshold : 1024;
  return (option_enabled && seq_len > thr) ? ATTN_KERNEL_ONLINE : ATTN_KERNEL_NAIVE;
}

int attn_fwd_auto(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                  int S, int d, float scale, int layout, int dtype, int option_enabled,
                  int threshold, void* workspace, size_t ws_bytes, void* stream, int* chosen) {
  const int kind = attn_select_kernel(option_enabled, S, threshold);
  if (chosen) *chosen = kind;
  if (kind == ATTN_KERNEL_ONLINE)
    return attn_fwd(q, k, v, o, lse, B, h, S, d, scale, layout, dtype, stream);
  return attn_fwd_naive(q, k, v, o, lse, B, h, S, d, scale, layout, dtype, workspace, ws_bytes,
                        stream);
}

int attn_compare(const void* a, const void* b, long long n, int dtype, float atol, float* max_abs,
                 void* stream) {
  if (max_abs) *max_abs = 0.f;
  if (!a || !b) return ATTN_E_NULL;
  if (dtype != ATTN_F32 && dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_E_DTYPE;
  if (n < 0 || !(atol >= 0.f)) return ATTN_E_SHAPE;
  DeviceState* ds = nullptr;
  int rc = device_setup(&ds);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float result = 0.f;
  if (n > 0) {
    rc = to_rc(attn::launch_max_abs_diff(a, b, n, dtype, &result, st));
    if (rc) return rc;
  }
  if (max_abs) *max_abs = result;
  return (result <= atol) ? ATTN_OK : ATTN_E_MISMATCH;
}

int attn_selftest_wait_timeout(long long limit_cycles, void* stream) {
  if (limit_cycles < 1 || limit_cycles > 10000000000LL) return ATTN_E_SHAPE;
  DeviceState* ds = nullptr;
  int rc = device_setup(&ds);
  if (rc) return rc;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(ds->status, limit_cycles);
  return to_rc(cudaGetLastError());
}

int attn_get_device_status(void* stream, unsigned int* detail) {
  if (detail) *detail = 0;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return static_cast<int>(e);
  DeviceState* ds = nullptr;
  int rc = device_setup(&ds);
  if (rc) return rc;
  unsigned v = 0, zero = 0;
  if ((e = cudaMemcpy(&v, ds->status, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return static_cast<int>(e);
  if ((e = cudaMemcpy(ds->status, &zero, sizeof zero, cudaMemcpyHostToDevice)) != cudaSuccess)
    return static_cast<int>(e);
  if (detail) *detail = v;
  return v ? ATTN_E_TIMEOUT : ATTN_OK;
}

}  // extern "C"
