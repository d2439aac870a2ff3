// qkv_proj_attn_noalloc: the fused QKV projection + attention for callers
// that cannot allocate device memory (see include/attn.h for who they are).
//
// The projection [B, S, 3D] normally lives in a workspace the caller
// allocates.  Here it lives in a fixed array declared statically in device
// memory, so the call allocates nothing: no cudaMalloc, no cudaFree, no
// allocating library routine.  The array is resolved once per device
// (cudaGetSymbolAddress with that device current) and then handed to the
// unchanged qkv_proj_attn path as its workspace.

#include <mutex>

#include "attn.h"
#include "common.h"

namespace {

// Shared by every call on a device; holds the last call's projection.  The
// projection GEMM writes every element the attention kernel then reads, so
// nothing here has to be cleared between calls.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device, resolved on
// the first call per device.  The name g_noalloc_scratch in host code is only
// a host-side handle, never a device address.
int scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_E_DEVICE;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (!p) return ATTN_E_DEVICE;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int qkv_proj_attn_noalloc(const void* x, const void* w_qkv, void* o, int B, int S, int D,
                                     int h, int dtype, void* stream) {
  // The same checks as qkv_proj_attn first, so that a bad argument is named
  // as such even on a problem too large for the scratch.
  const int rc0 = attn::validate_qkv_proj(x, w_qkv, o, B, S, D, h, dtype);
  if (rc0) return rc0;
  const size_t need = qkv_proj_attn_workspace_bytes(B, S, D, dtype);
  if (need > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_E_SCRATCH_LIMIT;
  void* ws = nullptr;
  const int rc = scratch_on_current_device(&ws);
  if (rc) return rc;
  return qkv_proj_attn(x, w_qkv, o, B, S, D, h, dtype, ws, ATTN_NOALLOC_SCRATCH_BYTES, stream);
}
