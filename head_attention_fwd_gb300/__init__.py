"""GB300 (sm_103a) multi-head attention forward: Python binding.

A thin ctypes layer over ``libattn_gb300.so`` (C ABI in ``include/attn.h``).
It only marshals arguments -- every step of the computation runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  There is
no fallback: if the library is not built, every call raises.

Entry points (same names as the C ABI):

* ``attn_fwd(q, k, v, ...)``        fused online-softmax attention (through
  ``attn_fwd_ws`` with a small scratch unless ``split=False``)
* ``attn_fwd_mixed(q, k, v, ...)``  fp32 inputs, 16-bit output (converted once, then fused)
* ``attn_fwd_naive(q, k, v, ...)``  unfused two-pass-softmax comparison path
* ``qkv_proj_attn(x, w_qkv, h, ...)`` fused QKV projection, then attention
* ``qkv_proj_attn_fused(x, w_qkv, h, ...)`` the same in one kernel (d = 64, S <= 512)
* ``qkv_proj_attn_noalloc(x, w_qkv, h, ...)`` the same without a workspace argument
* ``attn_get_device_status()``, ``attn_status_string(rc)``
"""

from __future__ import annotations

import ctypes
import os
import threading

LAYOUT_BHSD = 0  # contiguous [B, h, S, d]
LAYOUT_BSHD = 1  # head-interleaved [B, S, h, d]
LAYOUT_GROUPED = 2  # head groups [B, h/hg, S, hg, d] (attn_fwd_grouped)
ATTN_F32, ATTN_F16, ATTN_BF16 = 0, 1, 2
ATTN_OK = 0
ATTN_E_TIMEOUT = -9
ATTN_E_MISMATCH = -11
ATTN_KERNEL_NAIVE, ATTN_KERNEL_ONLINE = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn_gb300.so")
_lib = None
_lock = threading.Lock()


class AttnError(RuntimeError):
    def __init__(self, rc: int, what: str):
        self.rc = rc
        super().__init__(f"{what} failed: {attn_status_string(rc)} (status {rc})")


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            vp, ci, cf, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci, ci, vp]
            L.attn_fwd.restype = ci
            L.attn_fwd_ws.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci, ci, vp, sz, vp]
            L.attn_fwd_ws.restype = ci
            L.attn_fwd_ws_bytes.argtypes = [ci, ci, ci, ci, ci]
            L.attn_fwd_ws_bytes.restype = sz
            L.attn_fwd_mixed.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci, ci, vp, sz, vp]
            L.attn_fwd_mixed.restype = ci
            L.attn_fwd_mixed_workspace_bytes.argtypes = [ci, ci, ci, ci, ci]
            L.attn_fwd_mixed_workspace_bytes.restype = sz
            L.attn_fwd_grouped.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp]
            L.attn_fwd_grouped.restype = ci
            L.attn_fwd_naive.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci, ci, vp, sz, vp]
            L.attn_fwd_naive.restype = ci
            L.attn_fwd_naive_workspace_bytes.argtypes = [ci, ci, ci, ci]
            L.attn_fwd_naive_workspace_bytes.restype = sz
            L.qkv_proj_attn.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, vp, sz, vp]
            L.qkv_proj_attn.restype = ci
            L.qkv_proj_attn_fused.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, vp]
            L.qkv_proj_attn_fused.restype = ci
            L.qkv_proj_attn_noalloc.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, vp]
            L.qkv_proj_attn_noalloc.restype = ci
            L.qkv_proj_attn_workspace_bytes.argtypes = [ci, ci, ci, ci]
            L.qkv_proj_attn_workspace_bytes.restype = sz
            L.attn_status_string.argtypes = [ci]
            L.attn_status_string.restype = ctypes.c_char_p
            L.attn_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
            L.attn_get_device_status.restype = ci
            L.attn_selftest_wait_timeout.argtypes = [ctypes.c_longlong, vp]
            L.attn_selftest_wait_timeout.restype = ci
            L.attn_select_kernel.argtypes = [ci, ci, ci]
            L.attn_select_kernel.restype = ci
            L.attn_fwd_auto.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci, ci, ci, ci, vp, sz, vp,
                                        ctypes.POINTER(ci)]
            L.attn_fwd_auto.restype = ci
            L.attn_compare.argtypes = [vp, vp, ctypes.c_longlong, ci, cf, ctypes.POINTER(cf), vp]
            L.attn_compare.restype = ci
            L.attn_flash_schedule.argtypes = [ci, ci, ci, ci, ci, ci, ctypes.POINTER(ci), ctypes.POINTER(ci),
                                              ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_longlong),
                                              ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ci)]
            L.attn_flash_schedule.restype = ci
            L.attn_abi_version.argtypes = []
            L.attn_abi_version.restype = ci
            _lib = L
    return _lib


def attn_status_string(rc: int) -> str:
    return lib().attn_status_string(int(rc)).decode()


def _torch():
    import torch
    return torch


def dtype_code(dt) -> int:
    torch = _torch()
    codes = {torch.float32: ATTN_F32, torch.float16: ATTN_F16, torch.bfloat16: ATTN_BF16}
    if dt not in codes:
        raise TypeError(f"unsupported dtype {dt}")
    return codes[dt]


def _stream_ptr(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dims(q, layout):
    if q.dim() != 4:
        raise ValueError("q must be 4-d")
    if layout == LAYOUT_BHSD:
        B, h, S, d = q.shape
    elif layout == LAYOUT_BSHD:
        B, S, h, d = q.shape
    else:
        raise ValueError("layout must be 0 ([B,h,S,d]) or 1 ([B,S,h,d])")
    return int(B), int(h), int(S), int(d)


def _check_dense(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def attn_flash_schedule(B: int, h: int, S: int, d: int, num_sms: int, split: bool = True) -> dict:
    """The attention kernel's work schedule for a problem on num_sms SMs (host
    only, nothing is launched): mode, grid, dp_end, sk_units and, when items
    are cut (mode 2), the run bounds `cut` and the merge ranges `g_last`."""
    mode, grid = ctypes.c_int(), ctypes.c_int()
    dp_end, sk_units = ctypes.c_longlong(), ctypes.c_longlong()
    cut = (ctypes.c_longlong * 257)()
    g_last = (ctypes.c_int * 256)()
    rc = lib().attn_flash_schedule(B, h, S, d, num_sms, int(bool(split)), ctypes.byref(mode), ctypes.byref(grid),
                                   ctypes.byref(dp_end), ctypes.byref(sk_units), cut, g_last)
    if rc != 0:
        raise ValueError(f"attn_flash_schedule: {attn_status_string(rc)}")
    out = {"mode": mode.value, "grid": grid.value, "dp_end": dp_end.value, "sk_units": sk_units.value}
    if sk_units.value > 0:
        out["cut"] = list(cut[: grid.value + 1])
        out["g_last"] = list(g_last[: grid.value])
    return out


def attn_fwd_ws_bytes(B: int, h: int, S: int, d: int, dtype) -> int:
    """Scratch bytes attn_fwd_ws needs on the current device (0: none)."""
    return int(lib().attn_fwd_ws_bytes(B, h, S, d, dtype_code(dtype)))


def attn_fwd(q, k, v, o=None, lse=None, *, layout: int = LAYOUT_BHSD, scale: float | None = None,
             want_lse: bool = False, stream=None, split: bool = True, workspace=None):
    """O = softmax(scale·Q·K^T)·V (fused, one launch).  Returns (o, lse or None).

    split=True calls the C entry attn_fwd_ws with a scratch buffer (``workspace``,
    or one taken from torch's allocator), which lets the kernel cut the last
    wave of work items along the key axis; split=False calls attn_fwd."""
    torch = _torch()
    B, h, S, d = _dims(q, layout)
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share shape and dtype")
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, h, S), dtype=torch.float32, device=q.device)
    _check_dense(q, k, v, o, lse)
    sc = float(scale) if scale else 0.0
    if not split:
        rc = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, h, S, d, sc, layout,
                            dtype_code(q.dtype), _stream_ptr(stream))
        if rc:
            raise AttnError(rc, "attn_fwd")
        return o, lse
    if workspace is None:
        need = attn_fwd_ws_bytes(B, h, S, d, q.dtype)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            if isinstance(stream, torch.cuda.Stream):
                workspace.record_stream(stream)
    _check_dense(workspace)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().attn_fwd_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, h, S, d, sc, layout,
                           dtype_code(q.dtype), _ptr(workspace), nbytes, _stream_ptr(stream))
    if rc:
        raise AttnError(rc, "attn_fwd_ws")
    return o, lse


def attn_fwd_mixed_workspace_bytes(B: int, h: int, S: int, d: int, out_dtype) -> int:
    return int(lib().attn_fwd_mixed_workspace_bytes(B, h, S, d, dtype_code(out_dtype)))


def attn_fwd_mixed(q, k, v, o=None, lse=None, workspace=None, *, out_dtype=None, layout: int = LAYOUT_BHSD,
                   scale: float | None = None, want_lse: bool = False, stream=None):
    """fp32 q, k, v -> 16-bit o (out_dtype, default float16).  Returns (o, lse or None, workspace)."""
    torch = _torch()
    out_dtype = out_dtype or torch.float16
    B, h, S, d = _dims(q, layout)
    if q.dtype != torch.float32 or k.dtype != torch.float32 or v.dtype != torch.float32:
        raise ValueError("q, k, v must be float32")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one shape")
    if o is None:
        o = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, h, S), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(attn_fwd_mixed_workspace_bytes(B, h, S, d, out_dtype), dtype=torch.uint8,
                                device=q.device)
        if isinstance(stream, torch.cuda.Stream):
            workspace.record_stream(stream)
    _check_dense(q, k, v, o, lse, workspace)
    rc = lib().attn_fwd_mixed(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, h, S, d,
                              float(scale) if scale else 0.0, layout, dtype_code(o.dtype), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if rc:
        raise AttnError(rc, "attn_fwd_mixed")
    return o, lse, workspace


def attn_fwd_grouped(q, k, v, o=None, lse=None, *, scale: float | None = None, want_lse: bool = False,
                     stream=None):
    """attn_fwd on the head-group layout: q, k, v are [B, h/hg, S, hg, d].  Returns (o, lse or None)."""
    torch = _torch()
    if q.dim() != 5:
        raise ValueError("q must be [B, h/hg, S, hg, d]")
    B, G, S, hg, d = (int(n) for n in q.shape)
    h = G * hg
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share shape and dtype")
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, h, S), dtype=torch.float32, device=q.device)
    _check_dense(q, k, v, o, lse)
    rc = lib().attn_fwd_grouped(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, h, S, d, hg,
                                float(scale) if scale else 0.0, dtype_code(q.dtype), _stream_ptr(stream))
    if rc:
        raise AttnError(rc, "attn_fwd_grouped")
    return o, lse


def attn_fwd_naive_workspace_bytes(B: int, h: int, S: int, dtype) -> int:
    return int(lib().attn_fwd_naive_workspace_bytes(B, h, S, dtype_code(dtype)))


def attn_fwd_naive(q, k, v, o=None, lse=None, workspace=None, *, layout: int = LAYOUT_BHSD,
                   scale: float | None = None, want_lse: bool = False, stream=None):
    """Unfused comparison path (S and P materialised).  Returns (o, lse or None, workspace)."""
    torch = _torch()
    B, h, S, d = _dims(q, layout)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, h, S), dtype=torch.float32, device=q.device)
    need = attn_fwd_naive_workspace_bytes(B, h, S, q.dtype)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check_dense(q, k, v, o, lse, workspace)
    rc = lib().attn_fwd_naive(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, h, S, d,
                              float(scale) if scale else 0.0, layout, dtype_code(q.dtype),
                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _stream_ptr(stream))
    if rc:
        raise AttnError(rc, "attn_fwd_naive")
    return o, lse, workspace


def qkv_proj_attn_workspace_bytes(B: int, S: int, D: int, dtype) -> int:
    return int(lib().qkv_proj_attn_workspace_bytes(B, S, D, dtype_code(dtype)))


def qkv_proj_attn(x, w_qkv, h: int, o=None, workspace=None, *, stream=None):
    """X [B,S,D] · W_qkv [D,3D] -> heads -> attention.  Returns (o [B,S,h,d], workspace [B,S,3D] bytes)."""
    torch = _torch()
    B, S, D = (int(n) for n in x.shape)
    if o is None:
        o = torch.empty((B, S, h, D // h), dtype=x.dtype, device=x.device)
    need = qkv_proj_attn_workspace_bytes(B, S, D, x.dtype)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _check_dense(x, w_qkv, o, workspace)
    rc = lib().qkv_proj_attn(_ptr(x), _ptr(w_qkv), _ptr(o), B, S, D, h, dtype_code(x.dtype),
                             _ptr(workspace), workspace.numel() * workspace.element_size(),
                             _stream_ptr(stream))
    if rc:
        raise AttnError(rc, "qkv_proj_attn")
    return o, workspace


def qkv_proj_attn_fused(x, w_qkv, h: int, o=None, *, stream=None):
    """qkv_proj_attn in one kernel launch (d = D/h = 64, S <= 512): the projection
    feeds the attention on chip, no workspace.  Returns o [B,S,h,d]."""
    torch = _torch()
    B, S, D = (int(n) for n in x.shape)
    if o is None:
        o = torch.empty((B, S, h, D // h), dtype=x.dtype, device=x.device)
    _check_dense(x, w_qkv, o)
    rc = lib().qkv_proj_attn_fused(_ptr(x), _ptr(w_qkv), _ptr(o), B, S, D, h, dtype_code(x.dtype),
                                   _stream_ptr(stream))
    if rc:
        raise AttnError(rc, "qkv_proj_attn_fused")
    return o


def qkv_proj_attn_noalloc(x, w_qkv, h: int, o=None, *, stream=None):
    """qkv_proj_attn without a workspace argument, for callers that cannot allocate
    device memory: the projection goes to the library's fixed static scratch
    (ATTN_NOALLOC_SCRATCH_BYTES = 32 MiB per device).  The C call allocates nothing;
    only the optional output below is allocated here, when ``o`` is not given.
    The scratch belongs to the current device, so the call runs with x's device
    made current.  Returns o [B,S,h,d]."""
    torch = _torch()
    B, S, D = (int(n) for n in x.shape)
    if o is None:
        o = torch.empty((B, S, h, D // h), dtype=x.dtype, device=x.device)
    _check_dense(x, w_qkv, o)
    if w_qkv.device != x.device or o.device != x.device:
        raise ValueError("x, w_qkv and o must be on one device")
    with torch.cuda.device(x.device):
        rc = lib().qkv_proj_attn_noalloc(_ptr(x), _ptr(w_qkv), _ptr(o), B, S, D, h, dtype_code(x.dtype),
                                         _stream_ptr(stream))
    if rc:
        raise AttnError(rc, "qkv_proj_attn_noalloc")
    return o


def select_kernel(option_enabled: bool, seq_len: int, threshold: int = 0) -> int:
    """ATTN_KERNEL_ONLINE when the option is on and seq_len > threshold (1024 by default)."""
    return int(lib().attn_select_kernel(int(bool(option_enabled)), int(seq_len), int(threshold)))


def attn_fwd_auto(q, k, v, o=None, lse=None, workspace=None, *, option_enabled: bool = True,
                  threshold: int = 0, layout: int = LAYOUT_BHSD, scale: float | None = None,
                  want_lse: bool = False, stream=None):
    """attn_fwd or attn_fwd_naive as select_kernel picks.  Returns (o, lse or None, kernel)."""
    torch = _torch()
    B, h, S, d = _dims(q, layout)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, h, S), dtype=torch.float32, device=q.device)
    if workspace is None and select_kernel(option_enabled, S, threshold) == ATTN_KERNEL_NAIVE:
        workspace = torch.empty(attn_fwd_naive_workspace_bytes(B, h, S, q.dtype), dtype=torch.uint8,
                                device=q.device)
    _check_dense(q, k, v, o, lse, workspace)
    chosen = ctypes.c_int(-1)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().attn_fwd_auto(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, h, S, d,
                             float(scale) if scale else 0.0, layout, dtype_code(q.dtype),
                             int(bool(option_enabled)), int(threshold), _ptr(workspace), nbytes,
                             _stream_ptr(stream), ctypes.byref(chosen))
    if rc:
        raise AttnError(rc, "attn_fwd_auto")
    return o, lse, chosen.value


def attn_compare(a, b, atol: float, stream=None) -> tuple[int, float]:
    """(status, max |a - b|) of two device tensors of one dtype (synchronises the stream)."""
    if a.shape != b.shape or a.dtype != b.dtype:
        raise ValueError("a and b must share shape and dtype")
    _check_dense(a, b)
    mx = ctypes.c_float(0.0)
    rc = lib().attn_compare(_ptr(a), _ptr(b), a.numel(), dtype_code(a.dtype), float(atol),
                            ctypes.byref(mx), _stream_ptr(stream))
    return int(rc), float(mx.value)


def assert_numerically_equal(out_naive, out_online, atol: float = 1e-3, stream=None) -> None:
    """Raises AssertionError when the two outputs differ by more than atol."""
    rc, mx = attn_compare(out_naive, out_online, atol, stream)
    if rc == ATTN_E_MISMATCH:
        raise AssertionError(f"online softmax disagrees with naive: max |diff| {mx:.3e} > {atol}")
    if rc:
        raise AttnError(rc, "attn_compare")


def attn_selftest_wait_timeout(limit_cycles: int, stream=None) -> None:
    """Launch the stalled-wait self-test (see include/attn.h); read the result
    with attn_get_device_status()."""
    rc = lib().attn_selftest_wait_timeout(int(limit_cycles), _stream_ptr(stream))
    if rc:
        raise AttnError(rc, "attn_selftest_wait_timeout")


def attn_get_device_status(stream=None) -> tuple[int, int]:
    """Synchronise the stream; return (status, raw detail) and clear the device status word."""
    detail = ctypes.c_uint(0)
    rc = lib().attn_get_device_status(_stream_ptr(stream), ctypes.byref(detail))
    return int(rc), int(detail.value)
