"""fp64 CPU oracle for the multi-head attention forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library (``head_attention_fwd_gb300``) never imports it, and the two
share no code: this package wraps ``attn_oracle.cpp`` (plain C++, fp64), built
with g++ into ``liboracle.so`` beside it.

Every function follows a passage of the pages (page title, section):

* ``softmax``                 -- "Transformer算子生态深度分析" ch.2 §2.3 (three-step stable softmax)
* ``online_softmax``          -- same chapter §2.6 (block merge of running max / exp-sum);
                                 "WebGPU 算子优化：QKV 内存合并与 FlashAttention 分块计算"
                                 §FlashAttention 分块计算原理与浏览器适配 (m_new, l_new);
                                 "[WebGPU] Proposal: ... online softmax ..." §四 (block size 1)
* ``attention``, ``attention_rows`` -- ch.2 §2.2-§2.4 (scores, softmax, weighted sum);
                                 layouts from the WebGPU page §QKV 矩阵的内存合并模式选择
* ``qkv_projection``, ``split_heads``, ``qkv_proj_attention`` -- ch.2 §2.1 (fused [D,3D] weight)
* ``attention_grouped``       -- the "split" (head-group) layout of the same WebGPU section
* ``decode``                  -- IEEE-754 binary16 / bfloat16 widening of the GPU's input bytes

The pins that tie each function to the pages and to mathematics (not to
itself) are in ``tests/test_oracle.py``.  Every function there is pinned;
nothing here is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# element-type codes understood by attn_oracle.cpp
ET_F64, ET_F32, ET_F16, ET_BF16 = 0, 1, 2, 3

_c_double_p = ctypes.POINTER(ctypes.c_double)
_c_i64_p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile liboracle.so with g++ when it is missing or older than its source."""
    with _lock:
        stale = force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        _lib = bind(ctypes.CDLL(build()))
    return _lib


def bind(lib):
    """Declare the C signatures on a loaded liboracle (or a test build of it)."""
    vp, i64, dbl, cint = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_int
    lib.oracle_threads.argtypes = [cint]
    lib.oracle_decode.argtypes = [vp, cint, i64, _c_double_p]
    lib.oracle_softmax.argtypes = [_c_double_p, i64, _c_double_p, _c_double_p, _c_double_p]
    lib.oracle_online_softmax.argtypes = [_c_double_p, i64, i64, _c_double_p, _c_double_p,
                                          _c_double_p, _c_double_p, _c_double_p]
    lib.oracle_attention.argtypes = [vp, vp, vp, cint, i64, i64, i64, i64, cint, dbl,
                                     _c_double_p, _c_double_p, cint]
    lib.oracle_attention_rows.argtypes = [vp, vp, vp, cint, i64, i64, i64, i64, cint, dbl,
                                          _c_i64_p, i64, _c_double_p, _c_double_p, cint]
    lib.oracle_qkv_projection.argtypes = [vp, vp, cint, i64, i64, i64, _c_double_p, cint]
    lib.oracle_split_heads.argtypes = [_c_double_p, i64, i64, i64, i64, _c_double_p,
                                       _c_double_p, _c_double_p]
    lib.oracle_qkv_proj_attention.argtypes = [vp, vp, cint, i64, i64, i64, i64, dbl,
                                              _c_double_p, _c_double_p, cint]
    lib.oracle_attention_grouped.argtypes = [vp, vp, vp, cint, i64, i64, i64, i64, i64, dbl,
                                             _c_double_p, _c_double_p, cint]
    return lib


def _dp(a: np.ndarray):
    return a.ctypes.data_as(_c_double_p)


def _raw(t):
    """(contiguous host array holding the exact element bytes, element-type code).

    Accepts numpy arrays (float64 / float32 / float16) and torch CPU tensors
    (float64 / float32 / float16 / bfloat16).  No arithmetic: the bytes are
    passed through and widened inside the oracle.
    """
    if isinstance(t, np.ndarray):
        a = np.ascontiguousarray(t)
        et = {np.dtype(np.float64): ET_F64, np.dtype(np.float32): ET_F32,
              np.dtype(np.float16): ET_F16}.get(a.dtype)
        if et is None:
            raise TypeError(f"oracle: unsupported numpy dtype {a.dtype}")
        return a, et
    import torch  # torch tensors: view the raw bits
    if t.device.type != "cpu":
        raise ValueError("oracle inputs must live in host memory")
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy(), ET_BF16
    et = {torch.float64: ET_F64, torch.float32: ET_F32, torch.float16: ET_F16}.get(t.dtype)
    if et is None:
        raise TypeError(f"oracle: unsupported torch dtype {t.dtype}")
    return t.numpy(), et


def threads(nthreads: int = 0) -> int:
    """Worker threads a call with ``nthreads`` uses (0 = all host cores)."""
    return int(_load().oracle_threads(int(nthreads)))


def decode(t) -> np.ndarray:
    """Widen the elements of ``t`` to float64 (flat array)."""
    a, et = _raw(t)
    out = np.empty(a.size, dtype=np.float64)
    if _load().oracle_decode(a.ctypes.data, et, a.size, _dp(out)):
        raise ValueError("oracle_decode: bad arguments")
    return out


def softmax(s) -> tuple[np.ndarray, float, float]:
    """Three-step stable softmax of a vector: (p, m, d)."""
    s = np.ascontiguousarray(s, dtype=np.float64)
    p = np.empty_like(s)
    m, d = ctypes.c_double(), ctypes.c_double()
    if _load().oracle_softmax(_dp(s), s.size, _dp(p), ctypes.byref(m), ctypes.byref(d)):
        raise ValueError("oracle_softmax: bad arguments")
    return p, m.value, d.value


def online_softmax(s, block: int = 1):
    """Blocked online softmax of a vector: (p, m, d, m_trace, d_trace)."""
    s = np.ascontiguousarray(s, dtype=np.float64)
    nblk = -(-s.size // block)
    p = np.empty_like(s)
    mt, dt = np.empty(nblk), np.empty(nblk)
    m, d = ctypes.c_double(), ctypes.c_double()
    if _load().oracle_online_softmax(_dp(s), s.size, block, _dp(p), _dp(mt), _dp(dt),
                                     ctypes.byref(m), ctypes.byref(d)):
        raise ValueError("oracle_online_softmax: bad arguments")
    return p, m.value, d.value, mt, dt


def _shape(q, layout):
    if layout == 0:
        B, H, S, d = q.shape
    elif layout == 1:
        B, S, H, d = q.shape
    else:
        raise ValueError("layout must be 0 ([B,H,S,d]) or 1 ([B,S,H,d])")
    return int(B), int(H), int(S), int(d)


def attention(q, k, v, layout: int = 0, scale: float | None = None, nthreads: int = 0):
    """O = softmax(scale·Q·K^T)·V and LSE for every query row.

    q, k, v: same shape and element type, [B,H,S,d] (layout 0) or [B,S,H,d]
    (layout 1).  Returns (o float64 in the same layout, lse float64 [B,H,S]).
    """
    B, H, S, d = _shape(q, layout)
    if tuple(k.shape) != tuple(q.shape) or tuple(v.shape) != tuple(q.shape):
        raise ValueError("q, k, v must have the same shape")
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    (qa, et), (ka, et_k), (va, et_v) = _raw(q), _raw(k), _raw(v)
    if not (et == et_k == et_v):
        raise TypeError("q, k, v must have the same element type")
    o = np.empty(tuple(q.shape), dtype=np.float64)
    lse = np.empty((B, H, S), dtype=np.float64)
    if _load().oracle_attention(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, et, B, H, S, d,
                                layout, scale, _dp(o), _dp(lse), nthreads):
        raise ValueError("oracle_attention: bad arguments")
    return o, lse


def attention_rows(q, k, v, rows, layout: int = 0, scale: float | None = None, nthreads: int = 0):
    """Like ``attention`` for selected query rows only.

    rows: flat indices (b*H + h)*S + i.  Returns (o [len(rows), d], lse [len(rows)]).
    """
    B, H, S, d = _shape(q, layout)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    (qa, et), (ka, _), (va, _) = _raw(q), _raw(k), _raw(v)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.empty((rows.size, d), dtype=np.float64)
    lse = np.empty(rows.size, dtype=np.float64)
    if _load().oracle_attention_rows(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, et, B, H, S,
                                     d, layout, scale, rows.ctypes.data_as(_c_i64_p), rows.size,
                                     _dp(o), _dp(lse), nthreads):
        raise ValueError("oracle_attention_rows: bad arguments")
    return o, lse


def qkv_projection(x, w, nthreads: int = 0) -> np.ndarray:
    """X [B,S,D] · W_qkv [D,3D] in fp64 -> [B,S,3D]."""
    B, S, D = (int(n) for n in x.shape)
    if tuple(w.shape) != (D, 3 * D):
        raise ValueError("w_qkv must be [D, 3D]")
    (xa, et), (wa, et_w) = _raw(x), _raw(w)
    if et != et_w:
        raise TypeError("x and w_qkv must have the same element type")
    out = np.empty((B, S, 3 * D), dtype=np.float64)
    if _load().oracle_qkv_projection(xa.ctypes.data, wa.ctypes.data, et, B, S, D, _dp(out), nthreads):
        raise ValueError("oracle_qkv_projection: bad arguments")
    return out


def split_heads(qkv: np.ndarray, h: int):
    """[B,S,3D] -> (q, k, v), each [B,S,h,d] (head-interleaved)."""
    qkv = np.ascontiguousarray(qkv, dtype=np.float64)
    B, S, D3 = qkv.shape
    D = D3 // 3
    q, k, v = (np.empty((B, S, h, D // h)) for _ in range(3))
    if _load().oracle_split_heads(_dp(qkv), B, S, D, h, _dp(q), _dp(k), _dp(v)):
        raise ValueError("oracle_split_heads: bad arguments")
    return q, k, v


def qkv_proj_attention(x, w, h: int, scale: float | None = None, nthreads: int = 0):
    """Fused projection then attention: (o [B,S,h,d] float64, lse [B,h,S])."""
    B, S, D = (int(n) for n in x.shape)
    d = D // h
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    (xa, et), (wa, _) = _raw(x), _raw(w)
    o = np.empty((B, S, h, d), dtype=np.float64)
    lse = np.empty((B, h, S), dtype=np.float64)
    if _load().oracle_qkv_proj_attention(xa.ctypes.data, wa.ctypes.data, et, B, S, D, h, scale,
                                         _dp(o), _dp(lse), nthreads):
        raise ValueError("oracle_qkv_proj_attention: bad arguments")
    return o, lse


def attention_grouped(q, k, v, hg: int, scale: float | None = None, nthreads: int = 0):
    """Attention on the head-group layout [B, H/hg, S, hg, d]: (o same layout, lse [B,H,S])."""
    B, G, S, hg_, d = (int(n) for n in q.shape)
    if hg_ != hg or tuple(k.shape) != tuple(q.shape) or tuple(v.shape) != tuple(q.shape):
        raise ValueError("q, k, v must be [B, H/hg, S, hg, d]")
    H = G * hg
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    (qa, et), (ka, _), (va, _) = _raw(q), _raw(k), _raw(v)
    o = np.empty(tuple(q.shape), dtype=np.float64)
    lse = np.empty((B, H, S), dtype=np.float64)
    if _load().oracle_attention_grouped(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, et, B, H, S,
                                        d, hg, scale, _dp(o), _dp(lse), nthreads):
        raise ValueError("oracle_attention_grouped: bad arguments")
    return o, lse
