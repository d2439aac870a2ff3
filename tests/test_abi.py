"""C-ABI checks that need no GPU: the library loads, exports every function
include/attn.h declares, and rejects invalid arguments with the documented
negative codes before making any CUDA call."""

import ctypes
import os
import re

import pytest
import torch

import head_attention_fwd_gb300 as attn
from head_attention_fwd_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
E = dict(OK=0, NULL=-1, SHAPE=-2, ALIGN=-3, LAYOUT=-4, DTYPE=-5, WORKSPACE=-6, ALIAS=-7, DEVICE=-8,
         TIMEOUT=-9)


@pytest.fixture(scope="module")
def L():
    _build.build()
    return attn.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["attn_fwd", "attn_fwd_naive", "attn_fwd_naive_workspace_bytes", "qkv_proj_attn",
              "qkv_proj_attn_workspace_bytes", "attn_status_string", "attn_get_device_status",
              "attn_abi_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), f"libattn_gb300.so does not export {n}"
    assert L.attn_abi_version() == 1


def test_status_strings(L):
    for name, code in E.items():
        s = attn.attn_status_string(code)
        assert s and (name in s or code == 0)
    assert "unknown" in attn.attn_status_string(-1234)


# Fake, never-dereferenced device addresses: every call below fails validation
# before the library makes its first CUDA call.
A = 1 << 32  # spacing larger than any tensor used below
Q, K, V, O = A, 2 * A, 3 * A, 4 * A
NULL = None


def fwd(L, q=Q, k=K, v=V, o=O, lse=NULL, B=1, h=2, S=64, d=64, scale=0.0, layout=0, dtype=1):
    vp = ctypes.c_void_p
    return L.attn_fwd(vp(q), vp(k), vp(v), vp(o), vp(lse), B, h, S, d, scale, layout, dtype, vp(0))


def test_attn_fwd_validation(L):
    assert fwd(L, q=NULL) == E["NULL"]
    assert fwd(L, o=NULL) == E["NULL"]
    assert fwd(L, layout=2) == E["LAYOUT"]
    assert fwd(L, dtype=7) == E["DTYPE"]
    assert fwd(L, S=0) == E["SHAPE"]            # empty input
    assert fwd(L, B=0) == E["SHAPE"]
    assert fwd(L, h=-1) == E["SHAPE"]
    assert fwd(L, d=96) == E["SHAPE"]           # 16-bit: d in {64, 128}
    assert fwd(L, d=32, dtype=2) == E["SHAPE"]
    assert fwd(L, d=300, dtype=0) == E["SHAPE"]  # fp32: d <= 256
    assert fwd(L, q=Q + 2) == E["ALIGN"]
    assert fwd(L, o=O + 8) == E["ALIGN"]
    assert fwd(L, lse=5 * A + 2) == E["ALIGN"]
    assert fwd(L, o=Q) == E["ALIAS"]             # output may not overlap an input
    assert fwd(L, o=K + 64) == E["ALIAS"]
    assert fwd(L, lse=O + 16) == E["ALIAS"]
    assert fwd(L, B=1 << 20, h=1 << 12, S=1 << 12) == E["SHAPE"]  # beyond 2^40 elements


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a GPU")
def test_valid_call_without_gpu_reports_device_error(L):
    assert fwd(L) == E["DEVICE"]


def test_attn_fwd_ws_validation(L):
    vp = ctypes.c_void_p
    WS = 64 * A

    def fwd_ws(ws=WS, nbytes=1 << 24, dtype=1, o=O, d=64):
        return L.attn_fwd_ws(vp(Q), vp(K), vp(V), vp(o), vp(None), 1, 16, 4096, d, 0.0, 0, dtype, vp(ws),
                             nbytes, vp(0))

    assert fwd_ws(o=None) == E["NULL"]
    assert fwd_ws(d=96) == E["SHAPE"]
    assert fwd_ws(ws=WS + 128) == E["WORKSPACE"]      # not 256-byte aligned
    assert fwd_ws(ws=None, nbytes=64) == E["WORKSPACE"]
    assert fwd_ws(ws=Q) == E["ALIAS"]
    assert fwd_ws(ws=O - 1024) == E["ALIAS"]
    assert L.attn_fwd_ws_bytes(1, 16, 4096, 64, 0) == 0   # fp32: no scratch
    assert L.attn_fwd_ws_bytes(1, 16, 4096, 96, 1) == 0   # unsupported d
    assert L.attn_fwd_ws_bytes(0, 16, 4096, 64, 1) == 0
    if not torch.cuda.is_available():
        assert L.attn_fwd_ws_bytes(1, 16, 4096, 64, 1) == 0  # depends on the device's SM count
        assert fwd_ws() == E["DEVICE"]
        assert fwd_ws(ws=None, nbytes=0) == E["DEVICE"]      # plain attn_fwd


def test_attn_fwd_mixed_validation_and_workspace(L):
    vp = ctypes.c_void_p
    n = 1 * 16 * 4096 * 64
    copies = 3 * ((n * 2 + 255) // 256 * 256)
    need = L.attn_fwd_mixed_workspace_bytes(1, 16, 4096, 64, 1)
    assert need >= copies
    if not torch.cuda.is_available():
        assert need == copies                       # no device: no balancing scratch counted
    assert L.attn_fwd_mixed_workspace_bytes(1, 16, 4096, 64, 0) == 0   # output must be 16-bit
    assert L.attn_fwd_mixed_workspace_bytes(1, 16, 4096, 96, 1) == 0
    WS = 64 * A

    def mixed(q=Q, o=O, ws=WS, nbytes=copies, out=1, d=64, layout=0):
        return L.attn_fwd_mixed(vp(q), vp(K), vp(V), vp(o), vp(None), 1, 16, 4096, d, 0.0, layout, out,
                                vp(ws), nbytes, vp(0))

    assert mixed(q=None) == E["NULL"]
    assert mixed(out=0) == E["DTYPE"]
    assert mixed(d=32) == E["SHAPE"]
    assert mixed(layout=2) == E["LAYOUT"]
    assert mixed(q=Q + 4) == E["ALIGN"]
    assert mixed(o=Q + 1024) == E["ALIAS"]          # the 16-bit output inside the fp32 input
    assert mixed(ws=None) == E["WORKSPACE"]
    assert mixed(nbytes=copies - 256) == E["WORKSPACE"]
    assert mixed(ws=WS + 64) == E["WORKSPACE"]
    assert mixed(ws=K) == E["ALIAS"]
    if not torch.cuda.is_available():
        assert mixed() == E["DEVICE"]


def test_naive_validation_and_workspace(L):
    vp = ctypes.c_void_p
    need = L.attn_fwd_naive_workspace_bytes(1, 16, 4096, 1)
    rows, sp = 16 * 4096, 4096
    assert need == rows * sp * 4 + rows * sp * 2 + 2 * rows * 4
    assert L.attn_fwd_naive_workspace_bytes(1, 1, 5, 1) == 256 + 256 + 2 * 256  # S padded to 8
    assert L.attn_fwd_naive_workspace_bytes(1, 1, 5, 0) == 0                     # fp32 not supported
    WS = 64 * A

    def naive(ws=WS, nbytes=need, dtype=1, S=4096):
        return L.attn_fwd_naive(vp(Q), vp(K), vp(V), vp(O), vp(None), 1, 16, S, 64, 0.0, 0, dtype,
                                vp(ws), nbytes, vp(0))

    assert naive(dtype=0) == E["DTYPE"]
    assert naive(ws=None) == E["WORKSPACE"]
    assert naive(nbytes=need - 1) == E["WORKSPACE"]
    assert naive(ws=WS + 128) == E["WORKSPACE"]
    assert naive(ws=Q) == E["ALIAS"]


def test_qkv_proj_attn_validation_and_workspace(L):
    vp = ctypes.c_void_p
    need = L.qkv_proj_attn_workspace_bytes(8, 512, 768, 1)
    assert need == 8 * 512 * 3 * 768 * 2
    assert L.qkv_proj_attn_workspace_bytes(8, 512, 768, 0) == 0
    WS = 64 * A

    def proj(x=Q, w=K, o=O, B=8, S=512, D=768, h=12, dtype=1, ws=WS, nbytes=need):
        return L.qkv_proj_attn(vp(x), vp(w), vp(o), B, S, D, h, dtype, vp(ws), nbytes, vp(0))

    assert proj(x=None) == E["NULL"]
    assert proj(dtype=0) == E["DTYPE"]
    assert proj(D=770) == E["SHAPE"]      # D % h != 0
    assert proj(h=8) == E["SHAPE"]        # d = 96
    assert proj(S=0) == E["SHAPE"]
    assert proj(x=Q + 4) == E["ALIGN"]
    assert proj(ws=None) == E["WORKSPACE"]
    assert proj(nbytes=need - 2) == E["WORKSPACE"]
    assert proj(o=Q + 1024) == E["ALIAS"]
    assert proj(ws=K) == E["ALIAS"]


def test_qkv_proj_attn_fused_validation(L):
    vp = ctypes.c_void_p

    def fused(x=Q, w=K, o=O, B=8, S=512, D=768, h=12, dtype=1):
        return L.qkv_proj_attn_fused(vp(x), vp(w), vp(o), B, S, D, h, dtype, vp(0))

    assert fused(x=None) == E["NULL"]
    assert fused(dtype=0) == E["DTYPE"]
    assert fused(S=513) == E["SHAPE"]        # one head's K and V must fit in shared memory
    assert fused(h=6) == E["SHAPE"]          # d = 128: not supported by the single kernel
    assert fused(D=770) == E["SHAPE"]
    assert fused(S=0) == E["SHAPE"]
    assert fused(w=K + 8) == E["ALIGN"]
    assert fused(o=Q + 1024) == E["ALIAS"]
    if not torch.cuda.is_available():
        assert fused() == E["DEVICE"]


def test_qkv_proj_attn_noalloc_checks_arguments_before_the_scratch_limit(L):
    """A bad argument is reported as such even on a problem too large for the
    fixed scratch; only a valid problem that is too large gets the limit code."""
    vp = ctypes.c_void_p
    SCRATCH_LIMIT = -10

    def noalloc(x=Q, w=K, o=O, B=8, S=1024, D=768, h=12, dtype=1):
        return L.qkv_proj_attn_noalloc(vp(x), vp(w), vp(o), B, S, D, h, dtype, vp(0))

    assert 8 * 1024 * 3 * 768 * 2 > 32 << 20              # the default problem is over the limit
    assert noalloc() == SCRATCH_LIMIT
    assert noalloc(h=8) == E["SHAPE"]                      # d = 96
    assert noalloc(D=770) == E["SHAPE"]                    # D % h != 0
    assert noalloc(x=None) == E["NULL"]
    assert noalloc(dtype=0) == E["DTYPE"]
    assert noalloc(w=K + 4) == E["ALIGN"]
    assert noalloc(o=Q + 1024) == E["ALIAS"]
    if not torch.cuda.is_available():
        assert noalloc(B=1, S=64) == E["DEVICE"]           # valid and within the limit


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(attn, "_lib", None)
    monkeypatch.setattr(attn, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        attn.lib()
