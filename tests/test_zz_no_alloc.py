"""qkv_proj_attn_noalloc, the entry point for callers that cannot allocate
device memory at the point where they run attention (a plugin handed only its
input and output buffers, a framework whose pool must account for every byte,
a loop that cannot take an allocation's implicit synchronisation).  It keeps
the projection in the library's fixed static scratch instead of a caller
workspace.

Checked here: its output against the fp64 oracle and against the workspace
entry point on two calls in a row; that a call, once the first one on the
device has run, changes neither torch's allocation count nor the device's free
memory; the Python wrapper; and the size limit.

This file sorts last so that a run stopping at the first failure has already
run every other test.  It also passes alone in a fresh process.
"""

import ctypes

import pytest
import torch

import head_attention_fwd_gb300 as attn
import oracle
from tests.gpu_common import TOL16_MAX, TOL16_MEAN, check_o, device_status_ok, gpu_or_skip

pytestmark = pytest.mark.gpu

ATTN_E_SCRATCH_LIMIT = -10
SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def dev():
    return gpu_or_skip()


def _inputs(B, S, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((B, S, D), generator=g).to(dtype)
    w = (torch.randn((D, 3 * D), generator=g) * 0.02).to(dtype)
    return x, w


def _noalloc_c_call(x, w, o, h):
    """The C entry point itself, called through ctypes with raw pointers."""
    B, S, D = (int(n) for n in x.shape)
    vp = ctypes.c_void_p
    stream = vp(torch.cuda.current_stream().cuda_stream)
    return attn.lib().qkv_proj_attn_noalloc(vp(x.data_ptr()), vp(w.data_ptr()), vp(o.data_ptr()), B, S,
                                            D, h, attn.dtype_code(x.dtype), stream)


CASES = [(8, 512, 768, 12, torch.float16, 1),   # BERT-base shape, 18.9 MB of scratch
         (2, 300, 256, 2, torch.bfloat16, 2)]   # a smaller, ragged second call


def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls_in_a_row(dev):
    host, refs, outs, inputs = [], [], [], []
    for B, S, D, h, dtype, seed in CASES:
        x, w = _inputs(B, S, D, dtype, seed)
        host.append((x, w, h))
        xd, wd = x.to(dev), w.to(dev)
        o_ref, _ = attn.qkv_proj_attn(xd, wd, h)      # existing entry point, caller workspace
        refs.append(o_ref)
        inputs.append((xd, wd, h))
        outs.append(torch.empty_like(o_ref))
    device_status_ok()
    for (x, w, h), o in zip(inputs, outs):            # two no-alloc calls back to back
        assert _noalloc_c_call(x, w, o, h) == 0
    device_status_ok()
    for (x, w, h), o, o_ref in zip(host, outs, refs):
        err = (o.float() - o_ref.float()).abs()
        assert err.max().item() <= TOL16_MAX and err.mean().item() <= TOL16_MEAN
        o_oracle, _ = oracle.qkv_proj_attention(x, w, h)
        check_o(o, o_oracle, x.dtype, f"qkv_proj_attn_noalloc {tuple(x.shape)}")


def test_noalloc_call_leaves_device_memory_unchanged(dev):
    B, S, D, h, dtype, seed = CASES[0]
    x, w = (t.to(dev) for t in _inputs(B, S, D, dtype, seed))
    o = torch.empty((B, S, h, D // h), dtype=dtype, device=dev)
    assert _noalloc_c_call(x, w, o, h) == 0          # the first call on the device may load the module
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        assert _noalloc_c_call(x, w, o, h) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0, (free0, free1)
    device_status_ok()


def test_noalloc_python_wrapper(dev):
    B, S, D, h, dtype, seed = CASES[1]
    x, w = _inputs(B, S, D, dtype, seed)
    o = attn.qkv_proj_attn_noalloc(x.to(dev), w.to(dev), h)
    device_status_ok()
    assert o.shape == (B, S, h, D // h) and o.dtype == dtype
    o_oracle, _ = oracle.qkv_proj_attention(x, w, h)
    check_o(o, o_oracle, dtype, "qkv_proj_attn_noalloc wrapper")


def test_noalloc_rejects_problems_beyond_its_scratch(dev):
    B, S, D, h = 8, 1024, 768, 12                    # needs 37.7 MB > 32 MiB
    assert B * S * 3 * D * 2 > SCRATCH_BYTES
    x, w = (t.to(dev) for t in _inputs(B, S, D, torch.float16, 3))
    o = torch.zeros((B, S, h, D // h), dtype=torch.float16, device=dev)
    assert _noalloc_c_call(x, w, o, h) == ATTN_E_SCRATCH_LIMIT
    assert "scratch" in attn.attn_status_string(ATTN_E_SCRATCH_LIMIT)
    device_status_ok()
    assert torch.count_nonzero(o).item() == 0        # nothing was launched
