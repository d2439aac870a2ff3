"""qkv_proj_attn_noalloc, the entry point for callers that cannot allocate
device memory at the point where they run attention (a plugin handed only its
input and output buffers, a framework whose pool must account for every byte,
a loop that cannot take an allocation's implicit synchronisation).  It keeps
the projection in the library's fixed static scratch instead of a caller
workspace.

This file sorts last so that a run stopping at the first failure has already
run every other test.  It also passes alone in a fresh process.
"""

import ctypes

import pytest
import torch

import head_attention_fwd_gb300 as attn
from tests.gpu_common import TOL16_MAX, TOL16_MEAN, device_status_ok, gpu_or_skip

pytestmark = pytest.mark.gpu

ATTN_E_SCRATCH_LIMIT = -10
SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def dev():
    return gpu_or_skip()


def _inputs(B, S, D, dtype, seed, dev):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((B, S, D), generator=g).to(dtype).to(dev)
    w = (torch.randn((D, 3 * D), generator=g) * 0.02).to(dtype).to(dev)
    return x, w


def _noalloc_c_call(x, w, o, h):
    """The C entry point itself, called through ctypes with raw pointers."""
    B, S, D = (int(n) for n in x.shape)
    vp = ctypes.c_void_p
    stream = vp(torch.cuda.current_stream().cuda_stream)
    return attn.lib().qkv_proj_attn_noalloc(vp(x.data_ptr()), vp(w.data_ptr()), vp(o.data_ptr()), B, S,
                                            D, h, attn.dtype_code(x.dtype), stream)


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(dev):
    cases = [(8, 512, 768, 12, torch.float16, 1),   # BERT-base shape, 18.9 MB of scratch
             (2, 300, 256, 2, torch.bfloat16, 2)]   # a smaller, ragged second call
    refs, outs, inputs = [], [], []
    for B, S, D, h, dtype, seed in cases:
        x, w = _inputs(B, S, D, dtype, seed, dev)
        o_ref, _ = attn.qkv_proj_attn(x, w, h)        # existing entry point, caller workspace
        refs.append(o_ref)
        inputs.append((x, w, h))
        outs.append(torch.empty_like(o_ref))
    device_status_ok()
    for (x, w, h), o in zip(inputs, outs):            # two no-alloc calls back to back
        assert _noalloc_c_call(x, w, o, h) == 0
    device_status_ok()
    for o, o_ref in zip(outs, refs):
        err = (o.float() - o_ref.float()).abs()
        assert err.max().item() <= TOL16_MAX and err.mean().item() <= TOL16_MEAN


def test_noalloc_rejects_problems_beyond_its_scratch(dev):
    B, S, D, h = 8, 1024, 768, 12                    # needs 37.7 MB > 32 MiB
    assert B * S * 3 * D * 2 > SCRATCH_BYTES
    x, w = _inputs(B, S, D, torch.float16, 3, dev)
    o = torch.zeros((B, S, h, D // h), dtype=torch.float16, device=dev)
    assert _noalloc_c_call(x, w, o, h) == ATTN_E_SCRATCH_LIMIT
    assert "scratch" in attn.attn_status_string(ATTN_E_SCRATCH_LIMIT)
    device_status_ok()
    assert torch.count_nonzero(o).item() == 0        # nothing was launched
