"""The resident-tile attention kernel (fused.cu, attention only), which
attn_fwd uses for d = 64 and S <= 512 when its size rule says it pays: one
CTA per (batch, head) holds the head's Q, K, V in shared memory.  Element-by-element parity with the fp64
oracle (O and LSE) over ragged lengths, both layouts and both 16-bit types,
scores that move the running maximum, and agreement with the streaming kernel
on the same inputs."""

import math

import pytest
import torch

import head_attention_fwd_gb300 as attn
import oracle
from tests.gpu_common import TOL16_MAX, TOL16_MEAN, check_lse, check_o, device_status_ok, gpu_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return gpu_or_skip()


@pytest.fixture(autouse=True)
def resident_kernel(monkeypatch):
    """Every d = 64, S <= 512 call here runs on the resident kernel, whatever
    the size rule would pick for these small head counts."""
    monkeypatch.setenv("ATTN_RESIDENT", "force")


def rand_qkv(B, h, S, layout, dtype, seed, kmul=None):
    g = torch.Generator().manual_seed(seed)
    shp = (B, h, S, 64) if layout == 0 else (B, S, h, 64)
    q, k, v = (torch.randn(shp, generator=g) for _ in range(3))
    if kmul is not None:
        k = k * kmul
    return q.to(dtype), k.to(dtype), v.to(dtype)


# (B, h, S): a single key, ragged tails inside the first and later key tiles,
# exact tiles, an odd number of 128-row blocks, S = 512.
SHAPES = [(1, 1, 1), (1, 2, 37), (2, 3, 128), (1, 2, 200), (2, 1, 256), (1, 3, 384), (2, 2, 511),
          (1, 2, 512), (3, 4, 300)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_resident_matches_oracle(dev, shape, layout, dtype):
    B, h, S = shape
    q, k, v = rand_qkv(B, h, S, layout, dtype, seed=B * 1000 + h * 100 + S + layout)
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), layout=layout, want_lse=True)
    device_status_ok()
    o_ref, lse_ref = oracle.attention(q, k, v, layout=layout, scale=1 / math.sqrt(64))
    check_o(o, o_ref, dtype, f"resident {shape} L{layout}")
    check_lse(lse, lse_ref, f"resident {shape} L{layout}")


@pytest.mark.parametrize("shape", [(2, 3, 300), (1, 4, 512)], ids=lambda s: "x".join(map(str, s)))
def test_resident_agrees_with_streaming_kernel(dev, shape, monkeypatch):
    B, h, S = shape
    q, k, v = (t.to(dev) for t in rand_qkv(B, h, S, 0, torch.float16, seed=S))
    o_r, lse_r = attn.attn_fwd(q, k, v, want_lse=True)
    monkeypatch.setenv("ATTN_RESIDENT", "never")
    o_s, lse_s = attn.attn_fwd(q, k, v, want_lse=True)
    device_status_ok()
    d = (o_r.float() - o_s.float()).abs()
    assert d.max().item() <= TOL16_MAX and d.mean().item() <= TOL16_MEAN
    assert ((lse_r - lse_s).abs() / lse_s.abs().clamp_min(1)).max().item() <= 1e-3


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_resident_peaky_and_growing_scores(dev, dtype):
    """Keys that grow along the sequence and a few 8x rows move the running
    maximum by more than 2^8 after the first key tile (the O rescale path)."""
    B, h, S = 1, 2, 480
    g = torch.Generator().manual_seed(11)
    q = torch.randn((B, h, S, 64), generator=g)
    ramp = torch.linspace(0.2, 3.0, S).view(1, 1, S, 1)
    k = torch.randn((B, h, S, 64), generator=g) * ramp
    k[:, :, 400:405, :] *= 8
    v = torch.randn((B, h, S, 64), generator=g)
    q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), want_lse=True)
    device_status_ok()
    o_ref, lse_ref = oracle.attention(q, k, v, layout=0, scale=1 / 8)
    check_o(o, o_ref, dtype, "resident peaky")
    check_lse(lse, lse_ref, "resident peaky")


def test_resident_explicit_scale_without_lse(dev):
    q, k, v = rand_qkv(2, 2, 333, 1, torch.float16, seed=9)
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), layout=1, scale=0.05)
    device_status_ok()
    assert lse is None
    o_ref, _ = oracle.attention(q, k, v, layout=1, scale=0.05)
    check_o(o, o_ref, torch.float16, "resident scale 0.05")
