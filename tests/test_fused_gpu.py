"""qkv_proj_attn_fused -- the QKV projection and the attention in one kernel
("Transformer算子生态深度分析" §2.7) -- against the fp64 oracle, element by
element: the BERT-base shape in full, and small shapes with ragged sequence
lengths, one or several heads, fp16 and bf16.  Also checked against the
two-launch qkv_proj_attn on the same inputs."""

import pytest
import torch

import head_attention_fwd_gb300 as attn
import oracle
from head_attention_fwd_gb300.inputs import WORKLOADS, make_proj_inputs
from tests.gpu_common import TOL16_MAX, TOL16_MEAN, check_o, device_status_ok, gpu_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return gpu_or_skip()


def _inputs(B, S, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((B, S, D), generator=g).to(dtype)
    w = (torch.randn((D, 3 * D), generator=g) * 0.02).to(dtype)
    return x, w


# (B, S, D, h): one key tile, exact tiles, ragged tails, an odd number of
# query blocks (the second block of the last pair is empty), S = 512.
SHAPES = [(1, 1, 64, 1), (2, 128, 128, 2), (1, 300, 256, 4), (2, 512, 192, 3), (1, 257, 64, 1),
          (3, 384, 128, 2), (1, 77, 320, 5)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_fused_matches_oracle(dev, shape, dtype):
    B, S, D, h = shape
    x, w = _inputs(B, S, D, dtype, seed=sum(shape) + (dtype == torch.bfloat16))
    o = attn.qkv_proj_attn_fused(x.to(dev), w.to(dev), h)
    device_status_ok()
    o_ref, _ = oracle.qkv_proj_attention(x, w, h)
    check_o(o, o_ref, dtype, f"fused {shape}")
    o2, _ = attn.qkv_proj_attn(x.to(dev), w.to(dev), h)     # the two-launch path on the same inputs
    device_status_ok()
    d = (o.float() - o2.float()).abs()
    assert d.max().item() <= TOL16_MAX and d.mean().item() <= TOL16_MEAN


def test_fused_bert_base_full(dev):
    wl = WORKLOADS["bert_base_qkv"]
    x, w = make_proj_inputs(wl)
    o = attn.qkv_proj_attn_fused(x.to(dev), w.to(dev), wl.h)
    device_status_ok()
    o_ref, _ = oracle.qkv_proj_attention(x, w, wl.h)
    check_o(o, o_ref, wl.torch_dtype, wl.name + " fused")
    # repeated calls give identical bytes (no state carried between launches)
    o_again = attn.qkv_proj_attn_fused(x.to(dev), w.to(dev), wl.h)
    device_status_ok()
    assert torch.equal(o, o_again)


def test_fused_rejects_unsupported_sizes(dev):
    x, w = _inputs(1, 513, 128, torch.float16, 5)
    with pytest.raises(attn.AttnError, match="ATTN_E_SHAPE"):
        attn.qkv_proj_attn_fused(x.to(dev), w.to(dev), 2)      # S > 512
    x, w = _inputs(1, 64, 256, torch.float16, 6)
    with pytest.raises(attn.AttnError, match="ATTN_E_SHAPE"):
        attn.qkv_proj_attn_fused(x.to(dev), w.to(dev), 2)      # d = 128
