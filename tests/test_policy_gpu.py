"""attn_fwd_auto runs the kernel the policy picks, its output matches the fp64
oracle, and the numeric-agreement guard passes on the two kernels' outputs and
catches a planted difference."""

import math

import pytest
import torch

import head_attention_fwd_gb300 as attn
import oracle
from tests.gpu_common import TOL16_MAX, check_o, device_status_ok, gpu_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return gpu_or_skip()


def _qkv(S, dev, dtype=torch.float16, seed=0):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((1, 4, S, 64), generator=g).to(dtype).to(dev) for _ in range(3)]


@pytest.mark.parametrize("opt,S,want", [(True, 2048, attn.ATTN_KERNEL_ONLINE),
                                        (True, 256, attn.ATTN_KERNEL_NAIVE),
                                        (False, 2048, attn.ATTN_KERNEL_NAIVE)])
def test_auto_runs_the_selected_kernel(dev, opt, S, want):
    q, k, v = _qkv(S, dev)
    o, _, kind = attn.attn_fwd_auto(q, k, v, option_enabled=opt)
    device_status_ok()
    assert kind == want
    # the policy's output against the fp64 oracle, element by element
    o_ref, _ = oracle.attention(q.cpu(), k.cpu(), v.cpu(), layout=0, scale=1 / math.sqrt(64))
    check_o(o, o_ref, q.dtype, f"attn_fwd_auto S={S} option={opt}")
    ref = (attn.attn_fwd(q, k, v, split=False)[0] if want == attn.ATTN_KERNEL_ONLINE
           else attn.attn_fwd_naive(q, k, v)[0])
    device_status_ok()
    assert torch.equal(o, ref)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_guard_accepts_online_vs_naive_and_catches_a_difference(dev, dtype):
    q, k, v = _qkv(1500, dev, dtype, seed=3)
    o_online = attn.attn_fwd(q, k, v)[0]
    o_naive = attn.attn_fwd_naive(q, k, v)[0]
    device_status_ok()
    rc, mx = attn.attn_compare(o_naive, o_online, TOL16_MAX)
    assert rc == 0 and mx <= TOL16_MAX
    assert mx == pytest.approx((o_naive.float() - o_online.float()).abs().max().item(), rel=1e-6)
    attn.assert_numerically_equal(o_naive, o_online, atol=TOL16_MAX)
    bad = o_online.clone()
    bad[0, 2, 777, 5] += 0.5
    with pytest.raises(AssertionError):
        attn.assert_numerically_equal(o_naive, bad, atol=TOL16_MAX)
    bad[0, 1, 3, 3] = float("nan")
    rc, mx = attn.attn_compare(o_online, bad, 10.0)
    assert rc == attn.ATTN_E_MISMATCH and mx == float("inf")
