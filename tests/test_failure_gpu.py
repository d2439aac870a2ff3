"""Failure reporting on the GPU, without a GPU fault: a pipeline wait that
can never complete gives up after its limit, the kernel records the stall in
the device status word and returns, and the context stays usable."""

import math

import pytest
import torch

import head_attention_fwd_gb300 as attn
import oracle
from tests.gpu_common import check_o, device_status_ok, gpu_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return gpu_or_skip()


def test_stalled_wait_reports_timeout_and_context_survives(dev):
    device_status_ok()  # start clean
    attn.attn_selftest_wait_timeout(2_000_000)  # about a millisecond of SM clock
    rc, detail = attn.attn_get_device_status()
    assert rc == attn.ATTN_E_TIMEOUT
    assert detail >> 24 == 15 and (detail >> 16) & 0xFF == 1
    # the status word was cleared by the read and the context still works
    device_status_ok()
    g = torch.Generator().manual_seed(4)
    q, k, v = (torch.randn((1, 2, 200, 64), generator=g).to(torch.float16) for _ in range(3))
    o, _ = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev))
    device_status_ok()
    o_ref, _ = oracle.attention(q, k, v, scale=1 / math.sqrt(64))
    check_o(o, o_ref, torch.float16, "after timeout")


def test_sticky_status_makes_later_kernels_skip(dev):
    """While a stall is recorded and not yet read, attention kernels do no work
    (they see the status word and return), so a failure is never hidden."""
    g = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn((1, 1, 256, 64), generator=g).to(torch.float16).to(dev) for _ in range(3))
    o = torch.zeros_like(q)
    attn.attn_selftest_wait_timeout(1_000_000)
    attn.attn_fwd(q, k, v, o)
    rc, _ = attn.attn_get_device_status()
    assert rc == attn.ATTN_E_TIMEOUT
    assert torch.count_nonzero(o).item() == 0
    attn.attn_fwd(q, k, v, o)
    device_status_ok()
    assert torch.count_nonzero(o).item() > 0


def test_selftest_rejects_bad_limits(dev):
    for bad in (0, -5, 10**11):
        with pytest.raises(attn.AttnError):
            attn.attn_selftest_wait_timeout(bad)
