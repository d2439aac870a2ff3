"""The naive/online selection policy (host logic, no GPU): the cases the
online-softmax proposal page tests (§七), the threshold of its §六, and the
library's own edges."""

import os

import pytest

import head_attention_fwd_gb300 as attn
from head_attention_fwd_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def _golden_cases():
    out = []
    with open(os.path.join(ROOT, "tests", "golden", "p2_policy_cases.txt")) as f:
        for line in f:
            if line.startswith("case:"):
                opt, n, kind = line.split(":")[1].split()
                out.append((bool(int(opt)), int(n), kind))
    return out


@pytest.mark.parametrize("opt,n,kind", _golden_cases())
def test_page_cases(opt, n, kind):
    want = attn.ATTN_KERNEL_ONLINE if kind == "online" else attn.ATTN_KERNEL_NAIVE
    assert attn.select_kernel(opt, n) == want


def test_threshold_is_strict_and_configurable():
    assert attn.select_kernel(True, 1024) == attn.ATTN_KERNEL_NAIVE
    assert attn.select_kernel(True, 1025) == attn.ATTN_KERNEL_ONLINE
    assert attn.select_kernel(True, 300, threshold=256) == attn.ATTN_KERNEL_ONLINE
    assert attn.select_kernel(False, 10**6, threshold=1) == attn.ATTN_KERNEL_NAIVE
    assert attn.select_kernel(True, 2048, threshold=-1) == attn.ATTN_KERNEL_ONLINE  # default 1024


def test_compare_validates_before_any_cuda_call():
    import ctypes
    L = attn.lib()
    vp = ctypes.c_void_p
    assert L.attn_compare(vp(None), vp(16), 4, 1, 1e-3, None, vp(0)) == -1
    assert L.attn_compare(vp(16), vp(32), 4, 9, 1e-3, None, vp(0)) == -5
    assert L.attn_compare(vp(16), vp(32), -1, 1, 1e-3, None, vp(0)) == -2
