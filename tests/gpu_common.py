"""Helpers shared by the GPU test files: tolerances and comparisons.

Tolerances (fixed for this method): fp32 path max|dO| <= 1e-4; 16-bit inputs
with fp32 accumulation max|dO| <= 2e-2 and mean|dO| <= 2e-3; LSE relative error
<= 1e-3, taken against max(|LSE|, 1) so that a log-sum-exp near zero (a single
key with a score near 0) does not turn rounding into a large relative error.
"""

import numpy as np
import pytest
import torch

TOL16_MAX, TOL16_MEAN = 2e-2, 2e-3
TOL32_MAX = 1e-4
LSE_REL = 1e-3


def gpu_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from head_attention_fwd_gb300 import _build
    _build.build()
    return torch.device("cuda:0")


def check_o(o_gpu, o_ref, dtype, what=""):
    o = o_gpu.detach().float().cpu().numpy().astype(np.float64)
    err = np.abs(o - o_ref)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    if dtype == torch.float32:
        assert err.max() <= TOL32_MAX, f"{what}: max|dO| {err.max():.3e} > {TOL32_MAX}"
    else:
        assert err.max() <= TOL16_MAX, f"{what}: max|dO| {err.max():.3e} > {TOL16_MAX}"
        assert err.mean() <= TOL16_MEAN, f"{what}: mean|dO| {err.mean():.3e} > {TOL16_MEAN}"
    return err.max(), err.mean()


def check_lse(lse_gpu, lse_ref, what=""):
    lse = lse_gpu.detach().cpu().numpy().astype(np.float64)
    rel = np.abs(lse - lse_ref) / np.maximum(np.abs(lse_ref), 1.0)
    assert rel.max() <= LSE_REL, f"{what}: LSE rel err {rel.max():.3e} > {LSE_REL}"
    return rel.max()


def device_status_ok():
    import head_attention_fwd_gb300 as attn
    rc, detail = attn.attn_get_device_status()
    assert rc == 0, f"device status {rc} ({attn.attn_status_string(rc)}), detail {detail:#x}"


def gather_rows(o, rows, B, h, S, layout):
    """GPU output rows at flat indices (b*h + head)*S + i -> [len(rows), d] on the host."""
    rows = torch.as_tensor(rows, dtype=torch.long)
    b, hh, i = rows // (h * S), (rows // S) % h, rows % S
    idx = (b.to(o.device), hh.to(o.device), i.to(o.device))
    sel = o[idx[0], idx[1], idx[2]] if layout == 0 else o[idx[0], idx[2], idx[1]]
    return sel.float().cpu().numpy().astype(np.float64)
