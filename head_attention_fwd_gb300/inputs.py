"""Seeded synthetic inputs for the attention forward.

This module only draws random numbers and lays them out; it holds none of
the attention arithmetic, so that the CUDA path and the fp64 oracle can both
be fed the exact same bytes from it.

Workloads (what they are, with their sizes):

* ``single_head_f32``   B=1 h=1 S=128 d=64, fp32, [B,h,S,d]
* ``mha_f16_s4096``     B=1 h=16 S=4096 d=64 (D=1024), fp16, [B,h,S,d]
                        (the shape of the memory table in "Transformer算子生态深度分析" ch.2 §2.5)
* ``bert_base_qkv``     X [8,512,768] fp16 ~ N(0,1), W_qkv [768,2304] fp16 ~ N(0,0.02^2),
                        h=12 d=64, output [B,S,h,d] (BERT-base shape, same chapter §2.1)
* ``long_seq_bf16_peaky``  B=2 h=16 S=8192 d=64, bf16, [B,h,S,d], 1% of K rows x8
* ``wide_head_bf16_bshd``  B=1 h=32 S=16384 d=128, bf16, [B,S,h,d], with LSE

All values are drawn in fp32 from a seeded ``torch.Generator`` (N(0,1), or
N(0, 0.02^2) for the projection weight) and then rounded to the workload's
dtype; the seed of each workload is fixed below.  For the peaky workload,
floor(0.01 * B*h*S) (b, h, s) key rows are chosen by a seeded permutation
and multiplied by 8 after rounding (exact in bf16).  Synthetic weights stand
in for trained ones; no dataset is involved.
"""

from __future__ import annotations

import dataclasses
import math

import torch

LAYOUT_BHSD = 0  # contiguous [B, h, S, d]
LAYOUT_BSHD = 1  # head-interleaved [B, S, h, d]

_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    h: int
    S: int
    d: int
    dtype: str  # "f32" | "f16" | "bf16"
    layout: int  # LAYOUT_BHSD | LAYOUT_BSHD
    seed: int
    peaky_frac: float = 0.0  # fraction of K rows multiplied by peaky_mult
    peaky_mult: float = 8.0
    qkv_proj: bool = False  # inputs are X [B,S,D] and W_qkv [D,3D] instead of Q, K, V
    w_std: float = 0.02
    want_lse: bool = False

    @property
    def D(self) -> int:
        return self.h * self.d

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return _DTYPES[self.dtype]

    @property
    def attn_flops(self) -> int:
        """4·B·h·S²·d: two S×S×d products per head."""
        return 4 * self.B * self.h * self.S * self.S * self.d

    @property
    def proj_flops(self) -> int:
        return 2 * self.B * self.S * self.D * 3 * self.D if self.qkv_proj else 0

    def shape(self) -> tuple[int, int, int, int]:
        if self.layout == LAYOUT_BHSD:
            return (self.B, self.h, self.S, self.d)
        return (self.B, self.S, self.h, self.d)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("single_head_f32", 1, 1, 128, 64, "f32", LAYOUT_BHSD, seed=1001),
        Workload("mha_f16_s4096", 1, 16, 4096, 64, "f16", LAYOUT_BHSD, seed=1002),
        Workload("bert_base_qkv", 8, 12, 512, 64, "f16", LAYOUT_BSHD, seed=1003, qkv_proj=True),
        Workload("long_seq_bf16_peaky", 2, 16, 8192, 64, "bf16", LAYOUT_BHSD, seed=1004,
                 peaky_frac=0.01),
        Workload("wide_head_bf16_bshd", 1, 32, 16384, 128, "bf16", LAYOUT_BSHD, seed=1005,
                 want_lse=True),
    ]
}


def make_qkv(w: Workload, device: str | torch.device = "cpu", seed: int | None = None):
    """Seeded (q, k, v) in the workload's dtype and layout.

    Drawn on the host in fp32 (so the bytes do not depend on the device),
    rounded to the dtype, then moved to ``device``.
    """
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    shp = w.shape()
    q = torch.randn(shp, generator=g, dtype=torch.float32).to(w.torch_dtype)
    k = torch.randn(shp, generator=g, dtype=torch.float32).to(w.torch_dtype)
    v = torch.randn(shp, generator=g, dtype=torch.float32).to(w.torch_dtype)
    if w.peaky_frac > 0:
        nrows = int(math.floor(w.peaky_frac * w.B * w.h * w.S))
        pick = torch.randperm(w.B * w.h * w.S, generator=g)[:nrows]
        b = pick // (w.h * w.S)
        hh = (pick // w.S) % w.h
        s = pick % w.S
        if w.layout == LAYOUT_BHSD:
            k[b, hh, s, :] *= w.peaky_mult
        else:
            k[b, s, hh, :] *= w.peaky_mult
    return q.to(device), k.to(device), v.to(device)


def make_proj_inputs(w: Workload, device: str | torch.device = "cpu", seed: int | None = None):
    """Seeded (x [B,S,D], w_qkv [D,3D]) for the fused-projection workload."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    x = torch.randn((w.B, w.S, w.D), generator=g, dtype=torch.float32).to(w.torch_dtype)
    wq = (torch.randn((w.D, 3 * w.D), generator=g, dtype=torch.float32) * w.w_std).to(w.torch_dtype)
    return x.to(device), wq.to(device)


def sample_rows(w: Workload, n: int, seed: int = 7) -> torch.Tensor:
    """n distinct flat query-row indices (b*h + head)*S + i, always including
    the first and the last row of the problem (tile edges and the ragged tail)."""
    total = w.B * w.h * w.S
    g = torch.Generator().manual_seed(seed)
    n = min(n, total)
    rows = torch.randperm(total, generator=g)[:n]
    rows[0] = 0
    if n > 1:
        rows[1] = total - 1
    return torch.unique(rows)
