"""GPU-vs-oracle parity on small shapes (element by element).

Every case compares the CUDA path, called through the C ABI, with the fp64
oracle on the same seeded input bytes.  Shapes span several 128-row tiles,
more than one Q-tile pair per head, ragged tails in both the query and the key
direction, and the degenerate single-key case.
"""

import math

import numpy as np
import pytest
import torch

import head_attention_fwd_gb300 as attn
import oracle
from tests.gpu_common import check_lse, check_o, device_status_ok, gpu_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return gpu_or_skip()


@pytest.fixture(autouse=True)
def streaming_kernel(monkeypatch):
    """This file covers the streaming kernel (flash_fwd.cu) at small sizes, so
    d = 64 problems with S <= 512 are kept off the resident-tile kernel here
    (tests/test_resident_gpu.py covers that one)."""
    monkeypatch.setenv("ATTN_RESIDENT", "never")


@pytest.fixture
def force_split(monkeypatch):
    """Cut the last wave even where the library's cost rule would not (short
    items), so that the cut-and-merge path is covered at small sizes."""
    monkeypatch.setenv("ATTN_SPLIT", "force")


def rand_qkv(B, h, S, d, dtype, layout, seed, qmul=1.0):
    g = torch.Generator().manual_seed(seed)
    shp = (B, h, S, d) if layout == 0 else (B, S, h, d)
    q = (torch.randn(shp, generator=g) * qmul).to(dtype)
    k = torch.randn(shp, generator=g).to(dtype)
    v = torch.randn(shp, generator=g).to(dtype)
    return q, k, v


SHAPES16 = [(1, 1, 1, 64), (1, 2, 128, 64), (2, 3, 300, 64), (1, 1, 513, 64), (1, 2, 257, 128),
            (2, 1, 640, 128), (1, 2, 1000, 64)]


@pytest.mark.parametrize("shape", SHAPES16, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("split", [True, False], ids=["split", "whole"])
def test_flash_matches_oracle(dev, shape, layout, dtype, split, monkeypatch):
    """split: items cut along the key axis over the SMs (forced: at these sizes
    every item is cut into pieces of one or a few key tiles); whole: attn_fwd."""
    if split:
        monkeypatch.setenv("ATTN_SPLIT", "force")
    B, h, S, d = shape
    q, k, v = rand_qkv(B, h, S, d, dtype, layout, seed=hash(shape) % 10000 + layout)
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), layout=layout, want_lse=True, split=split)
    device_status_ok()
    o_ref, lse_ref = oracle.attention(q, k, v, layout=layout, scale=1 / math.sqrt(d))
    check_o(o, o_ref, dtype, f"flash {shape} L{layout}")
    check_lse(lse, lse_ref, f"flash {shape} L{layout}")


# More work items (B·h·ceil(S/256)) than SMs: CTAs run several items in turn,
# and with a scratch the last one to two waves are cut along the key axis.
PERSISTENT = [(1, 80, 512, 64), (2, 41, 300, 64), (1, 77, 640, 128), (1, 160, 256, 128)]


@pytest.mark.parametrize("shape", PERSISTENT, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("split", [True, False], ids=["split", "whole"])
def test_flash_persistent_schedule_matches_oracle(dev, shape, split, monkeypatch):
    if split:
        monkeypatch.setenv("ATTN_SPLIT", "force")
    B, h, S, d = shape
    dtype = torch.bfloat16 if d == 128 else torch.float16
    q, k, v = rand_qkv(B, h, S, d, dtype, 0, seed=h * S + d)
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), want_lse=True, split=split)
    device_status_ok()
    o_ref, lse_ref = oracle.attention(q, k, v, scale=1 / math.sqrt(d))
    check_o(o, o_ref, dtype, f"persistent {shape}")
    check_lse(lse, lse_ref, f"persistent {shape}")


def test_split_and_whole_agree(dev):
    """The cut-and-merge schedule and the whole-item schedule give the same
    result up to fp32 summation order (one 16-bit rounding step apart at most)."""
    q, k, v = (t.to(dev) for t in rand_qkv(1, 16, 4096, 64, torch.float16, 0, seed=7))
    assert attn.attn_fwd_ws_bytes(1, 16, 4096, 64, torch.float16) > 0  # 256 items of 32 key tiles: cut by default
    o1, l1 = attn.attn_fwd(q, k, v, want_lse=True, split=True)
    o2, l2 = attn.attn_fwd(q, k, v, want_lse=True, split=False)
    device_status_ok()
    d = (o1.float() - o2.float()).abs()
    assert d.max().item() <= 2e-3 and d.mean().item() <= 1e-4
    assert (l1 - l2).abs().max().item() <= 1e-4


def test_split_workspace_too_small_is_rejected(dev, force_split):
    import ctypes
    q, k, v = (t.to(dev) for t in rand_qkv(1, 16, 1024, 64, torch.float16, 0, seed=8))
    o = torch.empty_like(q)
    need = attn.attn_fwd_ws_bytes(1, 16, 1024, 64, torch.float16)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    vp = ctypes.c_void_p
    L = attn.lib()
    args = [vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(o.data_ptr()), None, 1, 16, 1024, 64,
            0.0, 0, 1]
    assert L.attn_fwd_ws(*args, vp(ws.data_ptr()), need - 256, vp(0)) == -6
    assert L.attn_fwd_ws(*args, vp(ws.data_ptr() + 128), need - 256, vp(0)) == -6
    assert L.attn_fwd_ws(*args, vp(ws.data_ptr()), need, vp(0)) == 0
    device_status_ok()


def test_split_schedule_replays_in_a_cuda_graph(dev, force_split):
    """A captured split launch replays with a fixed tag; its piece flags are
    cleared inside the graph, so every replay waits for its own pieces."""
    B, h, S, d = 1, 24, 700, 64
    qs, ks, vs = (torch.empty((B, h, S, d), dtype=torch.float16, device=dev) for _ in range(3))
    os_ = torch.empty_like(qs)
    ws = torch.empty(attn.attn_fwd_ws_bytes(B, h, S, d, torch.float16), dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        attn.attn_fwd(qs, ks, vs, os_, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        attn.attn_fwd(qs, ks, vs, os_, workspace=ws)
    for seed in (1, 2, 3):
        q, k, v = rand_qkv(B, h, S, d, torch.float16, 0, seed=100 + seed)
        qs.copy_(q), ks.copy_(k), vs.copy_(v)
        g.replay()
        torch.cuda.synchronize()
        device_status_ok()
        o_eager, _ = attn.attn_fwd(qs, ks, vs, split=True)
        assert torch.equal(os_, o_eager)


@pytest.mark.parametrize("d", [64, 128])
def test_flash_explicit_scale_and_no_lse(dev, d):
    q, k, v = rand_qkv(1, 2, 384, d, torch.float16, 0, seed=11)
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), scale=0.3)
    assert lse is None
    device_status_ok()
    o_ref, _ = oracle.attention(q, k, v, scale=0.3)
    check_o(o, o_ref, torch.float16, "explicit scale")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_flash_peaky_and_growing_scores(dev, dtype, d):
    """Scores whose row maximum keeps growing from tile to tile (every key
    tile forces a rescale of the running output) plus isolated large keys."""
    B, h, S = 1, 2, 1100
    q, k, v = rand_qkv(B, h, S, d, torch.float32, 0, seed=5)
    ramp = torch.linspace(0.2, 3.0, S).view(1, 1, S, 1)
    k = k * ramp
    k[:, :, ::97] *= 6.0
    q = q * 2.0  # with scale 1/sqrt(d), the same spread of scaled scores at either head size
    q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), want_lse=True)
    device_status_ok()
    o_ref, lse_ref = oracle.attention(q, k, v, scale=1 / math.sqrt(d))
    check_o(o, o_ref, dtype, "peaky")
    check_lse(lse, lse_ref, "peaky")


def test_flash_constant_values_are_reproduced(dev):
    """Every probability row sums to 1: V rows all equal to c give O = c."""
    q, k, _ = rand_qkv(1, 2, 700, 128, torch.bfloat16, 1, seed=3)
    c = torch.randn(1, 1, 2, 128).to(torch.bfloat16)
    v = c.expand(1, 700, 2, 128).contiguous()
    o, _ = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), layout=1)
    device_status_ok()
    err = (o.float().cpu() - c.float().expand_as(o)).abs().max().item()
    assert err <= 2e-2


SHAPES32 = [(1, 1, 128, 64), (1, 1, 1, 64), (2, 3, 77, 32), (1, 2, 300, 128), (1, 1, 40, 256),
            (1, 1, 33, 5)]


@pytest.mark.parametrize("shape", SHAPES32, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", [0, 1])
def test_simt_fp32_matches_oracle(dev, shape, layout):
    B, h, S, d = shape
    q, k, v = rand_qkv(B, h, S, d, torch.float32, layout, seed=17 + S)
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), layout=layout, want_lse=True)
    device_status_ok()
    o_ref, lse_ref = oracle.attention(q, k, v, layout=layout, scale=1 / math.sqrt(d))
    check_o(o, o_ref, torch.float32, f"simt {shape}")
    check_lse(lse, lse_ref, f"simt {shape}")


NAIVE_SHAPES = [(1, 2, 128, 64), (2, 2, 300, 64), (1, 1, 203, 128), (1, 1, 1, 64)]


@pytest.mark.parametrize("shape", NAIVE_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_naive_matches_oracle(dev, shape, layout, dtype):
    B, h, S, d = shape
    q, k, v = rand_qkv(B, h, S, d, dtype, layout, seed=23 + S)
    o, lse, ws = attn.attn_fwd_naive(q.to(dev), k.to(dev), v.to(dev), layout=layout, want_lse=True)
    device_status_ok()
    o_ref, lse_ref = oracle.attention(q, k, v, layout=layout, scale=1 / math.sqrt(d))
    check_o(o, o_ref, dtype, f"naive {shape}")
    check_lse(lse, lse_ref, f"naive {shape}")
    # The workspace holds S (fp32) then P: each row of P sums to 1.
    sp = (S + 7) // 8 * 8
    rows = B * h * S
    off = (rows * sp * 4 + 255) // 256 * 256
    P = ws[off:off + rows * sp * 2].view(dtype).view(rows, sp)[:, :S].float()
    assert torch.allclose(P.sum(dim=1), torch.ones(rows, device=P.device), atol=S * 4e-3)


@pytest.mark.parametrize("B,S,D,h", [(2, 200, 128, 2), (1, 300, 256, 2), (2, 64, 768, 12)])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_qkv_proj_attn_matches_oracle(dev, B, S, D, h, dtype):
    g = torch.Generator().manual_seed(B * S + D)
    x = torch.randn((B, S, D), generator=g).to(dtype)
    w = (torch.randn((D, 3 * D), generator=g) * 0.02).to(dtype)
    o, ws = attn.qkv_proj_attn(x.to(dev), w.to(dev), h)
    device_status_ok()
    # projection in the workspace: [B, S, 3D], rounded to the dtype
    proj = ws[: B * S * 3 * D * 2].view(dtype).view(B, S, 3 * D).float().cpu().numpy()
    proj_ref = oracle.qkv_projection(x, w)
    perr = np.abs(proj - proj_ref)
    assert perr.max() <= 2e-2 * max(1.0, np.abs(proj_ref).max()), f"projection max err {perr.max()}"
    o_ref, _ = oracle.qkv_proj_attention(x, w, h)
    check_o(o, o_ref, dtype, f"qkv_proj_attn {B},{S},{D},{h}")


def test_back_to_back_calls_on_one_stream(dev):
    """Consecutive launches on one stream (the bench's pattern) give identical results."""
    q, k, v = (t.to(dev) for t in rand_qkv(1, 4, 777, 64, torch.float16, 0, seed=99))
    o1, _ = attn.attn_fwd(q, k, v)
    outs = [attn.attn_fwd(q, k, v)[0] for _ in range(5)]
    device_status_ok()
    for o in outs:
        assert torch.equal(o, o1)


GROUPED = [(1, 4, 300, 64, 2), (2, 8, 257, 64, 4), (1, 6, 129, 128, 3), (1, 4, 200, 64, 1),
           (1, 4, 200, 128, 4)]


@pytest.mark.parametrize("shape", GROUPED, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_grouped_layout_matches_oracle(dev, shape, dtype):
    """The head-group ("split") layout [B, h/hg, S, hg, d], hg = 1 and hg = h included."""
    B, h, S, d, hg = shape
    g = torch.Generator().manual_seed(h * S + hg)
    q, k, v = (torch.randn((B, h // hg, S, hg, d), generator=g).to(dtype) for _ in range(3))
    o, lse = attn.attn_fwd_grouped(q.to(dev), k.to(dev), v.to(dev), want_lse=True)
    device_status_ok()
    o_ref, lse_ref = oracle.attention_grouped(q, k, v, hg, scale=1 / math.sqrt(d))
    check_o(o, o_ref, dtype, f"grouped {shape}")
    check_lse(lse, lse_ref, f"grouped {shape}")


def test_grouped_layout_rejects_bad_groups(dev):
    import ctypes
    L = attn.lib()
    vp = ctypes.c_void_p
    q = torch.zeros((1, 2, 64, 3, 64), dtype=torch.float32, device=dev)  # large enough for either dtype
    o = torch.empty_like(q)
    p, po = vp(q.data_ptr()), vp(o.data_ptr())
    assert L.attn_fwd_grouped(p, p, p, po, None, 1, 6, 64, 64, 4, 0.0, 1, vp(0)) == -2  # 4 does not divide 6
    assert L.attn_fwd_grouped(p, p, p, po, None, 1, 6, 64, 64, 3, 0.0, 0, vp(0)) == -5  # fp32: not supported


MIXED = [(1, 2, 300, 64), (2, 3, 129, 128), (1, 20, 512, 64)]


@pytest.mark.parametrize("shape", MIXED, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_mixed_fp32_inputs_match_oracle(dev, shape, layout, out_dtype):
    """fp32 Q, K, V -> 16-bit O: against the oracle on the fp32 values, and bit-identical to
    attn_fwd_ws on the inputs rounded to the output type (the conversion rounds to nearest even)."""
    B, h, S, d = shape
    q, k, v = rand_qkv(B, h, S, d, torch.float32, layout, seed=S + d + layout)
    o, lse, ws = attn.attn_fwd_mixed(q.to(dev), k.to(dev), v.to(dev), out_dtype=out_dtype, layout=layout,
                                     want_lse=True)
    device_status_ok()
    assert o.dtype == out_dtype
    o_ref, lse_ref = oracle.attention(q, k, v, layout=layout, scale=1 / math.sqrt(d))
    check_o(o, o_ref, out_dtype, f"mixed {shape}")
    check_lse(lse, lse_ref, f"mixed {shape}")
    o16, lse16 = attn.attn_fwd(q.to(out_dtype).to(dev), k.to(out_dtype).to(dev), v.to(out_dtype).to(dev),
                               layout=layout, want_lse=True)
    device_status_ok()
    assert torch.equal(o, o16) and torch.equal(lse, lse16)
    n = B * h * S * d
    off = (n * 2 + 255) // 256 * 256
    assert torch.equal(ws[:n * 2].view(out_dtype).cpu(), q.to(out_dtype).reshape(-1))
    assert torch.equal(ws[2 * off:2 * off + n * 2].view(out_dtype).cpu(), v.to(out_dtype).reshape(-1))


def test_cut_rule_keeps_short_items_whole(dev):
    """Items of fewer than 16 key tiles are never cut by default (no scratch needed);
    long items that leave a partial wave are."""
    assert attn.attn_fwd_ws_bytes(8, 12, 512, 64, torch.float16) == 0
    assert attn.attn_fwd_ws_bytes(2, 16, 8192, 64, torch.bfloat16) > 0
    assert attn.attn_fwd_ws_bytes(1, 32, 16384, 128, torch.bfloat16) == 0   # d = 128: one item per CTA


def test_grouped_layout_on_a_persistent_grid(dev):
    """More (batch, head, 256-row) items than SMs in the head-group layout: CTAs take
    several items in turn (d = 64) or one each (d = 128)."""
    for d in (64, 128):
        B, h, S, hg = 2, 40, 300, 4          # 2 * 40 * 2 = 160 items
        g = torch.Generator().manual_seed(d)
        dtype = torch.bfloat16
        q, k, v = (torch.randn((B, h // hg, S, hg, d), generator=g).to(dtype) for _ in range(3))
        o, lse = attn.attn_fwd_grouped(q.to(dev), k.to(dev), v.to(dev), want_lse=True)
        device_status_ok()
        o_ref, lse_ref = oracle.attention_grouped(q, k, v, hg, scale=1 / math.sqrt(d))
        check_o(o, o_ref, dtype, f"grouped persistent d{d}")
        check_lse(lse, lse_ref, f"grouped persistent d{d}")


def test_split_launches_on_two_streams_do_not_interfere(dev, force_split):
    """Cut launches running concurrently on two streams, each with its own
    scratch: every result equals the same call made alone."""
    shapes = [(1, 24, 700, 64), (2, 20, 900, 64)]
    inputs, alone = [], []
    for i, (B, h, S, d) in enumerate(shapes):
        q, k, v = (t.to(dev) for t in rand_qkv(B, h, S, d, torch.float16, 0, seed=300 + i))
        inputs.append((q, k, v))
        alone.append(attn.attn_fwd(q, k, v, want_lse=True))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in shapes]
    outs = [[] for _ in shapes]
    for rep in range(4):
        for i, st in enumerate(streams):
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(st):
                q, k, v = inputs[i]
                outs[i].append(attn.attn_fwd(q, k, v, want_lse=True, stream=st))
    torch.cuda.synchronize()
    device_status_ok()
    for i in range(len(shapes)):
        for o, lse in outs[i]:
            assert torch.equal(o, alone[i][0]) and torch.equal(lse, alone[i][1])
