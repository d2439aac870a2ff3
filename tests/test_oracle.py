"""Pins for the fp64 oracle (CPU only).

Each test ties an oracle function to something other than the oracle itself:
the worked score vector printed on the online-softmax proposal page, library
routines (scipy.special.softmax / logsumexp, numpy matmul, numpy / torch dtype
conversions), closed forms and invariants of the definition, and a brute-force
direct summation on tiny inputs.  They are chosen so that a plausible slip in
the oracle -- a dropped scale, a transposed or mismatched index, a wrong sign in
the merge rule, a missing rescale, a layout mix-up -- fails at least one.
"""

import math

import numpy as np
import pytest
import scipy.special as sps
import torch

import oracle
from tests.conftest import load_golden

RNG = np.random.default_rng(20261202)


# --------------------------------------------------------------- decoders ----
def test_decode_f16_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.decode(bits.view(np.float16))
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_decode_bf16_every_bit_pattern():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    t = bits.view(torch.bfloat16)
    ref = t.to(torch.float64).numpy()
    got = oracle.decode(t)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_decode_f32():
    x = RNG.standard_normal(1000).astype(np.float32) * 1e3
    np.testing.assert_array_equal(oracle.decode(x), x.astype(np.float64))


# ------------------------------------------------- the pages' worked vector ----
def _worked():
    g = load_golden("p2_worked_scores.txt")
    return np.array([float(x) for x in g["scores"]]), float(g["atol"][0])


def test_worked_vector_three_step_matches_library():
    s, _ = _worked()
    p, m, d = oracle.softmax(s)
    np.testing.assert_allclose(p, sps.softmax(s), rtol=0, atol=1e-15)
    assert m == 3.0
    # d = sum exp(s - m) = exp(logsumexp(s) - m)
    assert d == pytest.approx(math.exp(sps.logsumexp(s) - 3.0), rel=1e-15)


@pytest.mark.parametrize("block", [1, 2, 3, 4, 7])
def test_worked_vector_online_matches_naive(block):
    """The page's claim: online and naive agree (its tolerance 1e-3); in fp64
    they agree to rounding."""
    s, atol = _worked()
    p_naive, m_naive, d_naive = oracle.softmax(s)
    p_on, m_on, d_on, _, _ = oracle.online_softmax(s, block)
    assert np.max(np.abs(p_on - p_naive)) <= atol
    np.testing.assert_allclose(p_on, p_naive, rtol=0, atol=1e-15)
    assert m_on == m_naive
    assert d_on == pytest.approx(d_naive, rel=1e-15)


def test_worked_vector_running_statistics():
    """Per-element recurrence: after element t the running max is the prefix
    max and the running sum is sum_{i<=t} exp(s_i - m_t) = exp(lse(prefix) - m_t)."""
    s, _ = _worked()
    _, _, _, mt, dt = oracle.online_softmax(s, 1)
    np.testing.assert_array_equal(mt, np.maximum.accumulate(s))
    for t in range(s.size):
        want = math.exp(sps.logsumexp(s[: t + 1]) - mt[t])
        assert dt[t] == pytest.approx(want, rel=1e-15)
    # block merge of {1, 2} and {0.5, 3}: per-block (m, d) then merged
    _, _, _, mt2, dt2 = oracle.online_softmax(s, 2)
    assert mt2[0] == 2.0 and dt2[0] == pytest.approx(1 + math.exp(-1), rel=1e-15)
    assert mt2[1] == 3.0 and dt2[1] == pytest.approx(dt[-1], rel=1e-15)


@pytest.mark.parametrize("n,block,mag", [(1, 1, 1.0), (37, 5, 1.0), (1000, 128, 30.0),
                                         (513, 64, 700.0), (64, 64, 1e4)])
def test_online_random_vectors(n, block, mag):
    s = RNG.standard_normal(n) * mag
    p_on, m, d, _, _ = oracle.online_softmax(s, block)
    ref = sps.softmax(s)
    assert np.all(np.isfinite(p_on))
    np.testing.assert_allclose(p_on, ref, rtol=1e-12, atol=1e-300)
    assert m + math.log(d) == pytest.approx(sps.logsumexp(s), rel=1e-13, abs=1e-13)


def test_softmax_shift_invariance():
    s = RNG.standard_normal(50)
    p0, m0, d0 = oracle.softmax(s)
    p1, m1, d1 = oracle.softmax(s + 123.25)
    np.testing.assert_allclose(p1, p0, rtol=1e-13)
    assert m1 == pytest.approx(m0 + 123.25) and d1 == pytest.approx(d0, rel=1e-13)
    assert abs(p0.sum() - 1.0) < 1e-15 * 50


# ------------------------------------------------------------ attention ----
def _lib_attention(q, k, v, scale):
    """Reference from library routines: numpy matmul + scipy softmax/logsumexp, [B,H,S,d]."""
    s = np.einsum("bhid,bhjd->bhij", q, k) * scale
    return sps.softmax(s, axis=-1) @ v, sps.logsumexp(s, axis=-1)


@pytest.mark.parametrize("B,H,S,d", [(1, 1, 1, 4), (2, 3, 5, 8), (1, 2, 17, 16), (2, 1, 64, 64)])
def test_attention_matches_library(B, H, S, d):
    q, k, v = (RNG.standard_normal((B, H, S, d)) for _ in range(3))
    scale = 1 / math.sqrt(d)
    o, lse = oracle.attention(q, k, v, layout=0, scale=scale)
    o_ref, lse_ref = _lib_attention(q, k, v, scale)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-13, atol=1e-13)


def _brute(q, k, v, scale):
    """Direct summation for one head: O_i = sum_j e^{s_ij} v_j / sum_j e^{s_ij} (no max trick)."""
    S, d = len(q), len(q[0])
    out = []
    for i in range(S):
        w = [math.exp(scale * sum(q[i][e] * k[j][e] for e in range(d))) for j in range(S)]
        tot = sum(w)
        out.append([sum(w[j] * v[j][e] for j in range(S)) / tot for e in range(d)])
    return out


@pytest.mark.parametrize("S,d", [(1, 1), (2, 3), (5, 4), (8, 8)])
def test_attention_bruteforce_tiny(S, d):
    q, k, v = (RNG.standard_normal((1, 1, S, d)) for _ in range(3))
    o, _ = oracle.attention(q, k, v, scale=0.7)
    ref = np.array(_brute(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), 0.7))
    np.testing.assert_allclose(o[0, 0], ref, rtol=1e-12, atol=1e-12)


def test_constant_value_rows_returned_unchanged():
    """Every probability row sums to 1, so V rows all equal to c give O_i = c."""
    B, H, S, d = 2, 2, 33, 8
    q, k = (RNG.standard_normal((B, H, S, d)) * 3 for _ in range(2))
    c = RNG.standard_normal((B, H, 1, d))
    v = np.broadcast_to(c, (B, H, S, d)).copy()
    o, _ = oracle.attention(q, k, v)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=1e-13, atol=1e-14)


def test_zero_query_gives_column_mean():
    B, H, S, d = 1, 3, 29, 8
    k, v = (RNG.standard_normal((B, H, S, d)) for _ in range(2))
    o, lse = oracle.attention(np.zeros((B, H, S, d)), k, v)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape),
                               rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(S), rtol=1e-14)


def test_single_key_returns_value():
    q, k, v = (RNG.standard_normal((2, 2, 1, 16)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, scale=0.25)
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(lse, 0.25 * np.sum(q * k, axis=-1), rtol=1e-14)


def test_identical_keys_give_value_mean():
    B, H, S, d = 1, 2, 20, 8
    q, v = (RNG.standard_normal((B, H, S, d)) for _ in range(2))
    k = np.broadcast_to(RNG.standard_normal((B, H, 1, d)), (B, H, S, d)).copy()
    o, _ = oracle.attention(q, k, v)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape),
                               rtol=1e-12, atol=1e-14)


def test_joint_key_value_permutation_invariance():
    B, H, S, d = 2, 2, 40, 8
    q, k, v = (RNG.standard_normal((B, H, S, d)) for _ in range(3))
    perm = RNG.permutation(S)
    o0, l0 = oracle.attention(q, k, v)
    o1, l1 = oracle.attention(q, k[:, :, perm], v[:, :, perm])
    np.testing.assert_allclose(o1, o0, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l0, rtol=1e-13)
    o2, _ = oracle.attention(q, k, v[:, :, perm])  # V alone permuted: must change
    assert np.max(np.abs(o2 - o0)) > 1e-3


def test_per_row_score_shift_via_appended_column():
    """Q' = [Q | c_i/scale], K' = [K | 1] adds c_i to every score of row i:
    O is unchanged and LSE moves by exactly c_i (max-subtraction argument,
    "Transformer算子生态深度分析" ch.2 §2.3)."""
    B, H, S, d = 1, 2, 31, 7
    scale = 0.4
    q, k, v = (RNG.standard_normal((B, H, S, d)) for _ in range(3))
    c = RNG.standard_normal((B, H, S)) * 50
    q2 = np.concatenate([q, (c / scale)[..., None]], axis=-1)
    k2 = np.concatenate([k, np.ones((B, H, S, 1))], axis=-1)
    v2 = np.concatenate([v, np.zeros((B, H, S, 1))], axis=-1)
    o0, l0 = oracle.attention(q, k, v, scale=scale)
    o1, l1 = oracle.attention(q2, k2, v2, scale=scale)
    np.testing.assert_allclose(o1[..., :d], o0, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(l1, l0 + c, rtol=1e-12, atol=1e-10)


def test_scale_is_applied_to_the_dot_product():
    q, k, v = (RNG.standard_normal((1, 1, 9, 4)) for _ in range(3))
    for scale in (0.5, 1.0, 2.0):
        o, lse = oracle.attention(q, k, v, scale=scale)
        o_ref, lse_ref = _lib_attention(q, k, v, scale)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-13)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    o_def, _ = oracle.attention(q, k, v)  # default scale = 1/sqrt(d) = 0.5
    np.testing.assert_allclose(o_def, oracle.attention(q, k, v, scale=0.5)[0], rtol=0, atol=0)


def test_head_interleaved_layout_is_a_transpose():
    B, H, S, d = 2, 3, 13, 8
    q, k, v = (RNG.standard_normal((B, H, S, d)) for _ in range(3))
    o0, l0 = oracle.attention(q, k, v, layout=0)
    t = lambda a: np.ascontiguousarray(a.transpose(0, 2, 1, 3))
    o1, l1 = oracle.attention(t(q), t(k), t(v), layout=1)
    np.testing.assert_array_equal(o1, t(o0))
    np.testing.assert_array_equal(l1, l0)


def test_attention_rows_match_full():
    B, H, S, d = 2, 2, 19, 8
    q, k, v = (RNG.standard_normal((B, S, H, d)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, layout=1)
    rows = np.array([0, 5, 18, 19, 40, B * H * S - 1])
    o_r, l_r = oracle.attention_rows(q, k, v, rows, layout=1)
    for t, r in enumerate(rows):
        b, h, i = r // (H * S), (r // S) % H, r % S
        np.testing.assert_array_equal(o_r[t], o[b, i, h])
        assert l_r[t] == lse[b, h, i]


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16, torch.float32])
def test_attention_reads_16bit_bytes_exactly(dt):
    B, H, S, d = 1, 2, 24, 16
    q, k, v = (torch.randn((B, H, S, d), dtype=torch.float32).to(dt) for _ in range(3))
    o, lse = oracle.attention(q, k, v)
    o_ref, lse_ref = _lib_attention(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                    1 / math.sqrt(d))
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-13)


def test_peaky_scores_stay_finite():
    """Scores of magnitude ~1e3 (exp would overflow without the max shift)."""
    q, k, v = (RNG.standard_normal((1, 2, 50, 8)) for _ in range(3))
    k[:, :, ::7] *= 300
    o, lse = oracle.attention(q, k, v, scale=1.0)
    o_ref, lse_ref = _lib_attention(q, k, v, 1.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-13)


# ----------------------------------------------------------- projection ----
def test_projection_selection_weights_and_head_split():
    """W = [I | 2I | 3I] gives Q = X, K = 2X, V = 3X; the split puts column c
    of each third into head c // d, feature c % d ("Transformer算子生态深度分析"
    ch.2 §2.1)."""
    B, S, D, h = 2, 3, 4, 2
    x = RNG.standard_normal((B, S, D))
    w = np.concatenate([np.eye(D), 2 * np.eye(D), 3 * np.eye(D)], axis=1)
    qkv = oracle.qkv_projection(x, w)
    np.testing.assert_array_equal(qkv, np.concatenate([x, 2 * x, 3 * x], axis=-1))
    q, k, v = oracle.split_heads(qkv, h)
    d = D // h
    for head in range(h):
        np.testing.assert_array_equal(q[:, :, head, :], x[:, :, head * d:(head + 1) * d])
        np.testing.assert_array_equal(k[:, :, head, :], 2 * x[:, :, head * d:(head + 1) * d])
        np.testing.assert_array_equal(v[:, :, head, :], 3 * x[:, :, head * d:(head + 1) * d])


def test_projection_triple_loop():
    B, S, D = 2, 4, 4
    x, w = RNG.standard_normal((B, S, D)), RNG.standard_normal((D, 3 * D))
    got = oracle.qkv_projection(x, w)
    for b in range(B):
        for s in range(S):
            for c in range(3 * D):
                want = sum(x[b, s, kk] * w[kk, c] for kk in range(D))
                assert got[b, s, c] == pytest.approx(want, rel=1e-14, abs=1e-14)


def test_projection_16bit_matches_matmul():
    x = torch.randn((2, 8, 24)).to(torch.float16)
    w = (torch.randn((24, 72)) * 0.02).to(torch.float16)
    got = oracle.qkv_projection(x, w)
    np.testing.assert_allclose(got, x.double().numpy() @ w.double().numpy(), rtol=1e-13, atol=1e-15)


def test_qkv_proj_attention_composition():
    B, S, D, h = 2, 11, 16, 4
    d = D // h
    x = RNG.standard_normal((B, S, D))
    w = RNG.standard_normal((D, 3 * D)) * 0.3
    o, lse = oracle.qkv_proj_attention(x, w, h)
    qkv = x @ w
    heads = lambda a: a.reshape(B, S, h, d).transpose(0, 2, 1, 3)  # -> [B,h,S,d]
    o_ref, lse_ref = _lib_attention(heads(qkv[..., :D]), heads(qkv[..., D:2 * D]),
                                    heads(qkv[..., 2 * D:]), 1 / math.sqrt(d))
    np.testing.assert_allclose(o, o_ref.transpose(0, 2, 1, 3), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12)


def test_bad_arguments_are_rejected():
    q = np.zeros((1, 1, 4, 4))
    with pytest.raises(ValueError):
        oracle.attention(q, q, q, layout=2)
    with pytest.raises(ValueError):
        oracle.attention(q, q, np.zeros((1, 1, 5, 4)))
    with pytest.raises(ValueError):
        oracle.attention_rows(q, q, q, [4])


# ------------------------------------------------------- grouped layout ----
def _to_grouped(a, hg):
    """[B,H,S,d] -> [B,H/hg,S,hg,d] by numpy reshape/transpose (the layout's definition)."""
    B, H, S, d = a.shape
    return np.ascontiguousarray(a.reshape(B, H // hg, hg, S, d).transpose(0, 1, 3, 2, 4))


@pytest.mark.parametrize("H,hg", [(4, 1), (4, 2), (4, 4), (6, 3)])
def test_grouped_layout_matches_contiguous(H, hg):
    B, S, d = 2, 11, 8
    q, k, v = (RNG.standard_normal((B, H, S, d)) for _ in range(3))
    o0, l0 = oracle.attention(q, k, v, layout=0)
    og, lg = oracle.attention_grouped(_to_grouped(q, hg), _to_grouped(k, hg), _to_grouped(v, hg), hg)
    np.testing.assert_array_equal(og, _to_grouped(o0, hg))
    np.testing.assert_array_equal(lg, l0)


def test_grouped_extremes_are_the_other_two_layouts():
    """hg = 1 is the contiguous layout byte for byte; hg = H the head-interleaved one."""
    B, H, S, d = 1, 3, 7, 4
    q, k, v = (RNG.standard_normal((B, H, S, d)) for _ in range(3))
    o1, _ = oracle.attention_grouped(q.reshape(B, H, S, 1, d), k.reshape(B, H, S, 1, d),
                                     v.reshape(B, H, S, 1, d), 1)
    np.testing.assert_array_equal(o1.reshape(B, H, S, d), oracle.attention(q, k, v, layout=0)[0])
    t = lambda a: np.ascontiguousarray(a.transpose(0, 2, 1, 3))
    oH, _ = oracle.attention_grouped(t(q).reshape(B, 1, S, H, d), t(k).reshape(B, 1, S, H, d),
                                     t(v).reshape(B, 1, S, H, d), H)
    np.testing.assert_array_equal(oH.reshape(B, S, H, d), oracle.attention(t(q), t(k), t(v), layout=1)[0])
