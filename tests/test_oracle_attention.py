"""Pins for the float64 attention oracle (CPU only).

Each check ties ``oracle.attention`` to something other than itself: a
pure-Python brute force, closed forms, or the identities the pages state.
"""
import math

import numpy as np
import pytest

from attn_inputs import draw_fp32
from conftest import read_golden_kv
from oracle import attention as A
from oracle.exp2_model import bf16_round


def brute_force(q, k, v, causal, scale):
    """Pure-Python loops with math.exp; no NumPy arithmetic."""
    B, H, N, d = q.shape
    dv = v.shape[-1]
    o = [[[[0.0] * dv for _ in range(N)] for _ in range(H)] for _ in range(B)]
    lse = [[[0.0] * N for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            for i in range(N):
                allowed = [j for j in range(N) if (not causal or j <= i)]
                s = []
                for j in allowed:
                    acc = 0.0
                    for t in range(d):
                        acc += float(q[b, h, i, t]) * float(k[b, h, j, t])
                    s.append(scale * acc)
                mx = max(s)
                w = [math.exp(x - mx) for x in s]
                tot = sum(w)
                for c in range(dv):
                    o[b][h][i][c] = sum(w[n] * float(v[b, h, j, c]) for n, j in enumerate(allowed)) / tot
                lse[b][h][i] = mx + math.log(tot)
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 5, 3), (1, 2, 9, 4), (2, 1, 16, 8)])
def test_brute_force_matches(shape, causal):
    q, k, v = (x.astype(np.float64) for x in draw_fp32(*shape, seed=3))
    scale = 0.7
    o_ref, lse_ref = brute_force(q, k, v, causal, scale)
    o, lse = A.attention_fwd(q, k, v, causal, scale, row_chunk=4)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12


def test_brute_force_non_square_head_dims():
    # d != dv and N != d, so a transposed operand cannot go unnoticed
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 1, 7, 3))
    k = rng.standard_normal((1, 1, 7, 3))
    v = rng.standard_normal((1, 1, 7, 5))
    o_ref, lse_ref = brute_force(q, k, v, False, 0.4)
    o, lse = A.attention_fwd(q, k, v, False, 0.4)
    assert np.max(np.abs(o - o_ref)) < 1e-12 and np.max(np.abs(lse - lse_ref)) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_averages_values(causal):
    # q = 0: every allowed score is 0, so O_i is the mean of the allowed v_j and
    # LSE_i = ln(number of allowed keys).
    _, k, v = (x.astype(np.float64) for x in draw_fp32(1, 1, 12, 4, seed=1))
    q = np.zeros_like(k)
    o, lse = A.attention_fwd(q, k, v, causal, 0.5)
    for i in range(12):
        n = i + 1 if causal else 12
        assert np.allclose(o[0, 0, i], v[0, 0, :n].mean(axis=0), atol=1e-14)
        assert abs(lse[0, 0, i] - math.log(n)) < 1e-14


def test_two_keys_closed_form():
    # one query, two keys with q.k1 = x and q.k2 = 0: the weights are the
    # logistic pair, LSE = ln(e^{s x} + 1).
    x, s = 3.0, 0.8
    q = np.array([[[[1.0, 0.0]]]])
    k = np.array([[[[x, 0.0], [0.0, 5.0]]]])
    v = np.array([[[[2.0, -1.0], [0.5, 4.0]]]])
    o, lse = A.attention_fwd(q, k, v, False, s)
    w1 = 1.0 / (1.0 + math.exp(-s * x))
    expect = w1 * v[0, 0, 0] + (1.0 - w1) * v[0, 0, 1]
    assert np.allclose(o[0, 0, 0], expect, atol=1e-15)
    assert abs(lse[0, 0, 0] - math.log(math.exp(s * x) + 1.0)) < 1e-14


def test_causal_first_rows():
    q, k, v = (x.astype(np.float64) for x in draw_fp32(1, 1, 6, 4, seed=2))
    s = 0.3
    o, lse = A.attention_fwd(q, k, v, True, s)
    assert np.array_equal(o[0, 0, 0], v[0, 0, 0])                 # only key 0 allowed
    assert abs(lse[0, 0, 0] - s * float(q[0, 0, 0] @ k[0, 0, 0])) < 1e-14
    a = s * float(q[0, 0, 1] @ k[0, 0, 0])
    b = s * float(q[0, 0, 1] @ k[0, 0, 1])
    w0 = 1.0 / (1.0 + math.exp(b - a))
    assert np.allclose(o[0, 0, 1], w0 * v[0, 0, 0] + (1 - w0) * v[0, 0, 1], atol=1e-14)


def test_dominant_key():
    # a key whose score exceeds every other by more than 60 takes all the weight
    q, k, v = (x.astype(np.float64) for x in draw_fp32(1, 1, 8, 4, seed=4))
    unit = np.array([0.5, 0.5, 0.5, 0.5])
    k[0, 0, 5] = 10.0 * unit
    q[0, 0, 3] = 10.0 * unit                       # q.k5 = 100, |q.k_j| <= 10|k_j| otherwise
    assert np.max(np.abs(np.delete(k[0, 0], 5, axis=0) @ q[0, 0, 3])) < 40.0
    o, _ = A.attention_fwd(q, k, v, False, 1.0)
    assert np.allclose(o[0, 0, 3], v[0, 0, 5], atol=1e-12)


def test_blockwise_equals_one_shot_fp64():
    # "blockwise-LSE equals one-shot softmax" in float64, at the page's shape
    g = read_golden_kv("exactness_bands.txt")
    H, N, d, blk = int(g["H"]), int(g["N"]), int(g["d"]), int(g["block"])
    q, k, v = (x.astype(np.float64) for x in draw_fp32(1, H, N, d))
    o_ref, lse_ref = A.attention_fwd(q, k, v, False, 1.0 / math.sqrt(d))
    for blk_size in (blk, 128):
        o, lse, _ = A.blockwise_attention(q[0], k[0], v[0], False, 1.0 / math.sqrt(d), block=blk_size)
        assert np.max(np.abs(o - o_ref[0])) < 10 * g["fp64_max_abs"]
        assert np.max(np.abs(lse - lse_ref[0])) < 1e-12
    o2, lse2 = A.blockwise_attention_blockmax(q[0], k[0], v[0], False, 1.0 / math.sqrt(d), block=blk)
    assert np.max(np.abs(o2 - o_ref[0])) < 10 * g["fp64_max_abs"]
    assert np.max(np.abs(lse2 - lse_ref[0])) < 1e-12


@pytest.mark.parametrize("n", [256, 300])
def test_causal_block_skip_equals_masking(n):
    q, k, v = (x.astype(np.float64) for x in draw_fp32(1, 2, n, 32, seed=7))
    o_ref, lse_ref = A.attention_fwd(q, k, v, True, 0.25)
    o, lse, _ = A.blockwise_attention(q[0], k[0], v[0], True, 0.25, block=64)
    assert np.max(np.abs(o - o_ref[0])) < 1e-12
    assert np.max(np.abs(lse - lse_ref[0])) < 1e-12


def test_lagging_max_leaves_result_unchanged():
    # Q, K ~ N(0, 2^2): the running max keeps growing, so tau = 8 must actually
    # skip rescales, yet O and LSE must agree with tau = 0 in float64.
    q, k, v = (x.astype(np.float64) for x in draw_fp32(1, 2, 1024, 64, qk_std=2.0, seed=0))
    s = 1.0 / 8.0
    o0, lse0, f0 = A.blockwise_attention(q[0], k[0], v[0], True, s, block=128, tau=0.0)
    o8, lse8, f8 = A.blockwise_attention(q[0], k[0], v[0], True, s, block=128, tau=8.0)
    assert f8[..., 1:].sum() < f0[..., 1:].sum()
    assert np.max(np.abs(o8 - o0)) < 1e-12
    assert np.max(np.abs(lse8 - lse0)) < 1e-12
    o_ref, lse_ref = A.attention_fwd(q, k, v, True, s)
    assert np.max(np.abs(o8 - o_ref[0])) < 1e-12


def test_lse_combine_two_halves():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((5, 40)) * 3.0
    a, b = x[:, :17], x[:, 17:]
    m, l = A.lse_combine(a.max(1), np.exp(a - a.max(1, keepdims=True)).sum(1),
                         b.max(1), np.exp(b - b.max(1, keepdims=True)).sum(1))
    full = x.max(1) + np.log(np.exp(x - x.max(1, keepdims=True)).sum(1))
    assert np.max(np.abs(m + np.log(l) - full)) < 1e-14


def test_combine_partials_equals_one_shot():
    # attention over uneven key ranges, merged, is attention over all keys
    rng = np.random.default_rng(21)
    q, k, v = (rng.standard_normal((2, 3, 40, 16)) * 2.0 for _ in range(3))
    s = 0.3
    cuts = [0, 7, 26, 29, 40]
    parts = [A.attention_fwd(q, k[:, :, a:b], v[:, :, a:b], False, s) for a, b in zip(cuts[:-1], cuts[1:])]
    o, lse = A.combine_partials(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    o_ref, lse_ref = A.attention_fwd(q, k, v, False, s)
    assert np.max(np.abs(o - o_ref)) < 1e-12 and np.max(np.abs(lse - lse_ref)) < 1e-12
    # dropping a part's weight (averaging the parts instead) is far off
    o_bad = np.mean(np.stack([p[0] for p in parts]), axis=0)
    assert np.max(np.abs(o_bad - o_ref)) > 1e-2


def test_combine_partials_causal_chunks():
    # causal rows of query chunk i: full attention to earlier key chunks, the
    # chunk-local causal mask on its own chunk, nothing from later chunks
    rng = np.random.default_rng(5)
    n, c = 48, 16
    q, k, v = (rng.standard_normal((1, 2, n, 8)) for _ in range(3))
    s = 0.5
    o_ref, lse_ref = A.attention_fwd(q, k, v, True, s)
    for i in range(n // c):
        qs = q[:, :, i * c:(i + 1) * c]
        parts = [A.attention_fwd(qs, k[:, :, j * c:(j + 1) * c], v[:, :, j * c:(j + 1) * c], False, s)
                 for j in range(i)]
        parts.append(A.attention_fwd(qs, k[:, :, i * c:(i + 1) * c], v[:, :, i * c:(i + 1) * c], True, s))
        o, lse = A.combine_partials(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        assert np.max(np.abs(o - o_ref[:, :, i * c:(i + 1) * c])) < 1e-12
        assert np.max(np.abs(lse - lse_ref[:, :, i * c:(i + 1) * c])) < 1e-12


def test_combine_partials_special_cases():
    rng = np.random.default_rng(8)
    o1, l1 = rng.standard_normal((1, 4, 6, 5)), rng.standard_normal((1, 4, 6)) * 4
    # one part is itself
    o, lse = A.combine_partials(o1, l1)
    assert np.array_equal(o, o1[0]) and np.array_equal(lse, l1[0])
    # a part without keys (LSE = -inf) adds nothing
    o2 = rng.standard_normal((1, 4, 6, 5))
    o, lse = A.combine_partials(np.concatenate([o1, o2]), np.concatenate([l1, np.full((1, 4, 6), -np.inf)]))
    assert np.max(np.abs(o - o1[0])) < 1e-15 and np.array_equal(lse, l1[0])
    # no keys at all
    o, lse = A.combine_partials(o2, np.full((1, 4, 6), -np.inf))
    assert np.all(o == 0) and np.all(lse == -np.inf)
    # two equal parts: O unchanged, LSE + ln 2
    o, lse = A.combine_partials(np.concatenate([o1, o1]), np.concatenate([l1, l1]))
    assert np.max(np.abs(o - o1[0])) < 1e-14 and np.max(np.abs(lse - (l1[0] + math.log(2.0)))) < 1e-14
    # merging in two steps equals merging at once (associativity of the exact merge)
    o3, l3 = rng.standard_normal((1, 4, 6, 5)), rng.standard_normal((1, 4, 6)) * 4
    oa, la = A.combine_partials(np.concatenate([o1, o2]), np.concatenate([l1, l3]))
    ob, lb = A.combine_partials(np.stack([oa, o3[0]]), np.stack([la, l3[0] + 1.0]))
    oc, lc = A.combine_partials(np.concatenate([o1, o2, o3]), np.concatenate([l1, l3, l3 + 1.0]))
    assert np.max(np.abs(ob - oc)) < 1e-13 and np.max(np.abs(lb - lc)) < 1e-13


def test_precision_bands():
    # fp32 recurrence ~1e-5 and bf16 inputs with bf16 P ~5e-3..1e-2 against float64
    g = read_golden_kv("exactness_bands.txt")
    H, N, d = int(g["H"]), int(g["N"]), int(g["d"])
    q, k, v = draw_fp32(1, H, N, d)
    s = 1.0 / math.sqrt(d)
    o_ref, _ = A.attention_fwd(q, k, v, False, s)
    o32, _, _ = A.blockwise_attention(q[0], k[0], v[0], False, s, block=64, dtype=np.float32)
    e32 = np.max(np.abs(o32 - o_ref[0]))
    assert 1e-8 < e32 < 10 * g["fp32_max_abs"]
    qb, kb, vb = (bf16_round(x) for x in (q, k, v))
    o_refb, _ = A.attention_fwd(qb, kb, vb, False, s)
    ob, _, _ = A.blockwise_attention(qb[0], kb[0], vb[0], False, s, block=64, dtype=np.float32,
                                     p_cast=bf16_round)
    ob = bf16_round(ob)
    eb = np.max(np.abs(ob - o_refb[0]))
    assert eb < g["bf16_max_abs_hi"]


def test_blockwise_row_index_selects_rows():
    # the recurrence on a subset of query rows, given their positions, equals
    # the same rows of the full computation (causal mask by position)
    rng = np.random.default_rng(11)
    q, k, v = (rng.standard_normal((300, 32)) for _ in range(3))
    o, lse, _ = A.blockwise_attention(q, k, v, True, 0.2, block=64, tau=8.0)
    rows = np.array([0, 1, 63, 64, 150, 299])
    o_s, lse_s, _ = A.blockwise_attention(q[rows], k, v, True, 0.2, block=64, tau=8.0, row_index=rows)
    assert np.allclose(o_s, o[rows], rtol=0, atol=1e-12) and np.allclose(lse_s, lse[rows], rtol=0, atol=1e-12)
