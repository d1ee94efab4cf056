"""Pins for the float64 attention backward (CPU only): central finite
differences of the forward definition, an independent automatic
differentiation of a forward written here, and closed forms and invariants
the gradient must satisfy."""
import numpy as np
import pytest
import torch

from oracle.attention import attention_fwd
from oracle.backward import attention_bwd


def _case(n, d, dv, seed, causal, scale=0.7):
    rng = np.random.default_rng(seed)
    q, k = (rng.standard_normal((1, 1, n, d)) for _ in range(2))
    v = rng.standard_normal((1, 1, n, dv))
    do = rng.standard_normal((1, 1, n, dv))
    o, lse = attention_fwd(q, k, v, causal, scale)
    return q, k, v, do, o, lse, scale


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences(causal):
    # the loss sum(O * dO) has gradient (dQ, dK, dV); central differences of
    # the forward definition with step 1e-5 agree to ~1e-9
    q, k, v, do, o, lse, scale = _case(6, 3, 4, seed=5, causal=causal)
    dq, dk, dv = attention_bwd(q, k, v, o, do, lse, causal, scale)

    def loss(q_, k_, v_):
        return float((attention_fwd(q_, k_, v_, causal, scale)[0] * do).sum())

    h = 1e-5
    for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = xp, xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=0, atol=1e-8)


@pytest.mark.parametrize("causal", [False, True])
def test_autograd_of_a_plain_forward(causal):
    # torch differentiates a softmax forward written out here (no shared code
    # with the oracle's closed-form backward), in float64
    q, k, v, do, o, lse, scale = _case(70, 16, 8, seed=9, causal=causal)
    tq, tk, tv = (torch.tensor(x[0, 0], requires_grad=True) for x in (q, k, v))
    s = scale * tq @ tk.T
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(70, 70, dtype=torch.bool), 1), float("-inf"))
    out = torch.softmax(s, dim=-1) @ tv
    out.backward(torch.tensor(do[0, 0]))
    dq, dk, dv = attention_bwd(q, k, v, o, do, lse, causal, scale)
    for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        np.testing.assert_allclose(mine[0, 0], ref.numpy(), rtol=0, atol=1e-12)


def test_invariants():
    # adding one vector to every key shifts each score row by a constant, so
    # the keys' gradients sum to zero; each probability row sums to one, so
    # the values' gradients sum to the upstream gradients' sum
    for causal in (False, True):
        q, k, v, do, o, lse, scale = _case(200, 16, 16, seed=3, causal=causal)
        dq, dk, dv = attention_bwd(q, k, v, o, do, lse, causal, scale)
        np.testing.assert_allclose(dk[0, 0].sum(axis=0), 0.0, atol=1e-11)
        np.testing.assert_allclose(dv[0, 0].sum(axis=0), do[0, 0].sum(axis=0), atol=1e-11)


def test_closed_forms():
    q, k, v, do, o, lse, scale = _case(50, 8, 8, seed=4, causal=True)
    dq, dk, dv = attention_bwd(q, k, v, o, do, lse, True, scale)
    # causal row 0 sees key 0 alone: P = 1, dS = dP - D = 0, so dQ_0 = 0
    np.testing.assert_allclose(dq[0, 0, 0], 0.0, atol=1e-13)
    # the last key is seen by the last row alone: dV_{N-1} = P_{N-1,N-1} dO_{N-1}
    p_last = np.exp(scale * q[0, 0, -1] @ k[0, 0, -1] - lse[0, 0, -1])
    np.testing.assert_allclose(dv[0, 0, -1], p_last * do[0, 0, -1], atol=1e-13)
    # Q = 0: uniform probabilities, dV_j = sum over the rows that see key j of dO_i / (i + 1)
    n = 50
    q0 = np.zeros_like(q)
    o0, lse0 = attention_fwd(q0, k, v, True, scale)
    _, _, dv0 = attention_bwd(q0, k, v, o0, do, lse0, True, scale)
    want = np.array([sum(do[0, 0, i] / (i + 1) for i in range(j, n)) for j in range(n)])
    np.testing.assert_allclose(dv0[0, 0], want, atol=1e-12)


# ---------------------------------------------------------------- MXFP8 backward

def test_square_blocks_are_transpose_invariant():
    # square 32 x 32 blocks: quantising X^T gives the transpose of quantising X,
    # so one payload serves a product along either axis
    from oracle.mxfp8 import quantize_blocks
    rng = np.random.default_rng(11)
    x = rng.standard_normal((70, 45)) * np.exp2(rng.integers(-6, 6, size=(70, 45)))
    codes, e, deq = quantize_blocks(x)
    codes_t, e_t, deq_t = quantize_blocks(x.T)
    np.testing.assert_array_equal(codes_t, codes.T)
    np.testing.assert_array_equal(e_t, e.T)
    np.testing.assert_array_equal(deq_t, deq.T)


def _e4m3_value(x):
    from oracle.mxfp8 import e4m3_decode, e4m3_encode
    return float(e4m3_decode(e4m3_encode(np.array([x]))[0]))


def _block_round(x):
    """Brute force, one block and one element at a time: each 32 x 32 block
    (from row 0 and column 0) takes the smallest e with amax <= 448 * 2^e,
    found by counting up; an all-zero block takes e = 0."""
    R, C = x.shape
    out = np.zeros_like(x)
    for r0 in range(0, R, 32):
        for c0 in range(0, C, 32):
            amax = max(abs(x[r, c]) for r in range(r0, min(R, r0 + 32)) for c in range(c0, min(C, c0 + 32)))
            e = 0
            if amax > 0:
                e = -300
                while amax > 448.0 * 2.0 ** e:
                    e += 1
            for r in range(r0, min(R, r0 + 32)):
                for c in range(c0, min(C, c0 + 32)):
                    out[r, c] = _e4m3_value(x[r, c] / 2.0 ** e) * 2.0 ** e
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_mxfp8_backward_brute_force(causal):
    # every product written as loops over single terms, on a ragged size
    from oracle.backward import attention_bwd_mxfp8
    n, d, scale = 37, 8, 0.6
    rng = np.random.default_rng(21)
    q, k, v, do = (rng.standard_normal((1, 1, n, d)) for _ in range(4))
    o, lse = attention_fwd(q, k, v, causal, scale)
    got = attention_bwd_mxfp8(q, k, v, o, do, lse, causal, scale)
    qd, kd, vd, dod = (_block_round(x[0, 0]) for x in (q, k, v, do))
    P = np.zeros((n, n))
    dS = np.zeros((n, n))
    for i in range(n):
        drow = sum(dod[i, c] * o[0, 0, i, c] for c in range(d))
        for j in range(n):
            if causal and j > i:
                continue
            P[i, j] = np.exp(scale * sum(qd[i, c] * kd[j, c] for c in range(d)) - lse[0, 0, i])
            dp = sum(dod[i, c] * vd[j, c] for c in range(d))
            dS[i, j] = P[i, j] * (dp - drow)
    P8 = np.array([[_e4m3_value(P[i, j] * 256.0) / 256.0 for j in range(n)] for i in range(n)])
    dS8 = _block_round(dS)
    dq = np.array([[scale * sum(dS8[i, j] * kd[j, c] for j in range(n)) for c in range(d)] for i in range(n)])
    dk = np.array([[scale * sum(dS8[i, j] * qd[i, c] for i in range(n)) for c in range(d)] for j in range(n)])
    dv = np.array([[sum(P8[i, j] * dod[i, c] for i in range(n)) for c in range(d)] for j in range(n)])
    for g, want in zip(got, (dq, dk, dv)):
        np.testing.assert_allclose(g[0, 0], want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_mxfp8_backward_within_the_fp8_rounding_bound(causal):
    # against the float64 gradient of the same (dequantised) inputs: rounding P
    # to E4M3 moves each P by at most 2^-4 of itself (2^-18 absolute below
    # E4M3's normal range at the 2^-8 scale), rounding dS by at most 2^-4 of
    # itself plus 2^-17 of its block's amax; the outputs move by at most the
    # same bounds carried through the products' absolute values
    from oracle.backward import attention_bwd_mxfp8
    from oracle.mxfp8 import quantize_blocks
    n, d, scale = 200, 32, 0.3
    rng = np.random.default_rng(5)
    q, k, v, do = (rng.standard_normal((1, 1, n, d)) for _ in range(4))
    o, lse = attention_fwd(q, k, v, causal, scale)
    got_q, got_k, got_v = (g[0, 0] for g in attention_bwd_mxfp8(q, k, v, o, do, lse, causal, scale))
    qd, kd, vd, dod = (quantize_blocks(x[0, 0])[2] for x in (q, k, v, do))
    ex_q, ex_k, ex_v = (g[0, 0] for g in attention_bwd(qd[None, None], kd[None, None], vd[None, None], o, dod[None, None],
                                                      lse, causal, scale))
    s = scale * qd @ kd.T
    P = np.exp(s - lse[0, 0][:, None])
    if causal:
        P = np.where(np.tril(np.ones((n, n), dtype=bool)), P, 0.0)
    dS = P * (dod @ vd.T - (dod * o[0, 0]).sum(axis=1)[:, None])
    blk = np.abs(np.pad(dS, ((0, 24), (0, 24)))).reshape(7, 32, 7, 32).max(axis=(1, 3))
    amax = np.repeat(np.repeat(blk, 32, axis=0), 32, axis=1)[:n, :n]
    eps_ds = 2.0 ** -4 * np.abs(dS) + 2.0 ** -17 * amax
    eps_p = 2.0 ** -4 * P + 2.0 ** -18
    assert np.all(np.abs(got_v - ex_v) <= eps_p.T @ np.abs(dod) + 1e-12)
    assert np.all(np.abs(got_k - ex_k) <= scale * eps_ds.T @ np.abs(qd) + 1e-12)
    assert np.all(np.abs(got_q - ex_q) <= scale * eps_ds @ np.abs(kd) + 1e-12)
    # and the rounding is really there: the outputs differ from the exact ones
    assert np.abs(got_k - ex_k).max() > 1e-6 and np.abs(got_v - ex_v).max() > 1e-6


@pytest.mark.parametrize("causal", [False, True])
def test_mxfp8_rows_equal_the_whole_head(causal):
    # the row-sampled form computes the same numbers as the whole head, at
    # rows inside, at the edge of and across 32-row blocks, ragged tail included
    from oracle.backward import attention_bwd_mxfp8_head, attention_bwd_mxfp8_rows
    n, d, scale = 203, 16, 0.4
    rng = np.random.default_rng(8)
    q, k, v, do = (rng.standard_normal((1, 1, n, d)) for _ in range(4))
    o, lse = attention_fwd(q, k, v, causal, scale)
    args = (q[0, 0], k[0, 0], v[0, 0], o[0, 0], do[0, 0], lse[0, 0], causal, scale)
    dq, dk, dv = attention_bwd_mxfp8_head(*args)
    rows = np.array([0, 31, 32, 95, 100, 191, 192, 202])
    got = attention_bwd_mxfp8_rows(*args, rows, rows[::-1])
    np.testing.assert_allclose(got["dq"], dq[rows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["dk"], dk[rows[::-1]], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["dv"], dv[rows[::-1]], rtol=0, atol=1e-12)
