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
