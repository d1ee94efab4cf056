"""Pins for the parity gates themselves (CPU only).

A float32 simulation of the kernel's arithmetic stands in for the GPU: scores
as a float32 product of the bf16 inputs, the running max moved by the tau rule,
P = exp2 in float32, P rounded to bf16 for P V, the row sum and P V
accumulated in float32, O / l rounded to bf16. The method bound must hold
for it. Each of four plausible kernel mistakes must break it: P truncated
instead of rounded, the row sum taken from the rounded P, the row sum left
unscaled when the max moves, and a causal mask that also hides the diagonal.
(A rescale decision taken at growth == tau instead of above it is invisible
in O whenever the growth is exactly tau and tau is an integer: both choices
scale P by an exact power of two. The kernel's decisions are checked directly
by the GPU test of the decision log.)
"""
import math

import numpy as np
import pytest

from oracle.attention import attention_fwd
from parity import bf16_rn, bf16_ulp, compare, compare_method, method_reference

LOG2E = 1.0 / math.log(2.0)


def _bf16(x):
    return bf16_rn(x)


def _trunc_bf16(x):
    mant, expo = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.trunc(mant * 256.0) / 256.0, expo)


def simulate_kernel(q, k, v, causal, scale, tau, p_round=_bf16, sum_rounded=False, sum_unscaled=False,
                    mask_diagonal=False, block=128):
    """Forward pass in float32 the way the kernel orders it (one head)."""
    q32, k32, v32 = (np.asarray(x, dtype=np.float32) for x in (q, k, v))
    n, nk = q32.shape[0], k32.shape[0]
    sl2 = np.float32(scale * LOG2E)
    m = np.full(n, -np.inf, dtype=np.float32)
    l = np.zeros(n, dtype=np.float32)
    o = np.zeros((n, v32.shape[1]), dtype=np.float32)
    rows = np.arange(n)
    for j0 in range(0, nk, block):
        j1 = min(nk, j0 + block)
        s = (q32 @ k32[j0:j1].T).astype(np.float32)
        if causal:
            keep = (np.arange(j0, j1)[None, :] < rows[:, None]) if mask_diagonal else \
                (np.arange(j0, j1)[None, :] <= rows[:, None])
            s = np.where(keep, s, np.float32(-np.inf))
        bm = s.max(axis=1)
        m_new = np.maximum(m, bm)
        with np.errstate(invalid="ignore"):
            g = (m_new - m) * sl2
        fire = ~(g <= tau)
        fire &= np.isfinite(m_new)
        m_new = np.where(fire, m_new, m)
        with np.errstate(invalid="ignore"):
            corr = np.where(fire, np.where(np.isfinite(m), np.exp2((m - m_new) * sl2), 0.0), 1.0).astype(np.float32)
            neg = np.where(np.isfinite(m_new), -(m_new * sl2), 0.0).astype(np.float32)
            p = np.exp2((s * sl2 + neg[:, None]).astype(np.float32)).astype(np.float32)
        p = np.where(np.isfinite(s), p, np.float32(0.0))
        pr = p_round(p).astype(np.float32)
        l_corr = np.where(np.isfinite(m), np.float32(1.0), corr) if sum_unscaled else corr
        l = (l * l_corr + (pr if sum_rounded else p).sum(axis=1, dtype=np.float32)).astype(np.float32)
        o = (o * corr[:, None] + (pr @ v32[j0:j1]).astype(np.float32)).astype(np.float32)
        m = m_new
    with np.errstate(divide="ignore", invalid="ignore"):
        out = _bf16((o * (np.float32(1.0) / l)[:, None]).astype(np.float32))
    with np.errstate(divide="ignore"):
        lse = (m.astype(np.float64) * scale + np.log(l.astype(np.float64)))
    return out, lse


def _peaked(n=512, d=64, qk_std=4.0, seed=21):
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((n, d)).astype(np.float32) for _ in range(3))
    q *= np.float32(qk_std)
    k *= np.float32(qk_std)
    return _bf16(q), _bf16(k), _bf16(v)


@pytest.mark.parametrize("tau", [0.0, 8.0, 16.0])
@pytest.mark.parametrize("causal", [False, True])
def test_method_bound_holds_for_fp32_arithmetic(tau, causal):
    q, k, v = _peaked()
    scale = 64 ** -0.5
    o, _ = simulate_kernel(q, k, v, causal, scale, tau)
    o_m, _, delta, big_a, suspect = method_reference(q, k, v, causal, scale, tau)
    st = compare_method(o, o_m, delta, big_a, suspect, f"sim tau={tau} causal={causal}")
    # the bound on the arithmetic's error is much tighter than the envelope
    # 2^-8 A it replaces (both before the output's own half-ulp rounding)
    assert st["delta_mean"] < 0.2 * st["p_rounding_envelope_mean"]


def test_plain_gate_passes_fp32_arithmetic_on_unit_inputs():
    rng = np.random.default_rng(3)
    q, k, v = (_bf16(rng.standard_normal((1, 1, 700, 64))) for _ in range(3))
    o, lse = simulate_kernel(q[0, 0], k[0, 0], v[0, 0], True, 0.125, 8.0)
    o_ref, lse_ref = attention_fwd(q, k, v, True, 0.125)
    st = compare(o[None, None], lse[None, None], o_ref, lse_ref, "sim unit")
    assert st["o_over_1e-2"] == 0


@pytest.mark.parametrize("mistake", ["truncated_p", "sum_of_rounded_p", "sum_unscaled", "mask_diagonal"])
def test_method_bound_catches_plausible_mistakes(mistake):
    q, k, v = _peaked(n=384, seed=5)
    scale = 64 ** -0.5
    tau = 8.0
    kw = {"truncated_p": {"p_round": _trunc_bf16}, "sum_of_rounded_p": {"sum_rounded": True},
          "sum_unscaled": {"sum_unscaled": True}, "mask_diagonal": {"mask_diagonal": True}}[mistake]
    causal = mistake == "mask_diagonal"
    o, _ = simulate_kernel(q, k, v, causal, scale, tau, **kw)
    o_m, _, delta, big_a, suspect = method_reference(q, k, v, causal, scale, tau)
    if causal:
        o, o_m, delta, big_a, suspect = o[1:], o_m[1:], delta[1:], big_a[1:], suspect[1:]   # row 0 sees no key
    with pytest.raises(AssertionError):
        compare_method(o, o_m, delta, big_a, np.zeros_like(suspect), mistake)


def test_floor_exception_is_one_bf16_step():
    # |O_ref| = 5.01: RN_bf16 is 5.0, floor 0.01 < 1e-2 -> plain gate;
    # |O_ref| = 6.012: RN is 6.0 (ulp 2^-5), floor 0.012 > 1e-2 -> one step allowed
    o_ref = np.array([5.01, 6.012, 6.012, 6.012])
    lse = np.zeros(4)
    ok = np.array([5.0, 6.0, 6.03125, 5.96875])
    st = compare(ok, lse, o_ref, lse, "steps", mean_gate=False)
    assert st["floor_exceptions"] == 3 and st["o_over_1e-2"] == 3
    with pytest.raises(AssertionError):
        compare(np.array([5.0, 6.0625, 6.0, 6.0]), lse, o_ref, lse, "two steps", mean_gate=False)
    with pytest.raises(AssertionError):
        # 5.01 -> 4.99 is 0.02 away: its floor is below 1e-2, so no exception
        compare(np.array([4.96875, 6.0, 6.0, 6.0]), lse, o_ref, lse, "plain", mean_gate=False)


def test_max_history_is_the_running_max():
    # with tau = 0 the reference max of block b is the max over blocks 0..b
    rng = np.random.default_rng(0)
    q, k, v = (rng.standard_normal((200, 16)) for _ in range(3))
    from oracle.attention import blockwise_attention
    _, _, _, mh = blockwise_attention(q, k, v, False, 0.25, block=32, tau=0.0, max_history=True)
    s = q @ k.T
    bm = np.stack([s[:, j:j + 32].max(axis=1) for j in range(0, 200, 32)], axis=1)
    assert np.array_equal(mh, np.maximum.accumulate(bm, axis=1))
    # with tau the history is non-decreasing and ends at most tau below the true max
    _, _, _, mh8 = blockwise_attention(q, k, v, False, 0.25, block=32, tau=8.0, max_history=True)
    assert np.all(np.diff(mh8, axis=1) >= 0)
    assert np.all((s.max(axis=1) - mh8[:, -1]) * 0.25 * LOG2E <= 8.0 + 1e-12)


def test_method_floor_exempts_only_what_the_method_itself_misses():
    # peaked rows with tau = 4: the method (float64, P rounded to bf16, bf16
    # output) is itself more than 1e-2 from the exact result on a few elements
    q, k, v = _peaked(n=640, d=64, qk_std=4.0, seed=9)
    scale = 64 ** -0.5
    o_ref, lse_ref = attention_fwd(q[None, None], k[None, None], v[None, None], True, scale)
    o_ref, lse_ref = o_ref[0, 0], lse_ref[0, 0]
    o_m, lse_m, delta, _, _ = method_reference(q, k, v, True, scale, 4.0)
    out = bf16_rn(o_m)
    with pytest.raises(AssertionError):
        compare(out, lse_m, o_ref, lse_ref, "no method floor")        # the flat 1e-2 cannot hold
    st = compare(out, lse_m, o_ref, lse_ref, "method floor", method=(o_m, delta))
    assert st["method_floor_exceptions"] > 0 and st["o_over_1e-2"] <= st["method_floor_exceptions"]
    # an exempt element two bf16 steps away from the method fails
    i = np.argwhere(np.abs(out - o_ref) > 1e-2)[0]
    bad = out.copy()
    bad[tuple(i)] += 2 * 2.0 ** (np.floor(np.log2(abs(bad[tuple(i)]))) - 7) * np.sign(bad[tuple(i)])
    with pytest.raises(AssertionError):
        compare(bad, lse_m, o_ref, lse_ref, "two steps off the method", method=(o_m, delta))


def test_method_floor_covers_the_band_the_method_admits():
    # An element whose method result rounds to within 1e-2 of the exact one,
    # while the method's band (o_m +- delta, then the bf16 rounding) reaches
    # past 1e-2: the other bf16 neighbour, inside the band, is an output the
    # method's arithmetic admits and passes; two steps further out it fails.
    q, k, v = _peaked(n=640, d=64, qk_std=2.0, seed=0)
    scale = 0.37
    o_ref, lse_ref = attention_fwd(q[None, None], k[None, None], v[None, None], True, scale)
    o_ref, lse_ref = o_ref[0, 0], lse_ref[0, 0]
    o_m, lse_m, delta, _, suspect = method_reference(q, k, v, True, scale, 8.0)
    mbound = delta + 0.5 * bf16_ulp(np.abs(o_m) + delta)
    rnd = bf16_rn(o_m)
    step = bf16_ulp(np.abs(rnd))
    away = rnd + np.sign(rnd - o_ref) * step            # the neighbour away from O_ref
    band_only = ((np.abs(rnd - o_ref) <= 1e-2) & (np.abs(o_m - o_ref) + mbound > 1e-2)
                 & (np.abs(away - o_m) <= mbound) & (np.abs(away - o_ref) > 1e-2) & ~suspect[:, None]
                 & (np.abs(bf16_rn(o_ref) - o_ref) <= 1e-2))
    i = tuple(np.argwhere(band_only)[0])
    # the method's own output is within 1e-2 there, the neighbour is not
    assert abs(rnd[i] - o_ref[i]) <= 1e-2 < abs(away[i] - o_ref[i])
    base = compare(rnd, lse_m, o_ref, lse_ref, "method output", method=(o_m, delta))
    out = rnd.copy()
    out[i] = away[i]
    st = compare(out, lse_m, o_ref, lse_ref, "band element", method=(o_m, delta))
    assert st["exceptions_failed"] == 0 and st["o_over_1e-2_floor_ok"] == 0
    assert st["o_over_1e-2"] == base["o_over_1e-2"] + 1
    far = out.copy()
    far[i] = away[i] + 2 * np.sign(rnd[i] - o_ref[i]) * step[i]
    with pytest.raises(AssertionError):
        compare(far, lse_m, o_ref, lse_ref, "two steps past the band element", method=(o_m, delta))
