"""Parity helpers shared by the GPU tests.

Gate against the float64 oracle (the kernel's bf16 output, the same bf16
inputs on both sides):
  * O, elementwise: |O - O_ref| <= 1e-2, the required bound. The one exception
    is an element whose own rounding floor |RN_bf16(O_ref) - O_ref| already
    exceeds 1e-2, which no bf16 output can meet. Half a bf16 ulp only exceeds
    1e-2 where the ulp is 2^-5 or more, i.e. |O_ref| >= 4 (in [2, 4) the ulp
    is 2^-6 = 0.0156, so half of it is 0.0078 < 1e-2). Such an element must be
    RN_bf16(O_ref) or one of its two bf16 neighbours. Every exception is
    counted and reported, never hidden.
  * O, mean over all compared elements: <= 1e-3.
  * LSE: |LSE - LSE_ref| <= 1e-3.

Stress inputs outside the five workloads (tau = 16, scaled-score standard
deviations near 16, scale 0.37) have peaked rows. On those rows the kernel's
correct rounding of P to bf16 alone moves O by more than 1e-2 from the exact
result, because with a lagging max the dominant P is 2^delta, not exactly 1.
They are gated instead against the method at the kernel's precision. That is
the oracle's blockwise recurrence with the kernel's 128-key blocks and tau,
P rounded to bf16 (RN) before P V, and the row sum taken from the unrounded P.
The bound below is derived from the arithmetic (``method_reference``).

The kernel computes each P in fp32 with a small relative error E_ij. The bound
takes E_ij from the MUFU exp2, the fp32 rounding of the exponent, and the fp32
dot product of S and of the row max. The kernel's bf16 P can then differ from
the method's bf16 P only where a bf16 rounding midpoint lies within E_ij P_ij
of P_ij (an "at-risk" term), and there by one bf16 ulp at most. So
  |O~ - O_m| <= sum_{j at risk} ulp(P_ij)/P_ij w_ij |V_jc|  +  slack * A_ic
with w_ij the final softmax weights, A_ic = sum_j w_ij |V_jc|, and slack
covering the relative error of the fp32 row sum, the fp32 accumulation of the
products and the correction factors. The output's bf16 rounding adds half an
ulp. Rows whose rescale decision lies within the score error of tau could
rescale differently; they are reported and gated by the looser envelope
2^-8 A + ulp/2 + 1e-3 (the bound for any placement of the running max).
"""
from __future__ import annotations

import math

import numpy as np

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3
LOG2E = 1.0 / math.log(2.0)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.float64(2.0 ** -126))
    return np.ldexp(1.0, np.floor(np.log2(ax)).astype(np.int64) - 7)


def bf16_rn(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even), as float64."""
    mant, expo = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.rint(mant * 256.0) / 256.0, expo)


def _bf16_steps(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """How many bf16 values apart a and b are (both exact bf16 values)."""
    ia = (np.asarray(a, dtype=np.float32).view(np.int32) >> 16).astype(np.int64)
    ib = (np.asarray(b, dtype=np.float32).view(np.int32) >> 16).astype(np.int64)
    # map sign-magnitude to a monotone integer line
    ia = np.where(ia < 0, -(ia & 0x7FFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFF), ib)
    return np.abs(ia - ib)


def compare(o, lse, o_ref, lse_ref, what: str = "", max_gate: bool = True, mean_gate: bool = True,
            method=None) -> dict:
    """Assert the gate against the exact oracle; returns the statistics.

    ``method`` = (o_m, delta), the method at the kernel's precision and its
    bound (``method_reference``), adds the method's floor. The kernel may land
    anywhere in o_m +- delta before its output is rounded to bf16, so every
    output the method admits lies within delta + half an ulp of o_m. An
    element where some of those outputs lie more than 1e-2 from O_ref
    (|o_m - O_ref| + delta + half an ulp > 1e-2) is gated at |O - o_m| <=
    delta + half an ulp instead of 1e-2: with a lagging max the bf16 rounding
    of the dominant P is the method's own error, up to 2^-9 |V|, and the
    output's half ulp comes on top of it. ``max_gate=False`` only reports the
    elementwise figures."""
    o = np.asarray(o, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    err = np.abs(o - o_ref)
    rnd = bf16_rn(o_ref)
    floor = np.abs(rnd - o_ref)
    exc = floor > O_MAX_ABS
    steps = _bf16_steps(o, rnd)
    ok_exc = exc & (steps <= 1)
    mexc = np.zeros_like(exc)
    if method is not None:
        o_m, delta = (np.asarray(x, dtype=np.float64) for x in method)
        mbound = delta + 0.5 * bf16_ulp(np.abs(o_m) + delta)
        mexc = (np.abs(o_m - o_ref) + mbound > O_MAX_ABS) & ~exc
        ok_exc = ok_exc | ((exc | mexc) & (np.abs(o - o_m) <= mbound))
    lerr = np.abs(np.asarray(lse, dtype=np.float64) - np.asarray(lse_ref, dtype=np.float64))
    plain = ~(exc | mexc)
    stats = {
        "o_max_abs": float(err.max()) if err.size else 0.0,
        "o_mean_abs": float(err.mean()) if err.size else 0.0,
        "o_over_1e-2": int((err > O_MAX_ABS).sum()),
        "o_over_1e-2_floor_ok": int(((err > O_MAX_ABS) & plain).sum()),
        "floor_exceptions": int(exc.sum()),
        "method_floor_exceptions": int(mexc.sum()),
        "exceptions_failed": int(((exc | mexc) & ~ok_exc).sum()),
        "o_floor_max": float(floor.max()) if floor.size else 0.0,
        "lse_max_abs": float(lerr.max()) if lerr.size else 0.0,
        "finite": bool(np.isfinite(o).all() and np.isfinite(lse).all()),
    }
    print(f"parity {what}: {stats}")
    assert stats["finite"], f"{what}: non-finite output {stats}"
    if max_gate:
        assert stats["o_over_1e-2_floor_ok"] == 0, f"{what}: O beyond 1e-2 {stats}"
        assert stats["exceptions_failed"] == 0, f"{what}: O beyond its floor exception's bound {stats}"
    if mean_gate:
        assert stats["o_mean_abs"] <= O_MEAN_ABS, f"{what}: O mean error {stats}"
    assert stats["lse_max_abs"] <= LSE_MAX_ABS, f"{what}: LSE error {stats}"
    return stats


def compare_heads(o, lse, o_ref, lse_ref, q, k, v, causal: bool, scale: float, tau: float = 8.0,
                  what: str = "", rows=None, mean_gate: bool = True, exp_rel_err: float = 2.0 ** -21,
                  block: int = 128) -> dict:
    """``compare`` over [B, H, R, dv] outputs with the method's floor computed
    where it is needed: for every head with an element more than 1e-2 from
    O_ref (beyond its output-rounding floor), the method at the kernel's
    precision is formed for that head (q [B, H, R, d] the compared rows at
    positions ``rows``, default 0 .. R-1; k, v [B, H, N, *]) and the element is
    held to it. Heads without such an element are gated by the flat 1e-2.
    ``exp_rel_err`` is the relative error of the kernel's exp2 (the MUFU's by
    default; the software exp2's 8.77e-5 when a share of it is used);
    ``block`` the keys per block of the kernel's recurrence."""
    o = np.asarray(o, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    err = np.abs(o - o_ref)
    rnd = bf16_rn(o_ref)
    exc = np.abs(rnd - o_ref) > O_MAX_ABS
    suspect = ((err > O_MAX_ABS) & ~exc) | (exc & (_bf16_steps(o, rnd) > 1))
    o_m = o_ref.copy()
    delta = np.zeros_like(o_ref)
    heads = np.argwhere(suspect.any(axis=(2, 3)))
    for b, h in heads:
        o_m[b, h], _, delta[b, h], _, _ = method_reference(q[b, h], k[b, h], v[b, h], causal, scale, tau,
                                                           exp_rel_err=exp_rel_err, block=block, row_index=rows)
    st = compare(o, lse, o_ref, lse_ref, what, mean_gate=mean_gate, method=(o_m, delta))
    st["heads_with_method_floor"] = int(len(heads))
    return st


def method_reference(q, k, v, causal: bool, scale: float, tau: float, exp_rel_err: float = 2.0 ** -21,
                     block: int = 128, row_index=None):
    """The method at the kernel's precision for ONE head (float64 q [R, d]
    with its rows' positions ``row_index``, default 0 .. R-1; k [N, d], v [N,
    dv]) and the per-element bound of the module docstring.

    Returns (o_m, lse_m, delta, big_a, suspect_rows): delta [N, dv] bounds
    |O~ - o_m| before the output's bf16 rounding; big_a is A (the attention of
    |V|), from which ``compare_method`` forms the looser envelope used for the
    suspect rows (a rescale decision within the score error of tau)."""
    from oracle.attention import blockwise_attention
    from oracle.exp2_model import bf16_round
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, nk = q.shape[0], k.shape[0]
    rows = np.arange(n) if row_index is None else np.asarray(row_index)
    o_m, lse_m, _, m_used = blockwise_attention(q, k, v, causal, scale, block=block, tau=tau,
                                                p_cast=bf16_round, max_history=True, row_index=rows)
    sl2 = scale * LOG2E
    s = q @ k.T                                          # raw scores
    allowed = np.ones((n, nk), dtype=bool)
    if causal:
        allowed = np.arange(nk)[None, :] <= rows[:, None]
    nb = m_used.shape[1]
    ref = np.repeat(m_used, block, axis=1)[:, :nk]       # the max each key's P was taken against
    with np.errstate(invalid="ignore", over="ignore"):
        x = np.where(allowed, (s - ref) * sl2, -np.inf)
        p = np.exp2(x)                                   # the method's P (before rounding)
        w = np.where(allowed, np.exp(s * scale - lse_m[:, None]), 0.0)   # final softmax weights
    # relative error of the kernel's fp32 P: the exp2 itself, the fp32 rounding of
    # the exponent (and of -m s log2 e), and the fp32 dot products behind S_ij and m_i
    a = np.abs(q) @ np.abs(k).T                          # sum_c |q_ic k_jc|
    a_row = np.where(allowed, a, 0.0).max(axis=1, keepdims=True)
    e_rel = exp_rel_err + math.log(2.0) * (2.0 ** -23 * np.abs(np.where(allowed, x, 0.0))
                                           + 2.0 ** -23 * np.abs(np.where(np.isfinite(ref), ref, 0.0)) * sl2
                                           + 2.0 ** -22 * sl2 * (a + a_row))
    ulp_rel = np.where(p > 0, bf16_ulp(p) / np.where(p > 0, p, 1.0), 0.0)
    mant = np.where(p > 0, p / bf16_ulp(p), 0.0)         # position inside the bf16 binade, in ulps
    mid_dist = np.abs(mant - np.floor(mant) - 0.5) * ulp_rel   # relative distance to the nearest midpoint
    at_risk = allowed & (p > 0) & (mid_dist <= e_rel)
    av = np.abs(v)
    risk = (np.where(at_risk, ulp_rel * w, 0.0)) @ av
    big_a = w @ av
    slack = (e_rel.max(axis=1, keepdims=True) + (nk / 16 + 8) * 2.0 ** -22 + nb * 2.0 ** -21)
    delta = risk + slack * big_a
    # rows whose decision to move the max might go the other way in fp32
    suspect = np.zeros(n, dtype=bool)
    m_prev = np.full(n, -np.inf)
    for jb in range(nb):
        j0, j1 = jb * block, min(nk, (jb + 1) * block)
        sb = np.where(allowed[:, j0:j1], s[:, j0:j1], -np.inf)
        bmax = sb.max(axis=1)
        live = np.isfinite(m_prev) & np.isfinite(bmax)
        # signed growth: the max moves iff it exceeds tau (a block whose max lies
        # below the running one has growth 0, and so does not move it)
        g = np.where(live, (bmax - np.where(live, m_prev, 0.0)) * sl2, np.inf)
        margin = 2.0 ** -20 * sl2 * a_row[:, 0] + 2.0 ** -20 * np.abs(g)
        suspect |= live & (np.abs(g - tau) <= margin)
        m_prev = np.where(np.isfinite(m_used[:, jb]), m_used[:, jb], m_prev)
    return o_m, lse_m, delta, big_a, suspect


def compare_method(o, o_m, delta, big_a, suspect, what: str = "") -> dict:
    """Assert |O - o_m| <= delta + half an output ulp elementwise (the
    envelope 2^-8 A + ulp/2 + 1e-3 on suspect rows); returns the statistics,
    including the mean of delta against the mean of the 2^-8 A it replaces."""
    o = np.asarray(o, dtype=np.float64)
    err = np.abs(o - o_m)
    bound = delta + 0.5 * bf16_ulp(np.abs(o_m) + delta)
    envelope = 2.0 ** -8 * big_a + 1e-3 + 0.5 * bf16_ulp(o_m)
    bound = np.where(suspect[:, None], np.maximum(bound, envelope), bound)
    keep = ~suspect
    stats = {
        "o_max_abs_vs_method": float(err.max()) if err.size else 0.0,
        "o_over_bound": int((err > bound).sum()),
        "bound_max": float(bound.max()) if bound.size else 0.0,
        "delta_mean": float(delta[keep].mean()) if delta[keep].size else 0.0,
        "p_rounding_envelope_mean": float(2.0 ** -8 * big_a[keep].mean()) if big_a[keep].size else 0.0,
        "worst_err_over_bound": float((err / bound).max()) if err.size else 0.0,
        "suspect_rows": int(suspect.sum()),
    }
    print(f"method parity {what}: {stats}")
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    assert stats["o_over_bound"] == 0, f"{what}: O beyond the method bound {stats}"
    return stats


def sample_rows(N: int, rng: np.random.Generator, n_random: int = 24) -> np.ndarray:
    """Query rows to check at full size: the first rows, both sides of every
    128-row tile edge within the first and last 512 rows, the last rows, and
    random ones."""
    fixed = [0, 1, 2, 3, 63, 64, 126, 127, 128, 129, 254, 255, 256, 257, 383, 384, 511, 512]
    fixed += [N - 1, N - 2, N - 127, N - 128, N - 129, N - 255, N - 256, N - 257, N - 512]
    rnd = rng.integers(0, N, size=n_random).tolist()
    rows = sorted({r for r in fixed + rnd if 0 <= r < N})
    return np.array(rows, dtype=np.int64)
