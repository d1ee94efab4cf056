"""Float64 attention forward: the definition, and the online recurrence.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

``attention_fwd`` is the oracle: the one-shot safe softmax of the scaled scores
times V, with the per-row log-sum-exp. It follows "Lecture 2 - Online Softmax
and Numerical Correctness", section "The classical safe softmax" (softmax with
the row max subtracted; LSE = m + log of the shifted sum) and section "Causal
masking just changes which blocks contribute" (scores with j > i are -inf). The
scale multiplies the raw dot product before the softmax, as in the naive
three-step algorithm of "Flash Attention 4 - the algorithm and the two-MMA
problem", section "The memory-bound trap". All arithmetic is float64 and the
full score row is formed at once; rows are processed in chunks only to bound
memory.

``blockwise_attention`` restates the streaming recurrence (running max, running
sum, rescaled accumulator, normalisation deferred to the end) from "Flash
Attention 4 - the algorithm and the two-MMA problem", sections "Online softmax -
three running states" and "Deferred normalization", with the optional lagging
max of "FlashAttention-4's Softmax Tricks", section "Conditional rescaling, and
when it's exact". It exists only so the tests can check the one-shot definition
against the identities the pages state (blockwise equals one-shot in float64;
causal block skipping equals -inf masking; a stale max leaves O/l unchanged).
"""
from __future__ import annotations

import math

import numpy as np

LOG2E = 1.0 / math.log(2.0)


def _check(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> None:
    if q.ndim != 4 or k.shape != q.shape[:2] + k.shape[2:] or v.shape[:3] != k.shape[:3]:
        raise ValueError(f"bad shapes q{q.shape} k{k.shape} v{v.shape}")
    if q.shape[-1] != k.shape[-1]:
        raise ValueError("q and k head dims differ")


def attention_rows(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray, row_index: np.ndarray,
                   causal: bool, scale: float) -> tuple[np.ndarray, np.ndarray]:
    """One-shot attention for a set of query rows of ONE (batch, head).

    q_rows [R, d] (float64), k [Nk, d], v [Nk, dv]; row_index [R] holds each
    query row's position i, used only by the causal mask (key j allowed iff
    j <= i). Returns O [R, dv] and LSE [R], both float64.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = scale * (q_rows @ k.T)                      # [R, Nk] scaled scores
    if causal:
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j <= np.asarray(row_index)[:, None], s, -np.inf)
    m = s.max(axis=1)                               # row max (finite: key 0 is always allowed)
    e = np.exp(s - m[:, None])                      # exp(-inf) = 0 for masked keys
    l = e.sum(axis=1)
    o = (e @ v) / l[:, None]
    lse = m + np.log(l)
    return o, lse


def attention_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool, scale: float,
                  row_chunk: int = 512) -> tuple[np.ndarray, np.ndarray]:
    """O = softmax(s * Q K^T [masked]) V and LSE, float64, for [B,H,N,d] inputs."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    _check(q, k, v)
    B, H, N, _ = q.shape
    o = np.empty((B, H, N, v.shape[-1]), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for i0 in range(0, N, row_chunk):
                i1 = min(N, i0 + row_chunk)
                o[b, h, i0:i1], lse[b, h, i0:i1] = attention_rows(
                    q[b, h, i0:i1], k[b, h], v[b, h], np.arange(i0, i1), causal, scale)
    return o, lse


def blockwise_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool, scale: float,
                        block: int = 128, tau: float | None = None, dtype=np.float64,
                        p_cast=None, row_index: np.ndarray | None = None,
                        scores: np.ndarray | None = None, max_history: bool = False):
    """The streaming recurrence over key blocks, for one (batch, head) per call
    or for [..., N, d] batched inputs.

    Per key block: S = Q K_b^T (raw), block max on the raw scores, a candidate
    max; with ``tau`` given, the running max only moves when it would grow by
    more than tau in log2 units of the scaled score, otherwise the stale max is
    kept and the correction factor is 1. P = exp2((S - m) * s * log2 e), the
    running sum and the accumulator are multiplied by the correction factor and
    P's row sum / P V are added. After the last block O is divided by the sum
    once, and LSE = m*s + ln(sum).

    Causal: key blocks entirely above the diagonal of the query rows are
    skipped; the straddling block is masked to -inf for j > i.

    ``dtype`` runs the same recurrence in a narrower float type (inputs cast to
    it), for the precision-band checks; ``p_cast`` (optional) rounds P to the
    matrix-multiply input type before P V while the sum uses the unrounded P
    (the reading of "FlashAttention-4's Softmax Tricks", section "Conditional
    rescaling": the sum is taken from fp32 P, and P is cast to the MMA input
    type). ``row_index`` gives the sequence positions of q's rows (default
    0 .. n_q - 1) for the causal mask. ``scores`` (optional) gives the raw
    scores Q K^T [..., n_q, n_k] directly, for simulations over a chosen score
    distribution; q and k are then not used (pass None). Returns (O, LSE, fired) where fired
    [..., N, nblocks] is True where the running max moved (block 0 included).
    With ``max_history`` a fourth array [..., N, nblocks] is returned: the
    reference max (raw score units) that each block's P was taken against (a
    causal row's P is zero on keys it cannot see, whatever this value), -inf
    for blocks past the last causal row.
    """
    f = dtype
    v = np.asarray(v).astype(f)
    if scores is None:
        q = np.asarray(q).astype(f)
        k = np.asarray(k).astype(f)
        n_q, n_k = q.shape[-2], k.shape[-2]
        lead = q.shape[:-2]
    else:
        scores = np.asarray(scores).astype(f)
        n_q, n_k = scores.shape[-2], scores.shape[-1]
        lead = scores.shape[:-2]
    sl2 = f(scale * LOG2E)
    m = np.full(lead + (n_q,), -np.inf, dtype=f)
    l = np.zeros(lead + (n_q,), dtype=f)
    o = np.zeros(lead + (n_q, v.shape[-1]), dtype=f)
    nblocks = (n_k + block - 1) // block
    fired = np.zeros(lead + (n_q, nblocks), dtype=bool)
    m_used = np.full(lead + (n_q, nblocks), -np.inf, dtype=np.float64)
    rows = np.arange(n_q) if row_index is None else np.asarray(row_index)
    last_row = int(rows.max()) if rows.size else -1
    for jb in range(nblocks):
        j0, j1 = jb * block, min(n_k, (jb + 1) * block)
        if causal and j0 > last_row:
            break                                   # every remaining block is above the diagonal
        if scores is None:
            s = q @ np.swapaxes(k[..., j0:j1, :], -1, -2)   # raw scores [..., n_q, bk]
        else:
            s = scores[..., j0:j1]
        if causal and j1 - 1 > 0:
            cols = np.arange(j0, j1)
            s = np.where(cols[None, :] <= rows[:, None], s, f(-np.inf))
        bmax = s.max(axis=-1)
        cand = np.maximum(m, bmax)
        with np.errstate(invalid="ignore"):
            growth = (cand - m) * sl2              # +inf on the first block, nan if both -inf
        if tau is None:
            move = cand > m
        else:
            move = ~(growth <= f(tau))             # keep the stale max iff it grew by <= tau
        move &= np.isfinite(cand)
        m_new = np.where(move, cand, m)
        with np.errstate(invalid="ignore"):
            corr = np.where(move, np.exp2((m - m_new) * sl2), f(1.0))
        corr = np.where(np.isfinite(m), corr, f(0.0)).astype(f)
        with np.errstate(invalid="ignore"):
            p = np.exp2((s - m_new[..., None]) * sl2)
        p = np.where(np.isfinite(s), p, f(0.0)).astype(f)
        l = (corr * l + p.sum(axis=-1)).astype(f)
        pv = p if p_cast is None else np.asarray(p_cast(p)).astype(f)
        o = (corr[..., None] * o + pv @ v[..., j0:j1, :]).astype(f)
        m = m_new.astype(f)
        fired[..., jb] = move
        m_used[..., jb] = m
    out = o / l[..., None]
    lse = m.astype(np.float64) * scale + np.log(l.astype(np.float64))
    if max_history:
        return out, lse, fired, m_used
    return out, lse, fired


def blockwise_attention_blockmax(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool,
                                 scale: float, block: int = 64) -> tuple[np.ndarray, np.ndarray]:
    """The per-block-max form of the recurrence (float64).

    Each key block keeps its own max m_b and local sum l_b; the running state
    and the block are brought to the common max with two factors,
    exp(m - m_new) and exp(m_b - m_new), as in "Lecture 2 - Online Softmax and
    Numerical Correctness", sections "Combining two blocks exactly" and
    "Carrying the output along". Scores are scaled before the max here, unlike
    ``blockwise_attention``; the two readings agree for s > 0.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_q, n_k = q.shape[-2], k.shape[-2]
    lead = q.shape[:-2]
    m = np.full(lead + (n_q,), -np.inf)
    l = np.zeros(lead + (n_q,))
    o = np.zeros(lead + (n_q, v.shape[-1]))
    rows = np.arange(n_q)
    for j0 in range(0, n_k, block):
        j1 = min(n_k, j0 + block)
        s = scale * (q @ np.swapaxes(k[..., j0:j1, :], -1, -2))
        if causal:
            cols = np.arange(j0, j1)
            s = np.where(cols[None, :] <= rows[:, None], s, -np.inf)
        m_b = s.max(axis=-1)
        with np.errstate(invalid="ignore"):
            p_b = np.exp(s - m_b[..., None])
        p_b = np.where(np.isfinite(s), p_b, 0.0)
        l_b = p_b.sum(axis=-1)
        m_new = np.maximum(m, m_b)
        with np.errstate(invalid="ignore"):
            a_old = np.where(np.isfinite(m), np.exp(m - m_new), 0.0)
            a_blk = np.where(np.isfinite(m_b), np.exp(m_b - m_new), 0.0)
        o = a_old[..., None] * o + a_blk[..., None] * (p_b @ v[..., j0:j1, :])
        l = a_old * l + a_blk * l_b
        m = m_new
    return o / l[..., None], m + np.log(l)


def lse_combine(m_a: np.ndarray, l_a: np.ndarray, m_b: np.ndarray, l_b: np.ndarray):
    """Exact merge of two blocks' (max, shifted sum) statistics: the combined max
    is the larger one and each sum is brought to it by exp of the max gap
    ("Lecture 2 - Online Softmax and Numerical Correctness", section
    "Combining two blocks exactly")."""
    m = np.maximum(m_a, m_b)
    return m, np.exp(m_a - m) * l_a + np.exp(m_b - m) * l_b


def combine_partials(o_parts: np.ndarray, lse_parts: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Merge attention results computed over disjoint sets of keys into the
    result over their union, float64.

    o_parts [P, ..., R, dv]: each part's normalised output O_p; lse_parts
    [P, ..., R]: its log-sum-exp LSE_p = m_p + ln l_p of the scaled scores.
    "Lecture 2 - Online Softmax and Numerical Correctness", section "Combining
    two blocks exactly": the merged max is m = max_p m_p and the merged sum is
    l = sum_p exp(m_p - m) l_p. Each part enters with the statistics
    (m_p, l_p) = (LSE_p, 1), which have the same log-sum-exp, so l = sum_p
    exp(LSE_p - m), LSE = m + ln l, and the merged numerator sum_p exp(m_p - m)
    l_p O_p divided by l gives O. A part with LSE_p = -inf (no keys) adds
    nothing; a row whose parts are all -inf gets O = 0 and LSE = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    if o_parts.shape[:-1] != lse_parts.shape:
        raise ValueError(f"bad shapes o{o_parts.shape} lse{lse_parts.shape}")
    m = lse_parts.max(axis=0)
    live = np.isfinite(m)
    w = np.exp(lse_parts - np.where(live, m, 0.0))        # exp(m_p - m) l_p with l_p = 1
    l = w.sum(axis=0)
    with np.errstate(invalid="ignore", divide="ignore"):
        o = (w[..., None] * o_parts).sum(axis=0) / l[..., None]
        lse = m + np.log(l)
    o = np.where(live[..., None], o, 0.0)
    lse = np.where(live, lse, -np.inf)
    return o, lse
