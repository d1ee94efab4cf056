"""Lagging-max rescale simulator -- TEST INFRASTRUCTURE ONLY.

Restates the rule of "FlashAttention-4's Softmax Tricks", section "Conditional
rescaling, and when it's exact": per key block the candidate max is
max(m_old, block max); the rescale fires only when the scaled growth exceeds
tau (log2 units), otherwise the stale max is kept and the correction factor is
1. Scores here are already in log2 units of the scaled score, so the growth is
compared to tau directly.

``rescale_rates`` returns the two statistics that page tabulates: the share of
(row, block) pairs where a row's max moved, and the share of (warp, block)
pairs where any of a warp's 32 rows moved. Block 0 is left out (its "rescale"
multiplies an empty accumulator).
"""
from __future__ import annotations

import numpy as np


def fired_matrix(scores_log2: np.ndarray, block: int = 128, tau: float = 0.0) -> np.ndarray:
    """bool [rows, nblocks]: where the running max of each row moved."""
    s = np.asarray(scores_log2, dtype=np.float64)
    rows, n_keys = s.shape
    nblocks = n_keys // block
    m = np.full(rows, -np.inf)
    fired = np.zeros((rows, nblocks), dtype=bool)
    for jb in range(nblocks):
        cand = np.maximum(m, s[:, jb * block:(jb + 1) * block].max(axis=1))
        grew = cand - m                      # +inf on block 0
        move = grew > tau                    # keep the stale max iff growth <= tau
        m = np.where(move, cand, m)
        fired[:, jb] = move
    return fired


def rescale_rates(scores_log2: np.ndarray, block: int = 128, tau: float = 0.0,
                  warp: int = 32) -> tuple[float, float]:
    """(rows %, warps %) of rescale events, block 0 excluded."""
    f = fired_matrix(scores_log2, block, tau)[:, 1:]
    rows, nb = f.shape
    per_warp = f.reshape(rows // warp, warp, nb).any(axis=1)
    return 100.0 * float(f.mean()), 100.0 * float(per_warp.mean())
