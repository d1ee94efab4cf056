"""Float64 attention backward -- TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The pages do not print the backward equations; they say what it consumes and
how it is organised: "Lecture 2 - Online Softmax and Numerical Correctness",
section "Use it in the real stack", notes that the forward's per-row
log-sum-exp side output is what makes the backward pass cheap, and "PyTorch
FlashAttention-4 adds MXFP8 block-scaled forward and backward for Blackwell",
section "TMEM allocation and scale factor placement", describes a backward of
five matrix products with dK and dV accumulated per key tile.

The reading taken here is the plain gradient of the forward's definition
O = softmax(s Q K^T [causal mask]) V for an upstream gradient dO:

  P  = exp(s Q K^T - LSE)          the probabilities, rebuilt from the LSE
  dV = P^T dO
  dP = dO V^T
  D  = rowsum(dO * O)              = rowsum(P * dP), since O = P V
  dS = P * (dP - D)                the chain rule through the row softmax
  dQ = s dS K,   dK = s dS^T Q

(the five products: S, dP, dV, dK, dQ). Masked scores have P = 0, so they
contribute nothing. Everything is float64, one (batch, head) at a time, rows
in chunks only to bound memory.

The MXFP8 backward (``attention_bwd_mxfp8``) is the same method with every
product's inputs in MXFP8. The page on the MXFP8 extension, section
"Quantization along both axes and jagged tensors", quantises Q, K and dO in
square 32 x 32 blocks, so that one E4M3 payload serves both products that read
a tensor (along d for S and dP, along the sequence for dV, dK and dQ), and
quantises dS the same way so that dK and dQ read one representation. Its
section "Softmax conversion and unroll-KV" converts P online and notes that a
constant scale for P is robust, P being in [0, 1]. The readings taken here:
  * V is quantised in the same square blocks (it enters only dP, along d);
  * P enters dV as E4M3 with the constant scale 2^-8 (``p_to_mxfp8_constant``);
    dS = P (dP - D) takes the unrounded P;
  * dS is rounded in 32 x 32 blocks of (queries, keys) by the block rule of
    ``quantize_blocks``, the blocks starting at query 0 and key 0, entries
    outside the sequence or masked being zero;
  * D = rowsum(dO * O) takes the dequantised dO, the one dP is built from.
"""
from __future__ import annotations

import numpy as np

from oracle.mxfp8 import p_to_mxfp8_constant, quantize_blocks


def attention_bwd_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, o: np.ndarray, do: np.ndarray,
                       lse: np.ndarray, causal: bool, scale: float, row_chunk: int = 512,
                       p_cast=None, ds_cast=None, dv_p_cast=None) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """dQ, dK, dV (float64) of one (batch, head): q [N, d], k [N, d], v [N, dv],
    o and do [N, dv], lse [N] (natural log of the scaled scores' row sums).

    ``p_cast`` / ``ds_cast`` (optional) round P before it enters dV and dS,
    and dS before it enters dQ and dK, to a matrix-multiply input type: the
    same method in the precision a kernel feeds its tensor cores, for tight
    parity checks (the forward's reading: P takes the MMA input type).
    ``dv_p_cast`` (optional) rounds only the P that enters dV; dS then takes
    P as it was. ``row_chunk`` must be a multiple of 32 when ``ds_cast``
    rounds in 32-row blocks."""
    q, k, v, o, do, lse = (np.asarray(x, dtype=np.float64) for x in (q, k, v, o, do, lse))
    n = q.shape[0]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    d_row = (do * o).sum(axis=1)                     # D_i
    for i0 in range(0, n, row_chunk):
        i1 = min(n, i0 + row_chunk)
        s = scale * (q[i0:i1] @ k.T)                 # [R, N] scaled scores
        p = np.exp(s - lse[i0:i1, None])
        if causal:
            j = np.arange(k.shape[0])[None, :]
            p = np.where(j <= np.arange(i0, i1)[:, None], p, 0.0)
        if p_cast is not None:
            p = np.asarray(p_cast(p), dtype=np.float64)
        p_dv = p if dv_p_cast is None else np.asarray(dv_p_cast(p), dtype=np.float64)
        dv += p_dv.T @ do[i0:i1]
        dp = do[i0:i1] @ v.T
        ds = p * (dp - d_row[i0:i1, None])
        if ds_cast is not None:
            ds = np.asarray(ds_cast(ds), dtype=np.float64)
        dq[i0:i1] = scale * (ds @ k)
        dk += scale * (ds.T @ q[i0:i1])
    return dq, dk, dv


def attention_bwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, o: np.ndarray, do: np.ndarray,
                  lse: np.ndarray, causal: bool, scale: float) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """dQ, dK, dV (float64) for [B, H, N, d] inputs and lse [B, H, N]."""
    q = np.asarray(q)
    B, H = q.shape[:2]
    out = [np.empty(np.shape(x), dtype=np.float64) for x in (q, k, v)]
    for b in range(B):
        for h in range(H):
            g = attention_bwd_head(q[b, h], k[b, h], v[b, h], o[b, h], do[b, h], lse[b, h], causal, scale)
            for dst, src in zip(out, g):
                dst[b, h] = src
    return out[0], out[1], out[2]


def attention_bwd_abs_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, o: np.ndarray, do: np.ndarray,
                           lse: np.ndarray, causal: bool, scale: float,
                           row_chunk: int = 512) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """The same three products with every factor replaced by its absolute
    value: s |dS| |K|, s |dS|^T |Q|, |P|^T |dO| (float64). They bound how far
    a rounding of P or dS by a relative epsilon can move each output element,
    which is how the GPU tests size their tolerances."""
    q, k, v, o, do, lse = (np.asarray(x, dtype=np.float64) for x in (q, k, v, o, do, lse))
    n = q.shape[0]
    aq = np.zeros_like(q)
    ak = np.zeros_like(k)
    av = np.zeros_like(v)
    d_row = (do * o).sum(axis=1)
    for i0 in range(0, n, row_chunk):
        i1 = min(n, i0 + row_chunk)
        p = np.exp(scale * (q[i0:i1] @ k.T) - lse[i0:i1, None])
        if causal:
            j = np.arange(k.shape[0])[None, :]
            p = np.where(j <= np.arange(i0, i1)[:, None], p, 0.0)
        av += p.T @ np.abs(do[i0:i1])
        ds = np.abs(p * (do[i0:i1] @ v.T - d_row[i0:i1, None]))
        aq[i0:i1] = scale * (ds @ np.abs(k))
        ak += scale * (ds.T @ np.abs(q[i0:i1]))
    return aq, ak, av



def attention_bwd_mxfp8_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, o: np.ndarray, do: np.ndarray,
                             lse: np.ndarray, causal: bool, scale: float) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """dQ, dK, dV (float64) of one (batch, head) in MXFP8: q, k, v, do [N, d]
    are the unquantised inputs (rounded here in 32 x 32 blocks), o [N, d] the
    forward's output and lse [N] its LSE, both taken as given."""
    qd, kd, vd, dod = (quantize_blocks(np.asarray(x, dtype=np.float64))[2] for x in (q, k, v, do))
    return attention_bwd_head(qd, kd, vd, o, dod, lse, causal, scale, row_chunk=512,
                              ds_cast=lambda ds: quantize_blocks(ds)[2], dv_p_cast=p_to_mxfp8_constant)


def attention_bwd_mxfp8(q: np.ndarray, k: np.ndarray, v: np.ndarray, o: np.ndarray, do: np.ndarray,
                        lse: np.ndarray, causal: bool, scale: float) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """``attention_bwd_mxfp8_head`` over [B, H, N, d] inputs and lse [B, H, N]."""
    q = np.asarray(q)
    B, H = q.shape[:2]
    out = [np.empty(np.shape(x), dtype=np.float64) for x in (q, k, v)]
    for b in range(B):
        for h in range(H):
            g = attention_bwd_mxfp8_head(q[b, h], k[b, h], v[b, h], o[b, h], do[b, h], lse[b, h], causal, scale)
            for dst, src in zip(out, g):
                dst[b, h] = src
    return out[0], out[1], out[2]


def attention_bwd_mxfp8_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, o: np.ndarray, do: np.ndarray,
                             lse: np.ndarray, causal: bool, scale: float, q_rows, k_rows) -> dict:
    """``attention_bwd_mxfp8_head`` at chosen rows only, for long sequences:
    dQ at the query rows ``q_rows`` and dK, dV at the key rows ``k_rows`` of
    one head (inputs as there). dS is rounded in the same 32 x 32 blocks, so a
    query row needs the dS rows of its 32-row block against every key, and a
    key row the dS columns of its 32-key block against every query; those are
    the only parts computed. Returns a dict with dq, dk, dv (rows in the given
    order) and the rounded dS rows ("ds_rows"), dS columns ("ds_cols") and P
    columns ("p_cols") they were summed from."""
    qd, kd, vd, dod = (quantize_blocks(np.asarray(x, dtype=np.float64))[2] for x in (q, k, v, do))
    o, lse = np.asarray(o, dtype=np.float64), np.asarray(lse, dtype=np.float64)
    n = qd.shape[0]
    d_row = (dod * o).sum(axis=1)
    out = {"dq": [], "ds_rows": [], "dk": [], "dv": [], "ds_cols": [], "p_cols": []}
    rows_of_block = {}
    for i in q_rows:
        rows_of_block.setdefault(int(i) // 32, []).append(int(i))
    dq_at = {}
    for b, rows in rows_of_block.items():
        r0, r1 = 32 * b, min(n, 32 * b + 32)
        p = np.exp(scale * (qd[r0:r1] @ kd.T) - lse[r0:r1, None])
        if causal:
            p = np.where(np.arange(n)[None, :] <= np.arange(r0, r1)[:, None], p, 0.0)
        ds8 = quantize_blocks(p * (dod[r0:r1] @ vd.T - d_row[r0:r1, None]))[2]
        for i in rows:
            dq_at[i] = (scale * (ds8[i - r0] @ kd), ds8[i - r0])
    for i in q_rows:
        out["dq"].append(dq_at[int(i)][0])
        out["ds_rows"].append(dq_at[int(i)][1])
    cols_of_block = {}
    for j in k_rows:
        cols_of_block.setdefault(int(j) // 32, []).append(int(j))
    dk_at = {}
    for c, cols in cols_of_block.items():
        c0, c1 = 32 * c, min(n, 32 * c + 32)
        p = np.exp(scale * (qd @ kd[c0:c1].T) - lse[:, None])
        if causal:
            p = np.where(np.arange(c0, c1)[None, :] <= np.arange(n)[:, None], p, 0.0)
        ds8 = quantize_blocks(p * (dod @ vd[c0:c1].T - d_row[:, None]))[2]
        p8 = p_to_mxfp8_constant(p)
        for j in cols:
            dk_at[j] = (scale * (ds8[:, j - c0] @ qd), p8[:, j - c0] @ dod, ds8[:, j - c0], p8[:, j - c0])
    for j in k_rows:
        dk, dv, dsc, pc = dk_at[int(j)]
        out["dk"].append(dk)
        out["dv"].append(dv)
        out["ds_cols"].append(dsc)
        out["p_cols"].append(pc)
    return {key: np.array(val) for key, val in out.items()}
