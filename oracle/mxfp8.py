"""MXFP8 (E4M3 payload, E8M0 block scales) quantiser -- TEST INFRASTRUCTURE ONLY.

"PyTorch FlashAttention-4 adds MXFP8 block-scaled forward and backward for
Blackwell", section "Quantization along both axes and jagged tensors": Q and K
are quantised along the embedding dimension and V along the sequence, with
square 32 x 32 blocks, each block sharing one E8M0 (power of two) scale.

The pages do not state the scale rule. The reading taken here: a block's scale
is the smallest power of two 2^e with amax / 2^e <= 448 (the largest finite
E4M3 value), so the block's largest element lands in the top binade of E4M3
without saturating; an all-zero block takes e = 0. Elements are divided by 2^e
(exact) and rounded to E4M3, nearest with ties to even, saturating at +-448.

The same page, section "Softmax conversion and unroll-KV", converts P (the
probabilities, all in [0, 1]) to MXFP8 inside the kernel for the P V product,
one E8M0 scale per 32 consecutive keys of a row: ``p_to_mxfp8`` applies the
same scale rule to each such group of a row (the group's amax is the largest
P in it). The same section notes that a constant scale for P also works,
since softmax keeps P in [0, 1]: ``p_to_mxfp8_constant`` divides every P by
2^-8 (P = 1 lands on 256, inside E4M3's 448) and rounds it to E4M3.

E4M3 (the OCP "E4M3FN" encoding): 1 sign bit, 4 exponent bits with bias 7,
3 mantissa bits; exponent field 0 encodes subnormals m * 2^-9; the code
S.1111.111 is NaN and there are no infinities, so the largest finite value is
1.75 * 2^8 = 448 and the smallest subnormal 2^-9.

"FlashAttention-4's Softmax Tricks", section "Where 'exact' breaks: P in
FP8", compares P held in E4M3 with P held in E5M2 under a constant 2^8
offset: E5M2 (OCP): 1 sign bit, 5 exponent bits with bias 15, 2 mantissa
bits; exponent field 0 encodes subnormals m * 2^-16, exponent field 31 the
infinities and NaNs, so the largest finite value is 1.75 * 2^15 = 57344.
``p_to_fp8_constant`` converts P to either format with the constant scale;
conversions saturate to the largest finite value (the kernels' "satfinite").
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BLOCK = 32


def e4m3_decode(codes) -> np.ndarray:
    """Values (float64) of E4M3 byte codes; NaN for the NaN codes."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


E5M2_MAX = 57344.0


def e5m2_decode(codes) -> np.ndarray:
    """Values (float64) of E5M2 byte codes; +-inf and NaN for exponent field 31."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 2) & 0x1F
    m = c & 0x3
    mag = np.where(e == 0, m * 2.0 ** -16, (1.0 + m / 4.0) * np.exp2(e - 15.0))
    mag = np.where(e == 31, np.where(m == 0, np.inf, np.nan), mag)
    return sign * mag


def _round_to_codes(x, codes: np.ndarray, values: np.ndarray, vmax: float) -> np.ndarray:
    """Nearest of the ascending non-negative finite ``values`` (with their byte
    ``codes``), ties to the even code (even mantissa), magnitudes above vmax
    saturating to vmax; the sign bit (0x80) is kept, also for a zero result."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.minimum(np.abs(x), vmax)
    # index of the largest representable value <= mag
    lo = np.clip(np.searchsorted(values, mag, side="right") - 1, 0, len(values) - 1)
    hi = np.minimum(lo + 1, len(values) - 1)
    vlo, vhi = values[lo], values[hi]
    dlo, dhi = mag - vlo, vhi - mag
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi != lo) & ((codes[lo] & 1) == 1))
    code = np.where(pick_hi, codes[hi], codes[lo])
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


_POS_CODES = np.arange(0, 0x7F)      # E4M3 non-negative finite codes 0x00 .. 0x7E, ascending values
_POS_VALUES = e4m3_decode(_POS_CODES)
_E5_CODES = np.arange(0, 0x7C)       # E5M2 non-negative finite codes 0x00 .. 0x7B
_E5_VALUES = e5m2_decode(_E5_CODES)


def e4m3_encode(x) -> np.ndarray:
    """Round float values to E4M3 codes: nearest, ties to the even code
    (even mantissa), magnitudes above 448 saturate to 448. NaN is not expected."""
    return _round_to_codes(x, _POS_CODES, _POS_VALUES, E4M3_MAX)


def e5m2_encode(x) -> np.ndarray:
    """Round float values to E5M2 codes: nearest, ties to the even code,
    magnitudes above 57344 saturate to 57344. NaN is not expected."""
    return _round_to_codes(x, _E5_CODES, _E5_VALUES, E5M2_MAX)


def e8m0_exponent(amax) -> np.ndarray:
    """Smallest integer e with amax <= 448 * 2^e (0 for amax == 0)."""
    # amax = m * 2^E with m in [0.5, 1) and 448 = 0.875 * 2^9, so
    # amax <= 448 * 2^e  <=>  e >= E - 9 when m <= 0.875, else e >= E - 8.
    a = np.asarray(amax, dtype=np.float64)
    m, E = np.frexp(a)
    e = np.where(m <= 0.875, E - 9, E - 8)
    return np.where(a > 0, e, 0).astype(np.int64)


def quantize_blocks(x: np.ndarray) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Quantise [..., R, C] with one scale per 32 x 32 block (R, C padded up to
    multiples of 32 with zeros for the amax only).

    Returns (codes uint8 [..., R, C], e int64 [..., ceil(R/32), ceil(C/32)],
    dequantised float64 [..., R, C] = e4m3_decode(codes) * 2^e)."""
    x = np.asarray(x, dtype=np.float64)
    *lead, R, C = x.shape
    rb, cb = -(-R // BLOCK), -(-C // BLOCK)
    pad = np.zeros((*lead, rb * BLOCK, cb * BLOCK))
    pad[..., :R, :C] = x
    blocks = pad.reshape(*lead, rb, BLOCK, cb, BLOCK)
    amax = np.abs(blocks).max(axis=(-3, -1))                     # [..., rb, cb]
    e = e8m0_exponent(amax)
    scale_full = np.repeat(np.repeat(np.exp2(e.astype(np.float64)), BLOCK, axis=-2), BLOCK, axis=-1)
    scaled = pad / scale_full
    codes_full = e4m3_encode(scaled)
    codes = codes_full[..., :R, :C]
    deq = e4m3_decode(codes) * scale_full[..., :R, :C]
    return codes, e, deq


def p_to_mxfp8(p: np.ndarray) -> np.ndarray:
    """Values of P [..., rows, keys] after the MXFP8 conversion: each run of 32
    consecutive keys of a row (from key 0 of the block) shares one E8M0 scale
    chosen by the rule above from the run's largest P, and every P is divided
    by it and rounded to E4M3. Returns the dequantised values (float64)."""
    p = np.asarray(p, dtype=np.float64)
    out = np.empty_like(p)
    for g0 in range(0, p.shape[-1], BLOCK):
        run = p[..., g0:g0 + BLOCK]
        scale = np.exp2(e8m0_exponent(np.abs(run).max(axis=-1)).astype(np.float64))[..., None]
        out[..., g0:g0 + BLOCK] = e4m3_decode(e4m3_encode(run / scale)) * scale
    return out


P_CONST_EXP = -8


def p_to_mxfp8_constant(p: np.ndarray) -> np.ndarray:
    """Values of P after conversion to E4M3 with the constant scale 2^-8
    (float64): P / 2^-8 rounded to E4M3 (nearest even, saturating at 448),
    times 2^-8."""
    return p_to_fp8_constant(p, "e4m3")


def p_to_fp8_constant(p: np.ndarray, fmt: str) -> np.ndarray:
    """Values of P after conversion to ``fmt`` ("e4m3" or "e5m2") with the
    constant scale 2^-8 (the 2^8 offset of "FlashAttention-4's Softmax
    Tricks", section "Where 'exact' breaks: P in FP8"): P / 2^-8 rounded to the
    format (nearest even, saturating at its largest finite value), times 2^-8.
    A stale maximum lets P reach 2^tau: E4M3 saturates once 2^(tau + 8) > 448,
    E5M2 once 2^(tau + 8) > 57344."""
    scale = 2.0 ** P_CONST_EXP
    x = np.asarray(p, dtype=np.float64) / scale
    if fmt == "e4m3":
        return e4m3_decode(e4m3_encode(x)) * scale
    if fmt == "e5m2":
        return e5m2_decode(e5m2_encode(x)) * scale
    raise ValueError(f"unknown FP8 format {fmt!r}")
