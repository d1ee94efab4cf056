"""Software exp2 on the FMA pipe: NumPy model and accuracy statistics.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The method ("FlashAttention-4's Softmax Tricks", section "The emulated exp2";
"Software-Emulated Exponential" on the KernelWiki page) splits
2^x = 2^floor(x) * 2^frac(x):

  1. clamp x from below at -127;
  2. add 2^23 + 2^22 with rounding toward -inf, which leaves floor(x) as an
     integer in the low mantissa bits of the sum;
  3. subtract the constant again (exact) and take frac = x - floor(x) in [0, 1);
  4. evaluate 2^frac with a degree-3 polynomial in Horner form (3 FMAs), using
     the Sollya fpminimax coefficients printed on the first page (constant
     term 1);
  5. add floor(x) << 23 to the polynomial's bit pattern as a 32-bit integer,
     which multiplies it by 2^floor(x) (floor(x) taken mod 512).

This NumPy model is for the statistics only. Its multiply-add is "exact product
in float64, one float64 add, one rounding to float32", which double-rounds in
rare cases; the bit-exact scalar model with a true fused multiply-add is
``exp2_model.c`` (``oracle.cmodel``).
"""
from __future__ import annotations

import numpy as np

# Degree-3 coefficients, constant term first ("FlashAttention-4's Softmax
# Tricks", section "The emulated exp2", the P3 tuple: Sollya fpminimax for
# relative error with p0 = 1). Degree 4 and 5 coefficients are not printed.
POLY3 = (1.0, 0.695146143436431884765625, 0.227564394474029541015625,
         0.077119089663028717041015625)
ROUND_MAGIC = float(2 ** 23 + 2 ** 22)
CLAMP_LO = -127.0


def _mul_add_f32(a: np.ndarray, b: np.ndarray, c: float) -> np.ndarray:
    # float32*float32 is exact in float64; the sum is rounded, then narrowed.
    return (a.astype(np.float64) * b.astype(np.float64) + np.float64(np.float32(c))).astype(np.float32)


def exp2_emulated(x) -> np.ndarray:
    """Software exp2 of float32 inputs, float32 result (NumPy model)."""
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(CLAMP_LO))
    # Step 2 leaves MAGIC + floor(x) in the sum; for x in [-127, 2^22) that sum is
    # an exactly representable float32, so form it directly from floor(x).
    whole = np.floor(x.astype(np.float64))
    rounded = (whole + ROUND_MAGIC).astype(np.float32)
    frac = x - (rounded - np.float32(ROUND_MAGIC))          # exact, in [0, 1)
    poly = np.full(x.shape, np.float32(POLY3[-1]), dtype=np.float32)
    for coef in reversed(POLY3[:-1]):
        poly = _mul_add_f32(poly, frac, coef)
    with np.errstate(over="ignore"):
        shifted = rounded.view(np.int32) << np.int32(23)    # keeps floor(x) mod 512
        bits = shifted + poly.view(np.int32)                # 32-bit wrap-around add
    return bits.view(np.float32)


def bf16_round(y) -> np.ndarray:
    """Round float values (float32 or float64) to the nearest bfloat16, ties to
    even, returned as float64. Done from the value itself (no float32 step)."""
    y = np.asarray(y, dtype=np.float64)
    mant, expo = np.frexp(y)                                # y = mant * 2^expo, |mant| in [0.5, 1)
    return np.ldexp(np.rint(mant * 256.0) / 256.0, expo)    # 8 significant bits


def bf16_bits(y) -> np.ndarray:
    """bfloat16 bit patterns (as int32) of bf16_round(y), for positive finite y."""
    r = bf16_round(y).astype(np.float32)                    # exact: bf16 values fit float32
    return (r.view(np.int32) >> 16).astype(np.int32)


def accuracy(x, y) -> dict:
    """Accuracy of approximations y ~ 2^x against float64 exp2, in the four
    columns of the accuracy table on "FlashAttention-4's Softmax Tricks",
    section "The emulated exp2": max and mean float32 relative error, share of
    inputs whose bf16 rounding is bit-identical to the exact value's bf16
    rounding, and share within one bf16 ulp."""
    x = np.asarray(x, dtype=np.float32)
    y = np.asarray(y, dtype=np.float32)
    exact = np.exp2(x.astype(np.float64))
    rel = np.abs(y.astype(np.float64) - exact) / exact
    dbits = np.abs(bf16_bits(y) - bf16_bits(exact))
    return {
        "max_rel": float(rel.max()),
        "mean_rel": float(rel.mean()),
        "bf16_identical": float((dbits == 0).mean()),
        "bf16_within_1ulp": float((dbits <= 1).mean()),
    }
