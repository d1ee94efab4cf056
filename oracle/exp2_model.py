"""Software exp2: accuracy statistics, and the bf16 rounding they need.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The software exp2 itself is modelled once, in scalar C (``exp2_model.c``,
loaded by ``oracle.cmodel``): a true fused multiply-add and one add rounded
toward minus infinity, so it gives the device's bits. That model follows the
method of "FlashAttention-4's Softmax Tricks", section "The emulated exp2", and
"Software-Emulated Exponential" on the KernelWiki page. The input is clamped
at -127. The integer part comes from a rounding-down add of 2^23 + 2^22, and
the fraction from subtracting it back. A degree-3 polynomial (the printed
coefficients below, constant term 1) gives 2^frac in Horner form. Shifting the
integer into the exponent field by an integer add finishes it.

This module holds what the tests compare that model (and the device) against:
the four accuracy columns the page prints for it, measured against float64
exp2, and a bf16 rounding taken from the value itself.
"""
from __future__ import annotations

import numpy as np

# Degree-3 coefficients, constant term first, as printed on "FlashAttention-4's
# Softmax Tricks", section "The emulated exp2" (Sollya fpminimax for relative
# error with the constant term fixed at 1). Degree 4 and 5 are not printed.
POLY3 = (1.0, 0.695146143436431884765625, 0.227564394474029541015625,
         0.077119089663028717041015625)


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
