"""Pins for the software-exp2 model (CPU only).

The accuracy statistics the first page prints for degree 3 over [-20, 8] pin
the scalar C model; closed forms pin the range reduction and the exponent add.
"""
import numpy as np
import pytest

from attn_inputs import uniform_fp32
from conftest import read_golden_kv
from oracle import cmodel, exp2_model


@pytest.fixture(scope="module")
def sweep():
    g = read_golden_kv("sw_exp2_accuracy.txt")
    x = uniform_fp32(int(g["inputs"]), g["domain_lo"], g["domain_hi"], seed=0)
    return g, x


def _check_table(g, acc):
    # printed to 3 significant digits; bit-identical share printed as 99.000 %
    assert round(acc["max_rel"], 7) == pytest.approx(g["max_rel"], abs=5e-8)
    assert round(acc["mean_rel"], 7) == pytest.approx(g["mean_rel"], abs=5e-8)
    assert 100 * acc["bf16_identical"] == pytest.approx(g["bf16_identical_pct"], abs=0.05)
    assert 100 * acc["bf16_within_1ulp"] == g["bf16_within_1ulp_pct"]


def test_c_model_reproduces_accuracy_table(sweep):
    g, x = sweep
    _check_table(g, exp2_model.accuracy(x, cmodel.exp2_emulated(x)))


def test_integers_are_exact_powers():
    model = cmodel.exp2_emulated
    # frac = 0, so the polynomial returns its constant term 1 and the exponent
    # add must give exactly 2^n
    n = np.arange(-126, 128, dtype=np.float32)
    y = model(n)
    assert np.array_equal(y.astype(np.float64), np.exp2(n.astype(np.float64)))


def test_clamp_gives_zero():
    model = cmodel.exp2_emulated
    # x <= -127 clamps to -127: 1.0 shifted down by 127 binades is +0 exactly,
    # so a masked score (-inf) contributes nothing
    y = model(np.array([-np.inf, -1e30, -200.0, -127.0], dtype=np.float32))
    assert np.all(y == 0.0) and not np.any(np.signbit(y))


def test_half_integers():
    model = cmodel.exp2_emulated
    # 2^(n + 1/2) = sqrt(2) * 2^n within the degree-3 relative error
    n = np.arange(-20, 8, dtype=np.float32) + np.float32(0.5)
    y = model(n).astype(np.float64)
    rel = np.abs(y / np.exp2(n.astype(np.float64)) - 1.0)
    assert rel.max() < 8.8e-5
    # the fraction is the same for all n, so every result has the same mantissa
    mant = (y / np.exp2(np.floor(n.astype(np.float64))))
    assert np.all(mant == mant[0])


def test_c_model_is_fused():
    # one input where a double-rounded multiply-add and a fused one differ would
    # show up as a mismatch; here check the fused model against exact rational
    # evaluation of the Horner steps on a few fractions
    from fractions import Fraction
    c = [Fraction(v) for v in exp2_model.POLY3]
    for xf in (0.1, 0.33, 0.5, 0.77, 0.999):
        x = np.float32(xf)
        f = Fraction(float(x))
        p = np.float32(c[3])
        for coef in (c[2], c[1], c[0]):
            p = np.float32(float(Fraction(float(p)) * f + coef))  # one rounding of the exact value
        y = cmodel.exp2_emulated(np.array([x]))[0]
        assert y == p
