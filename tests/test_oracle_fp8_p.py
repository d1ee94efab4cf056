"""Pins for P held in FP8 (CPU only): the E5M2 codec against its definition,
and the output-error table of "FlashAttention-4's Softmax Tricks", section
"Where 'exact' breaks: P in FP8", reproduced with the oracle's streaming
recurrence (lagging maximum, row sum from the unrounded P) and its FP8
conversions under the constant 2^8 offset."""
import math

import numpy as np
import pytest

from attn_inputs import fp8_sim_values, rescale_scores
from conftest import read_golden_table
from oracle import mxfp8 as M
from oracle.attention import blockwise_attention

TABLE = read_golden_table("fp8_p_offset.txt")


def test_e5m2_decode_is_the_top_byte_of_binary16():
    # E5M2 shares binary16's sign, exponent and bias; its 2 mantissa bits are
    # binary16's top two, so code c is the binary16 with bits c << 8
    codes = np.arange(256)
    want = (codes.astype(np.uint16) << 8).view(np.float16).astype(np.float64)
    got = M.e5m2_decode(codes)
    finite = np.isfinite(want)
    assert np.array_equal(got[finite], want[finite])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(np.isinf(got), np.isinf(want))
    assert M.e5m2_decode(0x7B) == M.E5M2_MAX == 57344.0
    assert M.e5m2_decode(0x01) == 2.0 ** -16 and M.e5m2_decode(0x04) == 2.0 ** -14


def test_e5m2_encode_nearest_even_saturating():
    codes = np.arange(0x7C)
    assert np.array_equal(M.e5m2_encode(M.e5m2_decode(codes)), codes)
    assert M.e5m2_encode(1.125) == 0x3C        # halfway 1.0 (0x3C) / 1.25 (0x3D): even
    assert M.e5m2_encode(1.375) == 0x3E        # halfway 1.25 (0x3D) / 1.5 (0x3E): even
    assert M.e5m2_encode(2.0 ** -17) == 0x00   # half the smallest subnormal
    assert M.e5m2_encode(1e9) == 0x7B and M.e5m2_encode(-1e9) == 0xFB
    # brute force: the chosen value is a nearest one of the whole grid
    rng = np.random.default_rng(3)
    x = np.exp2(rng.uniform(-18, 16, 4000)) * rng.choice([-1.0, 1.0], 4000)
    got = M.e5m2_decode(M.e5m2_encode(x))
    grid = np.concatenate([-M._E5_VALUES[::-1], M._E5_VALUES])
    best = np.abs(np.abs(x)[:, None].clip(max=M.E5M2_MAX) - np.abs(grid)[None, :]).min(axis=1)
    assert np.array_equal(np.abs(np.abs(got) - np.abs(x).clip(max=M.E5M2_MAX)), best)


def test_p_to_fp8_constant_formats():
    p = np.array([1.0, 2.0, 4.0, 2.0 ** 7.9, 2.0 ** -20])
    e4 = M.p_to_fp8_constant(p, "e4m3")
    e5 = M.p_to_fp8_constant(p, "e5m2")
    assert np.array_equal(e4, M.p_to_mxfp8_constant(p))
    assert e4[1] == 1.75 and e4[2] == 1.75        # 2^(1 + 8) > 448: saturated
    assert e5[1] == 2.0 and e5[2] == 4.0          # E5M2 keeps them
    assert e5[3] == 224.0                         # 2^(7.9 + 8) rounds to the top value 57344 / 2^8
    assert e4[4] == 0.0 and e5[4] == 2.0 ** -20   # below E4M3's subnormals, inside E5M2's
    with pytest.raises(ValueError):
        M.p_to_fp8_constant(p, "e3m4")


def _rel_l2(kind, fmt, tau, exact_cache={}):
    s = rescale_scores(kind)
    v = fp8_sim_values()
    scale = math.log(2.0)          # scores are already in log2 units: scale * log2(e) = 1
    if kind not in exact_cache:
        exact_cache[kind] = blockwise_attention(None, None, v, False, scale, scores=s)[0]
    exact = exact_cache[kind]
    o = blockwise_attention(None, None, v, False, scale, tau=tau, scores=s,
                            p_cast=lambda p: M.p_to_fp8_constant(p, fmt))[0]
    return np.linalg.norm(o - exact) / np.linalg.norm(exact)


@pytest.mark.parametrize("kind", sorted(TABLE))
def test_fp8_p_error_table(kind):
    e4_0, e4_4, e5_0, e5_4 = TABLE[kind]
    got = {(f, t): _rel_l2(kind, f, t) for f in ("e4m3", "e5m2") for t in (0.0, 4.0)}
    # the unsaturated cells are rounding noise (seed spread ~5%); the saturated
    # E4M3 cell depends on how many rows overshoot 448 (seed spread ~15%)
    assert got["e4m3", 0.0] == pytest.approx(e4_0, rel=0.12)
    assert got["e5m2", 0.0] == pytest.approx(e5_0, rel=0.12)
    assert got["e5m2", 4.0] == pytest.approx(e5_4, rel=0.15)
    assert got["e4m3", 4.0] == pytest.approx(e4_4, rel=0.25)
    # the page's reading: E4M3 saturates under tau = 4, E5M2 has the headroom
    assert got["e4m3", 4.0] > 5 * got["e4m3", 0.0]
    assert got["e5m2", 4.0] < 2.5 * got["e5m2", 0.0]
