"""Pins for the MXFP8 quantiser of the oracle (CPU only): the E4M3 format's
closed forms, PyTorch's float8_e4m3fn conversion as a library cross-check, the
E8M0 scale rule as a property, and the 32 x 32 block structure."""
import numpy as np
import pytest
import torch

from oracle import mxfp8 as M


def test_e4m3_known_codes():
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5, 0x38: 1.0,
             0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for code, val in table.items():
        assert M.e4m3_decode(code) == val
    assert np.isnan(M.e4m3_decode(0x7F)) and np.isnan(M.e4m3_decode(0xFF))


def test_round_trip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(M.e4m3_encode(M.e4m3_decode(codes)), codes)


def test_ties_go_to_even_and_saturation():
    assert M.e4m3_encode(1.0625) == 0x38      # between 1.0 (0x38) and 1.125 (0x39)
    assert M.e4m3_encode(1.1875) == 0x3A      # between 1.125 (0x39) and 1.25 (0x3A)
    assert M.e4m3_encode(1.9375) == 0x40      # between 1.875 (0x3F) and 2.0 (0x40)
    assert M.e4m3_encode(2.0 ** -10) == 0x00  # half the smallest subnormal -> 0 (even)
    assert M.e4m3_encode(3 * 2.0 ** -10) == 0x02
    for big, code in ((448.0, 0x7E), (460.0, 0x7E), (500.0, 0x7E), (1e9, 0x7E), (-1e9, 0xFE)):
        assert M.e4m3_encode(big) == code


def test_agrees_with_torch_float8_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-448, 448, 200000), rng.standard_normal(200000) * 3,
                        rng.standard_normal(100000) * 1e-2]).astype(np.float32)
    ours = M.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_scale_rule_is_the_smallest_power_of_two():
    rng = np.random.default_rng(1)
    amax = np.concatenate([np.exp(rng.uniform(-20, 20, 10000)), 448.0 * np.exp2(np.arange(-10, 10.0)),
                           [1.0, 1.75, 448.0, 449.0]])
    e = M.e8m0_exponent(amax)
    assert np.all(amax <= 448.0 * np.exp2(e))
    assert np.all(amax > 448.0 * np.exp2(e - 1))
    assert list(M.e8m0_exponent([448.0, 449.0, 1.0, 1.75, 1.76, 0.0])) == [0, 1, -8, -8, -7, 0]


def test_block_structure_and_error_bound():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 3, 96, 128))
    x[0, 0, 32:64, 64:96] *= 1000.0            # one loud block must not change its neighbours
    codes, e, deq = M.quantize_blocks(x)
    assert codes.shape == x.shape and e.shape == (2, 3, 3, 4)
    amax = np.abs(x.reshape(2, 3, 3, 32, 4, 32)).max(axis=(3, 5))
    assert np.array_equal(e, M.e8m0_exponent(amax))
    assert e[0, 0, 1, 2] > e[0, 0, 1, 1] + 8
    # every block's largest element reaches at least the top half of E4M3's range
    assert np.all(amax / np.exp2(e) > 224.0)
    # 3 mantissa bits: relative error <= 2^-4 for elements in E4M3's normal range
    normal = np.abs(x) / np.repeat(np.repeat(np.exp2(e.astype(float)), 32, -2), 32, -1) >= 2.0 ** -6
    rel = np.abs(deq - x)[normal] / np.abs(x)[normal]
    assert rel.max() <= 2.0 ** -4 + 1e-12


def test_ragged_rows_are_padded_for_amax_only():
    x = np.ones((1, 1, 40, 64))
    codes, e, deq = M.quantize_blocks(x)
    assert codes.shape == (1, 1, 40, 64) and e.shape == (1, 1, 2, 2)
    assert np.array_equal(deq, x)


# ---- P converted to MXFP8 (one scale per 32 consecutive keys of a row)

def test_p_runs_of_representable_values_are_unchanged():
    # a run whose largest value is 1 takes scale 2^-8; values k/8 * 2^-n are
    # E4M3 values times that scale when they stay in E4M3's range
    vals = M.e4m3_decode(np.arange(0x08, 0x7F)) * 2.0 ** -8      # normal E4M3 values, scaled
    vals = vals[vals <= 1.0]
    rng = np.random.default_rng(5)
    p = rng.choice(vals, size=(7, 32))
    p[:, 0] = 1.0
    assert np.array_equal(M.p_to_mxfp8(p), p)


def test_p_runs_follow_the_scale_rule_and_nearest_rounding():
    # brute force: every element is the nearest of all E4M3 values times the
    # run's 2^e, e the smallest exponent with amax <= 448 * 2^e
    rng = np.random.default_rng(6)
    p = np.exp2(-rng.uniform(0, 12, size=(5, 96)))
    p[2, 32:64] *= 1e-3                         # a quiet run must get its own, smaller scale
    got = M.p_to_mxfp8(p)
    grid = M.e4m3_decode(np.arange(0x00, 0x7F))
    for r in range(p.shape[0]):
        for g0 in range(0, 96, 32):
            run = p[r, g0:g0 + 32]
            e = 0
            while run.max() > 448.0 * 2.0 ** e:
                e += 1
            while run.max() <= 448.0 * 2.0 ** (e - 1):
                e -= 1
            cand = grid * 2.0 ** e
            want = cand[np.abs(run[:, None] - cand[None, :]).argmin(axis=1)]
            assert np.array_equal(got[r, g0:g0 + 32], want)


def test_p_relative_error_and_run_boundaries():
    rng = np.random.default_rng(7)
    p = rng.uniform(0.0, 1.0, size=(4, 70))     # runs [0, 32), [32, 64), [64, 70)
    got = M.p_to_mxfp8(p)
    for a, b in ((0, 32), (32, 64), (64, 70)):
        run, out = p[:, a:b], got[:, a:b]
        scale = np.exp2(M.e8m0_exponent(run.max(axis=1)).astype(float))[:, None]
        normal = run / scale >= 2.0 ** -6       # E4M3's normal range after scaling
        rel = np.abs(out - run)[normal] / run[normal]
        assert rel.max() <= 2.0 ** -4 + 1e-12
    # changing one run leaves the others alone
    q = p.copy()
    q[:, 32:64] *= 1e-4
    got_q = M.p_to_mxfp8(q)
    assert np.array_equal(got_q[:, :32], got[:, :32]) and np.array_equal(got_q[:, 64:], got[:, 64:])


def test_p_constant_scale_conversion():
    # P in [0, 1.75] with the constant scale 2^-8: every E4M3 value times
    # 2^-8 is kept, everything else goes to the nearest one (brute force), and
    # nothing saturates below 448 / 256
    grid = M.e4m3_decode(np.arange(0x00, 0x7F)) * 2.0 ** -8
    keep = grid[grid <= 1.75]
    assert np.array_equal(M.p_to_mxfp8_constant(keep), keep)
    rng = np.random.default_rng(8)
    p = np.concatenate([rng.uniform(0, 1.75, 5000), np.exp2(-rng.uniform(0, 20, 5000))])
    want = grid[np.abs(p[:, None] - grid[None, :]).argmin(axis=1)]
    assert np.array_equal(M.p_to_mxfp8_constant(p), want)
    assert M.p_to_mxfp8_constant(np.array([1.0]))[0] == 1.0
    assert M.p_to_mxfp8_constant(np.array([2.0]))[0] == 1.75   # saturates at 448 * 2^-8
