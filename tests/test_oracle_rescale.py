"""Pins for the lagging-max rescale simulator (CPU only): the rescale-rate
table printed on the first page, and the 1/(j+1) record rate of iid scores."""
import numpy as np
import pytest

from attn_inputs import rescale_scores
from conftest import read_golden_table
from oracle.rescale_stats import fired_matrix, rescale_rates

TABLE = read_golden_table("rescale_rates.txt")


@pytest.mark.parametrize("kind", sorted(TABLE))
def test_rates_match_table(kind):
    s = rescale_scores(kind)
    r0, w0 = rescale_rates(s, tau=0.0)
    r8, w8 = rescale_rates(s, tau=8.0)
    t0r, t0w, t8r, t8w = TABLE[kind]
    # the table prints 2-3 digits; the ramp rows' noise is a reading
    assert r0 == pytest.approx(t0r, abs=1.0)
    assert w0 == pytest.approx(t0w, abs=5.0)
    assert r8 == pytest.approx(t8r, abs=1.0)
    assert w8 == pytest.approx(t8w, abs=5.0)


def test_iid_record_rate():
    # without tau, an iid row sets a new record in block j with probability
    # 1/(j+1) (the page's "about 1/j" remark); average over blocks 1..63
    s = rescale_scores("iid1.5")
    f = fired_matrix(s, tau=0.0)
    expect = np.mean([1.0 / (j + 1) for j in range(1, 64)])
    assert f[:, 1:].mean() == pytest.approx(expect, abs=0.005)
    assert f[:, 0].all()


def test_growth_equal_to_tau_keeps_stale_max():
    # growth of exactly tau keeps the stale max; a hair more moves it
    s = np.zeros((32, 256))
    s[:, 0] = 1.0
    s[:16, 200] = 9.0
    s[16:, 200] = 9.0 + 1e-9
    f = fired_matrix(s, block=128, tau=8.0)
    assert not f[:16, 1].any() and f[16:, 1].all()
