"""Pins for oracle.closed_forms against the numbers the P-cast page prints
(tests/golden/page_numbers.txt) and against the E4M3 decode table."""
import math

import numpy as np
import pytest

from oracle import closed_forms as cf
from tests.golden.pages import page_numbers

PAGE = page_numbers()


def test_round_to_zero_in_nats():
    assert cf.ROUND_TO_ZERO_NATS == pytest.approx(-math.log(PAGE["round_to_zero_threshold"]), rel=1e-15)
    assert round(cf.ROUND_TO_ZERO_NATS, 2) == PAGE["round_to_zero_nats"]


def test_delta_k_for_four_sinks():
    dk = cf.delta_k(4)
    assert round(dk, 1) == PAGE["delta_k_for_k4"]
    assert dk == pytest.approx(1.0293753730, abs=1e-9)   # E[max of 4 N(0,1)]
    assert cf.delta_k(1) == pytest.approx(0.0, abs=1e-12)
    assert cf.delta_k(2) == pytest.approx(1.0 / math.sqrt(math.pi), abs=1e-12)


def test_collapse_onset_for_S1():
    lo, hi = PAGE["collapse_onset_S1_low"], PAGE["collapse_onset_S1_high"]
    dc = cf.critical_delta(1.0)          # 10 ln 2 - delta_4 = 5.90
    assert round(dc) == lo
    assert cf.underflow_fraction(dc, 1.0) == pytest.approx(0.5, abs=1e-12)
    # the collapse switches on across delta ~ 6-7: half the non-sink P at 6, most by 7
    assert cf.underflow_fraction(lo - 2, 1.0) < 0.05
    assert cf.underflow_fraction(lo, 1.0) > 0.5 and cf.underflow_fraction(hi, 1.0) > 0.8
    # larger S moves the onset by ln S
    assert cf.critical_delta(256.0) - dc == pytest.approx(math.log(256.0), abs=1e-12)


def test_reverse_bound():
    bound = cf.reverse_bound(int(PAGE["reverse_bound_max_N"]), 256.0)
    assert bound < PAGE["reverse_nonsink_bound"]
    assert bound == pytest.approx(2.6e-13, rel=0.1)


def test_dp_sawtooth(orc):
    table = orc.e4m3_decode_table()
    for k in range(0, 9):
        assert cf.d_p(2.0 ** k, table) == PAGE["dp_floor_power_of_two"]
    excess = cf.d_p(448.0, table) / cf.d_p(256.0, table) - 1.0
    assert round(excess, 2) == PAGE["dp_excess_S448"]
    # power-of-two scales sit on the lower envelope
    for S in np.linspace(1.5, 447.0, 300):
        assert cf.d_p(float(S), table) >= PAGE["dp_floor_power_of_two"] - 1e-15


def test_normal_coverage(orc):
    table = orc.e4m3_decode_table()
    assert cf.normal_coverage(PAGE["largest_pow2_no_overflow"], table) == PAGE["normal_coverage_S256"]
    pow2 = [2.0 ** k for k in range(12) if 2.0 ** k <= PAGE["e4m3_max_finite"]]
    assert max(pow2) == PAGE["largest_pow2_no_overflow"]
