"""Pins of the oracle's historical-query sensitivity s_c = mean_i q_ic^2
(QuantWM Abstract, "historical Query sensitivity"; roboind article, "Step 1").

The values come from worked examples derived by hand
(`tests/golden/sensitivity_hand.json`), not from the oracle; two plausible
slips (summing instead of averaging, dividing by n_h - 1) are planted in the
oracle and must fail the pin.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import qwm_oracle as O


@pytest.fixture(scope="module")
def golden(golden_dir):
    with open(os.path.join(golden_dir, "sensitivity_hand.json")) as f:
        return json.load(f)


def _want_a(g):
    a = g["case_a"]
    return [Fraction(n, a["s_den"]) for n in a["s_num"]]


def test_sensitivity_hand_worked_example(golden):
    q = np.array(golden["case_a"]["q_hist"], dtype=np.float64)
    got = O.sensitivity(q)
    for c, want in enumerate(_want_a(golden)):
        assert abs(got[c] - float(want)) <= 1e-15 * float(want)


def test_sensitivity_per_head_axis(golden):
    """[H, n_h, d]: every head gets its own mean; the heads do not mix."""
    q = np.array(golden["case_a"]["q_hist"], dtype=np.float64)
    stacked = np.stack([q, 2.0 * q])
    got = O.sensitivity(stacked)
    want = np.array([float(x) for x in _want_a(golden)])
    assert np.allclose(got[0], want, rtol=1e-15) and np.allclose(got[1], 4.0 * want, rtol=1e-15)


def test_group_weights_of_squared_ramp(golden):
    """s_c = c^2 from two opposite ramps; w_g is the closed-form sum of squares."""
    b = golden["case_b"]
    c = np.arange(b["d"], dtype=np.float64)
    s = O.sensitivity(np.stack([c, -c]))
    assert s.tolist() == (c * c).tolist()
    assert O.group_weights(s.astype(np.float32)).tolist() == b["w"]


@pytest.mark.parametrize("slip", ["sum", "n_minus_1"])
def test_planted_normalisation_slip_is_caught(golden, monkeypatch, slip):
    """A sensitivity that sums, or divides by n_h - 1, misses the hand values."""
    def bad(q_hist):
        q = np.asarray(q_hist, dtype=np.float64)
        tot = (q * q).sum(axis=-2)
        return tot if slip == "sum" else tot / (q.shape[-2] - 1)
    monkeypatch.setattr(O, "sensitivity", bad)
    got = O.sensitivity(np.array(golden["case_a"]["q_hist"], dtype=np.float64))
    want = [float(x) for x in _want_a(golden)]
    assert any(abs(g - w) > 1e-6 * w for g, w in zip(got, want))
