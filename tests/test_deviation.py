"""Deviation statistics (host logic, CPU only): closed-form cases."""
import math

import numpy as np
import pytest

from precision_numerics_gb300.deviation import deviation


def test_constant_offset():
    ref = np.array([[1.0, -2.0], [3.0, 0.5]])
    d = deviation(ref - 0.25, ref)
    assert d["max_abs"] == 0.25 and d["mean_abs"] == 0.25
    assert d["signed_mean"] == -0.25  # the sign says which way the result is biased
    assert math.isclose(d["rel_l2"], 0.25 * 2 / math.sqrt(1 + 4 + 9 + 0.25))
    assert math.isclose(d["max_rel"], 0.25 / 3.0)


def test_errors_of_both_signs_cancel_only_in_the_signed_mean():
    ref = np.zeros(4) + 2.0
    d = deviation(ref + np.array([0.5, -0.5, 0.5, -0.5]), ref)
    assert d["signed_mean"] == 0.0
    assert d["mean_abs"] == 0.5 and d["max_abs"] == 0.5
    assert math.isclose(d["rel_l2"], 1.0 / 4.0)


def test_exact_match_and_zero_reference():
    ref = np.arange(6.0).reshape(2, 3)
    assert all(v == 0.0 for v in deviation(ref.copy(), ref).values())
    d = deviation(np.array([0.0, 3.0, -4.0]), np.zeros(3))
    assert d["rel_l2"] == 5.0 and d["max_rel"] == 4.0  # absolute figures when ref is 0


def test_inputs_are_widened_before_subtracting():
    ref = np.float32(1.0) + np.float32(2 ** -23) * np.arange(3, dtype=np.float32)
    d = deviation(ref.astype(np.float32), np.ones(3, np.float32))
    assert math.isclose(d["max_abs"], 2 * 2 ** -23)


def test_empty_and_shape_mismatch():
    assert deviation(np.zeros((0, 4)), np.zeros((0, 4)))["max_abs"] == 0.0
    with pytest.raises(ValueError):
        deviation(np.zeros(3), np.zeros(4))
