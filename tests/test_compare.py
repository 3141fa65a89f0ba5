"""The tolerance checks flag what they should (CPU only)."""
import numpy as np

from oracle import compare


def test_y_bf16_bar():
    ref = np.array([0.5, 2.0, -300.0])
    assert compare.check_y(ref + np.array([0.0099, 0.0199, 2.99]), ref, "bf16").ok
    assert not compare.check_y(ref + np.array([0.0101, 0.0, 0.0]), ref, "bf16").ok
    assert not compare.check_y(ref + np.array([0.0, 0.0, 3.01]), ref, "bf16").ok


def test_y_f32_relative():
    ref = np.array([1.0, 1e-3])
    assert compare.check_y(ref * (1 + 9e-6), ref, "f32").ok
    assert not compare.check_y(ref * np.array([1.0, 1 + 2e-5]), ref, "f32").ok


def test_dx_and_dgamma_scaled_by_terms():
    ref = np.array([1e-9, 1.0])
    scale = np.array([10.0, 1.0])
    assert compare.check_dx(ref + np.array([5e-5, 0.0]), ref, scale, "f32").ok
    assert not compare.check_dx(ref + np.array([2e-4, 0.0]), ref, scale, "f32").ok
    assert compare.check_dgamma(ref + np.array([1e-3, 0.0]), ref, scale, "f32").ok
    assert not compare.check_dgamma(ref + np.array([2e-3, 0.0]), ref, scale, "f32").ok


def test_nonfinite_handling():
    ref = np.array([np.nan, np.inf, 1.0])
    assert compare.check_y(np.array([np.nan, np.inf, 1.0]), ref, "f32").ok
    assert not compare.check_y(np.array([1.0, np.inf, 1.0]), ref, "f32").ok
    assert not compare.check_y(np.array([np.nan, np.inf, np.nan]), ref, "f32").ok


def test_rstd_bar():
    ref = np.array([0.25, 100.0])
    assert compare.check_rstd(ref * (1 + 9e-7), ref).ok
    assert not compare.check_rstd(ref * (1 + 2e-6), ref).ok
