"""Planted mistakes in copies of the oracle must each fail at least one pin.

This shows the pins are sensitive to the plausible ways the oracle could be
wrong: a dropped term, a wrong sign or exponent, a wrong denominator, a
missing factor, a mean where a sum belongs.  Every mistake is planted in a
fresh copy of the oracle module, on the CPU; the oracle itself is untouched.
"""
import importlib.util
import os

import numpy as np
import pytest

from tests.oracle_pins import ALL_PINS

ORACLE_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "rmsnorm_oracle.py")


def _fresh_copy(tag):
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{tag}", ORACLE_PATH)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _pow2(n):
    return 1 << (int(n) - 1).bit_length()


def _bwd_factory(variant):
    """A backward with one planted mistake; the rest as the definition."""
    def rms_backward(x, gamma, dy, eps, gemma=0, with_scales=False, _m=None):
        m = _m
        x = np.asarray(x, np.float64)
        dy = np.asarray(dy, np.float64)
        n = x.shape[-1]
        r = m.rms_rstd(x, eps)
        g = m.weight(gamma, gemma)
        u = dy if variant == "u_without_gamma" else dy * g[None, :]
        if variant == "bwd_block_denominator":
            c = np.sum(u * x, axis=-1) / _pow2(n)
        else:
            c = np.mean(u * x, axis=-1)
        if variant == "r_squared_in_dx":
            dx = r[:, None] * u - x * (r ** 2 * c)[:, None]
        elif variant == "dx_second_term_dropped":
            dx = r[:, None] * u
        elif variant == "dx_sign_flip":
            dx = r[:, None] * u + x * (r ** 3 * c)[:, None]
        else:
            dx = r[:, None] * u - x * (r ** 3 * c)[:, None]
        if variant == "dgamma_mean":
            dgamma = np.mean(dy * x * r[:, None], axis=0)
        elif variant == "dgamma_without_r":
            dgamma = np.sum(dy * x, axis=0)
        elif variant == "dgamma_times_weight":
            dgamma = np.sum(u * x * r[:, None], axis=0)
        else:
            dgamma = np.sum(dy * x * r[:, None], axis=0)
        if not with_scales:
            return dx, dgamma
        dxs = r[:, None] * np.abs(u) + np.abs(x) * (r ** 3 * np.mean(np.abs(u * x), axis=-1))[:, None]
        return dx, dgamma, dxs, np.sum(np.abs(dy * x * r[:, None]), axis=0)
    return rms_backward


def mutant(name):
    m = _fresh_copy(name)
    if name == "fwd_block_denominator":
        m.rms_rstd = lambda x, eps: 1.0 / np.sqrt(
            np.sum(np.asarray(x, np.float64) ** 2, axis=-1) / _pow2(np.shape(x)[-1]) + eps)
    elif name == "eps_outside_sqrt":
        m.rms_rstd = lambda x, eps: 1.0 / (np.sqrt(np.mean(np.asarray(x, np.float64) ** 2, axis=-1)) + eps)
    elif name == "eps_dropped":
        m.rms_rstd = lambda x, eps: 1.0 / np.sqrt(np.mean(np.asarray(x, np.float64) ** 2, axis=-1))
    elif name == "rms_not_mean_square":
        m.rms_rstd = lambda x, eps: 1.0 / np.sqrt(np.mean(np.abs(np.asarray(x, np.float64)), axis=-1) + eps)
    elif name == "dgamma_only_mean":
        orig = m.rms_dgamma
        m.rms_dgamma = lambda x, dy, eps, with_scales=False, _o=orig: (
            (lambda r: (r[0] / np.shape(x)[0], r[1]) if with_scales else r / np.shape(x)[0])(
                _o(x, dy, eps, with_scales)))
    elif name == "gemma_ignored":
        m.weight = lambda gamma, gemma=0: np.asarray(gamma, np.float64)
    elif name == "gamma_reversed":
        orig = m.weight
        m.weight = lambda gamma, gemma=0: orig(gamma, gemma)[::-1].copy()
    elif name == "normed_form_missing_n":
        def bad(x, gamma, dy, eps, gemma=0, _m=m):
            x = np.asarray(x, np.float64)
            r = _m.rms_rstd(x, eps)
            normed = x * r[:, None]
            dyw = np.asarray(dy, np.float64) * _m.weight(gamma, gemma)[None, :]
            s = np.sum(dyw * normed, axis=-1)
            return r[:, None] * (dyw - normed * s[:, None])
        m.rms_backward_normed_form = bad
    elif name == "emulation_single_rounding":
        def once(x, gamma, eps, gemma=0, dtype="bf16", _m=m):
            y, _ = _m.rms_forward(x, gamma, eps, gemma)
            return _m._round_bf16(y).astype(np.float64)
        m.emulate_forward_lowp = once
    elif name == "emulation_weight_first":
        def wfirst(x, gamma, eps, gemma=0, dtype="bf16", _m=m):
            xf = _m._round_f32(x)
            gf = _m._round_f32(_m.weight(gamma, gemma))
            r32 = _m._round_f32(_m.rms_rstd(x, eps))
            xg = _m._round_bf16(xf.astype(np.float64) * gf[None, :])
            return _m._round_bf16(_m._round_f32(xg.astype(np.float64) * r32[:, None])).astype(np.float64)
        m.emulate_forward_lowp = wfirst
    else:
        bwd = _bwd_factory(name)
        m.rms_backward = lambda *a, _b=bwd, _m=m, **k: _b(*a, _m=_m, **k)
    return m


MUTANTS = [
    "fwd_block_denominator",
    "eps_outside_sqrt",
    "eps_dropped",
    "rms_not_mean_square",
    "gemma_ignored",
    "gamma_reversed",
    "u_without_gamma",
    "bwd_block_denominator",
    "r_squared_in_dx",
    "dx_second_term_dropped",
    "dx_sign_flip",
    "dgamma_mean",
    "dgamma_without_r",
    "dgamma_times_weight",
    "dgamma_only_mean",
    "normed_form_missing_n",
    "emulation_single_rounding",
    "emulation_weight_first",
]


def _caught_by(m):
    caught = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(m)
        except (AssertionError, FloatingPointError, ValueError, ZeroDivisionError):
            caught.append(pin.__name__)
    return caught


@pytest.mark.parametrize("name", MUTANTS)
def test_mutant_is_caught(name):
    caught = _caught_by(mutant(name))
    assert caught, f"planted mistake {name!r} passes every pin"


def test_unmutated_copy_passes_every_pin():
    assert _caught_by(_fresh_copy("clean")) == []
