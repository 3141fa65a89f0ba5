"""The E4M3 output oracle against facts fixed outside it (CPU only): torch's
float8_e4m3fn conversion bit for bit, the format's closed forms, and the
per-row scale's invariants; planted mistakes must fail a pin."""
import importlib.util
import os

import numpy as np
import pytest

ORACLE_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "rmsnorm_oracle.py")


def _load(tag):
    spec = importlib.util.spec_from_file_location(f"rms_oracle_q_{tag}", ORACLE_PATH)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _probe_values():
    rng = np.random.default_rng(8)
    mag = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 20000))
    v = mag * rng.choice([-1.0, 1.0], mag.size)
    grid = np.arange(-448, 449, 0.0625)  # many exact ties between E4M3 neighbours
    ties = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -11, 2.0 ** -6 - 2.0 ** -10, 240.0,
                     232.0, 0.0, -0.0, 448.0, -448.0])
    return np.concatenate([v, grid, ties]).astype(np.float32).astype(np.float64)


def pin_matches_torch_float8(o):
    import torch

    v = _probe_values()
    t = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn)
    assert np.array_equal(o.round_e4m3(v), t.to(torch.float64).numpy())
    assert np.array_equal(o.e4m3_code(o.round_e4m3(v)), t.view(torch.uint8).numpy())


def pin_format_closed_forms(o):
    # every finite positive E4M3 value round-trips, and the ladder is the format's
    vals = np.array([k * 2.0 ** -9 for k in range(1, 8)]
                    + [(1 + m / 8) * 2.0 ** e for e in range(-6, 9) for m in range(8)
                       if not (e == 8 and m == 7)])
    assert np.array_equal(o.round_e4m3(vals), vals)
    assert vals.max() == 448.0 and len(vals) == 126
    assert np.array_equal(o.e4m3_code(vals), np.arange(1, 127, dtype=np.uint8))
    assert o.round_e4m3(np.array([1e6, -1e6])).tolist() == [448.0, -448.0]  # saturating


def pin_row_scale_invariants(o):
    rng = np.random.default_rng(9)
    y = rng.standard_normal((40, 300)) * np.exp(rng.uniform(-8, 8, 40))[:, None]
    y = y.astype(np.float32).astype(np.float64)
    y[3] = 0.0
    q, s = o.quantize_rows_e4m3(y)
    amax = np.abs(y).max(axis=1)
    nz = amax > 0
    assert np.allclose(s[nz], amax[nz] / 448.0, rtol=2 ** -23)
    assert s[3] == 1.0 and np.all(q[3] == 0)
    # the largest element of each row lands on 448 in magnitude
    assert np.all(np.abs(q[nz]).max(axis=1) == 448.0)
    # every code is the nearest E4M3 value to y/scale, within half a spacing
    v = y[nz] / s[nz, None]
    _, ex = np.frexp(np.maximum(np.abs(v), 2.0 ** -6))
    half = np.ldexp(1.0, ex - 1 - 3) / 2
    assert np.all(np.abs(q[nz] - v) <= half * (1 + 1e-6))


ALL_PINS = [pin_matches_torch_float8, pin_format_closed_forms, pin_row_scale_invariants]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_quant_oracle_pin(pin):
    pin(_load("real"))


def _mutant(name):
    m = _load(name)
    if name == "round_half_up":
        def r(v, _m=m):
            v = np.asarray(v, np.float64)
            a = np.abs(v)
            _, ex = np.frexp(np.maximum(a, 2.0 ** -6))
            sp = np.ldexp(1.0, ex - 4)
            return np.copysign(np.minimum(np.floor(a / sp + 0.5) * sp, 448.0), v)
        m.round_e4m3 = r
    elif name == "no_subnormals":
        orig = m.round_e4m3
        m.round_e4m3 = lambda v, _o=orig: np.where(np.abs(np.asarray(v)) < 2.0 ** -6, 0.0, _o(v))
    elif name == "scale_by_max_448":
        orig = m.quantize_rows_e4m3
        def qr(y, _o=orig):
            q, s = _o(y)
            return q, s * 448.0 / 240.0
        m.quantize_rows_e4m3 = qr
    elif name == "bias_8":
        orig = m.e4m3_code
        m.e4m3_code = lambda q, _o=orig: (_o(q) + 8).astype(np.uint8)
    return m


@pytest.mark.parametrize("name", ["round_half_up", "no_subnormals", "scale_by_max_448", "bias_8"])
def test_quant_mutant_is_caught(name):
    m = _mutant(name)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(m)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name!r} passes every E4M3 pin"
