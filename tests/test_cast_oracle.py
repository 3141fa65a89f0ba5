"""Pins of the oracle's weight-type cast (``cast_to_weight_dtype``): the
float32 weight gradient rounded to the weight's own type, as the source's
backward wrapper does after its float32 column sum ("Hướng dẫn Triton
RMSNorm", section "Reduce dgamma không có race khi ghi").

Pinned against hand-worked ties and overflow cases, and against torch's own
CPU conversions (a library routine: IEEE round to nearest even) on random
float32 bit patterns, so that truncation, ties away from zero or a dropped
carry into the exponent each fail here."""
import importlib.util
import os

import numpy as np
import pytest
import torch

from oracle import rmsnorm_oracle as o


def _f32(vals):
    return np.asarray(vals, dtype=np.float32)


def test_bf16_ties_go_to_even(o=o):
    # bfloat16 keeps 8 significand bits: near 1 its spacing is 2^-7.
    one = 1.0
    vals = _f32([one + 2.0 ** -8,            # halfway 1 .. 1+2^-7: even is 1
                 one + 3 * 2.0 ** -8,        # halfway 1+2^-7 .. 1+2^-6: even is 1+2^-6
                 one + 2.0 ** -8 + 2.0 ** -20,  # just past halfway: up
                 -(one + 2.0 ** -8),         # sign symmetric
                 2.0 - 2.0 ** -9])           # rounds up across the binade to 2
    want = [1.0, 1.0 + 2.0 ** -6, 1.0 + 2.0 ** -7, -1.0, 2.0]
    assert o.cast_to_weight_dtype(vals, "bf16").tolist() == want


def test_f16_ties_and_range(o=o):
    # float16 keeps 11 significand bits: near 1 its spacing is 2^-10.
    vals = _f32([1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 65504.0, 65520.0, 2.0 ** -24,
                 2.0 ** -26, 3 * 2.0 ** -25])
    got = o.cast_to_weight_dtype(vals, "f16").tolist()
    # ties to even; 65504 the largest finite, 65520 halfway to the next
    # power of two rounds to infinity; 2^-24 the smallest subnormal, 2^-26
    # under half of it rounds to zero, 1.5 * 2^-24 halfway rounds to even 2^-23.
    assert got == [1.0, 1.0 + 2.0 ** -9, 65504.0, float("inf"), 2.0 ** -24, 0.0, 2.0 ** -23]


def test_bf16_overflow_to_infinity(o=o):
    big = np.float32(np.finfo(np.float32).max)
    got = o.cast_to_weight_dtype(_f32([big, -big, 3.3895313892515355e38]), "bf16")
    assert np.isinf(got[0]) and got[0] > 0 and np.isinf(got[1]) and got[1] < 0
    assert got[2] == 3.3895313892515355e38  # bf16's largest finite value stays


def test_f32_is_unchanged():
    v = _f32([1.0 + 2.0 ** -23, -3.5e38, 1e-45])
    assert np.array_equal(o.cast_to_weight_dtype(v, "f32"), v.astype(np.float64))


@pytest.mark.parametrize("wdtype,tdt", [("bf16", torch.bfloat16), ("f16", torch.float16)])
def test_matches_torch_round_to_nearest_even(wdtype, tdt):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    # and values in each type's own range, with the low bits random
    v = np.concatenate([v, (rng.standard_normal(100_000) * 10.0 ** rng.integers(-8, 5, 100_000))
                        .astype(np.float32)])
    want = torch.from_numpy(v.copy()).to(tdt).to(torch.float64).numpy()
    got = o.cast_to_weight_dtype(v, wdtype)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), v[~same][:5]


# ---- planted mistakes, each in a fresh copy of the oracle (CPU only) ----

def _fresh_copy(tag):
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                        "rmsnorm_oracle.py")
    spec = importlib.util.spec_from_file_location(f"oracle_cast_mutant_{tag}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _bf16_truncate(a):
    f = np.ascontiguousarray(np.asarray(a, np.float64).astype(np.float32))
    return ((f.view(np.uint32) >> 16) << 16).astype(np.uint32).view(np.float32)


def _bf16_ties_away(a):
    f = np.ascontiguousarray(np.asarray(a, np.float64).astype(np.float32))
    bits = f.view(np.uint32).astype(np.uint64)
    return (((bits + 0x8000) >> 16) << 16).astype(np.uint32).view(np.float32)


def _bf16_no_carry(a):
    # rounds the 7 stored bits but drops the carry into the exponent
    f = np.ascontiguousarray(np.asarray(a, np.float64).astype(np.float32))
    bits = f.view(np.uint32).astype(np.uint64)
    keep = (bits >> 16) & 1
    mant = (((bits & 0x7FFFFF) + 0x7FFF + keep) >> 16) & 0x7F
    return (((bits >> 23) << 23) | (mant << 16)).astype(np.uint32).view(np.float32)


def _f16_truncate(a):
    f = np.asarray(a, np.float64).astype(np.float32)
    h = f.astype(np.float16)
    lower = np.where(np.abs(h.astype(np.float32)) > np.abs(f),
                     np.nextafter(h, np.float16(0)), h)
    return lower.astype(np.float32)


@pytest.mark.parametrize("name,attr,fn,pin", [
    ("bf16_truncate", "_round_bf16", _bf16_truncate, test_bf16_ties_go_to_even),
    ("bf16_ties_away", "_round_bf16", _bf16_ties_away, test_bf16_ties_go_to_even),
    ("bf16_no_carry", "_round_bf16", _bf16_no_carry, test_bf16_ties_go_to_even),
    ("f16_truncate", "_round_f16", _f16_truncate, test_f16_ties_and_range),
])
def test_planted_rounding_mistake_is_caught(name, attr, fn, pin):
    m = _fresh_copy(name)
    setattr(m, attr, fn)
    with pytest.raises(AssertionError):
        pin(o=m)
    pin(o=_fresh_copy(name + "_clean"))  # the unmutated copy passes the same pin
