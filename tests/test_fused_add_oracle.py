"""The fused residual-add oracle functions against facts fixed outside them
(CPU only): torch's own float32/bfloat16/float16 addition for h, and float64
autograd through h = x + residual, y = rms_norm(h) for the gradients; planted
mistakes in copies of the oracle must fail a pin."""
import importlib.util
import os

import numpy as np
import pytest

from synthetic.generator import bf16_bits_to_float32, float_to_bf16_bits

ORACLE_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "rmsnorm_oracle.py")


def _load(tag):
    spec = importlib.util.spec_from_file_location(f"rms_oracle_add_{tag}", ORACLE_PATH)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _dtype_values(rng, shape, dtype, scale=1.0):
    v = scale * rng.standard_normal(shape)
    if dtype == "bf16":
        return bf16_bits_to_float32(float_to_bf16_bits(v)).astype(np.float64)
    if dtype == "f16":
        return v.astype(np.float16).astype(np.float64)
    return v.astype(np.float32).astype(np.float64)


def pin_h_matches_torch_dtype_add(o):
    import torch

    rng = np.random.default_rng(3)
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
    for dtype in ("bf16", "f16", "f32"):
        for scale_b in (1.0, 1e-3, 300.0):  # include sums where the smaller term is mostly lost
            a = _dtype_values(rng, (37, 53), dtype)
            b = _dtype_values(rng, (37, 53), dtype, scale_b)
            h = o.residual_add(a, b, dtype)
            ref = (torch.tensor(a).to(tdt[dtype]) + torch.tensor(b).to(tdt[dtype])).double().numpy()
            assert np.array_equal(h, ref), (dtype, scale_b)


def pin_gradients_match_autograd(o):
    import torch
    import torch.nn.functional as F

    rng = np.random.default_rng(4)
    for M, N, eps, gemma in [(5, 33, 1e-6, 0), (3, 128, 1e-2, 1), (7, 1, 1e-5, 0)]:
        x = rng.standard_normal((M, N))
        res = rng.standard_normal((M, N))
        g = rng.uniform(0.5, 1.5, N)
        dy = rng.standard_normal((M, N))
        dh = rng.standard_normal((M, N))
        tx = torch.tensor(x, requires_grad=True)
        tr = torch.tensor(res, requires_grad=True)
        tg = torch.tensor(g, requires_grad=True)
        h = tx + tr
        w = (1.0 + tg) if gemma else tg
        y = F.rms_norm(h, (N,), w, eps)
        ((torch.tensor(dy) * y).sum() + (torch.tensor(dh) * h).sum()).backward()
        hh = x + res  # exact in float64 for these inputs' purpose: the pin is on the gradient algebra
        dx, dg = o.rms_backward_add(hh, g, dy, dh, eps, gemma)
        assert np.allclose(dx, tx.grad.numpy(), rtol=1e-10, atol=1e-12)
        assert np.allclose(dx, tr.grad.numpy(), rtol=1e-10, atol=1e-12)
        assert np.allclose(dg, tg.grad.numpy(), rtol=1e-10, atol=1e-12)
        yy, r, _ = o.rms_forward_add(x, res, g, eps, gemma, "f32")
        hf = (x.astype(np.float32) + res.astype(np.float32)).astype(np.float64)
        ty = F.rms_norm(torch.tensor(hf), (N,), torch.tensor((1.0 + g) if gemma else g), eps)
        assert np.allclose(yy, ty.numpy(), rtol=1e-12, atol=1e-14)


ALL_PINS = [pin_h_matches_torch_dtype_add, pin_gradients_match_autograd]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_fused_add_oracle_pin(pin):
    pin(_load("real"))


def _mutant(name):
    m = _load(name)
    if name == "h_without_residual":
        m.residual_add = lambda x, r, dtype="f32": np.asarray(x, np.float64)
    elif name == "h_rounded_in_float64":
        def ra(x, r, dtype="f32", _m=m):
            rnd = {"bf16": _m._round_bf16, "f16": _m._round_f16}.get(dtype, _m._round_f32)
            return rnd(np.asarray(x, np.float64) + np.asarray(r, np.float64)).astype(np.float64)
        m.residual_add = ra
    elif name == "dh_dropped":
        orig = m.rms_backward
        m.rms_backward_add = lambda h, g, dy, dh, eps, gemma=0, with_scales=False, _o=orig: \
            _o(h, g, dy, eps, gemma)
    elif name == "dh_doubled":
        orig = m.rms_backward_add
        m.rms_backward_add = lambda h, g, dy, dh, eps, gemma=0, with_scales=False, _o=orig: (
            _o(h, g, dy, dh, eps, gemma)[0] + np.asarray(dh), _o(h, g, dy, dh, eps, gemma)[1])
    return m


@pytest.mark.parametrize("name", ["h_without_residual", "h_rounded_in_float64", "dh_dropped",
                                  "dh_doubled"])
def test_fused_add_mutant_is_caught(name):
    m = _mutant(name)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(m)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name!r} passes every fused-add pin"
