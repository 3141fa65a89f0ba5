"""Pins of the fp64 oracle against facts fixed outside it.

Each ``pin_*`` takes an implementation object exposing the oracle's function
names (``rms_forward``, ``rms_backward``, ``rms_rstd``,
``rms_backward_normed_form``, ``emulate_forward_lowp``) and raises
AssertionError when the implementation disagrees with:

* values the pages print for worked examples (``tests/golden``);
* the exact central-difference gradient of L = sum(dy * y);
* ``torch.nn.functional.rms_norm`` and autograd in float64 (a library
  routine the oracle does not call);
* closed forms and invariants derived from the definitions.

``tests/test_oracle_pins.py`` runs every pin on the oracle;
``tests/test_oracle_mutants.py`` runs them on copies of the oracle with a
planted mistake and requires each copy to fail at least one pin.
"""
from __future__ import annotations

import json
import math
from pathlib import Path

import numpy as np

GOLDEN = json.loads((Path(__file__).parent / "golden" / "worked_examples.json").read_text())
CASES = {c["id"]: c for c in GOLDEN["cases"]}


def _close_printed(got, printed, decimals):
    """A value printed with ``decimals`` decimals matches within half a unit there."""
    got = np.asarray(got, np.float64)
    printed = np.asarray(printed, np.float64)
    half = 0.5 * 10.0 ** (-decimals) * (1 + 1e-9)
    assert got.shape == printed.shape, (got.shape, printed.shape)
    assert np.all(np.abs(got - printed) <= half), (got, printed)


def pin_worked_forward(impl):
    c = CASES["forward_3_4_unit_gamma"]
    y, r = impl.rms_forward(np.array(c["x"]), np.array(c["gamma"]), c["eps"])
    _close_printed(y, c["y"], c["decimals"])
    _close_printed(r, [c["r"]], c["decimals"])
    _close_printed(1.0 / r, [c["denominator"]], c["decimals"])
    _close_printed(1.0 / r[0] ** 2 - c["eps"], c["mean_square"], 9)
    c = CASES["forward_3_4_gamma_2_half"]
    y, _ = impl.rms_forward(np.array(c["x"]), np.array(c["gamma"]), c["eps"])
    _close_printed(y, c["y"], c["decimals"])


def pin_worked_backward(impl):
    c = CASES["backward_3_4_dy_1_2"]
    x, g, dy = np.array(c["x"]), np.array(c["gamma"]), np.array(c["dy"])
    dx, _ = impl.rms_backward(x, g, dy, c["eps"])
    _close_printed(dx, c["dx"], c["decimals"])
    # The printed intermediate mean(u*x) = 5.5 fixes the second term: with r
    # from the forward, dx = r*u - x*r^3*5.5 must reproduce dx.
    _, r = impl.rms_forward(x, g, c["eps"])
    u = np.array(c["u"])
    alt = r[0] * u - x * r[0] ** 3 * c["mean_ux"]
    assert np.allclose(dx, alt, rtol=1e-12, atol=1e-15), (dx, alt)


def pin_masked_denominator(impl):
    c = CASES["masked_denominator_257_ones"]
    n = c["N"]
    x = np.full((1, n), c["value"])
    g = np.full(n, c["gamma"])
    y, r = impl.rms_forward(x, g, c["eps"])
    _close_printed(y[0], np.full(n, c["correct"]["y"]), c["decimals"])
    _close_printed(1.0 / r, [c["correct"]["denominator"]], c["decimals"])
    wrong = c["wrong_block_divisor"]["y"]
    assert np.all(np.abs(y - wrong) > 0.4)
    # The same row at N=256 and N=257 normalises to the same value: only the
    # true N enters the mean.
    y256, _ = impl.rms_forward(np.ones((1, 256)), np.ones(256), c["eps"])
    assert np.allclose(y256[0, 0], y[0, 0], rtol=1e-15)
    c3 = CASES["masked_denominator_3_ones_block_4"]
    _, r3 = impl.rms_forward(np.array(c3["x"]), np.ones(3), 0.0)
    assert abs(1.0 / r3[0] ** 2 - c3["correct_mean"]) < 1e-15, r3


def pin_sum_not_mean(impl):
    c = CASES["dgamma_sum_not_mean"]
    # With x rows of ones and eps = 0, r = 1 and the per-row contributions
    # dy*x*r are dy itself: the table's contributions.
    contrib = np.array(c["contributions"])
    x = np.ones_like(contrib)
    _, dg = impl.rms_backward(x, np.ones(contrib.shape[1]), contrib, 0.0)
    assert np.array_equal(dg, np.array(c["expected_sum"])), dg
    assert not np.allclose(dg, np.array(c["wrong_mean"]))
    # M = 1 versus M = 17 copies of the same row: the sum scales by 17.
    rng = np.random.default_rng(17)
    x1 = rng.standard_normal((1, 9))
    dy1 = rng.standard_normal((1, 9))
    g = rng.uniform(0.5, 1.5, 9)
    _, dg1 = impl.rms_backward(x1, g, dy1, 1e-6)
    _, dg17 = impl.rms_backward(np.repeat(x1, 17, 0), g, np.repeat(dy1, 17, 0), 1e-6)
    assert np.allclose(dg17, 17.0 * dg1, rtol=1e-13, atol=1e-15)
    # The dgamma-only sum: the table, and agreement with the full backward.
    assert np.array_equal(impl.rms_dgamma(x, contrib, 0.0), np.array(c["expected_sum"]))
    xs = rng.standard_normal((23, 11)) * rng.uniform(0.1, 10.0, (23, 1))
    dys = rng.standard_normal((23, 11))
    _, dgf = impl.rms_backward(xs, rng.uniform(0.5, 1.5, 11), dys, 1e-5)
    dgo, sc = impl.rms_dgamma(xs, dys, 1e-5, with_scales=True)
    assert np.allclose(dgo, dgf, rtol=1e-14, atol=1e-14 * sc.max())
    assert np.all(sc >= np.abs(dgo))


def _fd_loss_grads(impl, x, g, dy, eps, gemma, h_rel=1e-6):
    """Central differences of sum(dy * y) using the implementation's forward."""
    def L(xx, gg):
        y, _ = impl.rms_forward(xx, gg, eps, gemma)
        return float(np.sum(dy * y))
    x = x.copy()
    g = g.copy()
    dx = np.zeros_like(x)
    dg = np.zeros_like(g)
    for idx in np.ndindex(*x.shape):
        a = x[idx]
        h = h_rel * max(1.0, abs(a))
        x[idx] = a + h
        lp = L(x, g)
        x[idx] = a - h
        lm = L(x, g)
        x[idx] = a
        dx[idx] = (lp - lm) / (2 * h)
    for j in range(g.size):
        a = g[j]
        h = h_rel * max(1.0, abs(a))
        g[j] = a + h
        lp = L(x, g)
        g[j] = a - h
        lm = L(x, g)
        g[j] = a
        dg[j] = (lp - lm) / (2 * h)
    return dx, dg


FD_SHAPES = [
    # (M, N, gemma, eps, seed)
    (3, 5, 0, 1e-6, 1),
    (2, 7, 1, 1e-6, 2),
    (1, 1, 0, 1e-6, 3),
    (17, 9, 0, 1e-5, 4),
    (4, 257, 0, 1e-6, 5),
    (3, 6, 1, 0.3, 6),
]


def pin_finite_differences(impl):
    for M, N, gemma, eps, seed in FD_SHAPES:
        rng = np.random.default_rng(seed)
        x = rng.standard_normal((M, N)) * rng.uniform(0.2, 3.0, (M, 1))
        g = rng.normal(0.0 if gemma else 1.0, 0.3, N)
        dy = rng.standard_normal((M, N))
        dx, dg = impl.rms_backward(x, g, dy, eps, gemma)
        fdx, fdg = _fd_loss_grads(impl, x, g, dy, eps, gemma)
        sx = np.abs(dx).max() + 1.0
        sg = np.abs(dg).max() + 1.0
        assert np.max(np.abs(dx - fdx)) <= 2e-7 * sx * math.sqrt(M * N), (M, N, gemma, np.max(np.abs(dx - fdx)))
        assert np.max(np.abs(dg - fdg)) <= 2e-7 * sg * math.sqrt(M * N), (M, N, gemma, np.max(np.abs(dg - fdg)))


def pin_torch_float64(impl):
    import torch
    import torch.nn.functional as F

    for M, N, gemma, eps, seed in [(5, 33, 0, 1e-6, 11), (4, 257, 1, 1e-5, 12), (8, 128, 0, 0.0, 13)]:
        rng = np.random.default_rng(seed)
        x = rng.standard_normal((M, N)) * rng.uniform(0.1, 10.0, (M, 1))
        g = rng.normal(0.0 if gemma else 1.0, 0.2, N)
        dy = rng.standard_normal((M, N))
        tx = torch.tensor(x, dtype=torch.float64, requires_grad=True)
        tg = torch.tensor(g, dtype=torch.float64, requires_grad=True)
        w = (1.0 + tg) if gemma else tg
        ty = F.rms_norm(tx, (N,), weight=w, eps=eps)
        ty.backward(torch.tensor(dy, dtype=torch.float64))
        y, _ = impl.rms_forward(x, g, eps, gemma)
        dx, dg = impl.rms_backward(x, g, dy, eps, gemma)
        ref_y = ty.detach().numpy()
        assert np.allclose(y, ref_y, rtol=1e-13, atol=1e-14 * np.abs(ref_y).max()), "y vs torch"
        assert np.allclose(dx, tx.grad.numpy(), rtol=1e-11, atol=1e-12 * np.abs(dx).max()), "dx vs torch"
        assert np.allclose(dg, tg.grad.numpy(), rtol=1e-11, atol=1e-12 * np.abs(dg).max()), "dgamma vs torch"


def pin_invariants(impl):
    rng = np.random.default_rng(21)
    M, N = 6, 40
    x = rng.standard_normal((M, N)) * rng.uniform(0.1, 10.0, (M, 1))
    g = rng.uniform(0.5, 1.5, N)
    dy = rng.standard_normal((M, N))
    # Scale invariance at eps = 0: exact for powers of two, ~1 ulp otherwise.
    y0, _ = impl.rms_forward(x, g, 0.0)
    for k in (-3, 1, 5):
        yk, _ = impl.rms_forward(x * 2.0 ** k, g, 0.0)
        assert np.array_equal(yk, y0), k
    y3, _ = impl.rms_forward(3.0 * x, g, 0.0)
    assert np.allclose(y3, y0, rtol=1e-14, atol=0)
    # mean_j (y/g)^2 = ms / (ms + eps); checked at eps comparable to ms.
    for eps in (1e-6, 0.5, 4.0):
        y, _ = impl.rms_forward(x, g, eps)
        ms = np.array([sum(v * v for v in row) / N for row in x])
        lhs = np.mean((y / g) ** 2, axis=1)
        assert np.allclose(lhs, ms / (ms + eps), rtol=1e-13), eps
    # sum_j x_j dx_j = eps * r^3 * sum_j u_j x_j  (x is orthogonal to dx as eps -> 0).
    for eps in (1e-6, 0.25):
        dx, _ = impl.rms_backward(x, g, dy, eps)
        ms = np.array([sum(v * v for v in row) / N for row in x])
        r = 1.0 / np.sqrt(ms + eps)
        sux = np.array([sum(dy[i, j] * g[j] * x[i, j] for j in range(N)) for i in range(M)])
        lhs = np.sum(x * dx, axis=1)
        scale = np.sum(np.abs(x * dx), axis=1)
        assert np.allclose(lhs, eps * r ** 3 * sux, rtol=1e-9, atol=1e-12 * scale.max()), eps
    # Zero row: y = 0, r = eps^-1/2, dx = u / sqrt(eps), no dgamma contribution.
    eps = 1e-4
    z = np.zeros((1, 7))
    gz = rng.uniform(0.5, 1.5, 7)
    dyz = rng.standard_normal((1, 7))
    yz, rz = impl.rms_forward(z, gz, eps)
    assert np.array_equal(yz, z) and abs(rz[0] - 100.0) < 1e-12
    dxz, dgz = impl.rms_backward(z, gz, dyz, eps)
    assert np.allclose(dxz, dyz * gz / math.sqrt(eps), rtol=1e-14)
    assert np.array_equal(dgz, np.zeros(7))
    # N = 1: r = 1/sqrt(x^2+eps), y = x r g, dx = u * eps * r^3.
    for xv, eps in ((0.7, 1e-6), (-2.5, 0.5), (3.0, 1.0)):
        x1 = np.array([[xv]])
        y1, r1 = impl.rms_forward(x1, np.array([1.5]), eps)
        rr = 1.0 / math.sqrt(xv * xv + eps)
        assert abs(r1[0] - rr) <= 1e-15 * rr and abs(y1[0, 0] - xv * rr * 1.5) <= 1e-15 * abs(xv * rr * 1.5)
        dx1, dg1 = impl.rms_backward(x1, np.array([1.5]), np.array([[0.3]]), eps)
        # dx = r u - x r^3 (u x) cancels to u eps r^3: bound the error by the terms.
        terms = rr * 0.45 + xv * xv * rr ** 3 * 0.45
        assert abs(dx1[0, 0] - 0.45 * eps * rr ** 3) <= 1e-14 * terms, (xv, eps)
        assert abs(dg1[0] - 0.3 * xv * rr) <= 1e-15 * abs(0.3 * xv * rr)
    # Gemma(gamma) equals the plain form with weight 1 + gamma.
    gg = rng.normal(0.0, 0.1, N)
    ya, _ = impl.rms_forward(x, gg, 1e-6, 1)
    yb, _ = impl.rms_forward(x, 1.0 + gg, 1e-6, 0)
    assert np.array_equal(ya, yb)
    dxa, dga = impl.rms_backward(x, gg, dy, 1e-6, 1)
    dxb, dgb = impl.rms_backward(x, 1.0 + gg, dy, 1e-6, 0)
    assert np.array_equal(dxa, dxb) and np.array_equal(dga, dgb)


def pin_two_forms_agree(impl):
    for M, N, gemma, seed in [(7, 64, 0, 31), (5, 257, 1, 32), (2, 3, 0, 33)]:
        rng = np.random.default_rng(seed)
        x = rng.standard_normal((M, N)) * rng.uniform(0.01, 100.0, (M, 1))
        g = rng.normal(0.0 if gemma else 1.0, 0.2, N)
        dy = rng.standard_normal((M, N))
        dx, _, dxs, _ = impl.rms_backward(x, g, dy, 1e-6, gemma, with_scales=True)
        dx2 = impl.rms_backward_normed_form(x, g, dy, 1e-6, gemma)
        assert np.all(np.abs(dx - dx2) <= 1e-13 * (np.abs(dx) + dxs)), (M, N, gemma)


def pin_lowp_emulation(impl):
    """Cast-order emulation versus torch's own float32/bfloat16 conversions."""
    import torch

    rng = np.random.default_rng(41)
    M, N = 16, 96
    # inputs exactly representable in bf16
    x = torch.tensor(rng.standard_normal((M, N)) * 3.0, dtype=torch.float32).to(torch.bfloat16).float()
    g = torch.tensor(rng.uniform(0.5, 1.5, N), dtype=torch.float32).to(torch.bfloat16).float()
    eps = 1e-6
    r32 = torch.tensor(impl.rms_rstd(x.double().numpy(), eps), dtype=torch.float32)
    normed = (x * r32[:, None]).to(torch.bfloat16).float()
    ref = (normed * g[None, :]).to(torch.bfloat16).double().numpy()
    got = impl.emulate_forward_lowp(x.double().numpy(), g.double().numpy(), eps, 0, "bf16")
    assert np.array_equal(got, ref)
    gw = (1.0 + g.double()).float()
    ref_g = ((x * r32[:, None]) * gw[None, :]).to(torch.bfloat16).double().numpy()
    got_g = impl.emulate_forward_lowp(x.double().numpy(), g.double().numpy(), eps, 1, "bf16")
    assert np.array_equal(got_g, ref_g)
    # Within two bf16 roundings (unit roundoff 2^-8 each) of the exact value,
    # and not always equal to a single rounding of it.
    exact, _ = impl.rms_forward(x.double().numpy(), g.double().numpy(), eps)
    assert np.all(np.abs(got - exact) <= (2.0 ** -7 + 2.0 ** -16) * np.abs(exact) + 1e-30)
    once = torch.tensor(exact).float().to(torch.bfloat16).double().numpy()
    assert not np.array_equal(got, once)
    # float16 I/O: the same order with torch's float16 conversions.
    xh = torch.tensor(rng.standard_normal((M, N)) * 3.0, dtype=torch.float32).to(torch.float16).float()
    gh = torch.tensor(rng.uniform(0.5, 1.5, N), dtype=torch.float32).to(torch.float16).float()
    r16 = torch.tensor(impl.rms_rstd(xh.double().numpy(), eps), dtype=torch.float32)
    ref_h = ((xh * r16[:, None]).to(torch.float16).float() * gh[None, :]).to(torch.float16)
    got_h = impl.emulate_forward_lowp(xh.double().numpy(), gh.double().numpy(), eps, 0, "f16")
    assert np.array_equal(got_h, ref_h.double().numpy())
    # bf16 activations with a float32 weight: x*r stays float32, one rounding at the end.
    gw = torch.tensor(rng.uniform(0.5, 1.5, N), dtype=torch.float32)
    ref_w = ((x * r32[:, None]) * gw[None, :]).to(torch.bfloat16).double().numpy()
    got_w = impl.emulate_forward_lowp(x.double().numpy(), gw.double().numpy(), eps, 0, "bf16", "f32")
    assert np.array_equal(got_w, ref_w)


ALL_PINS = [
    pin_worked_forward,
    pin_worked_backward,
    pin_masked_denominator,
    pin_sum_not_mean,
    pin_finite_differences,
    pin_torch_float64,
    pin_invariants,
    pin_two_forms_agree,
    pin_lowp_emulation,
]
