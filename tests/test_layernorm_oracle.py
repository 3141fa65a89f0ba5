"""The fp64 LayerNorm oracle against facts fixed outside it (CPU only), and
planted mistakes in copies of it that the pins must catch."""
import importlib.util
import os

import numpy as np
import pytest

ORACLE_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "layernorm_oracle.py")


def _load(tag):
    spec = importlib.util.spec_from_file_location(f"ln_oracle_{tag}", ORACLE_PATH)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _case(M, N, seed, shift=-2.3, scale=0.5):
    # the LN chapter's test draws x = -2.3 + 0.5 * randn, w, b ~ U(0, 1), dy = 0.1 * randn
    rng = np.random.default_rng(seed)
    x = shift + scale * rng.standard_normal((M, N))
    w = rng.uniform(0.0, 1.0, N)
    b = rng.uniform(0.0, 1.0, N)
    dy = 0.1 * rng.standard_normal((M, N))
    return x, w, b, dy


def pin_torch_float64(o):
    import torch
    import torch.nn.functional as F

    for M, N, eps, seed in [(6, 33, 1e-5, 1), (3, 257, 1e-6, 2), (4, 128, 0.5, 3)]:
        x, w, b, dy = _case(M, N, seed)
        tx = torch.tensor(x, requires_grad=True)
        tw = torch.tensor(w, requires_grad=True)
        tb = torch.tensor(b, requires_grad=True)
        ty = F.layer_norm(tx, (N,), tw, tb, eps)
        ty.backward(torch.tensor(dy))
        y, mean, rstd = o.ln_forward(x, w, b, eps)
        dx, dw, db = o.ln_backward(x, w, dy, eps)
        assert np.allclose(y, ty.detach().numpy(), rtol=1e-12, atol=1e-13)
        assert np.allclose(dx, tx.grad.numpy(), rtol=1e-10, atol=1e-12 * np.abs(dx).max())
        assert np.allclose(dw, tw.grad.numpy(), rtol=1e-10, atol=1e-12 * np.abs(dw).max())
        assert np.allclose(db, tb.grad.numpy(), rtol=1e-12, atol=1e-14)


def pin_finite_differences(o):
    for M, N, eps, seed in [(3, 5, 1e-5, 11), (2, 7, 0.3, 12), (5, 2, 1e-3, 13)]:
        x, w, b, dy = _case(M, N, seed)
        dx, dw, db = o.ln_backward(x, w, dy, eps)
        fx, fw, fb = o.ln_fd_gradients(x, w, b, dy, eps)
        for a, f in ((dx, fx), (dw, fw), (db, fb)):
            assert np.max(np.abs(a - f)) <= 1e-6 * (1 + np.abs(a).max()), (M, N, np.abs(a - f).max())


def pin_invariants(o):
    x, w, b, dy = _case(9, 48, 21, shift=0.7, scale=3.0)
    # shift invariance: adding a constant to a row changes nothing
    y0, _, _ = o.ln_forward(x, w, b, 1e-5)
    y1, _, _ = o.ln_forward(x + 5.0, w, b, 1e-5)
    assert np.allclose(y0, y1, rtol=1e-11, atol=1e-11)
    # with w = 1, b = 0: each row of y has mean 0 and mean square var/(var+eps)
    for eps in (1e-6, 0.5):
        y, mean, rstd = o.ln_forward(x, np.ones(48), np.zeros(48), eps)
        var = np.array([sum((v - sum(row) / 48) ** 2 for v in row) / 48 for row in x])
        assert np.allclose(np.mean(y, axis=1), 0.0, atol=1e-12)
        assert np.allclose(np.mean(y * y, axis=1), var / (var + eps), rtol=1e-12)
        assert np.allclose(mean, x.mean(axis=1), rtol=1e-14)
    # dx sums to zero over each row; sum_j dx_j xhat_j = N c1 eps rstd^3
    for eps in (1e-5, 0.25):
        dx, _, _ = o.ln_backward(x, w, dy, eps)
        scale = np.abs(dx).sum(axis=1)
        assert np.all(np.abs(dx.sum(axis=1)) <= 1e-12 * scale)
        mean, rstd = o.ln_stats(x, eps)
        xhat = (x - mean[:, None]) * rstd[:, None]
        c1 = np.array([sum(xhat[i, j] * w[j] * dy[i, j] for j in range(48)) / 48 for i in range(9)])
        lhs = np.sum(dx * xhat, axis=1)
        assert np.allclose(lhs, 48 * c1 * eps * rstd ** 3, rtol=1e-8, atol=1e-12 * scale.max())
    # db is the column sum of dy (sum, not mean); dw of one row is dy * xhat
    _, _, db = o.ln_backward(x, w, dy, 1e-5)
    assert np.allclose(db, [sum(dy[i, j] for i in range(9)) for j in range(48)], rtol=1e-13)
    _, dw1, _ = o.ln_backward(x[:1], w, dy[:1], 1e-5)
    _, dw17, db17 = o.ln_backward(np.repeat(x[:1], 17, 0), w, np.repeat(dy[:1], 17, 0), 1e-5)
    assert np.allclose(dw17, 17 * dw1, rtol=1e-13)
    assert np.allclose(db17, 17 * dy[0], rtol=1e-13)
    # a constant row: x - mean = 0, so y = b and rstd = eps^-1/2
    yc, mc, rc = o.ln_forward(np.full((1, 6), 3.5), w[:6], b[:6], 1e-4)
    assert np.allclose(yc[0], b[:6], rtol=0, atol=1e-15) and abs(rc[0] - 100.0) < 1e-12 and mc[0] == 3.5
    # without bias
    yn, _, _ = o.ln_forward(x, w, None, 1e-5)
    assert np.allclose(yn + b[None, :], y0, rtol=1e-14, atol=1e-14)


def pin_two_pass_variance(o):
    """A large common offset: the centred second pass keeps the variance, a
    one-pass E[x^2]-E[x]^2 in float64 would lose most of its digits."""
    rng = np.random.default_rng(5)
    base = rng.standard_normal((1, 64))
    x = 1e7 + base
    _, rstd = o.ln_stats(x, 0.0)
    var_true = np.var(base)  # the offset does not change the variance
    assert abs(1.0 / rstd[0] ** 2 - var_true) <= 1e-7 * var_true


def pin_wsum_term_scales(o):
    """The sizes of dw's row terms, by plain loops, and what the second one
    bounds: moving each row's mean by d (|mean| + mean|x|) and its rstd by a
    factor (1 + d) changes dw by at most d times it (to first order)."""
    x, w, b, dy = _case(5, 6, 31)
    eps = 1e-5
    s_abs, s_stat = o.ln_wsum_term_scales(x, dy, eps)
    M, N = x.shape
    for j in range(N):
        a = st = 0.0
        for i in range(M):
            mu = sum(x[i]) / N
            var = sum((v - mu) ** 2 for v in x[i]) / N
            r = 1.0 / (var + eps) ** 0.5
            xh = (x[i, j] - mu) * r
            a += abs(dy[i, j] * xh)
            st += abs(dy[i, j]) * (abs(xh) + (abs(mu) + sum(abs(v) for v in x[i]) / N) * r)
        assert abs(s_abs[j] - a) <= 1e-13 * a and abs(s_stat[j] - st) <= 1e-13 * st, j
    _, dw, _ = o.ln_backward(x, w, dy, eps)
    assert np.all(s_abs >= np.abs(dw) * (1 - 1e-14))
    mean, rstd = o.ln_stats(x, eps)
    d = 1e-6
    rng = np.random.default_rng(4)
    for _ in range(4):
        sg1, sg2 = rng.choice([-1.0, 1.0], M), rng.choice([-1.0, 1.0], M)
        m2 = mean + sg1 * d * (np.abs(mean) + np.mean(np.abs(x), axis=1))
        r2 = rstd * (1 + sg2 * d)
        dw2 = np.sum(dy * (x - m2[:, None]) * r2[:, None], axis=0)
        assert np.all(np.abs(dw2 - dw) <= d * s_stat * (1 + 1e-6))


ALL_PINS = [pin_torch_float64, pin_finite_differences, pin_invariants, pin_two_pass_variance,
            pin_wsum_term_scales]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_layernorm_oracle_pin(pin):
    pin(_load("real"))


def _mutant(name):
    m = _load(name)
    if name == "no_mean_subtraction":
        m.ln_stats = lambda x, eps: (np.zeros(np.shape(x)[0]),
                                     1.0 / np.sqrt(np.mean(np.asarray(x) ** 2, axis=-1) + eps))
    elif name == "unbiased_variance":
        def st(x, eps):
            x = np.asarray(x, np.float64)
            mu = np.mean(x, axis=-1)
            return mu, 1.0 / np.sqrt(np.var(x, axis=-1, ddof=1) + eps)
        m.ln_stats = st
    elif name == "one_pass_variance":
        def st(x, eps):
            x = np.asarray(x, np.float64)
            mu = np.mean(x, axis=-1)
            return mu, 1.0 / np.sqrt(np.mean(x * x, axis=-1) - mu * mu + eps)
        m.ln_stats = st
    elif name in ("dx_without_c2", "dx_without_c1", "dw_mean", "db_mean", "dw_without_xhat"):
        orig = m.ln_backward

        def bwd(x, w, dy, eps, with_scales=False, _m=m, _v=name):
            x = np.asarray(x, np.float64)
            dy = np.asarray(dy, np.float64)
            mean, rstd = _m.ln_stats(x, eps)
            xhat = (x - mean[:, None]) * rstd[:, None]
            gh = dy * np.asarray(w)[None, :]
            c1 = 0.0 if _v == "dx_without_c1" else np.mean(xhat * gh, axis=-1)[:, None]
            c2 = 0.0 if _v == "dx_without_c2" else np.mean(gh, axis=-1)[:, None]
            dx = (gh - (xhat * c1 + c2)) * rstd[:, None]
            dw = (np.mean if _v == "dw_mean" else np.sum)(dy * (x if _v == "dw_without_xhat" else xhat), axis=0)
            db = (np.mean if _v == "db_mean" else np.sum)(dy, axis=0)
            return dx, dw, db
        m.ln_backward = bwd
    elif name == "bias_ignored":
        orig = m.ln_forward
        m.ln_forward = lambda x, w, b, eps, _o=orig: _o(x, w, None, eps)
    return m


LN_MUTANTS = ["no_mean_subtraction", "unbiased_variance", "one_pass_variance", "dx_without_c2",
              "dx_without_c1", "dw_mean", "db_mean", "dw_without_xhat", "bias_ignored"]


@pytest.mark.parametrize("name", LN_MUTANTS)
def test_layernorm_mutant_is_caught(name):
    m = _mutant(name)
    caught = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(m)
        except (AssertionError, FloatingPointError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name!r} passes every LayerNorm pin"
