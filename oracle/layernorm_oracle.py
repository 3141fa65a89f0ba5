"""Plain fp64 CPU oracle for row-wise LayerNorm, forward and backward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  It shares no
code with the CUDA library.

Source: "第 07 章:LayerNorm——反向传播与原子锁" ([LN]):
  - step 3 (forward): per row mean = Σx/N, var = Σ(x − mean)²/N (a second
    pass over the centred values), rstd = 1/sqrt(var + eps),
    y = (x − mean)·rstd·w + b; mean and rstd are kept for the backward;
  - § 3.0 (backward): x̂ = (x − mean)·rstd, ĝ = w·dy, c1 = Σ x̂·ĝ / N,
    c2 = Σ ĝ / N, dx = (ĝ − (x̂·c1 + c2))·rstd; the weight and bias
    gradients are the row contributions dy·x̂ and dy summed over all rows.

Every function evaluates those definitions directly in float64 on the exact
values of the (dtype-rounded) inputs.  Library primitives used as steps:
``np.mean`` / ``np.sum``, ``np.sqrt``.  Every function is pinned by
``tests/test_layernorm_oracle.py`` (torch's float64 layer_norm and autograd,
central differences, closed forms, invariants); none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def ln_stats(x, eps: float):
    """(mean, rstd) per row: mean = Σx/N, var = Σ(x − mean)²/N, rstd = 1/sqrt(var + eps)."""
    x = _f64(x)
    mean = np.mean(x, axis=-1)
    d = x - mean[:, None]
    var = np.mean(d * d, axis=-1)
    return mean, 1.0 / np.sqrt(var + eps)


def ln_forward(x, w, b, eps: float, with_scales: bool = False):
    """y = (x − mean)·rstd·w + b (b may be None: no bias).  Returns (y, mean, rstd).

    With ``with_scales`` also ``y_scale = X·|w| + |b|`` with ``X = (|x| +
    |mean|)·rstd`` (the magnitudes of the terms y is made of before
    x − mean and the bias cancel, for tolerances) and ``abs_mean = Σ|x|/N``
    per row (the size of the terms of the mean).
    """
    x = _f64(x)
    mean, rstd = ln_stats(x, eps)
    xhat = (x - mean[:, None]) * rstd[:, None]
    y = xhat * _f64(w)[None, :]
    if b is not None:
        y = y + _f64(b)[None, :]
    if not with_scales:
        return y, mean, rstd
    X = (np.abs(x) + np.abs(mean)[:, None]) * rstd[:, None]
    y_scale = X * np.abs(_f64(w))[None, :]
    if b is not None:
        y_scale = y_scale + np.abs(_f64(b))[None, :]
    return y, mean, rstd, y_scale, np.mean(np.abs(x), axis=-1)


def ln_backward(x, w, dy, eps: float, with_scales: bool = False):
    """Gradients of L = Σ dy ⊙ y: (dx, dw, db), from the [LN] § 3.0 closed form.

    With ``with_scales`` also the sizes of the terms each output is built
    from, for tolerances where they cancel, with ``X = (|x| + |mean|)·rstd``
    standing for x̂ before x − mean cancels: ``dx_scale = rstd·(|ĝ| +
    mean|ĝ| + X·mean(X·|ĝ|))``, ``dw_scale = Σ_i |dy|·X`` and ``db_scale =
    Σ_i |dy|``.
    """
    x = _f64(x)
    dy = _f64(dy)
    mean, rstd = ln_stats(x, eps)
    xhat = (x - mean[:, None]) * rstd[:, None]
    gh = dy * _f64(w)[None, :]
    c1 = np.mean(xhat * gh, axis=-1)
    c2 = np.mean(gh, axis=-1)
    dx = (gh - (xhat * c1[:, None] + c2[:, None])) * rstd[:, None]
    dw = np.sum(dy * xhat, axis=0)
    db = np.sum(dy, axis=0)
    if not with_scales:
        return dx, dw, db
    X = (np.abs(x) + np.abs(mean)[:, None]) * rstd[:, None]
    dx_scale = rstd[:, None] * (np.abs(gh) + np.mean(np.abs(gh), axis=-1)[:, None]
                                + X * np.mean(X * np.abs(gh), axis=-1)[:, None])
    dw_scale = np.sum(np.abs(dy) * X, axis=0)
    db_scale = np.sum(np.abs(dy), axis=0)
    return dx, dw, db, dx_scale, dw_scale, db_scale


def ln_wsum_term_scales(x, dy, eps: float):
    """Sizes of dw's row terms, for its error bound: ``(sum_i |dy·x̂|,
    sum_i |dy|·(|x̂| + (|mean| + mean|x|)·rstd))`` per column, the second
    being how far x̂ moves per unit relative error of the stored mean
    (relative to |mean| + mean|x|) and rstd."""
    x = _f64(x)
    dy = _f64(dy)
    mean, rstd = ln_stats(x, eps)
    xhat = (x - mean[:, None]) * rstd[:, None]
    stat = (np.abs(mean) + np.mean(np.abs(x), axis=-1)) * rstd
    return (np.sum(np.abs(dy * xhat), axis=0),
            np.sum(np.abs(dy) * (np.abs(xhat) + stat[:, None]), axis=0))


def ln_loss(x, w, b, dy, eps: float) -> float:
    y, _, _ = ln_forward(x, w, b, eps)
    return float(np.sum(_f64(dy) * y))


def ln_fd_gradients(x, w, b, dy, eps: float, h_rel: float = 1e-6):
    """Central differences of ``ln_loss`` for every entry of x, w and b (tiny inputs)."""
    x = _f64(x).copy()
    w = _f64(w).copy()
    b = _f64(b).copy()
    grads = []
    for arr in (x, w, b):
        g = np.zeros_like(arr)
        for idx in np.ndindex(*arr.shape):
            a = arr[idx]
            h = h_rel * max(1.0, abs(a))
            arr[idx] = a + h
            lp = ln_loss(x, w, b, dy, eps)
            arr[idx] = a - h
            lm = ln_loss(x, w, b, dy, eps)
            arr[idx] = a
            g[idx] = (lp - lm) / (2.0 * h)
        grads.append(g)
    return tuple(grads)
