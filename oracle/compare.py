"""Tolerance checks of CUDA results against the fp64 oracle.

TEST INFRASTRUCTURE ONLY (imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg).

Bars, per output and I/O dtype:

* f32 I/O: y rel <= 1e-5; dx rel <= 1e-5; dgamma rel <= 1e-4.
* bf16 I/O: y and dx ``|err| <= 1e-2 * max(1, |ref|)``; dgamma (accumulated in
  fp32, stored fp32) rel <= 2e-3.
* f16 I/O: y and dx ``|err| <= 3e-3 + 3e-3 |ref|`` (the Triton RMSNorm
  tutorial's published FP16 bar, atol = rtol = 3e-3, § "Các phép đo trước khi
  xem kết quả"); dgamma rel <= 1e-3.
* rstd (always fp32): rel <= 1e-6.

"rel" is read elementwise against the size of the terms the value is built
from, because dx and dgamma are differences/sums of signed terms that can
cancel to ~0 (where a plain |err|/|ref| is ill-posed):

* y:      |e| <= tol * |ref|
* dx:     |e| <= tol * (|ref| + r|u| + |x| r^3 mean|u x|)   (c = mean(u x) is
          itself a sum of signed terms)
* dgamma: |e| <= tol * (|ref| + sum_i |dy x r|)

LayerNorm keeps the per-dtype bars and adds a float32 term for what the
method's float32 mean costs: x - mean cancels, so the rounding of the mean
(relative to |x| + |mean|) reaches xhat multiplied by rstd.  With X = (|x| +
|mean|) rstd standing for xhat before that cancellation (the fp64 LayerNorm
oracle reports these scales):

* y:      |e| <= bar(y) + 1e-5 (X |w| + |b|)
* dx:     |e| <= bar(dx) + 1e-5 rstd (|g| + mean|g| + X mean(X |g|))
* dw, db: the dgamma bar with scales sum_i |dy| X and sum_i |dy|
* mean:   |e| <= 1e-5 (|ref| + mean|x|), rstd: rel <= 1e-5.  Both are float32
          sums of up to a few hundred terms in sequence (a thread's share of
          a row, then the tree): (L + depth) u <= ~1e-5 relative to the sum of
          magnitudes, with u = 2^-24.

bar() is RMSNorm's y/dx bar for the dtype (for f32: 1e-5 |ref|).

Each check also reports the plain max abs / max rel error and the normwise
relative error ||e|| / ||ref|| for information.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

TOL = {
    "f32": {"y": 1e-5, "dx": 1e-5, "dgamma": 1e-4, "rstd": 1e-6},
    "bf16": {"y": 1e-2, "dx": 1e-2, "dgamma": 2e-3, "rstd": 1e-6},
    "f16": {"y": 3e-3, "dx": 3e-3, "dgamma": 1e-3, "rstd": 1e-6},
}


@dataclass
class Check:
    name: str
    ok: bool
    n: int
    n_bad: int
    max_abs: float
    max_rel: float
    norm_rel: float
    worst_ratio: float  # max |e| / allowed; <= 1 means pass

    def __str__(self) -> str:
        return (f"{self.name}: {'ok' if self.ok else 'FAIL'} n={self.n} bad={self.n_bad} "
                f"max_abs={self.max_abs:.3e} max_rel={self.max_rel:.3e} "
                f"norm_rel={self.norm_rel:.3e} worst/allowed={self.worst_ratio:.3f}")


def _check(name: str, got, ref, allowed) -> Check:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    allowed = np.broadcast_to(np.asarray(allowed, dtype=np.float64), ref.shape)
    with np.errstate(invalid="ignore"):
        err = np.abs(got - ref)
    finite = np.isfinite(got) & np.isfinite(ref)
    same_nonfinite = (~np.isfinite(ref)) & (
        (np.isnan(ref) & np.isnan(got)) | (ref == got))
    bad = ~((finite & (err <= allowed)) | same_nonfinite)
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(np.abs(ref) > 0, err / np.abs(ref), np.where(err > 0, np.inf, 0.0))
        ratio = np.where(allowed > 0, err / allowed, np.where(err > 0, np.inf, 0.0))
    fin = finite
    nref = float(np.linalg.norm(ref[fin])) if fin.any() else 0.0
    nerr = float(np.linalg.norm(err[fin])) if fin.any() else 0.0
    return Check(
        name=name,
        ok=not bool(bad.any()),
        n=int(ref.size),
        n_bad=int(bad.sum()),
        max_abs=float(err[fin].max()) if fin.any() else 0.0,
        max_rel=float(rel[fin].max()) if fin.any() else 0.0,
        norm_rel=(nerr / nref) if nref > 0 else nerr,
        worst_ratio=float(ratio[fin].max()) if fin.any() else 0.0,
    )


def check_rstd(got, ref) -> Check:
    return _check("rstd", got, ref, TOL["f32"]["rstd"] * np.abs(np.asarray(ref, np.float64)))


def check_y(got, ref, dtype: str) -> Check:
    ref = np.asarray(ref, np.float64)
    if dtype == "bf16":
        allowed = TOL["bf16"]["y"] * np.maximum(1.0, np.abs(ref))
    elif dtype == "f16":
        allowed = TOL["f16"]["y"] * (1.0 + np.abs(ref))
    else:
        allowed = TOL["f32"]["y"] * np.abs(ref)
    return _check("y", got, ref, allowed)


def check_dx(got, ref, scale, dtype: str) -> Check:
    ref = np.asarray(ref, np.float64)
    if dtype == "bf16":
        allowed = TOL["bf16"]["dx"] * np.maximum(1.0, np.abs(ref))
    elif dtype == "f16":
        allowed = TOL["f16"]["dx"] * (1.0 + np.abs(ref))
    else:
        allowed = TOL["f32"]["dx"] * (np.abs(ref) + np.asarray(scale, np.float64))
    return _check("dx", got, ref, allowed)


def check_dgamma(got, ref, scale, dtype: str) -> Check:
    ref = np.asarray(ref, np.float64)
    tol = TOL[dtype]["dgamma"]
    return _check("dgamma", got, ref, tol * (np.abs(ref) + np.asarray(scale, np.float64)))


# ---- LayerNorm ----
LN_STAT_TOL = 1e-5


def check_ln_y(got, ref, scale, dtype: str) -> Check:
    ref = np.asarray(ref, np.float64)
    extra = TOL["f32"]["y"] * np.asarray(scale, np.float64)
    return _check("y", got, ref, _bar(ref, dtype, "y") + extra)


def check_ln_mean(got, ref, abs_mean) -> Check:
    ref = np.asarray(ref, np.float64)
    return _check("mean", got, ref, LN_STAT_TOL * (np.abs(ref) + np.asarray(abs_mean, np.float64)))


def check_ln_rstd(got, ref) -> Check:
    ref = np.asarray(ref, np.float64)
    return _check("rstd", got, ref, LN_STAT_TOL * np.abs(ref))


def check_ln_dx(got, ref, scale, dtype: str) -> Check:
    ref = np.asarray(ref, np.float64)
    extra = TOL["f32"]["dx"] * np.asarray(scale, np.float64)
    return _check("dx", got, ref, _bar(ref, dtype, "dx") + extra)


def _bar(ref, dtype: str, what: str):
    if dtype == "bf16":
        return TOL["bf16"][what] * np.maximum(1.0, np.abs(ref))
    if dtype == "f16":
        return TOL["f16"][what] * (1.0 + np.abs(ref))
    return TOL["f32"][what] * np.abs(ref)


def check_ln_wsum(name: str, got, ref, scale, dtype: str) -> Check:
    """dw or db (float32 sums over rows), at the dgamma bar."""
    c = check_dgamma(got, ref, scale, dtype)
    c.name = name
    return c
