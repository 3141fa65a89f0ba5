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

The scaled dgamma bar above grows with sum_i |terms| (like M) while dgamma
itself grows like sqrt(M) for signed terms, so at large M it cannot see a
few dropped rows.  Two more checks stand beside it for every column sum
(dgamma; LayerNorm's dw and db):

* normwise: ||e|| / ||ref|| <= the dtype's dgamma tolerance (the stated
  "rel <= 2e-3" for bf16, read over the whole vector);
* tight elementwise: |e| <= tol |ref| + (g_D + t) S + s S_stat, derived
  from how the kernels sum, not fitted:
  - the sum runs through P float32 partial rows, each of at most n rows'
    terms (both reported by the library's rms_bwd_reduction /
    ln_bwd_reduction for the call's mapping).  Any fixed order of float32
    additions of k terms carries each term through at most k - 1
    roundings, so with D = n + P the summation adds at most
    g_D = D u / (1 - D u) of S = sum_i |term| (u = 2^-24, the float32
    unit roundoff);
  - t is each term's own relative error before it is added: RMSNorm forms
    dy * (x r) from the forward's stored r, so t = rstd's bar (1e-6, the
    bound the same tests enforce on that r) + 2u (x r rounded, the product
    rounded); LayerNorm's dw forms dy * xhat with xhat = fma(x, rstd,
    -mean rstd): t = u, and the stored mean and rstd (checked at 1e-5)
    move xhat by at most (1e-5 + 2u)(|xhat| + (|mean| + mean|x|) rstd),
    which enters through S_stat = sum_i |dy| (|xhat| + (|mean| + mean|x|)
    rstd); db sums dy itself (t = 0).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

U32 = 2.0 ** -24  # float32 unit roundoff

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
    err_sq: float = 0.0  # sum of squared errors (finite elements), for merging blocks
    ref_sq: float = 0.0  # sum of squared reference values (finite elements)

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
    ref_sq = float(np.sum(np.square(ref[fin]))) if fin.any() else 0.0
    err_sq = float(np.sum(np.square(err[fin]))) if fin.any() else 0.0
    nref, nerr = float(np.sqrt(ref_sq)), float(np.sqrt(err_sq))
    return Check(
        name=name,
        ok=not bool(bad.any()),
        n=int(ref.size),
        n_bad=int(bad.sum()),
        max_abs=float(err[fin].max()) if fin.any() else 0.0,
        max_rel=float(rel[fin].max()) if fin.any() else 0.0,
        norm_rel=(nerr / nref) if nref > 0 else nerr,
        worst_ratio=float(ratio[fin].max()) if fin.any() else 0.0,
        err_sq=err_sq,
        ref_sq=ref_sq,
    )


def merge(checks) -> Check:
    """One check over the union of the elements of several blocks' checks
    (of the same bar): counts add, maxima are taken, the normwise error is
    recomputed from the blocks' sums of squares."""
    checks = list(checks)
    err_sq = sum(c.err_sq for c in checks)
    ref_sq = sum(c.ref_sq for c in checks)
    nerr, nref = float(np.sqrt(err_sq)), float(np.sqrt(ref_sq))
    return Check(
        name=checks[0].name,
        ok=all(c.ok for c in checks),
        n=sum(c.n for c in checks),
        n_bad=sum(c.n_bad for c in checks),
        max_abs=max(c.max_abs for c in checks),
        max_rel=max(c.max_rel for c in checks),
        norm_rel=(nerr / nref) if nref > 0 else nerr,
        worst_ratio=max(c.worst_ratio for c in checks),
        err_sq=err_sq,
        ref_sq=ref_sq,
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


# ---- column sums: normwise and depth-derived elementwise bars ----

def sum_error_factor(reduction) -> float:
    """g_D = D u / (1 - D u), D = rows_per_partial + partials, for the
    library's reported (partials, rows_per_partial) of a column sum."""
    partials, rows = (int(v) for v in reduction)
    d = rows + partials
    return d * U32 / (1.0 - d * U32)


def check_normwise(name: str, got, ref, tol: float) -> Check:
    """||got - ref|| / ||ref|| <= tol over the whole vector."""
    c = _check(name, got, ref, np.inf)
    c.name = name
    c.ok = c.ok and c.norm_rel <= tol
    c.worst_ratio = c.norm_rel / tol
    return c


def check_sum_tight(name: str, got, ref, scale, dtype: str, reduction, term_rel: float,
                    stat_scale=None, stat_rel: float = 0.0) -> Check:
    """|e| <= tol |ref| + (g_D + term_rel) scale + stat_rel stat_scale."""
    ref = np.asarray(ref, np.float64)
    allowed = (TOL[dtype]["dgamma"] * np.abs(ref)
               + (sum_error_factor(reduction) + term_rel) * np.asarray(scale, np.float64))
    if stat_scale is not None:
        allowed = allowed + stat_rel * np.asarray(stat_scale, np.float64)
    c = _check(name, got, ref, allowed)
    return c


# Each RMSNorm dgamma term dy * (x r): r within rstd's bar, x r and the
# product each rounded once.
RMS_TERM_REL = TOL["f32"]["rstd"] + 2 * U32


def dgamma_checks(got, ref, scale, dtype: str, reduction, name: str = "dgamma"):
    """The scaled bar, the normwise bar and the tight elementwise bar."""
    c0 = check_dgamma(got, ref, scale, dtype)
    c0.name = name
    return [c0,
            check_normwise(name + "_normwise", got, ref, TOL[dtype]["dgamma"]),
            check_sum_tight(name + "_tight", got, ref, scale, dtype, reduction, RMS_TERM_REL)]


def ln_wsum_checks(got_dw, dw, dw_scale, dw_abs, dw_stat, got_db, db, db_scale, dtype: str,
                   reduction):
    """LayerNorm's dw (and db unless got_db is None): the scaled, normwise
    and tight bars.  dw_abs = sum_i |dy xhat|, dw_stat = sum_i |dy| (|xhat| +
    (|mean| + mean|x|) rstd), db_scale = sum_i |dy| (exact terms)."""
    out = [check_ln_wsum("dw", got_dw, dw, dw_scale, dtype),
           check_normwise("dw_normwise", got_dw, dw, TOL[dtype]["dgamma"]),
           check_sum_tight("dw_tight", got_dw, dw, dw_abs, dtype, reduction, U32,
                           dw_stat, LN_STAT_TOL + 2 * U32)]
    if got_db is not None:
        out += [check_ln_wsum("db", got_db, db, db_scale, dtype),
                check_normwise("db_normwise", got_db, db, TOL[dtype]["dgamma"]),
                check_sum_tight("db_tight", got_db, db, db_scale, dtype, reduction, 0.0)]
    return out


# ---- the weight gradient rounded to the weight's type ----

# Unit roundoff and smallest subnormal spacing of each weight type.
WEIGHT_ROUNDOFF = {"bf16": (2.0 ** -8, 2.0 ** -133), "f16": (2.0 ** -11, 2.0 ** -24),
                   "f32": (0.0, 0.0)}


def check_weight_cast(got, ref, scale, dtype: str, wdtype: str, reduction) -> Check:
    """dgamma after its rounding to the weight type ``wdtype``: the tight
    float32 bar b of the column sum, then one round to nearest in the weight
    type, |e| <= b + u_w (|ref| + b) + s_w / 2 (u_w the type's unit
    roundoff, s_w its subnormal spacing)."""
    ref = np.asarray(ref, np.float64)
    b = (TOL[dtype]["dgamma"] * np.abs(ref)
         + (sum_error_factor(reduction) + RMS_TERM_REL) * np.asarray(scale, np.float64))
    u, s = WEIGHT_ROUNDOFF[wdtype]
    c = _check("dgamma_cast", got, ref, b + u * (np.abs(ref) + b) + 0.5 * s)
    return c
