"""Plain fp64 CPU oracle for row-wise RMSNorm, forward and backward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The CUDA
library never calls it and shares no code with it; the only thing both sides
share is the seeded input generator in ``synthetic/``.

Every function evaluates the textbook definition directly in float64 on the
exact values of the (already dtype-rounded) inputs: no blocking, fusion or
reordering beyond what the definition states.  Library primitives used as
steps: ``np.mean`` / ``np.sum`` (the row mean and the column sum), ``np.sqrt``.

Sources (web pages on row-wise RMS normalisation):

* [TUT] "Hướng dẫn Triton RMSNorm: kernel, backward…" (partitech.com):
  - § "Vấn đề và công thức tham chiếu": r = 1/sqrt(mean(x²)+eps),
    y = x·r·gamma, eps added under the square root;
  - § "Vì sao cần một lượt đi và một lượt về?": u = dy·gamma,
    dx = r·u − x·r³·mean(u·x) (mean over the N columns of a row),
    dgamma = Σ_rows dy·x·r (a sum over the M rows);
  - § "Lập phương của r từ đâu?": ∂r/∂x_i = −x_i·r³/N;
  - § "N và BLOCK: hai kích thước không được nhầm": divide by the true N.
* [UNS] "02 · 手写 Triton kernel:RMSNorm / RoPE / SwiGLU", § 3 (RMSNorm):
  - the alternative closed form dX = inv_var/n·(n·dY_W − normed·Σ(dY_W·normed));
  - Gemma weight semantics (1 + W);
  - § 2 item 3 and § 3: normed is cast to the weight dtype, then multiplied
    by the weight (the order ``emulate_forward_lowp`` reproduces).

* Fused residual add ([UNS] §§ 1-2: neighbouring elementwise work is kept
  in registers, each tensor read and written once): ``residual_add``,
  ``rms_forward_add`` and ``rms_backward_add`` compose the definitions above
  with h = x + residual as the residual stream stores it (the float32 sum
  rounded once to the I/O dtype) and dx = dRMS + dh.

* The weight gradient in the weight's type ([TUT] § "Reduce dgamma không có
  race khi ghi": reduced in fp32, then converted to gamma's dtype):
  ``cast_to_weight_dtype``, pinned by ``tests/test_cast_oracle.py``.

* Output quantised to FP8 E4M3 for the next GEMM (the same fusion principle):
  ``round_e4m3`` / ``e4m3_code`` (the format: sign, 4 exponent bits with
  bias 7, 3 mantissa bits, subnormals, no infinities, largest 448; round to
  nearest even, saturating) and ``quantize_rows_e4m3`` / ``rms_forward_quant``
  (per-row scale amax/448, codes of y·(448/amax) in float32).

Every function here is pinned by ``tests/test_oracle_pins.py`` (and, for the
fused residual add and the E4M3 output, ``tests/test_fused_add_oracle.py``
and ``tests/test_quant_oracle.py``) against values the
pages print, closed forms, invariants, finite differences, torch's own
dtype arithmetic and ``torch.nn.functional.rms_norm`` with autograd in
float64; none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def weight(gamma, gemma: int = 0) -> np.ndarray:
    """Effective per-column weight g: gamma, or 1 + gamma for Gemma ([UNS] § 3)."""
    g = _f64(gamma)
    return 1.0 + g if gemma else g


def rms_rstd(x, eps: float) -> np.ndarray:
    """r_i = 1 / sqrt(mean_j x_ij² + eps), mean over the true N ([TUT] reference formula)."""
    x = _f64(x)
    ms = np.mean(x * x, axis=-1)
    return 1.0 / np.sqrt(ms + eps)


def rms_forward(x, gamma, eps: float, gemma: int = 0):
    """y_ij = x_ij · r_i · g_j and r ([TUT] reference formula; [UNS] § 3 for Gemma).

    Returns (y, r) in float64; x is (M, N), gamma is (N,).
    """
    x = _f64(x)
    r = rms_rstd(x, eps)
    y = x * r[:, None] * weight(gamma, gemma)[None, :]
    return y, r


def rms_backward(x, gamma, dy, eps: float, gemma: int = 0, with_scales: bool = False):
    """Closed-form gradients of L = Σ dy ⊙ y ([TUT] backward formulas).

    u = dy · g;  c_i = mean_j(u_ij · x_ij);  dx = r·u − x·r³·c;
    dgamma_j = Σ_i dy_ij · x_ij · r_i  (a sum over rows, not a mean; for
    Gemma the same, since d(1+gamma)/dgamma = 1).

    With ``with_scales`` it also returns the magnitudes the two outputs are
    built from, used to scale tolerances where the terms cancel:
    ``dx_scale = r·|u| + |x|·r³·mean_j|u·x|`` (c is itself a mean of signed
    terms, so its rounding error scales with the mean of their sizes) and
    ``dgamma_scale = Σ_i |dy·x·r|``.
    """
    x = _f64(x)
    dy = _f64(dy)
    r = rms_rstd(x, eps)
    u = dy * weight(gamma, gemma)[None, :]
    c = np.mean(u * x, axis=-1)
    r3 = r ** 3
    dx = r[:, None] * u - x * (r3 * c)[:, None]
    dgamma = np.sum(dy * x * r[:, None], axis=0)
    if not with_scales:
        return dx, dgamma
    dx_scale = r[:, None] * np.abs(u) + np.abs(x) * (r3 * np.mean(np.abs(u * x), axis=-1))[:, None]
    dgamma_scale = np.sum(np.abs(dy * x * r[:, None]), axis=0)
    return dx, dgamma, dx_scale, dgamma_scale


def rms_dgamma(x, dy, eps: float, with_scales: bool = False):
    """dgamma_j = Σ_i dy_ij · x_ij · r_i alone ([TUT] § "Tổng không phải trung bình").

    The same sum ``rms_backward`` returns, without forming dx; with
    ``with_scales`` also Σ_i |dy·x·r| (the size of the summed terms).
    """
    x = _f64(x)
    dy = _f64(dy)
    r = rms_rstd(x, eps)
    terms = dy * x * r[:, None]
    dgamma = np.sum(terms, axis=0)
    if not with_scales:
        return dgamma
    return dgamma, np.sum(np.abs(terms), axis=0)


def rms_backward_normed_form(x, gamma, dy, eps: float, gemma: int = 0):
    """dx in [UNS] § 3's form: inv_var/n · (n·dY_W − normed·Σ_j(dY_W·normed)).

    normed = x·r, dY_W = dy·g.  Algebraically equal to ``rms_backward``'s dx.
    """
    x = _f64(x)
    dy = _f64(dy)
    n = x.shape[-1]
    r = rms_rstd(x, eps)
    normed = x * r[:, None]
    dyw = dy * weight(gamma, gemma)[None, :]
    s = np.sum(dyw * normed, axis=-1)
    return (r / n)[:, None] * (n * dyw - normed * s[:, None])


# --- low-precision cast-order emulation ------------------------------------

def _round_f32(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64).astype(np.float32)


def _round_bf16(a) -> np.ndarray:
    """float32 values rounded to the nearest bfloat16, ties to even (finite inputs)."""
    f = np.ascontiguousarray(_round_f32(a))
    bits = f.view(np.uint32).astype(np.uint64)
    keep = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + keep) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32)


def _round_f16(a) -> np.ndarray:
    """float32 values rounded to the nearest float16, ties to even (numpy's conversion)."""
    return _round_f32(a).astype(np.float16).astype(np.float32)


def emulate_forward_lowp(x, gamma, eps: float, gemma: int = 0, dtype: str = "bf16",
                         weight_dtype: str = ""):
    """The forward as a fp32-accumulating kernel with ``dtype`` I/O rounds it.

    Follows the cast order of [UNS] § 3: normed = fp32(x·r) is rounded to the
    weight dtype (``weight_dtype``, default ``dtype``; float32 makes this
    rounding exact) first, then multiplied by the weight in fp32 and rounded
    to ``dtype``.  For Gemma the weight (1+gamma) is formed in fp32 and the
    product x·r·(1+gamma) is rounded once (the pages state no order there).
    r is the fp64 value rounded to fp32.  Returns float64 values of the
    rounded y.
    """
    rounders = {"bf16": _round_bf16, "f16": _round_f16}
    rnd = rounders.get(dtype, _round_f32)
    rnd_w = rounders.get(weight_dtype or dtype, _round_f32)
    xf = _round_f32(x)
    gf = _round_f32(gamma)
    r32 = _round_f32(rms_rstd(x, eps))
    xr = _round_f32(xf.astype(np.float64) * r32[:, None])
    if gemma:
        w = _round_f32(1.0 + gf.astype(np.float64))
        y = rnd(_round_f32(xr.astype(np.float64) * w[None, :]))
    else:
        normed = rnd_w(xr)
        y = rnd(_round_f32(normed.astype(np.float64) * gf[None, :]))
    return y.astype(np.float64)


# ---- the weight gradient in the weight's own type ------------------------------

def cast_to_weight_dtype(v, wdtype: str) -> np.ndarray:
    """float32 values rounded to the weight type ``wdtype`` ("bf16" or "f16";
    "f32" leaves them unchanged), to nearest with ties to even; values past
    the type's largest finite one become infinities.  Returned as float64.

    [TUT] § "Reduce dgamma không có race khi ghi": the partial sums are
    reduced in fp32, and the result is then converted to gamma's dtype.
    """
    f = _round_f32(v)
    if wdtype == "bf16":
        return _round_bf16(f).astype(np.float64)
    if wdtype == "f16":
        return _round_f16(f).astype(np.float64)
    return f.astype(np.float64)


# ---- fused residual add ------------------------------------------------------

def residual_add(x, residual, dtype: str = "f32") -> np.ndarray:
    """h = x + residual as stored in ``dtype``: the IEEE float32 sum of the two
    (dtype-exact) inputs, rounded once more to ``dtype`` (nothing more for
    float32).  Returns the float64 values of h."""
    s = _round_f32(x) + _round_f32(residual)  # numpy float32 arithmetic: one rounding
    rnd = {"bf16": _round_bf16, "f16": _round_f16}.get(dtype, _round_f32)
    return rnd(s).astype(np.float64)


def rms_forward_add(x, residual, gamma, eps: float, gemma: int = 0, dtype: str = "f32"):
    """(y, r, h): h = residual_add(x, residual), then the RMSNorm of h."""
    h = residual_add(x, residual, dtype)
    y, r = rms_forward(h, gamma, eps, gemma)
    return y, r, h


def rms_backward_add(h, gamma, dy, dh, eps: float, gemma: int = 0, with_scales: bool = False):
    """dx = dRMS(dy; h) + dh (the gradient reaching h through the residual
    path) and dgamma of the RMSNorm of h.  With ``with_scales`` the dx scale
    is rms_backward's plus |dh|."""
    out = rms_backward(h, gamma, dy, eps, gemma, with_scales=with_scales)
    dx = out[0] + _f64(dh)
    if not with_scales:
        return dx, out[1]
    return dx, out[1], out[2] + np.abs(_f64(dh)), out[3]


# ---- FP8 E4M3 output ---------------------------------------------------------

E4M3_MAX = 448.0


def round_e4m3(v) -> np.ndarray:
    """Nearest E4M3 value (ties to even), saturating at ±448: spacing 2^(e-3)
    for |v| in [2^e, 2^(e+1)), e >= -6, and 2^-9 below 2^-6 (subnormals)."""
    v = _f64(v)
    a = np.abs(v)
    _, ex = np.frexp(np.maximum(a, 2.0 ** -6))  # a = m * 2^ex, m in [0.5, 1)
    spacing = np.ldexp(1.0, ex - 1 - 3)
    q = np.minimum(np.round(a / spacing) * spacing, E4M3_MAX)  # np.round: half to even
    return np.copysign(q, v)


def e4m3_code(q) -> np.ndarray:
    """The byte of E4M3 values (as round_e4m3 returns them)."""
    q = _f64(q)
    a = np.abs(q)
    sign = (np.signbit(q)).astype(np.uint8) << 7
    sub = a < 2.0 ** -6
    _, ex = np.frexp(np.where(sub, 1.0, a))
    e = ex - 1
    expf = np.where(sub, 0, e + 7)
    mant = np.where(sub, np.round(a / 2.0 ** -9), np.round((a / np.ldexp(1.0, e) - 1.0) * 8))
    return (sign | (expf.astype(np.uint8) << 3) | mant.astype(np.uint8)).astype(np.uint8)


def quantize_rows_e4m3(y):
    """Codes and per-row scales of y (values exact in float32): amax = max|y|,
    scale = amax/448 (1 for a zero row), codes of y·(448/amax), the reciprocal
    and the product each rounded once in float32.  Returns (q values, scale)."""
    y32 = _round_f32(y)
    amax = np.max(np.abs(y32), axis=-1)
    nz = amax > 0
    safe = np.where(nz, amax, np.float32(1))
    inv = np.where(nz, np.float32(E4M3_MAX) / safe, np.float32(1)).astype(np.float32)
    scale = np.where(nz, safe / np.float32(E4M3_MAX), np.float32(1)).astype(np.float32)
    v = (y32 * inv[:, None]).astype(np.float32)
    return round_e4m3(v.astype(np.float64)), scale.astype(np.float64)


def rms_forward_quant(x, gamma, eps: float, gemma: int = 0, dtype: str = "bf16",
                      weight_dtype: str = ""):
    """(q values, scale, r): y as the forward stores it (the cast-order
    emulation, in ``dtype``), then quantize_rows_e4m3."""
    y = emulate_forward_lowp(x, gamma, eps, gemma, dtype, weight_dtype)
    q, scale = quantize_rows_e4m3(y)
    return q, scale, rms_rstd(x, eps)
