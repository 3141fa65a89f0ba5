"""Seeded synthetic inputs for RMSNorm and LayerNorm row workloads.

Every tensor is drawn in float64 from numpy's SFC64 bit generator, seeded by
``SeedSequence([seed, tensor_id])`` so that x, gamma, dy and the row scales
are independent streams.  Values are drawn row-chunk by row-chunk (a fixed
chunk size per workload), transformed by the distribution's affine map and
the optional per-row scale, then rounded to the I/O dtype:

* ``f32``  : float64 -> float32, round to nearest even (numpy ``astype``);
* ``f16``  : float64 -> float16, round to nearest even (numpy ``astype``);
* ``bf16`` : float64 -> float32 (RNE) -> bfloat16 (RNE on the 16 dropped
  mantissa bits).  bf16 tensors are returned as their ``uint16`` bit
  patterns, which is how both the CUDA side (viewed as ``torch.bfloat16``)
  and the oracle side (decoded exactly with ``storage_to_float64``) read
  them.

The rounded tensor is the one input both sides see.  Nothing here computes
any part of the normalisation.

Distributions are written ``("normal", mean, std)``, ``("uniform", lo, hi)``
and, for the per-row scale, ``("loguniform", a, b)``: ``s_i = exp(U(ln a,
ln b))`` multiplied into row i of x.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import numpy as np

_TENSOR_IDS = {"x": 1, "gamma": 2, "dy": 3, "row_scale": 4, "beta": 5, "residual": 6, "dh": 7}
_CHUNK_ELEMS = 1 << 22

Dist = Tuple[str, float, float]


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: the operation ("rms", "ln", "rms_add": the
    residual add fused into RMSNorm, or "rms_quant": the forward with an FP8
    E4M3 output), shapes, dtype, eps, flags and input laws.  For LayerNorm ``gamma`` is the weight w and ``beta`` the bias law
    (None: no bias); for "rms_add" ``residual`` is the law of the residual
    stream added to x, and the gradient dh reaching h through the residual
    path follows the dy law."""

    name: str
    M: int
    N: int
    dtype: str  # "f32", "bf16" or "f16"
    eps: float
    x: Dist = ("normal", 0.0, 1.0)
    gamma: Dist = ("uniform", 0.5, 1.5)
    dy: Dist = ("normal", 0.0, 1.0)
    row_scale: Optional[Dist] = None
    gemma: int = 0
    inplace_dx: int = 0
    seed: int = 0
    weight_dtype: str = ""  # "" (the activations' dtype) or "f32"
    op: str = "rms"  # "rms", "ln", "rms_add" or "rms_quant"
    beta: Optional[Dist] = None  # LayerNorm bias law
    residual: Optional[Dist] = None  # fused residual add: law of the residual stream
    note: str = field(default="", compare=False)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def wdtype(self) -> str:
        """The weight's dtype."""
        return self.weight_dtype or self.dtype

    def with_shape(self, M: int, N: Optional[int] = None, name: Optional[str] = None) -> "Workload":
        return replace(self, M=M, N=self.N if N is None else N,
                       name=name or f"{self.name}@{M}x{self.N if N is None else N}")


def _sweep(N: int) -> Workload:
    M = (1 << 27) // N  # x is 256 MiB of bf16, rounded down when N does not divide 2^27
    return Workload(name=f"sweep_bf16_N{N}", M=M, N=N, dtype="bf16", eps=1e-6,
                    note="row-width sweep, x ~ 256 MiB")


# The five workload families of the row-wise RMSNorm benchmark, plus the
# extra parity shapes the pages single out (N=257 vs 256, M=1 vs 17, the
# 128x257 fp32 timing shape, the 1151x8192 LayerNorm test shape).
WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_f32_64x128", 64, 128, "f32", 1e-6,
                 note="tiny fp32 fwd+bwd"),
        Workload("llama7b_bf16_8192x4096", 8192, 4096, "bf16", 1e-6,
                 gamma=("normal", 1.0, 0.1), dy=("normal", 0.0, 1e-2),
                 row_scale=("loguniform", 0.1, 10.0),
                 note="Llama-7B-shaped: 4x2048 tokens, hidden 4096"),
        Workload("wide_bf16_16384x8192", 16384, 8192, "bf16", 1e-5,
                 gamma=("normal", 1.0, 0.2), dy=("normal", 0.0, 1.0),
                 row_scale=("loguniform", 0.01, 100.0),
                 note="large hidden size; the headline workload"),
        Workload("gemma_bf16_32768x3072", 32768, 3072, "bf16", 1e-6,
                 gamma=("normal", 0.0, 0.1), gemma=1, inplace_dx=1,
                 note="Gemma (1+gamma) weight, dx written into dy"),
        *[_sweep(n) for n in (512, 1000, 2048, 5120, 11008, 16384)],
        *[Workload(f"widerows_bf16_N{n}", (1 << 27) // n, n, "bf16", 1e-6,
                   note="rows wider than one CTA's shared memory (cluster split)")
          for n in (32768, 65536, 131072)],
        *[Workload(f"widerows_bf16_N{n}", (1 << 27) // n, n, "bf16", 1e-6,
                   note="rows wider than a cluster holds (chunked mapping)")
          for n in (262144, 1048576)],
        Workload("wide_f16_16384x8192", 16384, 8192, "f16", 1e-5,
                 gamma=("normal", 1.0, 0.2), dy=("normal", 0.0, 1.0),
                 row_scale=("loguniform", 0.01, 100.0),
                 note="the large-hidden workload with fp16 I/O"),
        Workload("llama7b_bf16w32_8192x4096", 8192, 4096, "bf16", 1e-6,
                 gamma=("normal", 1.0, 0.1), dy=("normal", 0.0, 1e-2),
                 row_scale=("loguniform", 0.1, 10.0), weight_dtype="f32",
                 note="the Llama-7B shape with a float32 weight (mixed precision)"),
        Workload("timing_f32_128x257", 128, 257, "f32", 1e-6,
                 note="the tutorial's timing shape, ragged N"),
        Workload("rms_bf16_1151x8192", 1151, 8192, "bf16", 1e-5,
                 note="RMSNorm at the LayerNorm chapter's unit-test shape"),
        # LayerNorm: the chapter's unit test (1151 x 8192 fp16, x = -2.3 + 0.5 N(0,1),
        # w, b ~ U(0,1), dy = 0.1 N(0,1), eps 1e-5) and its backward benchmark
        # (M = 4096 fp16, N = 512 k for k = 2..31), plus the large-hidden shape.
        Workload("ln_test_f16_1151x8192", 1151, 8192, "f16", 1e-5, op="ln",
                 x=("normal", -2.3, 0.5), gamma=("uniform", 0.0, 1.0), beta=("uniform", 0.0, 1.0),
                 dy=("normal", 0.0, 0.1), note="the LayerNorm chapter's unit test"),
        *[Workload(f"ln_bench_f16_4096x{n}", 4096, n, "f16", 1e-5, op="ln",
                   x=("normal", -2.3, 0.5), gamma=("uniform", 0.0, 1.0),
                   beta=("uniform", 0.0, 1.0), dy=("normal", 0.0, 0.1),
                   note="the LayerNorm chapter's backward benchmark")
          for n in (1024, 4096, 8192, 15872)],
        # The residual add fused into RMSNorm at the Llama-7B and large-hidden
        # shapes (the residual stream as large as x).
        Workload("resadd_llama7b_bf16_8192x4096", 8192, 4096, "bf16", 1e-6, op="rms_add",
                 gamma=("normal", 1.0, 0.1), dy=("normal", 0.0, 1e-2),
                 row_scale=("loguniform", 0.1, 10.0), residual=("normal", 0.0, 1.0),
                 note="residual add + RMSNorm, Llama-7B shape"),
        Workload("resadd_wide_bf16_16384x8192", 16384, 8192, "bf16", 1e-5, op="rms_add",
                 gamma=("normal", 1.0, 0.2), dy=("normal", 0.0, 1.0),
                 row_scale=("loguniform", 0.01, 100.0), residual=("normal", 0.0, 1.0),
                 note="residual add + RMSNorm, large-hidden shape"),
        # The forward with its output quantised to FP8 E4M3 (one byte per
        # element and a scale per row) at the same two shapes.
        Workload("quant_llama7b_bf16_8192x4096", 8192, 4096, "bf16", 1e-6, op="rms_quant",
                 gamma=("normal", 1.0, 0.1), row_scale=("loguniform", 0.1, 10.0),
                 note="RMSNorm + E4M3 output, Llama-7B shape"),
        Workload("quant_wide_bf16_16384x8192", 16384, 8192, "bf16", 1e-5, op="rms_quant",
                 gamma=("normal", 1.0, 0.2), row_scale=("loguniform", 0.01, 100.0),
                 note="RMSNorm + E4M3 output, large-hidden shape"),
        Workload("quant_widerows_bf16_N65536", 2048, 65536, "bf16", 1e-6, op="rms_quant",
                 note="RMSNorm + E4M3 output, rows of 128 KiB (x 256 MiB)"),
        Workload("ln_wide_bf16_16384x8192", 16384, 8192, "bf16", 1e-5, op="ln",
                 x=("normal", -2.3, 0.5), gamma=("uniform", 0.0, 1.0), beta=("uniform", 0.0, 1.0),
                 dy=("normal", 0.0, 0.1), note="LayerNorm at the large-hidden shape"),
    ]
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def _generator(seed: int, tensor: str) -> np.random.Generator:
    return np.random.Generator(np.random.SFC64(np.random.SeedSequence([seed, _TENSOR_IDS[tensor]])))


def _draw(gen: np.random.Generator, dist: Dist, out: np.ndarray) -> None:
    kind, a, b = dist
    if kind == "normal":
        gen.standard_normal(out=out)
        if b != 1.0:
            out *= b
        if a != 0.0:
            out += a
    elif kind == "uniform":
        out[...] = gen.uniform(a, b, size=out.shape)
    elif kind == "loguniform":
        out[...] = np.exp(gen.uniform(math.log(a), math.log(b), size=out.shape))
    else:
        raise ValueError(f"unknown distribution {kind!r}")


def float_to_bf16_bits(a) -> np.ndarray:
    """Round float values to bfloat16 bit patterns: float32 RNE, then RNE on 16 bits."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32)
    lsb = (u >> 16) & np.uint32(1)
    return ((u + lsb + np.uint32(0x7FFF)) >> 16).astype(np.uint16)


def bf16_bits_to_float32(bits) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def storage_to_float64(arr, dtype: str) -> np.ndarray:
    """Exact float64 values of a stored tensor (float32 array or bf16 bits)."""
    if dtype == "bf16":
        return bf16_bits_to_float32(arr).astype(np.float64)
    if dtype == "f16":
        return np.asarray(arr, dtype=np.float16).astype(np.float64)
    return np.asarray(arr, dtype=np.float32).astype(np.float64)


def _store(vals64: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return float_to_bf16_bits(vals64)
    if dtype == "f16":
        return vals64.astype(np.float16)
    return vals64.astype(np.float32)


def _matrix(w: Workload, tensor: str, dist: Dist, row_scale: Optional[np.ndarray]) -> np.ndarray:
    gen = _generator(w.seed, tensor)
    out = np.empty((w.M, w.N), dtype={"bf16": np.uint16, "f16": np.float16}.get(w.dtype, np.float32))
    rows = max(1, _CHUNK_ELEMS // max(1, w.N))
    buf = np.empty((min(rows, max(w.M, 1)), w.N), dtype=np.float64)
    for r0 in range(0, w.M, rows):
        r1 = min(w.M, r0 + rows)
        blk = buf[: r1 - r0]
        _draw(gen, dist, blk)
        if row_scale is not None:
            blk *= row_scale[r0:r1, None]
        out[r0:r1] = _store(blk, w.dtype)
    return out


def make_inputs(w: Workload) -> dict:
    """Draw x (M,N), gamma (N,) and dy (M,N) for a workload, in storage form
    (gamma in the weight dtype).

    Returns a dict with keys ``x``, ``gamma``, ``dy`` (float32 arrays for f32
    workloads, float16 arrays for f16 ones, uint16 bf16 bit patterns for bf16
    ones), ``beta`` (the LayerNorm bias in the weight dtype, or None),
    ``row_scale`` (float64, or None) and, for workloads with a residual law,
    ``residual`` and ``dh`` (activation dtype).
    """
    scale = None
    if w.row_scale is not None:
        scale = np.empty(w.M, dtype=np.float64)
        _draw(_generator(w.seed, "row_scale"), w.row_scale, scale)
    gvals = np.empty(w.N, dtype=np.float64)
    _draw(_generator(w.seed, "gamma"), w.gamma, gvals)
    beta = None
    if w.beta is not None:
        bvals = np.empty(w.N, dtype=np.float64)
        _draw(_generator(w.seed, "beta"), w.beta, bvals)
        beta = _store(bvals, w.wdtype)
    fused = {}
    if w.residual is not None:
        fused["residual"] = _matrix(w, "residual", w.residual, None)
        fused["dh"] = _matrix(w, "dh", w.dy, None)
    return {
        **fused,
        "x": _matrix(w, "x", w.x, scale),
        "gamma": _store(gvals, w.wdtype),
        "beta": beta,
        "dy": _matrix(w, "dy", w.dy, None),
        "row_scale": scale,
    }
