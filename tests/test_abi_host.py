"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects invalid arguments on the host before any CUDA call.

The pointers passed here are never dereferenced: every case fails
validation, which runs before the library touches CUDA.
"""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "rmsnorm.h"

(OK, INVALID, UNSUPPORTED, ALIGNMENT, WORKSPACE, CUDA, TIMEOUT) = range(7)
A = 1 << 24  # fake, 256-byte aligned addresses A, 2A, ... that are never dereferenced
FAKE = A


@pytest.fixture(scope="module")
def lib():
    from row_wise_normalization_rms_gb300 import build

    build.build()
    from row_wise_normalization_rms_gb300 import _lib

    return _lib.load()


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:rms|ln)_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 8, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in rmsnorm.h but not exported"
    from row_wise_normalization_rms_gb300 import _lib

    assert sorted(_lib.SIGNATURES) == names


def test_status_strings(lib):
    for s in range(7):
        assert lib.rms_status_string(s)
    assert b"unknown" in lib.rms_status_string(99)


def fwd(lib, x=A, g=2 * A, y=3 * A, r=4 * A, M=4, N=8, eps=1e-6,
        dtype=1, gemma=0, path=0):
    return lib.rms_fwd_ex(x, g, y, r, M, N, eps, dtype, gemma, path, None)


def test_fwd_rejects_bad_arguments(lib):
    nan, inf = float("nan"), float("inf")
    assert fwd(lib, dtype=5) == INVALID
    assert fwd(lib, dtype=-1) == INVALID
    assert fwd(lib, gemma=2) == INVALID
    assert fwd(lib, M=-1) == INVALID
    assert fwd(lib, N=0) == INVALID
    assert fwd(lib, N=-5) == INVALID
    assert fwd(lib, eps=nan) == INVALID
    assert fwd(lib, eps=inf) == INVALID
    assert fwd(lib, eps=-1e-6) == INVALID
    assert fwd(lib, path=7) == INVALID
    assert fwd(lib, path=5) == INVALID
    assert fwd(lib, x=None) == INVALID
    assert fwd(lib, g=None) == INVALID
    assert fwd(lib, y=None) == INVALID
    assert fwd(lib, r=None) == INVALID
    assert fwd(lib, N=1 << 40) == UNSUPPORTED
    assert fwd(lib, M=1 << 62, N=1 << 20) == INVALID  # size overflows int64


def test_fwd_rejects_overlap(lib):
    assert fwd(lib, y=A + 16) == INVALID          # y inside x
    assert fwd(lib, y=2 * A - 16) == INVALID      # y's tail runs into gamma
    assert fwd(lib, r=A + 8) == INVALID           # rstd inside x
    assert fwd(lib, r=3 * A + 60) == INVALID      # rstd inside y


def test_fwd_empty_batch_is_a_noop(lib):
    assert fwd(lib, M=0, x=None, g=None, y=None, r=None) == OK


def bwd(lib, dy=A, x=2 * A, g=3 * A, r=4 * A, dx=5 * A, dg=6 * A, ws=7 * A, wsb=1 << 30, M=4,
        N=8, dtype=1, gemma=0, inplace=0,
        path=0):
    return lib.rms_bwd_ex(dy, x, g, r, dx, dg, ws, wsb, M, N, dtype, gemma, inplace, path, None)


def test_bwd_rejects_bad_arguments(lib):
    assert bwd(lib, dtype=5) == INVALID
    assert bwd(lib, gemma=-1) == INVALID
    assert bwd(lib, inplace=2) == INVALID
    assert bwd(lib, M=-3) == INVALID
    assert bwd(lib, N=0) == INVALID
    assert bwd(lib, path=-1) == INVALID
    assert bwd(lib, path=5) == INVALID
    assert bwd(lib, dg=None) == INVALID
    assert bwd(lib, dx=None) == INVALID
    assert bwd(lib, x=None) == INVALID
    assert bwd(lib, dy=None) == INVALID
    assert bwd(lib, g=None) == INVALID
    assert bwd(lib, r=None) == INVALID
    # in place: dx must be NULL or dy itself
    assert bwd(lib, inplace=1, dx=9 * A) == INVALID
    # the workspace is required when there are rows
    assert bwd(lib, ws=None) == WORKSPACE


def test_set_wait_limit_roundtrip(lib):
    prev = lib.rms_set_wait_limit(123)
    assert lib.rms_set_wait_limit(-1) == 123
    assert lib.rms_set_wait_limit(prev) > 0


def test_python_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from row_wise_normalization_rms_gb300 import _lib

    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        _lib.load()


def ln_f(lib, x=A, w=2 * A, b=3 * A, y=4 * A, mu=5 * A, r=6 * A, M=4, N=8, eps=1e-5, dtype=1,
         path=0):
    return lib.ln_fwd_ex(x, w, b, y, mu, r, M, N, eps, dtype, path, None)


def test_ln_fwd_rejects_bad_arguments(lib):
    assert ln_f(lib, dtype=5) == INVALID
    assert ln_f(lib, M=-1) == INVALID
    assert ln_f(lib, N=0) == INVALID
    assert ln_f(lib, eps=float("nan")) == INVALID
    assert ln_f(lib, eps=-1.0) == INVALID
    assert ln_f(lib, path=9) == INVALID
    assert ln_f(lib, path=2) == UNSUPPORTED  # no staged forward mapping
    assert ln_f(lib, path=4) == UNSUPPORTED  # no chunked LayerNorm mapping
    for k in ("x", "w", "y", "mu", "r"):
        assert ln_f(lib, **{k: None}) == INVALID, k
    assert ln_f(lib, N=1 << 40) == UNSUPPORTED


def test_ln_fwd_rejects_overlap(lib):
    assert ln_f(lib, y=A + 16) == INVALID        # y inside x
    assert ln_f(lib, y=3 * A - 16) == INVALID    # y's tail runs into b
    assert ln_f(lib, mu=4 * A + 4) == INVALID    # mean inside y
    assert ln_f(lib, r=5 * A + 8) == INVALID     # rstd overlaps mean
    assert ln_f(lib, mu=2 * A) == INVALID        # mean on w


def test_ln_fwd_empty_batch_is_a_noop(lib):
    assert ln_f(lib, M=0, x=None, w=None, b=None, y=None, mu=None, r=None) == OK


def ln_b(lib, dy=A, x=2 * A, w=3 * A, mu=4 * A, r=5 * A, dx=6 * A, dw=7 * A, db=8 * A, ws=9 * A,
         wsb=1 << 30, M=4, N=8, dtype=1, inplace=0, path=0):
    return lib.ln_bwd_ex(dy, x, w, mu, r, dx, dw, db, ws, wsb, M, N, dtype, inplace, path, None)


def test_ln_bwd_rejects_bad_arguments(lib):
    assert ln_b(lib, dtype=7) == INVALID
    assert ln_b(lib, inplace=3) == INVALID
    assert ln_b(lib, M=-2) == INVALID
    assert ln_b(lib, N=0) == INVALID
    assert ln_b(lib, path=5) == INVALID
    assert ln_b(lib, path=1) == UNSUPPORTED  # no register backward mapping
    assert ln_b(lib, path=4) == UNSUPPORTED  # no chunked LayerNorm mapping
    assert ln_b(lib, dw=None) == INVALID
    for k in ("dy", "x", "w", "mu", "r", "dx"):
        assert ln_b(lib, **{k: None}) == INVALID, k
    assert ln_b(lib, inplace=1, dx=10 * A) == INVALID
    assert ln_b(lib, ws=None) == WORKSPACE


def test_fused_add_rejects_bad_arguments(lib):
    # rms_fwd_add_ex(x, residual, gamma, y, h, rstd, M, N, eps, dtype, gemma, path, stream)
    f = lambda **k: lib.rms_fwd_add_ex(k.get("x", A), k.get("res", 2 * A), k.get("g", 3 * A),
                                       k.get("y", 4 * A), k.get("h", 5 * A), k.get("r", 6 * A),
                                       k.get("M", 4), k.get("N", 8), 1e-6, 1, 0,
                                       k.get("path", 0), None)
    assert f(res=None) == INVALID
    assert f(h=None) == INVALID
    assert f(h=A) == INVALID           # h over x
    assert f(h=4 * A) == INVALID       # h over y
    assert f(path=5) == INVALID
    assert f(M=0, x=None, res=None, g=None, y=None, h=None, r=None) == OK
    # rms_bwd_add_ex(dy, h, gamma, rstd, dh, dx, dgamma, ws, wsb, M, N, dtype, gemma, inplace, path, s)
    b = lambda **k: lib.rms_bwd_add_ex(A, 2 * A, 3 * A, 4 * A, k.get("dh", 5 * A),
                                       k.get("dx", 6 * A), 7 * A, 8 * A, 1 << 30, 4, 8, 1, 0,
                                       k.get("inplace", 0), 0, None)
    assert b(dh=None) == INVALID
    assert b(inplace=1, dx=5 * A) == INVALID  # in place means dx is dy


def test_quant_rejects_bad_arguments(lib):
    f = lambda **k: lib.rms_fwd_quant_ex(k.get("x", A), k.get("g", 2 * A), k.get("q", 3 * A),
                                         k.get("s", 4 * A), k.get("r", 5 * A), k.get("M", 4),
                                         k.get("N", 8), 1e-6, k.get("dtype", 1), 0,
                                         k.get("path", 0), None)
    assert f(dtype=5) == INVALID
    assert f(q=None) == INVALID
    assert f(s=None) == INVALID
    assert f(path=2) == UNSUPPORTED
    assert f(path=4, q=A + 4) == INVALID  # the any-width mapping: still checked on the host
    assert f(path=5) == INVALID
    assert f(q=A + 4) == INVALID          # codes over x
    assert f(s=3 * A + 8) == INVALID      # scale over the codes
    assert f(M=0, x=None, g=None, q=None, s=None, r=None) == OK


def test_reduction_queries_reject_bad_arguments(lib):
    p, n = ctypes.c_int64(7), ctypes.c_int64(7)
    P, R = ctypes.byref(p), ctypes.byref(n)
    q = lambda M=4, N=8, dtype=1, gemma=0, res=0, path=0, a=P, b=R: lib.rms_bwd_reduction(
        M, N, dtype, gemma, res, path, a, b)
    assert q(dtype=5) == INVALID
    assert q(gemma=2) == INVALID
    assert q(res=2) == INVALID
    assert q(M=-1) == INVALID
    assert q(N=0) == INVALID
    assert q(path=5) == INVALID
    assert q(a=None) == INVALID
    assert q(b=None) == INVALID
    assert q(N=1 << 40) == UNSUPPORTED
    assert q(M=0) == OK and p.value == 0 and n.value == 0  # no rows: nothing to sum
    lq = lambda M=4, N=8, dtype=1, path=0, a=P, b=R: lib.ln_bwd_reduction(M, N, dtype, path, a, b)
    assert lq(dtype=9) == INVALID
    assert lq(N=-3) == INVALID
    assert lq(path=1) == UNSUPPORTED  # no register backward mapping
    assert lq(path=4) == UNSUPPORTED
    assert lq(a=None) == INVALID
    p.value = n.value = 7
    assert lq(M=0) == OK and p.value == 0 and n.value == 0


def test_noalloc_answers_bad_shapes_before_its_scratch(lib):
    # rms_bwd_noalloc(dy, x, gamma, rstd, dx, dgamma, M, N, dtype, gemma, inplace, stream):
    # a bad shape or flag is rms_bwd's error, found before any device lookup
    f = lambda M=4, N=8, dtype=1, gemma=0, inplace=0, dg=6 * A: lib.rms_bwd_noalloc(
        A, 2 * A, 3 * A, 4 * A, 5 * A, dg, M, N, dtype, gemma, inplace, None)
    assert f(M=-1) == INVALID
    assert f(N=0) == INVALID
    assert f(M=0, dtype=7) == INVALID
    assert f(M=0, gemma=3) == INVALID
    assert f(M=0, dg=None) == INVALID


def test_dgamma_cast_rejects_bad_arguments(lib):
    # rms_dgamma_cast(dgamma, out, N, dtype, stream)
    f = lambda src=A, dst=2 * A, N=8, dtype=1: lib.rms_dgamma_cast(src, dst, N, dtype, None)
    assert f(src=None) == INVALID
    assert f(dst=None) == INVALID
    assert f(N=0) == INVALID
    assert f(N=-3) == INVALID
    assert f(dtype=-1) == INVALID
    assert f(dtype=5) == INVALID
    # bf16 output of 8 elements (16 bytes) inside the 32-byte float32 source
    assert f(dst=A + 16) == INVALID
    # a float32 output overlapping the source's tail
    assert f(dst=A + 28, dtype=0) == INVALID
