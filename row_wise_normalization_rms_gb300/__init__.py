"""Python binding of librmsnorm.so, the GB300 fused RMSNorm library.

Argument marshalling only: every function below derives sizes, dtype codes,
device pointers and the current CUDA stream from torch tensors and calls the
C entry point of the same name (declared in include/rmsnorm.h).  All
computation happens in the library's CUDA kernels; when the library is
missing, calls raise instead of falling back to anything else.

Forward:  r = 1/sqrt(mean(x^2) + eps),  y = x * r * g  (g = gamma or 1+gamma)
Backward: u = dy*g,  dx = r*u - x*r^3*mean(u*x),  dgamma = sum_rows dy*x*r

LayerNorm on the same engine (ln_fwd / ln_bwd):
  xhat = (x - mean)*rstd,  y = xhat*w + b
  g = dy*w,  dx = (g - (xhat*mean(xhat*g) + mean(g)))*rstd,
  dw = sum_rows dy*xhat,  db = sum_rows dy
"""
from __future__ import annotations

from . import _lib

RMS_F32, RMS_BF16, RMS_F16, RMS_BF16_W32, RMS_F16_W32 = 0, 1, 2, 3, 4
RMS_PATH_AUTO, RMS_PATH_REGISTERS, RMS_PATH_STAGED, RMS_PATH_SCALAR, RMS_PATH_CHUNKED = 0, 1, 2, 3, 4
(RMS_OK, RMS_ERR_INVALID_ARG, RMS_ERR_UNSUPPORTED, RMS_ERR_ALIGNMENT, RMS_ERR_WORKSPACE,
 RMS_ERR_CUDA, RMS_ERR_TIMEOUT) = range(7)
PATHS = {"auto": RMS_PATH_AUTO, "registers": RMS_PATH_REGISTERS, "staged": RMS_PATH_STAGED,
         "scalar": RMS_PATH_SCALAR, "chunked": RMS_PATH_CHUNKED}

__all__ = [
    "RmsError", "lib", "rms_fwd", "rms_bwd", "rms_bwd_noalloc", "rms_bwd_workspace_size",
    "rms_bwd_reduction", "ln_bwd_reduction", "rms_dgamma_combine", "rms_dgamma_cast",
    "rms_status_string",
    "rms_last_device_status", "rms_set_wait_limit", "rms_launch_count", "dtype_code",
]


class RmsError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {rms_status_string(status)} (status {status})")


_LIB = None  # the loaded library, kept once found (calls skip the loader's lock)


def lib():
    """The raw ctypes library (see _lib.SIGNATURES for the argument types)."""
    global _LIB
    if _LIB is None:
        _LIB = _lib.load()
    return _LIB


def rms_status_string(status: int) -> str:
    return lib().rms_status_string(int(status)).decode()


_DTYPES = None  # (activation dtype, weight dtype) -> rms_dtype code, built on first use


def _dtype_table():
    global _DTYPES
    if _DTYPES is None:
        import torch

        f32, bf16, f16 = torch.float32, torch.bfloat16, torch.float16
        _DTYPES = {(f32, f32): RMS_F32, (bf16, bf16): RMS_BF16, (f16, f16): RMS_F16,
                   (bf16, f32): RMS_BF16_W32, (f16, f32): RMS_F16_W32}
    return _DTYPES


def dtype_code(t, gamma=None) -> int:
    """The rms_dtype code of activations ``t`` and weight ``gamma`` (default: same type)."""
    code = _dtype_table().get((t.dtype, t.dtype if gamma is None else gamma.dtype))
    if code is not None:
        return code
    if (t.dtype, t.dtype) not in _DTYPES:
        raise ValueError(f"unsupported dtype {t.dtype}: float32, bfloat16 or float16")
    raise ValueError(f"unsupported weight dtype {gamma.dtype} for {t.dtype} activations")


_RAW_STREAM = None  # () -> the current device's current cudaStream_t as an int


def _current_stream_getter():
    """torch's raw-stream query (one call, no Stream object), else the public
    torch.cuda.current_stream(); both name the current device's current stream."""
    import torch

    torch.cuda.init()
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    dev = getattr(torch._C, "_cuda_getDevice", None)
    if raw is not None and dev is not None:
        try:
            if raw(dev()) == torch.cuda.current_stream().cuda_stream:
                return lambda: raw(dev())
        except (RuntimeError, TypeError):
            pass
    return lambda: torch.cuda.current_stream().cuda_stream


def _stream_handle(stream):
    global _RAW_STREAM
    if stream is None:
        if _RAW_STREAM is None:
            _RAW_STREAM = _current_stream_getter()
        return _RAW_STREAM()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous row-major")
    return t.data_ptr()


# The C ABI takes plain device pointers and cannot see buffer sizes; the
# binding checks what it can from the tensors before handing their pointers
# over: every tensor lives on x's CUDA device and holds at least the bytes
# the call reads or writes there.  None is passed through (the library
# decides whether that argument may be NULL).

def _rows(x, name="x"):
    """M, N and the CUDA device index of the 2-D row-major tensor x."""
    if x.dim() != 2:
        raise ValueError(f"{name} must be 2-D (rows, N), got shape {tuple(x.shape)}")
    dev = x.get_device()
    if dev < 0:
        raise ValueError(f"{name} must be a CUDA tensor, got one on {x.device}")
    M, N = x.shape
    return M, N, dev


def _arg(t, nbytes, name, dev):
    """The device pointer of ``t`` after checking its device and byte size."""
    if t is None:
        return None
    if t.get_device() != dev:
        raise ValueError(f"{name} is on {t.device}; every tensor must be on cuda:{dev}, as x")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name} holds {have} bytes; the call needs {nbytes}")
    return _ptr(t)


def _weight(t, N, name, dev):
    """As _arg for a weight vector, which needs N elements of its own type."""
    if t is not None and t.numel() < N:
        raise ValueError(f"{name} has {t.numel()} elements; the call needs {N}")
    return _arg(t, 0, name, dev)


def _path(path) -> int:
    return PATHS[path] if isinstance(path, str) else int(path)


def rms_fwd(x, gamma, y, rstd, eps: float = 1e-6, gemma: int = 0, stream=None, path="auto"):
    """y and rstd from x (M,N) and gamma (N,); writes into y (M,N) and rstd (M,) float32."""
    M, N, dev = _rows(x)
    mn = M * N * x.element_size()
    st = lib().rms_fwd_ex(_ptr(x), _weight(gamma, N, "gamma", dev),
                          _arg(y, mn, "y", dev), _arg(rstd, 4 * M, "rstd", dev), M, N,
                          float(eps), dtype_code(x, gamma), int(gemma), _path(path),
                          _stream_handle(stream))
    if st != RMS_OK:
        raise RmsError(st, "rms_fwd")


def rms_bwd(dy, x, gamma, rstd, dx, dgamma, workspace, gemma: int = 0, inplace_dx: int = 0,
            stream=None, path="auto"):
    """dx (M,N) and dgamma (N,) float32; with inplace_dx=1 dx is written into dy (pass dx=None)."""
    M, N, dev = _rows(x)
    mn = M * N * x.element_size()
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().rms_bwd_ex(_arg(dy, mn, "dy", dev), _ptr(x),
                          _weight(gamma, N, "gamma", dev),
                          _arg(rstd, 4 * M, "rstd", dev), _arg(dx, mn, "dx", dev),
                          _arg(dgamma, 4 * N, "dgamma", dev), _arg(workspace, 0, "workspace", dev),
                          ws_bytes, M, N, dtype_code(x, gamma), int(gemma), int(inplace_dx),
                          _path(path), _stream_handle(stream))
    if st != RMS_OK:
        raise RmsError(st, "rms_bwd")


def rms_bwd_noalloc(dy, x, gamma, rstd, dx, dgamma, gemma: int = 0, inplace_dx: int = 0,
                    stream=None):
    """rms_bwd with the library's built-in scratch instead of a workspace
    argument, for callers that cannot allocate device scratch themselves
    (see include/rmsnorm.h for the size limit and the sharing rules)."""
    M, N, dev = _rows(x)
    mn = M * N * x.element_size()
    st = lib().rms_bwd_noalloc(_arg(dy, mn, "dy", dev), _ptr(x),
                               _weight(gamma, N, "gamma", dev),
                               _arg(rstd, 4 * M, "rstd", dev), _arg(dx, mn, "dx", dev),
                               _arg(dgamma, 4 * N, "dgamma", dev), M, N, dtype_code(x, gamma),
                               int(gemma), int(inplace_dx), _stream_handle(stream))
    if st != RMS_OK:
        raise RmsError(st, "rms_bwd_noalloc")


def rms_dgamma_combine(parts, dgamma, stream=None):
    """dgamma (N,) = the rows of parts (ranks, N) float32 added in increasing
    row order: the exchange step of a row-sharded backward."""
    if parts.dim() != 2:
        raise ValueError(f"parts must be 2-D (ranks, N), got shape {tuple(parts.shape)}")
    R, N = parts.shape
    dev = parts.get_device()
    if dev < 0:
        raise ValueError(f"parts must be a CUDA tensor, got one on {parts.device}")
    if parts.dtype != dgamma.dtype or parts.element_size() != 4:
        raise ValueError("parts and dgamma must be float32")
    st = lib().rms_dgamma_combine(_ptr(parts), R, N, _arg(dgamma, 4 * N, "dgamma", dev),
                                  _stream_handle(stream))
    if st != RMS_OK:
        raise RmsError(st, "rms_dgamma_combine")


def rms_dgamma_cast(dgamma, out, stream=None):
    """out (N,) = dgamma (N,) float32 rounded to out's type (bfloat16 or float16,
    ties to even; a float32 out is a copy): the weight gradient in the weight's
    own type."""
    if dgamma.dim() != 1 or out.dim() != 1:
        raise ValueError("dgamma and out must be 1-D")
    if dgamma.dtype != _torch().float32:
        raise ValueError("dgamma must be float32")
    N = dgamma.numel()
    dev = dgamma.get_device()
    if dev < 0:
        raise ValueError(f"dgamma must be a CUDA tensor, got one on {dgamma.device}")
    code = {_torch().float32: RMS_F32, _torch().bfloat16: RMS_BF16,
            _torch().float16: RMS_F16}.get(out.dtype)
    if code is None:
        raise ValueError(f"unsupported weight dtype {out.dtype}")
    st = lib().rms_dgamma_cast(_ptr(dgamma), _arg(out, N * out.element_size(), "out", dev), N,
                               code, _stream_handle(stream))
    if st != RMS_OK:
        raise RmsError(st, "rms_dgamma_cast")


def _torch():
    import torch

    return torch


def rms_fwd_add(x, residual, gamma, y, h, rstd, eps: float = 1e-6, gemma: int = 0, stream=None,
                path="auto"):
    """Fused residual add + RMSNorm: h = x + residual (rounded to x's dtype;
    h may be residual itself) and y, rstd = RMSNorm(h)."""
    M, N, dev = _rows(x)
    mn = M * N * x.element_size()
    st = lib().rms_fwd_add_ex(_ptr(x), _arg(residual, mn, "residual", dev),
                              _weight(gamma, N, "gamma", dev),
                              _arg(y, mn, "y", dev), _arg(h, mn, "h", dev),
                              _arg(rstd, 4 * M, "rstd", dev), M, N, float(eps),
                              dtype_code(x, gamma), int(gemma), _path(path),
                              _stream_handle(stream))
    if st != RMS_OK:
        raise RmsError(st, "rms_fwd_add")


def rms_bwd_add(dy, h, gamma, rstd, dh, dx, dgamma, workspace, gemma: int = 0, inplace_dx: int = 0,
                stream=None, path="auto"):
    """Backward of rms_fwd_add: dx = dRMS + dh (dx may be dh itself, or dy
    with inplace_dx=1 and dx=None); dgamma as rms_bwd."""
    M, N, dev = _rows(h, "h")
    mn = M * N * h.element_size()
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().rms_bwd_add_ex(_arg(dy, mn, "dy", dev), _ptr(h),
                              _weight(gamma, N, "gamma", dev),
                              _arg(rstd, 4 * M, "rstd", dev), _arg(dh, mn, "dh", dev),
                              _arg(dx, mn, "dx", dev), _arg(dgamma, 4 * N, "dgamma", dev),
                              _arg(workspace, 0, "workspace", dev), ws_bytes, M, N,
                              dtype_code(h, gamma), int(gemma), int(inplace_dx), _path(path),
                              _stream_handle(stream))
    if st != RMS_OK:
        raise RmsError(st, "rms_bwd_add")


def rms_fwd_quant(x, gamma, q, scale, rstd, eps: float = 1e-6, gemma: int = 0, stream=None,
                  path="auto"):
    """RMSNorm forward quantised to FP8 E4M3: q (M,N) uint8 codes (or a
    torch.float8_e4m3fn tensor), scale and rstd (M,) float32."""
    M, N, dev = _rows(x)
    st = lib().rms_fwd_quant_ex(_ptr(x), _weight(gamma, N, "gamma", dev),
                                _arg(q, M * N, "q", dev), _arg(scale, 4 * M, "scale", dev),
                                _arg(rstd, 4 * M, "rstd", dev), M, N, float(eps),
                                dtype_code(x, gamma), int(gemma), _path(path),
                                _stream_handle(stream))
    if st != RMS_OK:
        raise RmsError(st, "rms_fwd_quant")


def ln_fwd(x, w, b, y, mean, rstd, eps: float = 1e-5, stream=None, path="auto"):
    """LayerNorm forward: y (M,N), mean and rstd (M,) float32 from x (M,N),
    w (N,) and b (N,) or None (no bias)."""
    M, N, dev = _rows(x)
    if b is not None and b.dtype != w.dtype:
        raise ValueError("w and b must share one dtype")
    st = lib().ln_fwd_ex(_ptr(x), _weight(w, N, "w", dev), _weight(b, N, "b", dev),
                         _arg(y, M * N * x.element_size(), "y", dev),
                         _arg(mean, 4 * M, "mean", dev), _arg(rstd, 4 * M, "rstd", dev), M, N,
                         float(eps), dtype_code(x, w), _path(path), _stream_handle(stream))
    if st != RMS_OK:
        raise RmsError(st, "ln_fwd")


def ln_bwd(dy, x, w, mean, rstd, dx, dw, db, workspace, inplace_dx: int = 0, stream=None,
           path="auto"):
    """LayerNorm backward: dx (M,N); dw and db (N,) float32 (db may be None);
    with inplace_dx=1 dx is written into dy (pass dx=None)."""
    M, N, dev = _rows(x)
    mn = M * N * x.element_size()
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().ln_bwd_ex(_arg(dy, mn, "dy", dev), _ptr(x), _weight(w, N, "w", dev),
                         _arg(mean, 4 * M, "mean", dev), _arg(rstd, 4 * M, "rstd", dev),
                         _arg(dx, mn, "dx", dev), _arg(dw, 4 * N, "dw", dev),
                         _arg(db, 4 * N, "db", dev), _arg(workspace, 0, "workspace", dev),
                         ws_bytes, M, N, dtype_code(x, w), int(inplace_dx), _path(path),
                         _stream_handle(stream))
    if st != RMS_OK:
        raise RmsError(st, "ln_bwd")


def ln_bwd_workspace_size(M: int, N: int) -> int:
    return int(lib().ln_bwd_workspace_size(int(M), int(N)))


def rms_bwd_workspace_size(M: int, N: int) -> int:
    return int(lib().rms_bwd_workspace_size(int(M), int(N)))


def _reduction(fn, where, *args):
    import ctypes

    p = ctypes.c_int64(0)
    n = ctypes.c_int64(0)
    st = fn(*args, ctypes.byref(p), ctypes.byref(n))
    if st != RMS_OK:
        raise RmsError(st, where)
    return int(p.value), int(n.value)


def rms_bwd_reduction(M: int, N: int, dtype: int, gemma: int = 0, residual: int = 0,
                      path="auto"):
    """(P, rows_per_partial): the partial rows the backward's dgamma sum adds
    and the most rows one partial row sums (``dtype`` an rms_dtype code)."""
    return _reduction(lib().rms_bwd_reduction, "rms_bwd_reduction", int(M), int(N), int(dtype),
                      int(gemma), int(residual), _path(path))


def ln_bwd_reduction(M: int, N: int, dtype: int, path="auto"):
    """(P, rows_per_partial) of ln_bwd's dw and db sums."""
    return _reduction(lib().ln_bwd_reduction, "ln_bwd_reduction", int(M), int(N), int(dtype),
                      _path(path))


def rms_last_device_status(stream=None) -> int:
    return int(lib().rms_last_device_status(_stream_handle(stream)))


def rms_set_wait_limit(polls: int) -> int:
    return int(lib().rms_set_wait_limit(int(polls)))


def rms_launch_count() -> int:
    return int(lib().rms_launch_count())
