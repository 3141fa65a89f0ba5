"""The Python binding's own checks, without a GPU: every tensor handed to the
C ABI lives on x's CUDA device and holds the bytes the call reads or writes.
Stand-in tensors (device index, element count and size, a fake address) and
a stand-in library that records its calls replace torch's CUDA tensors and
librmsnorm.so, so each wrapper runs end to end on the CPU."""
import pytest
import torch

import row_wise_normalization_rms_gb300 as rms


class T:
    """A contiguous tensor stand-in on CUDA device ``dev`` (-1: the host)."""

    _next = 1 << 24

    def __init__(self, *shape, dtype=torch.bfloat16, dev=0):
        self.shape = shape
        self.dtype = dtype
        self._dev = dev
        self.device = f"cuda:{dev}" if dev >= 0 else "cpu"
        self._ptr = T._next
        T._next += 1 << 24

    def dim(self):
        return len(self.shape)

    def get_device(self):
        return self._dev

    def numel(self):
        n = 1
        for s in self.shape:
            n *= s
        return n

    def element_size(self):
        return {torch.bfloat16: 2, torch.float16: 2, torch.float32: 4, torch.uint8: 1}[self.dtype]

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return self._ptr


class FakeLib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def f(*args):
            self.calls.append((name, args))
            return 0
        return f


@pytest.fixture()
def lib(monkeypatch):
    fake = FakeLib()
    monkeypatch.setattr(rms, "_LIB", fake)
    return fake


M, N = 6, 64
F32 = torch.float32


def args_of(op):
    """Arguments of a valid call of ``op`` (stream given: no CUDA query)."""
    x = T(M, N)
    if op == "rms_fwd":
        return (x, T(N), T(M, N), T(M, dtype=F32)), {}
    if op == "rms_bwd":
        return (T(M, N), x, T(N), T(M, dtype=F32), T(M, N), T(N, dtype=F32),
                T(4096, dtype=torch.uint8)), {}
    if op == "rms_bwd_noalloc":
        return (T(M, N), x, T(N), T(M, dtype=F32), T(M, N), T(N, dtype=F32)), {}
    if op == "rms_fwd_add":
        return (x, T(M, N), T(N), T(M, N), T(M, N), T(M, dtype=F32)), {}
    if op == "rms_bwd_add":
        return (T(M, N), x, T(N), T(M, dtype=F32), T(M, N), T(M, N), T(N, dtype=F32),
                T(4096, dtype=torch.uint8)), {}
    if op == "rms_fwd_quant":
        return (x, T(N), T(M, N, dtype=torch.uint8), T(M, dtype=F32), T(M, dtype=F32)), {}
    if op == "ln_fwd":
        return (x, T(N), T(N), T(M, N), T(M, dtype=F32), T(M, dtype=F32)), {}
    if op == "ln_bwd":
        return (T(M, N), x, T(N), T(M, dtype=F32), T(M, dtype=F32), T(M, N), T(N, dtype=F32),
                T(N, dtype=F32), T(4096, dtype=torch.uint8)), {}
    raise KeyError(op)


OPS = ["rms_fwd", "rms_bwd", "rms_bwd_noalloc", "rms_fwd_add", "rms_bwd_add", "rms_fwd_quant",
       "ln_fwd", "ln_bwd"]
X_POS = {"rms_bwd": 1, "rms_bwd_noalloc": 1, "rms_bwd_add": 1, "ln_bwd": 1}


@pytest.mark.parametrize("op", OPS)
def test_valid_call_reaches_the_library(lib, op):
    a, kw = args_of(op)
    getattr(rms, op)(*a, stream=0, **kw)
    assert len(lib.calls) == 1
    name, cargs = lib.calls[0]
    assert name.startswith(op)
    # every tensor's address is passed on, in order
    ptrs = [t.data_ptr() for t in a if isinstance(t, T)]
    assert [c for c in cargs if c in ptrs] == ptrs


@pytest.mark.parametrize("op", OPS)
def test_short_buffers_are_refused_before_the_library(lib, op):
    a, _ = args_of(op)
    xi = X_POS.get(op, 0)
    for i, t in enumerate(a):
        if not isinstance(t, T) or i == xi or t.dtype == torch.uint8 and t.shape == (4096,):
            continue  # x defines the sizes; the workspace size is the library's check
        short = list(a)
        shape = list(t.shape)
        shape[-1] -= 1
        short[i] = T(*shape, dtype=t.dtype)
        with pytest.raises(ValueError, match="needs"):
            getattr(rms, op)(*short, stream=0)
    assert lib.calls == []


@pytest.mark.parametrize("op", OPS)
def test_tensors_off_the_device_of_x_are_refused(lib, op):
    a, _ = args_of(op)
    xi = X_POS.get(op, 0)
    for i, t in enumerate(a):
        if not isinstance(t, T):
            continue
        for dev in (-1, 1):  # the host, another GPU
            moved = list(a)
            moved[i] = T(*t.shape, dtype=t.dtype, dev=dev)
            # x on the host is not a CUDA tensor; any other move splits the devices
            msg = "CUDA tensor" if (i == xi and dev < 0) else "must be on"
            with pytest.raises(ValueError, match=msg):
                getattr(rms, op)(*moved, stream=0)
    assert lib.calls == []


def test_none_is_left_to_the_library(lib):
    """NULL arguments are the library's to accept or refuse (dx with inplace_dx=1)."""
    a, _ = args_of("rms_bwd")
    a = list(a)
    a[4] = None
    rms.rms_bwd(*a, inplace_dx=1, stream=0)
    assert lib.calls[0][1][4] is None


def test_rows_must_be_two_dimensional(lib):
    with pytest.raises(ValueError, match="2-D"):
        rms.rms_fwd(T(M * N), T(N), T(M, N), T(M, dtype=F32), stream=0)
