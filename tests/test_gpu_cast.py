"""rms_dgamma_cast on GB300: the float32 weight gradient rounded to the
weight's own type ("Hướng dẫn Triton RMSNorm", section "Reduce dgamma không
có race khi ghi": reduced in float32, then converted to gamma's dtype).

The rounding is an integer decision taken in float32 on both sides, so on
seeded float32 vectors (ties, overflow, subnormals, ragged and misaligned
tails) the kernel must equal the oracle's round-to-nearest-even bit for bit;
after a backward it must sit within the column sum's float32 bar plus one
rounding of the oracle's fp64 dgamma."""
import ctypes

import numpy as np
import pytest
import torch

from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import row_wise_normalization_rms_gb300 as rms
    from oracle import compare
    from oracle import rmsnorm_oracle as orc
    from synthetic import WORKLOADS

TYPES = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def _vectors(N, seed):
    """Seeded float32 values: finite random bit patterns, values in the 16-bit
    types' ranges, exact ties of both types, and both types' extremes."""
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2 ** 32, size=N, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32).copy()
    v[~np.isfinite(v)] = 1.0
    k = rng.integers(0, 5, size=N)
    scale = 10.0 ** rng.integers(-9, 6, size=N)
    v = np.where(k == 1, (rng.standard_normal(N) * scale).astype(np.float32), v)
    # exact bf16 ties: a bf16 value plus half its spacing
    b = (rng.standard_normal(N) * scale).astype(np.float32)
    b = ((b.view(np.uint32) >> 16) << 16).view(np.float32)
    tie_bf16 = (b.view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    v = np.where(k == 2, tie_bf16, v)
    # exact f16 ties: an f16 value plus half its spacing (normal range)
    h = (rng.standard_normal(N) * 10.0 ** rng.integers(-3, 4, size=N)).astype(np.float16)
    h32 = h.astype(np.float32)
    tie_f16 = (h32.view(np.uint32) | np.uint32(1 << 12)).view(np.float32)
    v = np.where(k == 3, tie_f16, v)
    extremes = np.array([65504.0, 65520.0, -65520.0, 2.0 ** -24, 3 * 2.0 ** -25, 2.0 ** -26,
                         3.3895313892515355e38, np.finfo(np.float32).max, -0.0, 0.0],
                        dtype=np.float32)
    v[:min(N, extremes.size)] = extremes[:min(N, extremes.size)]
    return v


@pytest.mark.parametrize("wdtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("N", [1, 3, 4, 5, 1000, 4097, (1 << 20) + 3])
@pytest.mark.parametrize("offset", [0, 1])
def test_cast_bit_exact_against_oracle(wdtype, N, offset):
    v = _vectors(N, seed=N * 7 + offset)
    # offset 1: the float32 source and the output start one element past a
    # 16-byte boundary, which takes the element-wise form
    src = torch.empty(N + offset, dtype=torch.float32, device="cuda")
    src[offset:] = torch.from_numpy(v).cuda()
    out = torch.full((N + offset + 2,), float("nan"), dtype=TYPES[wdtype], device="cuda")
    rms.rms_dgamma_cast(src[offset:], out[offset:offset + N])
    torch.cuda.synchronize()
    want = orc.cast_to_weight_dtype(v, wdtype)
    got = out[offset:offset + N].to(torch.float64).cpu().numpy()
    same = (got == want) & (np.signbit(got) == np.signbit(want))
    assert same.all(), (v[~same][:4], got[~same][:4], want[~same][:4])
    # nothing written outside the N outputs
    assert torch.isnan(out[offset + N:]).all() and (offset == 0 or torch.isnan(out[:offset]).all())


@pytest.mark.parametrize("code", [0, 3, 4])  # RMS_F32, RMS_BF16_W32, RMS_F16_W32: a float32 weight
def test_cast_to_float32_weight_is_a_copy(code):
    v = torch.from_numpy(_vectors(4099, seed=code)).cuda()
    out = torch.full((4099,), float("nan"), device="cuda")
    st = rms.lib().rms_dgamma_cast(v.data_ptr(), out.data_ptr(), 4099, code,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), v.view(torch.int32))


def test_cast_rejects_bad_arguments():
    v = torch.zeros(64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    L = rms.lib()
    assert L.rms_dgamma_cast(None, v.data_ptr(), 8, 1, s) == rms.RMS_ERR_INVALID_ARG
    assert L.rms_dgamma_cast(v.data_ptr(), None, 8, 1, s) == rms.RMS_ERR_INVALID_ARG
    assert L.rms_dgamma_cast(v.data_ptr(), v[32:].data_ptr(), 0, 1, s) == rms.RMS_ERR_INVALID_ARG
    assert L.rms_dgamma_cast(v.data_ptr(), v[32:].data_ptr(), 8, 9, s) == rms.RMS_ERR_INVALID_ARG
    # output overlapping the source (bf16 output of 16 elements inside it)
    assert L.rms_dgamma_cast(v.data_ptr(), v[4:].data_ptr(), 16, 1, s) == rms.RMS_ERR_INVALID_ARG


@pytest.mark.parametrize("name,M", [("llama7b_bf16_8192x4096", None),
                                    ("wide_f16_16384x8192", 2048),
                                    ("timing_f32_128x257", None)])
def test_backward_then_cast_against_oracle(name, M):
    w = WORKLOADS[name]
    if M is not None:
        w = w.with_shape(M)
    inp = H.inputs_for(w)
    res = H.run_gpu(w, inp)
    out = torch.empty(w.N, dtype=TYPES[w.wdtype], device="cuda")
    rms.rms_dgamma_cast(res.dgamma, out)
    torch.cuda.synchronize()
    ref, scale = H.oracle_dgamma(w, inp)
    c = compare.check_weight_cast(H.to_host64(out), ref, scale, w.dtype, w.wdtype, res.reduction)
    assert c.ok, str(c)
    # the cast of the same float32 dgamma twice gives the same bits
    again = torch.empty_like(out)
    rms.rms_dgamma_cast(res.dgamma, again)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16 if out.element_size() == 2 else torch.int32),
                       again.view(torch.int16 if out.element_size() == 2 else torch.int32))
