"""rms_bwd_noalloc, the backward for callers that cannot allocate device
scratch (a plugin whose host program owns all device memory, a latency-
critical loop that cannot afford cudaMalloc's device-wide synchronisation).

It is called through the C ABI (ctypes, raw pointers) and must give what
rms_bwd gives with a caller workspace, on two calls in a row (the second
call finds the first call's partial sums still in the shared scratch
array).  Both entry points take the same row mapping and the same partial
rows, so dx and dgamma must agree bit for bit; the result is also checked
against the fp64 oracle.  This file is collected last so a failure here
does not stop the rest of the suite.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _case(name, M=None):
    from synthetic import WORKLOADS

    w = WORKLOADS[name]
    return w if M is None else w.with_shape(M)


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


@pytest.mark.parametrize("name,M", [("llama7b_bf16_8192x4096", None),
                                    ("gemma_bf16_32768x3072", 4096),
                                    ("tiny_f32_64x128", None)])
def test_noalloc_matches_workspace_entry_point(name, M):
    import row_wise_normalization_rms_gb300 as rms
    from tests import gpu_helpers as H

    w = _case(name, M)
    inp = H.inputs_for(w)
    code = rms.RMS_BF16 if w.dtype == "bf16" else rms.RMS_F32
    x = H.to_device(inp["x"], w.dtype)
    g = H.to_device(inp["gamma"], w.dtype)
    r = torch.empty(w.M, device="cuda")
    y = torch.empty_like(x)
    rms.rms_fwd(x, g, y, r, w.eps, w.gemma)

    # The existing entry point, with a caller-provided workspace.
    dy_ref = H.to_device(inp["dy"], w.dtype)
    dx_ref = torch.empty_like(x)
    dg_ref = torch.empty(w.N, device="cuda")
    ws = torch.empty(rms.rms_bwd_workspace_size(w.M, w.N), dtype=torch.uint8, device="cuda")
    rms.rms_bwd(dy_ref, x, g, r, None if w.inplace_dx else dx_ref, dg_ref, ws, w.gemma,
                w.inplace_dx)
    if w.inplace_dx:
        dx_ref = dy_ref
    torch.cuda.synchronize()

    lib = rms.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        dy = H.to_device(inp["dy"], w.dtype)
        dx = dy if w.inplace_dx else torch.empty_like(x)
        dg = torch.full((w.N,), float("nan"), device="cuda")
        st = lib.rms_bwd_noalloc(dy.data_ptr(), x.data_ptr(), g.data_ptr(), r.data_ptr(),
                                 None if w.inplace_dx else dx.data_ptr(), dg.data_ptr(), w.M, w.N,
                                 code, w.gemma, w.inplace_dx, stream)
        assert st == rms.RMS_OK, lib.rms_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(_bits(dx), _bits(dx_ref)), f"call {call}: dx differs from rms_bwd's"
        assert torch.equal(dg.view(torch.int32), dg_ref.view(torch.int32)), \
            f"call {call}: dgamma differs from rms_bwd's"
    # and against the oracle, with the parity tests' bars
    red = rms.rms_bwd_reduction(w.M, w.N, code, w.gemma)
    H.assert_parity(w, inp, H.GpuResult(y, r, dx, dg, True, red), H.sample_rows(w.M))


def test_noalloc_at_its_size_limit_through_the_binding():
    """The widest bf16 rows (a multiple of 8) whose workspace need fits the
    32 MiB scratch, with at least as many rows as the backward has partial
    rows: the partial rows run to the end of the array's reach."""
    import row_wise_normalization_rms_gb300 as rms

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    limit = 32 << 20
    N = (limit // (4 * sms * 4)) // 8 * 8
    M = 4 * sms + 37
    assert rms.rms_bwd_workspace_size(M, N) <= limit < rms.rms_bwd_workspace_size(M, N + 64)
    gen = torch.Generator(device="cuda").manual_seed(5)
    x = torch.randn(M, N, device="cuda", generator=gen).to(torch.bfloat16)
    g = (1 + 0.2 * torch.randn(N, device="cuda", generator=gen)).to(torch.bfloat16)
    dy = torch.randn(M, N, device="cuda", generator=gen).to(torch.bfloat16)
    y = torch.empty_like(x)
    r = torch.empty(M, device="cuda")
    rms.rms_fwd(x, g, y, r, 1e-6)
    dx_ref, dg_ref = torch.empty_like(x), torch.empty(N, device="cuda")
    ws = torch.empty(rms.rms_bwd_workspace_size(M, N), dtype=torch.uint8, device="cuda")
    rms.rms_bwd(dy, x, g, r, dx_ref, dg_ref, ws)
    for _ in range(2):
        dx, dg = torch.empty_like(x), torch.full((N,), float("nan"), device="cuda")
        rms.rms_bwd_noalloc(dy, x, g, r, dx, dg)
        torch.cuda.synchronize()
        assert torch.equal(dx.view(torch.int16), dx_ref.view(torch.int16))
        assert torch.equal(dg.view(torch.int32), dg_ref.view(torch.int32))
    assert rms.rms_last_device_status() == rms.RMS_OK


def test_noalloc_empty_batch_zeroes_dgamma():
    import row_wise_normalization_rms_gb300 as rms

    N = 96
    x = torch.empty(0, N, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(N, device="cuda", dtype=torch.bfloat16)
    dg = torch.full((N,), float("nan"), device="cuda")
    rms.rms_bwd_noalloc(x, x, g, torch.empty(0, device="cuda"), torch.empty_like(x), dg)
    torch.cuda.synchronize()
    assert bool((dg == 0).all())


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import row_wise_normalization_rms_gb300 as rms

    lib = rms.lib()
    M, N = 4096, 16384  # min(M, 4*SMs) * N * 4 bytes > 32 MiB on a 148- or 152-SM GB300
    assert rms.rms_bwd_workspace_size(M, N) > (32 << 20)
    x = torch.empty(8, device="cuda")  # never touched: the size check comes first
    p = x.data_ptr()
    st = lib.rms_bwd_noalloc(p, p + 1024, p + 2048, p + 3072, p + 4096, p + 5120, M, N,
                             rms.RMS_BF16, 0, 0, None)
    assert st == rms.RMS_ERR_WORKSPACE
