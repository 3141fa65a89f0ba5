"""rms_bwd_noalloc, the backward for callers that cannot allocate device
scratch (a plugin whose host program owns all device memory, a latency-
critical loop that cannot afford cudaMalloc's device-wide synchronisation).

It is called through the C ABI (ctypes, raw pointers) and must give what
rms_bwd gives with a caller workspace, within the tolerances of the parity
tests, on two calls in a row (the second call finds the first call's
partial sums still in the shared scratch array).  This file is collected
last so a failure here does not stop the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _case(name, M=None):
    from synthetic import WORKLOADS

    w = WORKLOADS[name]
    return w if M is None else w.with_shape(M)


@pytest.mark.parametrize("name,M", [("llama7b_bf16_8192x4096", None),
                                    ("gemma_bf16_32768x3072", 4096),
                                    ("tiny_f32_64x128", None)])
def test_noalloc_matches_workspace_entry_point(name, M):
    import row_wise_normalization_rms_gb300 as rms
    from oracle import compare
    from tests import gpu_helpers as H

    w = _case(name, M)
    inp = H.inputs_for(w)
    dt = H.tdtype(w.dtype)
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
        ref_dx = H.to_host64(dx_ref)
        ref_dg = H.to_host64(dg_ref)
        c_dx = compare.check_dx(H.to_host64(dx), ref_dx, np.abs(ref_dx), w.dtype)
        c_dg = compare.check_dgamma(H.to_host64(dg), ref_dg, np.abs(ref_dg), w.dtype)
        assert c_dx.ok and c_dg.ok, (call, str(c_dx), str(c_dg))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import row_wise_normalization_rms_gb300 as rms

    lib = rms.lib()
    M, N = 4096, 16384  # min(M, 4*SMs) * N * 4 bytes > 32 MiB on a 152-SM GB300
    assert rms.rms_bwd_workspace_size(M, N) > (32 << 20)
    x = torch.empty(8, device="cuda")  # never touched: the size check comes first
    p = x.data_ptr()
    st = lib.rms_bwd_noalloc(p, p + 1024, p + 2048, p + 3072, p + 4096, p + 5120, M, N,
                             rms.RMS_BF16, 0, 0, None)
    assert st == rms.RMS_ERR_WORKSPACE
