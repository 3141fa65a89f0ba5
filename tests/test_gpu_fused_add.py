"""The residual add fused into RMSNorm (rms_fwd_add / rms_bwd_add) versus the
fp64 oracle through the C ABI: h bit for bit (the stored float32 sum), y,
rstd, dx and dgamma within the bars, on every mapping, with the in-place
aliases the API allows.  The fused calls also reproduce the unfused ones
bit for bit where the arithmetic and the grid are the same."""
import dataclasses

import numpy as np
import pytest
import torch

from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import row_wise_normalization_rms_gb300 as rms
    from synthetic import WORKLOADS, Workload


def _aw(M, N, dtype, gemma=0, seed=0):
    from synthetic import Workload

    wd = ""
    if dtype.endswith("w32"):
        dtype, wd = dtype[:-3], "f32"
    return Workload(name=f"add{M}x{N}_{dtype}{wd}_g{gemma}", M=M, N=N, dtype=dtype, eps=1e-6,
                    op="rms_add", gemma=gemma, seed=seed, weight_dtype=wd,
                    gamma=("normal", 0.0, 0.1) if gemma else ("uniform", 0.5, 1.5),
                    row_scale=("loguniform", 0.01, 100.0), residual=("normal", 0.0, 1.0))


SHAPES = [(3, 7), (17, 8), (64, 128), (31, 257), (40, 1000), (300, 2048), (65, 4096),
          (33, 8192), (70, 10240), (5, 16384), (2, 65536)]
PATHS = ["auto", "registers", "staged", "scalar", "chunked"]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "bf16w32"])
@pytest.mark.parametrize("M,N", SHAPES, ids=[f"{m}x{n}" for m, n in SHAPES])
@pytest.mark.parametrize("path", PATHS)
def test_fused_add_parity(M, N, dtype, path):
    w = _aw(M, N, dtype, seed=M + 2 * N)
    inp = H.inputs_for(w)
    if path in ("registers", "staged", "chunked") and (N * w.elem_bytes) % 16 != 0:
        with pytest.raises(rms.RmsError) as ei:
            H.run_fused(w, inp, path=path)
        assert ei.value.status == rms.RMS_ERR_ALIGNMENT
        return
    try:
        res = H.run_fused(w, inp, path=path)
    except rms.RmsError as e:
        assert e.status == rms.RMS_ERR_UNSUPPORTED and path != "auto", str(e)
        pytest.skip(f"{path} mapping does not take N={N}")
    H.assert_fused_parity(w, inp, res)


@pytest.mark.parametrize("h_alias,dx_alias", [(True, "none"), (False, "dh"), (True, "dy"),
                                              (True, "dh")])
@pytest.mark.parametrize("gemma", [0, 1])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("path", ["auto", "registers", "staged", "scalar", "chunked"])
def test_fused_add_aliases(h_alias, dx_alias, gemma, dtype, path):
    """h written over the residual; dx accumulated into dh or written into dy."""
    w = _aw(129, 2048, dtype, gemma=gemma, seed=17)
    inp = H.inputs_for(w)
    H.assert_fused_parity(w, inp, H.run_fused(w, inp, path=path, h_alias=h_alias,
                                               dx_alias=dx_alias))


@pytest.mark.parametrize("h_alias,dx_alias", [(True, "dy"), (True, "dh"), (False, "none")])
@pytest.mark.parametrize("gemma", [0, 1])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_add_aliases_cluster_rows(h_alias, dx_alias, gemma, dtype):
    """The aliases on rows the chunked mapping splits over a cluster of CTAs
    (65536 columns: 4 CTAs a row for bf16, 8 for f32)."""
    w = _aw(6, 65536, dtype, gemma=gemma, seed=29)
    inp = H.inputs_for(w)
    H.assert_fused_parity(w, inp, H.run_fused(w, inp, path="chunked", h_alias=h_alias,
                                               dx_alias=dx_alias))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("path", ["registers", "staged", "scalar", "chunked"])
def test_fused_matches_unfused_bitwise(dtype, path):
    """y and rstd of rms_fwd_add equal rms_fwd on the stored h, bit for bit on
    the same mapping, and so does dgamma of rms_bwd_add against rms_bwd on h
    where both use the same grid (the staged backward stages dh as a third
    tensor, so its ring, and with it the persistent grid and the partial-sum
    order, differ: there dgamma agrees within the float32 bar)."""
    w = _aw(700, 4096, dtype, seed=23)
    inp = H.inputs_for(w)
    a = H.run_fused(w, inp, path=path)
    g = H.to_device(inp["gamma"], dtype)
    dy = H.to_device(inp["dy"], dtype)
    h = a.h.clone()
    y = torch.empty_like(h)
    r = torch.empty(w.M, device="cuda")
    rms.rms_fwd(h, g, y, r, w.eps, path=path)
    dx = torch.empty_like(h)
    dg = torch.empty(w.N, device="cuda")
    ws = torch.empty(rms.rms_bwd_workspace_size(w.M, w.N), dtype=torch.uint8, device="cuda")
    rms.rms_bwd(dy, h, g, r, dx, dg, ws, path=path)
    torch.cuda.synchronize()
    bits = torch.int32 if dtype == "f32" else torch.int16
    assert torch.equal(a.y.view(bits), y.view(bits))
    assert torch.equal(a.rstd.view(torch.int32), r.view(torch.int32))
    if path != "staged":
        assert torch.equal(a.dgamma.view(torch.int32), dg.view(torch.int32))
    else:
        assert torch.allclose(a.dgamma, dg, rtol=1e-5, atol=1e-5 * float(dg.abs().max()))


FUSED_FULL = ([n for n, w in WORKLOADS.items() if w.op == "rms_add"]
              if torch.cuda.is_available() else [])


@pytest.mark.parametrize("name", FUSED_FULL)
def test_fused_add_full_size(name):
    w = WORKLOADS[name]
    inp = H.inputs_for(w)
    res = H.run_fused(w, inp)
    H.assert_fused_parity(w, inp, res)  # every row


def test_fused_add_rejects_bad_aliases():
    M, N = 64, 1024
    x = torch.randn(M, N, device="cuda")
    res = torch.randn(M, N, device="cuda")
    g = torch.ones(N, device="cuda")
    y = torch.empty_like(x)
    r = torch.empty(M, device="cuda")
    with pytest.raises(rms.RmsError) as ei:  # h over x
        rms.rms_fwd_add(x, res, g, y, x, r)
    assert ei.value.status == rms.RMS_ERR_INVALID_ARG
    with pytest.raises(rms.RmsError) as ei:  # h over y
        rms.rms_fwd_add(x, res, g, y, y, r)
    assert ei.value.status == rms.RMS_ERR_INVALID_ARG
    h = torch.empty_like(x)
    rms.rms_fwd_add(x, res, g, y, h, r)
    dy = torch.randn(M, N, device="cuda")
    dg = torch.empty(N, device="cuda")
    ws = torch.empty(rms.rms_bwd_workspace_size(M, N), dtype=torch.uint8, device="cuda")
    with pytest.raises(rms.RmsError) as ei:  # dh over dy
        rms.rms_bwd_add(dy, h, g, r, dy, torch.empty_like(x), dg, ws)
    assert ei.value.status == rms.RMS_ERR_INVALID_ARG
    with pytest.raises(rms.RmsError) as ei:  # dx over h
        rms.rms_bwd_add(dy, h, g, r, torch.randn_like(x), h, dg, ws)
    assert ei.value.status == rms.RMS_ERR_INVALID_ARG
    torch.cuda.synchronize()


def test_fused_add_launch_count():
    M, N = 256, 2048
    x = torch.randn(M, N, device="cuda", dtype=torch.bfloat16)
    res = torch.randn_like(x)
    g = torch.ones(N, device="cuda", dtype=torch.bfloat16)
    y = torch.empty_like(x)
    r = torch.empty(M, device="cuda")
    dg = torch.empty(N, device="cuda")
    ws = torch.empty(rms.rms_bwd_workspace_size(M, N), dtype=torch.uint8, device="cuda")
    n0 = rms.rms_launch_count()
    rms.rms_fwd_add(x, res, g, y, res, r)
    rms.rms_bwd_add(torch.randn_like(x), res, g, r, torch.randn_like(x), torch.empty_like(x), dg,
                    ws)
    torch.cuda.synchronize()
    assert rms.rms_launch_count() - n0 == 1 + 2  # one fused kernel each way + column reduction
