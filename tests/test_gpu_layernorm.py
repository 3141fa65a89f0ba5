"""LayerNorm on the CUDA engine versus the fp64 LayerNorm oracle, element by
element, through the C ABI (ln_fwd / ln_bwd).

Small shapes are compared in full; the full-size LayerNorm workloads on
sampled rows for y, mean, rstd and dx and in full for dw and db.
Tolerances are those of ``oracle.compare`` (LayerNorm section).
"""
import numpy as np
import pytest
import torch

from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import row_wise_normalization_rms_gb300 as rms
    from synthetic import WORKLOADS, Workload


def _lw(M, N, dtype, seed=0, eps=1e-5, inplace=0, bias=True, row_scale=True):
    """A LayerNorm test workload with the LayerNorm chapter's laws (x = -2.3 +
    0.5 N(0,1), w, b ~ U(0,1), dy = 0.1 N(0,1)) and, by default, a per-row
    scale spanning 1e-2..1e2 so that eps matters on some rows."""
    from synthetic import Workload

    wd = ""
    if dtype.endswith("w32"):
        dtype, wd = dtype[:-3], "f32"
    return Workload(name=f"ln{M}x{N}_{dtype}{wd}_i{inplace}", M=M, N=N, dtype=dtype, eps=eps,
                    op="ln", x=("normal", -2.3, 0.5), gamma=("uniform", 0.0, 1.0),
                    beta=("uniform", 0.0, 1.0) if bias else None, dy=("normal", 0.0, 0.1),
                    row_scale=("loguniform", 0.01, 100.0) if row_scale else None,
                    inplace_dx=inplace, seed=seed, weight_dtype=wd)


SHAPES = [
    (1, 1), (3, 7), (17, 8), (5, 64), (31, 257), (128, 257), (40, 1000), (9, 1024), (2000, 512),
    (7, 2048), (6, 3072), (900, 4096), (4, 5120), (700, 8192), (3, 11008), (60, 15872),
    (30, 16384), (2, 32768), (2, 40000),
]
PATHS = {"auto": ("auto", "auto"), "vector": ("registers", "staged"), "scalar": ("scalar", "scalar")}


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "bf16w32", "f16w32"])
@pytest.mark.parametrize("M,N", SHAPES, ids=[f"{m}x{n}" for m, n in SHAPES])
@pytest.mark.parametrize("path", list(PATHS))
def test_ln_small_shapes_full_parity(M, N, dtype, path):
    w = _lw(M, N, dtype, seed=M + 3 * N)
    inp = H.inputs_for(w)
    fp, bp = PATHS[path]
    if path == "vector" and (N * w.elem_bytes) % 16 != 0:
        with pytest.raises(rms.RmsError) as ei:
            H.run_ln(w, inp, fwd_path=fp, bwd_path=bp)
        assert ei.value.status == rms.RMS_ERR_ALIGNMENT
        return
    try:
        res = H.run_ln(w, inp, fwd_path=fp, bwd_path=bp)
    except rms.RmsError as e:
        assert e.status == rms.RMS_ERR_UNSUPPORTED and path == "vector", str(e)
        pytest.skip(f"the vector mappings do not take N={N}")
    H.assert_ln_parity(w, inp, res)


@pytest.mark.parametrize("bias,with_db", [(False, True), (True, False), (False, False)])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16w32"])
@pytest.mark.parametrize("path", list(PATHS))
def test_ln_without_bias_or_db(bias, with_db, dtype, path):
    w = _lw(300, 2048, dtype, seed=4)
    inp = H.inputs_for(w)
    fp, bp = PATHS[path]
    res = H.run_ln(w, inp, fwd_path=fp, bwd_path=bp, with_db=with_db, bias=bias)
    H.assert_ln_parity(w, inp, res, bias=bias)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "bf16w32"])
@pytest.mark.parametrize("M,N", [(257, 3072), (65, 1000), (31, 257)])
def test_ln_inplace_dx(M, N, dtype):
    w = _lw(M, N, dtype, seed=7, inplace=1)
    inp = H.inputs_for(w)
    H.assert_ln_parity(w, inp, H.run_ln(w, inp))


LN_FULL = [n for n, w in WORKLOADS.items() if w.op == "ln"] if torch.cuda.is_available() else []


@pytest.mark.parametrize("name", LN_FULL)
def test_ln_workload_full_size(name):
    """Every LayerNorm workload at full size in the mapping the benchmark uses."""
    w = WORKLOADS[name]
    inp = H.inputs_for(w)
    res = H.run_ln(w, inp)
    H.assert_ln_parity(w, inp, res)  # every row


def test_ln_chapter_unit_test_bar():
    """The LayerNorm chapter's unit test: 1151 x 8192 fp16, eps 1e-5, every
    output within an absolute 1e-2 of the reference (its bar), here the fp64
    oracle on the same inputs; the stricter per-dtype bars hold as well."""
    w = WORKLOADS["ln_test_f16_1151x8192"]
    inp = H.inputs_for(w)
    res = H.run_ln(w, inp)
    y, mean, rstd, _, _, dx, _ = H.ln_oracle_rows(w, inp, np.arange(w.M))
    dw, db = H.ln_oracle_wsums(w, inp)[:2]
    for got, ref in ((res.y, y), (res.dx, dx), (res.dw, dw), (res.db, db)):
        assert np.max(np.abs(H.to_host64(got) - ref)) <= 1e-2
    H.assert_ln_parity(w, inp, res)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("path", list(PATHS))
def test_ln_inplace_matches_out_of_place_bitwise(dtype, path):
    w = _lw(500, 4096, dtype, seed=21)
    inp = H.inputs_for(w)
    fp, bp = PATHS[path]
    a = H.run_ln(w, inp, fwd_path=fp, bwd_path=bp, inplace=0)
    b = H.run_ln(w, inp, fwd_path=fp, bwd_path=bp, inplace=1)
    for u, v in ((a.y, b.y), (a.dx, b.dx), (a.dw, b.dw), (a.db, b.db)):
        assert torch.equal(u.view(torch.uint8) if u.dtype != torch.float32 else u.view(torch.int32),
                           v.view(torch.uint8) if v.dtype != torch.float32 else v.view(torch.int32))


def test_ln_dw_db_bitwise_reproducible():
    """A static row assignment and fixed-order sums: repeated calls give the
    same bits for dw and db."""
    w = WORKLOADS["ln_bench_f16_4096x8192"]
    inp = H.inputs_for(w)
    first = H.run_ln(w, inp)
    for _ in range(3):
        again = H.run_ln(w, inp)
        assert torch.equal(first.dw.view(torch.int32), again.dw.view(torch.int32))
        assert torch.equal(first.db.view(torch.int32), again.db.view(torch.int32))
        assert torch.equal(first.dx.view(torch.int16), again.dx.view(torch.int16))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_ln_edge_rows(dtype):
    """A constant row (variance 0: y = b, rstd = eps^-1/2; 1.5 so that the
    float32 row sum is exact), a row of zeros, one nonzero element, and (f32)
    a row far from zero relative to its spread."""
    w = _lw(6, 1024, dtype, seed=3, row_scale=False)
    inp = H.inputs_for(w)
    x = inp["x"].copy()
    one = np.asarray(1.0).astype(x.dtype) if dtype != "bf16" else np.uint16(0x3F80)
    x[0] = np.asarray(1.5).astype(x.dtype) if dtype != "bf16" else np.uint16(0x3FC0)
    x[1] = 0
    x[2] = 0
    x[2, 17] = one
    if dtype == "f32":
        x[3] = (1000.0 + np.linspace(-1, 1, 1024)).astype(np.float32)
    inp = dict(inp, x=x)
    H.assert_ln_parity(w, inp, H.run_ln(w, inp))
    H.assert_ln_parity(w, inp, H.run_ln(w, inp, path="scalar"))


def test_ln_empty_batch():
    N = 512
    w = torch.rand(N, device="cuda")
    x = torch.empty(0, N, device="cuda")
    y = torch.empty(0, N, device="cuda")
    mu = torch.empty(0, device="cuda")
    r = torch.empty(0, device="cuda")
    rms.ln_fwd(x, w, None, y, mu, r)
    dw = torch.full((N,), 7.0, device="cuda")
    db = torch.full((N,), 7.0, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    rms.ln_bwd(x, x, w, mu, r, y, dw, db, ws)
    torch.cuda.synchronize()
    assert bool((dw == 0).all()) and bool((db == 0).all())


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_ln_misaligned_pointers_use_scalar_path(dtype):
    w = _lw(100, 1024, dtype, seed=9)
    inp = H.inputs_for(w)
    dt = H.tdtype(dtype)
    M, N = w.M, w.N
    x = torch.empty(M * N + 1, dtype=dt, device="cuda")[1:].view(M, N)
    x.copy_(H.to_device(inp["x"], dtype))
    g = H.to_device(inp["gamma"], dtype)
    b = H.to_device(inp["beta"], dtype)
    y = torch.empty(M * N + 1, dtype=dt, device="cuda")[1:].view(M, N)
    mu = torch.empty(M, device="cuda")
    r = torch.empty(M, device="cuda")
    with pytest.raises(rms.RmsError) as ei:
        rms.ln_fwd(x, g, b, y, mu, r, w.eps, path="registers")
    assert ei.value.status == rms.RMS_ERR_ALIGNMENT
    rms.ln_fwd(x, g, b, y, mu, r, w.eps)
    dy = H.to_device(inp["dy"], dtype)
    dx = torch.empty(M * N + 1, dtype=dt, device="cuda")[1:].view(M, N)
    dw = torch.empty(N, device="cuda")
    db = torch.empty(N, device="cuda")
    ws = torch.empty(rms.ln_bwd_workspace_size(M, N), dtype=torch.uint8, device="cuda")
    with pytest.raises(rms.RmsError) as ei:
        rms.ln_bwd(dy, x, g, mu, r, dx, dw, db, ws, path="staged")
    assert ei.value.status == rms.RMS_ERR_ALIGNMENT
    rms.ln_bwd(dy, x, g, mu, r, dx, dw, db, ws)
    torch.cuda.synchronize()
    red = rms.ln_bwd_reduction(M, N, rms.dtype_code(x, g), "scalar")
    H.assert_ln_parity(w, inp, H.LnResult(y, mu, r, dx, dw, db, True, red))


def test_ln_workspace_and_launch_count():
    w = _lw(1000, 2048, "bf16", seed=1)
    inp = H.inputs_for(w)
    M, N = w.M, w.N
    assert rms.ln_bwd_workspace_size(M, N) == 2 * rms.rms_bwd_workspace_size(M, N)
    x = H.to_device(inp["x"], "bf16")
    g = H.to_device(inp["gamma"], "bf16")
    dy = H.to_device(inp["dy"], "bf16")
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    mu = torch.empty(M, device="cuda")
    r = torch.empty(M, device="cuda")
    dw = torch.empty(N, device="cuda")
    db = torch.empty(N, device="cuda")
    need = rms.ln_bwd_workspace_size(M, N)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    rms.ln_fwd(x, g, None, y, mu, r)
    with pytest.raises(rms.RmsError) as ei:
        rms.ln_bwd(dy, x, g, mu, r, dx, dw, db, small)
    assert ei.value.status == rms.RMS_ERR_WORKSPACE
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(rms.RmsError) as ei:  # misaligned workspace
        rms.ln_bwd(dy, x, g, mu, r, dx, dw, db, ws[16:])
    assert ei.value.status == rms.RMS_ERR_WORKSPACE
    n0 = rms.rms_launch_count()
    rms.ln_fwd(x, g, None, y, mu, r)
    rms.ln_bwd(dy, x, g, mu, r, dx, dw, db, ws)
    rms.ln_bwd(dy, x, g, mu, r, dx, dw, None, ws)
    # forward; rows kernel + one column-sum launch for dw and db; the same without db
    assert rms.rms_launch_count() - n0 == 1 + 2 + 2
    with pytest.raises(rms.RmsError) as ei:  # dx on top of x
        rms.ln_bwd(dy, x, g, mu, r, x, dw, db, ws)
    assert ei.value.status == rms.RMS_ERR_INVALID_ARG


@pytest.mark.parametrize("N", [1024, 8192])
def test_ln_staged_wait_timeout_reports_status(N):
    """With the poll limit at 0 the staged backward gives up at its first
    wait: it drains its copies, raises the device status and returns; the
    host sees RMS_ERR_TIMEOUT and the context stays usable."""
    w = _lw(600, N, "bf16", seed=11)
    inp = H.inputs_for(w)
    x = H.to_device(inp["x"], "bf16")
    g = H.to_device(inp["gamma"], "bf16")
    b = H.to_device(inp["beta"], "bf16")
    dy = H.to_device(inp["dy"], "bf16")
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    mu = torch.empty(w.M, device="cuda")
    r = torch.empty(w.M, device="cuda")
    dw = torch.empty(w.N, device="cuda")
    db = torch.empty(w.N, device="cuda")
    ws = torch.empty(rms.ln_bwd_workspace_size(w.M, w.N), dtype=torch.uint8, device="cuda")
    rms.ln_fwd(x, g, b, y, mu, r, w.eps)
    torch.cuda.synchronize()
    assert rms.rms_last_device_status() == rms.RMS_OK
    prev = rms.rms_set_wait_limit(0)
    try:
        rms.ln_bwd(dy, x, g, mu, r, dx, dw, db, ws, path="staged")
        assert rms.rms_last_device_status() == rms.RMS_ERR_TIMEOUT
        assert rms.rms_last_device_status() == rms.RMS_OK
    finally:
        rms.rms_set_wait_limit(prev)
    H.assert_ln_parity(w, inp, H.run_ln(w, inp, bwd_path="staged"))
