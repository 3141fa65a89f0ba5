"""CUDA path versus the fp64 oracle, element by element, through the C ABI.

Every row and column is compared, the full-size workloads included (the
oracle runs block by block on the host); a few extra wide-row cases compare
sampled rows.  Tolerances are those of ``oracle.compare``.
"""
import dataclasses

import numpy as np
import pytest
import torch

from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import row_wise_normalization_rms_gb300 as rms
    from oracle import rmsnorm_oracle as orc
    from synthetic import WORKLOADS, Workload, storage_to_float64


def _w(M, N, dtype, gemma=0, inplace=0, eps=1e-6, seed=0, **kw):
    """A test workload; dtype "bf16w32"/"f16w32" means 16-bit activations, float32 weight."""
    from synthetic import Workload

    wd = ""
    if dtype.endswith("w32"):
        dtype, wd = dtype[:-3], "f32"
    return Workload(name=f"t{M}x{N}_{dtype}{wd}_g{gemma}_i{inplace}", M=M, N=N, dtype=dtype,
                    eps=eps, gemma=gemma, inplace_dx=inplace, seed=seed, weight_dtype=wd,
                    gamma=("normal", 0.0, 0.1) if gemma else ("uniform", 0.5, 1.5),
                    row_scale=("loguniform", 0.01, 100.0), **kw)


SMALL_SHAPES = [
    (1, 1), (3, 7), (17, 8), (5, 64), (64, 128), (33, 256), (31, 257), (128, 257), (40, 1000),
    (9, 1024), (2000, 512), (1200, 1000), (7, 2048), (6, 3072), (900, 4096), (4, 5120),
    (700, 8192), (3, 11008), (300, 16384), (2, 32768),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "bf16w32", "f16w32"])
@pytest.mark.parametrize("M,N", SMALL_SHAPES, ids=[f"{m}x{n}" for m, n in SMALL_SHAPES])
@pytest.mark.parametrize("path", ["auto", "registers", "staged", "scalar", "chunked"])
def test_small_shapes_full_parity(M, N, dtype, path):
    w = _w(M, N, dtype, seed=M + N)
    b = 4 if w.dtype == "f32" else 2
    inp = H.inputs_for(w)
    if path in ("registers", "staged", "chunked") and (N * b) % 16 != 0:
        with pytest.raises(rms.RmsError) as ei:
            H.run_gpu(w, inp, path=path)
        assert ei.value.status == rms.RMS_ERR_ALIGNMENT
        return
    try:
        res = H.run_gpu(w, inp, path=path)
    except rms.RmsError as e:
        assert e.status == rms.RMS_ERR_UNSUPPORTED and path != "auto", str(e)
        pytest.skip(f"{path} mapping does not take N={N}")
    H.assert_parity(w, inp, res)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "bf16w32", "f16w32"])
@pytest.mark.parametrize("M,N", [(400, 10240), (153, 11008), (300, 12288), (161, 5120)])
@pytest.mark.parametrize("gemma", [0, 1])
def test_wide_rows_one_cta_per_sm(M, N, dtype, gemma):
    """Backward rows that leave the staged mapping one CTA per SM (16-bit rows
    of 19-24 KiB, float32 rows of 20 KiB) take three vectors a thread; each
    persistent CTA works through several rows."""
    w = _w(M, N, dtype, gemma=gemma, seed=M)
    inp = H.inputs_for(w)
    for path in ("auto", "staged"):
        H.assert_parity(w, inp, H.run_gpu(w, inp, path=path))


@pytest.mark.parametrize("gemma,inplace", [(0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "bf16w32", "f16w32"])
@pytest.mark.parametrize("M,N", [(257, 3072), (65, 1000), (31, 257)])
def test_gemma_and_inplace(M, N, dtype, gemma, inplace):
    w = _w(M, N, dtype, gemma=gemma, inplace=inplace, seed=7)
    inp = H.inputs_for(w)
    H.assert_parity(w, inp, H.run_gpu(w, inp))


FULL = [n for n, w in WORKLOADS.items() if w.op == "rms"] if torch.cuda.is_available() else []


@pytest.mark.parametrize("name", FULL)
def test_workload_full_size(name):
    """Every workload at its full size, in the mapping the benchmark uses,
    compared on every row (block by block on the host)."""
    w = WORKLOADS[name]
    inp = H.inputs_for(w)
    res = H.run_gpu(w, inp)
    H.assert_parity(w, inp, res)


@pytest.mark.parametrize("path", ["registers", "staged"])
def test_headline_workload_both_mappings(path):
    """16384 x 8192 bf16 through each vector mapping, full size, every row."""
    w = WORKLOADS["wide_bf16_16384x8192"]
    inp = H.inputs_for(w)
    H.assert_parity(w, inp, H.run_gpu(w, inp, path=path))


@pytest.mark.parametrize("name", ["wide_bf16_16384x8192", "gemma_bf16_32768x3072"])
def test_dgamma_bar_sees_dropped_rows(name):
    """dgamma from the GPU passes the tight and normwise bars; the same
    dgamma with one row's contribution taken out (a middle row, the last
    row), or the last eight rows', fails the tight bar."""
    from oracle import compare

    w = WORKLOADS[name]
    inp = H.inputs_for(w)
    res = H.run_gpu(w, inp)
    ref, scale = H.oracle_dgamma(w, inp)
    got = H.to_host64(res.dgamma)
    ok = compare.dgamma_checks(got, ref, scale, w.dtype, res.reduction)
    assert all(c.ok for c in ok), [str(c) for c in ok]
    for lo, hi in ((w.M // 2, w.M // 2 + 1), (w.M - 1, w.M), (w.M - 8, w.M)):
        x = storage_to_float64(inp["x"][lo:hi], w.dtype)
        dy = storage_to_float64(inp["dy"][lo:hi], w.dtype)
        part = orc.rms_dgamma(x, dy, w.eps)
        tight = compare.dgamma_checks(got - part, ref, scale, w.dtype, res.reduction)[2]
        assert not tight.ok, f"rows {lo}..{hi - 1} dropped: {tight}"


def test_dgamma_bitwise_reproducible():
    w = WORKLOADS["llama7b_bf16_8192x4096"]
    inp = H.inputs_for(w)
    a = H.run_gpu(w, inp)
    b = H.run_gpu(w, inp)
    c = H.run_gpu(w, inp)
    assert torch.equal(a.dgamma.view(torch.int32), b.dgamma.view(torch.int32))
    assert torch.equal(a.dgamma.view(torch.int32), c.dgamma.view(torch.int32))
    assert torch.equal(a.dx.view(torch.int16), b.dx.view(torch.int16))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("path", ["auto", "registers", "staged", "scalar", "chunked"])
def test_inplace_matches_out_of_place_bitwise(dtype, path):
    w = _w(1500, 2048, dtype, seed=3)
    inp = H.inputs_for(w)
    a = H.run_gpu(w, inp, path=path, inplace=0)
    b = H.run_gpu(w, inp, path=path, inplace=1)
    bits = torch.int32 if dtype == "f32" else torch.int16
    assert torch.equal(a.dx.view(bits), b.dx.view(bits))
    assert torch.equal(a.dgamma.view(torch.int32), b.dgamma.view(torch.int32))


@pytest.mark.parametrize("N", [1000, 4096, 8192])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "bf16w32", "f16w32"])
def test_lowp_cast_order(N, dtype):
    """y rounds x*r to the I/O type before the weight multiply: nearly every
    element equals the oracle's emulation of that order bit for bit, and many
    elements differ from a single rounding of the exact product.  Where the
    device's fp32 rstd rounds differently from the oracle's, the rounded x*r
    moves by one unit in the last place, and the weight (up to ~1.5) carries
    that into at most two units of y."""
    w = _w(256, N, dtype, seed=N)
    inp = H.inputs_for(w)
    res = H.run_gpu(w, inp)
    x = storage_to_float64(inp["x"], w.dtype)
    g = storage_to_float64(inp["gamma"], w.wdtype)
    emu = orc.emulate_forward_lowp(x, g, w.eps, 0, w.dtype, w.wdtype)
    got = H.to_host64(res.y)
    same = np.mean(got == emu)
    assert same >= 0.999, same
    diff = got != emu
    step = 2.0 ** -6 if w.dtype == "bf16" else 2.0 ** -9  # two units in the last place, relative
    assert np.all(np.abs(got[diff] - emu[diff]) <= step * np.abs(emu[diff]))
    if not w.weight_dtype:  # with a float32 weight there is only one rounding
        exact, _ = orc.rms_forward(x, g, w.eps)
        once = torch.tensor(exact).float().to(H.tdtype(w.dtype)).double().numpy()
        assert np.mean(got != once) > 0.01


def test_gemma_equals_plain_with_shifted_weight_f32():
    w = _w(300, 1024, "f32", gemma=1, seed=5)
    inp = H.inputs_for(w)
    a = H.run_gpu(w, inp)
    shifted = dict(inp)
    shifted["gamma"] = (1.0 + inp["gamma"].astype(np.float32)).astype(np.float32)
    b = H.run_gpu(dataclasses.replace(w, gemma=0), shifted)
    assert torch.equal(a.y, b.y) and torch.equal(a.dx, b.dx) and torch.equal(a.dgamma, b.dgamma)


def test_printed_worked_examples_fp32():
    """The tutorial's hand-worked rows through the CUDA path."""
    x = torch.tensor([[3.0, 4.0]], device="cuda")
    y = torch.empty_like(x)
    r = torch.empty(1, device="cuda")
    for gamma, expect in (([1.0, 1.0], [0.848528, 1.131371]), ([2.0, 0.5], [1.697056, 0.565685])):
        g = torch.tensor(gamma, device="cuda")
        rms.rms_fwd(x, g, y, r, 1e-6)
        torch.cuda.synchronize()
        assert np.all(np.abs(y.cpu().numpy()[0] - expect) <= 5e-7 + 1e-6 * np.abs(expect))
    assert abs(r.item() - 0.282843) <= 5e-7
    g = torch.ones(2, device="cuda")
    rms.rms_fwd(x, g, y, r, 1e-6)
    dy = torch.tensor([[1.0, 2.0]], device="cuda")
    dx = torch.empty_like(x)
    dg = torch.empty(2, device="cuda")
    ws = torch.empty(rms.rms_bwd_workspace_size(1, 2), dtype=torch.uint8, device="cuda")
    rms.rms_bwd(dy, x, g, r, dx, dg, ws)
    torch.cuda.synchronize()
    assert np.all(np.abs(dx.cpu().numpy()[0] - [-0.090510, 0.067882]) <= 5e-7 + 1e-6)
    # 257 ones: divide by N = 257, not by a padded 512.
    ones = torch.ones(1, 257, device="cuda")
    y1 = torch.empty_like(ones)
    rms.rms_fwd(ones, torch.ones(257, device="cuda"), y1, r, 1e-6)
    torch.cuda.synchronize()
    assert torch.all((y1 - 0.9999995).abs() <= 5e-7)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_sum_not_mean_on_gpu(dtype):
    dt = H.tdtype(dtype)
    x = torch.ones(2, 8, device="cuda", dtype=dt)
    dy = torch.tensor([[1.0, 2.0] * 4, [3.0, 4.0] * 4], device="cuda", dtype=dt)
    g = torch.ones(8, device="cuda", dtype=dt)
    r = torch.ones(2, device="cuda")  # eps = 0 on rows of ones
    dx = torch.empty_like(x)
    dg = torch.empty(8, device="cuda")
    ws = torch.empty(rms.rms_bwd_workspace_size(2, 8), dtype=torch.uint8, device="cuda")
    rms.rms_bwd(dy, x, g, r, dx, dg, ws)
    torch.cuda.synchronize()
    assert dg.tolist() == [4.0, 6.0] * 4


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_edge_rows(dtype):
    dt = H.tdtype(dtype)
    eps = 1e-4
    x = torch.zeros(3, 64, device="cuda", dtype=dt)
    x[1] = torch.linspace(-2, 2, 64, device="cuda").to(dt)
    x[2, 5] = float("nan")
    g = torch.full((64,), 1.5, device="cuda", dtype=dt)
    y = torch.empty_like(x)
    r = torch.empty(3, device="cuda")
    rms.rms_fwd(x, g, y, r, eps)
    dy = torch.ones_like(x)
    dx = torch.empty_like(x)
    dg = torch.empty(64, device="cuda")
    ws = torch.empty(rms.rms_bwd_workspace_size(3, 64), dtype=torch.uint8, device="cuda")
    rms.rms_bwd(dy, x, g, r, dx, dg, ws)
    torch.cuda.synchronize()
    assert torch.all(y[0] == 0) and abs(r[0].item() - 100.0) < 1e-4
    assert torch.allclose(dx[0].float(), torch.full((64,), 150.0, device="cuda"), rtol=1e-2)
    assert torch.isnan(y[2]).all() and torch.isnan(r[2])
    # eps = 0 on a zero row: r = inf and y = NaN, no special case.
    rms.rms_fwd(x[:1].contiguous(), g, y[:1], r[:1], 0.0)
    torch.cuda.synchronize()
    assert torch.isinf(r[0]) and torch.isnan(y[0]).all()


def test_empty_batch():
    x = torch.empty(0, 128, device="cuda")
    g = torch.ones(128, device="cuda")
    rms.rms_fwd(x, g, torch.empty_like(x), torch.empty(0, device="cuda"))
    dg = torch.full((128,), 7.0, device="cuda")
    rms.rms_bwd(x, x, g, torch.empty(0, device="cuda"), torch.empty_like(x), dg,
                torch.empty(0, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert torch.all(dg == 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_misaligned_pointers_use_scalar_path(dtype):
    """Views offset by one element are legal inputs; a forced vector mapping
    refuses them instead of reading unaligned vectors."""
    w = _w(100, 1024, dtype, seed=9)
    inp = H.inputs_for(w)
    dt = H.tdtype(dtype)
    M, N = w.M, w.N
    xb = torch.empty(M * N + 1, dtype=dt, device="cuda")
    x = xb[1:].view(M, N)
    x.copy_(H.to_device(inp["x"], dtype))
    g = H.to_device(inp["gamma"], dtype)
    yb = torch.empty(M * N + 1, dtype=dt, device="cuda")
    y = yb[1:].view(M, N)
    r = torch.empty(M, device="cuda")
    with pytest.raises(rms.RmsError) as ei:
        rms.rms_fwd(x, g, y, r, w.eps, path="registers")
    assert ei.value.status == rms.RMS_ERR_ALIGNMENT
    rms.rms_fwd(x, g, y, r, w.eps)
    dy = H.to_device(inp["dy"], dtype)
    dx = torch.empty(M * N + 1, dtype=dt, device="cuda")[1:].view(M, N)
    dg = torch.empty(N, device="cuda")
    ws = torch.empty(rms.rms_bwd_workspace_size(M, N), dtype=torch.uint8, device="cuda")
    rms.rms_bwd(dy, x, g, r, dx, dg, ws)
    torch.cuda.synchronize()
    red = rms.rms_bwd_reduction(M, N, rms.dtype_code(x, g), 0, 0, "scalar")
    res = H.GpuResult(y, r, dx, dg, True, red)
    H.assert_parity(w, inp, res)


def test_workspace_checks():
    M, N = 4096, 1024
    x = torch.randn(M, N, device="cuda")
    g = torch.ones(N, device="cuda")
    r = torch.ones(M, device="cuda")
    need = rms.rms_bwd_workspace_size(M, N)
    assert need > 0 and need % 256 == 0
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(rms.RmsError) as ei:
        rms.rms_bwd(x, x.clone(), g, r, torch.empty_like(x), torch.empty(N, device="cuda"), small)
    assert ei.value.status == rms.RMS_ERR_WORKSPACE
    odd = torch.empty(need + 512, dtype=torch.uint8, device="cuda")[16:]
    with pytest.raises(rms.RmsError) as ei:
        rms.rms_bwd(x, x.clone(), g, r, torch.empty_like(x), torch.empty(N, device="cuda"), odd)
    assert ei.value.status == rms.RMS_ERR_WORKSPACE


def test_overlapping_outputs_rejected_on_device_buffers():
    M, N = 64, 256
    buf = torch.randn(2 * M * N, device="cuda")
    x = buf[: M * N].view(M, N)
    y = buf[M * N // 2: M * N // 2 + M * N].view(M, N)
    with pytest.raises(rms.RmsError) as ei:
        rms.rms_fwd(x, torch.ones(N, device="cuda"), y, torch.empty(M, device="cuda"))
    assert ei.value.status == rms.RMS_ERR_INVALID_ARG


def test_launch_count_and_status():
    before = rms.rms_launch_count()
    w = _w(64, 128, "f32")
    inp = H.inputs_for(w)
    H.run_gpu(w, inp)
    assert rms.rms_launch_count() - before == 3
    assert rms.rms_last_device_status() == rms.RMS_OK


@pytest.mark.parametrize("N", [8192, 16384])
def test_both_vector_mappings_on_wide_rows(N):
    """Rows of 16 and 32 KiB run through both the register and the staged
    mapping, each checked against the oracle."""
    w = _w(2048, N, "bf16", seed=N + 1)
    inp = H.inputs_for(w)
    for path in ("registers", "staged"):
        H.assert_parity(w, inp, H.run_gpu(w, inp, path=path), H.sample_rows(w.M, 64))


@pytest.mark.parametrize("dtype,N", [("bf16", 32768), ("bf16", 65536), ("bf16", 131072),
                                     ("bf16", 22024), ("f32", 16384), ("f32", 32768),
                                     ("f16", 32768)])
@pytest.mark.parametrize("gemma,inplace", [(0, 0), (1, 1)])
def test_cluster_split_rows(dtype, N, gemma, inplace):
    """Rows wider than one CTA's stages are split across a thread-block
    cluster (column slices, row sums exchanged through distributed shared
    memory).  N = 22024 bf16 gives slices of unequal length."""
    w = _w(48, N, dtype, gemma=gemma, inplace=inplace, seed=N + gemma)
    inp = H.inputs_for(w)
    H.assert_parity(w, inp, H.run_gpu(w, inp, path="staged"))


@pytest.mark.parametrize("bwd", [False, True])
@pytest.mark.parametrize("N", [4096, 65536])
def test_staged_wait_timeout_reports_status(bwd, N):
    """With the poll limit at 0 every staged wait gives up at once: the
    kernel drains its copies, raises the device status and returns; the
    host sees RMS_ERR_TIMEOUT and the context stays usable."""
    w = _w(600 if N <= 4096 else 40, N, "bf16", seed=11)
    inp = H.inputs_for(w)
    x = H.to_device(inp["x"], "bf16")
    g = H.to_device(inp["gamma"], "bf16")
    dy = H.to_device(inp["dy"], "bf16")
    y = torch.empty_like(x)
    r = torch.empty(w.M, device="cuda")
    dx = torch.empty_like(x)
    dg = torch.empty(w.N, device="cuda")
    ws = torch.empty(rms.rms_bwd_workspace_size(w.M, w.N), dtype=torch.uint8, device="cuda")
    rms.rms_fwd(x, g, y, r, w.eps, path="staged")
    torch.cuda.synchronize()
    assert rms.rms_last_device_status() == rms.RMS_OK
    prev = rms.rms_set_wait_limit(0)
    try:
        if bwd:
            rms.rms_bwd(dy, x, g, r, dx, dg, ws, path="staged")
        else:
            rms.rms_fwd(x, g, y, r, w.eps, path="staged")
        assert rms.rms_last_device_status() == rms.RMS_ERR_TIMEOUT
        assert rms.rms_last_device_status() == rms.RMS_OK  # cleared by the read
    finally:
        rms.rms_set_wait_limit(prev)
    H.assert_parity(w, inp, H.run_gpu(w, inp, path="staged"))


@pytest.mark.parametrize("N", [8192, 65536, 262144])
def test_chunked_exchange_wait_limit_reports_status(N):
    """One-pass chunked mapping with the poll limit at 0: every row-partial
    wait runs past the limit, so the kernels raise the device status, yet
    they wait the exchange out (bounded) instead of skipping a row: the
    outputs still match and the host reads RMS_ERR_TIMEOUT once."""
    w = _w(24, N, "bf16", seed=13)
    inp = H.inputs_for(w)
    prev = rms.rms_set_wait_limit(0)
    try:
        res = H.run_gpu(w, inp, path="chunked", expect_status=rms.RMS_ERR_TIMEOUT)
        assert rms.rms_last_device_status() == rms.RMS_OK  # cleared by the read
    finally:
        rms.rms_set_wait_limit(prev)
    H.assert_parity(w, inp, res)


def test_more_than_2_31_elements():
    """2,097,157 x 1024 bf16 (2^31 + 5120 elements per matrix): 64-bit
    indexing in every kernel.  Inputs are drawn on the device with a seeded
    torch generator; sampled rows (including the last ones) are copied back
    and checked against the oracle; dgamma is checked by additivity: the
    full-matrix result equals the sum of three row blocks' results."""
    from oracle import compare

    M, N = (1 << 21) + 5, 1024
    gen = torch.Generator(device="cuda").manual_seed(0)
    x = torch.randn(M, N, device="cuda", generator=gen).to(torch.bfloat16)
    dy = torch.randn(M, N, device="cuda", generator=gen).to(torch.bfloat16)
    g = (torch.rand(N, device="cuda", generator=gen) + 0.5).to(torch.bfloat16)
    y = torch.empty_like(x)
    r = torch.empty(M, device="cuda")
    dx = torch.empty_like(x)
    dg = torch.empty(N, device="cuda")
    ws = torch.empty(rms.rms_bwd_workspace_size(M, N), dtype=torch.uint8, device="cuda")
    eps = 1e-6
    rms.rms_fwd(x, g, y, r, eps)
    rms.rms_bwd(dy, x, g, r, dx, dg, ws)
    torch.cuda.synchronize()
    rows = torch.tensor([0, 1, 2097151, 2097152, 2097153, M - 2, M - 1] + list(range(1000, M, 99991)),
                        device="cuda")
    xs = H.to_host64(x.index_select(0, rows))
    dys = H.to_host64(dy.index_select(0, rows))
    gs = H.to_host64(g)
    y_ref, r_ref = orc.rms_forward(xs, gs, eps)
    dx_ref, _, dxs, _ = orc.rms_backward(xs, gs, dys, eps, with_scales=True)
    for c in (compare.check_y(H.to_host64(y.index_select(0, rows)), y_ref, "bf16"),
              compare.check_rstd(H.to_host64(r.index_select(0, rows)), r_ref),
              compare.check_dx(H.to_host64(dx.index_select(0, rows)), dx_ref, dxs, "bf16")):
        assert c.ok, str(c)
    parts = np.zeros(N)
    for a, b in ((0, 700001), (700001, 2097152), (2097152, M)):
        dgb = torch.empty(N, device="cuda")
        wsb = torch.empty(rms.rms_bwd_workspace_size(b - a, N), dtype=torch.uint8, device="cuda")
        rms.rms_bwd(dy[a:b], x[a:b], g, r[a:b], dx[a:b], dgb, wsb)
        torch.cuda.synchronize()
        parts += H.to_host64(dgb)
    full = H.to_host64(dg)
    assert np.all(np.abs(full - parts) <= 2e-5 * (np.abs(full) + np.sqrt(M))), np.abs(full - parts).max()


@pytest.mark.parametrize("N", [32768, 65536, 131072, 262144])
def test_widest_rows(N):
    """Wide bf16 rows in the automatic mapping: cluster split up to 128K
    (backward) / 256K (forward), the chunked mapping beyond."""
    w = _w(64, N, "bf16", seed=N)
    inp = H.inputs_for(w)
    H.assert_parity(w, inp, H.run_gpu(w, inp))


def test_chunked_many_short_rows():
    """Forced chunked mapping on many 16-byte rows (M > N): the one-pass
    cluster mapping keeps no per-row values in the workspace, so the shape
    the three-pass mapping had no room for runs."""
    M, N = 5000, 8
    w = _w(M, N, "bf16", seed=1)
    inp = H.inputs_for(w)
    H.assert_parity(w, inp, H.run_gpu(w, inp, fwd_path="chunked", bwd_path="chunked"))


@pytest.mark.parametrize("gemma,inplace", [(0, 0), (1, 1)])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "bf16w32"])
@pytest.mark.parametrize("M,N", [(257, 3072), (1000, 512), (3, 65536), (700, 8192), (37, 40960),
                                 (19, 131072)])
def test_chunked_mapping(M, N, dtype, gemma, inplace):
    """The chunked mapping forced on ordinary shapes: one-pass clusters of 1,
    2, 3, 4, 8 and 16 CTAs (N = 131072 f32), Gemma and in-place dx."""
    w = _w(M, N, dtype, gemma=gemma, inplace=inplace, seed=M * 7 + N)
    inp = H.inputs_for(w)
    H.assert_parity(w, inp, H.run_gpu(w, inp, path="chunked"))


@pytest.mark.parametrize("M,N", [(3000, 4096), (300, 65536), (40, 1 << 20)])
def test_chunked_dgamma_bitwise_reproducible(M, N):
    """Run to run: one CTA per row (N = 4096), a 4-CTA cluster (65536), the
    three-pass backward (2^20)."""
    w = _w(M, N, "bf16", seed=5)
    inp = H.inputs_for(w)
    a = H.run_gpu(w, inp, path="chunked")
    b = H.run_gpu(w, inp, path="chunked")
    assert torch.equal(a.dgamma.view(torch.int32), b.dgamma.view(torch.int32))
    assert torch.equal(a.dx.view(torch.int16), b.dx.view(torch.int16))


@pytest.mark.parametrize("dtype,N,M", [("bf16", 262144, 48), ("f32", 200000, 12),
                                       ("bf16", 1 << 20, 6), ("f16", 393216, 9),
                                       ("f32", 600000, 3)])
def test_rows_beyond_the_cluster_split(dtype, N, M):
    """Rows wider than the staged cluster split holds take the chunked
    mapping automatically: one pass in a cluster of up to 16 CTAs (forward
    rows up to 2 MiB, backward up to 512 KiB), three passes beyond (the
    backward from 200000 f32 / 393216 f16 / 2^20 bf16 here, the forward at
    600000 f32)."""
    w = _w(M, N, dtype, seed=N % 1000 + M)
    inp = H.inputs_for(w)
    H.assert_parity(w, inp, H.run_gpu(w, inp))


@pytest.mark.parametrize("dtype,N", [("f32", 70001), ("bf16", 120003)])
def test_misaligned_wide_rows_scalar_workspace_partials(dtype, N):
    """Rows whose dgamma partials do not fit in shared memory, on the scalar
    mapping (N*b not a multiple of 16): the partials live in the workspace."""
    w = _w(9, N, dtype, seed=N % 977)
    inp = H.inputs_for(w)
    H.assert_parity(w, inp, H.run_gpu(w, inp))
