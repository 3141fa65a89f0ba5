"""RMSNorm forward quantised to FP8 E4M3 (rms_fwd_quant) against the fp64
oracle through the C ABI, and against the unfused composition on the GPU
(rms_fwd, then torch's float8 conversion of y * (448 / amax)) bit for bit."""
import numpy as np
import pytest
import torch

from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import row_wise_normalization_rms_gb300 as rms
    from oracle import rmsnorm_oracle as orc
    from synthetic import WORKLOADS, storage_to_float64

# the stored y may differ from the emulation by up to two units in its last place (rstd
# rounding), and the scale rounds once more: allow two units of the I/O type, three for f32
SCALE_TOL = {"bf16": 2 * 2.0 ** -8, "f16": 2 * 2.0 ** -11, "f32": 3 * 2.0 ** -23}


def _qw(M, N, dtype, gemma=0, seed=0):
    from synthetic import Workload

    wd = ""
    if dtype.endswith("w32"):
        dtype, wd = dtype[:-3], "f32"
    return Workload(name=f"q{M}x{N}_{dtype}{wd}_g{gemma}", M=M, N=N, dtype=dtype, eps=1e-6,
                    gemma=gemma, seed=seed, weight_dtype=wd,
                    gamma=("normal", 0.0, 0.1) if gemma else ("uniform", 0.5, 1.5),
                    row_scale=("loguniform", 0.01, 100.0))


def run_quant(w, inp, path="auto", x=None):
    x = H.to_device(inp["x"], w.dtype) if x is None else x
    g = H.to_device(inp["gamma"], w.wdtype)
    q = torch.empty(w.M, w.N, dtype=torch.uint8, device="cuda")
    s = torch.empty(w.M, device="cuda")
    r = torch.empty(w.M, device="cuda")
    rms.rms_fwd_quant(x, g, q, s, r, w.eps, w.gemma, path=path)
    torch.cuda.synchronize()
    return q, s, r


def assert_quant_parity(w, inp, q, s, r, rows=None):
    """rstd, the per-row scale and the codes against the oracle, block by
    block over ``rows`` (every row when None)."""
    g = storage_to_float64(inp["gamma"], w.wdtype)
    n_same = n_all = 0
    for blk in H.row_blocks(w.M, w.N, rows):
        x = storage_to_float64(inp["x"][blk], w.dtype)
        q_ref, s_ref, r_ref = orc.rms_forward_quant(x, g, w.eps, w.gemma, w.dtype, w.wdtype)
        idx = torch.as_tensor(blk, device="cuda")
        qb = q.index_select(0, idx).cpu().numpy()
        qv = torch.from_numpy(qb).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        sg = s.index_select(0, idx).cpu().numpy().astype(np.float64)
        rg = r.index_select(0, idx).cpu().numpy().astype(np.float64)
        assert np.all(np.abs(rg - r_ref) <= 1e-6 * r_ref), "rstd"
        assert np.all(np.abs(sg - s_ref) <= SCALE_TOL[w.dtype] * s_ref), "scale"
        n_same += int(np.sum(qb == orc.e4m3_code(q_ref)))
        n_all += qb.size
        # the rest within one step of the E4M3 ladder at that magnitude
        _, ex = np.frexp(np.maximum(np.abs(q_ref), 2.0 ** -6))
        step = np.ldexp(1.0, ex - 1 - 3)
        assert np.all(np.abs(qv - q_ref) <= step * (1 + 1e-9)), "a code more than one step off"
    same = n_same / max(1, n_all)
    assert same >= 0.999, f"only {same:.5f} of the codes equal the oracle's"


SHAPES = [(1, 8), (3, 64), (17, 128), (64, 1000), (33, 1024), (65, 4096), (9, 8192), (4, 16384),
          (2, 5000), (31, 257), (3, 32768), (2, 40008), (2, 70000)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "bf16w32"])
@pytest.mark.parametrize("M,N", SHAPES, ids=[f"{m}x{n}" for m, n in SHAPES])
@pytest.mark.parametrize("path", ["auto", "registers", "chunked", "scalar"])
@pytest.mark.parametrize("gemma", [0, 1])
def test_quant_parity(M, N, dtype, path, gemma):
    w = _qw(M, N, dtype, gemma=gemma, seed=M + N)
    inp = H.inputs_for(w)
    aligned = (N * w.elem_bytes) % 16 == 0
    if (path == "registers" and (not aligned or N * w.elem_bytes > 32768)) or (
            path == "chunked" and not aligned):
        with pytest.raises(rms.RmsError) as ei:
            run_quant(w, inp, path)
        assert ei.value.status in (rms.RMS_ERR_ALIGNMENT, rms.RMS_ERR_UNSUPPORTED)
        return
    assert_quant_parity(w, inp, *run_quant(w, inp, path))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("path", ["registers", "scalar"])
@pytest.mark.parametrize("N", [4096, 4104, 8192])
def test_quant_equals_unfused_composition(dtype, path, N):
    """Codes and scales equal, bit for bit, rms_fwd on the same mapping followed
    by the quantisation in torch: y * (448 / amax) in float32, then float8.
    Rows of more than 512 vectors run with half the register forward's
    threads, each holding two threads' vectors (4104 bf16: three warps
    standing for five), and must still sum in its order."""
    w = _qw(500, N, dtype, seed=4)
    inp = H.inputs_for(w)
    q, s, r = run_quant(w, inp, path)
    x = H.to_device(inp["x"], dtype)
    g = H.to_device(inp["gamma"], dtype)
    y = torch.empty_like(x)
    r2 = torch.empty(w.M, device="cuda")
    rms.rms_fwd(x, g, y, r2, w.eps, path=path)
    yf = y.float()
    amax = yf.abs().amax(dim=1)
    inv = torch.tensor(448.0, device="cuda") / amax
    codes = (yf * inv[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(r, r2)
    assert torch.equal(s, amax / torch.tensor(448.0, device="cuda"))
    assert torch.equal(q, codes)


def test_quant_edge_rows():
    w = _qw(6, 1024, "bf16", seed=2)
    inp = H.inputs_for(w)
    x = inp["x"].copy()
    x[0] = 0
    x[1] = 0
    x[1, 7] = np.uint16(0x3F80)  # one nonzero element: its code is the largest
    inp = dict(inp, x=x)
    for path in ("registers", "chunked", "scalar"):
        q, s, r = run_quant(w, inp, path)
        assert float(s[0]) == 1.0 and int(q[0].abs().sum()) == 0
        assert int(q[1, 7]) == 0x7E and int((q[1] != 0).sum()) == 1
        assert_quant_parity(w, inp, q, s, r)


def test_quant_misaligned_uses_scalar():
    w = _qw(50, 1024, "bf16", seed=6)
    inp = H.inputs_for(w)
    xb = torch.empty(w.M * w.N + 1, dtype=torch.bfloat16, device="cuda")
    x = xb[1:].view(w.M, w.N)
    x.copy_(H.to_device(inp["x"], "bf16"))
    with pytest.raises(rms.RmsError) as ei:
        run_quant(w, inp, "registers", x=x)
    assert ei.value.status == rms.RMS_ERR_ALIGNMENT
    assert_quant_parity(w, inp, *run_quant(w, inp, "auto", x=x))


def test_quant_full_size_headline_shape():
    w = WORKLOADS["wide_bf16_16384x8192"]
    inp = H.inputs_for(w)
    q, s, r = run_quant(w, inp)
    assert_quant_parity(w, inp, q, s, r)  # every row


def test_quant_full_size_wide_rows():
    """Rows of 128 KiB (too wide for the register mapping) at 256 MiB of x."""
    w = WORKLOADS["quant_widerows_bf16_N65536"]
    inp = H.inputs_for(w)
    q, s, r = run_quant(w, inp)
    assert_quant_parity(w, inp, q, s, r)  # every row


@pytest.mark.parametrize("dtype,N,M", [("bf16", 65536, 37), ("bf16", 262144, 9), ("f16", 98304, 11),
                                       ("f32", 65536, 13), ("bf16w32", 131072, 7)])
@pytest.mark.parametrize("path", ["auto", "chunked"])
def test_quant_cluster_mapping(dtype, N, M, path):
    """Rows of 64 KiB to 512 KiB: a cluster of 2 to 16 CTAs per row, one read
    of x, the sum of squares and the maximum |y| exchanged between the CTAs."""
    w = _qw(M, N, dtype, seed=N % 991 + M)
    inp = H.inputs_for(w)
    assert_quant_parity(w, inp, *run_quant(w, inp, path))
    assert rms.rms_last_device_status() == rms.RMS_OK


@pytest.mark.parametrize("dtype,N", [("bf16", 1 << 19), ("f32", 270000)])
def test_quant_rows_beyond_the_cluster(dtype, N):
    """Rows needing more than 16 slices of 32 KiB (1 MiB bf16, 1.03 MiB f32)
    fall back to a CTA per row walking the row three times."""
    w = _qw(3, N, dtype, seed=7)
    inp = H.inputs_for(w)
    for path in ("auto", "chunked"):
        assert_quant_parity(w, inp, *run_quant(w, inp, path))


def test_quant_cluster_exchange_wait_limit_reports_status():
    """The cluster mapping with the poll limit at 0: every exchange wait runs
    past the limit, so the kernel raises the device status but still waits
    each exchange out (bounded); the codes still match and the host reads
    RMS_ERR_TIMEOUT once."""
    w = _qw(20, 65536, "bf16", seed=21)
    inp = H.inputs_for(w)
    prev = rms.rms_set_wait_limit(0)
    try:
        q, s, r = run_quant(w, inp, "chunked")
        assert rms.rms_last_device_status() == rms.RMS_ERR_TIMEOUT
        assert rms.rms_last_device_status() == rms.RMS_OK  # cleared by the read
    finally:
        rms.rms_set_wait_limit(prev)
    assert_quant_parity(w, inp, q, s, r)
