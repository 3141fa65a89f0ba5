"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs and compare with the fp64 oracle on the same inputs."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import row_wise_normalization_rms_gb300 as rms
from oracle import compare
from oracle import layernorm_oracle as lno
from oracle import rmsnorm_oracle as orc
from synthetic import make_inputs, storage_to_float64

PAD = 64  # guard elements on each side of every output buffer
_SENTINEL = {"bf16": 0x7FC1, "f16": 0x7E01, "f32": 0x7FC00001}  # NaN payloads nothing else writes


def tdtype(dtype: str):
    return {"bf16": torch.bfloat16, "f16": torch.float16}.get(dtype, torch.float32)


def to_device(arr: np.ndarray, dtype: str) -> torch.Tensor:
    a = np.ascontiguousarray(arr)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()  # float32 or float16 arrays map directly


def to_host64(t: torch.Tensor) -> np.ndarray:
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


class Guarded:
    """A device tensor with sentinel-filled guard regions on both sides."""

    def __init__(self, shape, torch_dtype, sentinel_bits: int):
        n = int(np.prod(shape)) if len(shape) else 1
        self.bits_dtype = torch.int32 if torch_dtype == torch.float32 else torch.int16
        self.buf = torch.empty(n + 2 * PAD, dtype=torch_dtype, device="cuda")
        # the sentinels are positive in their signed view (0x7FC1, 0x7E01, 0x7FC00001)
        self.buf.view(self.bits_dtype).fill_(sentinel_bits)
        self.sentinel = sentinel_bits
        self.t = self.buf[PAD:PAD + n].view(*shape)

    def guards_intact(self) -> bool:
        b = self.buf.view(self.bits_dtype)
        return bool((b[:PAD] == self.sentinel).all() and (b[-PAD:] == self.sentinel).all())


@dataclass
class GpuResult:
    y: torch.Tensor
    rstd: torch.Tensor
    dx: torch.Tensor
    dgamma: torch.Tensor
    guards_ok: bool
    reduction: tuple  # (partials, rows_per_partial) of the backward's dgamma sum


def run_gpu(w, inp, path="auto", inplace=None, fwd_path=None, bwd_path=None,
            expect_status=None) -> GpuResult:
    """Forward then backward through the C ABI on device copies of ``inp``;
    the device status word read afterwards must be ``expect_status``
    (RMS_OK unless given)."""
    dt = tdtype(w.dtype)
    M, N = w.M, w.N
    inplace = w.inplace_dx if inplace is None else inplace
    x = to_device(inp["x"], w.dtype)
    g = to_device(inp["gamma"], w.wdtype)
    dy = to_device(inp["dy"], w.dtype)
    y = Guarded((M, N), dt, _SENTINEL[w.dtype])
    rstd = Guarded((M,), torch.float32, _SENTINEL["f32"])
    dg = Guarded((N,), torch.float32, _SENTINEL["f32"])
    dx = None if inplace else Guarded((M, N), dt, _SENTINEL[w.dtype])
    ws_bytes = rms.rms_bwd_workspace_size(M, N)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    rms.rms_fwd(x, g, y.t, rstd.t, w.eps, w.gemma, path=fwd_path or path)
    rms.rms_bwd(dy, x, g, rstd.t, None if inplace else dx.t, dg.t, ws, w.gemma, inplace,
                path=bwd_path or path)
    torch.cuda.synchronize()
    st = rms.rms_last_device_status()
    assert st == (rms.RMS_OK if expect_status is None else expect_status), st
    guards = y.guards_intact() and rstd.guards_intact() and dg.guards_intact() and (
        inplace or dx.guards_intact())
    red = rms.rms_bwd_reduction(M, N, rms.dtype_code(x, g), w.gemma, 0, bwd_path or path)
    return GpuResult(y.t, rstd.t, dy if inplace else dx.t, dg.t, guards, red)


def oracle_rows(w, inp, rows):
    """Oracle y, r, dx and the dx tolerance scale for the given rows."""
    x = storage_to_float64(inp["x"][rows], w.dtype)
    g = storage_to_float64(inp["gamma"], w.wdtype)
    dy = storage_to_float64(inp["dy"][rows], w.dtype)
    y, r = orc.rms_forward(x, g, w.eps, w.gemma)
    dx, _, dxs, _ = orc.rms_backward(x, g, dy, w.eps, w.gemma, with_scales=True)
    return y, r, dx, dxs


def oracle_dgamma(w, inp, block_rows: int = 1024):
    """Oracle dgamma over all M rows; the test sums it over row blocks to
    bound host memory (each block is the oracle's plain column sum)."""
    N = w.N
    total = np.zeros(N)
    scale = np.zeros(N)
    for r0 in range(0, w.M, block_rows):
        r1 = min(w.M, r0 + block_rows)
        x = storage_to_float64(inp["x"][r0:r1], w.dtype)
        dy = storage_to_float64(inp["dy"][r0:r1], w.dtype)
        d, s = orc.rms_dgamma(x, dy, w.eps, with_scales=True)
        total += d
        scale += s
    return total, scale


def sample_rows(M: int, n: int = 48, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    rows = set(np.linspace(0, M - 1, num=min(M, n // 2), dtype=np.int64).tolist())
    rows.update(rng.integers(0, M, size=min(M, n // 2)).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def row_blocks(M: int, N: int, rows=None, elems: int = 1 << 22):
    """The rows to compare (all when ``rows`` is None), in blocks of about
    ``elems`` elements so that the fp64 oracle's arrays stay small."""
    rows = np.arange(M, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
    step = max(1, elems // max(1, N))
    return [rows[i:i + step] for i in range(0, rows.size, step)]


def _take(t: torch.Tensor, rows: np.ndarray) -> np.ndarray:
    """Host float64 copy of the given rows of a device tensor."""
    if rows.size and rows[-1] - rows[0] + 1 == rows.size:  # contiguous block: a plain slice
        return to_host64(t[int(rows[0]):int(rows[-1]) + 1])
    return to_host64(t.index_select(0, torch.as_tensor(rows, device=t.device)))


def check_against_oracle(w, inp, res: GpuResult, rows=None):
    """All tolerance checks; ``rows`` None compares every row (block by block)."""
    parts = {"y": [], "rstd": [], "dx": []}
    for blk in row_blocks(w.M, w.N, rows):
        y_ref, r_ref, dx_ref, dxs = oracle_rows(w, inp, blk)
        parts["y"].append(compare.check_y(_take(res.y, blk), y_ref, w.dtype))
        parts["rstd"].append(compare.check_rstd(_take(res.rstd, blk), r_ref))
        parts["dx"].append(compare.check_dx(_take(res.dx, blk), dx_ref, dxs, w.dtype))
    dg_ref, dgs = oracle_dgamma(w, inp)
    checks = [compare.merge(parts[k]) for k in ("y", "rstd", "dx")]
    checks += compare.dgamma_checks(to_host64(res.dgamma), dg_ref, dgs, w.dtype, res.reduction)
    return checks


def assert_parity(w, inp, res: GpuResult, rows=None):
    assert res.guards_ok, "a kernel wrote outside its output buffer"
    checks = check_against_oracle(w, inp, res, rows)
    bad = [str(c) for c in checks if not c.ok]
    assert not bad, f"{w.name}: " + "; ".join(bad)
    return checks


def inputs_for(w):
    return make_inputs(w)


# ---------------------------------------------------------------- LayerNorm


@dataclass
class LnResult:
    y: torch.Tensor
    mean: torch.Tensor
    rstd: torch.Tensor
    dx: torch.Tensor
    dw: torch.Tensor
    db: "torch.Tensor | None"
    guards_ok: bool
    reduction: tuple  # (partials, rows_per_partial) of the dw and db sums


def run_ln(w, inp, path="auto", inplace=None, fwd_path=None, bwd_path=None, with_db=True,
           bias=True) -> LnResult:
    """LayerNorm forward then backward through the C ABI on device copies of ``inp``."""
    dt = tdtype(w.dtype)
    M, N = w.M, w.N
    inplace = w.inplace_dx if inplace is None else inplace
    x = to_device(inp["x"], w.dtype)
    g = to_device(inp["gamma"], w.wdtype)
    b = to_device(inp["beta"], w.wdtype) if (bias and inp["beta"] is not None) else None
    dy = to_device(inp["dy"], w.dtype)
    y = Guarded((M, N), dt, _SENTINEL[w.dtype])
    mean = Guarded((M,), torch.float32, _SENTINEL["f32"])
    rstd = Guarded((M,), torch.float32, _SENTINEL["f32"])
    dw = Guarded((N,), torch.float32, _SENTINEL["f32"])
    db = Guarded((N,), torch.float32, _SENTINEL["f32"])
    dx = None if inplace else Guarded((M, N), dt, _SENTINEL[w.dtype])
    ws = torch.empty(max(rms.ln_bwd_workspace_size(M, N), 256), dtype=torch.uint8, device="cuda")
    rms.ln_fwd(x, g, b, y.t, mean.t, rstd.t, w.eps, path=fwd_path or path)
    rms.ln_bwd(dy, x, g, mean.t, rstd.t, None if inplace else dx.t, dw.t,
               db.t if with_db else None, ws, inplace, path=bwd_path or path)
    torch.cuda.synchronize()
    assert rms.rms_last_device_status() == rms.RMS_OK
    guards = all(t.guards_intact() for t in (y, mean, rstd, dw, db)) and (
        inplace or dx.guards_intact())
    if not with_db:  # db must be untouched
        guards = guards and bool((db.t.view(torch.int32) == _SENTINEL["f32"]).all())
    red = rms.ln_bwd_reduction(M, N, rms.dtype_code(x, g), bwd_path or path)
    return LnResult(y.t, mean.t, rstd.t, dy if inplace else dx.t, dw.t,
                    db.t if with_db else None, guards, red)


def ln_oracle_rows(w, inp, rows, bias=True):
    x = storage_to_float64(inp["x"][rows], w.dtype)
    g = storage_to_float64(inp["gamma"], w.wdtype)
    b = storage_to_float64(inp["beta"], w.wdtype) if (bias and inp["beta"] is not None) else None
    dy = storage_to_float64(inp["dy"][rows], w.dtype)
    y, mean, rstd, ys, am = lno.ln_forward(x, g, b, w.eps, with_scales=True)
    dx, _, _, dxs, _, _ = lno.ln_backward(x, g, dy, w.eps, with_scales=True)
    return y, mean, rstd, ys, am, dx, dxs


def ln_oracle_wsums(w, inp, block_rows: int = 1024):
    """Oracle dw and db with their tolerance scales (dw_scale, db_scale, and
    the tight bar's dw_abs, dw_stat) over all M rows, summed over row blocks
    to bound host memory (each block is the oracle's column sum)."""
    N = w.N
    g = storage_to_float64(inp["gamma"], w.wdtype)
    acc = [np.zeros(N) for _ in range(6)]
    for r0 in range(0, w.M, block_rows):
        r1 = min(w.M, r0 + block_rows)
        x = storage_to_float64(inp["x"][r0:r1], w.dtype)
        dy = storage_to_float64(inp["dy"][r0:r1], w.dtype)
        _, dw, db, _, dws, dbs = lno.ln_backward(x, g, dy, w.eps, with_scales=True)
        wa, wst = lno.ln_wsum_term_scales(x, dy, w.eps)
        for a, v in zip(acc, (dw, db, dws, dbs, wa, wst)):
            a += v
    return tuple(acc)


def ln_checks(w, inp, res: LnResult, rows=None, bias=True):
    parts = {k: [] for k in ("y", "mean", "rstd", "dx")}
    for blk in row_blocks(w.M, w.N, rows):
        y, mean, rstd, ys, am, dx, dxs = ln_oracle_rows(w, inp, blk, bias)
        parts["y"].append(compare.check_ln_y(_take(res.y, blk), y, ys, w.dtype))
        parts["mean"].append(compare.check_ln_mean(_take(res.mean, blk), mean, am))
        parts["rstd"].append(compare.check_ln_rstd(_take(res.rstd, blk), rstd))
        parts["dx"].append(compare.check_ln_dx(_take(res.dx, blk), dx, dxs, w.dtype))
    dw, db, dws, dbs, wa, wst = ln_oracle_wsums(w, inp)
    checks = [compare.merge(parts[k]) for k in ("y", "mean", "rstd", "dx")]
    checks += compare.ln_wsum_checks(
        to_host64(res.dw), dw, dws, wa, wst,
        to_host64(res.db) if res.db is not None else None, db, dbs, w.dtype, res.reduction)
    return checks


def assert_ln_parity(w, inp, res: LnResult, rows=None, bias=True):
    assert res.guards_ok, "a kernel wrote outside its output buffer"
    checks = ln_checks(w, inp, res, rows, bias)
    bad = [str(c) for c in checks if not c.ok]
    assert not bad, f"{w.name}: " + "; ".join(bad)
    return checks


# ------------------------------------------------------- fused residual add


@dataclass
class AddResult:
    y: torch.Tensor
    rstd: torch.Tensor
    h: torch.Tensor
    dx: torch.Tensor
    dgamma: torch.Tensor
    guards_ok: bool
    reduction: tuple  # (partials, rows_per_partial) of the dgamma sum


def run_fused(w, inp, path="auto", fwd_path=None, bwd_path=None, h_alias=False, dx_alias="none",
              inplace=None) -> AddResult:
    """rms_fwd_add then rms_bwd_add through the C ABI.  ``h_alias``: h is
    written over the residual buffer; ``dx_alias``: "dh" (dx accumulated
    into dh), "dy" (in place into dy) or "none"."""
    dt = tdtype(w.dtype)
    M, N = w.M, w.N
    x = to_device(inp["x"], w.dtype)
    g = to_device(inp["gamma"], w.wdtype)
    dy = to_device(inp["dy"], w.dtype)
    res = to_device(inp["residual"], w.dtype)
    dh = to_device(inp["dh"], w.dtype)
    y = Guarded((M, N), dt, _SENTINEL[w.dtype])
    rstd = Guarded((M,), torch.float32, _SENTINEL["f32"])
    dg = Guarded((N,), torch.float32, _SENTINEL["f32"])
    hbuf = None if h_alias else Guarded((M, N), dt, _SENTINEL[w.dtype])
    h = res if h_alias else hbuf.t
    dxbuf = Guarded((M, N), dt, _SENTINEL[w.dtype]) if dx_alias == "none" else None
    ws = torch.empty(max(rms.rms_bwd_workspace_size(M, N), 256), dtype=torch.uint8, device="cuda")
    rms.rms_fwd_add(x, res, g, y.t, h, rstd.t, w.eps, w.gemma, path=fwd_path or path)
    if dx_alias == "dy":
        rms.rms_bwd_add(dy, h, g, rstd.t, dh, None, dg.t, ws, w.gemma, 1, path=bwd_path or path)
        dx = dy
    elif dx_alias == "dh":
        rms.rms_bwd_add(dy, h, g, rstd.t, dh, dh, dg.t, ws, w.gemma, 0, path=bwd_path or path)
        dx = dh
    else:
        rms.rms_bwd_add(dy, h, g, rstd.t, dh, dxbuf.t, dg.t, ws, w.gemma, 0, path=bwd_path or path)
        dx = dxbuf.t
    torch.cuda.synchronize()
    assert rms.rms_last_device_status() == rms.RMS_OK
    guards = y.guards_intact() and rstd.guards_intact() and dg.guards_intact() and (
        h_alias or hbuf.guards_intact()) and (dx_alias != "none" or dxbuf.guards_intact())
    red = rms.rms_bwd_reduction(M, N, rms.dtype_code(x, g), w.gemma, 1, bwd_path or path)
    return AddResult(y.t, rstd.t, h, dx, dg.t, guards, red)


def fused_checks(w, inp, res: AddResult, rows=None):
    """h bit-for-bit against the oracle's stored sum; y, rstd, dx, dgamma
    within the bars, with the oracle evaluated on that h (row blocks; all
    rows when ``rows`` is None)."""
    g = storage_to_float64(inp["gamma"], w.wdtype)
    h_bad = 0
    parts = {"y": [], "rstd": [], "dx": []}
    for blk in row_blocks(w.M, w.N, rows):
        x = storage_to_float64(inp["x"][blk], w.dtype)
        r_in = storage_to_float64(inp["residual"][blk], w.dtype)
        dy = storage_to_float64(inp["dy"][blk], w.dtype)
        dh = storage_to_float64(inp["dh"][blk], w.dtype)
        y_ref, r_ref, h_ref = orc.rms_forward_add(x, r_in, g, w.eps, w.gemma, w.dtype)
        dx_ref, _, dxs, _ = orc.rms_backward_add(h_ref, g, dy, dh, w.eps, w.gemma,
                                                 with_scales=True)
        h_bad += int(np.sum(_take(res.h, blk) != h_ref))
        parts["y"].append(compare.check_y(_take(res.y, blk), y_ref, w.dtype))
        parts["rstd"].append(compare.check_rstd(_take(res.rstd, blk), r_ref))
        parts["dx"].append(compare.check_dx(_take(res.dx, blk), dx_ref, dxs, w.dtype))
    checks = [compare.merge(parts[k]) for k in ("y", "rstd", "dx")]
    # dgamma over all rows, on the oracle's h
    total = np.zeros(w.N)
    scale = np.zeros(w.N)
    for r0 in range(0, w.M, 1024):
        r1 = min(w.M, r0 + 1024)
        hh = orc.residual_add(storage_to_float64(inp["x"][r0:r1], w.dtype),
                              storage_to_float64(inp["residual"][r0:r1], w.dtype), w.dtype)
        d, sc = orc.rms_dgamma(hh, storage_to_float64(inp["dy"][r0:r1], w.dtype), w.eps,
                               with_scales=True)
        total += d
        scale += sc
    checks += compare.dgamma_checks(to_host64(res.dgamma), total, scale, w.dtype, res.reduction)
    return h_bad, checks


def assert_fused_parity(w, inp, res: AddResult, rows=None):
    assert res.guards_ok, "a kernel wrote outside its output buffer"
    h_bad, checks = fused_checks(w, inp, res, rows)
    assert h_bad == 0, f"{w.name}: {h_bad} elements of h differ from the stored sum"
    bad = [str(c) for c in checks if not c.ok]
    assert not bad, f"{w.name}: " + "; ".join(bad)
