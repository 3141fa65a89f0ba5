"""The row-sharded backward's exchange step on one GPU: rms_dgamma_combine
adds per-rank vectors in rank order (bit for bit the sequential float32
sum), and two row blocks run separately and combined give dgamma within the
oracle's bars, bit for bit the same from run to run."""
import numpy as np
import pytest
import torch

from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import row_wise_normalization_rms_gb300 as rms
    from oracle import compare
    from row_wise_normalization_rms_gb300.sharded import row_block
    from synthetic import WORKLOADS


@pytest.mark.parametrize("R,N", [(1, 8), (2, 8192), (3, 1000), (8, 4096), (5, 3)])
def test_combine_is_the_rank_order_float32_sum(R, N):
    gen = torch.Generator().manual_seed(R * 1000 + N)
    parts = torch.randn(R, N, generator=gen) * torch.exp(torch.empty(R, N).uniform_(-12, 12,
                                                                                generator=gen))
    expect = parts[0].clone()
    for r in range(1, R):
        expect = expect + parts[r]  # IEEE float32 on the host, one rounding each
    out = torch.full((N,), float("nan"), device="cuda")
    rms.rms_dgamma_combine(parts.cuda(), out)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu().view(torch.int32), expect.view(torch.int32))
    # an unaligned output and an odd column count take the scalar loop
    buf = torch.full((N + 1,), float("nan"), device="cuda")
    rms.rms_dgamma_combine(parts.cuda(), buf[1:])
    torch.cuda.synchronize()
    assert torch.equal(buf[1:].cpu().view(torch.int32), expect.view(torch.int32))


def _sharded_dgamma(w, inp, world):
    """dgamma of the whole batch from ``world`` row blocks run one after the
    other on this GPU, then combined in rank order; the deepest block's
    reduction and the blocks' dx."""
    x = H.to_device(inp["x"], w.dtype)
    g = H.to_device(inp["gamma"], w.wdtype)
    dy = H.to_device(inp["dy"], w.dtype)
    y, dx = torch.empty_like(x), torch.empty_like(x)
    rstd = torch.empty(w.M, device="cuda")
    parts = torch.empty(world, w.N, device="cuda")
    depth = (0, 0)
    for r in range(world):
        lo, hi = row_block(w.M, world, r)
        ws = torch.empty(max(256, rms.rms_bwd_workspace_size(hi - lo, w.N)), dtype=torch.uint8,
                         device="cuda")
        rms.rms_fwd(x[lo:hi], g, y[lo:hi], rstd[lo:hi], w.eps, w.gemma)
        rms.rms_bwd(dy[lo:hi], x[lo:hi], g, rstd[lo:hi], dx[lo:hi], parts[r], ws, w.gemma)
        red = rms.rms_bwd_reduction(hi - lo, w.N, rms.dtype_code(x, g), w.gemma)
        depth = max(depth, red, key=lambda t: t[0] + t[1])
    dg = torch.full((w.N,), float("nan"), device="cuda")
    rms.rms_dgamma_combine(parts, dg)
    torch.cuda.synchronize()
    # the combine adds `world` more values per column after the deepest block
    return y, rstd, dx, dg, (depth[0] + world, depth[1])


@pytest.mark.parametrize("name,world", [("llama7b_bf16_8192x4096", 2),
                                        ("llama7b_bf16_8192x4096", 3),
                                        ("tiny_f32_64x128", 4)])
def test_row_blocks_combined_match_the_oracle(name, world):
    w = WORKLOADS[name]
    inp = H.inputs_for(w)
    y, rstd, dx, dg, red = _sharded_dgamma(w, inp, world)
    res = H.GpuResult(y, rstd, dx, dg, True, red)
    H.assert_parity(w, inp, res, None if w.M <= 64 else H.sample_rows(w.M))
    _, _, _, dg2, _ = _sharded_dgamma(w, inp, world)
    assert torch.equal(dg.view(torch.int32), dg2.view(torch.int32))
    assert rms.rms_last_device_status() == rms.RMS_OK
