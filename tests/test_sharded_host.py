"""The row-sharded path's host logic without a GPU: the row partition, and
the dgamma exchange over gloo at world sizes 2 and 3 (the per-rank vectors
gathered in rank order on every rank, then added in that order)."""
import os
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_row_blocks_cover_every_row_once():
    from row_wise_normalization_rms_gb300.sharded import row_block

    for M in (0, 1, 7, 16384, 16387):
        for world in (1, 2, 3, 8):
            blocks = [row_block(M, world, r) for r in range(world)]
            assert blocks[0][0] == 0 and blocks[-1][1] == M
            for (a0, a1), (b0, b1) in zip(blocks, blocks[1:]):
                assert a1 == b0  # contiguous, in rank order
            sizes = [b - a for a, b in blocks]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        row_block(10, 2, 2)


def _local_vector(rank, N=64):
    """Rank r's float32 vector: values of very different sizes, so that the
    order of the additions shows in the last bits."""
    rng = np.random.default_rng(100 + rank)
    v = rng.standard_normal(N) * np.exp(rng.uniform(-12, 12, N))
    return torch.tensor(v, dtype=torch.float32)


def _sequential(stacked, out):
    acc = stacked[0].clone()
    for r in range(1, stacked.shape[0]):
        acc = acc + stacked[r]  # float32 IEEE addition, one rounding each
    out.copy_(acc)


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    from row_wise_normalization_rms_gb300 import sharded

    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = _local_vector(rank)
    stacked = sharded.gather_rank_ordered(local)
    total = torch.empty_like(local)
    sharded.exchange_dgamma(local, total, combine=_sequential)
    # the product path has no CPU fallback: CPU tensors are refused
    refused = False
    try:
        sharded.exchange_dgamma(local, torch.empty_like(local))
    except (ValueError, RuntimeError):
        refused = True
    out[rank] = (stacked.numpy().tobytes(), total.numpy().tobytes(), refused)
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_dgamma_exchange_gloo_is_rank_ordered(world):
    port = 29700 + os.getpid() % 1000 + 10 * world
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    expect_stack = torch.stack([_local_vector(r) for r in range(world)])
    expect = torch.empty(expect_stack.shape[1])
    _sequential(expect_stack, expect)
    for r in range(world):
        stacked, total, refused = res[r]
        assert stacked == expect_stack.numpy().tobytes(), f"rank {r}: gather not in rank order"
        assert total == expect.numpy().tobytes(), f"rank {r}: not the rank-order sum"
        assert refused, f"rank {r}: CPU tensors went through the exchange's kernel path"
    if world >= 3:  # with three terms the order shows: the reversed sum differs in some bits
        rev = torch.empty_like(expect)
        _sequential(expect_stack.flip(0), rev)
        assert not torch.equal(rev.view(torch.int32), expect.view(torch.int32))


def test_single_rank_exchange_is_a_copy():
    from row_wise_normalization_rms_gb300 import sharded

    local = _local_vector(0)
    total = torch.empty_like(local)
    sharded.exchange_dgamma(local, total)
    assert torch.equal(total, local)
