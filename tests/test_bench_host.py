"""bench.py's host logic without a GPU: the multi-rank reduction over gloo
(world size 2), the byte formula, and the reference (oracle) arm."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    r, lr, w = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    m = bench.max_over_ranks(10.0 + 5.0 * r, dist)
    out[r] = (r, lr, w, m)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = 29500 + os.getpid() % 1000
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == (0, 0, 2, 15.0) and res[1] == (1, 1, 2, 15.0)


def test_step_bytes_formula():
    sys.path.insert(0, ROOT)
    import bench

    f, b = bench.step_bytes(16384, 8192, 2)
    assert f == 2 * 16384 * 8192 * 2 + 4 * 16384 + 8192 * 2
    assert b == 3 * 16384 * 8192 * 2 + 4 * 16384 + 8192 * 2 + 4 * 8192


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["M"] == 16384 and d["config"]["N"] == 8192


def test_reference_arm_other_ranks_are_silent():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_floor():
    r = subprocess.run([sys.executable, "bench.py", "--warmup", "2"], cwd=ROOT,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


def test_source_hash_ignores_comments_but_not_code():
    import bench

    src = 'int f(int a) {\n  return a * 2;  // twice\n}\nconst char* s = "x // y";\n'
    commented = ('/* header */\nint f(int a) {\n  /* multi\n line */ return a * 2;\n}\n'
                 'const char* s = "x // y";  // trailing\n')
    assert bench.code_tokens(src) == bench.code_tokens(commented)
    assert bench.code_tokens(src) != bench.code_tokens(src.replace("2", "3"))
    assert bench.code_tokens(src) != bench.code_tokens(src.replace("x // y", "x y"))
    assert len(bench.kernel_source_hash()) == 16


def test_cpu_baseline_times_each_direction():
    import bench
    from synthetic import workload

    w = workload("tiny_f32_64x128")
    cb = bench.cpu_oracle_throughput(w, seconds=0.3, rows_per_worker=8, workers=2)
    assert cb["kind"] == "oracle" and cb["cores"] == 2 and cb["unit"] == "GB/s"
    assert "2 host cores" in cb["sample"]
    assert cb["value"] > 0 and cb["fwd_gbs"] > 0 and cb["bwd_gbs"] > 0
    # the combined rate lies between the two directions' rates
    assert min(cb["fwd_gbs"], cb["bwd_gbs"]) * 0.99 <= cb["value"] <= max(cb["fwd_gbs"],
                                                                        cb["bwd_gbs"]) * 1.01


def test_workload_spec_from_the_command_line():
    import pytest

    import bench
    from synthetic import make_inputs

    w = bench.workload_from_spec("M=12,N=96,dtype=f16,eps=1e-5,gemma=1,inplace=1,seed=3")
    assert (w.M, w.N, w.dtype, w.eps, w.gemma, w.inplace_dx, w.seed, w.op) == \
        (12, 96, "f16", 1e-5, 1, 1, 3, "rms")
    for op in ("rms", "ln", "rms_add", "rms_quant"):
        wo = bench.workload_from_spec(f"M=5,N=64,op={op}")
        inp = make_inputs(wo)
        assert inp["x"].shape == (5, 64)
        if op == "rms_add":
            assert inp["residual"] is not None and inp["dh"] is not None
        if op == "ln":
            assert inp["beta"] is not None
    assert bench.workload_from_spec("M=2,N=8,weight=f32").wdtype == "f32"
    for bad in ("N=8", "M=2", "M=2,N=8,foo=1", "M=2,N=0", "M=2,N=8,dtype=f64", "M=2,N=8,gemma=2",
                "M=2,N=8,op=swiglu", "M=2,N8"):
        with pytest.raises(ValueError):
            bench.workload_from_spec(bad)


def test_oracle_pool_sums_worker_partials_in_worker_order():
    """The multi-core oracle's dgamma: each worker's rows, summed in worker
    order, equal the oracle over all the sample's rows."""
    import numpy as np

    import bench
    from oracle import rmsnorm_oracle as orc
    from synthetic import make_inputs, storage_to_float64, workload

    w = workload("tiny_f32_64x128")
    pool = bench.OraclePool(w.name, 5, 3)
    try:
        _, dg = pool.run("bwd")
    finally:
        pool.close()
    inp = make_inputs(w.with_shape(15))
    x = storage_to_float64(inp["x"], w.dtype)
    dy = storage_to_float64(inp["dy"], w.dtype)
    g = storage_to_float64(inp["gamma"], w.wdtype)
    _, ref = orc.rms_backward(x, g, dy, w.eps)
    assert np.allclose(dg, ref, rtol=1e-13, atol=1e-13 * np.abs(ref).max())
