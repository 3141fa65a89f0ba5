"""The seeded input generator: determinism, rounding, laws (CPU only)."""
import dataclasses

import numpy as np
import torch

from synthetic import (WORKLOADS, bf16_bits_to_float32, float_to_bf16_bits, make_inputs,
                       storage_to_float64, workload)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.uniform(-30, 30, 100000),
                        [0.0, -0.0, 1.0, 3.0e38, -3.4e38, 1e-40]]).astype(np.float32)
    ours = float_to_bf16_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(bf16_bits_to_float32(ours), torch.from_numpy(v).to(torch.bfloat16).float().numpy())


def test_deterministic_and_independent_streams():
    w = dataclasses.replace(workload("llama7b_bf16_8192x4096"), M=37, N=96)
    a, b = make_inputs(w), make_inputs(w)
    for k in ("x", "gamma", "dy"):
        assert np.array_equal(a[k], b[k])
    assert not np.array_equal(a["x"], a["dy"])
    c = make_inputs(dataclasses.replace(w, seed=1))
    assert not np.array_equal(a["x"], c["x"])


def test_laws_and_dtypes():
    w = dataclasses.replace(workload("wide_bf16_16384x8192"), M=512, N=512)
    d = make_inputs(w)
    assert d["x"].dtype == np.uint16 and d["x"].shape == (512, 512)
    x = storage_to_float64(d["x"], "bf16")
    s = d["row_scale"]
    assert s.min() >= 0.01 and s.max() <= 100.0
    z = x / s[:, None]
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    g = storage_to_float64(d["gamma"], "bf16")
    assert abs(g.mean() - 1.0) < 0.05 and abs(g.std() - 0.2) < 0.03
    t = make_inputs(workload("tiny_f32_64x128"))
    assert t["x"].dtype == np.float32 and t["gamma"].min() >= 0.5 and t["gamma"].max() <= 1.5


def test_sweep_row_counts():
    ms = {w.N: w.M for w in WORKLOADS.values() if w.name.startswith("sweep")}
    assert ms == {512: 262144, 1000: 134217, 2048: 65536, 5120: 26214, 11008: 12192, 16384: 8192}
