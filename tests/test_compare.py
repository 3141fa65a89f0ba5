"""The tolerance checks flag what they should (CPU only)."""
import numpy as np

from oracle import compare


def test_y_bf16_bar():
    ref = np.array([0.5, 2.0, -300.0])
    assert compare.check_y(ref + np.array([0.0099, 0.0199, 2.99]), ref, "bf16").ok
    assert not compare.check_y(ref + np.array([0.0101, 0.0, 0.0]), ref, "bf16").ok
    assert not compare.check_y(ref + np.array([0.0, 0.0, 3.01]), ref, "bf16").ok


def test_y_f32_relative():
    ref = np.array([1.0, 1e-3])
    assert compare.check_y(ref * (1 + 9e-6), ref, "f32").ok
    assert not compare.check_y(ref * np.array([1.0, 1 + 2e-5]), ref, "f32").ok


def test_dx_and_dgamma_scaled_by_terms():
    ref = np.array([1e-9, 1.0])
    scale = np.array([10.0, 1.0])
    assert compare.check_dx(ref + np.array([5e-5, 0.0]), ref, scale, "f32").ok
    assert not compare.check_dx(ref + np.array([2e-4, 0.0]), ref, scale, "f32").ok
    assert compare.check_dgamma(ref + np.array([1e-3, 0.0]), ref, scale, "f32").ok
    assert not compare.check_dgamma(ref + np.array([2e-3, 0.0]), ref, scale, "f32").ok


def test_nonfinite_handling():
    ref = np.array([np.nan, np.inf, 1.0])
    assert compare.check_y(np.array([np.nan, np.inf, 1.0]), ref, "f32").ok
    assert not compare.check_y(np.array([1.0, np.inf, 1.0]), ref, "f32").ok
    assert not compare.check_y(np.array([np.nan, np.inf, np.nan]), ref, "f32").ok


def test_rstd_bar():
    ref = np.array([0.25, 100.0])
    assert compare.check_rstd(ref * (1 + 9e-7), ref).ok
    assert not compare.check_rstd(ref * (1 + 2e-6), ref).ok


# ---- column sums: the depth-derived bar ---------------------------------------

U = 2.0 ** -24


def _f32_sum_like_the_kernels(terms, partials, tile):
    """float32 column sums in the kernels' order: tiles of ``tile`` rows dealt
    to ``partials`` units in turn, each unit adding its rows one by one into
    its partial row, then the partial rows added one by one."""
    M = terms.shape[0]
    t32 = terms.astype(np.float32)
    acc = np.zeros((partials, terms.shape[1]), np.float32)
    ntiles = -(-M // tile)
    for k in range(ntiles):
        p = k % partials
        for i in range(k * tile, min(M, (k + 1) * tile)):
            acc[p] = acc[p] + t32[i]  # one float32 rounding per addition
    out = np.zeros(terms.shape[1], np.float32)
    for p in range(partials):
        out = out + acc[p]
    rows = tile * -(-ntiles // partials)
    return out.astype(np.float64), (partials, rows)


def test_sum_error_factor_is_reached_by_half_ulp_terms():
    """1 followed by k terms of half an ulp: every addition rounds back to 1
    (ties to even), so float32 loses k u exactly, which is the first-order
    bound of a depth-k sum.  The bar's D = rows + P = k + 2 covers it; a
    depth counted three short (k - 1) would not."""
    for k in (5, 40, 300):
        terms = np.array([1.0] + [U] * k)[:, None]
        got, red = _f32_sum_like_the_kernels(terms, 1, 1)
        exact = 1.0 + k * U
        err = abs(got[0] - exact)
        assert err == k * U
        assert err <= compare.sum_error_factor(red) * np.sum(np.abs(terms))
        short = (red[0], red[1] - 3)  # an undercount of the depth
        assert err > compare.sum_error_factor(short) * np.sum(np.abs(terms))


def _rms_terms(M, N, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, N)) * np.exp(rng.uniform(np.log(0.01), np.log(100), (M, 1)))
    dy = rng.standard_normal((M, N))
    r = 1.0 / np.sqrt(np.mean(x * x, axis=1) + 1e-5)
    # as a kernel forms them: r stored in float32, x r rounded, the product rounded
    r32 = r.astype(np.float32)
    xn = (x.astype(np.float32) * r32[:, None]).astype(np.float32)
    t = (dy.astype(np.float32) * xn).astype(np.float32).astype(np.float64)
    exact = dy * x * r[:, None]
    return t, exact


def test_tight_dgamma_bar_holds_for_kernel_order_sums_and_sees_dropped_rows():
    M, N = 16384, 64
    t, exact = _rms_terms(M, N, 3)
    ref = exact.sum(axis=0)
    scale = np.abs(exact).sum(axis=0)
    for partials, tile in ((608, 1), (304, 2), (152, 4)):
        got, red = _f32_sum_like_the_kernels(t, partials, tile)
        checks = compare.dgamma_checks(got, ref, scale, "bf16", red)
        assert all(c.ok for c in checks), [str(c) for c in checks]
        # one row's contribution missing: the scaled bar does not see it,
        # the tight one does
        for row in (M // 2, M - 1):
            dropped = compare.dgamma_checks(got - t[row], ref, scale, "bf16", red)
            assert dropped[0].ok, "expected the scaled bar to be blind to one row"
            assert not dropped[2].ok, (row, str(dropped[2]))
        # the last tile wave (the last 8 rows)
        dropped = compare.dgamma_checks(got - t[-8:].sum(axis=0), ref, scale, "bf16", red)
        assert not dropped[2].ok, str(dropped[2])


def test_normwise_bar():
    ref = np.array([3.0, -4.0])  # norm 5
    assert compare.check_normwise("v", ref + np.array([0.009, 0.0]), ref, 2e-3).ok
    assert not compare.check_normwise("v", ref + np.array([0.011, 0.0]), ref, 2e-3).ok


def test_merged_blocks_equal_one_check():
    rng = np.random.default_rng(1)
    ref = rng.standard_normal((40, 7))
    got = ref + rng.standard_normal((40, 7)) * 1e-3
    whole = compare.check_y(got, ref, "bf16")
    parts = compare.merge(compare.check_y(got[i:i + 9], ref[i:i + 9], "bf16")
                          for i in range(0, 40, 9))
    assert (parts.ok, parts.n, parts.n_bad) == (whole.ok, whole.n, whole.n_bad)
    assert parts.max_abs == whole.max_abs and parts.worst_ratio == whole.worst_ratio
    assert abs(parts.norm_rel - whole.norm_rel) <= 1e-12 * whole.norm_rel
