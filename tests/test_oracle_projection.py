"""Pins for oracle.projection: the projection equals an exact integer product, the write path reduces to
the pinned pack when the weight selects hidden columns, and an odd trailing token is not packed."""

import numpy as np

from oracle import fp4, projection


def test_projection_equals_exact_integer_product():
    # small integers keep every dot product exact in fp32, so the projection must equal the int64 product
    rng = np.random.default_rng(0)
    h = rng.integers(-8, 9, (37, 640))
    w = rng.integers(-4, 5, (512, 640))
    exact = h.astype(np.int64) @ w.astype(np.int64).T
    x = projection.project(h, w)
    assert x.dtype == np.float32 and x.shape == (37, 512)
    np.testing.assert_array_equal(x.astype(np.int64), exact)


def test_projection_rounds_the_exact_sum_once():
    # the exact sum 1 + 2^-24 + 2^-25 lies above the fp32 midpoint 1 + 2^-24, so rounding it once gives
    # 1 + 2^-23; adding the terms in fp32 one by one would give 1.0 (1 + 2^-24 ties to even, 1.0, and
    # 1.0 + 2^-25 rounds back to 1.0)
    h = np.zeros((1, 64))
    w = np.zeros((512, 64))
    h[0, :3] = [1.0, 2.0 ** -24, 2.0 ** -25]
    w[0, :3] = 1.0
    x = projection.project(h, w)
    assert x[0, 0] == np.float32(1.0 + 2.0 ** -23)
    assert np.all(x[0, 1:] == 0)


def test_selecting_weight_reduces_to_the_pack():
    # w = [I | 0] picks the first 512 hidden columns: the write path is then the pinned pack of those
    rng = np.random.default_rng(1)
    h = rng.standard_normal((20, 768)).astype(np.float32)
    h = h.astype(np.float64)
    w = np.zeros((512, 768))
    w[:, :512] = np.eye(512)
    for rule in ("amax", "pow2"):
        got = projection.project_pack(h, w, rule, first_entry=3, n_blocks=3)
        want = fp4.pack(h[:, :512].astype(np.float32), 2, rule, first_entry=3, n_blocks=3)
        np.testing.assert_array_equal(got, want)


def test_odd_trailing_token_is_not_packed():
    rng = np.random.default_rng(2)
    h = rng.integers(-3, 4, (9, 128)).astype(np.float64)
    w = rng.integers(-2, 3, (512, 128)).astype(np.float64)
    full = projection.project_pack(h, w, "amax", n_blocks=1)
    even = projection.project_pack(h[:8], w, "amax", n_blocks=1)
    np.testing.assert_array_equal(full, even)
    codes, scales = fp4.unpack(full, 512, 8)
    assert np.all(codes[4:] == 0) and np.all(scales[4:] == 0)      # entries 4.. were never written
    assert np.any(scales[:4] != 0)
