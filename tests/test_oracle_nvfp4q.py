"""Pins for the NVFP4-query variant of oracle.attention (nvfp4_query, attend_kv, decode_attention_nvfp4q,
prefill_attention_nvfp4q): hand-worked roundings, the power-of-two equivariance the per-head pre-scale
gives, torch's fp64 attention with distinct keys and values, and reduction to the exact attention when the
query and the window keys are already on the FP4 grid."""

import os

import numpy as np
import pytest
import torch

from oracle import attention, fp4, indexer


def _golden(golden_dir):
    cases = []
    with open(os.path.join(golden_dir, "nvfp4_query.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            src, dst = line.split(";")
            q = np.zeros(512, np.float32)
            want = np.zeros(512, np.float32)
            for tok in src.split():
                i, v = tok.split("=")
                q[int(i)] = np.float32(float(v))
            for tok in dst.split():
                i, v = tok.split("=")
                want[int(i)] = np.float32(float(v))
            cases.append((q, want))
    return cases


def test_golden_query_roundings(golden_dir):
    cases = _golden(golden_dir)
    assert len(cases) == 5
    for q, want in cases:
        got = attention.nvfp4_query(q[None, :])[0]
        np.testing.assert_array_equal(got, want)


def test_power_of_two_equivariance():
    # the pre-scale depends only on the exponent of each head's maximum, so scaling a head by 2^k scales
    # its rounding by 2^k exactly (a missing or fixed pre-scale would saturate or flush the E4M3 scales)
    rng = np.random.default_rng(3)
    q = (rng.standard_normal((4, 512)) * np.array([[1.0], [50.0], [1e-3], [3e3]])).astype(np.float32)
    base = attention.nvfp4_query(q)
    for k in (-40, -7, -1, 1, 9, 33):
        f = np.float32(2.0 ** k)
        np.testing.assert_array_equal(attention.nvfp4_query(q * f), base * f)


def test_heads_are_independent_and_zero_heads_stay_zero():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((3, 512)).astype(np.float32)
    a = attention.nvfp4_query(q)
    q2 = q.copy()
    q2[1] *= np.float32(1000.0)
    q2[2] = 0.0
    b = attention.nvfp4_query(q2)
    np.testing.assert_array_equal(a[0], b[0])
    assert np.all(b[2] == 0)


def test_rounding_error_is_within_the_fp4_step():
    # every element moves by at most half an E2M1 step of its block scale, and the block maxima are
    # within the E4M3 rounding (6.25 %) of their value
    rng = np.random.default_rng(5)
    q = rng.standard_normal((8, 512)).astype(np.float32)
    r = attention.nvfp4_query(q)
    g = np.abs(q).reshape(8, 32, 16).max(-1)
    err = np.abs(r - q).reshape(8, 32, 16).max(-1)
    assert np.all(err <= g * (1.0 / 6.0) * 1.0625 + 1e-7)


def test_attend_kv_matches_torch_with_distinct_keys_and_values():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((5, 64))
    k = rng.standard_normal((23, 64))
    v = rng.standard_normal((23, 64))
    out, lse = attention.attend_kv(q, k, v, 0.125)
    t = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None], scale=0.125)[0]
    np.testing.assert_allclose(out, t.numpy(), rtol=0, atol=1e-12)
    z = (q @ k.T) * 0.125
    np.testing.assert_allclose(lse, np.log(np.exp(z).sum(1)), rtol=0, atol=1e-12)


def _grid_query(rng, heads):
    # heads whose elements are E2M1 codes times a block scale, each block holding a +-6 s element, with the
    # head maximum 6 s in [1024, 2048): exactly representable, so nvfp4_query leaves them unchanged
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    scales = np.array([176, 192, 208, 224, 240, 256, 288, 320], np.float32)
    q = np.zeros((heads, 512), np.float32)
    for h in range(heads):
        for g in range(32):
            s = scales[rng.integers(0, 8)] if g == 0 else np.float32(2.0 ** rng.integers(-3, 5))
            blk = mags[rng.integers(0, 8, 16)] * np.where(rng.random(16) < 0.5, -1, 1)
            blk[rng.integers(0, 16)] = 6.0
            q[h, 16 * g:16 * g + 16] = blk.astype(np.float32) * s
    return q


def _cache(rng, n_entries, cap):
    x = rng.standard_normal((2 * n_entries, 512)).astype(np.float32)
    blocks = fp4.pack(x, merge=2, rule="amax", n_blocks=(cap + 7) // 8)
    return fp4.dequantize(blocks, 512, cap)


def test_decode_reduces_to_exact_attention_on_fp4_inputs():
    rng = np.random.default_rng(7)
    q = _grid_query(rng, 4)
    np.testing.assert_array_equal(attention.nvfp4_query(q), q)
    entries = _cache(rng, 70, 80)
    idx = np.array([0, 3, 8, -1, 5])
    win = fp4.round_trip(rng.standard_normal((40, 512)).astype(np.float32) * 3, "amax")
    np.testing.assert_array_equal(fp4.round_trip(win, "amax"), win)
    a = attention.decode_attention_nvfp4q(q, entries, 70, idx, win, 0.04)
    b = attention.decode_attention(q, entries, 70, idx, win, 0.04)
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-12)


def test_window_values_stay_exact():
    # one window row and no cache rows: the softmax weight is 1, so the output is the row itself (not its
    # FP4 rounding), and lse is the logit of the rounded query against the rounded key
    rng = np.random.default_rng(8)
    q = rng.standard_normal((2, 512)).astype(np.float32)
    row = rng.standard_normal((1, 512)).astype(np.float32) * 7
    entries = np.zeros((8, 512))
    out, lse = attention.decode_attention_nvfp4q(q, entries, 0, np.array([-1]), row, 0.1)
    np.testing.assert_array_equal(out, np.broadcast_to(row.astype(np.float64), out.shape))
    z = attention.nvfp4_query(q).astype(np.float64) @ fp4.round_trip(row, "amax")[0].astype(np.float64) * 0.1
    np.testing.assert_allclose(lse, z, rtol=0, atol=1e-12)
    assert not np.array_equal(fp4.round_trip(row, "amax"), row)


@pytest.mark.parametrize("p", [0, 1, 2, 17, 60])
def test_prefill_reduces_to_exact_attention_on_fp4_inputs(p):
    rng = np.random.default_rng(9 + p)
    q = _grid_query(rng, 2)
    entries = _cache(rng, 40, 48)
    idx = np.array([0, 1, 2, 3, 4, -1])
    swa = fp4.round_trip(rng.standard_normal((64, 512)).astype(np.float32), "amax")
    a = attention.prefill_attention_nvfp4q(q, entries, 40, idx, swa, 0, p, 16, 0.05)
    b = attention.prefill_attention(q, entries, 40, idx, swa, 0, p, 16, 0.05)
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-12)
    # the causal rule is the indexer's: entries with 2e + 1 <= p, window tokens max(p - 15, 0) .. p
    el = indexer.eligibility(40, 48, q_pos=[p])[0]
    assert el.sum() == min(40, (p + 1) // 2)
