"""Pins for oracle.fp4 against values and properties that do not come from the oracle itself."""

import os

import numpy as np
import pytest
import torch

from oracle import fp4


def test_e2m1_table_all_codes():
    # OCP Microscaling Formats v1.0, FP4 E2M1: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign.
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = fp4.e2m1_value(np.arange(16))
    np.testing.assert_array_equal(got[:8], table)
    np.testing.assert_array_equal(got[8:], [-v for v in table])
    assert np.signbit(got[8])          # code 0x8 is negative zero


def test_e4m3_decode_matches_torch_float8():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp4.e4m3_value(np.arange(256))
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert fp4.e4m3_value(0x7E) == 448.0 and fp4.e4m3_value(0x01) == 2.0 ** -9
    assert fp4.e4m3_value(0x08) == 2.0 ** -6 and fp4.e4m3_value(0x38) == 1.0


def test_e4m3_rounding_matches_torch_float8():
    rng = np.random.default_rng(7)
    vals = [np.exp2(rng.uniform(-12, np.log2(448.0), 200000)).astype(np.float32)]
    # every midpoint between neighbouring finite values, and each value itself
    pos = fp4.e4m3_value(np.arange(0x7F))
    vals.append(((pos[:-1] + pos[1:]) / 2).astype(np.float32))
    vals.append(pos.astype(np.float32))
    vals.append(np.array([0.0, 2.0 ** -10, 2.0 ** -11, 1e-30, 447.9, 448.0], np.float32))
    x = np.concatenate(vals)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = fp4.e4m3_encode_nonneg(x)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_saturates_at_448():
    got = fp4.e4m3_encode_nonneg(np.array([448.0, 460.0, 1e6, np.inf], np.float32))
    np.testing.assert_array_equal(got, [0x7E] * 4)


def test_e2m1_nearest_and_ties_even():
    # defining property checked by brute force over a dense sweep: the chosen magnitude is a nearest
    # grid value, and at an exact midpoint the chosen code is even
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    y = np.concatenate([np.linspace(-7, 7, 28001), (grid[:-1] + grid[1:]) / 2,
                        -(grid[:-1] + grid[1:]) / 2]).astype(np.float32)
    codes = fp4.e2m1_encode(y).astype(np.int64)
    mag = grid[codes & 7]
    a = np.minimum(np.abs(y.astype(np.float64)), 6.0)
    best = np.abs(a[:, None] - grid[None, :]).min(axis=1)
    np.testing.assert_array_equal(np.abs(a - mag), best)
    tie = (np.abs(a[:, None] - grid[None, :]) == best[:, None]).sum(axis=1) == 2
    assert tie.sum() >= 14
    assert np.all((codes[tie] & 1) == 0)
    np.testing.assert_array_equal((codes >> 3) & 1, np.signbit(y))


def _golden_groups(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "fp4_groups.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rule, vals, codes, scale = [p.strip() for p in line.split(";")]
            rows.append((rule, np.array([float(v) for v in vals.split()], np.float32),
                         [int(c, 16) for c in codes.split()], int(scale, 16)))
    return rows


def test_golden_groups(golden_dir):
    rows = _golden_groups(golden_dir)
    assert len(rows) >= 9
    for rule, vals, codes, scale in rows:
        c, s = fp4.quantize(vals[None, :], rule)
        packed = (c[0, 0::2] | (c[0, 1::2] << 4)).tolist()
        assert packed == codes, (rule, vals, [hex(v) for v in packed])
        assert int(s[0, 0]) == scale


def test_pair_merge_is_rounded_mean():
    # for bf16 inputs fl32(fl32(a + b) * 0.5) equals the exact mean rounded once to fp32
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(4096, 64, generator=g) * torch.exp(torch.randn(4096, 64, generator=g) * 4))
    x = x.to(torch.bfloat16).float().numpy()
    m = fp4.pair_merge(x)
    ref = ((x[0::2].astype(np.float64) + x[1::2].astype(np.float64)) / 2).astype(np.float32)
    np.testing.assert_array_equal(m, ref)
    assert fp4.pair_merge(x[:5]).shape[0] == 2       # odd trailing row dropped


def test_quantize_picks_nearest_scaled_grid_value():
    rng = np.random.default_rng(11)
    m = (rng.standard_normal((2000, 64)) * np.exp2(rng.integers(-8, 8, (2000, 1)))).astype(np.float32)
    codes, scales = fp4.quantize(m, "amax")
    s = np.repeat(fp4.e4m3_value(scales), 16, axis=1)
    deq = fp4.e2m1_value(codes) * s
    cand = fp4.e2m1_value(np.arange(16))[None, None, :] * s[..., None]
    err = np.abs(m[..., None].astype(np.float64) - cand)
    best = err.min(axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):     # groups whose scale rounds to 0
        y = m.astype(np.float64) / s
    near_mid = np.min(np.abs(np.abs(y)[..., None] - np.array([.25, .75, 1.25, 1.75, 2.5, 3.5, 5.0])),
                      axis=-1) < 1e-5
    ok = np.isclose(np.abs(m - deq), best, rtol=0, atol=0) | near_mid
    assert ok.all()
    # the scale is the E4M3 value nearest amax / 6 (or 448)
    amax = np.abs(m.reshape(2000, 4, 16)).max(-1)
    sv = fp4.e4m3_value(scales)
    target = np.minimum(amax.astype(np.float64) / 6, 448)
    all_vals = fp4.e4m3_value(np.arange(0x7F))
    nearest = np.abs(target[..., None] - all_vals).min(-1)
    np.testing.assert_allclose(np.abs(sv - target), nearest, rtol=1e-6, atol=0)


def test_pow2_exact_for_integer_keys():
    rng = np.random.default_rng(5)
    k = rng.integers(-4, 5, (999, 128)).astype(np.float32)
    blocks = fp4.pack(k, merge=1, rule="pow2")
    back = fp4.dequantize(blocks, 128, 999)
    np.testing.assert_array_equal(back, k)
    _, scales = fp4.quantize(k, "pow2")
    vals = set(fp4.e4m3_value(np.unique(scales)).tolist())
    assert vals <= {0.0, 0.25, 0.5, 1.0}


def test_pow2_scale_clamps():
    s = fp4.scale_bytes(np.array([1e-20, 6 * 2.0 ** -9, 6 * 300.0, 6.0, 6.5], np.float32), "pow2")
    np.testing.assert_array_equal(fp4.e4m3_value(s), [2.0 ** -9, 2.0 ** -9, 256.0, 1.0, 2.0])


def test_block_layout_offsets():
    # dim 16: entry = 8 code bytes + 1 scale byte; block = 8 * 8 code bytes then 8 scale bytes = 72 B
    assert fp4.entry_bytes(512) == 288 and fp4.block_bytes(512) == 2304
    assert fp4.block_bytes(128) == 576 and fp4.block_bytes(16) == 72
    n = 11
    codes = np.zeros((n, 16), np.uint8)
    for i in range(n):
        codes[i, 0] = (i + 1) & 0xF    # low nibble of byte 0
        codes[i, 3] = 0x9              # high nibble of byte 1
    scales = np.arange(100, 100 + n, dtype=np.uint8)[:, None]
    out = fp4.layout(codes, scales, first_entry=3)
    assert out.shape == (2, 72)
    # entry i lands in slot 3 + i: block (3+i)//8, slot (3+i)%8
    assert out[0, 3 * 8] == 0x01 and out[0, 3 * 8 + 1] == 0x90 and out[0, 64 + 3] == 100
    assert out[0, 7 * 8] == 0x05 and out[0, 64 + 7] == 104
    assert out[1, 0] == 0x06 and out[1, 1] == 0x90 and out[1, 64] == 105
    assert out[1, 5 * 8] == 0x0B and out[1, 64 + 5] == 110
    assert out[0, 0] == 0 and out[0, 64] == 0          # slots before first_entry untouched
    c2, s2 = fp4.unpack(out, 16, 14)
    np.testing.assert_array_equal(c2[3:], codes)
    np.testing.assert_array_equal(s2[3:, 0], scales[:, 0])


def test_dequantize_is_code_times_scale():
    blocks = np.zeros((1, 2304), np.uint8)
    blocks[0, 0] = 0xF7            # entry 0: element 0 = +6, element 1 = -6 (code units)
    blocks[0, 2048] = 0x40         # entry 0 group 0 scale = 2.0
    blocks[0, 2048 + 31] = 0x30    # entry 0 group 31 scale = 0.5
    blocks[0, 255] = 0x20          # entry 0 element 511 = code 2 (1.0)
    d = fp4.dequantize(blocks, 512, 1)
    assert d[0, 0] == 12.0 and d[0, 1] == -12.0 and d[0, 511] == 0.5 and d[0, 2] == 0.0
