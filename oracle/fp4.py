"""FP4 cache format, restated plainly: pair-merge, E2M1 codes, E4M3 scales, block-major layout.

Test infrastructure only (see the package docstring).

What the pages fix: one 512-d latent per cache entry shared by keys and values ([digest] Core
Mechanics, "Channel"); two adjacent positions merged into one entry ([digest] Core Mechanics,
"Sequence"); FP4 storage of the global KV ([digest] Terminology "FP4"; [abstract] Abstract; [card] Key
ideas "FP4 global KV, trained that way"). Everything numeric below is this project's reading, because
the pages name no format:

  * merge(a, b) = fl32(fl32(a + b) * 0.5), a and b the bf16 inputs widened exactly to fp32.
  * E2M1 element: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is subnormal. The
    eight magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6 (OCP Microscaling Formats v1.0, FP4 E2M1).
  * E4M3 scale: OCP FP8 E4M3 (bias 7, subnormals, no infinities, S.1111.111 = NaN, max 448). Only
    non-negative scales occur.
  * One scale per 16 consecutive elements. AMAX rule: s = E4M3(round-to-nearest-even, saturating at
    448) of fl32(amax / 6). POW2 rule: s = the smallest power of two >= fl32(amax / 6), clamped to
    [2^-9, 256]. amax == 0 gives s == 0 and all-zero codes.
  * code = E2M1 nearest to fl32(m / s), ties to the even code, |value| saturating at 6, sign bit taken
    from the sign of fl32(m / s) (so -0.2 -> code 0x8).
  * Layout: entry e of a sequence lives in block e // 8, slot e % 8. A block holds the 8 slots' code
    bytes (dim/2 each, slot-major) followed by their scale bytes (dim/16 each, slot-major). Code byte j
    holds element 2j in the low nibble and element 2j+1 in the high nibble.
"""

import numpy as np

GROUP = 16
BLOCK = 8


# ---------------------------------------------------------------------------------------------
# Element formats (decode from the bit fields)
# ---------------------------------------------------------------------------------------------

def e2m1_value(code):
    """Value of E2M1 code(s) 0..15 from the bit fields (sign | exponent(2) | mantissa(1))."""
    code = np.asarray(code, dtype=np.int64)
    sign = np.where(code & 0x8, -1.0, 1.0)
    exponent = (code >> 1) & 0x3
    mantissa = code & 0x1
    magnitude = np.where(exponent == 0, 0.5 * mantissa,
                         np.exp2(exponent - 1.0) * (1.0 + 0.5 * mantissa))
    return sign * magnitude


def e4m3_value(byte):
    """Value of E4M3 byte(s) from the bit fields (sign | exponent(4), bias 7 | mantissa(3))."""
    b = np.asarray(byte, dtype=np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    exponent = (b >> 3) & 0xF
    mantissa = b & 0x7
    magnitude = np.where(exponent == 0, np.exp2(-6.0) * (mantissa / 8.0),
                         np.exp2(exponent - 7.0) * (1.0 + mantissa / 8.0))
    magnitude = np.where((b & 0x7F) == 0x7F, np.nan, magnitude)
    return sign * magnitude


# The 127 finite non-negative E4M3 values in byte order 0x00..0x7E (ascending in value).
_E4M3_NONNEG = e4m3_value(np.arange(0x7F))
# The 8 E2M1 magnitudes, code order 0..7 (ascending).
_E2M1_GRID = e2m1_value(np.arange(8))


def e4m3_encode_nonneg(x):
    """Round non-negative fp32 value(s) to E4M3 bytes: nearest value, ties to the even byte (even
    mantissa), values above 448 saturate to 448 (0x7E)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    if np.any(x < 0) or np.any(np.isnan(x)):
        raise ValueError("scale inputs must be non-negative numbers")
    lo = np.clip(np.searchsorted(_E4M3_NONNEG, x, side="right") - 1, 0, 0x7E)
    hi = np.minimum(lo + 1, 0x7E)
    v_lo, v_hi = _E4M3_NONNEG[lo], _E4M3_NONNEG[hi]
    mid = (v_lo + v_hi) / 2.0          # exact: both neighbours have 4 significant bits
    take_hi = (x > mid) | ((x == mid) & (hi % 2 == 0))
    out = np.where(take_hi, hi, lo)
    out = np.where(x >= 448.0, 0x7E, out)
    return out.astype(np.uint8)


def e2m1_encode(y):
    """E2M1 code(s) of fp32 value(s) y: the grid magnitude nearest |y| by brute force over all eight,
    ties to the even code, saturating at 6; the sign bit copies the sign bit of y."""
    y = np.asarray(y, dtype=np.float32)
    a = np.abs(y).astype(np.float64)
    a = np.where(np.isinf(a), 6.0, a)
    dist = np.abs(a[..., None] - _E2M1_GRID)            # [..., 8]
    best = dist.min(axis=-1, keepdims=True)
    ties = dist == best
    # among the nearest candidates prefer an even code; the grid is ascending so at most two tie
    even_tied = ties & (np.arange(8) % 2 == 0)
    idx = np.where(even_tied.any(axis=-1), np.argmax(even_tied, axis=-1), np.argmax(ties, axis=-1))
    sign = np.signbit(y).astype(np.int64) << 3
    return (idx | sign).astype(np.uint8)


# ---------------------------------------------------------------------------------------------
# Pair-merge and quantiser
# ---------------------------------------------------------------------------------------------

def pair_merge(x):
    """Merge rows 2i and 2i+1 of x (float32 [T, dim], exact bf16 values) into entry i:
    fl32(fl32(a + b) * 0.5). A trailing odd row is dropped ([digest] Core Mechanics, "Sequence")."""
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[0] // 2
    a = x[0:2 * n:2]
    b = x[1:2 * n:2]
    return (a + b) * np.float32(0.5)


def scale_bytes(amax, rule):
    """E4M3 scale byte for each group maximum (float32), rule 'amax' or 'pow2'."""
    amax = np.asarray(amax, dtype=np.float32)
    sf = amax / np.float32(6.0)                         # IEEE fp32 division
    if rule == "amax":
        return e4m3_encode_nonneg(sf)
    if rule != "pow2":
        raise ValueError(rule)
    mant, expo = np.frexp(sf.astype(np.float64))        # sf = mant * 2**expo, mant in [0.5, 1)
    k = np.where(mant == 0.5, expo - 1, expo)           # smallest power of two >= sf is 2**k
    k = np.clip(k, -9, 8)
    out = e4m3_encode_nonneg(np.exp2(k.astype(np.float64)).astype(np.float32))
    return np.where(sf == 0, 0, out).astype(np.uint8)


def quantize(m, rule, rows_per_chunk=4096):
    """Quantise rows m (float32 [n, dim], dim % 16 == 0). Returns (codes uint8 [n, dim] one code per
    element, scales uint8 [n, dim // 16]). Rows are independent; large inputs are processed a chunk of
    rows at a time only to bound the temporary memory of the brute-force search."""
    m = np.asarray(m, dtype=np.float32)
    n, dim = m.shape
    if dim % GROUP:
        raise ValueError("dim must be a multiple of 16")
    if n > rows_per_chunk:
        parts = [quantize(m[i:i + rows_per_chunk], rule, rows_per_chunk) for i in range(0, n, rows_per_chunk)]
        return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])
    g = m.reshape(n, dim // GROUP, GROUP)
    amax = np.abs(g).max(axis=-1)
    sb = scale_bytes(amax, rule)
    s = e4m3_value(sb).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = g / s[..., None]                             # IEEE fp32 division
    codes = e2m1_encode(y)
    codes = np.where((s == 0)[..., None], 0, codes).astype(np.uint8)
    return codes.reshape(n, dim), sb


def round_trip(x, rule):
    """Values of x (float32 [..., dim], dim % 16 == 0) after quantising them with `rule` and
    dequantising: the FP4 value each element is stored as."""
    x = np.asarray(x, dtype=np.float32)
    shape = x.shape
    rows = x.reshape(-1, shape[-1])
    codes, scales = quantize(rows, rule)
    s = np.repeat(e4m3_value(scales), GROUP, axis=1)
    return (e2m1_value(codes) * s).reshape(shape)


def entry_bytes(dim):
    return dim // 2 + dim // GROUP


def block_bytes(dim):
    return BLOCK * entry_bytes(dim)


def layout(codes, scales, first_entry=0, n_blocks=None, base=None):
    """Place quantised entries into block-major bytes. codes: [n, dim] one code per element;
    scales: [n, dim // 16]. Entry i goes to entry slot first_entry + i. Returns uint8
    [n_blocks, block_bytes(dim)] (a copy of `base` if given, else zeros)."""
    n, dim = codes.shape
    half, nsc = dim // 2, dim // GROUP
    last = first_entry + n
    if n_blocks is None:
        n_blocks = -(-last // BLOCK)
    out = np.zeros((n_blocks, block_bytes(dim)), np.uint8) if base is None else base.copy()
    packed = ((codes[:, 0::2] & 0xF) | ((codes[:, 1::2] & 0xF) << 4)).astype(np.uint8)
    e = first_entry + np.arange(n)
    blk, slot = e // BLOCK, e % BLOCK
    code_cols = slot[:, None] * half + np.arange(half)[None, :]
    out[blk[:, None], code_cols] = packed
    scale_cols = BLOCK * half + slot[:, None] * nsc + np.arange(nsc)[None, :]
    out[blk[:, None], scale_cols] = scales
    return out


def pack(x, merge, rule, first_entry=0, n_blocks=None, base=None):
    """csa_pack_fp4 for one sequence: merge (2) or take (1) rows of x, quantise, lay out."""
    x = np.asarray(x, dtype=np.float32)
    m = pair_merge(x) if merge == 2 else x
    codes, scales = quantize(m, rule)
    return layout(codes, scales, first_entry, n_blocks, base)


def unpack(blocks, dim, n_entries):
    """Inverse of layout: returns (codes [n_entries, dim], scales [n_entries, dim // 16])."""
    half, nsc = dim // 2, dim // GROUP
    e = np.arange(n_entries)
    blk, slot = e // BLOCK, e % BLOCK
    packed = blocks[blk[:, None], slot[:, None] * half + np.arange(half)[None, :]]
    codes = np.zeros((n_entries, dim), np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    scales = blocks[blk[:, None], BLOCK * half + slot[:, None] * nsc + np.arange(nsc)[None, :]]
    return codes, scales.astype(np.uint8)


def dequantize(blocks, dim, n_entries):
    """Dequantised entries (float64 [n_entries, dim]): E2M1 value times the group's E4M3 scale."""
    codes, scales = unpack(blocks, dim, n_entries)
    s = np.repeat(e4m3_value(scales), GROUP, axis=1)
    return e2m1_value(codes) * s
