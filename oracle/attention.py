"""Sparse attention over selected FP4 cache entries merged with the sliding window, in fp64.

Test infrastructure only (see the package docstring).

Follows [digest] Core Mechanics ("one 512-dim latent shares keys and values across all attention
heads"), [digest] Terminology (sliding window of 128) and [card] Key ideas ("Every layer keeps its own
query and sliding-window KV"). The reading taken: for query position u and head h the rows are the
dequantised eligible entries of the selected blocks together with the window rows; each row is both
key and value; z = scale * (q_h . row); out = softmax(z) @ rows; lse = log sum exp z. No rotary
embedding, sink or output projection. Duplicates between the window and the cache are kept.
"""

import numpy as np

from .fp4 import round_trip
from .indexer import eligibility

BLOCK = 8


def attend(q, rows, scale):
    """q: [H, D], rows: [n, D]; fp64. Returns (out [H, D], lse [H]). No rows: zeros and -inf."""
    q = np.asarray(q, np.float64)
    rows = np.asarray(rows, np.float64)
    if rows.shape[0] == 0:
        return np.zeros_like(q), np.full(q.shape[0], -np.inf)
    z = (q @ rows.T) * scale
    m = z.max(axis=1, keepdims=True)
    p = np.exp(z - m)
    l = p.sum(axis=1, keepdims=True)
    out = (p @ rows) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def selected_rows(entries, idx, eligible):
    """entries: dequantised [n_cap, D]; idx: block ids (-1 = empty); eligible: bool [n_cap].
    Returns the rows of eligible entries inside the listed blocks, in listing order."""
    out = []
    for b in np.asarray(idx):
        if b < 0:
            continue
        for e in range(b * BLOCK, b * BLOCK + BLOCK):
            if e < entries.shape[0] and eligible[e]:
                out.append(entries[e])
    if not out:
        return np.zeros((0, entries.shape[1]))
    return np.stack(out)


def decode_attention(q, entries, n_entries, idx, swa_rows, scale):
    """One decode query: q [H, D]; entries [n_cap, D]; idx [K]; swa_rows [w, D] (already cut to the
    rows in use). Every entry below n_entries is eligible. Returns (out, lse)."""
    el = eligibility(n_entries, entries.shape[0])[0]
    rows = np.concatenate([selected_rows(entries, idx, el), np.asarray(swa_rows, np.float64)], axis=0)
    return attend(q, rows, scale)


def prefill_window(swa, swa_first_pos, p, window):
    """Window rows for prefill position p: tokens max(p - window + 1, swa_first_pos) .. p; the row of
    token t is t - swa_first_pos."""
    lo = max(p - window + 1, swa_first_pos)
    return np.asarray(swa, np.float64)[lo - swa_first_pos:p - swa_first_pos + 1]


def prefill_attention(q, entries, n_entries, idx, swa, swa_first_pos, p, window, scale):
    """One causal query at token position p: the entries of the listed blocks that the indexer's
    eligibility rule admits at p (e < n_entries and 2e + 1 <= p), then the window rows of tokens
    max(p - window + 1, swa_first_pos) .. p. Used for prefill positions and for the draft positions of a
    multi-token decode step (speculative verification), which follow the same rule."""
    el = eligibility(n_entries, entries.shape[0], q_pos=[p])[0]
    rows = np.concatenate([selected_rows(entries, idx, el),
                           prefill_window(swa, swa_first_pos, p, window)], axis=0)
    return attend(q, rows, scale)


def dense_attention(q, entries, n_entries, swa_rows, scale):
    """Attention over every entry below n_entries plus the window, written without any block
    selection (used for the invariant that a Top-K covering every block equals dense attention)."""
    rows = np.concatenate([np.asarray(entries[:n_entries], np.float64),
                           np.asarray(swa_rows, np.float64)], axis=0)
    return attend(q, rows, scale)


# ---------------------------------------------------------------------------------------------
# NVFP4-query variant (opt-in): the logits q . k are taken with the query rounded to the cache's FP4
# format, so that the product can run on the block-scaled FP4 tensor cores, whose operands are both FP4.
# [card] Key ideas, "FP4 global KV, trained that way", stores the global KV in FP4; the pages give no
# query format, so this variant is this library's reading (an approximation the caller opts into):
#   * each query head h is scaled by 2^-e_h, e_h = floor(log2 max|q_h|) - 10 clamped to [-100, 100]
#     (0 for an all-zero head), so that every 16-element block's amax / 6 lies below 342 and its E4M3
#     scale stays inside the format; the scaled head is rounded with the AMAX rule of the cache format
#     and scaled back: q4_h = 2^e_h * round_trip(2^-e_h q_h, 'amax');
#   * window rows enter the logits as keys rounded with the same AMAX rule (no pre-scale), because the
#     block-scaled product needs both operands in FP4; cache rows are already in that format;
#   * every value (cache row or window row) stays exact, as in the exact path.
# ---------------------------------------------------------------------------------------------

def nvfp4_query(q):
    """Rounding of the query heads q [H, D] (float32 values) of the NVFP4-query variant (see above)."""
    q = np.asarray(q, np.float32)
    out = np.zeros_like(q)
    for h in range(q.shape[0]):
        amax = float(np.abs(q[h]).max()) if q.shape[1] else 0.0
        if amax == 0.0:
            e = 0
        else:
            _, k = np.frexp(amax)                       # amax = m * 2^k, m in [0.5, 1)
            e = int(np.clip(k - 1 - 10, -100, 100))
        f = np.float32(2.0 ** -e)
        out[h] = round_trip(q[h][None, :] * f, "amax")[0] * np.float32(2.0 ** e)
    return out


def attend_kv(q, keys, values, scale):
    """q: [H, D], keys and values: [n, D] (row i of keys scores value row i); fp64. Returns (out [H, D],
    lse [H]). No rows: zeros and -inf."""
    q = np.asarray(q, np.float64)
    keys = np.asarray(keys, np.float64)
    values = np.asarray(values, np.float64)
    if keys.shape[0] == 0:
        return np.zeros((q.shape[0], values.shape[1])), np.full(q.shape[0], -np.inf)
    z = (q @ keys.T) * scale
    m = z.max(axis=1, keepdims=True)
    p = np.exp(z - m)
    l = p.sum(axis=1, keepdims=True)
    out = (p @ values) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def _nvfp4_rows(cache_rows, window_rows):
    window_rows = np.asarray(window_rows, np.float32)
    keys = np.concatenate([np.asarray(cache_rows, np.float64),
                           round_trip(window_rows, "amax").astype(np.float64)], axis=0)
    values = np.concatenate([np.asarray(cache_rows, np.float64), window_rows.astype(np.float64)], axis=0)
    return keys, values


def decode_attention_nvfp4q(q, entries, n_entries, idx, swa_rows, scale):
    """decode_attention with the NVFP4-query logits: the rows are those of decode_attention; the keys of
    window rows are rounded to FP4 and the query heads by nvfp4_query; values are exact."""
    el = eligibility(n_entries, entries.shape[0])[0]
    keys, values = _nvfp4_rows(selected_rows(entries, idx, el), swa_rows)
    return attend_kv(nvfp4_query(q), keys, values, scale)


def prefill_attention_nvfp4q(q, entries, n_entries, idx, swa, swa_first_pos, p, window, scale):
    """prefill_attention (causal position p) with the NVFP4-query logits of decode_attention_nvfp4q."""
    el = eligibility(n_entries, entries.shape[0], q_pos=[p])[0]
    keys, values = _nvfp4_rows(selected_rows(entries, idx, el),
                               prefill_window(swa, swa_first_pos, p, window).astype(np.float32))
    return attend_kv(nvfp4_query(q), keys, values, scale)
