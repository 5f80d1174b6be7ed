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
