"""Block indexer and Top-K, restated plainly.

Test infrastructure only (see the package docstring).

Follows [card] Key ideas: layers either make the index (Full), "rescore with [their] own indexer
query" (Reindex) or reuse "Top-K indices" (Reuse); selection is over "blocks of 8", and "a
hierarchical sparse indexer (up to 2,048 blocks of 8 positions) trims decoder indexing". The pages give
no score function, tie rule or hierarchy shape; the readings taken here:

  * entry score (the plain definition, `entry_scores`): s_e = sum over heads h (in order 0, 1, ...) of
    fl32(w_h * r_h), r_h = max(0, q_h . k_e) with ReLU, plain q_h . k_e without, where k_e is the
    dequantised index key shared by all indexer heads. The dot products are taken in fp64 and rounded to
    fp32 (exact for the integer-valued inputs used throughout); the weighted head sum is taken in fp32 in
    that fixed order, and -0 is made +0.
  * query rounding (a separate step, `round_query`): before scoring, the selection calls
    (`flat_topk`, `hierarchical_topk`) round every indexer query to the cache's FP4 format with the POW2
    scale rule (one power-of-two scale per 16 elements), q^_h = dequant(quant_pow2(q_h)), and score with
    q^_h. This is part of the indexer call's contract, because its product takes both operands in FP4.
    For integer-valued queries in [-4, 4] the rounding is the identity.
  * a block's score is the maximum over its eligible entries; a block with no eligible entry is not a
    candidate (score -inf here).
  * Top-K: the min(K, #candidates) candidates with the largest scores, ties to the lower block id,
    listed in ascending block id and padded with -1.
  * hierarchical: super-block g covers blocks [64 g, 64 g + 64); its coarse key is the sum of the
    dequantised keys of its entries below n_entries, taken exactly and rounded once to fp32; super-blocks are
    scored with the same score function, the best keep_blocks / 64 are kept (ties to the lower id), and
    the block Top-K runs over their blocks only.
"""

import numpy as np

from . import fp4

BLOCK = 8
SUPER = 64
ENTRIES_PER_SUPER = BLOCK * SUPER


def round_query(q):
    """The indexer query as the selection calls score it: every group of 16 elements rounded to FP4 with
    the POW2 scale rule and dequantised (float32, same shape). The identity on integers in [-4, 4]."""
    return fp4.round_trip(np.asarray(q, dtype=np.float32), "pow2")


def entry_scores(q, keys, head_w=None, relu=True):
    """q: [Q, H, D] indexer queries, keys: [n_e, D] dequantised keys. Returns float32 [Q, n_e]:
    s_e = sum_h fl32(w_h * max(0, q_h . k_e)) in head order (no rounding of q here)."""
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    nq, nh, d = q.shape
    w = np.ones(nh, np.float32) if head_w is None else np.asarray(head_w, np.float32)
    dots = (q.reshape(nq * nh, d) @ keys.T).reshape(nq, nh, keys.shape[0])
    r = np.maximum(dots, 0.0) if relu else dots
    r32 = r.astype(np.float32)
    s = w[0] * r32[:, 0, :]
    for h in range(1, nh):
        s = s + w[h] * r32[:, h, :]
    return (s + np.float32(0.0)).astype(np.float32)


def block_scores(s, eligible):
    """s: float32 [Q, n_e]; eligible: bool [Q, n_e]. Returns float32 [Q, ceil(n_e / 8)], -inf where
    a block has no eligible entry."""
    nq, n_e = s.shape
    n_b = -(-n_e // BLOCK)
    v = np.full((nq, n_b * BLOCK), -np.inf, np.float32)
    v[:, :n_e] = np.where(eligible, s, -np.inf)
    return v.reshape(nq, n_b, BLOCK).max(axis=-1)


def eligibility(n_entries, n_e_total, q_pos=None):
    """bool [Q, n_e_total]: e < n_entries, and 2e + 1 <= p for prefill positions p."""
    e = np.arange(n_e_total)
    if q_pos is None:
        return (e < n_entries)[None, :]
    q_pos = np.asarray(q_pos, np.int64)
    return (e[None, :] < n_entries) & (2 * e[None, :] + 1 <= q_pos[:, None])


def topk(scores, k):
    """scores: float32 [n] with -inf for non-candidates. Returns int32 [k]: ascending ids of the
    chosen candidates (largest score first, ties to the lower id), padded with -1."""
    scores = np.asarray(scores, np.float32)
    cand = np.nonzero(scores != -np.inf)[0]
    order = np.lexsort((cand, -scores[cand].astype(np.float64)))
    chosen = np.sort(cand[order[:k]])
    out = np.full(k, -1, np.int32)
    out[:len(chosen)] = chosen
    return out


def flat_topk(q, keys, n_entries, k, head_w=None, relu=True, q_pos=None):
    """Index + Top-K for one sequence. q: [Q, H, D]; keys: dequantised [n_cap, D] (entries beyond
    n_entries are ignored). The queries are rounded by `round_query` first. Returns (idx int32 [Q, k],
    block scores float32 [Q, n_b])."""
    s = entry_scores(round_query(q), keys, head_w, relu)
    el = eligibility(n_entries, keys.shape[0], q_pos)
    el = np.broadcast_to(el, s.shape)
    S = block_scores(s, el)
    idx = np.stack([topk(S[j], k) for j in range(S.shape[0])])
    return idx, S


def coarse_keys(keys, n_entries):
    """Super-block coarse keys: float32 [ceil(n_entries / 512), D], each the sum of the dequantised keys of
    its entries below n_entries ([card] Key ideas, hierarchical indexer; the summary is this library's
    reading), taken exactly and rounded once to fp32. Dequantised FP4 keys are multiples of 2^-13 below
    2,688 in magnitude, so the fp64 sum of a super-block (at most 512 of them) is exact."""
    keys = np.asarray(keys, np.float64)[:n_entries]
    n_super = -(-n_entries // ENTRIES_PER_SUPER)
    d = keys.shape[1]
    padded = np.zeros((n_super * ENTRIES_PER_SUPER, d), np.float64)
    padded[:n_entries] = keys
    return padded.reshape(n_super, ENTRIES_PER_SUPER, d).sum(axis=1).astype(np.float32)


def hierarchical_topk(q, keys, n_entries, k, keep_blocks, head_w=None, relu=True, coarse=None):
    """Two-stage selection for one sequence (decode). q: [Q, H, D]; keys: dequantised [n_cap, D].
    The queries are rounded by `round_query` first, for both stages. Returns (idx int32 [Q, k], kept
    super-block ids int32 [Q, keep_blocks // 64])."""
    q = round_query(q)
    if coarse is None:
        coarse = coarse_keys(keys, n_entries)
    n_super = coarse.shape[0]
    keep_super = keep_blocks // SUPER
    cs = entry_scores(q, coarse, head_w, relu)                       # [Q, n_super]
    s = entry_scores(q, keys, head_w, relu)
    el = np.broadcast_to(eligibility(n_entries, keys.shape[0]), s.shape)
    S = block_scores(s, el)                                          # [Q, n_b]
    idx_all, kept_all = [], []
    for j in range(q.shape[0]):
        c = cs[j].copy()
        c[np.arange(n_super) * ENTRIES_PER_SUPER >= n_entries] = -np.inf
        kept = topk(c, keep_super)
        restricted = np.full(S.shape[1], -np.inf, np.float32)
        for g in kept[kept >= 0]:
            lo, hi = g * SUPER, min((g + 1) * SUPER, S.shape[1])
            restricted[lo:hi] = S[j, lo:hi]
        idx_all.append(topk(restricted, k))
        kept_all.append(kept)
    return np.stack(idx_all), np.stack(kept_all)
