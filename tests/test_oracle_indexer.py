"""Pins for oracle.indexer: integer brute force, brute-force Top-K, and the hierarchy's reduction to
flat selection."""

import itertools
import math

import numpy as np

from oracle import fp4, indexer


def _int_scores(q, k, w, relu):
    # int64 brute force, independent of the oracle's fp64 matmul and fp32 head sum
    nq, nh, d = q.shape
    out = np.zeros((nq, k.shape[0]), np.int64)
    for j in range(nq):
        for h in range(nh):
            dot = (q[j, h][None, :].astype(np.int64) * k.astype(np.int64)).sum(axis=1)
            out[j] += w[h] * (np.maximum(dot, 0) if relu else dot)
    return out


def test_entry_scores_match_integer_brute_force():
    rng = np.random.default_rng(1)
    for nh, d, relu in [(4, 128, True), (1, 64, True), (2, 64, False), (8, 128, True)]:
        q = rng.integers(-4, 5, (3, nh, d))
        k = rng.integers(-4, 5, (257, d))
        w = rng.integers(0, 4, nh)
        got = indexer.entry_scores(q, k, w.astype(np.float32), relu)
        np.testing.assert_array_equal(got.astype(np.int64), _int_scores(q, k, w, relu))
        assert not np.any(np.signbit(got) & (got == 0))           # no negative zeros


def test_scores_from_packed_keys_are_exact():
    rng = np.random.default_rng(2)
    q = rng.integers(-4, 5, (2, 4, 128))
    k = rng.integers(-4, 5, (100, 128)).astype(np.float32)
    deq = fp4.dequantize(fp4.pack(k, 1, "pow2"), 128, 100)
    got = indexer.entry_scores(q, deq)
    np.testing.assert_array_equal(got.astype(np.int64), _int_scores(q, k.astype(np.int64), [1] * 4, True))


def _brute_topk(scores, k):
    cand = [(float(s), i) for i, s in enumerate(scores) if s != -np.inf]
    cand.sort(key=lambda t: (-t[0], t[1]))
    chosen = sorted(i for _, i in cand[:k])
    return chosen + [-1] * (k - len(chosen))


def test_topk_matches_brute_force_sort():
    rng = np.random.default_rng(3)
    for trial in range(400):
        n = int(rng.integers(1, 65))
        kind = trial % 4
        if kind == 0:
            s = rng.integers(0, 4, n).astype(np.float32)          # heavy ties
        elif kind == 1:
            s = np.zeros(n, np.float32)                           # all equal
        elif kind == 2:
            s = rng.standard_normal(n).astype(np.float32)
        else:
            s = rng.integers(-2, 3, n).astype(np.float32)
            s[rng.random(n) < 0.3] = -np.inf                      # non-candidates
        k = int(rng.integers(1, 70))
        assert indexer.topk(s, k).tolist() == _brute_topk(s, k)


def test_topk_treats_signed_zeros_as_equal():
    s = np.array([-0.0, 0.0, -0.0, 0.0], np.float32)
    assert indexer.topk(s, 2).tolist() == [0, 1]


def test_block_scores_and_eligibility():
    s = np.arange(20, dtype=np.float32)[None, :]
    el = indexer.eligibility(13, 20)
    S = indexer.block_scores(s, el)
    np.testing.assert_array_equal(S, [[7, 12, -np.inf]])
    # prefill: entry e visible at token p iff 2e + 1 <= p
    el = indexer.eligibility(20, 20, q_pos=[0, 1, 2, 16, 17])
    assert el[0].sum() == 0 and el[1].sum() == 1 and el[2].sum() == 1
    assert el[3].sum() == 8 and el[4].sum() == 9


def test_hierarchical_with_everything_kept_equals_flat():
    rng = np.random.default_rng(4)
    for n_e in [512 * 5, 512 * 3 + 77, 200]:
        k = rng.integers(-4, 5, (n_e, 64)).astype(np.float32)
        q = rng.integers(-4, 5, (1, 4, 64))
        n_super = -(-n_e // 512)
        flat, _ = indexer.flat_topk(q, k, n_e, 16)
        hier, kept = indexer.hierarchical_topk(q, k, n_e, 16, keep_blocks=64 * n_super)
        np.testing.assert_array_equal(hier, flat)
        assert sorted(kept[0][kept[0] >= 0].tolist()) == list(range(n_super))


def test_hierarchical_restricts_to_kept_super_blocks():
    rng = np.random.default_rng(5)
    n_e = 512 * 8
    k = rng.integers(-1, 2, (n_e, 64)).astype(np.float32)
    q = np.ones((1, 1, 64), np.int64)
    k[512 * 5:512 * 6] = 4          # super-block 5 has the largest coarse key and every top entry
    k[512 * 2:512 * 3] = 3
    idx, kept = indexer.hierarchical_topk(q, k, n_e, 32, keep_blocks=64)
    assert kept[0].tolist() == [5]
    assert idx[0].tolist() == list(range(5 * 64, 5 * 64 + 32))
    idx2, kept2 = indexer.hierarchical_topk(q, k, n_e, 100, keep_blocks=128)
    assert kept2[0].tolist() == [2, 5]
    assert set(idx2[0].tolist()) <= set(range(128, 192)) | set(range(320, 384))


def test_coarse_keys_per_super_block():
    k = np.ones((1100, 8), np.float32)
    c = indexer.coarse_keys(k, 1100)
    np.testing.assert_array_equal(c[:, 0], [512, 512, 76])
    for a, b in itertools.product(range(2), range(2)):
        assert c[a, b] == 512


def test_coarse_keys_are_exact_sums_rounded_once():
    # 342 keys of 1536 (code 6 x scale 2^8) then 170 of 2^-5 (code 0.5 x 2^-4): a sum in entry order in fp32
    # loses every 2^-5 (half an ulp at 525,312, a tie that rounds to even), the exact sum keeps them
    k = np.zeros((512, 2), np.float32)
    k[:342] = 1536.0
    k[342:] = 2.0 ** -5
    c = indexer.coarse_keys(k, 512)
    assert c[0, 0] == np.float32(525312 + 170 * 2.0 ** -5)
    ordered = np.float32(0)
    for v in k[:, 0]:
        ordered = np.float32(ordered + v)
    assert ordered == np.float32(525312) != c[0, 0]


def test_coarse_keys_match_an_exactly_rounded_sum():
    # against Python's math.fsum (an exactly rounded sum), on dequantised FP4 keys of every magnitude
    rng = np.random.default_rng(13)
    x = rng.standard_normal((1100, 16)).astype(np.float32) * np.exp2(rng.integers(-12, 9, (1100, 1)))
    deq = fp4.dequantize(fp4.pack(x, 1, "pow2"), 16, 1100)
    c = indexer.coarse_keys(deq, 1100)
    for g in range(3):
        rows = deq[512 * g:min(512 * g + 512, 1100)]
        want = [np.float32(math.fsum(rows[:, j])) for j in range(16)]
        np.testing.assert_array_equal(c[g], want)


def test_query_rounding_is_identity_on_small_integers():
    # every integer in [-4, 4] survives the POW2 FP4 rounding, whatever the group's maximum magnitude
    rng = np.random.default_rng(11)
    for a in range(0, 5):
        for _ in range(200):
            g = rng.integers(-a, a + 1, 16).astype(np.float32)
            if a:
                g[rng.integers(16)] = a * (1 if rng.random() < 0.5 else -1)
            np.testing.assert_array_equal(indexer.round_query(g[None, None])[0, 0], g)


def test_query_rounding_hand_worked():
    # amax 5 -> 5/6 -> scale 1; 5 lies halfway between 4 (code 6) and 6 (code 7): ties go to the even code
    # amax 7 -> 7/6 -> scale 2; 7/2 = 3.5 lies halfway between 3 (code 5) and 4 (code 6) -> 4 -> 8
    # amax 0.3 -> 0.05 -> scale 2^-4; 0.3 / 2^-4 = 4.8 -> nearest grid value 4 -> 0.25
    for v, want in [(5.0, 4.0), (-5.0, -4.0), (7.0, 8.0), (0.3, 0.25)]:
        g = np.zeros((1, 1, 32), np.float32)
        g[0, 0, 3] = v
        g[0, 0, 16 + 5] = 1.0                         # the second group of 16 has its own scale
        out = indexer.round_query(g)[0, 0]
        assert out[3] == want and out[21] == 1.0
        assert np.all(np.delete(out, [3, 21]) == 0)


def test_entry_scores_do_not_round_the_query():
    # the plain score definition takes the query as given: 5s score as 5s (integer brute force)
    rng = np.random.default_rng(12)
    k = rng.integers(-4, 5, (64, 64))
    q = np.full((1, 1, 64), 5.0, np.float32)
    got = indexer.entry_scores(q, k)
    np.testing.assert_array_equal(got.astype(np.int64), _int_scores(np.full((1, 1, 64), 5), k, [1], True))


def test_selection_scores_the_rounded_query():
    # flat and hierarchical selection score with round_query(q): a query of 5s is rounded to 4s, so it
    # selects exactly like a query of 4s and its block scores equal the integer brute force of the 4s
    # query (a selection that skipped the rounding would report scores 5/4 as large)
    rng = np.random.default_rng(13)
    n_e = 512 * 3
    k = rng.integers(-4, 5, (n_e, 64)).astype(np.float32)
    q5 = np.full((1, 1, 64), 5.0, np.float32)
    q4 = np.full((1, 1, 64), 4.0, np.float32)
    a5, S5 = indexer.flat_topk(q5, k, n_e, 24)
    a4, S4 = indexer.flat_topk(q4, k, n_e, 24)
    np.testing.assert_array_equal(a5, a4)
    np.testing.assert_array_equal(S5, S4)
    h5, kept5 = indexer.hierarchical_topk(q5, k, n_e, 24, keep_blocks=128)
    h4, kept4 = indexer.hierarchical_topk(q4, k, n_e, 24, keep_blocks=128)
    np.testing.assert_array_equal(h5, h4)
    np.testing.assert_array_equal(kept5, kept4)
    # with rounding, block scores are the integer brute force of the rounded query
    s_int = _int_scores(np.full((1, 1, 64), 4), k.astype(np.int64), [1], True)
    el = np.arange(n_e) < n_e
    want = np.where(el, s_int[0], np.iinfo(np.int64).min).reshape(-1, 8).max(axis=1)
    np.testing.assert_array_equal(S5[0].astype(np.int64), want)
