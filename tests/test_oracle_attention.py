"""Pins for oracle.attention and oracle.chain: closed forms of softmax attention and the invariants
the method fixes (Top-K covering every block equals dense attention; Reuse layers reproduce their
source layer's indices)."""

import math

import numpy as np

from oracle import attention, chain, fp4, indexer


def test_two_row_closed_form():
    # rows e0 and e1, q = ln(3) e0, scale 1: softmax = (3/4, 1/4), out = (3/4, 1/4, 0, ...)
    d = 8
    rows = np.eye(2, d)
    q = np.zeros((1, d))
    q[0, 0] = math.log(3.0)
    out, lse = attention.attend(q, rows, 1.0)
    np.testing.assert_allclose(out[0, :2], [0.75, 0.25], rtol=0, atol=1e-15)
    assert np.all(out[0, 2:] == 0)
    assert abs(lse[0] - math.log(4.0)) < 1e-15
    # the scale multiplies the logits: q = 4 ln(3) e0 with scale 1/4 gives the same weights, and
    # lse = log(e^{ln 3} + e^0)
    q[0, 0] = 4 * math.log(3.0)
    out, lse = attention.attend(q, rows, 0.25)
    np.testing.assert_allclose(out[0, :2], [0.75, 0.25], rtol=0, atol=1e-15)
    assert abs(lse[0] - math.log(4.0)) < 1e-15


def test_zero_query_gives_mean_and_log_count():
    rng = np.random.default_rng(0)
    rows = rng.standard_normal((37, 16))
    out, lse = attention.attend(np.zeros((3, 16)), rows, 0.1)
    np.testing.assert_allclose(out, np.broadcast_to(rows.mean(0), (3, 16)), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(37), rtol=0, atol=1e-14)


def test_dominant_row_and_no_rows():
    rows = np.zeros((5, 4))
    rows[2] = [1.0, 2.0, 3.0, 4.0]
    q = np.array([[1000.0, 0, 0, 0]])
    out, _ = attention.attend(q, rows, 1.0)
    np.testing.assert_allclose(out[0], rows[2], rtol=0, atol=1e-12)
    out, lse = attention.attend(q, np.zeros((0, 4)), 1.0)
    assert np.all(out == 0) and lse[0] == -np.inf


def test_attend_equals_torch_sdpa_in_fp64():
    # torch's scaled-dot-product attention (its CPU math path, fp64) is an implementation independent of
    # the oracle; each row serves as both key and value, and the log-sum-exp comes from torch.logsumexp
    import torch
    rng = np.random.default_rng(5)
    for n, d, h, scale in ((1, 8, 1, 1.0), (37, 64, 4, 0.125), (300, 512, 16, 1 / math.sqrt(512))):
        rows = rng.standard_normal((n, d)) * 3
        q = rng.standard_normal((h, d)) * 2
        out, lse = attention.attend(q, rows, scale)
        tq = torch.from_numpy(q)[None, None]
        tr = torch.from_numpy(rows)[None, None]
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tr, tr, scale=scale)[0, 0].numpy()
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
        ref_lse = torch.logsumexp(torch.from_numpy(q) @ torch.from_numpy(rows).T * scale, dim=-1).numpy()
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-13, atol=1e-13)


def test_row_permutation_invariance():
    rng = np.random.default_rng(1)
    rows = rng.standard_normal((50, 32))
    q = rng.standard_normal((4, 32))
    a, la = attention.attend(q, rows, 0.3)
    b, lb = attention.attend(q, rows[rng.permutation(50)], 0.3)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(la, lb, rtol=1e-13)


def _cache(rng, n_tokens, dim=512):
    x = rng.standard_normal((n_tokens, dim)).astype(np.float32)
    blocks = fp4.pack(x, 2, "amax")
    n_e = n_tokens // 2
    return fp4.dequantize(blocks, dim, n_e), n_e


def test_topk_covering_every_block_equals_dense():
    rng = np.random.default_rng(2)
    entries, n_e = _cache(rng, 2 * 77)                # 77 entries -> 10 blocks, last one ragged
    swa = rng.standard_normal((19, 512))
    q = rng.standard_normal((8, 512))
    idx = np.array(list(range(9, -1, -1)) + [-1, -1])  # every block, any order, padded
    a, la = attention.decode_attention(q, entries, n_e, idx, swa, 1 / math.sqrt(512))
    b, lb = attention.dense_attention(q, entries, n_e, swa, 1 / math.sqrt(512))
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(la, lb, rtol=1e-12)


def test_selected_rows_respect_eligibility():
    entries = np.arange(20 * 4, dtype=np.float64).reshape(20, 4)
    el = np.arange(20) < 13
    rows = attention.selected_rows(entries, [1, -1, 0], el)
    assert [int(r[0]) // 4 for r in rows] == [8, 9, 10, 11, 12, 0, 1, 2, 3, 4, 5, 6, 7]


def test_prefill_window_rows():
    swa = np.arange(300, dtype=np.float64)[:, None] * np.ones((1, 4))
    w = attention.prefill_window(swa, 1000, 1200, 128)
    assert w.shape[0] == 128 and w[0, 0] == 1200 - 127 - 1000 and w[-1, 0] == 200
    w = attention.prefill_window(swa, 1000, 1005, 128)
    assert w.shape[0] == 6 and w[0, 0] == 0


def test_chain_modes_and_reuse_indices():
    m = chain.modes(20, 4)
    assert m.count(chain.FULL) == 1 and m.count(chain.REINDEX) == 4 and m.count(chain.REUSE) == 15
    src = chain.index_sources(m)
    assert src[:9] == [0, 0, 0, 0, 4, 4, 4, 4, 8] and src[19] == 16
    # running the chain: Reuse layers attend with exactly their source layer's indices
    rng = np.random.default_rng(3)
    keys = rng.integers(-4, 5, (400, 64)).astype(np.float32)
    per_layer_idx = {}
    for layer, mode in enumerate(m):
        if mode == chain.REUSE:
            per_layer_idx[layer] = per_layer_idx[src[layer]]
        else:
            q = rng.integers(-4, 5, (1, 1, 64))
            per_layer_idx[layer] = indexer.flat_topk(q, keys, 400, 8)[0]
    for layer, mode in enumerate(m):
        np.testing.assert_array_equal(per_layer_idx[layer], per_layer_idx[src[layer]])
    assert not np.array_equal(per_layer_idx[0], per_layer_idx[4])     # Reindex really rescored


def _row_count(lse):
    # with a zero query every logit is 0, so lse = log(number of rows)
    return int(round(math.exp(lse)))


def test_prefill_rows_counted_by_hand():
    # a hand-built cache of 20 entries (3 blocks, all listed) whose entry e holds the value e + 1 in every
    # column, and a window buffer that starts at token 0 with rows of zeros. At position p the entries
    # with 2e + 1 <= p are 0 .. floor((p - 1) / 2), i.e. floor((p + 1) / 2) of them, and the window has
    # the p + 1 rows of tokens 0 .. p (p < 128):
    #   p:        0  1  2  15  16  17
    #   entries:  0  1  1   8   8   9
    #   window:   1  2  3  16  17  18
    #   rows:     1  3  4  24  25  27
    entries = (np.arange(20, dtype=np.float64)[:, None] + 1) * np.ones((1, 16))
    swa = np.zeros((200, 16))
    q = np.zeros((2, 16))
    idx = np.array([2, 0, 1, -1])
    for p, n_ent, n_rows in [(0, 0, 1), (1, 1, 3), (2, 1, 4), (15, 8, 24), (16, 8, 25), (17, 9, 27)]:
        out, lse = attention.prefill_attention(q, entries, 20, idx, swa, 0, p, 128, 0.5)
        assert _row_count(lse[0]) == n_rows and _row_count(lse[1]) == n_rows
        # the output is the mean of the rows: sum of (e + 1) over the visible entries / rows
        want = sum(e + 1 for e in range(n_ent)) / n_rows
        np.testing.assert_allclose(out, want, rtol=0, atol=1e-14)
    # n_entries still bounds the visible entries at late positions, and the window keeps its last 128
    out, lse = attention.prefill_attention(q, entries, 13, idx, swa, 0, 199, 128, 0.5)
    assert _row_count(lse[0]) == 13 + 128
    np.testing.assert_allclose(out, sum(range(1, 14)) / (13 + 128), rtol=0, atol=1e-14)


def test_prefill_equals_decode_once_every_entry_is_visible():
    # at a position p >= 2 n_entries - 1 every entry below n_entries is visible, so the causal query equals
    # the decode query over the same blocks with the window rows of tokens p - 127 .. p
    rng = np.random.default_rng(4)
    entries, n_e = _cache(rng, 2 * 90)                # 90 entries, 12 blocks (the last ragged)
    swa = rng.standard_normal((1000, 512))
    first = 10                                        # token of window row 0; p - 127 >= first below
    q = rng.standard_normal((4, 512))
    idx = np.array([11, 3, -1, 7, 0, 5])
    scale = 1 / math.sqrt(512)
    for p in (2 * n_e - 1, 2 * n_e + 40, 900):
        a, la = attention.prefill_attention(q, entries, n_e, idx, swa, first, p, 128, scale)
        b, lb = attention.decode_attention(q, entries, n_e, idx, swa[p - 127 - first:p + 1 - first], scale)
        np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(la, lb, rtol=1e-13)
    # one position earlier the last entry (2e + 1 = 2 n_e - 1 > p) drops out, so the two differ
    p = 2 * n_e - 2
    a, _ = attention.prefill_attention(q, entries, n_e, np.array([11]), swa, first, p, 128, scale)
    b, _ = attention.decode_attention(q, entries, n_e, np.array([11]), swa[p - 127 - first:p + 1 - first], scale)
    assert not np.allclose(a, b)
