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
