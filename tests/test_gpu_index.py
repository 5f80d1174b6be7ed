"""csa_index_topk against the oracle: bit-exact block scores and Top-K indices (flat, prefill-causal,
hierarchical), ties, head weights, the no-ReLU form and more slots than candidates."""

import numpy as np
import pytest
import torch

from oracle import fp4 as o_fp4
from oracle import indexer as o_idx

from _pipeline import gpu_index, gpu_pack_sequences

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa():
    from compressed_sparse_attention_merge_b300 import binding
    binding.lib()
    return binding


def _keys(g, B, E, dim, zero_frac=0.0):
    k = torch.randint(-4, 5, (B, E, dim), generator=g, device=DEV).float()
    if zero_frac:
        k = torch.where(torch.rand(B, E, 1, generator=g, device=DEV) < zero_frac, 0.0, k)
    return k


@pytest.mark.parametrize("heads,dim,top_k,nq", [(4, 128, 32, 1), (1, 64, 64, 1), (2, 64, 16, 3),
                                                 (8, 256, 24, 1), (4, 128, 300, 2), (1, 64, 5, 9)])
def test_flat_topk_bit_exact(csa, heads, dim, top_k, nq):
    g = torch.Generator(device=DEV).manual_seed(10 + heads * dim + top_k)
    lengths = [1000, 37, 1024, 0]
    B, E = len(lengths), max(lengths)
    keys = _keys(g, B, E, dim, zero_frac=0.3)
    q_idx = torch.randint(-4, 5, (B, nq, heads, dim), generator=g, device=DEV).float()
    ws = csa.workspace(256, DEV)
    kc = gpu_pack_sequences(csa, keys, lengths, E, dim, 1, csa.SCALE_POW2, ws)
    n_entries = torch.tensor(lengths, dtype=torch.int32, device=DEV)
    idx, scores = gpu_index(csa, q_idx, kc, n_entries, E, top_k, want_scores=True)
    idx, scores = idx.cpu().numpy(), scores.cpu().numpy()
    kcpu, qcpu = keys.cpu().numpy(), q_idx.cpu().numpy()
    for b, n in enumerate(lengths):
        deq = o_fp4.dequantize(o_fp4.pack(kcpu[b, :n], 1, "pow2", n_blocks=-(-E // 8)), dim, E) if n else \
            np.zeros((E, dim))
        ref_idx, ref_S = o_idx.flat_topk(qcpu[b], deq, n, top_k)
        np.testing.assert_array_equal(idx[b], ref_idx, err_msg=f"seq {b}")
        nb = ref_S.shape[1]
        np.testing.assert_array_equal(scores[b, :, :nb], ref_S, err_msg=f"scores seq {b}")
        assert np.all(scores[b, :, nb:] == -np.inf)


def test_head_weights_and_no_relu(csa):
    g = torch.Generator(device=DEV).manual_seed(21)
    B, E, dim, heads = 2, 777, 128, 4
    keys = _keys(g, B, E, dim)
    q_idx = torch.randint(-4, 5, (B, 1, heads, dim), generator=g, device=DEV).float()
    w = torch.tensor([1.0, 0.5, 2.0, 0.25], device=DEV)
    ws = csa.workspace(256, DEV)
    kc = gpu_pack_sequences(csa, keys, [E, E], E, dim, 1, csa.SCALE_POW2, ws)
    n_entries = torch.tensor([E, E], dtype=torch.int32, device=DEV)
    for relu in (True, False):
        idx, scores = gpu_index(csa, q_idx, kc, n_entries, E, 40, head_w=w, relu=relu, want_scores=True)
        for b in range(B):
            deq = o_fp4.dequantize(o_fp4.pack(keys[b].cpu().numpy(), 1, "pow2"), dim, E)
            ref_idx, ref_S = o_idx.flat_topk(q_idx[b].cpu().numpy(), deq, E, 40, head_w=w.cpu().numpy(),
                                             relu=relu)
            np.testing.assert_array_equal(idx[b].cpu().numpy(), ref_idx)
            np.testing.assert_array_equal(scores[b].cpu().numpy()[:, :ref_S.shape[1]], ref_S)


def test_all_ties_pick_lowest_ids(csa):
    B, E, dim = 1, 800, 64
    keys = torch.zeros(B, E, dim, device=DEV)
    q_idx = torch.ones(B, 1, 1, dim, device=DEV)
    ws = csa.workspace(256, DEV)
    kc = gpu_pack_sequences(csa, keys, [E], E, dim, 1, csa.SCALE_POW2, ws)
    idx, _ = gpu_index(csa, q_idx, kc, torch.tensor([E], dtype=torch.int32, device=DEV), E, 7)
    assert idx[0, 0].tolist() == list(range(7))


def test_prefill_causal_positions(csa):
    g = torch.Generator(device=DEV).manual_seed(31)
    E, dim, heads, Q = 1500, 128, 4, 37
    keys = _keys(g, 1, E, dim)
    q_idx = torch.randint(-4, 5, (1, Q, heads, dim), generator=g, device=DEV).float()
    pos = torch.cat([torch.tensor([0, 1, 2, 15, 16, 17]), torch.randint(0, 2 * E + 10, (Q - 6,))]).to(torch.int32)
    q_pos = pos[None, :].to(DEV)
    ws = csa.workspace(256, DEV)
    kc = gpu_pack_sequences(csa, keys, [E], E, dim, 1, csa.SCALE_POW2, ws)
    idx, scores = gpu_index(csa, q_idx, kc, torch.tensor([E], dtype=torch.int32, device=DEV), E, 20,
                            q_pos=q_pos, want_scores=True)
    deq = o_fp4.dequantize(o_fp4.pack(keys[0].cpu().numpy(), 1, "pow2"), dim, E)
    ref_idx, ref_S = o_idx.flat_topk(q_idx[0].cpu().numpy(), deq, E, 20, q_pos=pos.numpy())
    np.testing.assert_array_equal(idx[0].cpu().numpy(), ref_idx)
    np.testing.assert_array_equal(scores[0].cpu().numpy()[:, :ref_S.shape[1]], ref_S)


@pytest.mark.parametrize("keep_blocks,top_k", [(192, 50), (64, 64), (4096, 40)])
def test_hierarchical_bit_exact(csa, keep_blocks, top_k):
    g = torch.Generator(device=DEV).manual_seed(41 + keep_blocks)
    lengths = [512 * 9 + 100, 512 * 2 + 3]
    B, E, dim = 2, max(lengths), 128
    keys = _keys(g, B, E, dim)
    # a few super-blocks with large keys, so that the coarse stage has a clear choice
    keys[0, 512 * 4:512 * 5] = 4.0
    keys[0, 512 * 7:512 * 7 + 40] = 3.0
    q_idx = torch.ones(B, 1, 4, dim, device=DEV)
    q_idx[:, :, 1:] = torch.randint(-4, 5, (B, 1, 3, dim), generator=g, device=DEV).float()
    ws = csa.workspace(256, DEV)
    coarse = csa.empty_coarse(B, E, dim, DEV)
    kc = gpu_pack_sequences(csa, keys, lengths, E, dim, 1, csa.SCALE_POW2, ws, coarse=coarse)
    n_entries = torch.tensor(lengths, dtype=torch.int32, device=DEV)
    idx, _ = gpu_index(csa, q_idx, kc, n_entries, E, top_k, coarse=coarse, keep_blocks=keep_blocks)
    for b, n in enumerate(lengths):
        deq = o_fp4.dequantize(o_fp4.pack(keys[b, :n].cpu().numpy(), 1, "pow2", n_blocks=-(-E // 8)), dim, E)
        ref_idx, _ = o_idx.hierarchical_topk(q_idx[b].cpu().numpy(), deq, n, top_k, keep_blocks)
        np.testing.assert_array_equal(idx[b].cpu().numpy(), ref_idx, err_msg=f"seq {b}")
        if keep_blocks >= 64 * (-(-n // 512)):
            flat, _ = o_idx.flat_topk(q_idx[b].cpu().numpy(), deq, n, top_k)
            np.testing.assert_array_equal(idx[b].cpu().numpy(), flat)


def test_off_grid_queries_are_rounded_like_the_oracle(csa):
    # queries outside the E2M1 grid (5, 7, fractions): both sides round them to FP4 with the POW2 rule
    g = torch.Generator(device=DEV).manual_seed(51)
    B, E, dim, heads = 2, 900, 128, 4
    keys = _keys(g, B, E, dim)
    vals = torch.tensor([5.0, -5.0, 7.0, 0.3, -0.75, 2.5, 1.0, 0.0], device=DEV)
    q_idx = vals[torch.randint(0, 8, (B, 1, heads, dim), generator=g, device=DEV)]
    ws = csa.workspace(256, DEV)
    kc = gpu_pack_sequences(csa, keys, [E, E - 13], E, dim, 1, csa.SCALE_POW2, ws)
    n_entries = torch.tensor([E, E - 13], dtype=torch.int32, device=DEV)
    idx, scores = gpu_index(csa, q_idx, kc, n_entries, E, 30, want_scores=True)
    for b, n in enumerate([E, E - 13]):
        deq = o_fp4.dequantize(o_fp4.pack(keys[b, :n].cpu().numpy(), 1, "pow2"), dim, n)
        ref_idx, ref_S = o_idx.flat_topk(q_idx[b].cpu().numpy(), deq, n, 30)
        np.testing.assert_array_equal(idx[b].cpu().numpy(), ref_idx)
        np.testing.assert_array_equal(scores[b].cpu().numpy()[:, :ref_S.shape[1]], ref_S)
