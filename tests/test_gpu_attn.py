"""csa_sparse_attn_decode / csa_sparse_attn_prefill against the fp64 oracle (max-abs 2e-3, max-rel 1e-2),
split-K against no split, empty and invalid inputs."""

import math

import numpy as np
import pytest
import torch

from oracle import attention as o_attn
from oracle import fp4 as o_fp4
from oracle import indexer as o_idx

from _pipeline import (SCALE, assert_attn_close, assert_lse_close, gpu_decode_attn, gpu_index, gpu_pack_sequences,
                       gpu_prefill_attn, to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa():
    from compressed_sparse_attention_merge_b300 import binding
    binding.lib()
    return binding


def _latents(g, B, T, outliers=0.01):
    x = torch.randn(B, T, 512, generator=g, device=DEV)
    x = torch.where(torch.rand(B, T, 512, generator=g, device=DEV) < outliers, x * 8, x)
    return x.to(torch.bfloat16)


def _random_idx(rng, n_b_list, B, Q, K, cap_blocks):
    idx = np.full((B, Q, K), -1, np.int32)
    for b in range(B):
        for j in range(Q):
            nb = n_b_list[b]
            k = min(K, nb)
            take = rng.choice(max(nb, 1), size=k, replace=False) if nb else np.zeros(0, np.int64)
            idx[b, j, :k] = take
            # a legal id past this sequence's valid blocks (inside capacity): must be ignored
            if k < K and nb < cap_blocks:
                idx[b, j, k] = cap_blocks - 1
    return idx


@pytest.mark.parametrize("heads,top_k,batch", [(64, 24, 3), (16, 64, 3), (32, 40, 2), (64, 16, 150)])
def test_decode_matches_oracle(csa, heads, top_k, batch):
    g = torch.Generator(device=DEV).manual_seed(100 + heads + top_k + batch)
    rng = np.random.default_rng(heads * 1000 + top_k + batch)
    base = [2000, 74, 1401, 1]
    tokens = [base[i % 4] + (i // 4) * 2 for i in range(batch)]
    B, T = batch, max(tokens)
    E = T // 2
    W = 128
    x = _latents(g, B, T)
    q = torch.randn(B, 1, heads, 512, generator=g, device=DEV).to(torch.bfloat16)
    swa = torch.randn(B, W, 512, generator=g, device=DEV).to(torch.bfloat16)
    swa_len = torch.tensor([[128, 5, 0, 77][i % 4] for i in range(B)], dtype=torch.int32, device=DEV)
    ws = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, tokens, E, 512, 2, csa.SCALE_AMAX, ws)
    n_e = [t // 2 for t in tokens]
    n_entries = torch.tensor(n_e, dtype=torch.int32, device=DEV)
    idx_np = _random_idx(rng, [-(-n // 8) for n in n_e], B, 1, top_k, -(-E // 8))
    idx = torch.from_numpy(idx_np).to(DEV)
    out, lse = gpu_decode_attn(csa, q, cache, n_entries, idx, swa, swa_len, E, W)
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    xf, qf, sf = to_np(x), to_np(q), to_np(swa)
    check = range(B) if B <= 8 else list(range(4)) + [B - 1]
    for b in check:
        entries = o_fp4.dequantize(o_fp4.pack(xf[b, :tokens[b]], 2, "amax", n_blocks=-(-E // 8)), 512, E)
        ref, ref_lse = o_attn.decode_attention(qf[b, 0].astype(np.float64), entries, n_e[b], idx_np[b, 0],
                                               sf[b, :int(swa_len[b])], SCALE)
        assert_attn_close(out[b, 0], ref, f"seq {b}")
        assert_lse_close(lse[b, 0], ref_lse, f"seq {b}")


def test_multi_query_decode_end_to_end(csa):
    # several independent queries per sequence in one decode call, each with its own indexer query and
    # Top-K; in decode every query sees the whole cache prefix and the same window
    g = torch.Generator(device=DEV).manual_seed(31)
    tokens, B, Q, H, K, W, HI, DI = [1800, 640], 2, 4, 64, 32, 128, 4, 128
    T = max(tokens)
    E = T // 2
    n_e = [t // 2 for t in tokens]
    x = _latents(g, B, T)
    keys = torch.randint(-4, 5, (B, E, DI), generator=g, device=DEV).float()
    q_idx = torch.randint(-4, 5, (B, Q, HI, DI), generator=g, device=DEV).float()
    q = torch.randn(B, Q, H, 512, generator=g, device=DEV).to(torch.bfloat16)
    swa = torch.randn(B, W, 512, generator=g, device=DEV).to(torch.bfloat16)
    swa_len = torch.tensor([W, 60], dtype=torch.int32, device=DEV)
    ws = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, tokens, E, 512, 2, csa.SCALE_AMAX, ws)
    kcache = gpu_pack_sequences(csa, keys, n_e, E, DI, 1, csa.SCALE_POW2, ws)
    n_entries = torch.tensor(n_e, dtype=torch.int32, device=DEV)
    idx, _ = gpu_index(csa, q_idx, kcache, n_entries, E, K)
    out, lse = gpu_decode_attn(csa, q, cache, n_entries, idx, swa, swa_len, E, W)
    idx, out, lse = idx.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy()
    xf, qf, sf, kf, qi = to_np(x), to_np(q), to_np(swa), keys.cpu().numpy(), q_idx.cpu().numpy()
    for b in range(B):
        deq_k = o_fp4.dequantize(o_fp4.pack(kf[b, :n_e[b]], 1, "pow2", n_blocks=-(-E // 8)), DI, E)
        ref_idx, _ = o_idx.flat_topk(qi[b], deq_k, n_e[b], K)
        np.testing.assert_array_equal(idx[b], ref_idx, err_msg=f"seq {b}")
        entries = o_fp4.dequantize(o_fp4.pack(xf[b, :tokens[b]], 2, "amax", n_blocks=-(-E // 8)), 512, E)
        for j in range(Q):
            ref, ref_lse = o_attn.decode_attention(qf[b, j].astype(np.float64), entries, n_e[b], ref_idx[j],
                                                   sf[b, :int(swa_len[b])], SCALE)
            assert_attn_close(out[b, j], ref, f"seq {b} query {j}")
            assert_lse_close(lse[b, j], ref_lse, f"seq {b} query {j}")


@pytest.mark.parametrize("prefix", [1001, 640])
def test_speculative_drafts_are_causal(csa, prefix):
    # multi-token decode for speculative verification: four draft tokens at positions p .. p + 3 follow a
    # prefix of p tokens. Draft j sees the cache entries with 2e + 1 <= p + j and the window tokens
    # p + j - 127 .. p + j. The drafts complete new entries (the pair (p - 1, p) for odd p, then the later
    # pairs), each visible from its completing draft on. All drafts share one indexer query and the new
    # entries' index keys are needles for it, so every draft's Top-K picks them as soon as they are visible.
    g = torch.Generator(device=DEV).manual_seed(41 + prefix)
    B, Q, H, K, W, HI, DI = 2, 4, 64, 24, 128, 4, 128
    T = prefix + Q
    E = T // 2
    x = _latents(g, B, T)
    keys = torch.randint(-4, 5, (B, E, DI), generator=g, device=DEV).float()
    q_idx = torch.randint(-4, 5, (B, 1, HI, DI), generator=g, device=DEV).float().expand(B, Q, HI, DI).contiguous()
    new_first = (prefix - 1) // 2                                   # first entry a draft completes or joins
    for b in range(B):
        keys[b, new_first:E] = 4.0 * torch.sign(q_idx[b, 0, 0])
    q = torch.randn(B, Q, H, 512, generator=g, device=DEV).to(torch.bfloat16)
    first_tok = prefix - W + 1                                      # window buffer: tokens p - 127 .. p + 3
    swa = torch.randn(B, W + Q - 1, 512, generator=g, device=DEV).to(torch.bfloat16)
    swa_first_pos = torch.full((B,), first_tok, dtype=torch.int32, device=DEV)
    q_pos = torch.arange(prefix, prefix + Q, dtype=torch.int32, device=DEV)[None].repeat(B, 1).contiguous()
    ws = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, [T] * B, E, 512, 2, csa.SCALE_AMAX, ws)
    kcache = gpu_pack_sequences(csa, keys, [E] * B, E, DI, 1, csa.SCALE_POW2, ws)
    n_entries = torch.full((B,), E, dtype=torch.int32, device=DEV)
    idx, _ = gpu_index(csa, q_idx, kcache, n_entries, E, K, q_pos=q_pos)
    out, lse = gpu_prefill_attn(csa, q, cache, n_entries, idx, q_pos, swa, swa_first_pos, E, W)
    idx, out, lse = idx.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy()
    xf, qf, sf, kf, qi = to_np(x), to_np(q), to_np(swa), keys.cpu().numpy(), q_idx.cpu().numpy()
    pos = np.arange(prefix, prefix + Q)
    for b in range(B):
        deq_k = o_fp4.dequantize(o_fp4.pack(kf[b], 1, "pow2", n_blocks=-(-E // 8)), DI, E)
        ref_idx, _ = o_idx.flat_topk(qi[b], deq_k, E, K, q_pos=pos)
        np.testing.assert_array_equal(idx[b], ref_idx, err_msg=f"seq {b}")
        entries = o_fp4.dequantize(o_fp4.pack(xf[b], 2, "amax", n_blocks=-(-E // 8)), 512, E)
        seen = []
        for j in range(Q):
            p = int(pos[j])
            ref, ref_lse = o_attn.prefill_attention(qf[b, j].astype(np.float64), entries, E, ref_idx[j], sf[b],
                                                    first_tok, p, W, SCALE)
            assert_attn_close(out[b, j], ref, f"seq {b} draft {j}")
            assert_lse_close(lse[b, j], ref_lse, f"seq {b} draft {j}")
            listed = {8 * int(blk) + s for blk in ref_idx[j] if blk >= 0 for s in range(8)}
            seen.append({e for e in range(new_first, E) if e in listed and 2 * e + 1 <= p})
        # each new entry enters exactly at the draft whose token completes it
        for j in range(Q):
            want = {e for e in range(new_first, E) if 2 * e + 1 <= prefix + j}
            assert seen[j] == want, (j, seen[j], want)
        assert seen[0] != seen[Q - 1]


def test_split_and_unsplit_agree(csa):
    # the same query attended once as a lone sequence (many splits) and inside a batch of 148 (no split)
    g = torch.Generator(device=DEV).manual_seed(7)
    B, T, W, K = 148, 1200, 128, 64
    E = T // 2
    x = _latents(g, 1, T).expand(B, T, 512).contiguous()
    q = torch.randn(1, 1, 64, 512, generator=g, device=DEV).to(torch.bfloat16).expand(B, 1, 64, 512).contiguous()
    swa = torch.randn(1, W, 512, generator=g, device=DEV).to(torch.bfloat16).expand(B, W, 512).contiguous()
    swa_len = torch.full((B,), W, dtype=torch.int32, device=DEV)
    ws = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, [T] * B, E, 512, 2, csa.SCALE_AMAX, ws)
    n_entries = torch.full((B,), E, dtype=torch.int32, device=DEV)
    idx = torch.arange(K, dtype=torch.int32, device=DEV).view(1, 1, K).expand(B, 1, K).contiguous()
    many, lse_many = gpu_decode_attn(csa, q[:1], cache[:1], n_entries[:1], idx[:1], swa[:1], swa_len[:1], E, W)
    one, lse_one = gpu_decode_attn(csa, q, cache, n_entries, idx, swa, swa_len, E, W)
    # Each split rounds its probabilities to fp16 relative to its own running maximum, so the two runs
    # round different numbers (relative error up to 2^-11 per probability) and cannot agree bit for bit.
    # They must agree to half the oracle tolerance; the log-sum-exp is fp32 only and agrees closely.
    assert (many[0] - one[0]).abs().max().item() <= 1e-3
    assert torch.allclose(lse_many[0], lse_one[0], atol=1e-4, rtol=0)
    assert torch.equal(one[0], one[B - 1])


def test_topk_covering_everything_equals_dense(csa):
    g = torch.Generator(device=DEV).manual_seed(8)
    T, W = 2 * 203, 128
    E = T // 2
    x = _latents(g, 1, T)
    q = torch.randn(1, 1, 64, 512, generator=g, device=DEV).to(torch.bfloat16)
    swa = torch.randn(1, W, 512, generator=g, device=DEV).to(torch.bfloat16)
    ws = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, [T], E, 512, 2, csa.SCALE_AMAX, ws)
    nb = -(-E // 8)
    idx = torch.tensor(list(range(nb - 1, -1, -1)) + [-1] * 3, dtype=torch.int32, device=DEV).view(1, 1, -1)
    out, lse = gpu_decode_attn(csa, q, cache, torch.tensor([E], dtype=torch.int32, device=DEV), idx, swa,
                               torch.tensor([W], dtype=torch.int32, device=DEV), E, W)
    entries = o_fp4.dequantize(o_fp4.pack(to_np(x)[0], 2, "amax"), 512, E)
    ref, ref_lse = o_attn.dense_attention(to_np(q)[0, 0].astype(np.float64), entries, E, to_np(swa)[0], SCALE)
    assert_attn_close(out[0, 0].cpu().numpy(), ref)
    assert_lse_close(lse[0, 0].cpu().numpy(), ref_lse)


def test_zero_query_is_mean_of_rows(csa):
    g = torch.Generator(device=DEV).manual_seed(9)
    T, W = 2 * 64, 128
    E = T // 2
    x = _latents(g, 1, T)
    q = torch.zeros(1, 1, 16, 512, dtype=torch.bfloat16, device=DEV)
    swa = torch.randn(1, W, 512, generator=g, device=DEV).to(torch.bfloat16)
    ws = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, [T], E, 512, 2, csa.SCALE_AMAX, ws)
    idx = torch.arange(8, dtype=torch.int32, device=DEV).view(1, 1, 8)
    out, lse = gpu_decode_attn(csa, q, cache, torch.tensor([E], dtype=torch.int32, device=DEV), idx, swa,
                               torch.tensor([10], dtype=torch.int32, device=DEV), E, W)
    entries = o_fp4.dequantize(o_fp4.pack(to_np(x)[0], 2, "amax"), 512, E)
    rows = np.concatenate([entries, to_np(swa)[0, :10]])
    np.testing.assert_allclose(out[0, 0].cpu().numpy(), np.broadcast_to(rows.mean(0), (16, 512)), atol=2e-3)
    np.testing.assert_allclose(lse[0, 0].cpu().numpy(), math.log(rows.shape[0]), atol=1e-4)


def test_no_rows_gives_zero_and_neg_inf(csa):
    E = 64
    cache = csa.empty_cache(1, E, 512, DEV)
    q = torch.ones(1, 1, 16, 512, dtype=torch.bfloat16, device=DEV)
    swa = torch.ones(1, 128, 512, dtype=torch.bfloat16, device=DEV)
    idx = torch.full((1, 1, 8), -1, dtype=torch.int32, device=DEV)
    out, lse = gpu_decode_attn(csa, q, cache, torch.tensor([E], dtype=torch.int32, device=DEV), idx, swa,
                               torch.tensor([0], dtype=torch.int32, device=DEV), E, 128)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_out_of_capacity_block_id_is_reported(csa):
    g = torch.Generator(device=DEV).manual_seed(10)
    T, W = 2 * 80, 128
    E = T // 2
    x = _latents(g, 1, T)
    q = torch.randn(1, 1, 16, 512, generator=g, device=DEV).to(torch.bfloat16)
    swa = torch.randn(1, W, 512, generator=g, device=DEV).to(torch.bfloat16)
    ws0 = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, [T], E, 512, 2, csa.SCALE_AMAX, ws0)
    idx = torch.tensor([[[3, 1000000, 0, -7]]], dtype=torch.int32, device=DEV)
    out = torch.empty(1, 1, 16, 512, device=DEV)
    n_entries = torch.tensor([E], dtype=torch.int32, device=DEV)
    swa_len = torch.tensor([W], dtype=torch.int32, device=DEV)
    args = csa.attn_args(q, cache, n_entries, idx, out, max_entries=E, window=W, scale=SCALE, swa=swa,
                         swa_len=swa_len)
    ws = csa.workspace(csa.sparse_attn_workspace_size(1, args), DEV)
    csa.sparse_attn_decode(q, cache, n_entries, idx, out, max_entries=E, window=W, scale=SCALE, ws=ws, swa=swa,
                           swa_len=swa_len)
    assert csa.device_status(ws) == csa.ERR_DEVICE_CHECK
    entries = o_fp4.dequantize(o_fp4.pack(to_np(x)[0], 2, "amax"), 512, E)
    ref, _ = o_attn.decode_attention(to_np(q)[0, 0].astype(np.float64), entries, E, [3, 0], to_np(swa)[0], SCALE)
    assert_attn_close(out[0, 0].cpu().numpy(), ref)


def test_prefill_matches_oracle(csa):
    g = torch.Generator(device=DEV).manual_seed(11)
    rng = np.random.default_rng(11)
    context, chunk_start, W, K, H = 1200, 1100, 128, 24, 64
    E = context // 2
    x = _latents(g, 1, context)
    ws = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, [context], E, 512, 2, csa.SCALE_AMAX, ws)
    pos = np.concatenate([[0, 1, 5, 200, 973, 1100, 1101], rng.integers(chunk_start, context, 26)]).astype(np.int32)
    Q = pos.size
    first = chunk_start - W + 1
    swa = torch.randn(1, context - first, 512, generator=g, device=DEV).to(torch.bfloat16)
    q = torch.randn(1, Q, H, 512, generator=g, device=DEV).to(torch.bfloat16)
    nb = -(-E // 8)
    idx_np = np.stack([rng.choice(nb, K, replace=False) for _ in range(Q)]).astype(np.int32)[None]
    idx_np[0, 0, -2:] = -1
    out, lse = gpu_prefill_attn(csa, q, cache, torch.tensor([E], dtype=torch.int32, device=DEV),
                                torch.from_numpy(idx_np).to(DEV), torch.from_numpy(pos)[None].to(DEV), swa,
                                torch.tensor([first], dtype=torch.int32, device=DEV), E, W)
    entries = o_fp4.dequantize(o_fp4.pack(to_np(x)[0], 2, "amax"), 512, E)
    qf, sf = to_np(q)[0], to_np(swa)[0]
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    for j in range(Q):
        ref, ref_lse = o_attn.prefill_attention(qf[j].astype(np.float64), entries, E, idx_np[0, j], sf, first,
                                                int(pos[j]), W, SCALE)
        assert_attn_close(out[0, j], ref, f"position {pos[j]}")
        assert_lse_close(lse[0, j], ref_lse, f"position {pos[j]}")


def test_bounded_wait_gives_up_and_the_context_survives(csa):
    # Failure path without a GPU fault: the test-only injection makes the attention withhold one internal
    # arrival, so the epilogue's wait (one cache tile per query, no window: one tile per CTA) gives up after
    # 64 polls, records CSA_ERR_TIMEOUT and the kernel returns. The same call then runs normally on the same
    # context and matches the oracle.
    g = torch.Generator(device=DEV).manual_seed(61)
    B, T, H, K = 2, 2 * 300, 64, 16
    E = T // 2
    x = _latents(g, B, T)
    q = torch.randn(B, 1, H, 512, generator=g, device=DEV).to(torch.bfloat16)
    ws0 = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, [T] * B, E, 512, 2, csa.SCALE_AMAX, ws0)
    n_entries = torch.full((B,), E, dtype=torch.int32, device=DEV)
    idx = torch.arange(K, dtype=torch.int32, device=DEV).view(1, 1, K).repeat(B, 1, 1).contiguous()
    out = torch.full((B, 1, H, 512), float("nan"), device=DEV)
    args = csa.attn_args(q, cache, n_entries, idx, out, max_entries=E, window=0, scale=SCALE)
    ws = csa.workspace(csa.sparse_attn_workspace_size(B, args), DEV)
    csa.debug_set_fault(csa.FAULT_WITHHOLD_ARRIVAL, 64)
    try:
        csa.sparse_attn_decode(q, cache, n_entries, idx, out, max_entries=E, window=0, scale=SCALE, ws=ws)
        status = csa.device_status(ws)
    finally:
        csa.debug_set_fault(csa.FAULT_NONE)
    assert status == csa.ERR_TIMEOUT
    csa.sparse_attn_decode(q, cache, n_entries, idx, out, max_entries=E, window=0, scale=SCALE, ws=ws)
    assert csa.device_status(ws) == csa.OK
    xf, qf, o = to_np(x), to_np(q), out.cpu().numpy()
    for b in range(B):
        entries = o_fp4.dequantize(o_fp4.pack(xf[b], 2, "amax", n_blocks=-(-E // 8)), 512, E)
        ref, _ = o_attn.decode_attention(qf[b, 0].astype(np.float64), entries, E, np.arange(K), np.zeros((0, 512)), SCALE)
        assert_attn_close(o[b, 0], ref, f"seq {b} after the timeout")


def test_queries_beyond_fp16_range_and_window_overflow(csa):
    # Queries of any finite bf16 magnitude: heads 0-15 up to ~1e5 (beyond fp16), heads 16-31 around 1e-6
    # (fp16 subnormals), the rest N(0, 1); every head matches the fp64 oracle. A window value beyond the
    # fp16 range is outside the call's contract and is reported as a device check.
    g = torch.Generator(device=DEV).manual_seed(62)
    B, T, H, K, W = 2, 2 * 700, 64, 32, 128
    E = T // 2
    x = _latents(g, B, T)
    q = torch.randn(B, 1, H, 512, generator=g, device=DEV)
    q[:, :, :16] *= 3.0e4
    q[:, :, 16:32] *= 1.0e-6
    q = q.to(torch.bfloat16)
    swa = torch.randn(B, W, 512, generator=g, device=DEV).to(torch.bfloat16)
    swa_len = torch.tensor([W, 90], dtype=torch.int32, device=DEV)
    ws0 = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, [T] * B, E, 512, 2, csa.SCALE_AMAX, ws0)
    n_entries = torch.full((B,), E, dtype=torch.int32, device=DEV)
    rng = np.random.default_rng(62)
    idx_np = np.stack([rng.choice(-(-E // 8), K, replace=False) for _ in range(B)]).astype(np.int32)[:, None, :]
    idx = torch.from_numpy(idx_np).to(DEV)
    out, lse = gpu_decode_attn(csa, q, cache, n_entries, idx, swa, swa_len, E, W)
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    xf, qf, sf = to_np(x), to_np(q), to_np(swa)
    assert np.abs(qf[:, :, :16]).max() > 65504
    for b in range(B):
        entries = o_fp4.dequantize(o_fp4.pack(xf[b], 2, "amax", n_blocks=-(-E // 8)), 512, E)
        ref, ref_lse = o_attn.decode_attention(qf[b, 0].astype(np.float64), entries, E, idx_np[b, 0],
                                               sf[b, :int(swa_len[b])], SCALE)
        assert_attn_close(out[b, 0], ref, f"seq {b}")
        # lse grows with |q|: compare it relative to its size for the large heads
        np.testing.assert_allclose(lse[b, 0], ref_lse, rtol=1e-5, atol=2e-3)
    swa[1, 5, 100] = 1.0e5
    bad = torch.empty(B, 1, H, 512, device=DEV)
    args = csa.attn_args(q, cache, n_entries, idx, bad, max_entries=E, window=W, scale=SCALE, swa=swa, swa_len=swa_len)
    ws = csa.workspace(csa.sparse_attn_workspace_size(B, args), DEV)
    csa.sparse_attn_decode(q, cache, n_entries, idx, bad, max_entries=E, window=W, scale=SCALE, ws=ws, swa=swa,
                           swa_len=swa_len)
    assert csa.device_status(ws) == csa.ERR_DEVICE_CHECK


def test_extreme_query_magnitudes(csa):
    # heads around 1e30 and 1e-30 (any finite bf16 magnitude): the logits of the large heads reach ~1e31, so the
    # softmax must subtract its maximum from the same rounded products it took the maximum of
    g = torch.Generator(device=DEV).manual_seed(63)
    B, T, H, K, W = 2, 1800, 64, 24, 128
    E = T // 2
    x = _latents(g, B, T)
    mag = torch.tensor([1e30, 1e-30, 3e5, 1.0], device=DEV).repeat(16).view(1, 1, H, 1)
    q = (torch.randn(B, 1, H, 512, generator=g, device=DEV) * mag).to(torch.bfloat16)
    swa = torch.randn(B, W, 512, generator=g, device=DEV).to(torch.bfloat16)
    swa_len = torch.tensor([W, 7], dtype=torch.int32, device=DEV)
    ws0 = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, [T] * B, E, 512, 2, csa.SCALE_AMAX, ws0)
    rng = np.random.default_rng(63)
    idx_np = np.stack([rng.choice(-(-E // 8), K, replace=False) for _ in range(B)]).astype(np.int32)[:, None, :]
    out, lse = gpu_decode_attn(csa, q, cache, torch.full((B,), E, dtype=torch.int32, device=DEV),
                               torch.from_numpy(idx_np).to(DEV), swa, swa_len, E, W)
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    xf, qf, sf = to_np(x), to_np(q), to_np(swa)
    for b in range(B):
        entries = o_fp4.dequantize(o_fp4.pack(xf[b], 2, "amax", n_blocks=-(-E // 8)), 512, E)
        ref, ref_lse = o_attn.decode_attention(qf[b, 0].astype(np.float64), entries, E, idx_np[b, 0],
                                               sf[b, :int(swa_len[b])], SCALE)
        assert_attn_close(out[b, 0], ref, f"seq {b}")
        np.testing.assert_allclose(lse[b, 0], ref_lse, rtol=1e-5, atol=2e-3)
