"""csa_sparse_attn_decode_nvfp4q / csa_sparse_attn_prefill_nvfp4q (block-scaled FP4 logits) against the fp64
oracle of the variant (max-abs 2e-3, max-rel 1e-2), and against the exact calls where the query and the
window keys are already on the FP4 grid."""

import numpy as np
import pytest
import torch

from oracle import attention as o_attn
from oracle import fp4 as o_fp4

from _pipeline import (SCALE, assert_attn_close, assert_lse_close, gpu_decode_attn, gpu_pack_sequences,
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


def _random_idx(rng, n_b_list, B, K, cap_blocks):
    idx = np.full((B, 1, K), -1, np.int32)
    for b in range(B):
        nb = n_b_list[b]
        k = min(K, nb)
        if k:
            idx[b, 0, :k] = rng.choice(nb, size=k, replace=False)
        if k < K and nb < cap_blocks:
            idx[b, 0, k] = cap_blocks - 1          # a legal id past the valid blocks: ignored
    return idx


@pytest.mark.parametrize("heads,top_k,batch", [(64, 24, 3), (16, 64, 3), (32, 40, 2), (64, 16, 150)])
def test_decode_matches_oracle(csa, heads, top_k, batch):
    g = torch.Generator(device=DEV).manual_seed(700 + heads + top_k + batch)
    rng = np.random.default_rng(7 * heads + top_k + batch)
    base = [2000, 74, 1401, 1]
    tokens = [base[i % 4] + (i // 4) * 2 for i in range(batch)]
    B, T = batch, max(tokens)
    E = T // 2
    W = 128
    x = _latents(g, B, T)
    q = (torch.randn(B, 1, heads, 512, generator=g, device=DEV) *
         torch.tensor([1.0, 30.0, 0.01], device=DEV).repeat(heads)[:heads].view(1, 1, heads, 1)).to(torch.bfloat16)
    swa = torch.randn(B, W, 512, generator=g, device=DEV).to(torch.bfloat16)
    swa_len = torch.tensor([[128, 5, 0, 77][i % 4] for i in range(B)], dtype=torch.int32, device=DEV)
    ws = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, tokens, E, 512, 2, csa.SCALE_AMAX, ws)
    n_e = [t // 2 for t in tokens]
    idx_np = _random_idx(rng, [-(-n // 8) for n in n_e], B, top_k, -(-E // 8))
    out, lse = gpu_decode_attn(csa, q, cache, torch.tensor(n_e, dtype=torch.int32, device=DEV),
                               torch.from_numpy(idx_np).to(DEV), swa, swa_len, E, W, nvfp4q=True)
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    xf, qf, sf = to_np(x), to_np(q), to_np(swa)
    check = range(B) if B <= 8 else list(range(4)) + [B - 1]
    for b in check:
        entries = o_fp4.dequantize(o_fp4.pack(xf[b, :tokens[b]], 2, "amax", n_blocks=-(-E // 8)), 512, E)
        ref, ref_lse = o_attn.decode_attention_nvfp4q(qf[b, 0], entries, n_e[b], idx_np[b, 0],
                                                      sf[b, :int(swa_len[b])], SCALE)
        assert_attn_close(out[b, 0], ref, f"seq {b}")
        assert_lse_close(lse[b, 0], ref_lse, f"seq {b}")


@pytest.mark.parametrize("W", [128, 300])
def test_prefill_matches_oracle(csa, W):
    # W = 300 gives three window tiles per position: the FP4 window keys of one tile are written into the
    # stage the previous tile's logits have just finished with
    g = torch.Generator(device=DEV).manual_seed(12 + W)
    rng = np.random.default_rng(12 + W)
    context, chunk_start, K, H = 1200, 1100, 24, 64
    E = context // 2
    x = _latents(g, 1, context)
    ws = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, [context], E, 512, 2, csa.SCALE_AMAX, ws)
    pos = np.concatenate([[0, 1, 5, 200, 973, 1100, 1101], rng.integers(chunk_start, context, 9)]).astype(np.int32)
    Q = pos.size
    first = chunk_start - W + 1
    swa = torch.randn(1, context - first, 512, generator=g, device=DEV).to(torch.bfloat16)
    q = torch.randn(1, Q, H, 512, generator=g, device=DEV).to(torch.bfloat16)
    nb = -(-E // 8)
    idx_np = np.stack([rng.choice(nb, K, replace=False) for _ in range(Q)]).astype(np.int32)[None]
    idx_np[0, 0, -2:] = -1
    out, lse = gpu_prefill_attn(csa, q, cache, torch.tensor([E], dtype=torch.int32, device=DEV),
                                torch.from_numpy(idx_np).to(DEV), torch.from_numpy(pos)[None].to(DEV), swa,
                                torch.tensor([first], dtype=torch.int32, device=DEV), E, W, nvfp4q=True)
    entries = o_fp4.dequantize(o_fp4.pack(to_np(x)[0], 2, "amax"), 512, E)
    qf, sf = to_np(q)[0], to_np(swa)[0]
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    for j in range(Q):
        ref, ref_lse = o_attn.prefill_attention_nvfp4q(qf[j], entries, E, idx_np[0, j], sf, first, int(pos[j]), W,
                                                       SCALE)
        assert_attn_close(out[0, j], ref, f"position {pos[j]}")
        assert_lse_close(lse[0, j], ref_lse, f"position {pos[j]}")


def _grid_query(rng, B, H):
    # every head exactly representable by the variant's rounding: each 16-element block holds a +-6 s element
    # and E2M1 multiples of its scale s, and the head's maximum 6 s lies in [1024, 2048)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    q = np.zeros((B, 1, H, 512), np.float32)
    for b in range(B):
        for h in range(H):
            for gi in range(32):
                s = np.float32([176, 192, 224, 256, 320][rng.integers(0, 5)]) if gi == 0 else \
                    np.float32(2.0 ** rng.integers(-2, 5))
                blk = mags[rng.integers(0, 8, 16)] * np.where(rng.random(16) < 0.5, -1, 1)
                blk[rng.integers(0, 16)] = 6.0
                q[b, 0, h, 16 * gi:16 * gi + 16] = blk * s / np.float32(1024.0)
    return q


def test_equals_exact_call_on_fp4_inputs(csa):
    # queries and window rows already on the FP4 grid: the variant's roundings change nothing, so both calls
    # compute the same attention (up to the order of fp32 accumulation)
    g = torch.Generator(device=DEV).manual_seed(31)
    rng = np.random.default_rng(31)
    B, T, H, K, W = 4, 3000, 64, 40, 128
    E = T // 2
    x = _latents(g, B, T)
    q_np = _grid_query(rng, B, H)
    assert np.array_equal(o_attn.nvfp4_query(q_np[0, 0]), q_np[0, 0])
    q = torch.from_numpy(q_np).to(DEV).to(torch.bfloat16)
    assert np.array_equal(to_np(q), q_np)
    w_np = o_fp4.round_trip(rng.standard_normal((B * W, 512)).astype(np.float32), "amax").reshape(B, W, 512)
    swa = torch.from_numpy(w_np).to(DEV).to(torch.bfloat16)
    assert np.array_equal(to_np(swa), w_np)
    swa_len = torch.tensor([128, 100, 1, 0], dtype=torch.int32, device=DEV)
    ws = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, [T] * B, E, 512, 2, csa.SCALE_AMAX, ws)
    n_entries = torch.full((B,), E, dtype=torch.int32, device=DEV)
    idx_np = _random_idx(rng, [-(-E // 8)] * B, B, K, -(-E // 8))
    idx = torch.from_numpy(idx_np).to(DEV)
    a, la = gpu_decode_attn(csa, q, cache, n_entries, idx, swa, swa_len, E, W, nvfp4q=True)
    b_, lb = gpu_decode_attn(csa, q, cache, n_entries, idx, swa, swa_len, E, W)
    assert_attn_close(a.cpu().numpy(), b_.cpu().numpy(), "variant against the exact call")
    assert_lse_close(la.cpu().numpy(), lb.cpu().numpy(), "variant against the exact call")
    entries = o_fp4.dequantize(o_fp4.pack(to_np(x)[1], 2, "amax"), 512, E)
    ref, ref_lse = o_attn.decode_attention(q_np[1, 0], entries, E, idx_np[1, 0], w_np[1, :100], SCALE)
    assert_attn_close(a[1, 0].cpu().numpy(), ref, "variant against the exact oracle")
    assert_lse_close(la[1, 0].cpu().numpy(), ref_lse, "variant against the exact oracle")


def test_large_and_tiny_query_heads(csa):
    # the per-head power of two keeps the E4M3 block scales in range at any magnitude bf16 allows
    g = torch.Generator(device=DEV).manual_seed(41)
    rng = np.random.default_rng(41)
    B, T, H, K, W = 2, 900, 64, 20, 128
    E = T // 2
    x = _latents(g, B, T)
    mag = torch.tensor([1e30, 1e-30, 3e5, 1.0], device=DEV).repeat(16).view(1, 1, H, 1)
    q = (torch.randn(B, 1, H, 512, generator=g, device=DEV) * mag).to(torch.bfloat16)
    swa = torch.randn(B, W, 512, generator=g, device=DEV).to(torch.bfloat16)
    swa_len = torch.tensor([128, 3], dtype=torch.int32, device=DEV)
    ws = csa.workspace(256, DEV)
    cache = gpu_pack_sequences(csa, x, [T] * B, E, 512, 2, csa.SCALE_AMAX, ws)
    idx_np = _random_idx(rng, [-(-E // 8)] * B, B, K, -(-E // 8))
    out, lse = gpu_decode_attn(csa, q, cache, torch.full((B,), E, dtype=torch.int32, device=DEV),
                               torch.from_numpy(idx_np).to(DEV), swa, swa_len, E, W, nvfp4q=True)
    qf, sf = to_np(q), to_np(swa)
    for b in range(B):
        entries = o_fp4.dequantize(o_fp4.pack(to_np(x)[b], 2, "amax"), 512, E)
        ref, ref_lse = o_attn.decode_attention_nvfp4q(qf[b, 0], entries, E, idx_np[b, 0], sf[b, :int(swa_len[b])],
                                                      SCALE)
        assert_attn_close(out[b, 0].cpu().numpy(), ref, f"seq {b}")
        np.testing.assert_allclose(lse[b, 0].cpu().numpy(), ref_lse, rtol=1e-5, atol=2e-3)


def test_no_rows_gives_zero_and_neg_inf(csa):
    q = torch.ones(2, 1, 16, 512, dtype=torch.bfloat16, device=DEV)
    cache = csa.empty_cache(2, 8, 512, DEV)
    swa = torch.zeros(2, 128, 512, dtype=torch.bfloat16, device=DEV)
    out, lse = gpu_decode_attn(csa, q, cache, torch.zeros(2, dtype=torch.int32, device=DEV),
                               torch.full((2, 1, 4), -1, dtype=torch.int32, device=DEV), swa,
                               torch.zeros(2, dtype=torch.int32, device=DEV), 8, 128, nvfp4q=True)
    assert torch.all(out == 0)
    assert torch.all(torch.isinf(lse)) and torch.all(lse < 0)
