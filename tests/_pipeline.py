"""Shared helpers for the GPU parity tests: run the CUDA path through the C-ABI binding and the CPU
oracle on the same seeded inputs, and compare. Not collected as tests."""

import math

import numpy as np
import torch

from oracle import attention as o_attn
from oracle import fp4 as o_fp4
from oracle import indexer as o_idx

ATOL = 2e-3          # max-abs error of attention outputs against the fp64 oracle
RTOL = 1e-2          # max relative error where |oracle| >= ATOL / RTOL
SCALE = 1.0 / math.sqrt(512)


def to_np(t):
    return t.detach().to("cpu").float().numpy() if t.dtype in (torch.bfloat16, torch.float16) \
        else t.detach().to("cpu").numpy()


def assert_attn_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref)
    assert err.max() <= ATOL, f"{what}: max abs err {err.max():.3e}"
    big = np.abs(ref) >= ATOL / RTOL
    if big.any():
        rel = (err[big] / np.abs(ref[big])).max()
        assert rel <= RTOL, f"{what}: max rel err {rel:.3e}"


def assert_lse_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    inf = np.isinf(ref)
    assert np.array_equal(np.isinf(got), inf), what
    if (~inf).any():
        err = np.abs(got[~inf] - ref[~inf]).max()
        assert err <= ATOL, f"{what}: lse err {err:.3e}"


# ------------------------------------------------------------------------------------------------
# Oracle side (CPU, numpy)
# ------------------------------------------------------------------------------------------------

def oracle_latent_cache(tokens_f32, n_blocks):
    """Packed latent cache of one sequence from its bf16 tokens (as float32), pair-merged."""
    return o_fp4.pack(tokens_f32, 2, "amax", n_blocks=n_blocks)


def oracle_key_cache(keys_f32, n_blocks):
    return o_fp4.pack(keys_f32, 1, "pow2", n_blocks=n_blocks)


# ------------------------------------------------------------------------------------------------
# CUDA side (through the binding)
# ------------------------------------------------------------------------------------------------

def gpu_pack_sequences(csa, tokens, lengths, max_entries, dim, merge, rule, ws, coarse=None):
    """Packs every sequence b's first lengths[b] rows of tokens [B, T, dim] into a new cache, one call per
    sequence (so that ragged sequences pack exactly their own rows)."""
    B = tokens.shape[0]
    cache = csa.empty_cache(B, max_entries, dim, tokens.device)
    for b in range(B):
        if lengths[b] // merge == 0:
            continue
        csa.pack_fp4(tokens[b:b + 1, :lengths[b]], cache[b:b + 1], merge=merge, scale_rule=rule,
                     max_entries=max_entries, ws=ws, coarse_sum=None if coarse is None else coarse[b:b + 1])
    return cache


def gpu_index(csa, q_idx, keys_cache, n_entries, max_entries, top_k, coarse=None, keep_blocks=0, q_pos=None,
              head_w=None, relu=True, want_scores=False):
    B, Q = q_idx.shape[0], q_idx.shape[1]
    out = torch.empty(B, Q, top_k, dtype=torch.int32, device=q_idx.device)
    scores = None
    if want_scores:
        scores = torch.empty(B, Q, -(-max_entries // 8), dtype=torch.float32, device=q_idx.device)
    args = csa.index_args(q_idx, keys_cache, n_entries, out, max_entries=max_entries, top_k=top_k, head_w=head_w,
                          relu=relu, q_pos=q_pos, coarse_sum=coarse, keep_blocks=keep_blocks,
                          out_block_scores=scores)
    ws = csa.workspace(csa.index_topk_workspace_size(B, args), q_idx.device)
    csa.index_topk(q_idx, keys_cache, n_entries, out, max_entries=max_entries, top_k=top_k, ws=ws, head_w=head_w,
                   relu=relu, q_pos=q_pos, coarse_sum=coarse, keep_blocks=keep_blocks, out_block_scores=scores)
    assert csa.device_status(ws) == csa.OK
    return out, scores


def gpu_decode_attn(csa, q, cache, n_entries, idx, swa, swa_len, max_entries, window, want_lse=True, nvfp4q=False):
    B, Q, H = q.shape[0], q.shape[1], q.shape[2]
    out = torch.empty(B, Q, H, 512, dtype=torch.float32, device=q.device)
    lse = torch.empty(B, Q, H, dtype=torch.float32, device=q.device) if want_lse else None
    args = csa.attn_args(q, cache, n_entries, idx, out, max_entries=max_entries, window=window, scale=SCALE,
                         swa=swa, swa_len=swa_len, out_lse=lse)
    ws = csa.workspace(csa.sparse_attn_workspace_size(B, args), q.device)
    fn = csa.sparse_attn_decode_nvfp4q if nvfp4q else csa.sparse_attn_decode
    fn(q, cache, n_entries, idx, out, max_entries=max_entries, window=window, scale=SCALE, ws=ws, swa=swa,
       swa_len=swa_len, out_lse=lse)
    assert csa.device_status(ws) == csa.OK
    return out, lse


def gpu_prefill_attn(csa, q, cache, n_entries, idx, q_pos, swa, swa_first_pos, max_entries, window, nvfp4q=False):
    B, Q, H = q.shape[0], q.shape[1], q.shape[2]
    out = torch.empty(B, Q, H, 512, dtype=torch.float32, device=q.device)
    lse = torch.empty(B, Q, H, dtype=torch.float32, device=q.device)
    args = csa.attn_args(q, cache, n_entries, idx, out, max_entries=max_entries, window=window, scale=SCALE,
                         swa=swa, swa_first_pos=swa_first_pos, q_pos=q_pos, out_lse=lse)
    ws = csa.workspace(csa.sparse_attn_workspace_size(B, args), q.device)
    fn = csa.sparse_attn_prefill_nvfp4q if nvfp4q else csa.sparse_attn_prefill
    fn(q, cache, n_entries, idx, out, q_pos=q_pos, max_entries=max_entries, window=window, scale=SCALE, ws=ws,
       swa=swa, swa_first_pos=swa_first_pos, out_lse=lse)
    assert csa.device_status(ws) == csa.OK
    return out, lse


def oracle_flat_topk(q_idx_b, keys_deq, n_e, top_k, q_pos=None, head_w=None, relu=True):
    return o_idx.flat_topk(q_idx_b, keys_deq, n_e, top_k, head_w=head_w, relu=relu, q_pos=q_pos)


def oracle_decode(q_b, entries, n_e, idx_b, swa_rows):
    return o_attn.decode_attention(q_b.astype(np.float64), entries, n_e, idx_b, swa_rows, SCALE)
