"""Seeded synthetic inputs for the CSA2 path. Random numbers only: nothing here computes any step of
the method, so both the CUDA path and the CPU oracle can be fed from it.

Value recipes (the pages publish no workload data; these follow the shapes they describe):
  latent tokens      bf16 N(0, 1); optionally a fraction of elements (i.i.d.) multiplied by 8 (outliers)
  attention queries  bf16 N(0, 1)
  window rows        bf16 N(0, 1)
  index keys         fp32 integers uniform in [-4, 4], one row per cache entry
  index queries      fp32 integers uniform in [-4, 4]
  needle blocks      a fraction of blocks whose 8 key rows are 4 * sign(first index query, head 0), so the
                     Top-K has structure to find
  hidden rows        bf16 N(0, 1), projected by a bf16 N(0, 1 / hidden) weight (latents about N(0, 1))
Every generator takes an explicit seed and device; large tensors are generated one sequence at a
time to bound the temporary fp32 memory.
"""

from dataclasses import dataclass, field

import torch

LATENT = 512


def generator(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def latent_tokens(g, shape, device, outlier_frac=0.0):
    """bf16 N(0, 1) values of the given shape; outlier_frac of the elements scaled by 8."""
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if outlier_frac > 0:
        mask = torch.rand(shape, generator=g, device=device) < outlier_frac
        x = torch.where(mask, x * 8.0, x)
    return x.to(torch.bfloat16)


def int_values(g, shape, device, lo=-4, hi=4):
    """fp32 integers uniform in [lo, hi]."""
    return torch.randint(lo, hi + 1, shape, generator=g, device=device, dtype=torch.int32).to(torch.float32)


def normal_bf16(g, shape, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def plant_needles(g, keys, q_idx, frac, block=8):
    """In place: each block of `keys` [B, n_e, D] is, with probability frac, overwritten by
    4 * sign(q_idx[b, 0, 0, :])."""
    if frac <= 0:
        return keys
    bsz, n_e, _ = keys.shape
    n_b = n_e // block
    for b in range(bsz):
        pick = torch.rand(n_b, generator=g, device=keys.device) < frac
        ids = torch.nonzero(pick).flatten()
        if ids.numel() == 0:
            continue
        needle = 4.0 * torch.sign(q_idx[b, 0, 0, :])
        rows = (ids[:, None] * block + torch.arange(block, device=keys.device)[None, :]).flatten()
        keys[b, rows] = needle
    return keys


@dataclass
class DecodeCase:
    """A decode workload: batch sequences with tokens[b] tokens each (pair-merged into tokens[b] // 2
    entries), n_query queries per sequence. With `causal_drafts`, the n_query queries of a sequence are
    the draft positions of a multi-token decode step (speculative verification): the last n_query tokens
    of the sequence, each seeing only the cache entries and window rows at or before its own position."""
    name: str
    tokens: list
    heads: int = 64
    idx_heads: int = 4
    idx_dim: int = 128
    top_k: int = 256
    window: int = 128
    n_query: int = 1
    outlier_frac: float = 0.0
    needle_frac: float = 0.0
    hier_keep: int = 0            # > 0: hierarchical selection keeping this many blocks
    layers: int = 1               # > 1: layer chain with per-layer queries and windows
    distinct_index_queries: int = 1
    causal_drafts: bool = False
    nvfp4q: bool = False          # attention by the NVFP4-query variant (block-scaled FP4 logits)
    seed: int = 0
    swa_len: list = field(default_factory=list)

    @property
    def batch(self):
        return len(self.tokens)

    @property
    def max_tokens(self):
        return max(self.tokens)

    @property
    def max_entries(self):
        return self.max_tokens // 2


def make_decode(case, device):
    """Returns a dict of tensors on `device`:
    tokens [B, T, 512] bf16, keys [B, E, D_i] f32, n_entries [B] i32, q [L, B, Q, H, 512] bf16,
    q_idx [Lq, B, Q, H_i, D_i] f32, swa [L, B, W, 512] bf16, swa_len [B] i32.
    With causal_drafts (every sequence T tokens long): q_pos [B, Q] i32 = T - Q .. T - 1, and the window
    buffer holds the W + Q - 1 tokens T - Q - W + 1 .. T - 1: swa [L, B, W + Q - 1, 512] bf16 with
    swa_first_pos [B] i32 = T - Q - W + 1."""
    g = generator(case.seed, device)
    B, T, E = case.batch, case.max_tokens, case.max_entries
    tokens = torch.empty(B, T, LATENT, dtype=torch.bfloat16, device=device)
    for b in range(B):
        tokens[b] = latent_tokens(g, (T, LATENT), device, case.outlier_frac)
    keys = torch.empty(B, E, case.idx_dim, dtype=torch.float32, device=device)
    for b in range(B):
        keys[b] = int_values(g, (E, case.idx_dim), device)
    n_entries = torch.tensor([t // 2 for t in case.tokens], dtype=torch.int32, device=device)
    nq = case.distinct_index_queries
    q_idx = int_values(g, (nq, B, case.n_query, case.idx_heads, case.idx_dim), device)
    plant_needles(g, keys, q_idx[0], case.needle_frac)
    L = case.layers
    q = normal_bf16(g, (L, B, case.n_query, case.heads, LATENT), device)
    Q = case.n_query
    swa_rows = case.window + (Q - 1 if case.causal_drafts else 0)
    swa = normal_bf16(g, (L, B, swa_rows, LATENT), device)
    sl = case.swa_len or [case.window] * B
    swa_len = torch.tensor(sl, dtype=torch.int32, device=device)
    out = dict(tokens=tokens, keys=keys, n_entries=n_entries, q=q, q_idx=q_idx, swa=swa, swa_len=swa_len)
    if case.causal_drafts:
        if any(t != T for t in case.tokens):
            raise ValueError("causal drafts need sequences of equal length")
        out["q_pos"] = torch.arange(T - Q, T, dtype=torch.int32, device=device)[None, :].repeat(B, 1).contiguous()
        out["swa_first_pos"] = torch.full((B,), T - Q - case.window + 1, dtype=torch.int32, device=device)
    return out


@dataclass
class PrefillCase:
    """A prefill chunk of `chunk` positions at the end of a `context`-token sequence (batch 1)."""
    name: str
    context: int
    chunk: int
    heads: int = 64
    idx_heads: int = 4
    idx_dim: int = 128
    top_k: int = 256
    window: int = 128
    outlier_frac: float = 0.0
    nvfp4q: bool = False          # attention by the NVFP4-query variant (block-scaled FP4 logits)
    seed: int = 0

    @property
    def max_entries(self):
        return self.context // 2

    @property
    def first_pos(self):
        return self.context - self.chunk


def make_prefill(case, device):
    """Returns: prior [1, P, 512] bf16 (tokens before the chunk), chunk [1, C, 512] bf16, keys
    [1, E, D_i] f32 (one row per entry, prior and chunk), q [1, C, H, 512] bf16, q_idx [1, C, H_i, D_i]
    f32, q_pos [1, C] i32, swa [1, C + window - 1, 512] bf16 (row r = token first_pos - window + 1 + r),
    swa_first_pos [1] i32, n_entries [1] i32."""
    g = generator(case.seed, device)
    P, C, E = case.first_pos, case.chunk, case.max_entries
    prior = latent_tokens(g, (1, P, LATENT), device, case.outlier_frac)
    chunk = latent_tokens(g, (1, C, LATENT), device, case.outlier_frac)
    keys = int_values(g, (1, E, case.idx_dim), device)
    q = normal_bf16(g, (1, C, case.heads, LATENT), device)
    q_idx = int_values(g, (1, C, case.idx_heads, case.idx_dim), device)
    q_pos = torch.arange(P, P + C, dtype=torch.int32, device=device)[None, :]
    swa_rows = C + case.window - 1
    swa = normal_bf16(g, (1, swa_rows, LATENT), device)
    swa_first_pos = torch.tensor([P - case.window + 1], dtype=torch.int32, device=device)
    n_entries = torch.tensor([E], dtype=torch.int32, device=device)
    return dict(prior=prior, chunk=chunk, keys=keys, q=q, q_idx=q_idx, q_pos=q_pos, swa=swa,
                swa_first_pos=swa_first_pos, n_entries=n_entries)


# The five workloads of the method's decode/prefill path, named by what they are.
@dataclass
class ProjectCase:
    """The cache write path: hidden rows of `batch` sequences of `tokens` tokens, projected to the latent by a
    [512][hidden] weight and packed (merge 2)."""
    name: str
    batch: int = 1
    tokens: int = 131072
    hidden: int = 4096
    seed: int = 30000


def make_project(case, device):
    """Hidden rows bf16 N(0, 1) [batch, tokens, hidden] and a weight bf16 N(0, 1 / hidden) [512, hidden], so
    that the latents are about N(0, 1)."""
    g = generator(case.seed, device)
    h = torch.empty(case.batch, case.tokens, case.hidden, dtype=torch.bfloat16, device=device)
    for b in range(case.batch):
        h[b] = torch.randn(case.tokens, case.hidden, generator=g, device=device).to(torch.bfloat16)
    w = (torch.randn(LATENT, case.hidden, generator=g, device=device) / case.hidden ** 0.5).to(torch.bfloat16)
    return {"h": h, "w": w}


TINY_DECODE_4K = DecodeCase("tiny_decode_4k_b1_h16", tokens=[4096], heads=16, idx_heads=1, idx_dim=64, top_k=64,
                            seed=20261)
DECODE_64K_B32 = DecodeCase("decode_64k_b32_h64", tokens=[65536] * 32, outlier_frac=0.01, needle_frac=0.01,
                            seed=20262)
DECODE_1M_B4_HIER = DecodeCase("decode_1m_b4_h64_hier2048", tokens=[1 << 20] * 4, outlier_frac=0.01,
                               needle_frac=0.01, hier_keep=2048, seed=20263)
CHAIN_128K_B64 = DecodeCase("chain20_128k_b64_h64", tokens=[131072] * 64, outlier_frac=0.01, needle_frac=0.01,
                            layers=20, distinct_index_queries=5, seed=20264)
PREFILL_2K_AT_128K = PrefillCase("prefill_2048_at_128k_h64", context=131072, chunk=2048, seed=20265)
# The prefill workload above with the opt-in NVFP4-query attention (same inputs, same seed).
PREFILL_2K_AT_128K_NVFP4Q = PrefillCase("prefill_2048_at_128k_h64_nvfp4q", context=131072, chunk=2048, nvfp4q=True,
                                        seed=20265)
# Multi-token decode at the 64K shape: four draft positions per sequence (speculative verification), the
# last four tokens of each sequence, causal among themselves.
DECODE_64K_B32_Q4 = DecodeCase("decode_64k_b32_h64_q4", tokens=[65536] * 32, n_query=4, outlier_frac=0.01,
                               needle_frac=0.01, causal_drafts=True, seed=20266)
# The decode workload above with the opt-in NVFP4-query attention (same inputs, same seed).
DECODE_64K_B32_NVFP4Q = DecodeCase("decode_64k_b32_h64_nvfp4q", tokens=[65536] * 32, outlier_frac=0.01,
                                   needle_frac=0.01, nvfp4q=True, seed=20262)

# The cache write path over one 128K-token sequence with a 4,096-wide hidden state (the pages give no hidden
# width; 4,096 is a common one for a model of this size class).
PROJECT_128K_H4096 = ProjectCase("project_pack_128k_h4096", batch=1, tokens=131072, hidden=4096, seed=30001)
