"""csa_index_topk_static, the indexer entry point for callers that cannot allocate device memory (a host
framework whose allocator owns the GPU, a plug-in limited to the buffers it is handed, a serving loop
that must not allocate once running). It takes its scratch from the library's own fixed device array
instead of a caller workspace, so it must select exactly what csa_index_topk selects with a workspace.

This file is collected last on purpose: the static array keeps the previous call's contents, and the
test must pass both in a fresh process and after every other test has used the library."""

import numpy as np
import pytest
import torch

from _pipeline import gpu_index, gpu_pack_sequences

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa():
    from compressed_sparse_attention_merge_b300 import binding
    binding.lib()
    return binding


def _case(csa, seed, lengths, dim, heads, nq):
    g = torch.Generator(device=DEV).manual_seed(seed)
    B, E = len(lengths), max(lengths)
    keys = torch.randint(-4, 5, (B, E, dim), generator=g, device=DEV).float()
    q_idx = torch.randint(-4, 5, (B, nq, heads, dim), generator=g, device=DEV).float()
    ws = csa.workspace(256, DEV)
    kc = gpu_pack_sequences(csa, keys, lengths, E, dim, 1, csa.SCALE_POW2, ws)
    return q_idx, kc, torch.tensor(lengths, dtype=torch.int32, device=DEV), E


def test_static_scratch_matches_workspace_call_twice_in_a_row(csa):
    # two different problems back to back: the second call must not see anything the first one left
    cases = [(_case(csa, 71, [5000, 1203, 4096], 128, 4, 2), 96),
             (_case(csa, 72, [777, 2500], 64, 1, 3), 40)]
    for (q_idx, kc, n_entries, E), top_k in cases:
        ref, _ = gpu_index(csa, q_idx, kc, n_entries, E, top_k)
        got = torch.full_like(ref, -7)
        status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
        csa.index_topk_static(q_idx, kc, n_entries, got, max_entries=E, top_k=top_k, status_out=status)
        torch.cuda.synchronize()
        assert int(status.item()) == csa.OK
        np.testing.assert_array_equal(got.cpu().numpy(), ref.cpu().numpy())


def test_static_scratch_rejects_too_large_a_call(csa):
    # 64 queries x 65,536 blocks of scores need 16 MiB, more than the 4 MiB array: refused, nothing launched
    E = 8 * 65536
    q_idx = torch.zeros(1, 64, 4, 128, device=DEV)
    kc = torch.zeros(1, 1, 16, dtype=torch.uint8, device=DEV)
    n_entries = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((1, 64, 8), -7, dtype=torch.int32, device=DEV)
    with pytest.raises(csa.CsaError) as err:
        csa.index_topk_static(q_idx, kc, n_entries, out, max_entries=E, top_k=8)
    assert err.value.status == csa.ERR_WORKSPACE_TOO_SMALL
    assert "static array" in str(err.value)
    torch.cuda.synchronize()
    assert torch.all(out == -7)
