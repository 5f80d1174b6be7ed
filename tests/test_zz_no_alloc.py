"""csa_index_topk_static, the indexer entry point for callers that cannot allocate device memory (a host
framework whose allocator owns the GPU, a plug-in limited to the buffers it is handed, a serving loop
that must not allocate once running). It takes its scratch from the library's own fixed device array
instead of a caller workspace, so it must select exactly what csa_index_topk selects with a workspace.

This file is collected last on purpose: the static array keeps the previous call's contents, and the
test must pass both in a fresh process and after every other test has used the library."""

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


def test_static_scratch_matches_the_oracle_flat_and_hierarchical(csa):
    # the static entry point against the CPU oracle directly: a flat call, then a hierarchical call that uses
    # the coarse-score and kept-super-block regions of the array, then the flat call again
    g = torch.Generator(device=DEV).manual_seed(73)
    lengths, dim, heads, top_k, keep = [3 * 512 + 77, 512 * 5], 128, 4, 48, 128
    B, E = len(lengths), max(lengths)
    keys = torch.randint(-4, 5, (B, E, dim), generator=g, device=DEV).float()
    q_idx = torch.randint(-4, 5, (B, 1, heads, dim), generator=g, device=DEV).float()
    ws = csa.workspace(256, DEV)
    coarse = csa.empty_coarse(B, E, dim, DEV)
    kc = gpu_pack_sequences(csa, keys, lengths, E, dim, 1, csa.SCALE_POW2, ws, coarse=coarse)
    n_entries = torch.tensor(lengths, dtype=torch.int32, device=DEV)
    kf, qi = keys.cpu().numpy(), q_idx.cpu().numpy()
    for hier in (False, True, False):
        got = torch.full((B, 1, top_k), -7, dtype=torch.int32, device=DEV)
        status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
        extra = dict(coarse_sum=coarse, keep_blocks=keep) if hier else {}
        csa.index_topk_static(q_idx, kc, n_entries, got, max_entries=E, top_k=top_k, status_out=status, **extra)
        torch.cuda.synchronize()
        assert int(status.item()) == csa.OK
        for b in range(B):
            n = lengths[b]
            deq = o_fp4.dequantize(o_fp4.pack(kf[b, :n], 1, "pow2", n_blocks=-(-E // 8)), dim, E)
            if hier:
                ref, _ = o_idx.hierarchical_topk(qi[b], deq, n, top_k, keep)
            else:
                ref, _ = o_idx.flat_topk(qi[b], deq, n, top_k)
            np.testing.assert_array_equal(got[b].cpu().numpy(), ref, err_msg=f"hier={hier} seq {b}")


def test_static_scratch_reports_a_device_check_then_recovers(csa):
    # an entry count beyond max_entries is clamped by the kernels and reported through status_out; the
    # next call starts from a cleared status word and reports 0
    q_idx, kc, n_entries, E = _case(csa, 74, [900, 640], 64, 2, 1)
    top_k = 16
    bad = n_entries.clone()
    bad[1] = E + 100
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    out = torch.empty(2, 1, top_k, dtype=torch.int32, device=DEV)
    csa.index_topk_static(q_idx, kc, bad, out, max_entries=E, top_k=top_k, status_out=status)
    torch.cuda.synchronize()
    assert int(status.item()) == csa.ERR_DEVICE_CHECK
    csa.index_topk_static(q_idx, kc, n_entries, out, max_entries=E, top_k=top_k, status_out=status)
    torch.cuda.synchronize()
    assert int(status.item()) == csa.OK
    ref, _ = gpu_index(csa, q_idx, kc, n_entries, E, top_k)
    np.testing.assert_array_equal(out.cpu().numpy(), ref.cpu().numpy())
