"""csa_pack_fp4 against the oracle: bit-exact bytes, coarse sums, appends, capacity errors."""

import numpy as np
import pytest
import torch

from oracle import fp4 as o_fp4
from oracle import indexer as o_idx

from _pipeline import to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    from compressed_sparse_attention_merge_b300 import binding
    binding.lib()
    return binding


DEV = "cuda"


def test_latent_pack_bit_exact_ragged(csa):
    g = torch.Generator(device=DEV).manual_seed(1)
    lengths = [401, 2 * 77, 64, 1]                   # odd tail, partial last block, one block, nothing
    T, E = max(lengths), max(lengths) // 2
    x = (torch.randn(4, T, 512, generator=g, device=DEV) *
         torch.where(torch.rand(4, T, 512, generator=g, device=DEV) < 0.01, 8.0, 1.0)).to(torch.bfloat16)
    ws = csa.workspace(256, DEV)
    cache = csa.empty_cache(4, E, 512, DEV)
    for b, n in enumerate(lengths):
        csa.pack_fp4(x[b:b + 1, :n], cache[b:b + 1], merge=2, scale_rule=csa.SCALE_AMAX, max_entries=E, ws=ws)
    assert csa.device_status(ws) == csa.OK
    got = cache.cpu().numpy()
    xf = to_np(x)
    for b, n in enumerate(lengths):
        ref = o_fp4.pack(xf[b, :n], 2, "amax", n_blocks=got.shape[1])
        np.testing.assert_array_equal(got[b], ref, err_msg=f"sequence {b}")


def test_fp32_extremes_bit_exact(csa):
    # saturation (scale 448, codes at 6), subnormal E4M3 scales, zeros of both signs, exact ties
    g = torch.Generator(device=DEV).manual_seed(2)
    n = 512
    base = torch.randn(1, n, 512, generator=g, device=DEV)
    mag = torch.exp2(torch.randint(-16, 14, (1, n, 32, 1), generator=g, device=DEV).float())
    x = (base.view(1, n, 32, 16) * mag).view(1, n, 512)
    x[0, 0, :16] = torch.tensor([6, -6, 3, 0, .25, -.25, .75, 1.25, 1.75, 2.5, 3.5, 5, -5, 1, .5, -0.0])
    x[0, 1, :16] = -0.0
    x[0, 2, :16] = 5000.0
    x[0, 3, :16] = 1e-6
    ws = csa.workspace(256, DEV)
    cache = csa.empty_cache(1, n, 512, DEV)
    csa.pack_fp4(x, cache, merge=1, scale_rule=csa.SCALE_AMAX, max_entries=n, ws=ws)
    ref = o_fp4.pack(x[0].cpu().numpy(), 1, "amax")
    np.testing.assert_array_equal(cache[0].cpu().numpy(), ref)


def test_pow2_keys_and_coarse_sums(csa):
    g = torch.Generator(device=DEV).manual_seed(3)
    for dim in (64, 128, 256):
        E = 512 * 3 + 77
        keys = torch.randint(-4, 5, (2, E, dim), generator=g, device=DEV).float()
        lengths = [E, 512 * 2 + 5]
        ws = csa.workspace(256, DEV)
        coarse = csa.empty_coarse(2, E, dim, DEV)
        cache = csa.empty_cache(2, E, dim, DEV)
        for b in range(2):
            csa.pack_fp4(keys[b:b + 1, :lengths[b]], cache[b:b + 1], merge=1, scale_rule=csa.SCALE_POW2,
                         max_entries=E, ws=ws, coarse_sum=coarse[b:b + 1])
        assert csa.device_status(ws) == csa.OK
        kc = keys.cpu().numpy()
        for b in range(2):
            ref = o_fp4.pack(kc[b, :lengths[b]], 1, "pow2", n_blocks=cache.shape[1])
            np.testing.assert_array_equal(cache[b].cpu().numpy(), ref)
            deq = o_fp4.dequantize(ref, dim, lengths[b])
            c_ref = o_idx.coarse_keys(deq, lengths[b])
            np.testing.assert_array_equal(coarse[b, :c_ref.shape[0]].cpu().numpy(), c_ref)


def test_coarse_sums_are_exact_sums(csa):
    # real-valued keys over a wide range of magnitudes, and a super-block whose sum in entry order in fp32 would
    # lose 170 half-ulp increments: the coarse sums equal the exact sum rounded once, bit for bit
    g = torch.Generator(device=DEV).manual_seed(4)
    for dim in (64, 128, 256):
        E = 512 * 2 + 300
        x = torch.randn(1, E, dim, generator=g, device=DEV)
        x = x * torch.exp2(torch.randint(-12, 9, (1, E, 1), generator=g, device=DEV).float())
        x[0, :342] = 1536.0
        x[0, 342:512] = 2.0 ** -5
        ws = csa.workspace(256, DEV)
        coarse = csa.empty_coarse(1, E, dim, DEV)
        cache = csa.empty_cache(1, E, dim, DEV)
        csa.pack_fp4(x, cache, merge=1, scale_rule=csa.SCALE_POW2, max_entries=E, ws=ws, coarse_sum=coarse)
        assert csa.device_status(ws) == csa.OK
        ref = o_fp4.pack(x[0].cpu().numpy(), 1, "pow2", n_blocks=cache.shape[1])
        np.testing.assert_array_equal(cache[0].cpu().numpy(), ref)
        c_ref = o_idx.coarse_keys(o_fp4.dequantize(ref, dim, E), E)
        assert c_ref[0, 0] == np.float32(525312 + 170 * 2.0 ** -5)
        np.testing.assert_array_equal(coarse[0, :c_ref.shape[0]].cpu().numpy(), c_ref)


def test_append_at_first_entry(csa):
    g = torch.Generator(device=DEV).manual_seed(4)
    E = 3000
    prior = torch.randn(1, 2 * 1037, 512, generator=g, device=DEV).to(torch.bfloat16)
    chunk = torch.randn(1, 2 * 300, 512, generator=g, device=DEV).to(torch.bfloat16)
    ws = csa.workspace(256, DEV)
    cache = csa.empty_cache(1, E, 512, DEV)
    csa.pack_fp4(prior, cache, merge=2, scale_rule=csa.SCALE_AMAX, max_entries=E, ws=ws)
    first = torch.tensor([1037], dtype=torch.int32, device=DEV)
    csa.pack_fp4(chunk, cache, merge=2, scale_rule=csa.SCALE_AMAX, max_entries=E, ws=ws, first_entry=first)
    assert csa.device_status(ws) == csa.OK
    ref = o_fp4.pack(prior[0].float().cpu().numpy(), 2, "amax", n_blocks=cache.shape[1])
    ref = o_fp4.pack(chunk[0].float().cpu().numpy(), 2, "amax", first_entry=1037, base=ref)
    np.testing.assert_array_equal(cache[0].cpu().numpy(), ref)


def test_capacity_overflow_is_reported_not_written(csa):
    x = torch.ones(1, 64, 512, dtype=torch.bfloat16, device=DEV)
    ws = csa.workspace(256, DEV)
    cache = csa.empty_cache(1, 64, 512, DEV)
    first = torch.tensor([40], dtype=torch.int32, device=DEV)      # 40 + 32 > 64
    csa.pack_fp4(x, cache, merge=2, scale_rule=csa.SCALE_AMAX, max_entries=64, ws=ws, first_entry=first)
    assert csa.device_status(ws) == csa.ERR_DEVICE_CHECK
    assert int(cache.sum()) == 0
    assert csa.device_status(ws) == csa.OK                       # reading clears the status word


def test_multi_job_pack_equals_the_single_calls(csa):
    # a decode step's two appends in one launch (latent pair-merge under AMAX at first_entry, index keys
    # under POW2 with coarse sums), plus a job with no whole pair, which is skipped
    g = torch.Generator(device=DEV).manual_seed(6)
    B, E, D = 3, 1200, 128
    lat_prior = torch.randn(B, 2 * 900, 512, generator=g, device=DEV).to(torch.bfloat16)
    lat_new = torch.randn(B, 2 * 3, 512, generator=g, device=DEV).to(torch.bfloat16)
    keys = torch.randint(-4, 5, (B, 903, D), generator=g, device=DEV).float()
    ws = csa.workspace(256, DEV)
    cache = csa.empty_cache(B, E, 512, DEV)
    kcache = csa.empty_cache(B, E, D, DEV)
    coarse = csa.empty_coarse(B, E, D, DEV)
    csa.pack_fp4(lat_prior, cache, merge=2, scale_rule=csa.SCALE_AMAX, max_entries=E, ws=ws)
    csa.pack_fp4(keys[:, :900].contiguous(), kcache, merge=1, scale_rule=csa.SCALE_POW2, max_entries=E, ws=ws,
                 coarse_sum=coarse)
    first = torch.full((B,), 900, dtype=torch.int32, device=DEV)
    odd = torch.ones(B, 1, 512, dtype=torch.bfloat16, device=DEV)
    spare = csa.empty_cache(B, E, 512, DEV)
    csa.pack_fp4_multi([
        (lat_new, cache, dict(merge=2, scale_rule=csa.SCALE_AMAX, max_entries=E, first_entry=first)),
        (keys[:, 900:].contiguous(), kcache, dict(merge=1, scale_rule=csa.SCALE_POW2, max_entries=E,
                                                  first_entry=first, coarse_sum=coarse)),
        (odd, spare, dict(merge=2, scale_rule=csa.SCALE_AMAX, max_entries=E)),
    ], ws=ws)
    assert csa.device_status(ws) == csa.OK
    assert int(spare.sum()) == 0
    lp, ln, kc = to_np(lat_prior), to_np(lat_new), keys.cpu().numpy()
    for b in range(B):
        ref = o_fp4.pack(lp[b], 2, "amax", n_blocks=cache.shape[1])
        ref = o_fp4.pack(ln[b], 2, "amax", first_entry=900, base=ref)
        np.testing.assert_array_equal(cache[b].cpu().numpy(), ref, err_msg=f"latent {b}")
        kref = o_fp4.pack(kc[b], 1, "pow2", n_blocks=kcache.shape[1])
        np.testing.assert_array_equal(kcache[b].cpu().numpy(), kref, err_msg=f"keys {b}")
        c_ref = o_idx.coarse_keys(o_fp4.dequantize(kref, D, 903), 903)
        np.testing.assert_array_equal(coarse[b, :c_ref.shape[0]].cpu().numpy(), c_ref)


def test_multi_job_pack_bulk_and_overflow(csa):
    # a bulk job (one thread per group) next to a small one, then a job that overflows its capacity next
    # to one that fits: the overflow is reported and leaves its cache untouched, the other job is written
    g = torch.Generator(device=DEV).manual_seed(7)
    big = torch.randn(1, 2 * 3000, 512, generator=g, device=DEV).to(torch.bfloat16)
    small = torch.randn(2, 5, 256, generator=g, device=DEV)
    ws = csa.workspace(256, DEV)
    c_big = csa.empty_cache(1, 3000, 512, DEV)
    c_small = csa.empty_cache(2, 5, 256, DEV)
    csa.pack_fp4_multi([(big, c_big, dict(merge=2, scale_rule=csa.SCALE_AMAX, max_entries=3000)),
                        (small, c_small, dict(merge=1, scale_rule=csa.SCALE_AMAX, max_entries=5))], ws=ws)
    assert csa.device_status(ws) == csa.OK
    np.testing.assert_array_equal(c_big[0].cpu().numpy(), o_fp4.pack(to_np(big)[0], 2, "amax"))
    sm = small.cpu().numpy()
    for b in range(2):
        np.testing.assert_array_equal(c_small[b].cpu().numpy(), o_fp4.pack(sm[b], 1, "amax"))

    over = torch.ones(1, 64, 512, dtype=torch.bfloat16, device=DEV)
    c_over = csa.empty_cache(1, 64, 512, DEV)
    first = torch.tensor([40], dtype=torch.int32, device=DEV)      # 40 + 32 > 64
    c_ok = csa.empty_cache(2, 5, 256, DEV)
    csa.pack_fp4_multi([(over, c_over, dict(merge=2, scale_rule=csa.SCALE_AMAX, max_entries=64, first_entry=first)),
                        (small, c_ok, dict(merge=1, scale_rule=csa.SCALE_AMAX, max_entries=5))], ws=ws)
    assert csa.device_status(ws) == csa.ERR_DEVICE_CHECK
    assert int(c_over.sum()) == 0
    np.testing.assert_array_equal(c_ok.cpu().numpy(), c_small.cpu().numpy())
