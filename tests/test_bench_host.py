"""Host-side logic of bench.py, on CPU: the algorithmic byte counts behind the roofline line, the layer
modes of the chain workload against the oracle's, and the workload table against the shapes the method's
configurations state."""

import dataclasses
import bench
from oracle import chain


def test_attention_bytes_per_query():
    # 256 blocks of 2,304 B, 128 window rows of 1,024 B, 64 heads of query (1,024 B) and output
    # (2,048 B), 256 indices of 4 B
    assert bench.attn_bytes_per_query(64, 256, 128) == 256 * 2304 + 128 * 1024 + 64 * 3072 + 256 * 4 == 918_528
    assert 32 * bench.attn_bytes_per_query(64, 256, 128) == 29_392_896
    assert bench.attn_bytes_per_query(16, 64, 128) == 64 * 2304 + 128 * 1024 + 16 * 3072 + 64 * 4


def test_index_bytes_per_entry():
    # one packed key: dim / 2 code bytes and dim / 16 scale bytes
    assert bench.index_bytes_per_entry(128) == 72
    assert bench.index_bytes_per_entry(64) == 36
    assert 32 * 32768 * bench.index_bytes_per_entry(128) == 75_497_472


def test_chain_modes_match_the_oracle():
    assert bench.chain_modes(20) == chain.modes(20, 4)
    m = bench.chain_modes(20)
    assert (m.count("full"), m.count("reindex"), m.count("reuse")) == (1, 4, 15)


def test_workload_table():
    cases = bench._cases()
    assert bench.DEFAULT_WORKLOAD == "decode_64k_b32_h64"
    d = cases["decode_64k_b32_h64"]
    assert (d.batch, d.max_entries, d.heads, d.idx_heads, d.idx_dim, d.top_k, d.window, d.n_query) == \
        (32, 32768, 64, 4, 128, 256, 128, 1)
    t = cases["tiny_decode_4k_b1_h16"]
    assert (t.batch, t.max_entries, t.heads, t.idx_heads, t.idx_dim, t.top_k) == (1, 2048, 16, 1, 64, 64)
    h = cases["decode_1m_b4_h64_hier2048"]
    assert (h.batch, h.max_entries, h.hier_keep, h.top_k) == (4, 1 << 19, 2048, 256)
    c = cases["chain20_128k_b64_h64"]
    assert (c.batch, c.max_entries, c.layers, c.distinct_index_queries) == (64, 65536, 20, 5)
    p = cases["prefill_2048_at_128k_h64"]
    assert (p.chunk, p.max_entries, p.first_pos) == (2048, 65536, 131072 - 2048)
    q = cases["decode_64k_b32_h64_q4"]
    assert (q.batch, q.max_entries, q.n_query) == (32, 32768, 4)
    # the NVFP4-query workload is the decode workload with the other attention: same inputs, same seed
    v = cases["decode_64k_b32_h64_nvfp4q"]
    assert v.nvfp4q and not d.nvfp4q
    assert dataclasses.replace(v, name=d.name, nvfp4q=False) == d
    w = cases["prefill_2048_at_128k_h64_nvfp4q"]
    assert w.nvfp4q and not p.nvfp4q
    assert dataclasses.replace(w, name=p.name, nvfp4q=False) == p
    # every other workload draws from its own seed
    seeds = [cases[k].seed for k in cases if not k.endswith("_nvfp4q")]
    assert len(set(seeds)) == len(seeds)


def test_shards_draw_other_seeds_with_the_same_shapes():
    a, b = bench.shard_case("decode_64k_b32_h64", 0), bench.shard_case("decode_64k_b32_h64", 1)
    assert a.seed != b.seed
    assert (a.batch, a.max_entries, a.top_k) == (b.batch, b.max_entries, b.top_k)


def test_nvfp4q_workloads_share_the_byte_and_flop_models():
    # the NVFP4-query workloads move the same algorithmic bytes (and do the same attention work) as the exact
    # ones: the roofline lines of the two variants are comparable
    import dataclasses as dc
    cases = bench._cases()
    d, v = cases["decode_64k_b32_h64"], cases["decode_64k_b32_h64_nvfp4q"]
    per = bench.attn_bytes_per_query(d.heads, d.top_k, d.window)
    assert per == bench.attn_bytes_per_query(v.heads, v.top_k, v.window) == 918_528
    p, w = cases["prefill_2048_at_128k_h64"], cases["prefill_2048_at_128k_h64_nvfp4q"]
    assert dc.replace(w, name=p.name, nvfp4q=False) == p
