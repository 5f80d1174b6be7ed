"""The workloads of the method at full size, built and run exactly as bench.py times them (one
step of the path), checked against the oracle on sampled sequences, positions and layers:

  * FP4 cache bytes of sampled entries (latent and index key), bit-exact;
  * Top-K indices of sampled sequences / positions, bit-exact (flat, hierarchical, prefill-causal);
  * attention outputs of sampled queries within max-abs 2e-3 and max-rel 1e-2;
  * the layer chain: Full, Reindex and Reuse layers, Reuse indices equal to their source layer's.

The oracle scores every entry of a sampled sequence from its seeded integer index keys; that its own
quantise-dequantise round trip is the identity on such keys is checked first on a sample of rows.
Attention rows are the oracle's own pair-merged, packed and dequantised entries of the blocks its
own Top-K selects, plus the window rows."""

import math

import numpy as np
import pytest
import torch

import bench
from oracle import attention as o_attn
from oracle import fp4 as o_fp4
from oracle import indexer as o_idx

from _pipeline import SCALE, assert_attn_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _exact_keys(keys_np, rng):
    """The integer keys themselves, after checking on 512 random rows that the oracle's POW2 pack and
    dequantisation reproduce them exactly."""
    rows = rng.choice(keys_np.shape[0], size=min(512, keys_np.shape[0]), replace=False)
    sample = keys_np[rows]
    deq = o_fp4.dequantize(o_fp4.pack(sample, 1, "pow2"), sample.shape[1], sample.shape[0])
    np.testing.assert_array_equal(deq, sample)
    return keys_np.astype(np.float64)


def _pairs(tok, entries):
    """Token pairs (2e, 2e + 1) of the given entries from a device tensor [T, 512], as float32 [n, 2, 512]."""
    e = torch.as_tensor(np.asarray(entries, np.int64), device=tok.device)
    rows = torch.stack([2 * e, 2 * e + 1], dim=1).reshape(-1)
    return to_np(tok[rows]).reshape(len(entries), 2, -1)


def _check_pack(cache_b, tok, keys_b, kcache_b, entries, idx_dim):
    """Bytes of the given entries in the GPU caches against the oracle's pack of the same inputs."""
    pairs = _pairs(tok, entries)
    half, nsc = idx_dim // 2, idx_dim // 16
    for k, e in enumerate(entries):
        s = e % 8
        blk = o_fp4.pack(pairs[k], 2, "amax", first_entry=s, n_blocks=1)[0]
        got = cache_b[e // 8]
        np.testing.assert_array_equal(got[256 * s:256 * s + 256], blk[256 * s:256 * s + 256], err_msg=f"entry {e}")
        np.testing.assert_array_equal(got[2048 + 32 * s:2048 + 32 * s + 32], blk[2048 + 32 * s:2048 + 32 * s + 32])
        kb = o_fp4.pack(keys_b[e:e + 1], 1, "pow2", first_entry=s, n_blocks=1)[0]
        gk = kcache_b[e // 8]
        np.testing.assert_array_equal(gk[s * half:(s + 1) * half], kb[s * half:(s + 1) * half])
        np.testing.assert_array_equal(gk[8 * half + s * nsc:8 * half + (s + 1) * nsc],
                                      kb[8 * half + s * nsc:8 * half + (s + 1) * nsc])


def _oracle_rows(tok, blocks, eligible):
    """Dequantised entries of the listed blocks (in listing order) that pass `eligible(e)`: each is the
    oracle's pair-merge and FP4 pack of the entry's two tokens, dequantised."""
    entries = [e for b in blocks if b >= 0 for e in range(8 * b, 8 * b + 8) if eligible(e)]
    if not entries:
        return np.zeros((0, 512))
    pairs = _pairs(tok, entries)
    rows = [o_fp4.dequantize(o_fp4.pack(pairs[k], 2, "amax", n_blocks=1), 512, 1)[0] for k in range(len(entries))]
    return np.stack(rows)


def _decode_case(name, samples, layer_checks=None):
    w = bench.make_workload(name, DEV, replicas=1, keep_inputs=True)
    c = w.case
    L = len(w.modes)
    outs = [torch.empty_like(w.out) for _ in range(L)]
    w.step(0, layer_outs=outs)
    torch.cuda.synchronize()
    assert w.csa.device_status(w.ws_attn) == w.csa.OK and w.csa.device_status(w.ws_index) == w.csa.OK
    rng = np.random.default_rng(7)
    d = w.inputs
    E = w.E
    for b in samples:
        tok = d["tokens"][b]
        keys_np = d["keys"][b].cpu().numpy()
        keys = _exact_keys(keys_np, rng)
        probe = sorted(set(rng.choice(E, 24, replace=False).tolist()) | {0, E - 1})
        _check_pack(w.caches[0][b].cpu().numpy(), tok, keys_np, w.kcaches[0][b].cpu().numpy(), probe, c.idx_dim)
        sources, n_idx, src = [], 0, 0
        ref_idx = {}
        q_pos = d["q_pos"][b].cpu().numpy() if c.causal_drafts else None
        for layer, mode in enumerate(w.modes):
            if mode != "reuse":
                src = n_idx
                q_idx = d["q_idx"][n_idx % d["q_idx"].shape[0], b].cpu().numpy()
                if c.hier_keep:
                    ref, _ = o_idx.hierarchical_topk(q_idx, keys, E, c.top_k, c.hier_keep)
                else:
                    ref, _ = o_idx.flat_topk(q_idx, keys, E, c.top_k, q_pos=q_pos)
                np.testing.assert_array_equal(w.idx[src][b].cpu().numpy(), ref, err_msg=f"{name} seq {b} layer {layer}")
                ref_idx[src] = ref
                n_idx += 1
            sources.append(src)
        for layer in (layer_checks if layer_checks is not None else range(L)):
            ref = ref_idx[sources[layer]]
            for j in range(c.n_query):
                if q_pos is None:
                    swa = to_np(d["swa"][layer, b])[:int(d["swa_len"][b])].astype(np.float64)
                    rows = _oracle_rows(tok, ref[j], lambda e: e < E)
                else:
                    p = int(q_pos[j])
                    swa = o_attn.prefill_window(to_np(d["swa"][layer, b]), int(d["swa_first_pos"][b]), p, c.window)
                    rows = _oracle_rows(tok, ref[j], lambda e, p=p: e < E and 2 * e + 1 <= p)
                q = to_np(d["q"][layer, b, j]).astype(np.float64)
                if c.nvfp4q:
                    # the NVFP4-query attention: rounded query heads and window keys in the logits, exact values
                    keys = np.concatenate([rows, o_fp4.round_trip(np.asarray(swa, np.float32), "amax")])
                    want, _ = o_attn.attend_kv(o_attn.nvfp4_query(q.astype(np.float32)), keys,
                                               np.concatenate([rows, swa]), SCALE)
                else:
                    want, _ = o_attn.attend(q, np.concatenate([rows, swa]), SCALE)
                assert_attn_close(outs[layer][b, j, :c.heads].cpu().numpy(), want[:c.heads],
                                  f"{name} seq {b} layer {layer} ({w.modes[layer]})")
    return w


def test_tiny_decode_4k():
    _decode_case("tiny_decode_4k_b1_h16", samples=[0])


def test_decode_64k_batch32():
    _decode_case("decode_64k_b32_h64", samples=[0, 31])


def test_decode_64k_batch32_four_query_positions():
    _decode_case("decode_64k_b32_h64_q4", samples=[0, 31])


def test_decode_64k_batch32_nvfp4q():
    _decode_case("decode_64k_b32_h64_nvfp4q", samples=[0, 31])


def test_decode_1m_hierarchical():
    _decode_case("decode_1m_b4_h64_hier2048", samples=[2])


def test_chain_20_layers_128k_batch64():
    w = _decode_case("chain20_128k_b64_h64", samples=[5], layer_checks=[0, 1, 4, 7, 19])
    # Reuse layers attend with exactly their source layer's indices (one index buffer per Full/Reindex)
    assert len(w.idx) == sum(m != "reuse" for m in w.modes) == 5


def test_prefill_2048_at_128k():
    _prefill_case("prefill_2048_at_128k_h64")


def test_prefill_2048_at_128k_nvfp4q():
    _prefill_case("prefill_2048_at_128k_h64_nvfp4q")


def _prefill_case(name):
    w = bench.make_workload(name, DEV, replicas=1, keep_inputs=True)
    c = w.case
    w.step(0)
    torch.cuda.synchronize()
    assert w.csa.device_status(w.ws_attn) == w.csa.OK and w.csa.device_status(w.ws_index) == w.csa.OK
    d = w.inputs
    E, P, C = w.E, c.first_pos, c.chunk
    rng = np.random.default_rng(8)
    tok = torch.cat([d["prior"][0], d["chunk"][0]])
    keys_np = d["keys"][0].cpu().numpy()
    keys = _exact_keys(keys_np, rng)
    probe = sorted(set(rng.choice(E, 24, replace=False).tolist()) | {P // 2, P // 2 + 1, E - 1})
    _check_pack(w.caches[0][0].cpu().numpy(), tok, keys_np, w.kcaches[0][0].cpu().numpy(), probe, c.idx_dim)
    js = [0, 1, 2, 127, 128, 1000, C - 2, C - 1]
    pos = d["q_pos"][0].cpu().numpy()[js]
    ref, _ = o_idx.flat_topk(d["q_idx"][0].cpu().numpy()[js], keys, E, c.top_k, q_pos=pos)
    np.testing.assert_array_equal(w.idx[0].cpu().numpy()[js], ref)
    swa = to_np(d["swa"][0])
    first = int(d["swa_first_pos"][0])
    out = w.out[0].cpu().numpy()
    for k, j in enumerate(js):
        p = int(pos[k])
        rows = _oracle_rows(tok, ref[k], lambda e: e < E and 2 * e + 1 <= p)
        win = o_attn.prefill_window(swa, first, p, c.window)
        qj = to_np(d["q"][0, j]).astype(np.float64)
        if c.nvfp4q:
            keys = np.concatenate([rows, o_fp4.round_trip(np.asarray(win, np.float32), "amax")])
            want, _ = o_attn.attend_kv(o_attn.nvfp4_query(qj.astype(np.float32)), keys, np.concatenate([rows, win]),
                                       SCALE)
        else:
            want, _ = o_attn.attend(qj, np.concatenate([rows, win]), SCALE)
        assert_attn_close(out[j], want, f"{name} position {p}")


def test_chain_step_as_one_graph_replays_the_eager_step():
    # the 20-layer chain through the library's multi-layer entry point (csa_decode_layers) at a smaller size
    # (4 sequences of 8K tokens): captured once as a CUDA graph and replayed, it reproduces the eager step bit
    # for bit, and sampled layers match the oracle (Reuse layers with their source layer's indices)
    import dataclasses
    from compressed_sparse_attention_merge_b300 import synth
    case = dataclasses.replace(synth.CHAIN_128K_B64, name="chain20_8k_b4", tokens=[8192] * 4, seed=20299)
    w = bench.DecodeWorkload(case, torch.device(DEV), replicas=1, keep_inputs=True)
    L = len(w.modes)
    eager = [torch.empty_like(w.out) for _ in range(L)]
    graphed = [torch.full_like(w.out, float("nan")) for _ in range(L)]
    w.step(0, layer_outs=eager)
    torch.cuda.synchronize()
    idx_eager = [t.clone() for t in w.idx]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w.step(0, layer_outs=graphed)
    for t in w.idx:
        t.fill_(-9)
    g.replay()
    torch.cuda.synchronize()
    assert w.csa.device_status(w.ws_attn) == w.csa.OK and w.csa.device_status(w.ws_index) == w.csa.OK
    for layer in range(L):
        assert torch.equal(graphed[layer], eager[layer]), f"layer {layer}"
    for a, b in zip(w.idx, idx_eager):
        assert torch.equal(a, b)
    d = w.inputs
    E, b = w.E, 1
    tok = d["tokens"][b]
    keys = d["keys"][b].cpu().numpy().astype(np.float64)
    n_idx, src, ref_idx = 0, 0, {}
    sources = []
    for layer, mode in enumerate(w.modes):
        if mode != "reuse":
            src = n_idx
            ref, _ = o_idx.flat_topk(d["q_idx"][n_idx % d["q_idx"].shape[0], b].cpu().numpy(), keys, E, case.top_k)
            np.testing.assert_array_equal(w.idx[src][b].cpu().numpy(), ref, err_msg=f"layer {layer}")
            ref_idx[src] = ref
            n_idx += 1
        sources.append(src)
    for layer in (0, 1, 4, 5, 19):
        ref = ref_idx[sources[layer]]
        rows = _oracle_rows(tok, ref[0], lambda e: e < E)
        swa = to_np(d["swa"][layer, b])[:int(d["swa_len"][b])].astype(np.float64)
        want, _ = o_attn.attend(to_np(d["q"][layer, b, 0]).astype(np.float64), np.concatenate([rows, swa]), SCALE)
        assert_attn_close(graphed[layer][b, 0].cpu().numpy(), want, f"layer {layer} ({w.modes[layer]})")
