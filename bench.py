"""Benchmark of the CSA2 sparse-attention hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step is one pass of the whole path over one batch of synthetic input:
  decode workloads   re-pack the newest merged entry of every sequence (latent and index key; the bytes
                     written equal the ones already there, so the cache stays fixed across steps),
                     index + Top-K (flat or hierarchical), sparse decode attention with the window;
                     the layer chain runs this per layer with the Full / Reindex / Reuse pattern.
  prefill workload   pair-merge + FP4-pack the chunk, per-position index + Top-K, sparse prefill attention.

The default workload is decode at 64K tokens, batch 32, 64 heads. Each rank holds its own batch (weak
scaling, no collective on the data path); rank 0 prints one JSON line. `value` is query tokens per
second over all ranks with inputs resident in HBM; `e2e` repeats the measurement with the step's
inputs copied from pinned host memory and the attention output copied back inside the timed region.

L2: every timed step reads one of several cache replicas in rotation, so the touched set is larger
than the 126 MB L2. Per-kernel times come from the library's CUDA-event hooks on the launch stream.
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "decode query-tokens/s and achieved HBM GB/s for CSA2 sparse attn, 64K–1M ctx"
UNIT = "query-tokens/s"
SCALE = 1.0 / math.sqrt(512)
L2_BYTES = 126 * 1024 * 1024


# ------------------------------------------------------------------------------------------------
# Workloads
# ------------------------------------------------------------------------------------------------

def _cases():
    from compressed_sparse_attention_merge_b300 import synth
    return {
        "tiny_decode_4k_b1_h16": synth.TINY_DECODE_4K,
        "decode_64k_b32_h64": synth.DECODE_64K_B32,
        "decode_1m_b4_h64_hier2048": synth.DECODE_1M_B4_HIER,
        "chain20_128k_b64_h64": synth.CHAIN_128K_B64,
        "prefill_2048_at_128k_h64": synth.PREFILL_2K_AT_128K,
        "decode_64k_b32_h64_q4": synth.DECODE_64K_B32_Q4,
        "decode_64k_b32_h64_nvfp4q": synth.DECODE_64K_B32_NVFP4Q,
        "prefill_2048_at_128k_h64_nvfp4q": synth.PREFILL_2K_AT_128K_NVFP4Q,
        "project_pack_128k_h4096": synth.PROJECT_128K_H4096,
    }


DEFAULT_WORKLOAD = "decode_64k_b32_h64"


def chain_modes(n_layers):
    """Layer modes of the chain: layer 0 Full, every fourth layer Reindex, the rest Reuse."""
    return ["full" if l == 0 else ("reindex" if l % 4 == 0 else "reuse") for l in range(n_layers)]


def attn_bytes_per_query(heads, top_k, window):
    """Algorithmic HBM bytes of one decode query's attention: the selected blocks (2,304 B each), the
    window rows (1,024 B), the query (1,024 B per head), the output (2,048 B per head), the indices."""
    return 2304 * top_k + 1024 * window + 1024 * heads + 2048 * heads + 4 * top_k


def index_bytes_per_entry(idx_dim):
    """Algorithmic HBM bytes per scored entry: its packed index key (dim/2 codes + dim/16 scales)."""
    return idx_dim // 2 + idx_dim // 16


class DecodeWorkload:
    """Packed caches, queries and windows of a decode workload on one device, with `replicas` copies
    of the caches so that consecutive steps read different memory."""

    def __init__(self, case, device, replicas, keep_inputs=False):
        from compressed_sparse_attention_merge_b300 import binding as csa
        from compressed_sparse_attention_merge_b300 import synth
        self.csa, self.case, self.device = csa, case, device
        d = synth.make_decode(case, device)
        self.inputs = dict(d) if keep_inputs else None
        B, E, T = case.batch, case.max_entries, case.max_tokens
        self.B, self.E = B, E
        self.hier = case.hier_keep > 0
        ws = csa.workspace(256, device)
        cache = csa.empty_cache(B, E, 512, device)
        csa.pack_fp4(d["tokens"], cache, merge=2, scale_rule=csa.SCALE_AMAX, max_entries=E, ws=ws)
        kcache = csa.empty_cache(B, E, case.idx_dim, device)
        coarse = csa.empty_coarse(B, E, case.idx_dim, device) if self.hier else None
        csa.pack_fp4(d["keys"], kcache, merge=1, scale_rule=csa.SCALE_POW2, max_entries=E, ws=ws,
                     coarse_sum=coarse)
        if csa.device_status(ws) != csa.OK:
            raise RuntimeError("cache construction reported a device check")
        # the step's new tokens and index keys: the tokens of the entries the step's query positions complete
        # (the newest pair for one query; the pairs of the drafts for causal draft positions); re-packing
        # them rewrites those entries with the same bytes
        lo = 2 * ((T - case.n_query) // 2)
        self.new_tokens = d["tokens"][:, lo:T].contiguous()
        n_new = (T - lo) // 2
        self.new_keys = d["keys"][:, E - n_new:E].contiguous()
        self.first = (d["n_entries"] - n_new).contiguous()
        del d["tokens"], d["keys"]
        self.n_entries = d["n_entries"]
        self.q, self.q_idx, self.swa, self.swa_len = d["q"], d["q_idx"], d["swa"], d["swa_len"]
        self.causal = case.causal_drafts
        self.q_pos, self.swa_first_pos = d.get("q_pos"), d.get("swa_first_pos")
        self.caches = [cache] + [cache.clone() for _ in range(replicas - 1)]
        self.kcaches = [kcache] + [kcache.clone() for _ in range(replicas - 1)]
        self.coarses = [coarse] * replicas if coarse is None else [coarse] + [coarse.clone() for _ in
                                                                             range(replicas - 1)]
        self.layers = case.layers
        self.modes = chain_modes(case.layers) if case.layers > 1 else ["full"]
        n_idx_layers = sum(m != "reuse" for m in self.modes)
        K = case.top_k
        self.idx = [torch.empty(B, case.n_query, K, dtype=torch.int32, device=device) for _ in range(n_idx_layers)]
        self.out = torch.empty(B, case.n_query, case.heads, 512, dtype=torch.float32, device=device)
        ia = csa.index_args(self.q_idx[0], kcache, self.n_entries, self.idx[0], max_entries=E, top_k=K,
                            coarse_sum=coarse, keep_blocks=case.hier_keep, q_pos=self.q_pos)
        self.ws_index = csa.workspace(csa.index_topk_workspace_size(B, ia), device)
        # one pair of templates per cache replica (their pointers are the only per-replica fields)
        self.index_tmpl = [csa.index_args(self.q_idx[0], self.kcaches[r], self.n_entries, self.idx[0], max_entries=E,
                                          top_k=K, coarse_sum=self.coarses[r], keep_blocks=case.hier_keep,
                                          q_pos=self.q_pos) for r in range(replicas)]
        if self.causal:
            aa = csa.attn_args(self.q[0], cache, self.n_entries, self.idx[0], self.out, max_entries=E,
                               window=case.window, scale=SCALE, swa=self.swa[0], swa_first_pos=self.swa_first_pos,
                               q_pos=self.q_pos)
        else:
            aa = csa.attn_args(self.q[0], cache, self.n_entries, self.idx[0], self.out, max_entries=E,
                               window=case.window, scale=SCALE, swa=self.swa[0], swa_len=self.swa_len)
        self.ws_attn = csa.workspace(csa.sparse_attn_workspace_size(B, aa), device)
        if self.causal:
            self.attn_tmpl = [csa.attn_args(self.q[0], self.caches[r], self.n_entries, self.idx[0], self.out,
                                            max_entries=E, window=case.window, scale=SCALE, swa=self.swa[0],
                                            swa_first_pos=self.swa_first_pos, q_pos=self.q_pos)
                              for r in range(replicas)]
        else:
            self.attn_tmpl = [csa.attn_args(self.q[0], self.caches[r], self.n_entries, self.idx[0], self.out,
                                            max_entries=E, window=case.window, scale=SCALE, swa=self.swa[0],
                                            swa_len=self.swa_len) for r in range(replicas)]
        self.ws_pack = ws
        self.queries_per_step = B * case.n_query

    def step(self, r, q=None, q_idx=None, new_tokens=None, new_keys=None, out=None, layer_outs=None):
        """One decode step on replica r. Optional arguments replace the resident inputs (end-to-end
        mode passes freshly copied ones); layer_outs, if given, receives every layer's output."""
        csa, c = self.csa, self.case
        q = self.q if q is None else q
        q_idx = self.q_idx if q_idx is None else q_idx
        new_tokens = self.new_tokens if new_tokens is None else new_tokens
        new_keys = self.new_keys if new_keys is None else new_keys
        out = self.out if out is None else out
        cache, kcache, coarse = self.caches[r], self.kcaches[r], self.coarses[r]
        # both appends (latent pair, index key) in one launch
        csa.pack_fp4_multi([
            (new_tokens, cache, dict(merge=2, scale_rule=csa.SCALE_AMAX, max_entries=self.E, first_entry=self.first)),
            (new_keys, kcache, dict(merge=1, scale_rule=csa.SCALE_POW2, max_entries=self.E, first_entry=self.first,
                                    coarse_sum=coarse))], ws=self.ws_pack)
        # every layer (indexer for Full / Reindex, attention) through the library's multi-layer entry point
        layers, n_idx = [], 0
        for layer, mode in enumerate(self.modes):
            ent = {"mode": mode, "q": q[layer], "swa": self.swa[layer], "nvfp4q": c.nvfp4q,
                   "out": out if layer_outs is None else layer_outs[layer]}
            if mode != "reuse":
                ent["q_idx"] = q_idx[n_idx % q_idx.shape[0]]
                ent["idx"] = self.idx[n_idx]
                n_idx += 1
            layers.append(ent)
        csa.decode_layers(layers, index_tmpl=self.index_tmpl[r], attn_tmpl=self.attn_tmpl[r], ws_index=self.ws_index,
                          ws_attn=self.ws_attn)
        return out

    def algorithmic_bytes(self):
        """Per-kernel algorithmic HBM bytes of one step: {kernel: bytes per launch}."""
        c = self.case
        B = self.B
        per_q = attn_bytes_per_query(c.heads, c.top_k, c.window)
        out = {"sparse_attn": B * c.n_query * per_q}
        if self.hier:
            keep = c.hier_keep
            n_super = -(-self.E // 512)
            out["coarse_score"] = B * c.n_query * n_super * c.idx_dim * 4
            out["index_score_hier"] = B * c.n_query * keep * 8 * index_bytes_per_entry(c.idx_dim)
        else:
            out["index_score"] = B * self.E * index_bytes_per_entry(c.idx_dim)
        return out

    def step_bytes(self):
        c = self.case
        per = self.algorithmic_bytes()
        n_idx = sum(m != "reuse" for m in self.modes)
        total = per["sparse_attn"] * len(self.modes)
        for k, v in per.items():
            if k != "sparse_attn":
                total += v * n_idx
        return total

    def h2d_inputs(self):
        """The tensors a caller supplies per step (copied from pinned host memory in e2e mode)."""
        return {"q": self.q, "q_idx": self.q_idx, "new_tokens": self.new_tokens, "new_keys": self.new_keys}


class PrefillWorkload:
    """A prefill chunk at the end of a long context: the prior cache is built once; each step packs the
    chunk, selects per position and attends."""

    def __init__(self, case, device, replicas, keep_inputs=False):
        from compressed_sparse_attention_merge_b300 import binding as csa
        from compressed_sparse_attention_merge_b300 import synth
        self.csa, self.case, self.device = csa, case, device
        d = synth.make_prefill(case, device)
        self.inputs = dict(d) if keep_inputs else None
        E, P = case.max_entries, case.first_pos
        self.E = E
        ws = csa.workspace(256, device)
        cache = csa.empty_cache(1, E, 512, device)
        csa.pack_fp4(d["prior"], cache, merge=2, scale_rule=csa.SCALE_AMAX, max_entries=E, ws=ws)
        kcache = csa.empty_cache(1, E, case.idx_dim, device)
        csa.pack_fp4(d["keys"], kcache, merge=1, scale_rule=csa.SCALE_POW2, max_entries=E, ws=ws)
        if csa.device_status(ws) != csa.OK:
            raise RuntimeError("cache construction reported a device check")
        self.ws_pack = ws
        self.chunk = d["chunk"]
        self.chunk_keys = d["keys"][:, P // 2:].contiguous()
        self.first = torch.tensor([P // 2], dtype=torch.int32, device=device)
        self.caches = [cache] + [cache.clone() for _ in range(replicas - 1)]
        self.kcaches = [kcache] + [kcache.clone() for _ in range(replicas - 1)]
        self.q, self.q_idx, self.q_pos = d["q"], d["q_idx"], d["q_pos"]
        self.swa, self.swa_first_pos, self.n_entries = d["swa"], d["swa_first_pos"], d["n_entries"]
        C = case.chunk
        self.idx = torch.empty(1, C, case.top_k, dtype=torch.int32, device=device)
        self.out = torch.empty(1, C, case.heads, 512, dtype=torch.float32, device=device)
        ia = csa.index_args(self.q_idx, kcache, self.n_entries, self.idx, max_entries=E, top_k=case.top_k,
                            q_pos=self.q_pos)
        self.ws_index = csa.workspace(csa.index_topk_workspace_size(1, ia), device)
        aa = csa.attn_args(self.q, cache, self.n_entries, self.idx, self.out, max_entries=E, window=case.window,
                           scale=SCALE, swa=self.swa, swa_first_pos=self.swa_first_pos, q_pos=self.q_pos)
        self.ws_attn = csa.workspace(csa.sparse_attn_workspace_size(1, aa), device)
        self.queries_per_step = C
        self.modes = ["full"]

    def step(self, r, q=None, q_idx=None, new_tokens=None, new_keys=None, out=None):
        csa, c = self.csa, self.case
        q = self.q if q is None else q
        q_idx = self.q_idx if q_idx is None else q_idx
        chunk = self.chunk if new_tokens is None else new_tokens
        ckeys = self.chunk_keys if new_keys is None else new_keys
        out = self.out if out is None else out
        cache, kcache = self.caches[r], self.kcaches[r]
        csa.pack_fp4_multi([
            (chunk, cache, dict(merge=2, scale_rule=csa.SCALE_AMAX, max_entries=self.E, first_entry=self.first)),
            (ckeys, kcache, dict(merge=1, scale_rule=csa.SCALE_POW2, max_entries=self.E, first_entry=self.first))],
            ws=self.ws_pack)
        csa.index_topk(q_idx, kcache, self.n_entries, self.idx, max_entries=self.E, top_k=c.top_k,
                       ws=self.ws_index, q_pos=self.q_pos)
        attn = csa.sparse_attn_prefill_nvfp4q if c.nvfp4q else csa.sparse_attn_prefill
        attn(q, cache, self.n_entries, self.idx, out, q_pos=self.q_pos, max_entries=self.E, window=c.window,
             scale=SCALE, ws=self.ws_attn, swa=self.swa, swa_first_pos=self.swa_first_pos)
        return out

    def flops(self):
        """Algorithmic FLOPs per step: the indexer's dense product over eligible entries and the
        attention's two products over the selected entries and the window rows (per position)."""
        c = self.case
        P = c.first_pos
        idx_flops = 0
        att_rows = 0
        for j in range(c.chunk):
            p = P + j
            eligible = min(self.E, (p + 1) // 2)
            idx_flops += 2 * c.idx_heads * c.idx_dim * eligible
            att_rows += min(c.top_k * 8, eligible) + min(c.window, p - (P - c.window + 1) + 1)
        return {"index_score": idx_flops, "sparse_attn": 4 * c.heads * 512 * att_rows}

    def algorithmic_bytes(self):
        c = self.case
        return {"index_score": self.E * index_bytes_per_entry(c.idx_dim),
                "sparse_attn": c.chunk * attn_bytes_per_query(c.heads, c.top_k, c.window)}

    def step_bytes(self):
        return sum(self.algorithmic_bytes().values())

    def h2d_inputs(self):
        return {"q": self.q, "q_idx": self.q_idx, "new_tokens": self.chunk, "new_keys": self.chunk_keys}


class ProjectWorkload:
    """The cache write path: each step projects every hidden row of the batch to the latent and pair-merges
    and FP4-packs the result into the cache (csa_project_pack, one kernel)."""

    metric = "cache-write tokens/s (latent projection + pair-merge + FP4 pack)"
    unit = "tokens/s"
    dtype = "bf16 mma f32 accumulate, fp4-e2m1/e4m3 cache"

    def __init__(self, case, device, replicas, keep_inputs=False):
        from compressed_sparse_attention_merge_b300 import binding as csa
        from compressed_sparse_attention_merge_b300 import synth
        self.csa, self.case, self.device = csa, case, device
        d = synth.make_project(case, device)
        self.h, self.w = d["h"], d["w"]
        self.E = case.tokens // 2
        self.caches = [csa.empty_cache(case.batch, self.E, 512, device) for _ in range(replicas)]
        self.out = self.caches[0]
        self.ws_pack = csa.workspace(256, device)
        self.queries_per_step = case.batch * case.tokens
        self.modes = ["project"]

    def step(self, r, new_tokens=None, out=None, **_):
        h = self.h if new_tokens is None else new_tokens
        cache = self.caches[r] if out is None else out
        self.csa.project_pack(h, self.w, cache, scale_rule=self.csa.SCALE_AMAX, max_entries=self.E, ws=self.ws_pack)
        return cache

    def flops(self):
        c = self.case
        return {"project_pack": 2 * c.batch * c.tokens * c.hidden * 512}

    def algorithmic_bytes(self):
        c = self.case
        return {"project_pack": c.batch * c.tokens * c.hidden * 2 + 512 * c.hidden * 2 + c.batch * self.E * 288}

    def step_bytes(self):
        return sum(self.algorithmic_bytes().values())

    def h2d_inputs(self):
        return {"new_tokens": self.h}


def shard_case(name, shard):
    """The workload's case for one rank: rank r draws its own sequences (seed offset by 1000 r), so that N
    ranks hold N different shards of one global batch."""
    import dataclasses
    case = _cases()[name]
    return dataclasses.replace(case, seed=case.seed + 1000 * shard) if shard else case


def make_workload(name, device, replicas, keep_inputs=False, shard=0, batch=None):
    """The named workload; `batch` (decode workloads only) replaces the number of sequences, each as long as
    the workload's first."""
    import dataclasses
    case = shard_case(name, shard)
    if batch is not None:
        if not hasattr(case, "tokens") or not isinstance(case.tokens, list):
            raise ValueError("--batch applies to decode workloads")
        case = dataclasses.replace(case, tokens=[case.tokens[0]] * batch, swa_len=None)
    if name.startswith("project"):
        return ProjectWorkload(case, device, replicas, keep_inputs)
    if name.startswith("prefill"):
        return PrefillWorkload(case, device, replicas, keep_inputs)
    return DecodeWorkload(case, device, replicas, keep_inputs)


def touched_bytes(w):
    return w.step_bytes() if not isinstance(w, PrefillWorkload) else w.step_bytes()


# ------------------------------------------------------------------------------------------------
# Clocks
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


# ------------------------------------------------------------------------------------------------
# Our arm
# ------------------------------------------------------------------------------------------------

def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args):
    from compressed_sparse_attention_merge_b300 import binding as csa
    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    csa.lib()

    w = make_workload(args.workload, device, args.replicas, shard=rank, batch=args.batch)
    R = args.replicas
    stream = torch.cuda.current_stream(device)

    # eager warm-up: the first launches on the device set kernel attributes outside any capture
    for i in range(args.warmup):
        w.step(i % R)
    torch.cuda.synchronize(device)

    # one CUDA graph per cache replica holds a whole step; the timed loop replays them in rotation
    graphs = []
    for r in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            w.step(r)
        graphs.append(g)
    for i in range(args.warmup):
        graphs[i % R].replay()
    torch.cuda.synchronize(device)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    # The timed window is exactly K steps; it is repeated (the same K steps, back to back) until about
    # args.min_seconds have passed, so that the clock record holds many samples under load, and the median
    # window is reported with the repeat count.
    per_window = []
    t_begin = time.perf_counter()
    while True:
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _barrier(world)
        torch.cuda.synchronize(device)
        start.record(stream)
        for i in range(args.steps):
            graphs[i % R].replay()
        stop.record(stream)
        torch.cuda.synchronize(device)
        _barrier(world)
        per_window.append(start.elapsed_time(stop) / args.steps)
        done = len(per_window) >= 3 and time.perf_counter() - t_begin >= args.min_seconds
        if world > 1:
            flag = torch.tensor([1.0 if done else 0.0], device=device)
            import torch.distributed as dist
            dist.all_reduce(flag, op=dist.ReduceOp.MIN)
            done = flag.item() > 0.5
        if done or len(per_window) >= 100000:
            break
    clocks = sampler.stop() if sampler else None
    ms = statistics.median(per_window)
    ms = _max_over_ranks(ms, world, device)
    value = world * w.queries_per_step / (ms * 1e-3)

    # per-kernel device times: the same K steps captured with the library's event hooks (event nodes on
    # the launch stream around every kernel), replayed once
    csa.profile_begin(64 * args.steps * max(1, len(w.modes)) + 64)
    gp = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gp):
        for i in range(args.steps):
            w.step(i % R)
    gp.replay()
    torch.cuda.synchronize(device)
    kt, dropped = csa.profile_end()
    launches = sum(n for n, _ in kt.values())
    del gp

    # end to end through the binding: per step, H2D of the step's inputs from pinned host memory, the
    # path, D2H of the attention output; captured per replica like the device-resident steps, and also
    # run eagerly (one Python call per entry point) for comparison
    host_in = {k: v.to("cpu").pin_memory() for k, v in w.h2d_inputs().items()}
    dev_in = {k: torch.empty_like(v) for k, v in w.h2d_inputs().items()}
    host_out = torch.empty(w.out.shape, dtype=w.out.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step(r):
        for k in host_in:
            dev_in[k].copy_(host_in[k], non_blocking=True)
        out = w.step(r, **dev_in)
        host_out.copy_(out, non_blocking=True)

    def timed(fn):
        for i in range(args.warmup):
            fn(i % R)
        torch.cuda.synchronize(device)
        _barrier(world)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            fn(i % R)
        t1.record(stream)
        torch.cuda.synchronize(device)
        _barrier(world)
        return _max_over_ranks(t0.elapsed_time(t1) / args.steps, world, device)

    e2e_graphs = []
    for r in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            e2e_step(r)
        e2e_graphs.append(g)
    e2e_serial_ms = timed(lambda r: e2e_graphs[r].replay())
    e2e_eager_ms = timed(e2e_step)
    del e2e_graphs, graphs
    e2e_ms = e2e_pipelined(w, host_in, args, world, device, stream)
    # a device check or a bounded wait that gave up in any run above voids the measurement
    for ws_name in [n for n in ("ws_pack", "ws_index", "ws_attn") if hasattr(w, n)]:
        st = csa.device_status(getattr(w, ws_name))
        if st != csa.OK:
            raise RuntimeError(f"{ws_name}: device status {st} after the timed runs")

    peaks = _peaks()
    kernels = {}
    alg = w.algorithmic_bytes()
    flops = w.flops() if hasattr(w, "flops") else {}
    for name, (n, tot) in kt.items():
        avg_ms = tot / n
        ent = {"launches_per_step": n / args.steps, "avg_ms": round(avg_ms, 5),
               "share": round(tot / sum(t for _, t in kt.values()), 4)}
        if name in alg:
            ent["alg_bytes_per_launch"] = alg[name]
            ent["achieved_gbs"] = round(alg[name] / (avg_ms * 1e-3) / 1e9, 1)
            ent["frac_hbm"] = round(ent["achieved_gbs"] / peaks["hbm_gbs"], 4)
        if name in flops:
            per_launch = flops[name] / max(1.0, n / args.steps)
            ent["flops_per_launch"] = per_launch
            ent["achieved_tflops"] = round(per_launch / (avg_ms * 1e-3) / 1e12, 2)
        kernels[name] = ent
    # the dominant kernel: the one with the largest total time among those with a roofline model (algorithmic
    # bytes or FLOPs), else the largest overall
    modelled = [kv for kv in kt.items() if kv[0] in alg or kv[0] in flops]
    dom = max(modelled or list(kt.items()), key=lambda kv: kv[1][1])[0]
    if dom in flops:
        # the burst peak, unless the clock record shows the power cap active during the timed loop: then the
        # kernel ran in the regime of the sustained (power-capped) peak
        capped = bool(clocks) and "sw_power_cap" in clocks.get("reasons", []) and peaks["bf16_tflops_sustained"]
        peak = peaks["bf16_tflops_sustained"] if capped else peaks["bf16_tflops"]
        achieved = kernels[dom]["achieved_tflops"]
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": TRAFFIC.get((args.workload, dom)),
                "peak_source": peaks["source"] + (" bf16 sustained (power cap active in the timed loop)" if capped
                                                  else " bf16 burst"),
                "frac_of_burst": round(achieved / peaks["bf16_tflops"], 4)}
    else:
        achieved = kernels[dom].get("achieved_gbs")
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": None if achieved is None else round(achieved / peaks["hbm_gbs"], 4),
                "traffic": None if args.batch else TRAFFIC.get((args.workload, dom)),
                "peak_source": peaks["source"] + " copy"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, budget_s=args.cpu_budget)

    metric, unit = getattr(w, "metric", METRIC), getattr(w, "unit", UNIT)
    line = {
        "metric": metric, "value": round(value, 1), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "timing": {"windows": len(per_window), "steps_per_window": args.steps, "statistic": "median window",
                   "ms_per_step_min": round(min(per_window), 5), "ms_per_step_max": round(max(per_window), 5)}, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": getattr(w, "dtype", "fp4-e2m1/e4m3 cache, fp16 mma f32 accumulate"),
        "data": "synthetic",
        "config": {"workload": args.workload, "launch": "CUDA graph per step",
                   "batch_per_gpu": w.case.batch if hasattr(w.case, "batch") else 1,
                   "queries_per_step_per_gpu": w.queries_per_step, "layers": len(w.modes),
                   "l2": f"{R} cache replicas in rotation, {round(R * touched_bytes(w) / 1e6, 1)} MB touched "
                         f"per rotation > 126 MB L2",
                   "parallelism": f"replicas x{world} (batch sharded, no collective)"},
        "alg_bytes_per_step": w.step_bytes(),
        "achieved_step_gbs": round(w.step_bytes() / (ms * 1e-3) / 1e9, 1),
        "e2e": {"value": round(world * w.queries_per_step / (e2e_ms * 1e-3), 1), "unit": unit,
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "launch": "per step: inputs copied from pinned host memory on a copy stream, the "
                          "entry points on the compute stream, the output copied back on a third stream; "
                          "inputs and outputs double-buffered so step i+1's copy-in and step i-1's "
                          "copy-back overlap step i; one CUDA graph per pass over the cache replicas",
                "serial_value": round(world * w.queries_per_step / (e2e_serial_ms * 1e-3), 1),
                "serial_ms_per_step": round(e2e_serial_ms, 5),
                "eager_value": round(world * w.queries_per_step / (e2e_eager_ms * 1e-3), 1),
                "eager_ms_per_step": round(e2e_eager_ms, 5)},
        "gpu_launches": launches, "kernels": kernels, "roofline": roof, "clocks": clocks,
        "cpu_baseline": cpu, "impl": "ours",
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def e2e_pipelined(w, host_in, args, world, device, comp):
    """End-to-end ms per step through the binding with every step's host copies in the timed region,
    pipelined the way a serving loop runs: step i's inputs go up on a copy stream, its entry points run
    on the compute stream, its output comes back on a third stream; two sets of device inputs, device
    outputs and pinned host outputs let step i+1's copy-in and step i-1's copy-back overlap step i. The
    schedule of one pass over the cache replicas (all three streams, with their event dependencies) is
    captured as one CUDA graph, so the host launches one graph per pass."""
    R = args.replicas
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    bufs = [{k: torch.empty_like(v) for k, v in w.h2d_inputs().items()} for _ in range(2)]
    outs = [torch.empty_like(w.out) for _ in range(2)]
    host_out = [torch.empty(w.out.shape, dtype=w.out.dtype).pin_memory() for _ in range(2)]
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, done, copied = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    fork, up_end, down_end = ev(), ev(), ev()
    steps_per_pass = max(R, 2)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap = torch.cuda.current_stream(device)
        fork.record(cap)
        up.wait_event(fork)
        down.wait_event(fork)
        for i in range(steps_per_pass):
            b, r = i % 2, i % R
            if i >= 2:
                up.wait_event(done[b])
            with torch.cuda.stream(up):
                for k in host_in:
                    bufs[b][k].copy_(host_in[k], non_blocking=True)
            in_ready[b].record(up)
            cap.wait_event(in_ready[b])
            if i >= 2:
                cap.wait_event(copied[b])
            w.step(r, out=outs[b], **bufs[b])
            done[b].record(cap)
            down.wait_event(done[b])
            with torch.cuda.stream(down):
                host_out[b].copy_(outs[b], non_blocking=True)
            copied[b].record(down)
        up_end.record(up)
        down_end.record(down)
        cap.wait_event(up_end)
        cap.wait_event(down_end)

    passes = max(1, -(-args.steps // steps_per_pass))
    for _ in range(max(1, -(-args.warmup // steps_per_pass))):
        g.replay()
    torch.cuda.synchronize(device)
    _barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    for _ in range(passes):
        g.replay()
    t1.record(comp)
    torch.cuda.synchronize(device)
    _barrier(world)
    return _max_over_ranks(t0.elapsed_time(t1) / (passes * steps_per_pass), world, device)


# Per-launch DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of the current kernels, from one ncu
# capture of the same workload with one cache replica (still larger than L2):
#   python bench.py [--workload <name>] --steps 2 --warmup 3 --no-cpu-baseline --min-seconds 0 --replicas 1
# under ncu -k regex:<kernel> -s 2 -c 1. An entry is removed when its kernel changes; the roofline then
# reports traffic as null.
TRAFFIC = {
    # python bench.py --workload project_pack_128k_h4096 --steps 1 --warmup 3 --no-cpu-baseline --min-seconds 0
    #   --replicas 1 (ncu reports these in GB / MB with six digits)
    ("project_pack_128k_h4096", "project_pack"): 1_102_514_000 + 19_863_808,
    ("decode_64k_b32_h64", "sparse_attn"): 25_296_640 + 0,
    ("decode_64k_b32_h64_nvfp4q", "sparse_attn"): 24_971_520 + 0,
    ("decode_64k_b32_h64", "index_score"): 75_609_088 + 892_160,
}


# ------------------------------------------------------------------------------------------------
# The oracle arm and the CPU baseline
# ------------------------------------------------------------------------------------------------

def _blas_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        return max([i.get("num_threads", 1) for i in info] or [1])
    except Exception:
        return 1


class OracleDecodeSample:
    """One sequence of a decode workload, prepared for the CPU oracle (same shapes and value recipe)."""

    def __init__(self, case, seed_offset=0):
        from compressed_sparse_attention_merge_b300 import synth
        from oracle import fp4 as o_fp4
        from oracle import indexer as o_idx
        g = synth.generator(case.seed + 1000 + seed_offset, "cpu")
        T, E = case.max_tokens, case.max_entries
        self.case, self.E = case, E
        tokens = synth.latent_tokens(g, (T, 512), "cpu", case.outlier_frac).float().numpy()
        keys = synth.int_values(g, (1, E, case.idx_dim), "cpu")
        nq = case.distinct_index_queries
        q_idx = synth.int_values(g, (nq, 1, case.n_query, case.idx_heads, case.idx_dim), "cpu")
        synth.plant_needles(g, keys, q_idx[0], case.needle_frac)
        self.keys_f = keys[0].numpy()
        self.q_idx = q_idx[:, 0].numpy()                 # [distinct queries, Q, H_i, D_i]
        Q = case.n_query
        self.q = synth.normal_bf16(g, (case.layers, Q, case.heads, 512), "cpu").float().numpy()
        swa_rows = case.window + (Q - 1 if case.causal_drafts else 0)
        self.swa = synth.normal_bf16(g, (case.layers, swa_rows, 512), "cpu").float().numpy()
        self.q_pos = np.arange(T - Q, T) if case.causal_drafts else None
        self.swa_first_pos = T - Q - case.window + 1
        nb = -(-E // 8)
        lo = 2 * ((T - Q) // 2)
        self.first = E - (T - lo) // 2
        self.new_tokens = tokens[lo:T]
        self.new_key = self.keys_f[self.first:E]
        self.cache = o_fp4.pack(tokens, 2, "amax", n_blocks=nb)
        self.kcache = o_fp4.pack(self.keys_f, 1, "pow2", n_blocks=nb)
        self.coarse = None
        if case.hier_keep:
            self.coarse = o_idx.coarse_keys(o_fp4.dequantize(self.kcache, case.idx_dim, E), E)
        self.modes = chain_modes(case.layers) if case.layers > 1 else ["full"]

    def step(self):
        """The oracle's decode step for this one sequence; returns the attention outputs."""
        from oracle import attention as o_attn
        from oracle import fp4 as o_fp4
        from oracle import indexer as o_idx
        c, E = self.case, self.E
        cache = o_fp4.pack(self.new_tokens, 2, "amax", first_entry=self.first, base=self.cache)
        kcache = o_fp4.pack(self.new_key, 1, "pow2", first_entry=self.first, base=self.kcache)
        keys = o_fp4.dequantize(kcache, c.idx_dim, E)
        entries = o_fp4.dequantize(cache, 512, E)
        outs, idx = [], None
        n_idx = 0
        for layer, mode in enumerate(self.modes):
            if mode != "reuse":
                q_idx = self.q_idx[n_idx % self.q_idx.shape[0]]
                if c.hier_keep:
                    idx, _ = o_idx.hierarchical_topk(q_idx, keys, E, c.top_k, c.hier_keep, coarse=self.coarse)
                else:
                    idx, _ = o_idx.flat_topk(q_idx, keys, E, c.top_k, q_pos=self.q_pos)
                n_idx += 1
            for j in range(c.n_query):
                qj = self.q[layer, j].astype(np.float64)
                if self.q_pos is not None:
                    out, _ = o_attn.prefill_attention(qj, entries, E, idx[j], self.swa[layer], self.swa_first_pos,
                                                      int(self.q_pos[j]), c.window, SCALE)
                elif c.nvfp4q:
                    out, _ = o_attn.decode_attention_nvfp4q(self.q[layer, j], entries, E, idx[j], self.swa[layer],
                                                            SCALE)
                else:
                    out, _ = o_attn.decode_attention(qj, entries, E, idx[j], self.swa[layer], SCALE)
                outs.append(out)
        return outs


class OraclePrefillSample:
    """A few positions of the prefill workload for the CPU oracle."""

    def __init__(self, case, positions=4):
        from compressed_sparse_attention_merge_b300 import synth
        from oracle import fp4 as o_fp4
        g = synth.generator(case.seed + 1000, "cpu")
        self.case = case
        E, P, C = case.max_entries, case.first_pos, case.chunk
        self.E, self.P = E, P
        prior = synth.latent_tokens(g, (P, 512), "cpu", case.outlier_frac).float().numpy()
        self.chunk = synth.latent_tokens(g, (C, 512), "cpu", case.outlier_frac).float().numpy()
        self.keys = synth.int_values(g, (E, case.idx_dim), "cpu").numpy()
        self.cache = o_fp4.pack(prior, 2, "amax", n_blocks=-(-E // 8))
        self.kcache = o_fp4.pack(self.keys[:P // 2], 1, "pow2", n_blocks=-(-E // 8))
        self.positions = [P + (C - 1) * i // max(1, positions - 1) for i in range(positions)]
        self.q = synth.normal_bf16(g, (len(self.positions), case.heads, 512), "cpu").float().numpy()
        self.q_idx = synth.int_values(g, (len(self.positions), case.idx_heads, case.idx_dim), "cpu").numpy()
        self.swa = synth.normal_bf16(g, (C + case.window - 1, 512), "cpu").float().numpy()

    def step(self):
        from oracle import attention as o_attn
        from oracle import fp4 as o_fp4
        from oracle import indexer as o_idx
        c, E, P = self.case, self.E, self.P
        cache = o_fp4.pack(self.chunk, 2, "amax", first_entry=P // 2, base=self.cache)
        kcache = o_fp4.pack(self.keys[P // 2:], 1, "pow2", first_entry=P // 2, base=self.kcache)
        keys = o_fp4.dequantize(kcache, c.idx_dim, E)
        entries = o_fp4.dequantize(cache, 512, E)
        pos = np.array(self.positions)
        idx, _ = o_idx.flat_topk(self.q_idx, keys, E, c.top_k, q_pos=pos)
        outs = []
        attend = o_attn.prefill_attention_nvfp4q if c.nvfp4q else o_attn.prefill_attention
        for j, p in enumerate(self.positions):
            qj = self.q[j] if c.nvfp4q else self.q[j].astype(np.float64)
            out, _ = attend(qj, entries, E, idx[j], self.swa, P - c.window + 1, int(p), c.window, SCALE)
            outs.append(out)
        return outs


class OracleProjectSample:
    """A slice of the projection workload's tokens for the CPU oracle (the same value recipe, its own draw)."""

    def __init__(self, case, tokens=256, seed_offset=0):
        from compressed_sparse_attention_merge_b300 import synth
        g = synth.generator(case.seed + 1000 + seed_offset, "cpu")
        self.h = synth.normal_bf16(g, (tokens, case.hidden), "cpu").float().numpy()
        w = torch.randn(512, case.hidden, generator=g) / case.hidden ** 0.5
        self.w = w.to(torch.bfloat16).float().numpy()
        self.tokens = tokens

    def step(self):
        from oracle import projection as o_proj
        return o_proj.project_pack(self.h, self.w, "amax")


def _oracle_sample(workload, seed_offset=0):
    """(sample, units per step, what the sample is) for the CPU oracle."""
    case = _cases()[workload]
    if workload.startswith("project"):
        s = OracleProjectSample(case, seed_offset=seed_offset)
        return s, s.tokens, f"{s.tokens} tokens of one sequence (projection of the hidden rows, merge and pack)"
    if workload.startswith("prefill"):
        s = OraclePrefillSample(case)
        return s, len(s.positions), f"{len(s.positions)} positions of the chunk (pack of the whole chunk, " \
                                    f"dequantisation of the cache, per-position index + Top-K and attention)"
    s = OracleDecodeSample(case, seed_offset=seed_offset)
    return s, case.n_query, "one sequence of the batch (re-pack of the newest entry, dequantisation of the " \
                            "cache, index + Top-K, attention" + (" through all layers" if case.layers > 1 else "") \
                            + ")"


def _metric_unit(workload):
    return (ProjectWorkload.metric, ProjectWorkload.unit) if workload.startswith("project") else (METRIC, UNIT)


def _host_cpu():
    """nproc and the CPU model of this host."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return os.cpu_count() or 1, model


def _oracle_worker(args):
    """One process of the all-cores baseline: its own sequence sample (seed offset by its index), numpy
    limited to one thread, steps until the budget is spent. Returns (steps, seconds, queries per step)."""
    workload, index, budget_s = args
    try:
        import threadpoolctl
        threadpoolctl.threadpool_limits(1)
    except Exception:
        pass
    s, queries, _ = _oracle_sample(workload, seed_offset=index)
    s.step()
    n, t0 = 0, time.perf_counter()
    while True:
        s.step()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 50:
            return n, el, queries


def cpu_baseline(workload, budget_s=20.0, parallel=True):
    """The oracle, as it stands, timed on this host's cores on a bounded sample of the workload: one
    process with numpy's own threads, and (parallel) one single-threaded process per core, each on its own
    sequence of the workload, for the all-cores figure."""
    s, queries, what = _oracle_sample(workload)
    s.step()                               # warm caches of numpy's allocator
    n, t0 = 0, time.perf_counter()
    while True:
        s.step()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 50:
            break
    one = n * queries / el
    nproc, model = _host_cpu()
    out = {"value": round(one, 4), "unit": _metric_unit(workload)[1], "cores": _blas_threads(), "kind": "oracle",
           "sample": what + f"; {n} repetitions in {el:.1f} s", "host": {"nproc": nproc, "cpu": model}}
    if parallel and nproc > 1:
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        with ctx.Pool(nproc) as pool:
            res = pool.map(_oracle_worker, [(workload, i, budget_s) for i in range(nproc)])
        total = sum(n_i * q_i / el_i for n_i, el_i, q_i in res)
        out["all_cores"] = {"value": round(total, 4), "cores": nproc,
                            "sample": f"{nproc} single-threaded processes, each on its own sequence of the workload "
                                      f"for about {budget_s:.0f} s (sum of their rates)"}
        out["value"], out["cores"] = out["all_cores"]["value"], nproc
        out["single_process"] = {"value": round(one, 4), "cores": _blas_threads()}
    return out


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    s, queries, what = _oracle_sample(args.workload)
    for _ in range(args.warmup):
        s.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s.step()
    el = time.perf_counter() - t0
    value = args.steps * queries / el
    cores = _blas_threads()
    metric, unit = _metric_unit(args.workload)
    line = {"metric": metric, "value": round(value, 4), "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * el / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "launch": "the oracle (numpy, fp64) on the host cores",
                       "sample": what},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": what},
            "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(_cases().keys()), default=DEFAULT_WORKLOAD)
    ap.add_argument("--replicas", type=int, default=4)
    ap.add_argument("--batch", type=int, default=None,
                    help="decode workloads: number of sequences (each as long as the workload's first)")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--min-seconds", type=float, default=2.5,
                    help="the K-step timed window is repeated until this many seconds have passed")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
