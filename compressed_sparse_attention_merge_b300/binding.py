"""Python binding of the C ABI in include/csa.h (ctypes). Argument marshalling only: every step of the
path runs in the CUDA kernels of ``libcsa.so``. PyTorch supplies device memory and streams.

The library must have been built (``python -m compressed_sparse_attention_merge_b300.build``); loading
fails loudly otherwise, and there is no CPU fallback.
"""

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcsa.so")
_lib = None

LATENT_DIM = 512
BLOCK_ENTRIES = 8
SUPER_BLOCK = 64
WS_HEADER_BYTES = 256

OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_UNSUPPORTED_DEVICE = 0, 1, 2, 3
ERR_WORKSPACE_TOO_SMALL, ERR_CUDA, ERR_DEVICE_CHECK, ERR_TIMEOUT = 4, 5, 6, 7
DTYPE_BF16, DTYPE_F32 = 0, 1
SCALE_AMAX, SCALE_POW2 = 0, 1
IDX_RELU, IDX_HIER = 1, 2


class CsaError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        detail = ""
        if status == ERR_CUDA or (status == ERR_WORKSPACE_TOO_SMALL and where == "csa_index_topk_static"):
            detail = " [" + lib().csa_last_error().decode() + "]"
        super().__init__(f"{where}: {lib().csa_status_string(status).decode()} (status {status}){detail}")


class PackArgs(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("x_dtype", ctypes.c_int32), ("dim", ctypes.c_int32),
                ("x_stride_b", ctypes.c_int64), ("x_stride_t", ctypes.c_int64), ("n_tokens", ctypes.c_int64),
                ("merge", ctypes.c_int32), ("scale_rule", ctypes.c_int32), ("first_entry", ctypes.c_void_p),
                ("max_entries", ctypes.c_int64), ("cache", ctypes.c_void_p), ("cache_stride_b", ctypes.c_int64),
                ("coarse_sum", ctypes.c_void_p), ("coarse_stride_b", ctypes.c_int64)]


class ProjectArgs(ctypes.Structure):
    _fields_ = [("h", ctypes.c_void_p), ("h_stride_b", ctypes.c_int64), ("h_stride_t", ctypes.c_int64),
                ("hidden", ctypes.c_int64), ("w", ctypes.c_void_p), ("n_tokens", ctypes.c_int64),
                ("scale_rule", ctypes.c_int32), ("reserved", ctypes.c_int32), ("first_entry", ctypes.c_void_p),
                ("max_entries", ctypes.c_int64), ("cache", ctypes.c_void_p), ("cache_stride_b", ctypes.c_int64)]


class IndexArgs(ctypes.Structure):
    _fields_ = [("n_query", ctypes.c_int64), ("heads", ctypes.c_int32), ("dim", ctypes.c_int32),
                ("q_idx", ctypes.c_void_p), ("head_w", ctypes.c_void_p), ("flags", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("keys", ctypes.c_void_p), ("keys_stride_b", ctypes.c_int64),
                ("n_entries", ctypes.c_void_p), ("max_entries", ctypes.c_int64), ("q_pos", ctypes.c_void_p),
                ("coarse_sum", ctypes.c_void_p), ("coarse_stride_b", ctypes.c_int64),
                ("keep_blocks", ctypes.c_int32), ("reserved0", ctypes.c_int32), ("out_idx", ctypes.c_void_p),
                ("out_block_scores", ctypes.c_void_p)]


class AttnArgs(ctypes.Structure):
    _fields_ = [("n_query", ctypes.c_int64), ("heads", ctypes.c_int32), ("scale", ctypes.c_float),
                ("q", ctypes.c_void_p), ("cache", ctypes.c_void_p), ("cache_stride_b", ctypes.c_int64),
                ("n_entries", ctypes.c_void_p), ("max_entries", ctypes.c_int64), ("idx", ctypes.c_void_p),
                ("top_k", ctypes.c_int32), ("window", ctypes.c_int32), ("q_pos", ctypes.c_void_p),
                ("swa", ctypes.c_void_p), ("swa_stride_b", ctypes.c_int64), ("swa_rows", ctypes.c_int64),
                ("swa_len", ctypes.c_void_p), ("swa_first_pos", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("out_lse", ctypes.c_void_p)]


class LayerArgs(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("flags", ctypes.c_int32), ("q_idx", ctypes.c_void_p),
                ("idx", ctypes.c_void_p), ("q", ctypes.c_void_p), ("swa", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("out_lse", ctypes.c_void_p)]


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


def lib():
    """The loaded libcsa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"{_LIB_PATH} is missing: build it with "
                              "`python -m compressed_sparse_attention_merge_b300.build`")
        L = ctypes.CDLL(_LIB_PATH)
        P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        L.csa_abi_version.restype = I32
        L.csa_status_string.restype = ctypes.c_char_p
        L.csa_status_string.argtypes = [I32]
        L.csa_last_error.restype = ctypes.c_char_p
        L.csa_last_error.argtypes = []
        L.csa_entry_bytes.restype = SZ
        L.csa_entry_bytes.argtypes = [I32]
        L.csa_block_bytes.restype = SZ
        L.csa_block_bytes.argtypes = [I32]
        L.csa_workspace_reset.restype = I32
        L.csa_workspace_reset.argtypes = [P, SZ, P]
        L.csa_get_device_status.restype = I32
        L.csa_get_device_status.argtypes = [P, P]
        L.csa_pack_fp4.restype = I32
        L.csa_pack_fp4.argtypes = [I64, ctypes.POINTER(PackArgs), P, SZ, P]
        L.csa_pack_fp4_multi.restype = I32
        L.csa_project_pack.restype = I32
        L.csa_project_pack.argtypes = [I64, ctypes.POINTER(ProjectArgs), P, SZ, P]
        L.csa_pack_fp4_multi.argtypes = [I32, ctypes.POINTER(I64), ctypes.POINTER(PackArgs), P, SZ, P]
        L.csa_index_topk_workspace_size.restype = SZ
        L.csa_index_topk_workspace_size.argtypes = [I64, ctypes.POINTER(IndexArgs)]
        L.csa_index_topk.restype = I32
        L.csa_index_topk.argtypes = [I64, ctypes.POINTER(IndexArgs), P, SZ, P]
        L.csa_index_topk_static.restype = I32
        L.csa_index_topk_static.argtypes = [I64, ctypes.POINTER(IndexArgs), P, P]
        L.csa_sparse_attn_workspace_size.restype = SZ
        L.csa_sparse_attn_workspace_size.argtypes = [I64, ctypes.POINTER(AttnArgs)]
        for name in ("csa_sparse_attn_decode", "csa_sparse_attn_prefill", "csa_sparse_attn_decode_nvfp4q",
                     "csa_sparse_attn_prefill_nvfp4q"):
            f = getattr(L, name)
            f.restype = I32
            f.argtypes = [I64, ctypes.POINTER(AttnArgs), P, SZ, P]
        L.csa_decode_layers.restype = I32
        L.csa_decode_layers.argtypes = [I64, I32, ctypes.POINTER(LayerArgs), ctypes.POINTER(IndexArgs),
                                        ctypes.POINTER(AttnArgs), P, SZ, P, SZ, P]
        L.csa_debug_set_fault.restype = I32
        L.csa_debug_set_fault.argtypes = [I32, ctypes.c_uint32]
        L.csa_profile_begin.restype = I32
        L.csa_profile_begin.argtypes = [I32]
        L.csa_profile_end.restype = I32
        L.csa_profile_end.argtypes = [ctypes.POINTER(KernelTime), I32, ctypes.POINTER(ctypes.c_int),
                                      ctypes.POINTER(ctypes.c_int64)]
        _lib = L
    return _lib


def _check(status, where):
    if status != OK:
        raise CsaError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype=None, cuda=True):
    if t is None:
        raise ValueError(f"{name} is required")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


# ------------------------------------------------------------------------------------------------
# Sizes and workspaces
# ------------------------------------------------------------------------------------------------

def block_bytes(dim):
    return int(lib().csa_block_bytes(dim))


def cache_blocks(max_entries):
    return -(-max_entries // BLOCK_ENTRIES)


def empty_cache(batch, max_entries, dim, device):
    """A zeroed packed cache [batch, ceil(max_entries / 8), block_bytes(dim)] uint8."""
    return torch.zeros(batch, cache_blocks(max_entries), block_bytes(dim), dtype=torch.uint8, device=device)


def empty_coarse(batch, max_entries, dim, device):
    n_super = -(-max_entries // (BLOCK_ENTRIES * SUPER_BLOCK))
    return torch.zeros(batch, n_super, dim, dtype=torch.float32, device=device)


def workspace(nbytes, device):
    """A zeroed workspace of at least nbytes (torch's allocator returns 512-byte aligned storage)."""
    ws = torch.zeros(max(int(nbytes), WS_HEADER_BYTES), dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def workspace_reset(ws, stream=None):
    _check(lib().csa_workspace_reset(_ptr(ws), ws.numel(), _stream(stream)), "csa_workspace_reset")


def device_status(ws, stream=None):
    """Synchronizes the stream and returns (and clears) the workspace status code."""
    return int(lib().csa_get_device_status(_ptr(ws), _stream(stream)))


# ------------------------------------------------------------------------------------------------
# Entry points
# ------------------------------------------------------------------------------------------------

def pack_args(x, cache, *, merge, scale_rule, max_entries, first_entry=None, coarse_sum=None):
    _need(x, "x")
    _need(cache, "cache", torch.uint8)
    if x.dim() != 3:
        raise ValueError("x must be [batch, n_tokens, dim]")
    if x.stride(2) != 1:
        raise ValueError("x rows must be contiguous")
    a = PackArgs()
    a.x = x.data_ptr()
    a.x_dtype = {torch.bfloat16: DTYPE_BF16, torch.float32: DTYPE_F32}[x.dtype]
    a.dim = x.shape[2]
    a.x_stride_b, a.x_stride_t = x.stride(0), x.stride(1)
    a.n_tokens = x.shape[1]
    a.merge, a.scale_rule = merge, scale_rule
    a.first_entry = None if first_entry is None else _need(first_entry, "first_entry", torch.int32).data_ptr()
    a.max_entries = max_entries
    a.cache = cache.data_ptr()
    a.cache_stride_b = cache[0].numel() if cache.dim() > 1 else cache.numel()
    if coarse_sum is not None:
        _need(coarse_sum, "coarse_sum", torch.float32)
        a.coarse_sum = coarse_sum.data_ptr()
        a.coarse_stride_b = coarse_sum[0].numel()
    return a


def pack_fp4(x, cache, *, merge, scale_rule, max_entries, ws, first_entry=None, coarse_sum=None, stream=None):
    """csa_pack_fp4: pair-merge (merge=2) or take (merge=1) rows of x [B, T, dim] and FP4-pack them into
    cache [B, blocks, block_bytes] at entries first_entry[b]...; optional coarse-key maintenance."""
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    a = pack_args(x, cache, merge=merge, scale_rule=scale_rule, max_entries=max_entries,
                  first_entry=first_entry, coarse_sum=coarse_sum)
    _check(lib().csa_pack_fp4(x.shape[0], ctypes.byref(a), _ptr(ws), ws.numel(), _stream(stream)), "csa_pack_fp4")


def project_pack(h, w, cache, *, scale_rule, max_entries, ws, first_entry=None, stream=None):
    """csa_project_pack: project hidden rows h [B, T, hidden] (bf16) by w [512, hidden] (bf16) and pair-merge
    + FP4-pack the latents into cache [B, blocks, 2304] at entries first_entry[b]..."""
    _need(h, "h", torch.bfloat16)
    _need(w, "w", torch.bfloat16)
    _need(cache, "cache", torch.uint8)
    if h.dim() != 3 or h.stride(2) != 1:
        raise ValueError("h must be [batch, n_tokens, hidden] with contiguous rows")
    if w.dim() != 2 or w.shape[0] != 512 or w.shape[1] != h.shape[2] or not w.is_contiguous():
        raise ValueError("w must be a contiguous [512, hidden] tensor")
    a = ProjectArgs()
    a.h = h.data_ptr()
    a.h_stride_b, a.h_stride_t = h.stride(0), h.stride(1)
    a.hidden = h.shape[2]
    a.w = w.data_ptr()
    a.n_tokens = h.shape[1]
    a.scale_rule = scale_rule
    a.first_entry = None if first_entry is None else _need(first_entry, "first_entry", torch.int32).data_ptr()
    a.max_entries = max_entries
    a.cache = cache.data_ptr()
    a.cache_stride_b = cache[0].numel() if cache.dim() > 1 else cache.numel()
    _check(lib().csa_project_pack(h.shape[0], ctypes.byref(a), _ptr(ws), ws.numel(), _stream(stream)),
           "csa_project_pack")


PACK_MAX_JOBS = 4


def pack_fp4_multi(jobs, *, ws, stream=None):
    """csa_pack_fp4_multi: several pack_fp4 calls in one launch. jobs is a list of (x, cache, kwargs),
    kwargs being pack_fp4's keyword arguments other than ws and stream. No two jobs may write the same
    cache entries."""
    if not 1 <= len(jobs) <= PACK_MAX_JOBS:
        raise ValueError(f"1..{PACK_MAX_JOBS} jobs")
    arr = (PackArgs * len(jobs))()
    batches = (ctypes.c_int64 * len(jobs))()
    for j, (x, cache, kw) in enumerate(jobs):
        if not x.is_cuda:
            raise ValueError("x must be a CUDA tensor")
        arr[j] = pack_args(x, cache, **kw)
        batches[j] = x.shape[0]
    _check(lib().csa_pack_fp4_multi(len(jobs), batches, arr, _ptr(ws), ws.numel(), _stream(stream)),
           "csa_pack_fp4_multi")


def index_args(q_idx, keys, n_entries, out_idx, *, max_entries, top_k, head_w=None, relu=True, q_pos=None,
               coarse_sum=None, keep_blocks=0, out_block_scores=None):
    _need(q_idx, "q_idx", torch.float32)
    _need(keys, "keys", torch.uint8)
    _need(n_entries, "n_entries", torch.int32)
    _need(out_idx, "out_idx", torch.int32)
    if q_idx.dim() != 4:
        raise ValueError("q_idx must be [batch, n_query, heads, dim]")
    a = IndexArgs()
    a.n_query, a.heads, a.dim = q_idx.shape[1], q_idx.shape[2], q_idx.shape[3]
    a.q_idx = q_idx.data_ptr()
    a.head_w = None if head_w is None else _need(head_w, "head_w", torch.float32).data_ptr()
    a.flags = (IDX_RELU if relu else 0) | (IDX_HIER if coarse_sum is not None else 0)
    a.top_k = top_k
    a.keys = keys.data_ptr()
    a.keys_stride_b = keys[0].numel()
    a.n_entries = n_entries.data_ptr()
    a.max_entries = max_entries
    a.q_pos = None if q_pos is None else _need(q_pos, "q_pos", torch.int32).data_ptr()
    if coarse_sum is not None:
        _need(coarse_sum, "coarse_sum", torch.float32)
        a.coarse_sum = coarse_sum.data_ptr()
        a.coarse_stride_b = coarse_sum[0].numel()
        a.keep_blocks = keep_blocks
    a.out_idx = out_idx.data_ptr()
    a.out_block_scores = None if out_block_scores is None else _need(out_block_scores, "out_block_scores",
                                                                     torch.float32).data_ptr()
    return a


def index_topk_workspace_size(batch, args):
    return int(lib().csa_index_topk_workspace_size(batch, ctypes.byref(args)))


def index_topk(q_idx, keys, n_entries, out_idx, *, max_entries, top_k, ws, head_w=None, relu=True, q_pos=None,
               coarse_sum=None, keep_blocks=0, out_block_scores=None, stream=None):
    """csa_index_topk. Flat selection unless coarse_sum is given (hierarchical, keep_blocks blocks kept)."""
    a = index_args(q_idx, keys, n_entries, out_idx, max_entries=max_entries, top_k=top_k, head_w=head_w,
                   relu=relu, q_pos=q_pos, coarse_sum=coarse_sum, keep_blocks=keep_blocks,
                   out_block_scores=out_block_scores)
    _check(lib().csa_index_topk(q_idx.shape[0], ctypes.byref(a), _ptr(ws), ws.numel(), _stream(stream)),
           "csa_index_topk")


STATIC_INDEX_SCRATCH_BYTES = 4 << 20


def index_topk_static(q_idx, keys, n_entries, out_idx, *, max_entries, top_k, head_w=None, relu=True, q_pos=None,
                      coarse_sum=None, keep_blocks=0, status_out=None, stream=None):
    """csa_index_topk_static: the same selection as index_topk, for callers that cannot allocate device
    memory; the scratch is the library's own fixed 4 MiB device array (calls on one device must not
    overlap on the GPU). status_out: optional int32 CUDA tensor of one element that receives the device
    status word."""
    a = index_args(q_idx, keys, n_entries, out_idx, max_entries=max_entries, top_k=top_k, head_w=head_w,
                   relu=relu, q_pos=q_pos, coarse_sum=coarse_sum, keep_blocks=keep_blocks)
    st = None if status_out is None else _need(status_out, "status_out", torch.int32)
    _check(lib().csa_index_topk_static(q_idx.shape[0], ctypes.byref(a), _ptr(st), _stream(stream)),
           "csa_index_topk_static")


def attn_args(q, cache, n_entries, idx, out, *, max_entries, window, scale, swa=None, swa_len=None,
              swa_first_pos=None, q_pos=None, out_lse=None):
    _need(q, "q", torch.bfloat16)
    _need(cache, "cache", torch.uint8)
    _need(n_entries, "n_entries", torch.int32)
    _need(idx, "idx", torch.int32)
    _need(out, "out", torch.float32)
    if q.dim() != 4 or q.shape[3] != LATENT_DIM:
        raise ValueError("q must be [batch, n_query, heads, 512]")
    a = AttnArgs()
    a.n_query, a.heads, a.scale = q.shape[1], q.shape[2], float(scale)
    a.q = q.data_ptr()
    a.cache = cache.data_ptr()
    a.cache_stride_b = cache[0].numel()
    a.n_entries = n_entries.data_ptr()
    a.max_entries = max_entries
    a.idx = idx.data_ptr()
    a.top_k = idx.shape[-1]
    a.window = window
    a.q_pos = None if q_pos is None else _need(q_pos, "q_pos", torch.int32).data_ptr()
    if swa is not None:
        _need(swa, "swa", torch.bfloat16)
        a.swa = swa.data_ptr()
        a.swa_stride_b = swa[0].numel()
        a.swa_rows = swa.shape[1]
    a.swa_len = None if swa_len is None else _need(swa_len, "swa_len", torch.int32).data_ptr()
    a.swa_first_pos = None if swa_first_pos is None else _need(swa_first_pos, "swa_first_pos",
                                                               torch.int32).data_ptr()
    a.out = out.data_ptr()
    a.out_lse = None if out_lse is None else _need(out_lse, "out_lse", torch.float32).data_ptr()
    return a


def sparse_attn_workspace_size(batch, args):
    return int(lib().csa_sparse_attn_workspace_size(batch, ctypes.byref(args)))


def sparse_attn_decode(q, cache, n_entries, idx, out, *, max_entries, window, scale, ws, swa=None, swa_len=None,
                       out_lse=None, stream=None):
    """csa_sparse_attn_decode: q [B, Q, H, 512] bf16 attends to the blocks idx [B, Q, K] of the cache plus
    rows 0..swa_len[b]-1 of swa [B, rows, 512]."""
    a = attn_args(q, cache, n_entries, idx, out, max_entries=max_entries, window=window, scale=scale, swa=swa,
                  swa_len=swa_len, out_lse=out_lse)
    _check(lib().csa_sparse_attn_decode(q.shape[0], ctypes.byref(a), _ptr(ws), ws.numel(), _stream(stream)),
           "csa_sparse_attn_decode")


def sparse_attn_prefill(q, cache, n_entries, idx, out, *, q_pos, max_entries, window, scale, ws, swa=None,
                        swa_first_pos=None, out_lse=None, stream=None):
    """csa_sparse_attn_prefill: causal per-position attention (entry e visible iff 2e+1 <= q_pos) plus the
    window of tokens max(p - window + 1, swa_first_pos[b]) .. p from swa [B, rows, 512]."""
    a = attn_args(q, cache, n_entries, idx, out, max_entries=max_entries, window=window, scale=scale, swa=swa,
                  swa_first_pos=swa_first_pos, q_pos=q_pos, out_lse=out_lse)
    _check(lib().csa_sparse_attn_prefill(q.shape[0], ctypes.byref(a), _ptr(ws), ws.numel(), _stream(stream)),
           "csa_sparse_attn_prefill")


def sparse_attn_decode_nvfp4q(q, cache, n_entries, idx, out, *, max_entries, window, scale, ws, swa=None,
                              swa_len=None, out_lse=None, stream=None):
    """csa_sparse_attn_decode_nvfp4q: sparse_attn_decode with the logits on the block-scaled FP4 tensor cores
    (query heads and window keys rounded to FP4 inside the logits; values exact)."""
    a = attn_args(q, cache, n_entries, idx, out, max_entries=max_entries, window=window, scale=scale, swa=swa,
                  swa_len=swa_len, out_lse=out_lse)
    _check(lib().csa_sparse_attn_decode_nvfp4q(q.shape[0], ctypes.byref(a), _ptr(ws), ws.numel(), _stream(stream)),
           "csa_sparse_attn_decode_nvfp4q")


def sparse_attn_prefill_nvfp4q(q, cache, n_entries, idx, out, *, q_pos, max_entries, window, scale, ws, swa=None,
                               swa_first_pos=None, out_lse=None, stream=None):
    """csa_sparse_attn_prefill_nvfp4q: sparse_attn_prefill with the NVFP4-query logits."""
    a = attn_args(q, cache, n_entries, idx, out, max_entries=max_entries, window=window, scale=scale, swa=swa,
                  swa_first_pos=swa_first_pos, q_pos=q_pos, out_lse=out_lse)
    _check(lib().csa_sparse_attn_prefill_nvfp4q(q.shape[0], ctypes.byref(a), _ptr(ws), ws.numel(),
                                                _stream(stream)), "csa_sparse_attn_prefill_nvfp4q")


LAYER_FULL, LAYER_REINDEX, LAYER_REUSE = 0, 1, 2
LAYER_ATTN_NVFP4Q = 1
_LAYER_MODES = {"full": LAYER_FULL, "reindex": LAYER_REINDEX, "reuse": LAYER_REUSE}


def decode_layers(layers, *, index_tmpl, attn_tmpl, ws_index, ws_attn, stream=None):
    """csa_decode_layers: a step of several layers over one cache. layers: list of dicts with keys mode
    ("full" | "reindex" | "reuse"), q_idx and idx (Full / Reindex), q, swa (or None), out, out_lse (or
    None), and optionally nvfp4q (True: the layer's attention is the NVFP4-query variant). index_tmpl / attn_tmpl: IndexArgs / AttnArgs (from index_args / attn_args) holding the shared
    fields; a set q_pos in attn_tmpl makes the attention causal. The batch is taken from the first layer's q."""
    n = len(layers)
    arr = (LayerArgs * n)()
    for i, layer in enumerate(layers):
        arr[i].mode = _LAYER_MODES[layer["mode"]]
        arr[i].flags = LAYER_ATTN_NVFP4Q if layer.get("nvfp4q") else 0
        if layer["mode"] != "reuse":
            arr[i].q_idx = _need(layer["q_idx"], "q_idx", torch.float32).data_ptr()
            arr[i].idx = _need(layer["idx"], "idx", torch.int32).data_ptr()
        arr[i].q = _need(layer["q"], "q", torch.bfloat16).data_ptr()
        arr[i].swa = None if layer.get("swa") is None else _need(layer["swa"], "swa", torch.bfloat16).data_ptr()
        arr[i].out = _need(layer["out"], "out", torch.float32).data_ptr()
        arr[i].out_lse = None if layer.get("out_lse") is None else _need(layer["out_lse"], "out_lse",
                                                                         torch.float32).data_ptr()
    batch = layers[0]["q"].shape[0]
    _check(lib().csa_decode_layers(batch, n, arr, ctypes.byref(index_tmpl), ctypes.byref(attn_tmpl), _ptr(ws_index),
                                   ws_index.numel(), _ptr(ws_attn), ws_attn.numel(), _stream(stream)),
           "csa_decode_layers")


# ------------------------------------------------------------------------------------------------
# Kernel timing
# ------------------------------------------------------------------------------------------------

FAULT_NONE, FAULT_WITHHOLD_ARRIVAL = 0, 1


def debug_set_fault(fault, spin_limit=0):
    """csa_debug_set_fault (test-only): make later attention launches withhold one internal arrival so
    that a bounded wait gives up after spin_limit polls; FAULT_NONE restores normal launches."""
    _check(lib().csa_debug_set_fault(int(fault), int(spin_limit)), "csa_debug_set_fault")


def profile_begin(max_launches=4096):
    _check(lib().csa_profile_begin(max_launches), "csa_profile_begin")


def profile_end():
    """Returns ({kernel name: (launches, total_ms)}, dropped launches)."""
    out = (KernelTime * 64)()
    n = ctypes.c_int(0)
    dropped = ctypes.c_int64(0)
    _check(lib().csa_profile_end(out, 64, ctypes.byref(n), ctypes.byref(dropped)), "csa_profile_end")
    return {out[i].name.decode(): (int(out[i].launches), float(out[i].total_ms)) for i in range(n.value)}, \
        int(dropped.value)
