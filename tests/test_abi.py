"""The C-ABI library loads and exports every symbol include/csa.h declares; host-side validation that
needs no GPU rejects bad arguments before touching the device. No compute call runs here."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")


@pytest.fixture(scope="module")
def lib():
    from compressed_sparse_attention_merge_b300 import build, binding
    build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(csa_[a-z0-9_]+)\s*\(", text))
    return sorted(n for n in names if not n.endswith("_t"))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("csa_pack_fp4", "csa_pack_fp4_multi", "csa_index_topk", "csa_sparse_attn_decode",
              "csa_sparse_attn_prefill", "csa_sparse_attn_decode_nvfp4q", "csa_sparse_attn_prefill_nvfp4q",
              "csa_project_pack", "csa_decode_layers"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    path = lib._name
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (csa_[a-z0-9_]+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)


def test_project_pack_rejects_bad_arguments_before_any_device_call(lib):
    # pointers that are never dereferenced on the host
    from compressed_sparse_attention_merge_b300 import binding as b
    good = 0x10000
    pa = b.ProjectArgs()
    pa.h, pa.w, pa.cache = good, good, good
    pa.h_stride_b, pa.h_stride_t, pa.hidden, pa.n_tokens = 4 * 640, 640, 640, 4
    pa.scale_rule, pa.max_entries, pa.cache_stride_b = b.SCALE_AMAX, 8, 2304
    call = lambda batch: lib.csa_project_pack(batch, ctypes.byref(pa), None, 0, None)
    for field, bad, want in [("hidden", 600, b.ERR_INVALID_ARG),          # not a multiple of 64
                             ("hidden", 16448, b.ERR_INVALID_ARG),        # above 16,384
                             ("scale_rule", 7, b.ERR_INVALID_ARG),
                             ("reserved", 1, b.ERR_INVALID_ARG),
                             ("n_tokens", -1, b.ERR_INVALID_ARG),
                             ("h", good + 8, b.ERR_ALIGNMENT),
                             ("w", good + 4, b.ERR_ALIGNMENT),
                             ("h_stride_t", 644, b.ERR_ALIGNMENT),        # rows not 16-byte aligned
                             ("h_stride_t", 576, b.ERR_INVALID_ARG),      # shorter than a row
                             ("cache_stride_b", 2312, b.ERR_ALIGNMENT)]:
        old = getattr(pa, field)
        setattr(pa, field, bad)
        assert call(2) == want, field
        setattr(pa, field, old)
    pa.h_stride_b = 640                                  # sequences overlapping rows
    assert call(2) == b.ERR_INVALID_ARG
    pa.h = None                                          # a null pointer is fine when nothing is packed
    pa.n_tokens = 1
    assert call(2) not in (b.ERR_INVALID_ARG, b.ERR_ALIGNMENT)  # validation passes (device checks follow)


def test_constants_and_strings(lib):
    assert lib.csa_abi_version() == 1
    assert lib.csa_entry_bytes(512) == 288 and lib.csa_block_bytes(512) == 2304
    assert lib.csa_block_bytes(128) == 576 and lib.csa_block_bytes(64) == 288
    assert lib.csa_entry_bytes(10) == 0
    for s in range(8):
        assert lib.csa_status_string(s)
    assert b"unknown" in lib.csa_status_string(99)


def test_validation_rejects_before_any_device_call(lib):
    from compressed_sparse_attention_merge_b300 import binding as b
    # null argument blocks
    assert lib.csa_pack_fp4(1, None, None, 0, None) == b.ERR_INVALID_ARG
    assert lib.csa_index_topk(1, None, None, 0, None) == b.ERR_INVALID_ARG
    assert lib.csa_sparse_attn_decode(1, None, None, 0, None) == b.ERR_INVALID_ARG
    pa = b.PackArgs()
    pa.x_dtype, pa.dim, pa.merge, pa.scale_rule = 0, 100, 2, 0       # dim not a multiple of 64
    assert lib.csa_pack_fp4(1, ctypes.byref(pa), None, 0, None) == b.ERR_INVALID_ARG
    # multi-job pack: job count out of range, missing arrays, one bad job fails the call
    jobs = (b.PackArgs * 2)()
    batches = (ctypes.c_int64 * 2)(1, 1)
    assert lib.csa_pack_fp4_multi(0, batches, jobs, None, 0, None) == b.ERR_INVALID_ARG
    assert lib.csa_pack_fp4_multi(b.PACK_MAX_JOBS + 1, batches, jobs, None, 0, None) == b.ERR_INVALID_ARG
    assert lib.csa_pack_fp4_multi(1, None, jobs, None, 0, None) == b.ERR_INVALID_ARG
    jobs[0].x_dtype, jobs[0].dim, jobs[0].merge, jobs[0].scale_rule = 0, 512, 2, 0
    jobs[1].x_dtype, jobs[1].dim, jobs[1].merge, jobs[1].scale_rule = 0, 512, 3, 0     # merge 3
    assert lib.csa_pack_fp4_multi(2, batches, jobs, None, 0, None) == b.ERR_INVALID_ARG
    # unsupported indexer shape / attention head count
    ia = b.IndexArgs()
    ia.n_query, ia.heads, ia.dim, ia.top_k, ia.flags = 1, 3, 128, 8, b.IDX_RELU
    assert lib.csa_index_topk(1, ctypes.byref(ia), None, 0, None) == b.ERR_INVALID_ARG
    ia.heads, ia.top_k = 4, 5000
    assert lib.csa_index_topk(1, ctypes.byref(ia), None, 0, None) == b.ERR_INVALID_ARG
    ia.top_k, ia.flags = 8, b.IDX_RELU | b.IDX_HIER      # hierarchical without coarse keys
    assert lib.csa_index_topk(1, ctypes.byref(ia), None, 0, None) == b.ERR_INVALID_ARG
    aa = b.AttnArgs()
    aa.n_query, aa.heads, aa.top_k, aa.window, aa.scale = 1, 20, 8, 128, 0.04
    assert lib.csa_sparse_attn_decode(1, ctypes.byref(aa), None, 0, None) == b.ERR_INVALID_ARG
    aa.heads, aa.scale = 64, -1.0
    assert lib.csa_sparse_attn_prefill(1, ctypes.byref(aa), None, 0, None) == b.ERR_INVALID_ARG


def test_workspace_sizes_are_host_only(lib):
    from compressed_sparse_attention_merge_b300 import binding as b
    ia = b.IndexArgs()
    ia.n_query, ia.heads, ia.dim, ia.top_k, ia.flags, ia.max_entries = 1, 4, 128, 256, b.IDX_RELU, 32768
    n = lib.csa_index_topk_workspace_size(32, ctypes.byref(ia))
    assert n >= 256 + 32 * 4096 * 4 and n % 256 == 0
    ia.flags, ia.keep_blocks, ia.max_entries = b.IDX_RELU | b.IDX_HIER, 2048, 1 << 19
    n = lib.csa_index_topk_workspace_size(4, ctypes.byref(ia))
    assert n >= 256 + 4 * 2048 * 4 + 4 * 1024 * 4 + 4 * 32 * 4


def test_misaligned_pointers_rejected_before_any_device_call(lib):
    # pointers that are never dereferenced on the host: an 8-byte offset from a 16-byte boundary
    from compressed_sparse_attention_merge_b300 import binding as b
    bad, good = 0x10008, 0x10000
    pa = b.PackArgs()
    pa.x, pa.cache, pa.x_dtype, pa.dim, pa.merge, pa.scale_rule = bad, good, b.DTYPE_BF16, 512, 2, b.SCALE_AMAX
    pa.x_stride_b, pa.x_stride_t, pa.n_tokens, pa.max_entries = 4 * 512, 512, 4, 8
    assert lib.csa_pack_fp4(1, ctypes.byref(pa), None, 0, None) == b.ERR_ALIGNMENT
    pa.x, pa.x_stride_t = good, 516                      # a row stride of 1,032 bytes
    assert lib.csa_pack_fp4(1, ctypes.byref(pa), None, 0, None) == b.ERR_ALIGNMENT
    pa.x_stride_t = 512
    jobs = (b.PackArgs * 2)(pa, pa)
    jobs[1].cache = bad
    assert lib.csa_pack_fp4_multi(2, (ctypes.c_int64 * 2)(1, 1), jobs, None, 0, None) == b.ERR_ALIGNMENT
    ia = b.IndexArgs()
    ia.n_query, ia.heads, ia.dim, ia.top_k, ia.flags, ia.max_entries = 1, 4, 128, 8, b.IDX_RELU, 64
    ia.q_idx, ia.keys, ia.n_entries, ia.out_idx, ia.keys_stride_b = bad, good, good, good, 8 * 576
    assert lib.csa_index_topk(1, ctypes.byref(ia), None, 0, None) == b.ERR_ALIGNMENT
    aa = b.AttnArgs()
    aa.n_query, aa.heads, aa.top_k, aa.window, aa.scale, aa.max_entries = 1, 64, 8, 0, 0.04, 64
    aa.q, aa.cache, aa.n_entries, aa.idx, aa.out = good, good, good, good, bad
    assert lib.csa_sparse_attn_decode(1, ctypes.byref(aa), None, 0, None) == b.ERR_ALIGNMENT
    aa.out, aa.window, aa.swa, aa.swa_len, aa.swa_rows = good, 128, bad, good, 128
    assert lib.csa_sparse_attn_decode(1, ctypes.byref(aa), None, 0, None) == b.ERR_ALIGNMENT
    aa.swa, aa.cache = good, good + 16                   # 16-byte aligned is not enough for the latent cache
    assert lib.csa_sparse_attn_decode(1, ctypes.byref(aa), None, 0, None) == b.ERR_ALIGNMENT
    aa.cache, aa.cache_stride_b = good, 2304 * 8 + 16    # nor a stride that is not a multiple of 32
    assert lib.csa_sparse_attn_decode(2, ctypes.byref(aa), None, 0, None) == b.ERR_ALIGNMENT
    aa.cache_stride_b = 0
    # and the argument checks that come first
    aa.swa, aa.window = good, 2048                       # window above 1,024 rows
    assert lib.csa_sparse_attn_decode(1, ctypes.byref(aa), None, 0, None) == b.ERR_INVALID_ARG
    aa.window, aa.scale = 128, float("nan")
    assert lib.csa_sparse_attn_decode(1, ctypes.byref(aa), None, 0, None) == b.ERR_INVALID_ARG


def test_attention_workspace_size_is_host_only(lib):
    # without a device the size is the partials layout, 148 SMs assumed: 4 queries of
    # 16 cache tiles take 16 cache splits and a window split each, so 17 partials of (o, m, l) per head
    from compressed_sparse_attention_merge_b300 import binding as b
    aa = b.AttnArgs()
    aa.n_query, aa.heads, aa.top_k, aa.window, aa.scale = 1, 64, 256, 128, 0.04
    aa.max_entries, aa.swa_rows = 1 << 19, 128
    n = lib.csa_sparse_attn_workspace_size(4, ctypes.byref(aa))
    assert n % 256 == 0 and n >= 256 + 4 * 17 * 64 * (512 * 4 + 2 * 4)
    # one cache tile and one window tile: two splits, so partials; no window: one split, no partials
    aa.top_k = 16
    assert lib.csa_sparse_attn_workspace_size(1, ctypes.byref(aa)) >= 256 + 2 * 64 * (512 * 4 + 2 * 4)
    # no window: one split, no partials; the header and the NVFP4-query variant's rounded query (64 head rows
    # of 256 code bytes, 32 scale bytes and a 4-byte power of two)
    aa.swa_rows, aa.window = 0, 0
    assert lib.csa_sparse_attn_workspace_size(1, ctypes.byref(aa)) == 256 + 64 * 256 + 64 * 32 + 256


def test_static_index_validates_before_sizing(lib):
    # csa_index_topk_static checks its arguments first: a malformed call is CSA_ERR_INVALID_ARG (not a
    # workspace-size answer) and nothing is queued; without a device none of this needs one
    from compressed_sparse_attention_merge_b300 import binding as b
    ia = b.IndexArgs()
    ia.n_query, ia.heads, ia.dim, ia.top_k, ia.flags, ia.max_entries = -3, 4, 128, 8, b.IDX_RELU, 64
    assert lib.csa_index_topk_static(1, ctypes.byref(ia), None, None) == b.ERR_INVALID_ARG
    ia.n_query, ia.max_entries = 1, -5
    assert lib.csa_index_topk_static(1, ctypes.byref(ia), None, None) == b.ERR_INVALID_ARG
    # a call whose scratch would exceed the array but whose arguments are malformed (3 heads): invalid first
    ia.heads, ia.max_entries, ia.n_query = 3, 8 << 20, 64
    assert lib.csa_index_topk_static(4, ctypes.byref(ia), None, None) == b.ERR_INVALID_ARG
    # a well-formed call with misaligned queries: alignment, still before the size check
    ia.heads, ia.n_query, ia.max_entries = 4, 1, 64
    ia.q_idx, ia.keys, ia.n_entries, ia.out_idx, ia.keys_stride_b = 0x10008, 0x10000, 0x10000, 0x10000, 8 * 576
    assert lib.csa_index_topk_static(1, ctypes.byref(ia), None, None) == b.ERR_ALIGNMENT


def test_nvfp4q_attention_and_layer_flags_reject_before_any_device_call(lib):
    # the NVFP4-query calls share the exact calls' validation; csa_decode_layers checks every layer's flags
    # before anything is launched (none of this needs a device)
    from compressed_sparse_attention_merge_b300 import binding as b
    assert lib.csa_sparse_attn_decode_nvfp4q(1, None, None, 0, None) == b.ERR_INVALID_ARG
    assert lib.csa_sparse_attn_prefill_nvfp4q(1, None, None, 0, None) == b.ERR_INVALID_ARG
    aa = b.AttnArgs()
    aa.n_query, aa.heads, aa.top_k, aa.window, aa.scale = 1, 20, 8, 128, 0.04      # 20 heads
    assert lib.csa_sparse_attn_decode_nvfp4q(1, ctypes.byref(aa), None, 0, None) == b.ERR_INVALID_ARG
    aa.heads, aa.window = 64, 2048                                                 # window beyond 1,024
    assert lib.csa_sparse_attn_prefill_nvfp4q(1, ctypes.byref(aa), None, 0, None) == b.ERR_INVALID_ARG
    # a layer flag other than CSA_LAYER_ATTN_NVFP4Q
    layers = (b.LayerArgs * 1)()
    layers[0].mode, layers[0].flags = b.LAYER_FULL, 2
    ia, aa = b.IndexArgs(), b.AttnArgs()
    assert lib.csa_decode_layers(1, 1, layers, ctypes.byref(ia), ctypes.byref(aa), None, 0, None, 0,
                                 None) == b.ERR_INVALID_ARG
    # a first layer in Reuse mode (no indices to reuse)
    layers[0].mode, layers[0].flags = b.LAYER_REUSE, b.LAYER_ATTN_NVFP4Q
    assert lib.csa_decode_layers(1, 1, layers, ctypes.byref(ia), ctypes.byref(aa), None, 0, None, 0,
                                 None) == b.ERR_INVALID_ARG
