/*
 * csa.h -- C ABI of the CSA2 compressed-sparse-attention library for B300 (sm_103a).
 *
 * The library implements one data path: a shared FP4 global KV cache built by pair-merging adjacent
 * token latents, a block indexer with Top-K selection (flat or hierarchical), and sparse attention
 * over the selected cache blocks merged with each layer's own sliding-window KV.
 *
 * Sources the operations follow (web pages about the DeepSeek-V4.1-Flash technical report):
 *   [digest] "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression" (paper-digest.app),
 *            sections "Core Mechanics" and "Terminology".
 *   [abstract] "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (thelatestinai.com),
 *            section "Abstract".
 *   [card]   "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (observer.broadside card),
 *            section "Key ideas".
 *   [news]   "DeepSeek Releases V4.1 Flash with 4x KV Cache Compression for Long-Context Agent
 *            Workflows" (promptgoblins), section "Details".
 * The pages fix the structure only (one 512-d latent shared by K and V across heads, 2 positions merged
 * per entry, FP4 storage, blocks of 8, Top-K, hierarchical indexing up to 2,048 blocks, a 128-token
 * sliding window, Full/Reindex/Reuse layers). Every numeric format and rounding rule below is this
 * library's own definition; each is stated where it is used.
 *
 * Conventions shared by every call
 *   - All pointers marked "device" are CUDA device pointers on the current device. The caller owns every
 *     buffer; the library never allocates or frees device memory.
 *   - Every call is stream-ordered and asynchronous on `stream`. The returned csa_status reports host-side
 *     validation only; when it is not CSA_OK nothing was launched.
 *   - Problems only the device can see (an out-of-range block id, an entry count beyond capacity) never
 *     trap: the kernel skips the offending item and records a code in the workspace header, which
 *     csa_get_device_status() returns. The header must be zeroed once (csa_workspace_reset) before first
 *     use; csa_get_device_status() clears it again after reading.
 *   - Only sm_103 devices are accepted (CSA_ERR_UNSUPPORTED_DEVICE otherwise). There is no CPU fallback.
 *   - Calls are safe from several host threads as long as they use different workspaces. Calls that share
 *     a workspace must be ordered on one stream.
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CSA_ABI_VERSION 1

/* Width of the shared latent that serves as key and value for every head ([digest] Core Mechanics,
   "Channel"). */
#define CSA_LATENT_DIM 512
/* Cache entries per selectable block ([card] Key ideas, "blocks of 8"). */
#define CSA_BLOCK_ENTRIES 8
/* Elements that share one E4M3 scale byte (format of this library). */
#define CSA_SCALE_GROUP 16
/* Blocks per super-block of the hierarchical indexer (reading of [card] Key ideas, "hierarchical
   sparse indexer (up to 2,048 blocks of 8 positions)"). */
#define CSA_SUPER_BLOCK 64
/* Largest Top-K (in blocks) accepted by csa_index_topk and the attention calls. */
#define CSA_MAX_TOP_K 2048
/* Bytes at the start of every workspace reserved for the device status word. */
#define CSA_WS_HEADER_BYTES 256

typedef enum csa_status {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = 1,        /* null pointer, bad size, unsupported shape or flag */
  CSA_ERR_ALIGNMENT = 2,          /* a pointer or stride breaks the alignment stated for it */
  CSA_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not sm_103 */
  CSA_ERR_WORKSPACE_TOO_SMALL = 4,
  CSA_ERR_CUDA = 5,               /* a CUDA runtime call failed (launch, attribute query) */
  CSA_ERR_DEVICE_CHECK = 6,       /* a kernel found invalid data; see the conventions above */
  CSA_ERR_TIMEOUT = 7             /* a bounded device-side wait gave up */
} csa_status;

enum { CSA_DTYPE_BF16 = 0, CSA_DTYPE_F32 = 1 };

/* Scale rule of the FP4 quantiser (format of this library):
 *   CSA_SCALE_AMAX: s = E4M3_rne_satfinite(amax / 6), the usual rule for latents.
 *   CSA_SCALE_POW2: s = smallest power of two >= amax / 6, clamped to [2^-9, 256]; exact for index keys
 *                   whose values are integers in [-4, 4]. */
enum { CSA_SCALE_AMAX = 0, CSA_SCALE_POW2 = 1 };

/* Indexer flags. CSA_IDX_RELU: score = sum_h w_h * max(0, q_h . k). Without it the ReLU is dropped.
   CSA_IDX_HIER: two-stage (super-block, then block) selection; decode only. */
enum { CSA_IDX_RELU = 1, CSA_IDX_HIER = 2 };

int csa_abi_version(void);
const char* csa_status_string(csa_status status);

/* Text describing the most recent failure of a csa_* call of this thread that had more to say than its
   status code: a CUDA runtime failure behind CSA_ERR_CUDA ("<step>: <CUDA error string> (<code>)"), or
   the sizes behind a CSA_ERR_WORKSPACE_TOO_SMALL of csa_index_topk_static; "" if there was none. The
   string is owned by the library and stays valid until the thread's next failing call. */
const char* csa_last_error(void);

/* Bytes of one packed entry of width `dim` (dim/2 code bytes + dim/16 scale bytes), and of one block
   of 8 entries. dim = 512 gives 288 and 2,304. Returns 0 for a dim that is not a positive multiple of 16. */
size_t csa_entry_bytes(int dim);
size_t csa_block_bytes(int dim);

/* Zeroes the workspace header (status word). Async on `stream`. */
csa_status csa_workspace_reset(void* ws, size_t ws_bytes, cudaStream_t stream);

/* Synchronizes `stream`, reads the workspace status word, clears it, and returns CSA_OK,
   CSA_ERR_DEVICE_CHECK or CSA_ERR_TIMEOUT (or CSA_ERR_CUDA if the synchronize failed). */
csa_status csa_get_device_status(void* ws, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------------
 * csa_pack_fp4 -- pair-merge and FP4-pack token rows into cache entries.
 *
 * Follows [digest] Core Mechanics ("Sequence: the Encoder merges 2 adjacent positions into 1 cache
 * entry"), [digest] Terminology / [abstract] Abstract / [card] Key ideas ("FP4 global KV").
 *
 * For every sequence b and new entry i in [0, n_tokens / merge):
 *   m = merge == 2 ? fl32(fl32(x[2i] + x[2i+1]) * 0.5)  :  x[i]        (fp32, IEEE round-to-nearest)
 * then per group of 16 elements: amax = max |m|, scale s by `scale_rule`, code_j = E2M1_rne_satfinite(
 * fl32(m_j / s)) (sign kept, so a negative value that rounds to zero is code 0x8; s == 0 gives all-zero
 * codes). An odd trailing token (merge == 2) is not packed.
 *
 * Entry e = first_entry[b] + i is written to block e / 8, slot e % 8 of sequence b:
 *   block = [8 x dim/2 code bytes, slot-major][8 x dim/16 E4M3 scale bytes, slot-major]
 *   code byte j of an entry holds element 2j in its low nibble and 2j+1 in its high nibble.
 *
 * If coarse_sum is not NULL, after packing every super-block (64 blocks = 512 entries) that received a
 * new entry is recomputed: coarse_sum[b][g][d] = the exact sum, rounded once to fp32, of the dequantized
 * element d over entries [512 g, min(512 (g+1), first_entry[b] + n_new)). This assumes entries are appended
 * in order, so that [0, first_entry[b] + n_new) is the valid prefix. (Dequantized values are multiples of
 * 2^-13 below 2,688 in magnitude, so the sum is taken exactly in 64-bit fixed point.)
 *
 * Arguments (all strides in elements unless stated):
 *   x            device, [batch][n_tokens][dim] rows of x_dtype; each row contiguous; 16-byte aligned rows.
 *   dim          512 for latents; any multiple of 64 up to 1024 for index keys.
 *   first_entry  device int32 [batch], or NULL for 0. first_entry[b] + n_new must be <= max_entries
 *                (else the sequence is skipped and CSA_ERR_DEVICE_CHECK recorded).
 *   cache        device, 16-byte aligned; sequence b starts at cache + b * cache_stride_b (bytes, a multiple
 *                of 16, >= ceil(max_entries / 8) * csa_block_bytes(dim)).
 *   coarse_sum   device fp32 [batch][ceil(max_entries / 512)][dim] with stride coarse_stride_b, or NULL.
 *   ws           workspace of at least CSA_WS_HEADER_BYTES (status word only).
 * ------------------------------------------------------------------------------------------------ */
typedef struct csa_pack_args {
  const void* x;
  int32_t x_dtype;
  int32_t dim;
  int64_t x_stride_b;
  int64_t x_stride_t;
  int64_t n_tokens;
  int32_t merge;
  int32_t scale_rule;
  const int32_t* first_entry;
  int64_t max_entries;
  uint8_t* cache;
  int64_t cache_stride_b;
  float* coarse_sum;
  int64_t coarse_stride_b;
} csa_pack_args;

csa_status csa_pack_fp4(int64_t batch, const csa_pack_args* args, void* ws, size_t ws_bytes,
                        cudaStream_t stream);

/* ------------------------------------------------------------------------------------------------
 * csa_project_pack -- project hidden rows to 512-d latents, then pair-merge and FP4-pack them, in one
 * kernel (the latents never reach memory).
 *
 * Follows [card] Key ideas ("Causal Encoder-Decoder (CED)": the upper layers' global KV is projected from
 * the hidden state of a middle layer) and csa_pack_fp4 for the merge and the format.
 *
 * For every sequence b and token t in [0, n_tokens):
 *   x[t][j] = sum over k of h[b][t][k] * w[j][k]     (j < 512; bf16 inputs, fp32 accumulation on the tensor
 *                                                   cores, in an order of their own: the result equals the
 *                                                   exactly rounded sum whenever every partial sum is exact in
 *                                                   fp32, such as for small-integer inputs)
 * then the rows x go through csa_pack_fp4 with merge 2, dim 512 and scale_rule (an odd trailing token is
 * not packed): entry first_entry[b] + i holds the merged pair (2i, 2i + 1).
 *
 * Arguments (strides in elements):
 *   h            device bf16 [batch][n_tokens][hidden], rows contiguous; 16-byte aligned, with h_stride_t and
 *                h_stride_b multiples of 8 (h_stride_t >= hidden).
 *   hidden       64 .. 16,384, a multiple of 64.
 *   w            device bf16 [512][hidden] (output-major, like a linear layer's weight), contiguous,
 *                16-byte aligned.
 *   scale_rule, first_entry, max_entries, cache, cache_stride_b: as csa_pack_fp4 with dim 512.
 *   ws           workspace of at least CSA_WS_HEADER_BYTES (status word only).
 * Errors: CSA_ERR_INVALID_ARG / CSA_ERR_ALIGNMENT before any launch; a sequence whose first_entry[b] +
 * n_tokens / 2 exceeds max_entries is skipped and CSA_ERR_DEVICE_CHECK recorded; a bounded wait that runs
 * out records CSA_ERR_TIMEOUT.
 * ------------------------------------------------------------------------------------------------ */
typedef struct csa_project_args {
  const void* h;
  int64_t h_stride_b;
  int64_t h_stride_t;
  int64_t hidden;
  const void* w;
  int64_t n_tokens;
  int32_t scale_rule;
  int32_t reserved;          /* must be 0 */
  const int32_t* first_entry;
  int64_t max_entries;
  uint8_t* cache;
  int64_t cache_stride_b;
} csa_project_args;

csa_status csa_project_pack(int64_t batch, const csa_project_args* args, void* ws, size_t ws_bytes,
                            cudaStream_t stream);

/* csa_pack_fp4_multi -- n_jobs csa_pack_fp4 calls (job j: batch[j] sequences, args[j]) in as few
 * launches as their sizes allow. A decode step appends to the latent cache and to the index-key cache, and
 * this call does both in one launch. The result equals the calls made one after another in job order,
 * provided no two jobs write the same cache entry or the same coarse sums. If they do, the bytes are
 * undefined. Every job is validated as csa_pack_fp4 validates it before anything is launched; a job
 * that fails validation fails the whole call, and nothing is launched.
 *   n_jobs  1..CSA_PACK_MAX_JOBS.
 *   batch   host int64 [n_jobs].
 *   args    host [n_jobs].
 *   ws      one workspace header, shared by all jobs; it records the first device check of any job.
 * Jobs whose batch or new-entry count is 0 are skipped. */
#define CSA_PACK_MAX_JOBS 4
csa_status csa_pack_fp4_multi(int n_jobs, const int64_t* batch, const csa_pack_args* args, void* ws,
                              size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------------
 * csa_index_topk -- score cache blocks with an indexer query and select the Top-K blocks.
 *
 * Follows [card] Key ideas ("Reindex ... rescore with its own indexer query", "Reuse (reuse both KV and
 * Top-K indices)", "a hierarchical sparse indexer (up to 2,048 blocks of 8 positions) trims decoder
 * indexing") and [news] Details ("block-based approach").
 *
 * Per query u = (b, j):
 *   entry score   s_e = sum over h = 0..H-1, in that order, of fl32(w_h * r_{h,e}),
 *                 r_{h,e} = max(0, q^_h . k_e) (plain q^_h . k_e without CSA_IDX_RELU), where k_e is the
 *                 dequantized index key and q^_h is the query rounded to the same FP4 format with the
 *                 CSA_SCALE_POW2 rule (E2M1 codes, one power-of-two scale per 16 elements; the identity for
 *                 integer values in [-4, 4]). Both enter a block-scaled FP4 tensor-core product with fp32
 *                 accumulation, exact when the dequantized values are integers and |partial sums| < 2^24.
 *   eligible      e < n_entries[b], and 2e + 1 <= q_pos[b][j] when q_pos is given (prefill causality).
 *   block score   S_blk = max of s_e over eligible entries of the block; blocks with none are not
 *                 candidates.
 *   Top-K         the min(top_k, #candidates) candidates with the largest S, ties to the lower block id,
 *                 written in ascending block id and padded with -1.
 *   CSA_IDX_HIER  (q_pos must be NULL) super-block g (blocks [64 g, 64 g + 64)) is first scored with the
 *                 same score function applied to coarse_sum[b][g]; the keep_blocks / 64 best super-blocks
 *                 (ties to the lower id) are kept and the block Top-K runs over their blocks only.
 *
 * Arguments:
 *   q_idx     device fp32 [batch][n_query][heads][dim], contiguous; 16-byte aligned.
 *   heads     1, 2, 4 or 8.   dim: 64, 128 or 256.
 *   head_w    device fp32 [heads] or NULL for all ones.
 *   keys      device packed index keys (csa_pack_fp4 layout with width dim), 16-byte aligned; sequence b
 *             at keys + b * keys_stride_b bytes (a multiple of 16).
 *   n_entries device int32 [batch]; each in [0, max_entries].
 *   q_pos     device int32 [batch][n_query] token positions (prefill) or NULL (decode: every entry
 *             below n_entries is eligible).
 *   coarse_sum, coarse_stride_b   CSA_IDX_HIER only: as written by csa_pack_fp4.
 *   keep_blocks CSA_IDX_HIER only: a multiple of 64, at most 4096 (the pages' figure is 2,048).
 *   top_k     1..CSA_MAX_TOP_K.
 *   out_idx   device int32 [batch][n_query][top_k].
 *   out_block_scores  optional device fp32 [batch][n_query][ceil(max_entries / 8)] (flat mode only):
 *             the block scores, -inf for non-candidates.
 *   ws        at least csa_index_topk_workspace_size(batch, args) bytes, 256-byte aligned.
 * ------------------------------------------------------------------------------------------------ */
typedef struct csa_index_args {
  int64_t n_query;
  int32_t heads;
  int32_t dim;
  const float* q_idx;
  const float* head_w;
  int32_t flags;
  int32_t top_k;
  const uint8_t* keys;
  int64_t keys_stride_b;
  const int32_t* n_entries;
  int64_t max_entries;
  const int32_t* q_pos;
  const float* coarse_sum;
  int64_t coarse_stride_b;
  int32_t keep_blocks;
  int32_t reserved0;
  int32_t* out_idx;
  float* out_block_scores;
} csa_index_args;

size_t csa_index_topk_workspace_size(int64_t batch, const csa_index_args* args);
csa_status csa_index_topk(int64_t batch, const csa_index_args* args, void* ws, size_t ws_bytes,
                          cudaStream_t stream);

/* ------------------------------------------------------------------------------------------------
 * csa_index_topk_static -- csa_index_topk for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call: it exists for callers of this library that have no way to
 * hand csa_index_topk a workspace, such as code inside a host framework whose allocator owns all device
 * memory and forbids raw cudaMalloc, plug-ins that may only use the buffers they are given, or serving
 * loops that must not allocate once running. It computes exactly what csa_index_topk computes, with the
 * same arguments and validation, but takes its scratch from a fixed array that the library places in
 * device memory when it is loaded. It never calls cudaMalloc, cudaFree or any other allocating routine.
 *
 *   - The array holds CSA_STATIC_INDEX_SCRATCH_BYTES (4 MiB). A call whose csa_index_topk_workspace_size
 *     is larger is rejected with CSA_ERR_WORKSPACE_TOO_SMALL before anything is launched, and
 *     csa_last_error() gives both sizes. Every GPU that loads the library holds the array until exit.
 *   - The first call on a device (with that device current) looks up the array's device address; make
 *     that first call before capturing any stream on that device. A lookup that fails is retried by the
 *     next call. Invalid arguments are rejected (CSA_ERR_INVALID_ARG, CSA_ERR_ALIGNMENT) before the size
 *     check and before anything is queued.
 *   - Every call on a device shares the one array, and it keeps the previous call's contents; each call
 *     clears the status word itself. Calls whose work overlaps on the GPU (different streams, or
 *     different host threads, without ordering between them) race on the array and give undefined
 *     results: order them on one stream.
 *   - status_out: optional device int32. When given, it receives the call's device status word after
 *     the kernels finish (stream-ordered): 0, or CSA_ERR_DEVICE_CHECK / CSA_ERR_TIMEOUT as
 *     csa_get_device_status() would report for a workspace.
 * ------------------------------------------------------------------------------------------------ */
#define CSA_STATIC_INDEX_SCRATCH_BYTES (4u << 20)

csa_status csa_index_topk_static(int64_t batch, const csa_index_args* args, int32_t* status_out,
                                 cudaStream_t stream);

/* ------------------------------------------------------------------------------------------------
 * csa_sparse_attn_decode / csa_sparse_attn_prefill -- attention over the selected blocks of the shared
 * FP4 cache merged with the layer's own sliding-window KV.
 *
 * Follows [digest] Core Mechanics ("one 512-dim latent shares keys and values across all attention
 * heads"), [digest] Terminology ("SWA ... each token sees only a recent window (128 here)") and [card]
 * Key ideas ("Every layer keeps its own query and sliding-window KV").
 *
 * Per query u = (b, j) and head h, the rows are
 *   R = { dequantized entry e of every block listed in idx[u] (id >= 0), e eligible }  U  W_u
 * where eligibility is as for csa_index_topk and W_u is the window:
 *   decode : rows 0 .. swa_len[b]-1 of swa[b]
 *   prefill: the rows of tokens max(p - window + 1, swa_first_pos[b]) .. p, p = q_pos[b][j]; the row of
 *            token t is t - swa_first_pos[b].
 * A row c (512 values) is both key and value:
 *   z_c = scale * (q_h . c),  out[u][h] = sum_c softmax(z)_c * c,  out_lse[u][h] = log sum_c exp(z_c).
 * Duplicates between the cache and the window are not removed. A query with no rows gets out = 0 and
 * lse = -inf.
 *
 * Precision (library choice): cache rows are dequantized exactly (E2M1 x E4M3 products fit fp16). Each
 * head of q is scaled by the power of two that puts its largest magnitude in [2^14, 2^15) and converted
 * to fp16, exactly for any finite bf16 query (elements more than 2^28 below the head's largest lose bits),
 * the factor going into that head's softmax scale. Window rows are converted from bf16 to fp16 (exact for
 * 2^-14 <= |x| <= 65504; smaller magnitudes lose at most 2^-25 absolute); a window value beyond 65504
 * is outside the contract and is reported as CSA_ERR_DEVICE_CHECK (the outputs of that query are then
 * undefined). Products are accumulated in fp32, probabilities are rounded to fp16 for the value product,
 * sums are fp32.
 *
 * Causal and independent queries. csa_sparse_attn_prefill is the causal multi-query call: query j of
 * sequence b sits at token q_pos[b][j] and sees only what exists at that position. It serves prefill
 * chunks and also the draft positions of a multi-token decode step (speculative verification, [card] Key
 * ideas, "Near-flat decode cost": DSpark speculative decoding): drafts at tokens p .. p + Q - 1 pass
 * q_pos = p .. p + Q - 1 (to csa_index_topk as well), so draft j sees the entries with 2e + 1 <= p + j,
 * including an entry completed by an earlier draft, and the window tokens up to p + j.
 * csa_sparse_attn_decode with n_query > 1 instead runs independent queries that all see the whole cache
 * prefix (n_entries[b]) and the same window rows.
 *
 * Arguments:
 *   n_query   queries per sequence (decode: independent queries over the whole prefix; prefill: causal).
 *   heads     16, 32, 48 or 64.   scale: softmax scale (1/sqrt(512) for the pages' latent).
 *   q         device bf16 [batch][n_query][heads][512], contiguous, 16-byte aligned.
 *   cache     device packed latent cache (csa_pack_fp4, dim 512), 32-byte aligned (the kernel reads
 *             it in 32-byte sectors); stride in bytes, a multiple of 32.
 *   n_entries device int32 [batch]; max_entries bounds it and the block ids.
 *   idx       device int32 [batch][n_query][top_k] block ids (ascending not required; -1 = empty slot).
 *   window    sliding-window length in rows, 0..1024 (the pages use 128).
 *   swa       device bf16 [batch][swa_rows][512] (stride swa_stride_b elements, rows contiguous).
 *   swa_len   decode: device int32 [batch], each in [0, min(window, swa_rows)].
 *   swa_first_pos, q_pos  prefill: device int32 [batch] and [batch][n_query].
 *   out       device fp32 [batch][n_query][heads][512].   out_lse: device fp32 [batch][n_query][heads]
 *             or NULL.
 *   ws        at least csa_sparse_attn_workspace_size(batch, args) bytes, 256-byte aligned.
 * ------------------------------------------------------------------------------------------------ */
typedef struct csa_attn_args {
  int64_t n_query;
  int32_t heads;
  float scale;
  const void* q;
  const uint8_t* cache;
  int64_t cache_stride_b;
  const int32_t* n_entries;
  int64_t max_entries;
  const int32_t* idx;
  int32_t top_k;
  int32_t window;
  const int32_t* q_pos;
  const void* swa;
  int64_t swa_stride_b;
  int64_t swa_rows;
  const int32_t* swa_len;
  const int32_t* swa_first_pos;
  float* out;
  float* out_lse;
} csa_attn_args;

/* Workspace bytes for one call with these arguments on the current device (the same for the NVFP4-query
 * calls below). A query's rows are cut into 128-row tiles shared by several CTAs (splits), as many as fill the
 * device's SMs. With more than one split the workspace holds every split's partial (o, m, l), which a second
 * kernel merges. It also holds the NVFP4-query variant's rounded operands: 64 head rows per query of 288 bytes
 * plus a 4-byte power of two, and 288 bytes per window row. The answer depends on the device's SM count, so
 * query it with the device current that will run the call. */
size_t csa_sparse_attn_workspace_size(int64_t batch, const csa_attn_args* args);
csa_status csa_sparse_attn_decode(int64_t batch, const csa_attn_args* args, void* ws, size_t ws_bytes,
                                  cudaStream_t stream);
csa_status csa_sparse_attn_prefill(int64_t batch, const csa_attn_args* args, void* ws, size_t ws_bytes,
                                   cudaStream_t stream);

/* ------------------------------------------------------------------------------------------------
 * csa_sparse_attn_decode_nvfp4q / csa_sparse_attn_prefill_nvfp4q -- the same attention with the logits taken
 * on the block-scaled FP4 tensor cores (opt-in; an approximation of the calls above).
 *
 * [card] Key ideas, "FP4 global KV, trained that way", stores the global KV in FP4 with one scale per
 * 16 elements, the operand format of the block-scaled FP4 product, which needs both operands in FP4. The
 * pages give no query format; this variant is the library's reading. It computes what
 * csa_sparse_attn_decode / csa_sparse_attn_prefill compute (same rows, eligibility, window, outputs and
 * workspace) with two roundings inside the logits z_c = scale * (q4_h . k_c):
 *   q4_h  each query head scaled by 2^-e_h, e_h = floor(log2 max|q_h|) - 10 clamped to [-100, 100] (0 for an
 *         all-zero head), rounded like csa_pack_fp4 with CSA_SCALE_AMAX (per 16 elements an E4M3 scale of
 *         amax / 6, E2M1 codes), and scaled back by 2^e_h;
 *   k_c   a cache row as stored; a window row rounded like csa_pack_fp4 with CSA_SCALE_AMAX (no merge, no
 *         pre-scale; magnitudes above 2688 saturate).
 * Values are exact: out[u][h] = sum_c softmax(z)_c * c uses the dequantized cache rows and the bf16 window
 * rows, as in the exact calls. Logits are accumulated in fp32. A first kernel rounds every query head and
 * every window row once per call into the workspace; the attention kernel copies those and the cache's code
 * bytes in by tensor map (the cache's 32-byte alignment and stride rule apply, as above). All other argument
 * rules and error behaviour are those of the exact calls.
 * ------------------------------------------------------------------------------------------------ */
csa_status csa_sparse_attn_decode_nvfp4q(int64_t batch, const csa_attn_args* args, void* ws, size_t ws_bytes,
                                         cudaStream_t stream);
csa_status csa_sparse_attn_prefill_nvfp4q(int64_t batch, const csa_attn_args* args, void* ws, size_t ws_bytes,
                                          cudaStream_t stream);

/* ------------------------------------------------------------------------------------------------
 * csa_decode_layers -- a step of several layers over one shared cache: for every layer in order, the
 * indexer (Full and Reindex layers) and the sparse attention.
 *
 * Follows [card] Key ideas, "CSA2 with three static layer modes": a Full layer makes the global KV and
 * the index, a Reindex layer reuses the KV but rescores with its own indexer query, a Reuse layer reuses
 * both the KV and the Top-K indices; "Every layer keeps its own query and sliding-window KV".
 *
 * index_tmpl and attn_tmpl hold everything the layers share (keys, entry counts, Top-K size, flags,
 * hierarchical keys, cache, window lengths, scale, heads, and q_pos for causal positions); their per-layer
 * pointers (q_idx, out_idx; q, idx, swa, out, out_lse) are ignored and taken from layers[l]:
 *   CSA_LAYER_FULL / CSA_LAYER_REINDEX: csa_index_topk with q_idx into idx, then attention over idx;
 *   CSA_LAYER_REUSE: attention over the idx of the most recent Full or Reindex layer (layers[l].q_idx and
 *                    layers[l].idx are ignored).
 * Attention runs as csa_sparse_attn_prefill when attn_tmpl->q_pos is set (causal positions, e.g. the
 * draft tokens of a multi-token decode step) and as csa_sparse_attn_decode otherwise.
 * ws_index and ws_attn are sized by csa_index_topk_workspace_size / csa_sparse_attn_workspace_size for the
 * templates; they are reused by every layer, in order, on `stream`. Every layer is validated before
 * anything is launched; the first layer may not be a Reuse layer.
 * ------------------------------------------------------------------------------------------------ */
enum { CSA_LAYER_FULL = 0, CSA_LAYER_REINDEX = 1, CSA_LAYER_REUSE = 2 };
/* Layer flags. CSA_LAYER_ATTN_NVFP4Q: the layer's attention is the NVFP4-query variant
 * (csa_sparse_attn_decode_nvfp4q / csa_sparse_attn_prefill_nvfp4q). Other bits must be 0. */
enum { CSA_LAYER_ATTN_NVFP4Q = 1 };

typedef struct csa_layer_args {
  int32_t mode;
  int32_t flags;
  const float* q_idx;   /* indexer queries [batch][n_query][heads][dim] (Full / Reindex) */
  int32_t* idx;         /* Top-K output [batch][n_query][top_k] (Full / Reindex) */
  const void* q;        /* attention queries, bf16 [batch][n_query][heads][512] */
  const void* swa;      /* this layer's window rows (layout of csa_attn_args.swa), or NULL if window = 0 */
  float* out;           /* [batch][n_query][heads][512] */
  float* out_lse;       /* [batch][n_query][heads] or NULL */
} csa_layer_args;

csa_status csa_decode_layers(int64_t batch, int n_layers, const csa_layer_args* layers,
                             const csa_index_args* index_tmpl, const csa_attn_args* attn_tmpl, void* ws_index,
                             size_t ws_index_bytes, void* ws_attn, size_t ws_attn_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------------
 * csa_debug_set_fault -- test-only fault injection for the device-side failure path.
 *
 * Every wait inside the library's kernels is bounded: after a fixed number of polls it gives up, records
 * CSA_ERR_TIMEOUT in the workspace status word (read by csa_get_device_status) and the kernel's other
 * roles stop too, so the kernel returns and the CUDA context stays usable. This call lets a test make such
 * a wait run out without any GPU fault: with fault = CSA_FAULT_WITHHOLD_ARRIVAL, later attention launches
 * of this process withhold one internal arrival (the value products of a CTA's first tile never report
 * completion), so a wait behind it gives up after spin_limit polls (each poll suspends for at most about
 * 20 microseconds). fault = CSA_FAULT_NONE restores normal launches (spin_limit is then ignored and the
 * library's own limit applies). Process-wide, not thread-safe; not for production use.
 * ------------------------------------------------------------------------------------------------ */
enum { CSA_FAULT_NONE = 0, CSA_FAULT_WITHHOLD_ARRIVAL = 1 };
csa_status csa_debug_set_fault(int fault, uint32_t spin_limit);

/* ------------------------------------------------------------------------------------------------
 * Kernel timing (opt-in, not thread-safe). Between csa_profile_begin and csa_profile_end every kernel
 * this library launches is bracketed by two CUDA timing events recorded on its launch stream (also
 * inside stream capture, as external event nodes). csa_profile_end synchronizes the device and reports,
 * per kernel name, the number of launches and their summed device time. Launches beyond max_launches
 * are counted in *dropped but not timed.
 * ------------------------------------------------------------------------------------------------ */
typedef struct csa_kernel_time {
  char name[48];
  int64_t launches;
  double total_ms;
} csa_kernel_time;

csa_status csa_profile_begin(int max_launches);
csa_status csa_profile_end(csa_kernel_time* out, int max_out, int* n_out, int64_t* dropped);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H_ */
