// Internal declarations shared by the kernels and the C-ABI layer of the CSA2 library.
// Device helpers here implement the cache format stated in include/csa.h (E2M1 codes, one E4M3
// scale per 16 elements, block-major layout) from the format definitions themselves.
#pragma once

#include <cuda.h>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "../../include/csa.h"

namespace csa {

// ------------------------------------------------------------------------------------------------
// Workspace header: word 0 = first status code recorded, 1 = kernel id, 2 = detail, 3 = count.
// ------------------------------------------------------------------------------------------------
enum KernelId : uint32_t {
  KID_PACK = 1,
  KID_COARSE_SUM = 2,
  KID_INDEX_SCORE = 3,
  KID_COARSE_SCORE = 4,
  KID_TOPK = 5,
  KID_ATTN = 6,
  KID_COMBINE = 7,
  KID_PROJECT = 8,
};

__device__ __forceinline__ void report(uint32_t* hdr, uint32_t code, uint32_t kernel, uint32_t detail) {
  if (atomicCAS(hdr, 0u, code) == 0u) {
    hdr[1] = kernel;
    hdr[2] = detail;
  }
  atomicAdd(hdr + 3, 1u);
}

// ------------------------------------------------------------------------------------------------
// Format helpers
// ------------------------------------------------------------------------------------------------
constexpr int kBlockEntries = CSA_BLOCK_ENTRIES;
constexpr int kGroup = CSA_SCALE_GROUP;
constexpr int kLatent = CSA_LATENT_DIM;
constexpr int kSuper = CSA_SUPER_BLOCK;

__host__ __device__ constexpr int entry_bytes(int dim) { return dim / 2 + dim / kGroup; }
__host__ __device__ constexpr int block_bytes(int dim) { return kBlockEntries * entry_bytes(dim); }

// Two E2M1 codes (low nibble = first element) -> f16x2 (first element in the low half).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t out;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(out) : "r"(byte));
  return out;
}

// One E4M3 byte -> f16x2 holding the value twice (every E4M3 value is exact in fp16).
__device__ __forceinline__ uint32_t e4m3_to_f16x2_bcast(uint32_t byte) {
  uint32_t out;
  const uint16_t pair = (uint16_t)((byte & 0xFFu) | ((byte & 0xFFu) << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(pair));
  return out;
}

__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  const uint32_t h2 = e4m3_to_f16x2_bcast(byte);
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Non-negative fp32 -> E4M3 byte, round to nearest even, saturating at 448. Both halves of the
// converted pair receive x, so the low byte is the result whichever half the instruction fills first.
__device__ __forceinline__ uint32_t float_to_e4m3_satfinite(float x) {
  uint16_t out;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(out) : "f"(x));
  return out & 0xFFu;
}

// E2M1 code of y: nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6 to |y|, ties to the even code (the thresholds
// alternate between strict and non-strict at the midpoints 0.25, 0.75, ..., 5), saturating at 6; the
// sign bit copies the sign bit of y.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  const float a = fabsf(y);
  uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) +
               (a > 5.0f);
  return c | ((__float_as_uint(y) >> 31) << 3);
}

// Smallest power of two >= sf (sf > 0), clamped to [2^-9, 256]; returns the E4M3 byte and the value.
__device__ __forceinline__ uint32_t pow2_scale(float sf, float* value) {
  const uint32_t bits = __float_as_uint(sf);
  const int e = (int)((bits >> 23) & 0xFFu);
  const uint32_t mant = bits & 0x7FFFFFu;
  int k = (e == 0) ? -126 : (mant == 0u ? e - 127 : e - 126);
  k = k < -9 ? -9 : (k > 8 ? 8 : k);
  *value = __uint_as_float((uint32_t)(k + 127) << 23);
  return k >= -6 ? (uint32_t)(k + 7) << 3 : (0x08u >> (-6 - k));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// ------------------------------------------------------------------------------------------------
// mbarrier and bulk-copy helpers (PTX ISA: mbarrier, cp.async.bulk). Every wait is bounded: a poll
// suspends the thread in hardware until the phase completes or kWaitHintNs pass, and after kSpinLimit
// polls (a few seconds at most) the wait gives up and returns false; the caller records CSA_ERR_TIMEOUT.
// ------------------------------------------------------------------------------------------------
constexpr uint32_t kSpinLimit = 1u << 17;
constexpr uint32_t kWaitHintNs = 20000;

// One poll of the phase with the given parity: true once it has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t done;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(done) : "r"(bar_addr), "r"(parity), "r"(kWaitHintNs) : "memory");
  return done != 0;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
               :: "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
               :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// Non-blocking check of the phase with the given parity: true if it has completed (no suspension).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t done;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(done) : "r"(bar_addr), "r"(parity) : "memory");
  return done != 0;
}

// Polls the phase with the given parity; true once it has completed, false after kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(a, parity)) return true;
  return false;
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from global to this CTA's
// shared memory; completion is counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// ------------------------------------------------------------------------------------------------
// Launch parameter blocks (host -> kernel launchers)
// ------------------------------------------------------------------------------------------------
struct PackParams {
  const void* x;
  int x_dtype, dim, merge, scale_rule;
  int64_t x_stride_b, x_stride_t, n_new, batch, max_entries;
  const int32_t* first_entry;
  uint8_t* cache;
  int64_t cache_stride_b;
  float* coarse_sum;
  int64_t coarse_stride_b;
  uint32_t* hdr;
};

// Several pack jobs in one launch: job j covers CTAs [cta_begin[j], cta_begin[j + 1]).
struct PackMulti {
  PackParams job[CSA_PACK_MAX_JOBS];
  int64_t cta_begin[CSA_PACK_MAX_JOBS + 1];
  int n;
};

struct ScoreParams {
  // queries
  const float* q_idx;          // [batch][n_query][heads][dim]
  const float* head_w;         // [heads] or null
  int64_t n_query;
  int heads, dim, relu;
  // keys
  const uint8_t* keys;
  int64_t keys_stride_b;
  const int32_t* n_entries;
  int64_t max_entries;
  const int32_t* q_pos;        // [batch][n_query] or null
  // hierarchical restriction: per unit list of kept super-blocks (null in flat mode)
  const int32_t* kept;         // [units][keep_super]
  int keep_super;
  // output: per unit block scores
  float* scores;               // [units][score_stride]
  int64_t score_stride;
  int64_t n_slots;             // blocks (flat) or compact slots (hierarchical) per unit
  int64_t batch;
  uint32_t* hdr;
};

struct CoarseScoreParams {
  const float* q_idx;
  const float* head_w;
  int64_t n_query;
  int heads, dim, relu;
  const float* coarse;
  int64_t coarse_stride_b;
  const int32_t* n_entries;
  int64_t n_super;
  float* scores;               // [units][n_super]
  int64_t batch;
};

struct TopkParams {
  const float* scores;         // [units][score_stride]
  int64_t score_stride;
  int64_t n;                   // candidates per unit
  int k;
  int32_t* out;                // [units][out_stride]
  int64_t out_stride;
  const int32_t* map_super;    // hierarchical: slot s -> map_super[unit][s / 64] * 64 + s % 64
  int map_stride;
  int64_t units;
  uint32_t* hdr;
};

struct AttnParams {
  int64_t units, n_query;
  int heads;
  float scale_log2;            // softmax scale * log2(e)
  const __nv_bfloat16* q;      // [units][heads][512]
  const uint8_t* cache;
  int64_t cache_stride_b;
  const int32_t* n_entries;
  int64_t max_entries;
  const int32_t* idx;          // [units][top_k]
  int top_k, window;
  const int32_t* q_pos;        // [units] or null (decode)
  const __nv_bfloat16* swa;
  int64_t swa_stride_b, swa_rows;
  const int32_t* swa_len;
  const int32_t* swa_first_pos;
  // Work split (grid.x = splits): cache splits 0 .. cache_splits-1 share the n_ct cache tiles (16 selected
  // blocks = 128 rows each); the n_wt window tiles (128 rows each) go to a split of their own when
  // win_split is set, else to the last cache split.
  int splits, cache_splits, win_split, n_ct, n_wt;
  // last_ct >= 0: the last cache split, which then also takes the window tiles, gets cache tiles
  // [n_ct - last_ct, n_ct) and the others share the rest evenly; -1: every cache split gets an even share.
  int last_ct;
  float* part_o;               // [units][splits][heads][512]
  float* part_ml;              // [units][splits][heads][2]
  float* out;                  // used when splits == 1
  float* out_lse;
  uint32_t* hdr;
  int q4;                      // host side: the NVFP4-query variant (block-scaled FP4 logits)
  // NVFP4-query variant: operands rounded by the prepare kernel (workspace). Per unit, 64 head rows (zero
  // beyond heads) of 256 code bytes, 32 scale bytes and the head's power of two 2^e; per sequence, swa_rows
  // window rows of 256 code bytes and 32 scale bytes.
  uint8_t* q4_codes;           // [units][64][256]
  uint8_t* q4_sc;              // [units][64][32]
  float* q4_mult;              // [units][64]
  uint8_t* w4;                 // [batch][swa_rows][256]
  uint8_t* w4_sc;              // [batch][swa_rows][32]
  // Exact attention with several splits a query: the queries converted once by the prepare kernel, each head
  // scaled by its power of two (q4_mult) and rounded to fp16 (exact), 64 head rows a unit; null otherwise.
  __half* qh;                  // [units][64][512]
  // Bounded waits give up after this many polls (kSpinLimit unless a test lowered it), and a nonzero
  // fault makes the kernel withhold one arrival (csa_debug_set_fault).
  uint32_t spin_limit;
  int fault;
};

// The fault and poll limit that csa_debug_set_fault set for later attention launches of this process.
void debug_fault(int* fault, uint32_t* spin_limit);

// ------------------------------------------------------------------------------------------------
// Programmatic dependent launch. Within one call of the C ABI, every kernel after the first is launched as
// a programmatic dependent of the kernel before it: it may start (and run its prologue: tensor-memory
// allocation, barrier setup, loads of the call's inputs) once every CTA of that kernel has passed
// griddep_launch(). Each kernel calls griddep_wait() before it reads anything the kernel before it
// writes, and before it exits; the wait returns once that kernel has completed and its writes are
// visible. A kernel signals griddep_launch() only after its own wait, so at most two kernels overlap and
// every earlier one has completed. A kernel whose first action is the wait (pack, coarse sums, indexer,
// Top-K, combine) is launched as a dependent even as the first kernel of a call; the attention kernel reads
// the call's inputs before its wait, so it is a dependent only after a kernel of the same call.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------------------------------------
// Launchers (one per kernel file). Each returns the launch error, if any; `pdl` launches the kernel as a
// programmatic dependent of the kernel before it in the stream (see above).
// ------------------------------------------------------------------------------------------------
cudaError_t launch_pack(const PackParams& p, cudaStream_t s);
cudaError_t launch_pack_multi(const PackParams* jobs, int n, cudaStream_t s);
cudaError_t launch_coarse_sum(const PackParams& p, cudaStream_t s);

// Fused latent projection + pair-merge + FP4 pack (csa_project_pack).
struct ProjectParams {
  const __nv_bfloat16* h;
  int64_t h_stride_b, h_stride_t, hidden, n_tokens, batch, max_entries, cache_stride_b;
  const __nv_bfloat16* w;
  int scale_rule;
  const int32_t* first_entry;
  uint8_t* cache;
  uint32_t* hdr;
};
cudaError_t launch_project_pack(const ProjectParams& p, cudaStream_t s);
cudaError_t launch_index_score(const ScoreParams& p, int num_sms, cudaStream_t s, bool pdl);
cudaError_t launch_coarse_score(const CoarseScoreParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_topk(const TopkParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_attn(const AttnParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_attn_prep(const AttnParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_combine(const AttnParams& p, cudaStream_t s, bool pdl);

// Clears an error that an earlier runtime call of another component left in this thread's last-error
// slot without checking it, so that the check after a launch reports that launch alone. A sticky error
// (a faulted context) is not cleared by this and still fails the launch.
inline void clear_stale_error() { (void)cudaGetLastError(); }

// Raises a kernel's dynamic shared-memory limit to `bytes`, once per (device, kernel). The first
// launch of a kernel on a device should not be inside stream capture (the attribute call is not a
// stream operation); later launches find the limit in the table and skip it.
cudaError_t ensure_smem_limit_fn(const void* kernel, int bytes);

template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel kernel, int bytes) {
  return ensure_smem_limit_fn(reinterpret_cast<const void*>(kernel), bytes);
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime (no link to libcuda);
// null if the driver does not provide it.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// Host-side checks of csa_index_topk's arguments (shapes, flags, pointers, alignment); CSA_OK when the call
// may proceed. Touches no device state.
csa_status validate_index_args(int64_t batch, const csa_index_args* a);

// Records the text of a CUDA runtime failure for csa_last_error() and returns CSA_ERR_CUDA.
csa_status cuda_fail(cudaError_t e, const char* where);
// Records a printf-style message for csa_last_error().
void set_last_error(const char* fmt, ...);

// Kernel timing hooks (defined in csa_api.cu); no-ops unless profiling is on.
void prof_begin(const char* name, cudaStream_t s);
void prof_end(cudaStream_t s);

struct ProfScope {
  cudaStream_t s;
  ProfScope(const char* name, cudaStream_t st) : s(st) { prof_begin(name, st); }
  ~ProfScope() { prof_end(s); }
};

}  // namespace csa
