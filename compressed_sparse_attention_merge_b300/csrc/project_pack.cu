// Fused cache write: latent projection of hidden rows (a bf16 GEMM on the fifth-generation tensor cores),
// then pair-merge and FP4 pack in the epilogue, straight into the cache.
//
// Follows "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (card), Key ideas, "Causal
// Encoder-Decoder (CED)": the upper layers' global KV is projected from the hidden state of a middle layer.
// Also "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression" (paper-digest), Core Mechanics,
// "Sequence": two adjacent positions merge into one cache entry. The merge and the FP4 format are those of
// csa_pack_fp4 (include/csa.h), and the quantisation below takes the same steps in the same order.
//
// Design. The kernel is persistent: one CTA per SM loops over work items, an item being 128 tokens (64
// entries) of one sequence and one half (256 columns) of the 512 latent columns.
//   - One warp streams K-major 64-element slices of the hidden rows ([128 x 64]) and of the weight
//     ([256 x 64]) by tensor map into a 4-stage ring, 128-byte swizzled, item after item.
//   - One warp issues tcgen05.mma.kind::f16 (bf16 x bf16, fp32 accumulator, M = 128 tokens, N = 256) into one
//     of two accumulators in tensor memory (2 x 256 columns), so that the products of the next item run
//     while the epilogue reads the last one.
//   - Four epilogue warps (thread = token = tensor-memory lane) read an accumulator 32 columns at a time.
//     The two tokens of a pair sit in adjacent lanes, and each lane of a pair takes one of the two 16-column
//     groups. It gets the partner's half of that group with one shuffle per column, merges, quantises, and
//     stores its 8 code bytes and its scale byte.
// Neighbouring CTAs take the two column halves of a token tile at the same time, so the second reads the
// hidden rows from L2.
#include <cuda.h>

#include <cstring>

#include "csa_internal.cuh"
#include "tc.cuh"

namespace csa {
namespace {

constexpr int kTokTile = 128;                   // tokens per CTA: M of the product
constexpr int kNHalf = 256;                     // latent columns per CTA: N of the product
constexpr int kKStep = 64;                      // hidden elements per stage (128 bytes of bf16: one swizzle span)
constexpr int kStages = 4;
constexpr int kThreads = 192;                   // warp 0 copies, 1 MMA, 2-5 epilogue
constexpr int kAStage = kTokTile * kKStep * 2;  // 16 KB
constexpr int kBStage = kNHalf * kKStep * 2;    // 32 KB
constexpr int kAOff = 0;
constexpr int kBOff = kAOff + kStages * kAStage;
constexpr int kBarOff = kBOff + kStages * kBStage;
constexpr int kSmem = kBarOff + (2 * kStages + 5) * 8 + 16;
constexpr uint32_t kTmemCols = kNHalf;
constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kTokTile, kNHalf, 0, 0);
static_assert(kBOff % 1024 == 0 && kAStage % 1024 == 0 && kBStage % 1024 == 0, "swizzled stages on 1 KB");
static_assert(kSmem <= 232448, "shared memory");

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
               " [%0], [%1, {%2, %3}], [%4];"
               :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
               " [%0], [%1, {%2, %3, %4}], [%5];"
               :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
                  "r"(smem_addr(bar)) : "memory");
}

// Bounded wait that gives up (and records a timeout) after kSpinLimit polls or once another role gave up.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint32_t* hdr) {
  const uint32_t a = smem_addr(bar);
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 7u) == 7u && *abort_flag) return false;
  }
  *abort_flag = 1;
  report(hdr, CSA_ERR_TIMEOUT, KID_PROJECT, blockIdx.x);
  return false;
}

// The same wait taken by a whole warp; the result is the same on every lane.
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint32_t* hdr) {
  return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag, hdr));
}

// Bounded wait that ignores the abort flag (work in flight that must finish before the CTA exits).
__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(a, parity)) return;
}

__global__ void __launch_bounds__(kThreads, 1) project_pack_kernel(const ProjectParams p, int64_t tiles,
                                                                    const __grid_constant__ CUtensorMap h_map,
                                                                    const __grid_constant__ CUtensorMap w_map) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;            // [2]: an accumulator holds a finished item
  uint64_t* acc_empty = acc_full + 2;              // [2]: the epilogue has read it
  uint64_t* done = acc_empty + 2;
  uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_ptr + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // setup (no global memory: this overlaps the kernel before)
  if (warp == 1) tc::alloc(tmem_ptr, 2 * kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], 4); }
    mbar_init(done, 1);
    fence_mbar_init();
    *abort_flag = 0;
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  griddep_wait();                                  // before any global access: the cache may still be read before
  griddep_launch();
  const uint32_t tbase = *tmem_ptr;
  const int nk = (int)(p.hidden / kKStep);
  // Work items: item i is column half i & 1 of token tile (i >> 1) % tiles of sequence (i >> 1) / tiles. A CTA
  // takes items blockIdx.x, blockIdx.x + gridDim.x, ...; the grid is even, so the two halves of a tile run at
  // the same time on neighbouring CTAs.
  const int64_t total = 2 * tiles * p.batch;

  if (warp == 0) {
    // ---------------- tensor-map copies of the hidden and weight slices, item after item ----------------
    if (lane == 0) {
      int64_t g = 0;                               // stages issued by this CTA
      bool ok = true;
      for (int64_t item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const int half = (int)(item & 1);
        const int64_t t0 = ((item >> 1) % tiles) * kTokTile, b = (item >> 1) / tiles;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int slot = (int)(g % kStages);
          if (g >= kStages && !wait_or_abort(&empty[slot], (uint32_t)((g / kStages) - 1) & 1u, abort_flag, p.hdr)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[slot], kAStage + kBStage);
          tma_load_3d(smem + kAOff + slot * kAStage, &h_map, kb * kKStep, (int)t0, (int)b, &full[slot]);
          tma_load_2d(smem + kBOff + slot * kBStage, &w_map, kb * kKStep, kNHalf * half, &full[slot]);
        }
      }
      // no copy into this CTA's shared memory may still be in flight when it exits
      for (int64_t k = g - kStages < 0 ? 0 : g - kStages; k < g; ++k) drain(&full[k % kStages], (uint32_t)(k / kStages) & 1u);
    }
  } else if (warp == 1) {
    // ---------------- products: x[128 x 256] += h[128 x 64] . w[256 x 64]^T per stage, into accumulator
    // j & 1 for the CTA's j-th item ----------------
    const uint32_t a0 = smem_addr(smem + kAOff), b0 = smem_addr(smem + kBOff);
    int64_t g = 0;
    int j = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; item < total && ok; item += gridDim.x, ++j) {
      const int acc = j & 1;
      // the epilogue has read what item j - 2 left in this accumulator
      if (j >= 2 && !wait_bar_warp(&acc_empty[acc], (uint32_t)((j >> 1) - 1) & 1u, abort_flag, p.hdr)) break;
      tc::fence_after();
      const uint32_t d = tbase + acc * kTmemCols;
      for (int kb = 0; kb < nk; ++kb, ++g) {
        const int slot = (int)(g % kStages);
        if (!wait_bar_warp(&full[slot], (uint32_t)(g / kStages) & 1u, abort_flag, p.hdr)) { ok = false; break; }
        tc::fence_after();
#pragma unroll
        for (int ks = 0; ks < kKStep / 16; ++ks) {
          const uint64_t a = tc::smem_desc(a0 + slot * kAStage + ks * 32, 16, 1024, tc::kSwizzle128B);
          const uint64_t bd = tc::smem_desc(b0 + slot * kBStage + ks * 32, 16, 1024, tc::kSwizzle128B);
          tc::mma_f16_warp(d, a, bd, kIdesc, (kb | ks) != 0 ? 1u : 0u);
        }
        tc::commit_warp(&empty[slot]);
      }
      if (ok) tc::commit_warp(&acc_full[acc]);
    }
    // every product issued must be complete before the tensor memory is released
    tc::commit_warp(done);
    drain(done, 0);
    __syncwarp();
  } else {
    // ---------------- epilogue: merge, quantise and store (thread = token row), item after item ----------------
    const int sp = warp & 3;
    const int r = sp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(sp * 32) << 16;
    const int64_t n_pairs = p.n_tokens / 2;
    const bool odd = (lane & 1) != 0;
    int j = 0;
    for (int64_t item = blockIdx.x; item < total; item += gridDim.x, ++j) {
      const int acc = j & 1;
      const int half = (int)(item & 1);
      const int64_t tile = (item >> 1) % tiles, b = (item >> 1) / tiles;
      if (!wait_bar_warp(&acc_full[acc], (uint32_t)(j >> 1) & 1u, abort_flag, p.hdr)) break;
      tc::fence_after();
      const int64_t pair = ((tile * kTokTile) + r) >> 1;        // tiles start on even tokens
      const int64_t first = p.first_entry ? (int64_t)p.first_entry[b] : 0;
      const bool seq_ok = first >= 0 && first + n_pairs <= p.max_entries;
      if (!seq_ok && tile == 0 && half == 0 && r == 0) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_PROJECT, (uint32_t)b);
      const bool store = seq_ok && pair < n_pairs;
      const int64_t e = first + pair;
      uint8_t* blk = p.cache + b * p.cache_stride_b + (e / kBlockEntries) * (int64_t)block_bytes(kLatent);
      const int slot = (int)(e % kBlockEntries);
#pragma unroll 1
      for (int c = 0; c < kNHalf / 32; ++c) {
        uint32_t x[32];
        tc::ld_32x32(tbase + acc * kTmemCols + lane_base + 32 * c, x);
        tc::wait_ld();
        // the even lane of a pair takes columns 0-15 of the chunk, the odd lane columns 16-31; each sends
        // the other its copy of the partner's group: m = fl32(fl32(x_2i + x_2i+1) * 0.5)
        float m[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float give = __uint_as_float(odd ? x[i] : x[16 + i]);
          const float recv = __shfl_xor_sync(0xffffffffu, give, 1);
          const float own = __uint_as_float(odd ? x[16 + i] : x[i]);
          m[i] = __fmul_rn(odd ? __fadd_rn(recv, own) : __fadd_rn(own, recv), 0.5f);
        }
        float amax = 0.0f;
#pragma unroll
        for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(m[k]));
        const float sf = __fdiv_rn(amax, 6.0f);
        uint32_t sbyte = 0;
        float sv = 0.0f;
        if (sf > 0.0f) {
          if (p.scale_rule == CSA_SCALE_AMAX) {
            sbyte = float_to_e4m3_satfinite(sf);
            sv = e4m3_to_float(sbyte);
          } else {
            sbyte = pow2_scale(sf, &sv);
          }
        }
        uint32_t codes[2] = {0u, 0u};                            // 8 code bytes, low nibble first
        if (sv > 0.0f) {
#pragma unroll
          for (int k = 0; k < 16; ++k) codes[k / 8] |= e2m1_code(__fdiv_rn(m[k], sv)) << (4 * (k % 8));
        }
        if (store) {
          const int g = kNHalf / kGroup * half + 2 * c + (odd ? 1 : 0);
          *reinterpret_cast<uint2*>(blk + slot * (kLatent / 2) + g * 8) = make_uint2(codes[0], codes[1]);
          blk[kBlockEntries * (kLatent / 2) + slot * (kLatent / kGroup) + g] = (uint8_t)sbyte;
        }
      }
      // this accumulator may take item j + 2 (every tensor-memory load above has completed)
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::dealloc(tbase, 2 * kTmemCols);
}

}  // namespace

cudaError_t launch_project_pack(const ProjectParams& p, cudaStream_t s) {
  const int64_t n_pairs = p.n_tokens / 2;
  if (p.batch == 0 || n_pairs == 0) return cudaSuccess;
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  // hidden rows as [batch][n_tokens][hidden] bf16 in [1 x 128 x 64] boxes; rows past n_tokens read as zero
  CUtensorMap h_map, w_map;
  std::memset(&h_map, 0, sizeof(h_map));
  std::memset(&w_map, 0, sizeof(w_map));
  {
    const int64_t seq_stride = p.batch > 1 ? p.h_stride_b : p.n_tokens * p.h_stride_t;
    const cuuint64_t dims[3] = {(cuuint64_t)p.hidden, (cuuint64_t)p.n_tokens, (cuuint64_t)p.batch};
    const cuuint64_t strides[2] = {(cuuint64_t)p.h_stride_t * 2, (cuuint64_t)seq_stride * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kKStep, (cuuint32_t)kTokTile, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&h_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(p.h), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)p.hidden, (cuuint64_t)kLatent};
    const cuuint64_t strides[1] = {(cuuint64_t)p.hidden * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kKStep, (cuuint32_t)kNHalf};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(p.w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  ProfScope prof("project_pack", s);
  clear_stale_error();
  cudaError_t e = ensure_smem_limit(project_pack_kernel, kSmem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (2 * n_pairs + kTokTile - 1) / kTokTile;
  // persistent: one CTA per SM (even), each looping over (token tile, column half) items
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int64_t items = 2 * tiles * p.batch;
  int64_t grid = (int64_t)(sms & ~1);
  if (grid > items) grid = items;
  if (grid < 1) grid = 1;
  // (a programmatic dependent: the kernel waits before its first global access)
  return launch_ex(project_pack_kernel, dim3((unsigned)grid), dim3(kThreads), (size_t)kSmem, s, true, p, tiles, h_map,
                   w_map);
}

}  // namespace csa
