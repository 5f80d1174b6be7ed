// Indexer: block-scaled FP4 products of the index keys with the indexer queries on the fifth-generation
// tensor cores (tcgen05.mma kind::mxf4nvf4), the weighted ReLU head sum, the causal mask and the maximum
// over each block of 8 entries; plus the super-block scores of the hierarchical stage.
//
// Follows "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (card), Key ideas: layers
// "rescore with [their] own indexer query" and select "blocks of 8"; "a hierarchical sparse indexer (up
// to 2,048 blocks of 8 positions) trims decoder indexing". The score function, the FP4 formats and the
// super-block shape are this library's readings, stated in include/csa.h.
//
// Design. The index keys are stored as E2M1 codes with one E4M3 scale per 16 elements, which is exactly
// the operand format of the block-scaled FP4 MMA, so the keys are never dequantised: a tensor-map copy
// streams each stage of 16 blocks (128 entries) into shared memory in the swizzled K-major layout the MMA
// reads, and the 128 entries are the M side of one product. The queries of one unit (a group of query
// positions of one sequence, all indexer heads) are rounded to the same FP4 format with power-of-two
// scales (exact for integer values in [-4, 4]) and form the N side. Each product lands in tensor memory;
// four epilogue warps (thread = entry) write the keys' scale factors into tensor memory before the product
// (as soon as a stage's copy has landed, between the epilogues of earlier stages) and afterwards apply ReLU, the head weights, the ordered head sum and the causal mask, and take the block
// maximum across the 8 lanes that hold one block. The accumulator is double-buffered so that the epilogue
// of one stage overlaps the product of the next, and the copy warp starts the first stages before the
// queries are prepared.
#include <cuda.h>

#include <cstring>

#include "csa_internal.cuh"
#include "tc.cuh"

namespace csa {
namespace {

constexpr int kStageBlocks = 16;
constexpr int kStageRows = kStageBlocks * kBlockEntries;     // 128 = M of the product
constexpr int kThreads = 192;                                 // warp 0 copies, 1 MMA, 2-5 scales + epilogue

template <int DI, int N>
struct Cfg {
  static constexpr int kRowCodes = DI / 2;
  static constexpr int kRowScales = DI / kGroup;
  static constexpr int kMmas = DI / 64;                       // K = 64 elements per block-scaled MMA
  static constexpr int kCodesStage = kStageRows * kRowCodes;
  static constexpr int kScalesStage = kStageRows * kRowScales;
  static constexpr uint32_t kSwizzle = DI == 64 ? 6u : (DI == 128 ? 4u : 2u);   // 32, 64, 128-byte swizzle
  static constexpr int kSwzShift = DI == 64 ? 2 : (DI == 128 ? 1 : 0);
  static constexpr int kSwzMask = DI == 64 ? 1 : (DI == 128 ? 3 : 7);
  static constexpr uint32_t kSbo = 8 * kRowCodes;
  // copy stages in flight: five at dim 128 (9,216 B each), so that four CTAs fit in one SM's shared memory
  static constexpr int kStages = DI == 128 ? 5 : 6;
  // shared memory (bytes)
  static constexpr int kCodesOff = 0;
  static constexpr int kScalesOff = kCodesOff + kStages * kCodesStage;
  static constexpr int kQOff = kScalesOff + kStages * kScalesStage;                // N rows of query codes
  static constexpr int kQScOff = kQOff + N * kRowCodes;                            // N x DI/16 query scales
  static constexpr int kPosOff = (kQScOff + N * kRowScales + 7) & ~7;             // NQ query positions
  static constexpr int kBarOff = (kPosOff + 4 * N + 7) & ~7;
  static constexpr int kSmem = kBarOff + (3 * kStages + 2 * 4 + 2) * 8 + 16;
  // pipeline depth in tensor memory: accumulator buffers and key-scale buffers (scales are written two
  // stages ahead of the product that reads them)
  static constexpr int kND = N <= 16 ? 4 : 2;
  static constexpr int kNSF = 4;
  // tensor memory columns
  static constexpr uint32_t kColD = 0;                              // kND x N
  static constexpr uint32_t kColSFA = kND * N;                      // kNSF x (4 per MMA)
  static constexpr uint32_t kColSFB = kColSFA + kNSF * 4 * kMmas;   // 4 per MMA
  static constexpr uint32_t kColsUsed = kColSFB + 4 * kMmas;
  static constexpr uint32_t kTmemCols = kColsUsed <= 32 ? 32 : (kColsUsed <= 64 ? 64 : (kColsUsed <= 128 ? 128 : (kColsUsed <= 256 ? 256 : 512)));
};

// Instruction descriptor of kind::mxf4nvf4: E2M1 A and B, UE4M3 scale factors, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc) : "memory");
}

__device__ __forceinline__ void st_32x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" :: "r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void ld_32x16(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w, uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
               " [%0], [%1, {%2, %3, %4, %5}], [%6];"
               :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w),
                  "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
               " [%0], [%1, {%2, %3, %4}], [%5];"
               :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
                  "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint32_t* hdr) {
  const uint32_t a = smem_addr(bar);
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 7u) == 7u && *abort_flag) return false;
  }
  *abort_flag = 1;
  report(hdr, CSA_ERR_TIMEOUT, KID_INDEX_SCORE, blockIdx.x);
  return false;
}

__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(a, parity)) return;
  }
}

// The FP4 rounding of 16 query values that both sides of the indexer use: power-of-two scale (the
// POW2 rule of the cache), E2M1 codes. Returns the scale byte; codes are packed two per byte.
__device__ __forceinline__ uint32_t quantize16_pow2(const float* v, uint32_t* lo, uint32_t* hi) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const float sf = __fdiv_rn(amax, 6.0f);
  uint32_t sbyte = 0;
  float s = 0.0f;
  if (sf > 0.0f) sbyte = pow2_scale(sf, &s);
  *lo = 0;
  *hi = 0;
  if (s > 0.0f) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t byte = e2m1_code(__fdiv_rn(v[2 * j], s)) | (e2m1_code(__fdiv_rn(v[2 * j + 1], s)) << 4);
      if (j < 4) *lo |= byte << (8 * j); else *hi |= byte << (8 * (j - 4));
    }
  }
  return sbyte;
}

struct IdxUnit {
  int64_t b, j0, row0, n_e, n_b;
  int nq;              // valid queries of the unit
};

template <int DI, int HI, int N>
__global__ void __launch_bounds__(kThreads, 1)
index_tc_kernel(const ScoreParams p, int64_t stages_per_unit, int splits, int groups_per_seq,
                const __grid_constant__ CUtensorMap codes_map, const __grid_constant__ CUtensorMap scales_map) {
  using C = Cfg<DI, N>;
  constexpr int NQ = N / HI;                    // query slots of the unit (columns n = q * HI + h)
  constexpr uint32_t kIdesc = idesc_mxf4(kStageRows, N);
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + C::kStages;
  uint64_t* sfr = empty + C::kStages;
  uint64_t* dfull = sfr + C::kStages;              // [kND]
  uint64_t* dempty = dfull + 4;                 // [kND]
  uint64_t* fin = dempty + 4;                   // [1]
  uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(fin + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_ptr + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Barriers and tensor memory touch no global memory. With a few query columns (decode) they are set up
  // before the wait on the kernel before, so that they overlap its end; with many (prefill) the wait comes
  // first (setting up first slowed prefill, measured).
  auto setup = [&]() {
    if (warp == 1) tc::alloc(tmem_ptr, C::kTmemCols);
    if (tid == 0) {
      for (int i = 0; i < C::kStages; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); mbar_init(&sfr[i], 4); }
      for (int i = 0; i < C::kND; ++i) { mbar_init(&dfull[i], 1); mbar_init(&dempty[i], 4); }
      mbar_init(fin, 1);
      fence_mbar_init();
      *abort_flag = 0;
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
  };
  if constexpr (N <= 16) setup();
  griddep_wait();                                  // (hierarchical) the kept super-blocks come from the kernel before
  griddep_launch();
  if constexpr (N > 16) setup();
  const bool hier = p.kept != nullptr;
  const int64_t unit = blockIdx.y;
  IdxUnit u;
  if (hier) {
    u.b = unit / p.n_query; u.j0 = unit % p.n_query; u.nq = 1; u.row0 = unit;
  } else {
    u.b = unit / groups_per_seq; u.j0 = (unit % groups_per_seq) * NQ;
    u.nq = (int)(p.n_query - u.j0 < NQ ? p.n_query - u.j0 : NQ);
    u.row0 = u.b * p.n_query + u.j0;
  }
  int64_t n_e = p.n_entries[u.b];
  if (n_e < 0 || n_e > p.max_entries) {
    if (tid == 0 && blockIdx.x == 0) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_INDEX_SCORE, (uint32_t)u.b);
    n_e = n_e < 0 ? 0 : p.max_entries;
  }
  u.n_e = n_e;
  u.n_b = (n_e + kBlockEntries - 1) / kBlockEntries;
  const int64_t k0 = stages_per_unit * blockIdx.x / splits;
  const int64_t k1 = stages_per_unit * (blockIdx.x + 1) / splits;
  const int n = (int)(k1 - k0);

  // ---------------- the copies start while the other warps prepare the unit's FP4 queries ----------------
  const uint32_t tbase = *tmem_ptr;
  const uint32_t s_base = smem_addr(smem);
  if (warp == 0) {
    // ---------------- tensor-map copies of the key stages ----------------
    if (lane == 0) {
      int issued = 0;
      for (int k = 0; k < n; ++k) {
        const int slot = k % C::kStages;
        if (k >= C::kStages && !wait_or_abort(&empty[slot], ((k / C::kStages) - 1) & 1, abort_flag, p.hdr)) break;
        const int64_t st = k0 + k;
        int64_t id0 = st * kStageBlocks;
        if (hier) {
          const int32_t g = p.kept[unit * p.keep_super + (st >> 2)];
          id0 = g < 0 ? -1 : (int64_t)g * kSuper + (st & 3) * kStageBlocks;
        }
        if (id0 >= 0 && id0 < u.n_b) {
          mbar_arrive_expect_tx(&full[slot], C::kCodesStage + C::kScalesStage);
          tma_load_4d(smem + C::kCodesOff + slot * C::kCodesStage, &codes_map, 0, 0, (int)id0, (int)u.b, &full[slot]);
          tma_load_3d(smem + C::kScalesOff + slot * C::kScalesStage, &scales_map, 0, (int)id0, (int)u.b, &full[slot]);
        } else {
          mbar_arrive(&full[slot]);
        }
        ++issued;
      }
      for (int k = issued - C::kStages < 0 ? 0 : issued - C::kStages; k < issued; ++k)
        drain(&full[k % C::kStages], (k / C::kStages) & 1);
    }
  } else {
  constexpr int kSetupThreads = kThreads - 32;
  const int qt = tid - 32;
  uint8_t* qcodes = smem + C::kQOff;
  uint8_t* qsc = smem + C::kQScOff;
  int32_t* pos_sh = reinterpret_cast<int32_t*>(smem + C::kPosOff);
  for (int q = qt; q < NQ; q += kSetupThreads)
    pos_sh[q] = (p.q_pos != nullptr && q < u.nq) ? __ldg(p.q_pos + u.b * p.n_query + u.j0 + q) : INT32_MAX;
  for (int t = qt; t < N * C::kRowScales; t += kSetupThreads) {
    const int row = t / C::kRowScales, g = t % C::kRowScales;       // row = q * HI + h
    const int q = row / HI, h = row % HI;
    float v[16];
    const bool have = q < u.nq && h < HI;
    const float* src = p.q_idx + ((u.b * p.n_query + u.j0 + q) * HI + h) * (int64_t)DI + g * 16;
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = have ? __ldg(src + j) : 0.0f;
    uint32_t lo, hi;
    const uint32_t sb = quantize16_pow2(v, &lo, &hi);
    const int chunk = (g * 8) >> 4, within = (g * 8) & 15;
    uint8_t* dst = qcodes + row * C::kRowCodes + ((chunk ^ ((row >> C::kSwzShift) & C::kSwzMask)) << 4) + within;
    *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
    qsc[row * C::kRowScales + g] = (uint8_t)sb;
  }
  tc::fence_proxy_async();
  asm volatile("bar.sync 1, %0;" :: "n"(kSetupThreads) : "memory");

  if (warp >= 2) {
    // query scale factors: column n at lane 32 j + n % 32, column kColSFB + 4 s + n / 32, for every
    // subpartition j (each epilogue warp writes its own copy)
    const int sp = warp & 3;
    const uint32_t lane_base = (uint32_t)(sp * 32) << 16;
#pragma unroll
    for (int s = 0; s < C::kMmas; ++s) {
#pragma unroll
      for (int c = 0; c < (N + 31) / 32; ++c) {
        const int nn = lane + 32 * c;
        uint32_t w = 0;
        if (nn < N) w = *reinterpret_cast<const uint32_t*>(qsc + nn * C::kRowScales + 4 * s);
        st_32x1(tbase + lane_base + C::kColSFB + 4 * s + c, w);
      }
    }
    tc::wait_st();
  }
  tc::fence_before();
  asm volatile("bar.sync 1, %0;" :: "n"(kSetupThreads) : "memory");
  tc::fence_after();

  if (warp == 1) {
    // ---------------- products ----------------
    if (lane == 0) {
      for (int k = 0; k < n; ++k) {
        const int slot = k % C::kStages, db = k % C::kND, sb = k % C::kNSF;
        if (!wait_or_abort(&sfr[slot], (k / C::kStages) & 1, abort_flag, p.hdr)) break;
        if (k >= C::kND && !wait_or_abort(&dempty[db], ((k / C::kND) - 1) & 1, abort_flag, p.hdr)) break;
        tc::fence_after();
        const uint32_t a0 = s_base + C::kCodesOff + slot * C::kCodesStage;
        const uint32_t b0 = s_base + C::kQOff;
#pragma unroll
        for (int s = 0; s < C::kMmas; ++s) {
          const uint64_t a = tc::smem_desc(a0 + 32 * s, 16, C::kSbo, C::kSwizzle);
          const uint64_t b = tc::smem_desc(b0 + 32 * s, 16, C::kSbo, C::kSwizzle);
          mma_mxf4(tbase + C::kColD + db * N, a, b, kIdesc, tbase + C::kColSFA + sb * 4 * C::kMmas + 4 * s,
                   tbase + C::kColSFB + 4 * s, s > 0 ? 1u : 0u);
        }
        tc::commit(&empty[slot]);
        tc::commit(&dfull[db]);
      }
      tc::commit(fin);
      drain(fin, 0);
    }
  } else {
    // ---------------- key scale factors and epilogue (thread = entry row of the stage) ----------------
    const int sp = warp & 3;
    const int m = sp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(sp * 32) << 16;
    float w[HI];
#pragma unroll
    for (int h = 0; h < HI; ++h) w[h] = p.head_w ? __ldg(p.head_w + h) : 1.0f;
    // key scale factors of stage k (whose copy has landed) into scale buffer k % kNSF (lane m, column
    // base + 4 s + m / 32)
    auto put_scales = [&](int k) {
      const int slot = k % C::kStages;
      const uint8_t* sc = smem + C::kScalesOff + slot * C::kScalesStage + (m >> 3) * (8 * C::kRowScales) +
                          (m & 7) * C::kRowScales;
#pragma unroll
      for (int s = 0; s < C::kMmas; ++s)
        st_32x1(tbase + lane_base + C::kColSFA + (k % C::kNSF) * 4 * C::kMmas + 4 * s + sp,
                *reinterpret_cast<const uint32_t*>(sc + 4 * s));
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfr[slot]);
    };
    int ks = 0;                                    // the next stage whose scale factors are written
    bool ok = true;
    for (int k = 0; k < n && ok; ++k) {
      const int db = k % C::kND;
      // Until stage k's product is complete, write the scale factors of every stage whose copy has landed and
      // whose scale buffer the products of stage ks - kNSF have finished with (their epilogue has begun), so
      // the products never wait for this loop to come round to them. Both barriers are polled; a round that
      // finds neither ready sleeps briefly.
      uint32_t spins = 0;
      for (;;) {
        if (ks < n && ks < k + C::kNSF &&
            __all_sync(0xffffffffu, mbar_test_wait(smem_addr(&full[ks % C::kStages]), (ks / C::kStages) & 1))) {
          put_scales(ks++);
          continue;
        }
        if (ks > k && __all_sync(0xffffffffu, mbar_test_wait(smem_addr(&dfull[db]), (k / C::kND) & 1))) break;
        if (++spins >= kSpinLimit * 8u) {
          if (lane == 0) {
            *abort_flag = 1;
            report(p.hdr, CSA_ERR_TIMEOUT, KID_INDEX_SCORE, blockIdx.x);
          }
          ok = false;
          break;
        }
        if ((spins & 7u) == 7u && __any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
        __nanosleep(32);
      }
      if (!ok) break;
      tc::fence_after();
      const int64_t st = k0 + k;
      const int64_t slot0 = st * kStageBlocks;
      int64_t id0 = slot0;
      if (hier) {
        const int32_t g = p.kept[unit * p.keep_super + (st >> 2)];
        id0 = g < 0 ? -1 : (int64_t)g * kSuper + (st & 3) * kStageBlocks;
      }
      const int64_t blk = id0 + (m >> 3);
      const int64_t e = blk * kBlockEntries + (m & 7);
      const bool row_ok = id0 >= 0 && blk < u.n_b && e < u.n_e;
      const int64_t slot = slot0 + (m >> 3);
      if constexpr (NQ >= 8) {
        // Many positions per unit: all N columns in one round of loads, then the block maximum of every
        // position at once by a transposing reduction over the 8 lanes of a block. At the step with offset
        // o a lane keeps the half of its positions selected by (lane & o) and takes the maximum with its
        // partner's copy of that half; after offsets 1, 2, 4, lane j of a block holds positions
        // (j & 1) NQ/2 + (j >> 1 & 1) NQ/4 + (j >> 2) NQ/8 + i, i < NQ/8. The maximum is exact, so the result
        // equals the per-position shuffles of the path below.
        uint32_t r[N];
#pragma unroll
        for (int c0 = 0; c0 < N; c0 += 16) ld_32x16(tbase + lane_base + C::kColD + db * N + c0, r + c0);
        tc::wait_ld();
        float v[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          float sum = 0.0f;
#pragma unroll
          for (int h = 0; h < HI; ++h) {
            const float dot = __uint_as_float(r[q * HI + h]);
            const float t = __fmul_rn(w[h], p.relu ? fmaxf(dot, 0.0f) : dot);
            sum = h == 0 ? t : __fadd_rn(sum, t);
          }
          const bool okq = row_ok && q < u.nq && 2 * e + 1 <= (int64_t)pos_sh[q];
          v[q] = okq ? __fadd_rn(sum, 0.0f) : -INFINITY;
        }
#pragma unroll
        for (int o = 1, n = NQ / 2; o <= 4; o <<= 1, n >>= 1) {
          const bool up = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < n; ++i) {
            const float keep = up ? v[n + i] : v[i];
            const float give = up ? v[i] : v[n + i];
            v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, o));
          }
        }
        const int j = lane & 7;
        const int qb = (j & 1) * (NQ / 2) + ((j >> 1) & 1) * (NQ / 4) + (j >> 2) * (NQ / 8);
        if (slot < p.n_slots) {
#pragma unroll
          for (int i = 0; i < NQ / 8; ++i) {
            const int q = qb + i;
            if (q < u.nq) p.scores[(u.row0 + q) * p.score_stride + slot] = v[i];
          }
        }
      } else {
#pragma unroll
        for (int c0 = 0; c0 < N; c0 += 16) {
          if (c0 >= u.nq * HI) break;
          uint32_t r[16];
          ld_32x16(tbase + lane_base + C::kColD + db * N + c0, r);
          tc::wait_ld();
#pragma unroll
          for (int qq = 0; qq < 16 / HI; ++qq) {
            const int q = c0 / HI + qq;
            if (q >= NQ || q >= u.nq) break;
            float sum = 0.0f;
#pragma unroll
            for (int h = 0; h < HI; ++h) {
              const float dot = __uint_as_float(r[qq * HI + h]);
              const float t = __fmul_rn(w[h], p.relu ? fmaxf(dot, 0.0f) : dot);
              sum = h == 0 ? t : __fadd_rn(sum, t);
            }
            const bool okq = row_ok && 2 * e + 1 <= (int64_t)pos_sh[q];
            float mx = okq ? __fadd_rn(sum, 0.0f) : -INFINITY;
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            if ((lane & 7) == 0 && slot < p.n_slots) {
              const int64_t row = hier ? u.row0 : u.row0 + q;
              p.scores[row * p.score_stride + slot] = mx;
            }
          }
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dempty[db]);
    }
  }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::dealloc(tbase, C::kTmemCols);
}

// Super-block scores. A CTA takes one unit and kCoarsePerCta super-blocks: it rounds the unit's queries
// to FP4 once (16-element groups, power-of-two scales: the rounding the block products use) into shared
// memory, then each warp scores its super-blocks with lanes over the feature index (per-lane fused
// multiply-adds in feature order, then a butterfly sum), the ReLU, the head weights and the ordered head
// sum. Two super-blocks a warp: with a few queries (the 1M decode has 4 x 1,024 super-blocks) more CTAs
// spread the latency-bound scoring over the SMs (16.1 -> 11.1 us against eight a warp).
constexpr int kCoarsePerWarp = 2;
constexpr int kCoarsePerCta = 8 * kCoarsePerWarp;

__global__ void __launch_bounds__(256) coarse_score_kernel(CoarseScoreParams p) {
  extern __shared__ float xq_sh[];                 // [heads][dim]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  griddep_wait();
  griddep_launch();
  const int64_t unit = blockIdx.y;
  const int64_t b = unit / p.n_query;
  const int64_t n_e = p.n_entries[b];
  const int groups = p.heads * p.dim / 16;
  for (int t = threadIdx.x; t < groups; t += blockDim.x) {
    const float* src = p.q_idx + unit * p.heads * (int64_t)p.dim + t * 16;
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __ldg(src + j);
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
    const float sf = __fdiv_rn(amax, 6.0f);
    float sc = 0.0f;
    if (sf > 0.0f) pow2_scale(sf, &sc);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float xq = 0.0f;
      if (sc > 0.0f) {
        const uint32_t h2 = e2m1x2_to_f16x2(e2m1_code(__fdiv_rn(v[j], sc)));
        xq = __fmul_rn(__half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))), sc);
      }
      xq_sh[t * 16 + j] = xq;
    }
  }
  __syncthreads();
  for (int j = 0; j < kCoarsePerWarp; ++j) {
    const int64_t g = (int64_t)blockIdx.x * kCoarsePerCta + warp * kCoarsePerWarp + j;
    if (g >= p.n_super) break;
    float* dst = p.scores + unit * p.n_super + g;
    if (g * (int64_t)kSuper * kBlockEntries >= n_e) {
      if (lane == 0) *dst = -INFINITY;
      continue;
    }
    const float* crow = p.coarse + b * p.coarse_stride_b + g * p.dim;
    float c[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) c[k] = 32 * k < p.dim ? __ldg(crow + 32 * k + lane) : 0.0f;
    float s = 0.0f;
    for (int h = 0; h < p.heads; ++h) {
      const float* xq = xq_sh + h * p.dim;
      float d = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (32 * k < p.dim) d = fmaf(xq[32 * k + lane], c[k], d);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
      if (p.relu) d = fmaxf(d, 0.0f);
      const float wgt = p.head_w ? __ldg(p.head_w + h) : 1.0f;
      const float t = __fmul_rn(wgt, d);
      s = (h == 0) ? t : __fadd_rn(s, t);
    }
    if (lane == 0) *dst = __fadd_rn(s, 0.0f);
  }
}

template <int DI, int HI, int N>
cudaError_t launch_tc(const ScoreParams& p, int num_sms, cudaStream_t s, bool pdl) {
  using C = Cfg<DI, N>;
  constexpr int NQ = N / HI;
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const int64_t n_b_cap = (p.max_entries + kBlockEntries - 1) / kBlockEntries;
  const int64_t bb = block_bytes(DI);
  const int64_t seq_stride = p.batch > 1 ? p.keys_stride_b : n_b_cap * bb;
  CUtensorMap codes_map, scales_map;
  {
    const cuuint64_t dims[4] = {(cuuint64_t)(DI / 2), 8, (cuuint64_t)n_b_cap, (cuuint64_t)p.batch};
    const cuuint64_t strides[3] = {(cuuint64_t)(DI / 2), (cuuint64_t)bb, (cuuint64_t)seq_stride};
    const cuuint32_t box[4] = {(cuuint32_t)(DI / 2), 8, (cuuint32_t)kStageBlocks, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle swz = DI == 64 ? CU_TENSOR_MAP_SWIZZLE_32B
                                            : (DI == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
    if (enc(&codes_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(p.keys), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)(DI / 2), (cuuint64_t)n_b_cap, (cuuint64_t)p.batch};
    const cuuint64_t strides[2] = {(cuuint64_t)bb, (cuuint64_t)seq_stride};
    const cuuint32_t box[3] = {(cuuint32_t)(DI / 2), (cuuint32_t)kStageBlocks, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&scales_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(p.keys) + kBlockEntries * (DI / 2), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const bool hier = p.kept != nullptr;
  const int groups_per_seq = hier ? 1 : (int)((p.n_query + NQ - 1) / NQ);
  const int64_t units = hier ? p.batch * p.n_query : p.batch * groups_per_seq;
  const int64_t spu = (p.n_slots + kStageBlocks - 1) / kStageBlocks;
  // one wave: as many CTAs per SM as shared memory, registers and tensor memory let stay resident (at most 4),
  // each with a contiguous range of one unit's stages
  if (units > 65535) return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem_limit(index_tc_kernel<DI, HI, N>, C::kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, smem_sm = 0, reserved = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess) return e;
  const int by_smem = smem_sm / (C::kSmem + reserved);
  int per_sm = (int)(512 / C::kTmemCols) < 4 ? (int)(512 / C::kTmemCols) : 4;
  if (by_smem < per_sm) per_sm = by_smem < 1 ? 1 : by_smem;
  int64_t splits = (int64_t)num_sms * per_sm / units;
  if (splits > spu) splits = spu;
  if (splits < 1) splits = 1;
  clear_stale_error();
  const dim3 grid((unsigned)splits, (unsigned)units);
  return launch_ex(index_tc_kernel<DI, HI, N>, grid, dim3(kThreads), (size_t)C::kSmem, s, pdl, p, spu, (int)splits,
                   groups_per_seq, codes_map, scales_map);
}

template <int DI, int HI>
cudaError_t launch_h(const ScoreParams& p, int num_sms, cudaStream_t s, bool pdl) {
  // one unit per query group that fits 16 columns (decode), else 64 columns (64 / HI query positions)
  if (p.kept != nullptr || p.n_query * HI <= 16) return launch_tc<DI, HI, 16>(p, num_sms, s, pdl);
  return launch_tc<DI, HI, 64>(p, num_sms, s, pdl);
}

template <int DI>
cudaError_t launch_d(const ScoreParams& p, int num_sms, cudaStream_t s, bool pdl) {
  switch (p.heads) {
    case 1: return launch_h<DI, 1>(p, num_sms, s, pdl);
    case 2: return launch_h<DI, 2>(p, num_sms, s, pdl);
    case 4: return launch_h<DI, 4>(p, num_sms, s, pdl);
    case 8: return launch_h<DI, 8>(p, num_sms, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_index_score(const ScoreParams& p, int num_sms, cudaStream_t s, bool pdl) {
  if (p.n_slots == 0) return cudaSuccess;
  ProfScope prof(p.kept ? "index_score_hier" : "index_score", s);
  switch (p.dim) {
    case 64: return launch_d<64>(p, num_sms, s, pdl);
    case 128: return launch_d<128>(p, num_sms, s, pdl);
    case 256: return launch_d<256>(p, num_sms, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_coarse_score(const CoarseScoreParams& p, cudaStream_t s, bool pdl) {
  const int64_t units = p.batch * p.n_query;
  if (units == 0 || p.n_super == 0) return cudaSuccess;
  if (units > 65535 || p.dim > 256) return cudaErrorInvalidValue;
  ProfScope prof("coarse_score", s);
  clear_stale_error();
  const dim3 grid((unsigned)((p.n_super + kCoarsePerCta - 1) / kCoarsePerCta), (unsigned)units);
  return launch_ex(coarse_score_kernel, grid, dim3(256), (size_t)p.heads * p.dim * sizeof(float), s, pdl, p);
}

}  // namespace csa
