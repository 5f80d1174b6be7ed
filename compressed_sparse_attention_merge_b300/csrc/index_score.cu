// Indexer: entry scores against the FP4 index keys, weighted ReLU head sum, and the warp-level max over
// each block of 8 entries.
//
// Follows "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (card), Key ideas: layers
// "rescore with [their] own indexer query" and select "blocks of 8"; "a hierarchical sparse indexer (up
// to 2,048 blocks of 8 positions) trims decoder indexing". The score function, the key format and the
// super-block shape are this library's readings, stated in include/csa.h.
//
// Design. The key stream is the HBM term, so the kernel reads every key byte once with coalesced
// 128-bit loads straight into registers and never stages it. A warp handles a tile of two blocks (16
// entries); the 16 x dim key tile is the A operand of mma.sync m16n8k16 (f16 in, f32 accumulate) with
// the entries as rows. Each A register is one code byte converted by cvt.rn.f16x2.e2m1x2 and multiplied
// by its f16 scale; this is exact, and because the dot product does not depend on the order of the
// feature index the kernel feeds every lane its own contiguous slice of a key row and permutes the query
// features the same way. The 8 MMA columns hold (query, head) pairs. Integer-valued inputs make every
// product and partial sum an integer below 2^24, so scores are exact.
// The epilogue applies ReLU and the head weights, sums the heads in a fixed order across the owning
// lanes, masks ineligible entries to -inf and takes the block max with three xor-shuffles over the 8
// lanes that hold one block's rows.
#include "csa_internal.cuh"

namespace csa {
namespace {

__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int DI>
struct RowRaw {
  static constexpr int kWords = DI / 32;     // DI/8 code bytes per lane per row
  uint32_t code[kWords];
  uint32_t scale;                             // DI/64 scale bytes, little-endian
};

template <int DI>
__device__ __forceinline__ void load_row(const uint8_t* blk, int r, int c, RowRaw<DI>& out) {
  constexpr int BPL = DI / 8, GPL = DI / 64;
  const uint8_t* cp = blk + r * (DI / 2) + c * BPL;
  if constexpr (BPL == 8) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(cp));
    out.code[0] = v.x; out.code[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < BPL / 16; ++i) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(cp) + i);
      out.code[4 * i] = v.x; out.code[4 * i + 1] = v.y; out.code[4 * i + 2] = v.z; out.code[4 * i + 3] = v.w;
    }
  }
  const uint8_t* sp = blk + kBlockEntries * (DI / 2) + r * (DI / 16) + c * GPL;
  if constexpr (GPL == 1) out.scale = __ldg(sp);
  else if constexpr (GPL == 2) out.scale = __ldg(reinterpret_cast<const unsigned short*>(sp));
  else out.scale = __ldg(reinterpret_cast<const unsigned int*>(sp));
}

template <int DI>
__device__ __forceinline__ void zero_row(RowRaw<DI>& out) {
#pragma unroll
  for (int i = 0; i < RowRaw<DI>::kWords; ++i) out.code[i] = 0u;
  out.scale = 0u;
}

// A fragment registers (rows r and r+8) for k-step kk from the raw bytes of the lane's slice.
template <int DI>
__device__ __forceinline__ void a_frag(const RowRaw<DI>& ra, const RowRaw<DI>& rb, const uint32_t* sa,
                                       const uint32_t* sb, int kk, uint32_t* a) {
  const int byte = 2 * kk;
  const uint32_t wa = ra.code[byte >> 2], wb = rb.code[byte >> 2];
  const int sh = (byte & 3) * 8;
  const int grp = kk >> 2;
  a[0] = hmul2_u32(e2m1x2_to_f16x2((wa >> sh) & 0xFFu), sa[grp]);
  a[1] = hmul2_u32(e2m1x2_to_f16x2((wb >> sh) & 0xFFu), sb[grp]);
  a[2] = hmul2_u32(e2m1x2_to_f16x2((wa >> (sh + 8)) & 0xFFu), sa[grp]);
  a[3] = hmul2_u32(e2m1x2_to_f16x2((wb >> (sh + 8)) & 0xFFu), sb[grp]);
}

// Query fragments (B operand) for the lane's column n = lane / 4: query jq, head n % HI.
template <int DI, int HI>
__device__ __forceinline__ void load_qfrag(const ScoreParams& p, int64_t b, int64_t jq, int lane,
                                           uint32_t (*bq)[2]) {
  constexpr int KS = DI / 16;
  const int n = lane >> 2, c = lane & 3;
  const int h = n % HI;
  if (jq >= p.n_query) {
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) { bq[kk][0] = 0u; bq[kk][1] = 0u; }
    return;
  }
  const float* qrow = p.q_idx + ((b * p.n_query + jq) * HI + h) * (int64_t)DI + c * (DI / 4);
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(qrow) + kk);
    bq[kk][0] = pack_half2(f.x, f.y);
    bq[kk][1] = pack_half2(f.z, f.w);
  }
}

template <int DI, int HI>
__global__ void __launch_bounds__(256) index_score_kernel(ScoreParams p) {
  constexpr int KS = DI / 16;
  constexpr int GPL = DI / 64;
  constexpr int BB = block_bytes(DI);
  constexpr int QPM = HI >= 8 ? 1 : 8 / HI;     // queries per MMA
  constexpr int LPQ = HI >= 2 ? HI / 2 : 1;     // lanes holding one query's heads
  constexpr int QPL = HI == 1 ? 2 : 1;          // queries held by one lane

  const int lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  const bool hier = p.kept != nullptr;
  const int64_t unit = blockIdx.y;              // hierarchical: (b, j); flat: b
  const int64_t b = hier ? unit / p.n_query : unit;
  const int64_t jq_fixed = hier ? unit % p.n_query : 0;

  int64_t n_e = p.n_entries[b];
  if (n_e < 0 || n_e > p.max_entries) {
    if (threadIdx.x == 0 && blockIdx.x == 0) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_INDEX_SCORE, (uint32_t)b);
    n_e = n_e < 0 ? 0 : p.max_entries;
  }
  const int64_t n_b = (n_e + kBlockEntries - 1) / kBlockEntries;
  const uint8_t* seq = p.keys + b * p.keys_stride_b;

  // head weights for the lane's two columns
  float w0 = 1.0f, w1 = 1.0f;
  if (p.head_w) { w0 = __ldg(p.head_w + (2 * c) % HI); w1 = __ldg(p.head_w + (2 * c + 1) % HI); }

  const int64_t n_qg = hier ? 1 : (p.n_query + QPM - 1) / QPM;
  uint32_t bq[KS][2];
  if (n_qg == 1) load_qfrag<DI, HI>(p, b, hier ? jq_fixed : (int64_t)(r / HI), lane, bq);

  const int64_t tiles = (p.n_slots + 1) / 2;
  const int64_t warp0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);

  for (int64_t t = warp0; t < tiles; t += wstride) {
    // ---- block ids of the tile's two slots
    int64_t blk[2];
    bool ok[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int64_t slot = 2 * t + i;
      int64_t id = -1;
      if (slot < p.n_slots) {
        if (hier) {
          const int32_t g = p.kept[unit * p.keep_super + slot / kSuper];
          id = g < 0 ? -1 : (int64_t)g * kSuper + slot % kSuper;
        } else {
          id = slot;
        }
      }
      blk[i] = id;
      ok[i] = id >= 0 && id < n_b;
    }
    if (!ok[0] && !ok[1]) {
      // nothing eligible: both slots are non-candidates for every query
      const int64_t rows = hier ? 1 : p.n_query;
      for (int64_t j = lane; j < rows; j += 32) {
        const int64_t row = hier ? unit : b * p.n_query + j;
#pragma unroll
        for (int i = 0; i < 2; ++i)
          if (2 * t + i < p.n_slots) p.scores[row * p.score_stride + 2 * t + i] = -INFINITY;
      }
      continue;
    }

    // ---- raw key bytes for rows r (block 0) and r (block 1): one 16-byte load per row for DI = 128
    RowRaw<DI> ra, rb;
    if (ok[0]) load_row<DI>(seq + blk[0] * BB, r, c, ra); else zero_row<DI>(ra);
    if (ok[1]) load_row<DI>(seq + blk[1] * BB, r, c, rb); else zero_row<DI>(rb);
    uint32_t sa[GPL], sb[GPL];
#pragma unroll
    for (int gi = 0; gi < GPL; ++gi) {
      sa[gi] = e4m3_to_f16x2_bcast((ra.scale >> (8 * gi)) & 0xFFu);
      sb[gi] = e4m3_to_f16x2_bcast((rb.scale >> (8 * gi)) & 0xFFu);
    }
    uint32_t af[KS][4];
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) a_frag<DI>(ra, rb, sa, sb, kk, af[kk]);

    const int64_t eA = blk[0] * kBlockEntries + r;
    const int64_t eB = blk[1] * kBlockEntries + r;

    for (int64_t qg = 0; qg < n_qg; ++qg) {
      if (n_qg > 1) load_qfrag<DI, HI>(p, b, qg * QPM + r / HI, lane, bq);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) mma16816(acc, af[kk], bq[kk][0], bq[kk][1]);

      // t = w_h * ReLU(dot) per column, rows r (acc0, acc1) and r + 8 (acc2, acc3)
      float tv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float d = p.relu ? fmaxf(acc[i], 0.0f) : acc[i];
        tv[i] = __fmul_rn((i & 1) ? w1 : w0, d);
      }
      // ordered head sums: s[row half][query slot of this lane]
      float s[2][QPL];
      if constexpr (HI == 1) {
        s[0][0] = tv[0]; s[0][1] = tv[1]; s[1][0] = tv[2]; s[1][1] = tv[3];
      } else {
        const int base = (lane & ~3) | (c - c % LPQ);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float acc_s = 0.0f;
#pragma unroll
          for (int i = 0; i < LPQ; ++i) {
            const float x0 = __shfl_sync(0xffffffffu, tv[2 * half], base + i);
            const float x1 = __shfl_sync(0xffffffffu, tv[2 * half + 1], base + i);
            acc_s = (i == 0) ? x0 : __fadd_rn(acc_s, x0);
            acc_s = __fadd_rn(acc_s, x1);
          }
          s[half][0] = acc_s;
        }
      }
      // mask ineligible entries, block max over the 8 lanes sharing c
#pragma unroll
      for (int k = 0; k < QPL; ++k) {
        const int64_t jq = hier ? jq_fixed : qg * QPM + (HI == 1 ? 2 * c + k : c / LPQ);
        int64_t pos = INT64_MAX;
        if (p.q_pos != nullptr && jq < p.n_query) pos = p.q_pos[b * p.n_query + jq];
        const bool vA = ok[0] && eA < n_e && 2 * eA + 1 <= pos;
        const bool vB = ok[1] && eB < n_e && 2 * eB + 1 <= pos;
        float mA = vA ? __fadd_rn(s[0][k], 0.0f) : -INFINITY;
        float mB = vB ? __fadd_rn(s[1][k], 0.0f) : -INFINITY;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, off));
          mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, off));
        }
        const bool owner = (r == 0) && (HI == 1 || c % LPQ == 0) && jq < p.n_query;
        if (owner) {
          const int64_t row = hier ? unit : b * p.n_query + jq;
          float* dst = p.scores + row * p.score_stride;
          if (2 * t < p.n_slots) dst[2 * t] = mA;
          if (2 * t + 1 < p.n_slots) dst[2 * t + 1] = mB;
        }
      }
    }
  }
}

// Super-block scores: one warp per (unit, super-block), lanes over the feature index.
__global__ void __launch_bounds__(256) coarse_score_kernel(CoarseScoreParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t units = p.batch * p.n_query;
  if (gw >= units * p.n_super) return;
  const int64_t unit = gw / p.n_super, g = gw % p.n_super;
  const int64_t b = unit / p.n_query;
  const int64_t n_e = p.n_entries[b];
  float* dst = p.scores + unit * p.n_super + g;
  if (g * (int64_t)kSuper * kBlockEntries >= n_e) {
    if (lane == 0) *dst = -INFINITY;
    return;
  }
  const float* crow = p.coarse + b * p.coarse_stride_b + g * p.dim;
  float s = 0.0f;
  for (int h = 0; h < p.heads; ++h) {
    const float* qrow = p.q_idx + (unit * p.heads + h) * (int64_t)p.dim;
    float d = 0.0f;
    for (int i = lane; i < p.dim; i += 32) d = fmaf(__ldg(qrow + i), __ldg(crow + i), d);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if (p.relu) d = fmaxf(d, 0.0f);
    const float w = p.head_w ? __ldg(p.head_w + h) : 1.0f;
    const float t = __fmul_rn(w, d);
    s = (h == 0) ? t : __fadd_rn(s, t);
  }
  if (lane == 0) *dst = __fadd_rn(s, 0.0f);
}

// ------------------------------------------------------------------------------------------------
// Streaming decode indexer (every unit's queries fit one MMA column group). The keys of all units are
// cut into stages of 16 consecutive blocks; each CTA takes a contiguous range of stages. A producer
// warp copies stages into a ring of shared-memory buffers with cp.async.bulk (one copy per stage: the
// 16 blocks are contiguous in the cache), completing on the stage's "full" mbarrier; each of the 8
// consumer warps takes two blocks of the stage into registers, releases the buffer on its "empty"
// mbarrier and then scores them exactly as the kernel above does. Many stages in flight per SM keep
// the HBM stream busy.
// ------------------------------------------------------------------------------------------------
constexpr int kStageBlocks = 16;
constexpr int kConsumerWarps = kStageBlocks / 2;
constexpr int kStreamThreads = (kConsumerWarps + 1) * 32;

template <int DI>
struct StreamCfg {
  static constexpr int BB = block_bytes(DI);
  static constexpr int stage_bytes = kStageBlocks * BB;
  static constexpr int stages = DI == 64 ? 16 : (DI == 128 ? 8 : 4);
  static constexpr int bar_off = stages * stage_bytes;
  static constexpr int smem = bar_off + 2 * stages * 8;
};

// Walks a CTA's contiguous range of stages in order without per-stage divisions: the unit and its
// data (sequence, query, valid entries) are refreshed only when the walk crosses into a new unit.
struct StageCursor {
  int64_t unit, st;         // unit index and stage within the unit
  int64_t b, jq0, n_e, n_b;
  int64_t slot0, id0;
  int valid;                // leading blocks of the stage that exist in the cache

  __device__ __forceinline__ void load_unit(const ScoreParams& p) {
    const bool hier = p.kept != nullptr;
    b = hier ? unit / p.n_query : unit;
    jq0 = hier ? unit % p.n_query : 0;
    int64_t n = p.n_entries[b];
    n_e = n < 0 ? 0 : (n > p.max_entries ? p.max_entries : n);
    n_b = (n_e + kBlockEntries - 1) / kBlockEntries;
  }
  __device__ __forceinline__ void load_stage(const ScoreParams& p) {
    slot0 = st * kStageBlocks;
    if (p.kept != nullptr) {
      const int32_t g = p.kept[unit * p.keep_super + (st >> 2)];       // 4 stages per super-block
      id0 = g < 0 ? -1 : (int64_t)g * kSuper + (slot0 & (kSuper - 1));
    } else {
      id0 = slot0;
    }
    int64_t v = id0 < 0 ? 0 : n_b - id0;
    v = v < 0 ? 0 : (v > kStageBlocks ? kStageBlocks : v);
    const int64_t slots_left = p.n_slots - slot0;
    valid = (int)(v < slots_left ? v : slots_left);
  }
  __device__ __forceinline__ void begin(const ScoreParams& p, int64_t gs, int64_t spu) {
    unit = gs / spu;
    st = gs - unit * spu;
    load_unit(p);
    load_stage(p);
  }
  __device__ __forceinline__ bool next(const ScoreParams& p, int64_t spu) {   // true if the unit changed
    bool changed = false;
    if (++st == spu) { st = 0; ++unit; load_unit(p); changed = true; }
    load_stage(p);
    return changed;
  }
};

template <int DI>
__device__ __forceinline__ void load_row_smem(const uint8_t* blk, int r, int c, RowRaw<DI>& out) {
  constexpr int BPL = DI / 8, GPL = DI / 64;
  const uint32_t cp = smem_addr(blk + r * (DI / 2) + c * BPL);
  if constexpr (BPL == 8) {
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(out.code[0]), "=r"(out.code[1]) : "r"(cp));
  } else {
#pragma unroll
    for (int i = 0; i < BPL / 16; ++i)
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(out.code[4 * i]), "=r"(out.code[4 * i + 1]), "=r"(out.code[4 * i + 2]),
                     "=r"(out.code[4 * i + 3])
                   : "r"(cp + 16 * i));
  }
  const uint8_t* sp = blk + kBlockEntries * (DI / 2) + r * (DI / 16) + c * GPL;
  if constexpr (GPL == 1) out.scale = *sp;
  else if constexpr (GPL == 2) out.scale = *reinterpret_cast<const unsigned short*>(sp);
  else out.scale = *reinterpret_cast<const unsigned int*>(sp);
}

template <int DI, int HI>
__global__ void __launch_bounds__(kStreamThreads, 2)
index_stream_kernel(ScoreParams p, int64_t total_stages, int64_t stages_per_unit) {
  using C = StreamCfg<DI>;
  constexpr int KS = DI / 16;
  constexpr int GPL = DI / 64;
  constexpr int QPM = HI >= 8 ? 1 : 8 / HI;
  constexpr int LPQ = HI >= 2 ? HI / 2 : 1;
  constexpr int QPL = HI == 1 ? 2 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::bar_off);
  uint64_t* empty = full + C::stages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t s0 = total_stages * blockIdx.x / gridDim.x;
  const int64_t s1 = total_stages * (blockIdx.x + 1) / gridDim.x;
  const bool hier = p.kept != nullptr;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---- producer: one lane issues every copy of this CTA's stages, in order
    if (lane != 0) return;
    int64_t issued = 0;
    StageCursor si;
    si.begin(p, s0, stages_per_unit);
    for (int64_t gs = s0; gs < s1; ++gs, ++issued) {
      const int64_t k = gs - s0;
      const int slot = (int)(k % C::stages);
      const uint32_t round = (uint32_t)(k / C::stages);
      if (k > 0) si.next(p, stages_per_unit);
      if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1u)) {
        report(p.hdr, CSA_ERR_TIMEOUT, KID_INDEX_SCORE, (uint32_t)blockIdx.x);
        break;
      }
      const uint32_t bytes = (uint32_t)si.valid * C::BB;
      if (bytes) {
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s(smem + slot * C::stage_bytes, p.keys + si.b * p.keys_stride_b + si.id0 * C::BB, bytes,
                 &full[slot]);
      } else {
        mbar_arrive(&full[slot]);
      }
    }
    // the CTA must not exit while a copy into its shared memory is still in flight
    for (int64_t k = issued - C::stages < 0 ? 0 : issued - C::stages; k < issued; ++k) {
      if (!mbar_wait(&full[k % C::stages], (uint32_t)(k / C::stages) & 1u)) {
        report(p.hdr, CSA_ERR_TIMEOUT, KID_INDEX_SCORE, (uint32_t)blockIdx.x);
        break;
      }
    }
    return;
  }

  // ---- consumers
  const int r = lane >> 2, c = lane & 3;
  float w0 = 1.0f, w1 = 1.0f;
  if (p.head_w) { w0 = __ldg(p.head_w + (2 * c) % HI); w1 = __ldg(p.head_w + (2 * c + 1) % HI); }
  uint32_t bq[KS][2];
  StageCursor si;
  si.begin(p, s0, stages_per_unit);
  load_qfrag<DI, HI>(p, si.b, hier ? si.jq0 : (int64_t)(r / HI), lane, bq);
  for (int64_t gs = s0; gs < s1; ++gs) {
    const int64_t k = gs - s0;
    const int slot = (int)(k % C::stages);
    const uint32_t round = (uint32_t)(k / C::stages);
    if (k > 0 && si.next(p, stages_per_unit))
      load_qfrag<DI, HI>(p, si.b, hier ? si.jq0 : (int64_t)(r / HI), lane, bq);
    const int64_t jq0 = si.jq0;
    if (!mbar_wait(&full[slot], round & 1u)) {
      if (lane == 0) report(p.hdr, CSA_ERR_TIMEOUT, KID_INDEX_SCORE, (uint32_t)blockIdx.x);
      return;
    }
    const uint8_t* st = smem + slot * C::stage_bytes;
    const int i0 = 2 * warp;
    const bool ok0 = i0 < si.valid, ok1 = i0 + 1 < si.valid;
    RowRaw<DI> ra, rb;
    if (ok0) load_row_smem<DI>(st + i0 * C::BB, r, c, ra); else zero_row<DI>(ra);
    if (ok1) load_row_smem<DI>(st + (i0 + 1) * C::BB, r, c, rb); else zero_row<DI>(rb);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (si.slot0 + i0 >= p.n_slots) continue;

    uint32_t sa[GPL], sb[GPL];
#pragma unroll
    for (int gi = 0; gi < GPL; ++gi) {
      sa[gi] = e4m3_to_f16x2_bcast((ra.scale >> (8 * gi)) & 0xFFu);
      sb[gi] = e4m3_to_f16x2_bcast((rb.scale >> (8 * gi)) & 0xFFu);
    }
    uint32_t af[KS][4];
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) a_frag<DI>(ra, rb, sa, sb, kk, af[kk]);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) mma16816(acc, af[kk], bq[kk][0], bq[kk][1]);

    float tv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float d = p.relu ? fmaxf(acc[i], 0.0f) : acc[i];
      tv[i] = __fmul_rn((i & 1) ? w1 : w0, d);
    }
    float sc[2][QPL];
    if constexpr (HI == 1) {
      sc[0][0] = tv[0]; sc[0][1] = tv[1]; sc[1][0] = tv[2]; sc[1][1] = tv[3];
    } else {
      const int base = (lane & ~3) | (c - c % LPQ);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float acc_s = 0.0f;
#pragma unroll
        for (int i = 0; i < LPQ; ++i) {
          const float x0 = __shfl_sync(0xffffffffu, tv[2 * half], base + i);
          const float x1 = __shfl_sync(0xffffffffu, tv[2 * half + 1], base + i);
          acc_s = (i == 0) ? x0 : __fadd_rn(acc_s, x0);
          acc_s = __fadd_rn(acc_s, x1);
        }
        sc[half][0] = acc_s;
      }
    }
    const int64_t eA = (si.id0 + i0) * kBlockEntries + r;
    const int64_t eB = eA + kBlockEntries;
#pragma unroll
    for (int kq = 0; kq < QPL; ++kq) {
      const int64_t jq = hier ? jq0 : (HI == 1 ? 2 * c + kq : c / LPQ);
      int64_t pos = INT64_MAX;
      if (p.q_pos != nullptr && jq < p.n_query) pos = p.q_pos[si.b * p.n_query + jq];
      const bool vA = ok0 && eA < si.n_e && 2 * eA + 1 <= pos;
      const bool vB = ok1 && eB < si.n_e && 2 * eB + 1 <= pos;
      float mA = vA ? __fadd_rn(sc[0][kq], 0.0f) : -INFINITY;
      float mB = vB ? __fadd_rn(sc[1][kq], 0.0f) : -INFINITY;
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, off));
        mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, off));
      }
      const bool owner = (r == 0) && (HI == 1 || c % LPQ == 0) && jq < p.n_query;
      if (owner) {
        const int64_t row = hier ? si.unit : si.b * p.n_query + jq;
        float* dst = p.scores + row * p.score_stride + si.slot0 + i0;
        dst[0] = mA;
        if (si.slot0 + i0 + 1 < p.n_slots) dst[1] = mB;
      }
    }
  }
}

template <int DI, int HI>
cudaError_t launch_score_t(const ScoreParams& p, int num_sms, cudaStream_t s) {
  constexpr int QPM = HI >= 8 ? 1 : 8 / HI;
  if (p.kept != nullptr || p.n_query <= QPM) {
    // every unit's queries fit one MMA column group: stream the keys through shared memory
    using C = StreamCfg<DI>;
    const int64_t units = p.kept ? p.batch * p.n_query : p.batch;
    const int64_t spu = (p.n_slots + kStageBlocks - 1) / kStageBlocks;
    const int64_t total = units * spu;
    int64_t grid = 2 * (int64_t)num_sms;
    if (grid > total) grid = total;
    if (grid < 1) return cudaSuccess;
    cudaError_t e = ensure_smem_limit(index_stream_kernel<DI, HI>, C::smem);
    if (e != cudaSuccess) return e;
    clear_stale_error();
    index_stream_kernel<DI, HI><<<(unsigned)grid, kStreamThreads, C::smem, s>>>(p, total, spu);
    return cudaGetLastError();
  }
  const int64_t units_y = p.kept ? p.batch * p.n_query : p.batch;
  const int64_t tiles = (p.n_slots + 1) / 2;
  constexpr int kThreads = 256, kWarps = kThreads / 32;
  int64_t want = ((int64_t)num_sms * 4 + units_y - 1) / units_y;   // ~4 CTAs per SM in total
  int64_t need = (tiles + kWarps - 1) / kWarps;
  int64_t bx = want < need ? want : need;
  if (bx < 1) bx = 1;
  dim3 grid((unsigned)bx, (unsigned)units_y);
  clear_stale_error();
  index_score_kernel<DI, HI><<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <int DI>
cudaError_t launch_score_d(const ScoreParams& p, int num_sms, cudaStream_t s) {
  switch (p.heads) {
    case 1: return launch_score_t<DI, 1>(p, num_sms, s);
    case 2: return launch_score_t<DI, 2>(p, num_sms, s);
    case 4: return launch_score_t<DI, 4>(p, num_sms, s);
    case 8: return launch_score_t<DI, 8>(p, num_sms, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_index_score(const ScoreParams& p, int num_sms, cudaStream_t s) {
  if (p.n_slots == 0) return cudaSuccess;
  ProfScope prof(p.kept ? "index_score_hier" : "index_score", s);
  switch (p.dim) {
    case 64: return launch_score_d<64>(p, num_sms, s);
    case 128: return launch_score_d<128>(p, num_sms, s);
    case 256: return launch_score_d<256>(p, num_sms, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_coarse_score(const CoarseScoreParams& p, cudaStream_t s) {
  const int64_t warps = p.batch * p.n_query * p.n_super;
  if (warps == 0) return cudaSuccess;
  ProfScope prof("coarse_score", s);
  const int64_t blocks = (warps + 7) / 8;
  clear_stale_error();
  coarse_score_kernel<<<(unsigned)blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace csa
