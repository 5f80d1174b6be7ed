// Sparse attention over selected FP4 cache blocks merged with the sliding window, on the fifth-generation
// tensor cores (tcgen05), split over the row list, plus the fixed-order log-sum-exp combine of the splits.
//
// Follows "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression" (paper-digest), Core
// Mechanics ("one 512-dim latent shares keys and values across all attention heads") and Terminology
// (sliding window of 128), and "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (card),
// Key ideas ("Every layer keeps its own query and sliding-window KV").
//
// Design. A CTA owns one query (all heads) and some 128-row tiles of its row list: the window tiles first,
// then a range of cache tiles (16 selected blocks each). Because one latent row c is both key and value,
// both products are taken with the rows as the 128-wide M side and the heads as N:
//   S^T [rows x heads]  = C [rows x 512] . Q^T                   (logits)
//   O^T [512 x heads]  += C^T [512 x rows] . P^T [rows x heads]  (values)
// Both read the same dequantised tile in shared memory: 128-byte-swizzled rows of 64 latent columns are the
// K-major layout of C and the MN-major layout of C^T. S and O accumulate in tensor memory; the row sums l
// are added up by one warp from the fp16 probabilities in shared memory (the same values the tensor core
// multiplies).
//   Every tile is dequantised once. Eight converter warps (thread = tensor-memory lane = tile row) read
//   their row's FP4 codes and scales straight from global memory (the gather warp prefetches each cache
//   tile's blocks into L2 three tiles ahead; a converter keeps the codes of its next two panels in flight in
//   registers, one 32-byte load each, and loads a tile's scale bytes once), convert a 64-column panel to
//   fp16 and write it into the tile buffer in shared memory. The buffer holds one whole tile and is recycled
//   per 128-latent chunk as the value products finish with it; both products wait for a chunk on the same
//   barrier. Window tiles come first: their bf16 rows are copied by tensor map straight into the buffer and
//   converted to fp16 in place by the same threads.
// Pipelining: S and P are double-buffered, so the softmax of tile t+1 can run while the values of tile t are
// multiplied; the converters of tile t+1 wait only for the value products of the chunk they overwrite (which
// complete after the same tile's logits). Both products are issued by whole warps (one elected lane
// issues).
//
// Warp roles: 0-3 softmax and epilogue (thread = tile row), 4-11 converters (warp 4 + 4 h + s covers
// subpartition s, panels of parity h), 12 gather (window copies, L2 prefetch, block-id checks), 13 logits
// MMA issue and tensor-memory allocation, 14 values MMA issue, 15 row sums. The softmax keeps, per head, a
// reference maximum that is raised only when a tile's maximum exceeds it by more than 8 (in log2 units),
// so the probabilities stay below 2^8 and the accumulators are rescaled rarely. When a query's rows are
// split over several CTAs, every split writes its unnormalised partial (o, m, l) and the combine kernel
// merges them in split order (measured faster than merging inside the kernel across a thread-block
// cluster, through distributed shared memory or through L2 copies).
//
// Prepared operands. A prepare kernel (attn_prep_kernel, the attention's predecessor) converts each query
// once into the workspace when many queries have several splits each, so that the splits copy the fp16
// panels in by tensor map instead of each converting them.
//
// NVFP4-query mode (attn_tc_kernel<true>, opt-in). The logits are taken on the block-scaled FP4 tensor cores
// (kind::mxf4nvf4): the prepare kernel rounds the query heads and the window rows to the cache's FP4 format;
// the logits warp copies each tile's FP4 keys (cache codes, or the rounded window rows) into a raw stage by
// tensor map as soon as the previous tile's logits are complete, and the converters, which still build the
// exact fp16 tile for the value products, write the keys' scale factors to tensor memory one tile ahead. The
// logits then never wait for the values buffer; the converters set the tile cadence.
#include <cuda.h>

#include <cstring>

#include "csa_internal.cuh"
#include "tc.cuh"

namespace csa {
namespace {

constexpr int kRows = 128;                                 // rows per tile: M of both products
constexpr int kTileBlocks = kRows / kBlockEntries;         // 16 cache blocks per tile
constexpr int kHeadsPad = 64;                              // N of both products (heads, zero-padded)
constexpr int kPanels = kLatent / 64;                      // 8 panels of 64 latent columns
constexpr int kChunks = kLatent / 128;                     // 4 chunks of 128 latent columns (M of a value product)
constexpr int kLatBlk = block_bytes(kLatent);              // 2304
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.0f;                      // log2 headroom before the reference max moves
constexpr float kMaxProb = 256.0f;                         // 2^kRescaleSlack

// shared-memory map (bytes); the operand regions start on 1024-byte boundaries
constexpr int kQPanel = kHeadsPad * 128;                   // 8 KB: [64 heads x 64 latent] fp16
constexpr int kQOff = 0;                                   // queries: 8 K-major panels, 64 KB
constexpr int kHalfBytes = kRows * 128;                    // 16 KB: 64 latent columns of a whole tile
constexpr int kChunkBytes = 2 * kHalfBytes;                // 32 KB: 128 latent columns of a whole tile
constexpr int kVOff = kQOff + kPanels * kQPanel;           // 65,536: the values buffer, 4 chunks
constexpr int kPBytes = kRows * 128;                       // 16 KB: one P^T buffer
constexpr int kPOff = kVOff + kChunks * kChunkBytes;       // 196,608: two P^T buffers
constexpr int kBarOff = kPOff + 2 * kPBytes;               // 229,376
constexpr int kNumBars = 32;
constexpr int kTmemPtrOff = kBarOff + kNumBars * 8;
constexpr int kFlagOff = kTmemPtrOff + 16;                 // int flag[2], abort, have, progress
constexpr int kMOff = kFlagOff + 32;                       // float m[64]
constexpr int kAlphaOff = kMOff + 64 * 4;                  // float alpha[2][64]: per P buffer
constexpr int kRedOff = kAlphaOff + 2 * 64 * 4;            // float red[4][64]
constexpr int kLsumOff = kRedOff + 4 * 64 * 4;             // float lsum[64]: final row sums
constexpr int kQScaleOff = kLsumOff + 64 * 4;              // float qscale[64]: per-head log2 softmax scale
constexpr int kQMaxOff = kQScaleOff + 64 * 4;              // uint qmax[64]: bits of each head's largest |q|
constexpr int kSmemBytes = kQMaxOff + 64 * 4;
static_assert(kVOff % 1024 == 0 && kPOff % 1024 == 0, "swizzled operands start on 1024-byte boundaries");
// NVFP4-query mode: the query region holds the FP4 query (B operand of the block-scaled logits), its scale
// bytes, and one stage of a tile's FP4 codes (A operand): block b of the tile at kRawOff + 2048 b, its 8 rows'
// first 128 code bytes (latent 0-255) then their last 128, each an 8-row 128-byte-swizzled atom.
constexpr int kQ4Off = 0;                                  // 2 K-halves x [64 heads x 128 B]: 16 KB
constexpr int kQ4ScOff = kQ4Off + 2 * kHeadsPad * 128;     // 64 heads x 32 scale bytes: 2 KB
constexpr int kRawOff = kQ4ScOff + kHeadsPad * 32;         // 16 blocks x 2 KB
constexpr int kRawBytes = kTileBlocks * 2048;
static_assert(kRawOff % 1024 == 0 && kRawOff + kRawBytes <= kVOff, "NVFP4-query operands fit the query region");
static_assert(kSmemBytes <= 232448, "shared memory");

enum Bar {
  V_FULL = 0,                           // tile buffer chunks: converters <-> logits and values issuers
  V_EMPTY = V_FULL + kChunks,
  S_FULL = V_EMPTY + kChunks,           // logits buffers: logits issuer <-> softmax
  S_EMPTY = S_FULL + 2,
  P_FULL = S_EMPTY + 2,                 // P buffers: softmax <-> values issuer and row sums
  P_EMPTY = P_FULL + 2,
  WIN_FULL = P_EMPTY + 2,               // a window tile's rows have landed in the values buffer
  SFX_FULL,                             // NVFP4-query mode: a tile's key scale factors are in tensor memory
                                        // (and a window tile's FP4 codes in the raw stage); one per parity
  RAW_FULL = SFX_FULL + 2,              // NVFP4-query mode: a cache tile's codes have landed in the raw stage
  RAW_DONE,                             // NVFP4-query mode: the logits of the tile in the raw stage are complete
  Q_FULL,                               // prepared fp16 queries have landed (exact attention with several splits)
  FIN_L, FIN_V, NUM_BARS
};

static_assert(NUM_BARS <= kNumBars, "barrier area");

constexpr int kConv0 = 4, kConvWarps = 8;      // converter warps 4..11
constexpr int kGatherWarp = 12, kLogitsWarp = 13, kValuesWarp = 14, kSumWarp = 15;
constexpr int kThreads = 16 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;   // S: two buffers of 64 columns; O^T: 4 x 64 columns
// NVFP4-query mode: key scale factors, two buffers of 8 products x 4 columns; query scale factors, 8 x 4
constexpr uint32_t kColSFA = 128, kColSFB = 192;

constexpr uint32_t kIdescS = tc::idesc_f16_f32(128, kHeadsPad, 0, 0);   // C K-major, Q K-major
constexpr uint32_t kIdescPV = tc::idesc_f16_f32(128, kHeadsPad, 1, 1);  // C^T MN-major, P^T MN-major
constexpr uint32_t kIdescS4 = tc::idesc_mxf4(128, kHeadsPad);            // FP4 codes, FP4 query

// Bounded wait that also gives up as soon as another role of the CTA has given up.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         uint32_t* hdr, uint32_t detail, uint32_t limit) {
  const uint32_t a = smem_addr(bar);
  if (mbar_test_wait(a, parity)) return true;      // the common case: the phase completed already
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 7u) == 7u && *abort_flag) return false;
  }
  *abort_flag = 1;
  report(hdr, CSA_ERR_TIMEOUT, KID_ATTN, detail);
  return false;
}

// The same wait taken by a whole warp; the result is the same on every lane.
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              uint32_t* hdr, uint32_t detail, uint32_t limit) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, hdr, detail, limit));
}

// Bounded wait that ignores the abort flag (draining copies that must land before the CTA exits).
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(a, parity)) return;
  }
}

// AND of v over the 128 softmax threads (named barrier 1), so that they all take the same branch.
__device__ __forceinline__ bool all_softmax(bool v) {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.and.pred p, 1, 128, q;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(r) : "r"((uint32_t)v) : "memory");
  return r != 0;
}

// OR of v over the 128 softmax threads (named barrier 1).
__device__ __forceinline__ bool any_softmax(bool v) {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, 1, 128, q;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(r) : "r"((uint32_t)v) : "memory");
  return r != 0;
}

// Tensor-map copy of a [1 x 128 x 64] box (batch, row, latent column) into shared memory.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
               " [%0], [%1, {%2, %3, %4}], [%5];"
               :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
                  "r"(smem_addr(bar)) : "memory");
}

// Tensor-map copy of one [8 x 128-byte] box (the code bytes of one cache block's 8 rows, one half of each
// row) into shared memory, 128-byte swizzled.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w, uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
               " [%0], [%1, {%2, %3, %4, %5}], [%6];"
               :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w),
                  "r"(smem_addr(bar)) : "memory");
}

// Two E2M1 codes (lo in the low nibble): the nearest E2M1 value, ties to the even code, saturating at 6, the
// sign kept (the hardware conversion with round-to-nearest-even and finite saturation).
__device__ __forceinline__ uint32_t e2m1x2_rn(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tmov.b32 %0, {t, t, t, t};\n\t}"
      : "=r"(r) : "f"(lo), "f"(hi));
  return r & 0xFFu;
}

// One 16-element group rounded with the AMAX rule of the cache format (the rule csa_pack_fp4 applies): the
// E4M3 scale byte of fl32(amax / 6) is returned, the E2M1 codes of fl32(v / s) go to *lo (elements 0-7) and
// *hi (8-15), low nibble first; a zero scale gives zero codes.
__device__ __forceinline__ uint32_t quant16_amax(const float* v, uint32_t* lo, uint32_t* hi) {
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[k]));
  const float sf = __fdiv_rn(amax, 6.0f);
  uint32_t sbyte = 0u;
  float s = 0.0f;
  if (sf > 0.0f) {
    sbyte = float_to_e4m3_satfinite(sf);
    s = e4m3_to_float(sbyte);
  }
  uint32_t c0 = 0u, c1 = 0u;
  if (s > 0.0f) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      c0 |= e2m1x2_rn(__fdiv_rn(v[2 * k], s), __fdiv_rn(v[2 * k + 1], s)) << (8 * k);
      c1 |= e2m1x2_rn(__fdiv_rn(v[8 + 2 * k], s), __fdiv_rn(v[9 + 2 * k], s)) << (8 * k);
    }
  }
  *lo = c0;
  *hi = c1;
  return sbyte;
}

struct UnitCtx {
  int64_t unit, b, n_e, n_b, nb_cap, pos, swa_first, swa_len;
  bool prefill;
};

// Block id of row r of the CTA's global cache tile t as stored in the index list (-1 past the list).
__device__ __forceinline__ int cache_id(const AttnParams& p, const UnitCtx& u, int t, int r) {
  const int slot = t * kTileBlocks + (r >> 3);
  return slot < p.top_k ? __ldg(p.idx + u.unit * p.top_k + slot) : -1;
}

// Whether row r (slot r & 7) of a block with stored id `id` is attended.
__device__ __forceinline__ bool cache_ok(const UnitCtx& u, int64_t id, int r) {
  if (id < 0 || id >= u.n_b) return false;
  const int64_t e = id * kBlockEntries + (r & 7);
  return e < u.n_e && 2 * e + 1 <= u.pos;
}

// Bulk prefetch of a global range into L2 (no shared-memory destination, no completion).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}

// Prefetch of one [1 x 128 x 64] box of a tensor map into L2.
__device__ __forceinline__ void prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
               :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z) : "memory");
}

// First window-buffer row of window tile tw (may be negative or past the buffer: those rows are filled
// with zeros by the tensor copy and are never attended).
__device__ __forceinline__ int64_t window_row0(const AttnParams& p, const UnitCtx& u, int tw) {
  return u.prefill ? u.pos - p.window + 1 + (int64_t)tw * kRows - u.swa_first : (int64_t)tw * kRows;
}

// Whether row r of window tile tw is attended; *oob reports a row the caller declared present but that
// lies outside the window buffer.
__device__ __forceinline__ bool window_row(const AttnParams& p, const UnitCtx& u, int tw, int r, bool* oob) {
  const int slot = tw * kRows + r;
  *oob = false;
  if (slot >= p.window) return false;
  const bool declared = u.prefill ? (u.pos - p.window + 1 + slot >= u.swa_first) : (slot < u.swa_len);
  const int64_t s = window_row0(p, u, tw) + r;
  if (declared && (s < 0 || s >= p.swa_rows)) { *oob = true; return false; }
  return declared;
}

// Copies window tile tw (128 rows x 512 bf16) into the values buffer: eight [128 x 64] boxes, box k going
// to chunk k / 2, half k % 2, in the buffer's 128-byte-swizzled layout.
__device__ __forceinline__ void copy_window_tile(const AttnParams& p, const UnitCtx& u, int tw, uint8_t* smem,
                                                 const CUtensorMap* map, uint64_t* bar) {
  const int64_t y0 = window_row0(p, u, tw);
  const int y = (int)(y0 < -(int64_t)kRows ? -kRows : (y0 > p.swa_rows ? p.swa_rows : y0));
  mbar_arrive_expect_tx(bar, kChunks * kChunkBytes);
#pragma unroll
  for (int k = 0; k < 2 * kChunks; ++k)
    tma_load_3d(smem + kVOff + k * kHalfBytes, map, 64 * k, y, (int)u.b, bar);
}

// 2^x by the hardware approximation (relative error near 2^-22; subnormal results flush to zero). The
// probabilities it produces are rounded to fp16 for the tensor core, so the approximation is invisible.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t x) {
  return f2_to_h2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
}

// Four code bytes (eight E2M1 elements, low nibble first) -> four f16x2, exact.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t* h) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
}

// One 64-column panel of a cache row: 32 code bytes (w) and 4 scale bytes (sc) -> 32 f16x2, exact.
// Zero codes and a zero scale (rows that are not attended) give exact zeros.
__device__ __forceinline__ void dequant_panel(const uint32_t* w, uint32_t sc, uint32_t* h) {
#pragma unroll
  for (int i = 0; i < 8; ++i) e2m1x8_to_f16x8(w[i], h + 4 * i);
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t s2 = e4m3_to_f16x2_bcast((sc >> (8 * g)) & 0xFFu);
#pragma unroll
    for (int k = 0; k < 8; ++k) h[8 * g + k] = hmul2_u32(h[8 * g + k], s2);
  }
}

// 32 bytes (one sector) of read-only global memory in one 256-bit load; p must be 32-byte aligned.
__device__ __forceinline__ void ld_nc_v8(const void* ptr, uint32_t* r) {
  asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "l"(ptr));
}

// 16 bytes of read-only global memory (a volatile load: issued where written and never repeated).
__device__ __forceinline__ uint4 ld_nc_v4(const void* ptr) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(ptr));
  return r;
}

// The scale words of the four panels of parity hp (panels hp, hp + 2, hp + 4, hp + 6) of one cache row:
// one 256-bit load of the row's 32 scale bytes; zeros for a row that is not attended.
__device__ __forceinline__ void load_scales(const uint8_t* seq, int id, bool ok, int row, int hp, uint32_t* sc) {
  uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
  if (ok) ld_nc_v8(seq + (int64_t)id * kLatBlk + 2048 + (row & 7) * 32, w);
#pragma unroll
  for (int c = 0; c < 4; ++c) sc[c] = hp ? w[2 * c + 1] : w[2 * c];
}

// NVFP4-query mode: the scale words of the four panels of parity hp of row `row` of window tile tw, from the
// window rows the prepare kernel rounded; zeros for a row that is not attended.
__device__ __forceinline__ void load_window_scales(const AttnParams& p, const UnitCtx& u, int tw, int row, int hp,
                                                   uint32_t* sc) {
  bool oob;
  uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
  if (window_row(p, u, tw, row, &oob)) ld_nc_v8(p.w4_sc + ((int64_t)u.b * p.swa_rows + window_row0(p, u, tw) + row) * 32, w);
#pragma unroll
  for (int c = 0; c < 4; ++c) sc[c] = hp ? w[2 * c + 1] : w[2 * c];
}

// NVFP4-query mode: a converter writes the key scale factors of its row and its four panels (panels hp,
// hp + 2, hp + 4, hp + 6 = block-scaled products of K = 64) of tile t into scale buffer t & 1 (row m's bytes
// of product s at lane m, column kColSFA + 32 (t & 1) + 4 s + m / 32) and arrives on that buffer's barrier.
__device__ __forceinline__ void put_key_scales(uint32_t tbase, int sp, int hp, int lane, int t, const uint32_t* sc,
                                               uint64_t* bars) {
  const uint32_t lb = (uint32_t)(sp * 32) << 16;
#pragma unroll
  for (int c = 0; c < 4; ++c) tc::st_32x1(tbase + lb + kColSFA + 32 * (t & 1) + 4 * (2 * c + hp) + sp, sc[c]);
  tc::wait_st();
  tc::fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars[SFX_FULL + (t & 1)]);
}

__device__ __forceinline__ uint32_t pick4(const uint32_t* v, int i) {
  return i == 0 ? v[0] : (i == 1 ? v[1] : (i == 2 ? v[2] : v[3]));
}

// NVFP4-query variant, first step: rounds every query head and every window row once per call. One warp per
// 512-element row, lane = one 16-element group. A query head is scaled by 2^-e, e = floor(log2 max|q_h|) - 10
// clamped to [-100, 100], which puts every block's amax / 6 below 342 (inside the E4M3 scale range); rows
// beyond the call's heads are zero so that each unit has 64 rows. Window rows are rounded as they are.
__global__ void __launch_bounds__(256) attn_prep_kernel(const AttnParams p) {
  griddep_launch();                                // the attention kernel may start its setup
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t qrows = p.units * 64;
  const int64_t wrows = p.q4 && p.window > 0 ? (p.units / p.n_query) * p.swa_rows : 0;
  float x[16];
  uint32_t w8[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
  if (r < qrows && !p.q4) {
    // exact attention: the head scaled by 2^-e, e = floor(log2 max|q_h|) - 14, which puts its largest magnitude
    // in [2^14, 2^15), and rounded to fp16 (exact for every finite bf16 value), as the attention kernel does
    // when it converts its own queries
    const int64_t unit = r >> 6;
    const int h = (int)(r & 63);
    if (h < p.heads) {
      const __nv_bfloat16* src = p.q + (unit * p.heads + h) * kLatent + lane * 16;
      const uint4 a = ld_nc_v4(src), b = ld_nc_v4(src + 8);
      w8[0] = a.x; w8[1] = a.y; w8[2] = a.z; w8[3] = a.w; w8[4] = b.x; w8[5] = b.y; w8[6] = b.z; w8[7] = b.w;
    }
    uint32_t m = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = max(m, max(w8[j] & 0x7FFFu, (w8[j] >> 16) & 0x7FFFu));
    m = __reduce_max_sync(0xffffffffu, m);
    int sh = m == 0u ? 0 : (int)((m >> 7) & 0xFFu) - 127 - 14;
    sh = sh < -100 ? -100 : (sh > 100 ? 100 : sh);
    const float f = __int_as_float((127 - sh) << 23);
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      o[j] = f2_to_h2(__uint_as_float(w8[j] << 16) * f, __uint_as_float(w8[j] & 0xFFFF0000u) * f);
    uint4* dst = reinterpret_cast<uint4*>(p.qh + r * kLatent + lane * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    if (lane == 0) p.q4_mult[r] = __int_as_float((127 + sh) << 23);
  } else if (r < qrows) {
    const int64_t unit = r >> 6;
    const int h = (int)(r & 63);
    if (h < p.heads) {
      const __nv_bfloat16* src = p.q + (unit * p.heads + h) * kLatent + lane * 16;
      const uint4 a = ld_nc_v4(src), b = ld_nc_v4(src + 8);
      w8[0] = a.x; w8[1] = a.y; w8[2] = a.z; w8[3] = a.w; w8[4] = b.x; w8[5] = b.y; w8[6] = b.z; w8[7] = b.w;
    }
    uint32_t m = 0u;                               // |x| bits: magnitudes compare as integers
#pragma unroll
    for (int j = 0; j < 8; ++j) m = max(m, max(w8[j] & 0x7FFFu, (w8[j] >> 16) & 0x7FFFu));
    m = __reduce_max_sync(0xffffffffu, m);
    int sh = m == 0u ? 0 : (int)((m >> 7) & 0xFFu) - 127 - 10;
    sh = sh < -100 ? -100 : (sh > 100 ? 100 : sh);
    const float f = __int_as_float((127 - sh) << 23);               // 2^-sh, exact
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      x[2 * j] = __fmul_rn(__uint_as_float(w8[j] << 16), f);
      x[2 * j + 1] = __fmul_rn(__uint_as_float(w8[j] & 0xFFFF0000u), f);
    }
    uint32_t lo, hi;
    const uint32_t sb = quant16_amax(x, &lo, &hi);
    *reinterpret_cast<uint2*>(p.q4_codes + r * 256 + lane * 8) = make_uint2(lo, hi);
    p.q4_sc[r * 32 + lane] = (uint8_t)sb;
    if (lane == 0) p.q4_mult[r] = __int_as_float((127 + sh) << 23);  // 2^sh
  } else if (r < qrows + wrows) {
    const int64_t wr = r - qrows;
    const int64_t b = wr / p.swa_rows, row = wr % p.swa_rows;
    const __nv_bfloat16* src = p.swa + b * p.swa_stride_b + row * kLatent + lane * 16;
    const uint4 a = ld_nc_v4(src), c = ld_nc_v4(src + 8);
    w8[0] = a.x; w8[1] = a.y; w8[2] = a.z; w8[3] = a.w; w8[4] = c.x; w8[5] = c.y; w8[6] = c.z; w8[7] = c.w;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      x[2 * j] = __uint_as_float(w8[j] << 16);
      x[2 * j + 1] = __uint_as_float(w8[j] & 0xFFFF0000u);
    }
    uint32_t lo, hi;
    const uint32_t sb = quant16_amax(x, &lo, &hi);
    *reinterpret_cast<uint2*>(p.w4 + wr * 256 + lane * 8) = make_uint2(lo, hi);
    p.w4_sc[wr * 32 + lane] = (uint8_t)sb;
  }
  // completes only after the kernel before it, so that its dependent, which waits for this kernel alone,
  // also sees everything before (the index list)
  griddep_wait();
}

template <bool kQ4>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const AttnParams p,
                                                               const __grid_constant__ CUtensorMap swa_map,
                                                               const __grid_constant__ CUtensorMap cache_map,
                                                               const __grid_constant__ CUtensorMap win4_map,
                                                               const __grid_constant__ CUtensorMap qh_map) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + kTmemPtrOff);
  volatile int* flag = reinterpret_cast<volatile int*>(smem + kFlagOff);
  volatile int* abort_flag = flag + 2;
  float* msh = reinterpret_cast<float*>(smem + kMOff);
  float* alpha = reinterpret_cast<float*>(smem + kAlphaOff);
  float* red = reinterpret_cast<float*>(smem + kRedOff);
  float* lsh = reinterpret_cast<float*>(smem + kLsumOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const int H = p.heads;

  UnitCtx u;
  u.unit = blockIdx.y;
  u.b = u.unit / p.n_query;
  u.n_e = __ldg(p.n_entries + u.b);
  if (u.n_e < 0 || u.n_e > p.max_entries) {
    if (tid == 0 && split == 0) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_ATTN, (uint32_t)u.b);
    u.n_e = u.n_e < 0 ? 0 : p.max_entries;
  }
  u.n_b = (u.n_e + kBlockEntries - 1) / kBlockEntries;
  u.nb_cap = (p.max_entries + kBlockEntries - 1) / kBlockEntries;
  u.prefill = p.q_pos != nullptr;
  u.pos = u.prefill ? (int64_t)__ldg(p.q_pos + u.unit) : INT64_MAX;
  u.swa_first = (u.prefill && p.window > 0) ? (int64_t)__ldg(p.swa_first_pos + u.b) : 0;
  u.swa_len = (!u.prefill && p.window > 0) ? (int64_t)__ldg(p.swa_len + u.b) : 0;

  // this CTA's tiles: nw window tiles first, then cache tiles [c0, c1)
  const bool win_only = p.win_split && split == p.splits - 1;
  int c0 = 0, c1 = 0;
  if (!win_only) {
    if (p.last_ct >= 0) {
      const int rest = p.n_ct - p.last_ct, others = p.cache_splits - 1;
      c0 = split < others ? split * rest / others : rest;
      c1 = split < others ? (split + 1) * rest / others : p.n_ct;
    } else {
      c0 = (int)((int64_t)split * p.n_ct / p.cache_splits);
      c1 = (int)((int64_t)(split + 1) * p.n_ct / p.cache_splits);
    }
  }
  const int nw = (win_only || (!p.win_split && split == p.cache_splits - 1)) ? p.n_wt : 0;
  const int n_cache = c1 - c0;
  const int n_tiles = nw + n_cache;
  const uint8_t* seq = p.cache + u.b * p.cache_stride_b;

  // ---------------- setup ----------------
  if (warp == kLogitsWarp) tc::alloc(tmem_ptr, kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < kChunks; ++i) {
      mbar_init(&bars[V_FULL + i], kConvWarps);
      mbar_init(&bars[V_EMPTY + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[S_FULL + i], 1);
      mbar_init(&bars[S_EMPTY + i], 4);
      mbar_init(&bars[P_FULL + i], 4);
      mbar_init(&bars[P_EMPTY + i], 2);        // the values' commit and the row-sum warp
    }
    mbar_init(&bars[WIN_FULL], 1);
    mbar_init(&bars[SFX_FULL], kConvWarps);
    mbar_init(&bars[SFX_FULL + 1], kConvWarps);
    mbar_init(&bars[RAW_FULL], 1);
    mbar_init(&bars[RAW_DONE], 1);
    mbar_init(&bars[Q_FULL], 1);
    mbar_init(&bars[FIN_L], 1);
    mbar_init(&bars[FIN_V], 1);
    fence_mbar_init();
    flag[0] = 0; flag[1] = 0; *abort_flag = 0; flag[3] = 0; flag[4] = -1;
    for (int h = 0; h < 64; ++h) reinterpret_cast<uint32_t*>(smem + kQMaxOff)[h] = 0u;
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tmem_ptr;
  const uint32_t s_base = smem_addr(smem);

  // The first window tile lands in the values buffer while the queries are loaded.
  if (warp == kGatherWarp && lane == 0 && nw > 0) copy_window_tile(p, u, 0, smem, &swa_map, &bars[WIN_FULL]);

  // Converters: their rows' block ids of the first three cache tiles, the scales of the first two and the
  // codes of the first two panels, loaded as soon as the queries are in shared memory. The codes of the
  // next two panels a converter handles form a queue in registers (q0 is the next to convert): each
  // conversion shifts the queue and loads the panel two places further on (the same tile's chunk c + 2, or
  // the next cache tile's chunk c - 2).
  const bool is_conv = warp >= kConv0 && warp < kConv0 + kConvWarps;
  const int sp = warp & 3;                         // tensor-memory subpartition of this warp
  const int hp = (warp - kConv0) >> 2;             // converters: panel parity
  const int row = sp * 32 + lane;                  // converters and softmax: tile row = tensor-memory lane
  uint32_t q0[8], q1[8], qs0 = 0u, qs1 = 0u;
  uint32_t sc_c[4] = {0u, 0u, 0u, 0u}, sc_n[4] = {0u, 0u, 0u, 0u};   // scale words of cache tiles 0 and 1
  int id_c = -1, id_n = -1, id_nn = -1;            // block ids of cache tiles 0, 1 and 2 for this row
#pragma unroll
  for (int i = 0; i < 8; ++i) { q0[i] = 0u; q1[i] = 0u; }
  if (warp != kGatherWarp) {
    // queries: bf16 -> fp16, K-major 128-byte-swizzled panels; heads beyond H are zero. Each head is first
    // scaled by a power of two 2^-k_h that puts its largest magnitude in [2^14, 2^15), so that every
    // finite bf16 query converts to fp16 exactly (bf16 carries 8 significant bits, fp16 11); the factor
    // 2^k_h goes into that head's softmax scale. Every load of a thread is issued before the first use.
    constexpr int kQThreads = kThreads - 32;
    constexpr int kQItems = kHeadsPad * 64;
    constexpr int kQPer = (kQItems + kQThreads - 1) / kQThreads;
    static_assert(kQThreads % 32 == 0 && kQItems % 32 == 0, "one head per warp and item batch");
    const int qt = tid < kGatherWarp * 32 ? tid : tid - 32;
    const __nv_bfloat16* qg = p.q + u.unit * (int64_t)H * kLatent;
    uint32_t* qmax = reinterpret_cast<uint32_t*>(smem + kQMaxOff);
    float* qscale = reinterpret_cast<float*>(smem + kQScaleOff);
    if constexpr (!kQ4) {
      if (p.qh != nullptr) {
        // the queries were converted by the prepare kernel (this kernel's predecessor): eight tensor-map boxes
        // of [64 heads x 64 latent] land as the eight 128-byte-swizzled panels
        griddep_wait();
        if (warp == kLogitsWarp && lane == 0) {
          mbar_arrive_expect_tx(&bars[Q_FULL], kPanels * kQPanel);
#pragma unroll 1
          for (int pp = 0; pp < kPanels; ++pp)
            tma_load_3d(smem + kQOff + pp * kQPanel, &qh_map, 64 * pp, 0, (int)u.unit, &bars[Q_FULL]);
        }
        if (qt < 64) qscale[qt] = p.scale_log2 * __ldg(p.q4_mult + u.unit * 64 + qt);
      } else {
        uint4 v[kQPer];
#pragma unroll
        for (int k = 0; k < kQPer; ++k) {
          const int i = qt + k * kQThreads;
          const int h = i >> 6, ch = i & 63;
          v[k] = make_uint4(0, 0, 0, 0);
          if (i < kQItems && h < H) v[k] = ld_nc_v4(qg + (int64_t)h * kLatent + ch * 8);
        }
#pragma unroll
        for (int k = 0; k < kQPer; ++k) {
          const int i = qt + k * kQThreads;
          if (i < kQItems) {
            // magnitudes compare as integers: the bits of |x| with the sign cleared
            // (the 32 lanes of a warp hold 32 consecutive items starting at a multiple of 32, so all lie in one
            // head's 64 and the warp reduces them before one atomic; the branch is uniform per warp, since
            // kQItems and kQThreads are multiples of 32)
            uint32_t m = 0u;
            const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) m = max(m, max(w4[j] & 0x7FFFu, (w4[j] >> 16) & 0x7FFFu));
            m = __reduce_max_sync(0xffffffffu, m);
            if (lane == 0) atomicMax(qmax + (i >> 6), m);
          }
        }
        asm volatile("bar.sync 3, %0;" :: "n"(kQThreads) : "memory");
#pragma unroll
        for (int k = 0; k < kQPer; ++k) {
          const int i = qt + k * kQThreads;
          if (i < kQItems) {
            const int h = i >> 6, ch = i & 63, pp = ch >> 3, c = ch & 7;
            const uint32_t mb = qmax[h];
            int sh = mb == 0u ? 0 : (int)((mb >> 7) & 0xFFu) - 127 - 14;    // exponent of the largest |q|, - 14
            sh = sh < -100 ? -100 : (sh > 100 ? 100 : sh);
            const float f = __int_as_float((127 - sh) << 23);                  // 2^-sh, exact
            const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
              o[j] = f2_to_h2(__uint_as_float(w4[j] << 16) * f, __uint_as_float(w4[j] & 0xFFFF0000u) * f);
            *reinterpret_cast<uint4*>(smem + kQOff + pp * kQPanel + h * 128 + ((c ^ (h & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        if (qt < 64) {
          const uint32_t mb = qmax[qt];
          int sh = mb == 0u ? 0 : (int)((mb >> 7) & 0xFFu) - 127 - 14;
          sh = sh < -100 ? -100 : (sh > 100 ? 100 : sh);
          qscale[qt] = p.scale_log2 * __int_as_float((127 + sh) << 23);      // scale_log2 * 2^sh
        }
      }
    } else {
      // NVFP4 query, rounded by the prepare kernel (this kernel's predecessor): the codes form the B operand of
      // the block-scaled logits (two K-halves of [64 heads x 128 bytes], 128-byte swizzle), the scale bytes go
      // to tensor memory, and the head's power of two goes into its softmax scale
      griddep_wait();
      const uint8_t* qsrc = p.q4_codes + u.unit * 64 * 256;
      for (int i = qt; i < 64 * 16; i += kQThreads) {
        const int n = i >> 4, j = i & 15, cc = j & 7;
        *reinterpret_cast<uint4*>(smem + kQ4Off + (j >> 3) * (kHeadsPad * 128) + n * 128 + ((cc ^ (n & 7)) << 4)) =
            ld_nc_v4(qsrc + i * 16);
      }
      if (qt < 64) qscale[qt] = p.scale_log2 * __ldg(p.q4_mult + u.unit * 64 + qt);
      if (warp < 4) {
        // query scale factors: head n's four bytes of product s at lane 32 j + n % 32 (every subpartition j
        // holds a copy; warp w writes subpartition w), column kColSFB + 4 s + n / 32
        const uint32_t lb = (uint32_t)(warp * 32) << 16;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t sc[8];
          ld_nc_v8(p.q4_sc + (u.unit * 64 + lane + 32 * c) * 32, sc);
#pragma unroll
          for (int s8 = 0; s8 < 8; ++s8) tc::st_32x1(tbase + lb + kColSFB + 4 * s8 + c, sc[s8]);
        }
        tc::wait_st();
      }
    }
    if (qt < 64) msh[qt] = -INFINITY;
    tc::fence_proxy_async();
    tc::fence_before();
    asm volatile("bar.sync 2, %0;" :: "n"(kThreads) : "memory");
    tc::fence_after();
    if (is_conv) {
      griddep_wait();                                // the index list comes from the kernel before
      id_c = n_cache > 0 ? cache_id(p, u, c0, row) : -1;
      id_n = n_cache > 1 ? cache_id(p, u, c0 + 1, row) : -1;
      id_nn = n_cache > 2 ? cache_id(p, u, c0 + 2, row) : -1;
      const bool ok0 = n_cache > 0 && cache_ok(u, id_c, row);
      if (ok0) {
        const uint8_t* e = seq + (int64_t)id_c * kLatBlk + (row & 7) * 256 + hp * 32;
        ld_nc_v8(e, q0);
        ld_nc_v8(e + 64, q1);
      }
      load_scales(seq, id_c, ok0, row, hp, sc_c);
      load_scales(seq, id_n, n_cache > 1 && cache_ok(u, id_n, row), row, hp, sc_n);
      qs0 = sc_c[0];
      qs1 = sc_c[1];
      // NVFP4-query mode: the key scale factors of the first tile (a later tile's are written while the tile
      // before it is converted)
      if (kQ4 && n_tiles > 0) {
        uint32_t sw[4] = {sc_c[0], sc_c[1], sc_c[2], sc_c[3]};
        if (nw > 0) load_window_scales(p, u, 0, row, hp, sw);
        put_key_scales(tbase, sp, hp, lane, 0, sw, bars);
      }
    }
  } else {
    // the gather warp starts its L2 prefetches once the queries have arrived, so that the queries and the
    // first tile's bytes (loaded by the converters) are not queued behind the later tiles
    asm volatile("bar.sync 2, %0;" :: "n"(kThreads) : "memory");
  }

  if (warp == kGatherWarp) {
    // ---------------- gather: block-id checks, L2 prefetch, later window tiles ----------------
    griddep_wait();
    // the blocks of cache tile k go to L2 when the converters start tile k - 3 (tiles 1 and 2 at once; the
    // converters load tile 0 themselves, so its ids are only checked); lanes 0-15 take one block each.
    // The pacing is a hint: a wait that runs out (or a CTA that gives up) just prefetches at once.
    volatile int* progress = flag + 4;
    for (int k = 0; k < n_cache; ++k) {
      const int target = nw + k - 3;
      for (uint32_t i = 0; k >= 3 && i < p.spin_limit && *progress < target && !*abort_flag; ++i) __nanosleep(64);
      const int slot = (c0 + k) * kTileBlocks + lane;
      if (lane < kTileBlocks && slot < p.top_k) {
        const int64_t id = __ldg(p.idx + u.unit * p.top_k + slot);
        if (id < -1 || id >= u.nb_cap) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_ATTN, (uint32_t)u.unit);
        if (k > 0 && id >= 0 && id < u.n_b) prefetch_l2(seq + id * kLatBlk, kLatBlk);
      }
    }
    if (lane == 0) {
      for (int tw = 1; tw < nw; ++tw) {
        const int64_t y0 = window_row0(p, u, tw);
        if (y0 < 0 || y0 + kRows > p.swa_rows) continue;
        for (int pp = 0; pp < kPanels; ++pp) prefetch_l2_3d(&swa_map, pp * 64, (int)y0, (int)u.b);
      }
      int copied = nw > 0 ? 1 : 0;
      for (int tw = 1; tw < nw; ++tw) {
        // the values buffer holds the previous tile until its value products are done
        bool ok = true;
        for (int c = 0; c < kChunks && ok; ++c) ok = wait_bar(&bars[V_EMPTY + c], (tw - 1) & 1, abort_flag, p.hdr, 9, p.spin_limit);
        if (!ok) break;
        copy_window_tile(p, u, tw, smem, &swa_map, &bars[WIN_FULL]);
        ++copied;
      }
      // no copy into this CTA's shared memory may still be in flight when it exits
      if (copied > 0) drain_bar(&bars[WIN_FULL], (copied - 1) & 1);
    }
  } else if (is_conv) {
    // ---------------- converters: one 64-column panel of every chunk of every tile ----------------
    volatile int* progress = flag + 4;
    bool stop = false;
    for (int it = 0; it < n_tiles && !stop; ++it) {
      if (warp == kConv0 && lane == 0) *progress = it;
      const bool win = it < nw;
      // NVFP4-query mode: the converters set the tile cadence and usually find the previous tile's value
      // products long complete; they complete in issue order, so one test of the last chunk's barrier stands in
      // for the four per-chunk waits
      bool prev_done = kQ4 && !win && it > 0 &&
                       __all_sync(0xffffffffu, mbar_test_wait(smem_addr(&bars[V_EMPTY + kChunks - 1]), (it - 1) & 1));
      const int k = it - nw;                       // cache tile index within this CTA
      bool vr = false;
      if (win) {
        bool oob;
        vr = window_row(p, u, it, row, &oob);
        if (oob && hp == 0) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_ATTN, (uint32_t)u.unit);
        if (!__all_sync(0xffffffffu, wait_bar(&bars[WIN_FULL], it & 1, abort_flag, p.hdr, 10, p.spin_limit))) break;
        // NVFP4-query mode: the next tile's key scale factors, one tile ahead
        if (kQ4 && it + 1 < n_tiles) {
          uint32_t sw[4] = {sc_c[0], sc_c[1], sc_c[2], sc_c[3]};
          if (it + 1 < nw) load_window_scales(p, u, it + 1, row, hp, sw);
          put_key_scales(tbase, sp, hp, lane, it + 1, sw, bars);
        }
      }
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c) {
        const int pnl = 2 * c + hp;
        uint8_t* vrow = smem + kVOff + c * kChunkBytes + hp * kHalfBytes + (row >> 3) * 1024 + (row & 7) * 128;
        uint32_t h[32];
        if (win) {
          // bf16 -> fp16 of this row's 64 columns, in place; rows that are not attended become zero. A value
          // beyond the fp16 range (|x| > 65504, outside the call's contract) becomes infinite: reported.
          uint32_t inf = 0u;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 x = *reinterpret_cast<const uint4*>(vrow + ((j ^ (row & 7)) << 4));
            h[4 * j] = vr ? bf2_to_h2(x.x) : 0u; h[4 * j + 1] = vr ? bf2_to_h2(x.y) : 0u;
            h[4 * j + 2] = vr ? bf2_to_h2(x.z) : 0u; h[4 * j + 3] = vr ? bf2_to_h2(x.w) : 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e)
              inf |= ((h[4 * j + e] & 0x7C00u) == 0x7C00u) | ((h[4 * j + e] & 0x7C000000u) == 0x7C000000u);
          }
          if (inf) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_ATTN, (uint32_t)u.unit);
        } else {
          dequant_panel(q0, qs0, h);
#pragma unroll
          for (int i = 0; i < 8; ++i) { q0[i] = q1[i]; q1[i] = 0u; }
          qs0 = qs1;
          qs1 = 0u;
          // the panel two places further on enters at the back of the queue
          const bool same = c + 2 < kChunks;
          const int id2 = same ? id_c : id_n;
          if (cache_ok(u, id2, row)) {
            ld_nc_v8(seq + (int64_t)id2 * kLatBlk + (row & 7) * 256 + (same ? pnl + 4 : pnl - 4) * 32, q1);
            qs1 = same ? pick4(sc_c, c + 2) : pick4(sc_n, c - 2);
          }
        }
        // values operand: the chunk must have been consumed by the previous tile's value products (a window
        // tile's chunks were, before its copy was issued)
        if (!win && it > 0 && !prev_done &&
            !__all_sync(0xffffffffu, wait_bar(&bars[V_EMPTY + c], (it - 1) & 1, abort_flag, p.hdr, 6, p.spin_limit))) {
          stop = true;
          break;
        }
        // NVFP4-query mode: the next cache tile's key scale factors go in once the value products of tile it - 1
        // have begun to free this tile's buffer (its logits, the last reader of that scale buffer, are complete)
        if (kQ4 && !win && c == 0 && it + 1 < n_tiles) put_key_scales(tbase, sp, hp, lane, it + 1, sc_n, bars);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(vrow + ((j ^ (row & 7)) << 4)) = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
        // publish the chunk to the value products; in NVFP4-query mode, where the converters set the cadence,
        // two chunks at a time (one proxy fence and round of arrivals per pair)
        if (!kQ4 || (c & 1)) {
          tc::fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            if (kQ4) mbar_arrive(&bars[V_FULL + c - 1]);
            mbar_arrive(&bars[V_FULL + c]);
          }
        }
      }
      if (!win) {
        // the scales of tile k + 2 are loaded a tile before the queue reaches it, its id one more tile earlier
#pragma unroll
        for (int i = 0; i < 4; ++i) sc_c[i] = sc_n[i];
        load_scales(seq, id_nn, k + 2 < n_cache && cache_ok(u, id_nn, row), row, hp, sc_n);
        id_c = id_n;
        id_n = id_nn;
        id_nn = k + 3 < n_cache ? cache_id(p, u, c0 + k + 3, row) : -1;
      }
    }
  } else if (kQ4 && warp == kLogitsWarp) {
    // ---------------- NVFP4-query logits: S^T(t) = C . Q4^T by block-scaled FP4 products ----------------
    // Each tile's FP4 keys are copied by tensor map into the raw stage once the previous tile's logits are
    // complete: a cache tile as 16 blocks (two [8 x 128-byte] boxes each, 8-row groups 2,048 bytes apart), a
    // window tile from the rounded window rows (two [128 x 128-byte] boxes, 8-row groups 1,024 bytes apart).
    // The key scale factors come from the converters, one tile ahead, so the logits never wait for the
    // values buffer.
    griddep_wait();                                  // the index list and the rounded window rows
    bool ok = true;
    int raw_issued = 0;
    int nid = (n_cache > 0 && lane < kTileBlocks) ? cache_id(p, u, c0, lane << 3) : -1;
    for (int it = 0; it < n_tiles && ok; ++it) {
      const int sb = it & 1;
      const bool win = it < nw;
      if (it > 0 && !wait_bar_warp(&bars[RAW_DONE], (it - 1) & 1, abort_flag, p.hdr, 14, p.spin_limit)) break;
      if (lane == 0) mbar_arrive_expect_tx(&bars[RAW_FULL], kRawBytes);
      __syncwarp();
      if (win) {
        if (lane == 0) {
          const int64_t y0 = window_row0(p, u, it);
          const int y = (int)(y0 < -(int64_t)kRows ? -kRows : (y0 > p.swa_rows ? p.swa_rows : y0));
          tma_load_3d(smem + kRawOff, &win4_map, 0, y, (int)u.b, &bars[RAW_FULL]);
          tma_load_3d(smem + kRawOff + kRawBytes / 2, &win4_map, 128, y, (int)u.b, &bars[RAW_FULL]);
        }
      } else {
        const int k = it - nw;
        if (lane < kTileBlocks) {
          uint8_t* dst = smem + kRawOff + lane * 2048;
          tma_load_4d(dst, &cache_map, 0, 0, nid, (int)u.b, &bars[RAW_FULL]);
          tma_load_4d(dst + 1024, &cache_map, 128, 0, nid, (int)u.b, &bars[RAW_FULL]);
        }
        nid = (k + 1 < n_cache && lane < kTileBlocks) ? cache_id(p, u, c0 + k + 1, lane << 3) : -1;
      }
      ++raw_issued;
      if (!wait_bar_warp(&bars[RAW_FULL], it & 1, abort_flag, p.hdr, 15, p.spin_limit)) break;
      if (!wait_bar_warp(&bars[SFX_FULL + sb], (it >> 1) & 1, abort_flag, p.hdr, 16, p.spin_limit)) break;
      if (it >= 2 && !wait_bar_warp(&bars[S_EMPTY + sb], ((it - 2) >> 1) & 1, abort_flag, p.hdr, 4, p.spin_limit)) break;
      tc::fence_after();
      const uint32_t d = tbase + kColS + 64 * sb;
      const uint32_t half_off = win ? kRawBytes / 2 : 1024, sbo = win ? 1024 : 2048;
#pragma unroll
      for (int s8 = 0; s8 < 8; ++s8) {
        const uint64_t a = tc::smem_desc(s_base + kRawOff + (s8 >> 2) * half_off + (s8 & 3) * 32, 16, sbo,
                                         tc::kSwizzle128B);
        const uint64_t b = tc::smem_desc(s_base + kQ4Off + (s8 >> 2) * (kHeadsPad * 128) + (s8 & 3) * 32, 16, 1024,
                                         tc::kSwizzle128B);
        tc::mma_mxf4_warp(d, a, b, kIdescS4, tbase + kColSFA + 32 * sb + 4 * s8, tbase + kColSFB + 4 * s8, s8 > 0 ? 1u : 0u);
      }
      tc::commit_warp(&bars[S_FULL + sb]);
      tc::commit_warp(&bars[RAW_DONE]);
    }
    // every MMA issued must be complete before the tensor memory is released, and no copy may still be in
    // flight into this CTA's shared memory when it exits
    tc::commit_warp(&bars[FIN_L]);
    drain_bar(&bars[FIN_L], 0);
    if (raw_issued > 0) drain_bar(&bars[RAW_FULL], (raw_issued - 1) & 1);
    __syncwarp();
  } else if (warp == kLogitsWarp) {
    // ---------------- logits MMA issue: S^T(t) = C . Q^T into S buffer t & 1 ----------------
    const uint32_t q_addr = s_base + kQOff;
    bool ok = p.qh == nullptr || wait_bar_warp(&bars[Q_FULL], 0, abort_flag, p.hdr, 17, p.spin_limit);
    for (int it = 0; it < n_tiles && ok; ++it) {
      const int sb = it & 1;
      if (it >= 2 && !wait_bar_warp(&bars[S_EMPTY + sb], ((it - 2) >> 1) & 1, abort_flag, p.hdr, 4, p.spin_limit)) break;
      const uint32_t d = tbase + kColS + 64 * sb;
      for (int c = 0; c < kChunks; ++c) {
        if (!wait_bar_warp(&bars[V_FULL + c], it & 1, abort_flag, p.hdr, 4, p.spin_limit)) { ok = false; break; }
        tc::fence_after();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int pnl = 2 * c + hh;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t a = tc::smem_desc(s_base + kVOff + c * kChunkBytes + hh * kHalfBytes + ks * 32, 16, 1024,
                                             tc::kSwizzle128B);
            const uint64_t bq = tc::smem_desc(q_addr + pnl * kQPanel + ks * 32, 16, 1024, tc::kSwizzle128B);
            tc::mma_f16_warp(d, a, bq, kIdescS, (pnl | ks) != 0);
          }
        }
      }
      if (ok) tc::commit_warp(&bars[S_FULL + sb]);
    }
    // every MMA issued must be complete before the tensor memory is released, and the query copy must have
    // landed before the CTA exits
    tc::commit_warp(&bars[FIN_L]);
    drain_bar(&bars[FIN_L], 0);
    if (p.qh != nullptr) drain_bar(&bars[Q_FULL], 0);
    __syncwarp();
  } else if (warp == kValuesWarp) {
    // ---------------- values MMA issue: O^T += C^T . P^T, chunk by chunk ----------------
    const uint32_t v_addr = s_base + kVOff;
    for (int it = 0; it < n_tiles; ++it) {
      const int pb = it & 1;
      const uint32_t p_addr = s_base + kPOff + pb * kPBytes;
      if (!wait_bar_warp(&bars[P_FULL + pb], (it >> 1) & 1, abort_flag, p.hdr, 5, p.spin_limit)) break;
      tc::fence_after();
      bool ok = true;
      for (int c = 0; c < kChunks; ++c) {
        if (!wait_bar_warp(&bars[V_FULL + c], it & 1, abort_flag, p.hdr, 6, p.spin_limit)) { ok = false; break; }
        tc::fence_after();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint64_t a = tc::smem_desc(v_addr + c * kChunkBytes + j * 2048, kHalfBytes, 1024, tc::kSwizzle128B);
          const uint64_t bp = tc::smem_desc(p_addr + j * 2048, 8192, 1024, tc::kSwizzle128B);
          tc::mma_f16_warp(tbase + kColO + 64 * c, a, bp, kIdescPV, (it > 0 || j > 0) ? 1u : 0u);
        }
        tc::commit_warp(&bars[V_EMPTY + c]);
      }
      if (!ok) break;
      if (!(p.fault == CSA_FAULT_WITHHOLD_ARRIVAL && it == 0)) tc::commit_warp(&bars[P_EMPTY + pb]);
    }
    tc::commit_warp(&bars[FIN_V]);
    drain_bar(&bars[FIN_V], 0);
    __syncwarp();
  } else if (warp == kSumWarp) {
    // ---------------- row sums: l += sum over the tile's rows of P (lane = heads 2 lane, 2 lane + 1) ----
    float l0 = 0.0f, l1 = 0.0f;
    const int h0 = 2 * lane;
    for (int it = 0; it < n_tiles; ++it) {
      const int pb = it & 1;
      if (!wait_bar_warp(&bars[P_FULL + pb], (it >> 1) & 1, abort_flag, p.hdr, 13, p.spin_limit)) break;
      if (flag[pb]) {
        // the softmax raised the reference maxima for this tile: rescale like O
        l0 *= alpha[64 * pb + h0];
        l1 *= alpha[64 * pb + h0 + 1];
      }
      const uint8_t* pbuf = smem + kPOff + pb * kPBytes + (lane & 3) * 4;
      float a0 = 0.0f, a1 = 0.0f, b0 = 0.0f, b1 = 0.0f;
#pragma unroll 8
      for (int r = 0; r < kRows; r += 2) {
        const uint32_t x = *reinterpret_cast<const uint32_t*>(pbuf + r * 128 + (((lane >> 2) ^ (r & 7)) << 4));
        const uint32_t y = *reinterpret_cast<const uint32_t*>(pbuf + (r + 1) * 128 + (((lane >> 2) ^ ((r + 1) & 7)) << 4));
        const float2 fx = __half22float2(*reinterpret_cast<const __half2*>(&x));
        const float2 fy = __half22float2(*reinterpret_cast<const __half2*>(&y));
        a0 += fx.x; a1 += fx.y; b0 += fy.x; b1 += fy.y;
      }
      l0 += a0 + b0;
      l1 += a1 + b1;
      if (it == n_tiles - 1) {
        lsh[h0] = l0;
        lsh[h0 + 1] = l1;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[P_EMPTY + pb]);
    }
  } else {
    // ---------------- softmax (warps 0-3, thread = tile row) ----------------
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float* qsc = reinterpret_cast<const float*>(smem + kQScaleOff);
    bool ok = true;
    griddep_wait();
    griddep_launch();
    int64_t sid_nxt = n_cache > 0 ? cache_id(p, u, c0, row) : -1;
    for (int it = 0; it < n_tiles; ++it) {
      const int sb = it & 1;
      bool valid;
      if (it < nw) {
        bool oob;
        valid = window_row(p, u, it, row, &oob);
      } else {
        valid = cache_ok(u, sid_nxt, row);
        sid_nxt = it - nw + 1 < n_cache ? cache_id(p, u, c0 + it - nw + 1, row) : -1;
      }
      if (!all_softmax(wait_bar(&bars[S_FULL + sb], (it >> 1) & 1, abort_flag, p.hdr, 7, p.spin_limit))) { ok = false; break; }
      tc::fence_after();
      // P buffer sb, alpha[sb] and flag[sb] were last read by the value products and row sums of tile it - 2
      if (it >= 2 && !all_softmax(wait_bar(&bars[P_EMPTY + sb], ((it - 2) >> 1) & 1, abort_flag, p.hdr, 12, p.spin_limit))) {
        ok = false;
        break;
      }
      float* al = alpha + 64 * sb;
      const uint32_t s_col = tbase + lane_base + kColS + 64 * sb;
      uint8_t* prow = smem + kPOff + sb * kPBytes + row * 128;
      // Probabilities against the current reference maxima, 32 heads at a time, written to row `row` of P
      // (fp16, MN-major: 64 heads contiguous, 128-byte swizzle). When a probability would exceed 2^8 (a
      // maximum moved by more than the slack, or none was set yet), the maxima are raised and the same loop
      // runs once more; after a raise every probability is at most 2^8, so there is no third pass.
      if (tid == 0) flag[sb] = 0;
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        // on the CTA's first tile every reference maximum is still -inf, so a first pass could only report an
        // overflow: it goes straight to the maxima (a tile without attended rows then leaves them at -inf and
        // the second pass writes zeros, as the first would have)
        const bool first = it == 0 && pass == 0;
        bool over = first;
#pragma unroll 1
        for (int half = 0; half < 2 && !first; ++half) {
          uint32_t sr[32];
          tc::ld_32x32(s_col + 32 * half, sr);
          tc::wait_ld();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 ma = *reinterpret_cast<const float4*>(msh + 32 * half + 8 * c);
            const float4 mb = *reinterpret_cast<const float4*>(msh + 32 * half + 8 * c + 4);
            const float mm[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
            const float4 sa = *reinterpret_cast<const float4*>(qsc + 32 * half + 8 * c);
            const float4 sbb = *reinterpret_cast<const float4*>(qsc + 32 * half + 8 * c + 4);
            const float ss[8] = {sa.x, sa.y, sa.z, sa.w, sbb.x, sbb.y, sbb.z, sbb.w};
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int h = 8 * c + 2 * k;
              // the scaled logit is rounded before the maximum is subtracted, as it was when the maximum was
              // taken, so the largest row gives exactly 2^0 at any magnitude (a fused multiply-add would leave
              // the product's rounding error in the exponent, which overflows for logits beyond 2^27)
              const float p0 = valid ? ex2(__fmul_rn(__uint_as_float(sr[h]), ss[2 * k]) - mm[2 * k]) : 0.0f;
              const float p1 = valid ? ex2(__fmul_rn(__uint_as_float(sr[h + 1]), ss[2 * k + 1]) - mm[2 * k + 1]) : 0.0f;
              over |= !(p0 <= kMaxProb) || !(p1 <= kMaxProb);
              w[k] = f2_to_h2(p0, p1);
            }
            const int pc = 4 * half + c;
            *reinterpret_cast<uint4*>(prow + ((pc ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        if (pass == 1 || !any_softmax(over)) break;
        // per-head maximum over the warp's 32 rows, 32 heads at a time, by a transposing reduction: at
        // the step with offset o a lane keeps the half of its values selected by (lane & o) and takes the
        // maximum with its partner's copy of that half, so after five steps lane l holds head 32 half + l
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t sr[32];
          tc::ld_32x32(s_col + 32 * half, sr);
          tc::wait_ld();
          float v[32];
#pragma unroll
          for (int h = 0; h < 32; ++h) v[h] = valid ? __fmul_rn(__uint_as_float(sr[h]), qsc[32 * half + h]) : -INFINITY;
#pragma unroll
          for (int n = 16, o = 16; n >= 1; n >>= 1, o >>= 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < n; ++i) {
              const float keep = up ? v[n + i] : v[i];
              const float give = up ? v[i] : v[n + i];
              v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, o));
            }
          }
          red[warp * 64 + 32 * half + lane] = v[0];
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (tid < 64) {
          const float tm = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
          const float mo = msh[tid];
          float mn = mo;
          if (tm > mo + kRescaleSlack) mn = tm;
          al[tid] = (mo == -INFINITY || mn == mo) ? 1.0f : exp2f(mo - mn);
          if (mn != mo && mo != -INFINITY) flag[sb] = 1;
          msh[tid] = mn;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (flag[sb]) {
          // every value product before this tile must be complete before O is rescaled (the ones of tile
          // it - 1 complete last: the values are issued in tile order); the row-sum warp rescales l itself
          if (it > 0) {
            if (!all_softmax(wait_bar(&bars[P_EMPTY + ((it - 1) & 1)], ((it - 1) >> 1) & 1, abort_flag, p.hdr, 12, p.spin_limit))) {
              ok = false;
              break;
            }
            tc::fence_after();
          }
          // raise the reference maximum of the accumulated O (32 columns = 32 heads at a time)
#pragma unroll 1
          for (int k = 0; k < 8; ++k) {
            uint32_t o[32];
            tc::ld_32x32(tbase + lane_base + kColO + 32 * k, o);
            tc::wait_ld();
            const float* ak = al + 32 * (k & 1);
#pragma unroll
            for (int h = 0; h < 32; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * ak[h]);
            tc::st_32x32(tbase + lane_base + kColO + 32 * k, o);
          }
          tc::wait_st();
        }
      }
      if (!ok) break;
      // S buffer sb has been read for the last time: the logits of tile it + 2 may overwrite it
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[S_EMPTY + sb]);
      tc::fence_proxy_async();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[P_FULL + sb]);
    }
    // ---------------- epilogue ----------------
    const int last = n_tiles - 1;
    const bool have = all_softmax(ok && n_tiles > 0 &&
                                  wait_bar(&bars[P_EMPTY + (last & 1)], (last >> 1) & 1, abort_flag, p.hdr, 8, p.spin_limit));
    tc::fence_after();
    // the row sums, one per head, written by the row-sum warp before its last arrival on P_EMPTY
    if (!have && tid < 64) lsh[tid] = 0.0f;
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const int64_t prow_base = (u.unit * p.splits + split) * H;
    if (tid == 0) flag[3] = have ? 1 : 0;
    if (p.splits == 1) {
      // 1 / l per head, over red (whose last use was the last tile's softmax)
      if (tid < 64) red[tid] = lsh[tid] > 0.0f ? 1.0f / lsh[tid] : 0.0f;
      asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll 1
      for (int k = 0; k < 8; ++k) {
        uint32_t o[32];
        if (have) {
          tc::ld_32x32(tbase + lane_base + kColO + 32 * k, o);
          tc::wait_ld();
        } else {
#pragma unroll
          for (int h = 0; h < 32; ++h) o[h] = 0u;
        }
        const int d = 128 * (k >> 1) + tid;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int h = 32 * (k & 1) + j;
          if (h >= H) break;
          p.out[(u.unit * H + h) * (int64_t)kLatent + d] = __uint_as_float(o[j]) * red[h];
        }
      }
      if (tid < H && p.out_lse != nullptr) {
        const float l = lsh[tid];
        p.out_lse[u.unit * H + tid] = l > 0.0f ? (msh[tid] + log2f(l)) * kLn2 : -INFINITY;
      }
    } else if (tid < H) {
      *reinterpret_cast<float2*>(p.part_ml + (prow_base + tid) * 2) = make_float2(have ? msh[tid] : -INFINITY, lsh[tid]);
    }
    tc::fence_before();
  }

  if (p.splits > 1) {
    // ---------------- this split's unnormalised o, written by all warps ----------------
    // Every product has completed (the softmax saw the last values finish). Warp w reads tensor-memory
    // subpartition w % 4 (latent column 32 (w % 4) + lane of each 128-column chunk), 32-column pieces
    // 2 (w / 4) and 2 (w / 4) + 1.
    __syncwarp();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const bool had = flag[3] != 0;
    const int64_t prow_base = (u.unit * p.splits + split) * H;
    {
      const uint32_t sp_base = (uint32_t)((warp & 3) * 32) << 16;
#pragma unroll 1
      for (int k = 2 * (warp >> 2); k < 2 * (warp >> 2) + 2; ++k) {
        uint32_t o[32];
        if (had) {
          tc::ld_32x32(tbase + sp_base + kColO + 32 * k, o);
          tc::wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = 0u;
        }
        const int d = 128 * (k >> 1) + 32 * (warp & 3) + lane;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int h = 32 * (k & 1) + j;
          if (h < H) p.part_o[(prow_base + h) * kLatent + d] = __uint_as_float(o[j]);
        }
      }
    }
  }
  __syncthreads();
  tc::fence_after();
  if (warp == kLogitsWarp) tc::dealloc(tbase, kTmemCols);
}

// out[u][h] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s, splits in order; lse = (M + log2 L) ln 2.
// One block per (unit, head), thread = 4 latent columns. The splits are read eight at a time, the (m, l)
// pairs and the o slices of a batch all issued before the first use; a later batch with a larger maximum
// rescales what the earlier batches added up (at most eight splits need no rescale).
__global__ void __launch_bounds__(128) combine_kernel(AttnParams p) {
  constexpr int kBatch = 8;
  griddep_wait();                                  // the partials come from the kernel before
  griddep_launch();
  const int64_t row = blockIdx.x;                 // unit * H + h
  const int64_t unit = row / p.heads;
  const int h = (int)(row % p.heads);
  const int S = p.splits, H = p.heads;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + unit * S * H + h;
  const float4* po = reinterpret_cast<const float4*>(p.part_o) + (unit * S * H + h) * (int64_t)(kLatent / 4) + threadIdx.x;
  float M = -INFINITY, L = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < S; s0 += kBatch) {
    float2 x[kBatch];
    float4 v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      x[i] = make_float2(-INFINITY, 0.0f);
      v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s0 + i < S) {
        x[i] = ml[(s0 + i) * H];
        v[i] = po[(int64_t)(s0 + i) * H * (kLatent / 4)];
      }
    }
    float Mb = M;
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (x[i].y > 0.0f) Mb = fmaxf(Mb, x[i].x);
    if (Mb == -INFINITY) continue;
    if (Mb != M && M != -INFINITY) {
      const float r = exp2f(M - Mb);
      acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
      L *= r;
    }
    M = Mb;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (!(x[i].y > 0.0f)) continue;
      const float w = exp2f(x[i].x - M);
      acc.x += w * v[i].x; acc.y += w * v[i].y; acc.z += w * v[i].z; acc.w += w * v[i].w;
      L += w * x[i].y;
    }
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  reinterpret_cast<float4*>(p.out)[row * (kLatent / 4) + threadIdx.x] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (threadIdx.x == 0 && p.out_lse != nullptr) p.out_lse[row] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_attn(const AttnParams& p, cudaStream_t s, bool pdl) {
  if (p.units == 0) return cudaSuccess;
  // window rows as a [batch][swa_rows][512] bf16 tensor, copied in [1 x 128 x 64] boxes with the
  // 128-byte swizzle of the kernel's panels; rows outside the tensor read as zero
  CUtensorMap map;
  std::memset(&map, 0, sizeof(map));
  if (p.n_wt > 0) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)kLatent, (cuuint64_t)p.swa_rows, (cuuint64_t)(p.units / p.n_query)};
    const cuuint64_t strides[2] = {(cuuint64_t)kLatent * 2, (cuuint64_t)p.swa_stride_b * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)kRows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(p.swa), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  // NVFP4-query mode: the cache's code bytes as a [batch][block][slot][256] byte tensor (block stride 2,304,
  // the scale bytes after each block's codes are skipped), copied in [8 x 128] boxes, one half of each of a
  // block's 8 rows, with the 128-byte swizzle of the block-scaled operand; ids outside the tensor read as zero
  CUtensorMap cmap;
  std::memset(&cmap, 0, sizeof(cmap));
  if (p.q4) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    const int64_t nb_cap = (p.max_entries + kBlockEntries - 1) / kBlockEntries;
    const int64_t batch = p.units / p.n_query;
    const cuuint64_t dims[4] = {256, (cuuint64_t)kBlockEntries, (cuuint64_t)(nb_cap > 0 ? nb_cap : 1), (cuuint64_t)batch};
    const int64_t sb = batch > 1 ? p.cache_stride_b : (nb_cap > 0 ? nb_cap : 1) * kLatBlk;
    const cuuint64_t strides[3] = {256, (cuuint64_t)kLatBlk, (cuuint64_t)sb};
    const cuuint32_t box[4] = {128, (cuuint32_t)kBlockEntries, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = enc(&cmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(p.cache), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  // NVFP4-query mode: the window rows rounded by the prepare kernel as a [batch][swa_rows][256] byte tensor,
  // copied in [128 x 128] boxes (one half of each of a window tile's rows) with the 128-byte swizzle; rows
  // outside the tensor read as zero
  CUtensorMap wmap;
  std::memset(&wmap, 0, sizeof(wmap));
  if (p.q4 && p.n_wt > 0) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {256, (cuuint64_t)p.swa_rows, (cuuint64_t)(p.units / p.n_query)};
    const cuuint64_t strides[2] = {256, (cuuint64_t)p.swa_rows * 256};
    const cuuint32_t box[3] = {128, (cuuint32_t)kRows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, p.w4, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  // exact attention with prepared queries: [units][64][512] fp16, copied in [1 x 64 x 64] boxes (one panel of
  // 64 latent columns for the 64 head rows) with the 128-byte swizzle of the query panels
  CUtensorMap qmap;
  std::memset(&qmap, 0, sizeof(qmap));
  if (p.qh != nullptr) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)kLatent, 64, (cuuint64_t)p.units};
    const cuuint64_t strides[2] = {(cuuint64_t)kLatent * 2, (cuuint64_t)64 * kLatent * 2};
    const cuuint32_t box[3] = {64, 64, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, p.qh, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  ProfScope prof("sparse_attn", s);
  clear_stale_error();
  if (p.q4) {
    cudaError_t e = ensure_smem_limit(attn_tc_kernel<true>, kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_ex(attn_tc_kernel<true>, dim3((unsigned)p.splits, (unsigned)p.units), dim3(kThreads),
                     (size_t)kSmemBytes, s, pdl, p, map, cmap, wmap, qmap);
  }
  cudaError_t e = ensure_smem_limit(attn_tc_kernel<false>, kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_ex(attn_tc_kernel<false>, dim3((unsigned)p.splits, (unsigned)p.units), dim3(kThreads),
                   (size_t)kSmemBytes, s, pdl, p, map, cmap, wmap, qmap);
}

cudaError_t launch_attn_prep(const AttnParams& p, cudaStream_t s, bool pdl) {
  if (p.units == 0) return cudaSuccess;
  const int64_t rows = p.units * 64 + (p.q4 && p.window > 0 ? (p.units / p.n_query) * p.swa_rows : 0);
  ProfScope prof("attn_prep", s);
  clear_stale_error();
  return launch_ex(attn_prep_kernel, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, s, pdl, p);
}

cudaError_t launch_combine(const AttnParams& p, cudaStream_t s, bool pdl) {
  if (p.units == 0 || p.splits == 1) return cudaSuccess;
  ProfScope prof("attn_combine", s);
  clear_stale_error();
  return launch_ex(combine_kernel, dim3((unsigned)(p.units * p.heads)), dim3(128), 0, s, pdl, p);
}

}  // namespace csa
