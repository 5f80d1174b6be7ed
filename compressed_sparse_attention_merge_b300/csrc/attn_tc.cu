// Sparse attention over selected FP4 cache blocks merged with the sliding window, on the fifth-generation
// tensor cores (tcgen05), split over the row list, plus the fixed-order log-sum-exp combine of the splits.
//
// Follows "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression" (paper-digest), Core
// Mechanics ("one 512-dim latent shares keys and values across all attention heads") and Terminology
// (sliding window of 128), and "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (card),
// Key ideas ("Every layer keeps its own query and sliding-window KV").
//
// Design. A CTA owns one query (all heads) and some 128-row tiles of its row list: a range of cache
// tiles (16 selected blocks each) and/or the window tiles. Because one latent row c is both key and
// value, both products are taken with the rows as the 128-wide M side and the heads as N:
//   S^T [rows x heads]  = C [rows x 512] . Q^T                   (logits)
//   O^T [512 x heads]  += C^T [512 x rows] . P^T [rows x heads]  (values)
// S and O accumulate in tensor memory; the row sums l are added up by one warp from the fp16
// probabilities in shared memory (the same values the tensor core multiplies).
//   Cache tiles: the gather warp copies the 16 raw FP4 blocks (36 KB) with cp.async.bulk into one of three
//   raw stages. Two groups of four warps dequantise every tile: group A writes the logits operand
//   straight into tensor memory (thread = row, 64-column panels, a four-panel ring); group B
//   writes the values operand into a two-slot shared-memory ring of [128 latent x 64 row] units in the
//   128-byte-swizzled MN-major layout.
//   Window tiles: a tensor-map copy (TMA, 128-byte swizzle) lands the 128 bf16 rows in panel layout over
//   the raw and ring areas; they are converted to fp16 in place and serve both products.
// Pipelining: S is double-buffered in tensor memory and the logits and the values have separate issuing
// threads, so that the logits of tile t+1 run while the softmax of tile t works; the softmax of tile t+1
// computes its probabilities while the values of tile t run and writes them once those have read P. A
// third raw stage lets the copy of tile t+2 start while tile t's values operand is still being built.
//
// Warp roles: 0-3 softmax and epilogue (thread = tile row), 4-7 group A, 8-11 group B, 12 gather,
// 13 logits MMA issue and tensor-memory allocation, 14 values MMA issue, 15 row sums. The softmax keeps,
// per head, a reference maximum that is raised only when a tile's maximum exceeds it by more than 8 (in
// log2 units), so the probabilities stay below 2^8 and the accumulators are rescaled rarely. Splits write
// unnormalised partials (o, m, l); the combine kernel merges them in split order. When the splits of a
// unit form one thread-block cluster, each CTA stages its (o, m, l) in its own shared memory instead and
// CTA r merges latent columns [512 r / S, 512 (r + 1) / S) of every split, in split order, through
// distributed shared memory.
#include <cuda.h>

#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "csa_internal.cuh"
#include "tc.cuh"

namespace csa {
namespace {

constexpr int kRows = 128;                                 // rows per tile: M of both products
constexpr int kTileBlocks = kRows / kBlockEntries;         // 16 cache blocks per tile
constexpr int kHeadsPad = 64;                              // N of both products (heads, zero-padded)
constexpr int kPanels = kLatent / 64;                      // 8 panels of 64 latent columns
constexpr int kLatBlk = block_bytes(kLatent);              // 2304
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.0f;                      // log2 headroom before the reference max moves
constexpr float kMaxProb = 256.0f;                         // 2^kRescaleSlack

// shared-memory map (bytes); the operand regions start on 1024-byte boundaries
constexpr int kQPanel = kHeadsPad * 128;                   // 8 KB
constexpr int kQOff = 0;                                   // queries: 8 K-major panels, 64 KB
constexpr int kPBytes = kRows * 128;                       // the P^T buffer: 16 KB
constexpr int kPOff = kQOff + kPanels * kQPanel;           // 65,536
// Staged blocks are padded by 16 bytes so that the same byte of a row falls in a different bank in each
// of 8 consecutive blocks.
constexpr int kRawBlk = kLatBlk + 16;                      // 2,320
constexpr int kRawStage = kTileBlocks * kRawBlk;           // 37,120
constexpr int kRawStages = 3;
constexpr int kRawOff = kPOff + kPBytes;                   // 81,920
constexpr int kUnitBytes = 2 * 64 * 128;                   // values unit: 128 latent columns x 64 rows
constexpr int kRing = 2;
constexpr int kRingOff = (kRawOff + kRawStages * kRawStage + 1023) & ~1023;   // 193,536
constexpr int kPanelBytes = kRows * 128;                   // 16 KB: one 64-column panel of a whole tile
constexpr int kWinOff = kRawOff;                           // window tile: 8 panels over the raw and ring areas
constexpr int kWinEnd = kWinOff + kPanels * kPanelBytes;   // 212,992: window panels, or the staged o
constexpr int kRingEnd = kRingOff + kRing * kUnitBytes;    // 226,304
constexpr int kBarOff = kRingEnd > kWinEnd ? kRingEnd : kWinEnd;
constexpr int kNumBars = 36;
constexpr int kTmemPtrOff = kBarOff + kNumBars * 8;
constexpr int kFlagOff = kTmemPtrOff + 16;                 // int flag[2], int abort, int have (cluster staging)
constexpr int kMOff = kFlagOff + 16;                       // float m[64]
constexpr int kAlphaOff = kMOff + 64 * 4;                  // float alpha[2][64]: per P buffer
constexpr int kRedOff = kAlphaOff + 2 * 64 * 4;            // float red[4][64]
constexpr int kLsumOff = kRedOff + 4 * 64 * 4;             // float lsum[64]: final row sums
constexpr int kSmemBytes = kLsumOff + 64 * 4;
static_assert(kWinOff % 1024 == 0 && kRingOff % 1024 == 0, "swizzled operands start on 1024-byte boundaries");
static_assert(kSmemBytes <= 232448, "shared memory");

constexpr int kTRing = 4;
enum Bar {
  RAW_FULL = 0,                         // raw stages: gather -> both dequantisation groups
  RAW_EMPTY = RAW_FULL + kRawStages,
  TRING_FULL = RAW_EMPTY + kRawStages,  // logits operand panels in tensor memory: group A <-> logits issuer
  TRING_EMPTY = TRING_FULL + kTRing,
  RING_FULL = TRING_EMPTY + kTRing,     // values operand units in shared memory: group B <-> values issuer
  RING_EMPTY = RING_FULL + kRing,
  S_FULL = RING_EMPTY + kRing,          // logits buffers: logits issuer <-> softmax
  S_EMPTY = S_FULL + 2,
  P_FULL = S_EMPTY + 2,                 // the P buffer, per tile parity: softmax <-> values issuer, row sums
  PV_DONE = P_FULL + 2,
  WIN_FULL = PV_DONE + 2, WIN_CVT, WIN_EMPTY,
  FIN_L, FIN_V, NUM_BARS
};

static_assert(NUM_BARS <= kNumBars, "barrier area");

constexpr int kGrpA0 = 4, kGrpB0 = 8;          // first warps of the two dequantisation groups
constexpr int kDqWarps = 8;
constexpr int kGatherWarp = 12, kLogitsWarp = 13, kValuesWarp = 14, kSumWarp = 15;
constexpr int kThreads = 16 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColA = 128, kColO = 256;   // S: two buffers of 64 columns; A: four panels

constexpr uint32_t kIdescS = tc::idesc_f16_f32(128, kHeadsPad, 0, 0);   // C K-major, Q K-major
constexpr uint32_t kIdescPV = tc::idesc_f16_f32(128, kHeadsPad, 1, 1);  // C^T MN-major, P^T MN-major

// Row of a cache tile held by tensor-memory lane l (0..127) in the logits. The 8 lanes of a quarter warp
// take 8 different blocks and 8 different slots, so that their raw loads and their P^T stores fall in
// different banks.
__device__ __forceinline__ int lane_row(int l) {
  const int h = l >> 3, i = l & 7;
  const int blk = i + 8 * (h & 1), slot = (i + (h >> 1)) & 7;
  return 8 * blk + slot;
}

// Bounded wait that also gives up as soon as another role of the CTA has given up.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         uint32_t* hdr, uint32_t detail) {
  const uint32_t a = smem_addr(bar);
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 7u) == 7u && *abort_flag) return false;
  }
  *abort_flag = 1;
  report(hdr, CSA_ERR_TIMEOUT, KID_ATTN, detail);
  return false;
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

// Tensor-map copy of a [1 x 128 x 64] box (batch, row, latent column) into shared memory.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
               " [%0], [%1, {%2, %3, %4}], [%5];"
               :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
                  "r"(smem_addr(bar)) : "memory");
}

// OR of v over the 128 softmax threads (named barrier 1).
__device__ __forceinline__ bool any_softmax(bool v) {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, 1, 128, q;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(r) : "r"((uint32_t)v) : "memory");
  return r != 0;
}

struct UnitCtx {
  int64_t unit, b, n_e, n_b, nb_cap, pos, swa_first, swa_len;
  bool prefill;
};

// Block id of row r of cache tile t as stored in the index list (-1 past the list).
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

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}

// Every thread of every CTA of the cluster arrives; shared-memory writes before it are visible after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
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

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const AttnParams p,
                                                               const __grid_constant__ CUtensorMap swa_map) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + kTmemPtrOff);
  volatile int* flag = reinterpret_cast<volatile int*>(smem + kFlagOff);
  volatile int* abort_flag = flag + 2;
  float* msh = reinterpret_cast<float*>(smem + kMOff);
  float* alpha = reinterpret_cast<float*>(smem + kAlphaOff);
  float* red = reinterpret_cast<float*>(smem + kRedOff);

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

  // this CTA's tiles: cache tiles [c0, c1), then nw window tiles
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
  const int n_tiles = n_cache + nw;
  const uint8_t* seq = p.cache + u.b * p.cache_stride_b;

  // ---------------- setup ----------------
  // The barriers first, so that the gather warp can start the first tiles' copies while the other warps
  // load and convert the queries.
  if (warp == kLogitsWarp) tc::alloc(tmem_ptr, kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < kTRing; ++i) {
      mbar_init(&bars[TRING_FULL + i], 4);
      mbar_init(&bars[TRING_EMPTY + i], 1);
    }
    for (int i = 0; i < kRawStages; ++i) {
      mbar_init(&bars[RAW_FULL + i], 1);
      mbar_init(&bars[RAW_EMPTY + i], kDqWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[S_FULL + i], 1);
      mbar_init(&bars[S_EMPTY + i], 4);
      mbar_init(&bars[P_FULL + i], 4);
      mbar_init(&bars[PV_DONE + i], 2);        // the values' commit and the row-sum warp
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&bars[RING_FULL + i], 4);
      mbar_init(&bars[RING_EMPTY + i], 1);
    }
    mbar_init(&bars[WIN_FULL], 1);
    mbar_init(&bars[WIN_CVT], kDqWarps);
    mbar_init(&bars[WIN_EMPTY], 1);
    mbar_init(&bars[FIN_L], 1);
    mbar_init(&bars[FIN_V], 1);
    fence_mbar_init();
    flag[0] = 0; flag[1] = 0; *abort_flag = 0;
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tmem_ptr;
  const uint32_t s_base = smem_addr(smem);
  if (warp != kGatherWarp) {
    // queries: bf16 -> fp16, K-major 128-byte-swizzled panels; heads beyond H are zero. Every load of a
    // thread is issued before the first conversion.
    constexpr int kQThreads = kThreads - 32;
    constexpr int kQItems = kHeadsPad * 64;
    constexpr int kQPer = (kQItems + kQThreads - 1) / kQThreads;
    const int qt = tid < kGatherWarp * 32 ? tid : tid - 32;
    const __nv_bfloat16* qg = p.q + u.unit * (int64_t)H * kLatent;
    uint4 v[kQPer];
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int i = qt + k * kQThreads;
      const int h = i >> 6, ch = i & 63;
      v[k] = make_uint4(0, 0, 0, 0);
      if (i < kQItems && h < H) v[k] = __ldg(reinterpret_cast<const uint4*>(qg + (int64_t)h * kLatent + ch * 8));
    }
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int i = qt + k * kQThreads;
      if (i < kQItems) {
        const int h = i >> 6, ch = i & 63, pp = ch >> 3, c = ch & 7;
        const uint4 w = make_uint4(bf2_to_h2(v[k].x), bf2_to_h2(v[k].y), bf2_to_h2(v[k].z), bf2_to_h2(v[k].w));
        *reinterpret_cast<uint4*>(smem + kQOff + pp * kQPanel + h * 128 + ((c ^ (h & 7)) << 4)) = w;
      }
    }
    if (qt < 64) msh[qt] = -INFINITY;
    tc::fence_proxy_async();
    asm volatile("bar.sync 2, %0;" :: "n"(kQThreads) : "memory");
  }

  if (warp == kGatherWarp) {
    // ---------------- gather: cache blocks (cp.async.bulk), window rows (tensor map) ----------------
    if (lane == 0) {
      int issued = 0, win_issued = 0;
      for (int it = 0; it < n_cache; ++it) {
        const int stage = it % kRawStages;
        if (it >= kRawStages && !wait_bar(&bars[RAW_EMPTY + stage], (it / kRawStages - 1) & 1, abort_flag, p.hdr, 1)) break;
        const int t = c0 + it;
        uint8_t* dst = smem + kRawOff + stage * kRawStage;
        uint32_t bytes = 0;
        int64_t ids[kTileBlocks];
#pragma unroll
        for (int j = 0; j < kTileBlocks; ++j) {
          const int slot = t * kTileBlocks + j;
          int64_t id = -1;
          if (slot < p.top_k) id = __ldg(p.idx + u.unit * p.top_k + slot);
          if (id < -1 || id >= u.nb_cap) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_ATTN, (uint32_t)u.unit);
          ids[j] = (id >= 0 && id < u.n_b) ? id : -1;
          if (ids[j] >= 0) bytes += kLatBlk;
        }
        if (bytes) {
          mbar_arrive_expect_tx(&bars[RAW_FULL + stage], bytes);
#pragma unroll
          for (int j = 0; j < kTileBlocks; ++j)
            if (ids[j] >= 0) bulk_g2s(dst + j * kRawBlk, seq + ids[j] * kLatBlk, kLatBlk, &bars[RAW_FULL + stage]);
        } else {
          mbar_arrive(&bars[RAW_FULL + stage]);
        }
        ++issued;
        if (it == kRawStages - 1 || (it < kRawStages - 1 && it == n_cache - 1)) {
          // the later tiles of this CTA go to L2 now, so that refilling a raw stage costs an L2 read
          for (int t2 = c0 + kRawStages; t2 < c1; ++t2) {
            for (int j = 0; j < kTileBlocks; ++j) {
              const int slot = t2 * kTileBlocks + j;
              const int64_t id = slot < p.top_k ? (int64_t)__ldg(p.idx + u.unit * p.top_k + slot) : -1;
              if (id >= 0 && id < u.n_b) prefetch_l2(seq + id * kLatBlk, kLatBlk);
            }
          }
          // and the window rows, read once the cache tiles are done (boxes inside the buffer only)
          for (int tw = 0; tw < nw; ++tw) {
            const int64_t y0 = window_row0(p, u, tw);
            if (y0 < 0 || y0 + kRows > p.swa_rows) continue;
            for (int pp = 0; pp < kPanels; ++pp) prefetch_l2_3d(&swa_map, pp * 64, (int)y0, (int)u.b);
          }
        }
      }
      if (issued == n_cache) {
        for (int tw = 0; tw < nw; ++tw) {
          // the window panels overlay the raw and ring buffers: wait until every earlier product is done
          const int need = tw + (n_cache > 0 ? 1 : 0);
          if (need > 0 && !wait_bar(&bars[WIN_EMPTY], (need - 1) & 1, abort_flag, p.hdr, 9)) break;
          const int64_t y0 = window_row0(p, u, tw);
          const int y = (int)(y0 < -(int64_t)kRows ? -kRows : (y0 > p.swa_rows ? p.swa_rows : y0));
          mbar_arrive_expect_tx(&bars[WIN_FULL], kPanels * kPanelBytes);
#pragma unroll
          for (int pp = 0; pp < kPanels; ++pp)
            tma_load_3d(smem + kWinOff + pp * kPanelBytes, &swa_map, pp * 64, y, (int)u.b, &bars[WIN_FULL]);
          ++win_issued;
        }
      }
      // no copy into this CTA's shared memory may still be in flight when it exits
      for (int it = issued - kRawStages < 0 ? 0 : issued - kRawStages; it < issued; ++it)
        drain_bar(&bars[RAW_FULL + it % kRawStages], (it / kRawStages) & 1);
      if (win_issued > 0) drain_bar(&bars[WIN_FULL], (win_issued - 1) & 1);
    }
  } else if (warp >= kGrpA0 && warp < kGrpA0 + kDqWarps) {
    // ---------------- dequantisation ----------------
    bool stop = false;
    if (warp < kGrpB0) {
      // group A: one warp per tensor-memory subpartition, thread = lane = row lane_row(lane); writes the 8
      // logits panels of a tile into the two-slot tensor-memory ring
      const int sp = warp & 3;
      const int l = sp * 32 + lane;
      const int r = lane_row(l);
      const int blk = r >> 3, sl = r & 7;
      const uint32_t lane_base = (uint32_t)(sp * 32) << 16;
      uint32_t t_k = 0;
      int id_next = n_cache > 0 ? cache_id(p, u, c0, r) : -1;
      for (int it = 0; it < n_cache && !stop; ++it) {
        const int stage = it % kRawStages;
        const bool vr = cache_ok(u, id_next, r);
        if (it + 1 < n_cache) id_next = cache_id(p, u, c0 + it + 1, r);
        if (!__all_sync(0xffffffffu, wait_bar(&bars[RAW_FULL + stage], (it / kRawStages) & 1, abort_flag, p.hdr, 2))) break;
        const uint8_t* raw = smem + kRawOff + stage * kRawStage + blk * kRawBlk;
        const uint8_t* codes = raw + sl * 256;
        const uint8_t* scales = raw + 2048 + sl * 32;
        // Panels go out in pairs: both are converted and stored, then one wait covers both stores. The
        // next panel's raw words are loaded while the current one is converted.
        uint4 wa = *reinterpret_cast<const uint4*>(codes);
        uint4 wb = *reinterpret_cast<const uint4*>(codes + 16);
        uint32_t ws = vr ? *reinterpret_cast<const uint32_t*>(scales) : 0u;
#pragma unroll 1
        for (int pp = 0; pp < kPanels && !stop; pp += 2) {
          uint32_t slots[2];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t h[32];
            e2m1x8_to_f16x8(wa.x, h);      e2m1x8_to_f16x8(wa.y, h + 4);
            e2m1x8_to_f16x8(wa.z, h + 8);  e2m1x8_to_f16x8(wa.w, h + 12);
            e2m1x8_to_f16x8(wb.x, h + 16); e2m1x8_to_f16x8(wb.y, h + 20);
            e2m1x8_to_f16x8(wb.z, h + 24); e2m1x8_to_f16x8(wb.w, h + 28);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              // a zero scale (rows that are not attended) gives exact zeros: E2M1 has no infinities or NaNs
              const uint32_t sc = e4m3_to_f16x2_bcast((ws >> (8 * g)) & 0xFFu);
#pragma unroll
              for (int k = 0; k < 8; ++k) h[8 * g + k] = hmul2_u32(h[8 * g + k], sc);
            }
            const int nx = pp + q + 1;
            if (nx < kPanels) {
              wa = *reinterpret_cast<const uint4*>(codes + nx * 32);
              wb = *reinterpret_cast<const uint4*>(codes + nx * 32 + 16);
              ws = vr ? *reinterpret_cast<const uint32_t*>(scales + nx * 4) : 0u;
            }
            const uint32_t slot = t_k % kTRing, n = t_k / kTRing;
            if (n > 0 && !__all_sync(0xffffffffu, wait_bar(&bars[TRING_EMPTY + slot], (n - 1) & 1u, abort_flag, p.hdr, 3))) {
              stop = true;
              break;
            }
            tc::fence_after();
            tc::st_32x32(tbase + lane_base + kColA + 32 * slot, h);
            slots[q] = slot;
            ++t_k;
          }
          if (stop) break;
          tc::wait_st();
          tc::fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bars[TRING_FULL + slots[0]]);
            mbar_arrive(&bars[TRING_FULL + slots[1]]);
          }
        }
        tc::wait_st();      // no tensor-memory store may be in flight if the loop gave up
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[RAW_EMPTY + stage]);
      }
    } else {
      // group B: writes the values operand as 8 units of [128 latent columns x 64 rows] per tile (unit
      // 2 ch + rh: latent chunk ch, rows 64 rh ..). Per unit a thread converts 8 chunks of 8 elements:
      // column chunk c of block 8 rh + 2 bsel + (k & 1), slot 2 wl + ((k >> 1) & 1), panel half k >> 2.
      const int wl = warp - kGrpB0;
      const int c = lane & 7, bsel = lane >> 3;
      uint32_t u_k = 0;
      // the 4 blocks of this thread's rows in a tile: 8 rh + 2 bsel + j (rh, j in {0, 1})
      int ids_next[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) ids_next[q] = n_cache > 0 ? cache_id(p, u, c0, 8 * (8 * (q >> 1) + 2 * bsel + (q & 1))) : -1;
      for (int it = 0; it < n_cache && !stop; ++it) {
        const int stage = it % kRawStages;
        uint32_t vmask = 0;       // bit 4 rh + (k & 3): row attended
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int r = 8 * (8 * rh + 2 * bsel + (k & 1)) + 2 * wl + (k >> 1);
            if (cache_ok(u, ids_next[2 * rh + (k & 1)], r)) vmask |= 1u << (4 * rh + k);
          }
        }
        if (it + 1 < n_cache) {
#pragma unroll
          for (int q = 0; q < 4; ++q) ids_next[q] = cache_id(p, u, c0 + it + 1, 8 * (8 * (q >> 1) + 2 * bsel + (q & 1)));
        }
        if (!__all_sync(0xffffffffu, wait_bar(&bars[RAW_FULL + stage], (it / kRawStages) & 1, abort_flag, p.hdr, 2))) break;
        const uint8_t* raw = smem + kRawOff + stage * kRawStage;
        for (int unit = 0; unit < 8; ++unit) {
          const int ch = unit >> 1, rh = unit & 1;
          // the unit's raw words first: one load latency per unit instead of one per item
          uint32_t cw[8], sb[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int bl = 2 * bsel + (k & 1), sl = 2 * wl + ((k >> 1) & 1), pnl = 2 * ch + (k >> 2);
            const uint8_t* src = raw + (8 * rh + bl) * kRawBlk;
            cw[k] = *reinterpret_cast<const uint32_t*>(src + sl * 256 + pnl * 32 + c * 4);
            sb[k] = src[2048 + sl * 32 + pnl * 4 + (c >> 1)];
          }
          const uint32_t slot = u_k % kRing, n = u_k / kRing;
          if (n > 0 && !__all_sync(0xffffffffu, wait_bar(&bars[RING_EMPTY + slot], (n - 1) & 1u, abort_flag, p.hdr, 3))) {
            stop = true;
            break;
          }
          uint8_t* dst = smem + kRingOff + slot * kUnitBytes;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int bl = 2 * bsel + (k & 1), sl = 2 * wl + ((k >> 1) & 1), ph = k >> 2;
            const uint32_t sc = (vmask >> (4 * rh + (k & 3))) & 1u ? e4m3_to_f16x2_bcast(sb[k]) : 0u;
            uint32_t hh[4];
            e2m1x8_to_f16x8(cw[k], hh);
#pragma unroll
            for (int e = 0; e < 4; ++e) hh[e] = hmul2_u32(hh[e], sc);
            const int rl = 8 * bl + sl;
            *reinterpret_cast<uint4*>(dst + ph * (kUnitBytes / 2) + rl * 128 + ((c ^ sl) << 4)) =
                make_uint4(hh[0], hh[1], hh[2], hh[3]);
          }
          tc::fence_proxy_async();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[RING_FULL + slot]);
          ++u_k;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[RAW_EMPTY + stage]);
      }
    }
    const int dt = tid - kGrpA0 * 32;          // 0..255 over both groups
    for (int tw = 0; tw < nw && !stop; ++tw) {
      if (!__all_sync(0xffffffffu, wait_bar(&bars[WIN_FULL], tw & 1, abort_flag, p.hdr, 10))) break;
      // in place: bf16 -> fp16, rows that are not attended -> 0; this thread's rows are (k & 3) * 32 + dt / 8
      bool vr[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        bool oob;
        vr[k] = window_row(p, u, tw, k * 32 + (dt >> 3), &oob);
        if (oob && (dt & 7) == 0) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_ATTN, (uint32_t)u.unit);
      }
#pragma unroll 4
      for (int k = 0; k < 32; ++k) {
        const int q = k * 256 + dt;
        const int pp = q >> 10, row = (q & 1023) >> 3, cc = q & 7;
        uint4* a = reinterpret_cast<uint4*>(smem + kWinOff + pp * kPanelBytes + row * 128 + ((cc ^ (row & 7)) << 4));
        const uint4 x = *a;
        const bool v = vr[k & 3];
        *a = v ? make_uint4(bf2_to_h2(x.x), bf2_to_h2(x.y), bf2_to_h2(x.z), bf2_to_h2(x.w)) : make_uint4(0, 0, 0, 0);
      }
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[WIN_CVT]);
    }
  } else if (warp == kLogitsWarp) {
    // ---------------- logits MMA issue: S^T(t) = C . Q^T into S buffer t & 1 ----------------
    if (lane == 0) {
      const uint32_t q_addr = s_base + kQOff, win_addr = s_base + kWinOff;
      uint32_t t_k = 0;
      bool ok = true;
      for (int it = 0; it < n_tiles && ok; ++it) {
        const int sb = it & 1;
        const bool cache = it < n_cache;
        if (it >= 2 && !wait_bar(&bars[S_EMPTY + sb], ((it - 2) >> 1) & 1, abort_flag, p.hdr, 4)) { ok = false; break; }
        if (!cache && !wait_bar(&bars[WIN_CVT], (it - n_cache) & 1, abort_flag, p.hdr, 11)) { ok = false; break; }
        const uint32_t d = tbase + kColS + 64 * sb;
        for (int pp = 0; pp < kPanels; ++pp) {
          uint32_t slot = 0;
          if (cache) {
            slot = t_k % kTRing;
            if (!wait_bar(&bars[TRING_FULL + slot], (t_k / kTRing) & 1u, abort_flag, p.hdr, 4)) { ok = false; break; }
          }
          tc::fence_after();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t bq = tc::smem_desc(q_addr + pp * kQPanel + ks * 32, 16, 1024, tc::kSwizzle128B);
            if (cache) {
              tc::mma_f16_ts(d, tbase + kColA + 32 * slot + 8 * ks, bq, kIdescS, (pp | ks) != 0);
            } else {
              const uint64_t a = tc::smem_desc(win_addr + pp * kPanelBytes + ks * 32, 16, 1024, tc::kSwizzle128B);
              tc::mma_f16(d, a, bq, kIdescS, (pp | ks) != 0);
            }
          }
          if (cache) { tc::commit(&bars[TRING_EMPTY + slot]); ++t_k; }
        }
        if (ok) tc::commit(&bars[S_FULL + sb]);
      }
      // every MMA issued must be complete before the tensor memory is released
      tc::commit(&bars[FIN_L]);
      drain_bar(&bars[FIN_L], 0);
    }
  } else if (warp == kValuesWarp) {
    // ---------------- values MMA issue: O^T += C^T . P^T and l += ones . P^T ----------------
    if (lane == 0) {
      const uint32_t ring_addr = s_base + kRingOff, win_addr = s_base + kWinOff;
      uint32_t u_k = 0;
      for (int it = 0; it < n_tiles; ++it) {
        const int pb = it & 1;
        const bool cache = it < n_cache;
        const uint32_t p_addr = s_base + kPOff;
        if (!wait_bar(&bars[P_FULL + pb], (it >> 1) & 1, abort_flag, p.hdr, 5)) break;
        tc::fence_after();
        bool ok = true;
        if (cache) {
          for (int unit = 0; unit < 8; ++unit) {
            const int ch = unit >> 1, rh = unit & 1;
            const uint32_t slot = u_k % kRing;
            if (!wait_bar(&bars[RING_FULL + slot], (u_k / kRing) & 1u, abort_flag, p.hdr, 6)) { ok = false; break; }
            tc::fence_after();
            const uint32_t c_addr = ring_addr + slot * kUnitBytes;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t a = tc::smem_desc(c_addr + j * 2048, kUnitBytes / 2, 1024, tc::kSwizzle128B);
              const uint64_t bp = tc::smem_desc(p_addr + rh * (kPBytes / 2) + j * 2048, 8192, 1024, tc::kSwizzle128B);
              tc::mma_f16(tbase + kColO + 64 * ch, a, bp, kIdescPV, (it > 0 || rh > 0 || j > 0) ? 1u : 0u);
            }
            tc::commit(&bars[RING_EMPTY + slot]);
            ++u_k;
          }
        } else {
          for (int ch = 0; ch < 4; ++ch) {
            const uint32_t c_addr = win_addr + 2 * ch * kPanelBytes;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint64_t a = tc::smem_desc(c_addr + j * 2048, kPanelBytes, 1024, tc::kSwizzle128B);
              const uint64_t bp = tc::smem_desc(p_addr + j * 2048, 8192, 1024, tc::kSwizzle128B);
              tc::mma_f16(tbase + kColO + 64 * ch, a, bp, kIdescPV, (it > 0 || j > 0) ? 1u : 0u);
            }
          }
        }
        if (!ok) break;
        tc::commit(&bars[PV_DONE + pb]);
        // the window panels overlay the raw and ring buffers: free them after the last cache tile and
        // after every window tile
        if ((cache && it == n_cache - 1 && nw > 0) || !cache) tc::commit(&bars[WIN_EMPTY]);
      }
      tc::commit(&bars[FIN_V]);
      drain_bar(&bars[FIN_V], 0);
    }
  } else if (warp == kSumWarp) {
    // ---------------- row sums: l += sum over the tile's rows of P (lane = heads 2 lane, 2 lane + 1) ----
    float l0 = 0.0f, l1 = 0.0f;
    const int h0 = 2 * lane;
    bool ok = true;
    for (int it = 0; it < n_tiles && ok; ++it) {
      const int pb = it & 1;
      if (!__all_sync(0xffffffffu, wait_bar(&bars[P_FULL + pb], (it >> 1) & 1, abort_flag, p.hdr, 13))) { ok = false; break; }
      if (flag[pb]) {
        // the softmax raised the reference maxima for this tile: rescale like O
        l0 *= alpha[64 * pb + h0];
        l1 *= alpha[64 * pb + h0 + 1];
      }
      const uint8_t* pbuf = smem + kPOff + (lane & 3) * 4;
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
        float* lsum = reinterpret_cast<float*>(smem + kLsumOff);
        lsum[h0] = l0;
        lsum[h0 + 1] = l1;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[PV_DONE + pb]);
    }
  } else {
    // ---------------- softmax (warps 0-3, thread = tile row) ----------------
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    bool ok = true;
    int id_next = n_cache > 0 ? cache_id(p, u, c0, lane_row(tid)) : -1;
    for (int it = 0; it < n_tiles; ++it) {
      const int sb = it & 1;
      // tensor-memory lane tid holds row lane_row(tid) of a cache tile (row tid of a window tile)
      const int row = it < n_cache ? lane_row(tid) : tid;
      bool valid;
      if (it < n_cache) {
        valid = cache_ok(u, id_next, row);
        if (it + 1 < n_cache) id_next = cache_id(p, u, c0 + it + 1, row);
      } else {
        bool oob;
        valid = window_row(p, u, it - n_cache, row, &oob);
      }
      const uint32_t s_col = kColS + 64 * sb;
      if (!all_softmax(wait_bar(&bars[S_FULL + sb], (it >> 1) & 1, abort_flag, p.hdr, 7))) { ok = false; break; }
      // alpha[sb] and flag[sb] were last read by the row sums of tile it - 2
      if (it >= 2) {
        if (!all_softmax(wait_bar(&bars[PV_DONE + sb], ((it - 2) >> 1) & 1, abort_flag, p.hdr, 12))) { ok = false; break; }
      }
      tc::fence_after();
      float* al = alpha + 64 * sb;
      // Fast path: probabilities against the current reference maxima; the full path runs only when a
      // probability would exceed 2^8 (a maximum moved by more than the slack, or none was set yet).
      uint32_t w[32];
      bool over = false;
      {
        uint32_t sr[64];
        tc::ld_32x64(tbase + lane_base + s_col, sr);
        tc::wait_ld();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 ma = *reinterpret_cast<const float4*>(msh + 8 * c);
          const float4 mb = *reinterpret_cast<const float4*>(msh + 8 * c + 4);
          const float mm[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int h = 8 * c + 2 * k;
            const float p0 = valid ? ex2(__uint_as_float(sr[h]) * p.scale_log2 - mm[2 * k]) : 0.0f;
            const float p1 = valid ? ex2(__uint_as_float(sr[h + 1]) * p.scale_log2 - mm[2 * k + 1]) : 0.0f;
            over |= !(p0 <= kMaxProb) || !(p1 <= kMaxProb);
            w[4 * c + k] = f2_to_h2(p0, p1);
          }
        }
      }
      const bool full = any_softmax(over);
      if (tid == 0) flag[sb] = 0;
      if (full) {
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          // per-head maximum over the warp's 32 rows (one warp reduction per head)
          uint32_t sr[32];
          tc::ld_32x32(tbase + lane_base + s_col + 32 * half, sr);
          tc::wait_ld();
#pragma unroll
          for (int h = 0; h < 32; ++h) {
            const float v = valid ? __uint_as_float(sr[h]) * p.scale_log2 : -INFINITY;
            float mx;
            asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(mx) : "f"(v));
            red[warp * 64 + 32 * half + h] = mx;
          }
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
          // the previous tile's value products must be complete before O is rescaled (the ones before it
          // completed earlier: the values are issued in tile order); the row-sum warp rescales l itself
          if (it > 0) {
            if (!all_softmax(wait_bar(&bars[PV_DONE + ((it - 1) & 1)], ((it - 1) >> 1) & 1, abort_flag, p.hdr, 12))) {
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
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sr[32];
          tc::ld_32x32(tbase + lane_base + s_col + 32 * half, sr);
          tc::wait_ld();
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float m0 = msh[32 * half + 2 * k], m1 = msh[32 * half + 2 * k + 1];
            const float p0 = (!valid || m0 == -INFINITY) ? 0.0f : ex2(__uint_as_float(sr[2 * k]) * p.scale_log2 - m0);
            const float p1 = (!valid || m1 == -INFINITY) ? 0.0f : ex2(__uint_as_float(sr[2 * k + 1]) * p.scale_log2 - m1);
            w[16 * half + k] = f2_to_h2(p0, p1);
          }
        }
      }
      // S buffer sb has been read for the last time: the logits of tile it + 2 may overwrite it
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[S_EMPTY + sb]);
      // P was read by the values and the row sums of tile it - 1
      if (it >= 1) {
        if (!all_softmax(wait_bar(&bars[PV_DONE + ((it - 1) & 1)], ((it - 1) >> 1) & 1, abort_flag, p.hdr, 14))) {
          ok = false;
          break;
        }
      }
      // probabilities, fp16, row `row` of P (MN-major: 64 heads contiguous, 128-byte swizzle)
      uint8_t* prow = smem + kPOff + row * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) << 4)) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
      tc::fence_proxy_async();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[P_FULL + sb]);
    }
    // ---------------- epilogue ----------------
    const int last = n_tiles - 1;
    const bool have = all_softmax(ok && n_tiles > 0 &&
                                  wait_bar(&bars[PV_DONE + (last & 1)], (last >> 1) & 1, abort_flag, p.hdr, 8));
    tc::fence_after();
    // the row sums, one per head, written by the row-sum warp before its last arrival on PV_DONE
    float* lsh = reinterpret_cast<float*>(smem + kLsumOff);
    if (!have && tid < 64) lsh[tid] = 0.0f;
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const int64_t prow_base = (u.unit * p.splits + split) * H;
    if (p.cluster) {
      // o is staged by every warp after the roles end; m and l are already in shared memory
      if (tid == 0) flag[3] = have ? 1 : 0;
      if (!have && tid < 64) msh[tid] = -INFINITY;
    }
#pragma unroll 1
    for (int k = 0; k < 8 && !p.cluster; ++k) {
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
        const float l = lsh[h];
        const float x = __uint_as_float(o[j]);
        if (p.splits == 1) p.out[(u.unit * H + h) * (int64_t)kLatent + d] = l > 0.0f ? x / l : 0.0f;
        else p.part_o[(prow_base + h) * kLatent + d] = x;
      }
    }
    if (tid < H && !p.cluster) {
      const float l = lsh[tid];
      const float m = have ? msh[tid] : -INFINITY;
      if (p.splits == 1) {
        if (p.out_lse != nullptr) p.out_lse[u.unit * H + tid] = l > 0.0f ? (m + log2f(l)) * kLn2 : -INFINITY;
      } else {
        *reinterpret_cast<float2*>(p.part_ml + (prow_base + tid) * 2) = make_float2(m, l);
      }
    }
    tc::fence_before();
  }

  if (p.cluster) {
    // ---------------- staging of o: [head][512] fp32 over the operand area ----------------
    // Every product has completed (the softmax saw the last values finish). Warp w reads tensor-memory
    // subpartition w % 4 (latent columns 32 (w % 4) .. of each 128-column chunk), 32-column pieces
    // 2 (w / 4) and 2 (w / 4) + 1.
    __syncwarp();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    {
      const bool had = flag[3] != 0;
      float* stage = reinterpret_cast<float*>(smem + kRawOff);
      const uint32_t sp_base = (uint32_t)((warp & 3) * 32) << 16;
#pragma unroll 1
      for (int k = 2 * (warp >> 2); k < 2 * (warp >> 2) + 2; ++k) {
        uint32_t o[32];
        if (had) {
          tc::ld_32x32(tbase + sp_base + kColO + 32 * k, o);
          tc::wait_ld();
        }
        const int d = 128 * (k >> 1) + 32 * (warp & 3) + lane;
#pragma unroll
        for (int j = 0; j < 32; ++j) stage[(32 * (k & 1) + j) * kLatent + d] = had ? __uint_as_float(o[j]) : 0.0f;
      }
    }
    // ---------------- merge of the cluster's splits ----------------
    // Thread = (head tid / 8, every eighth float4 column of this CTA's slice); the weights of the splits
    // for its head are computed once: w_s = 2^(m_s - M) / sum_s 2^(m_s - M) l_s over splits with l_s > 0.
    cluster_sync();
    const int S = p.splits;
    const int h = tid >> 3, t8 = tid & 7;
    const int c_lo = split * (kLatent / 4) / S, c_hi = (split + 1) * (kLatent / 4) / S;
    const float* stage = reinterpret_cast<const float*>(smem + kRawOff);
    const float* lsum = reinterpret_cast<const float*>(smem + kLsumOff);
    if (h < H) {
      float ms[8], ls[8];
      float M = -INFINITY;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        ms[s] = -INFINITY;
        ls[s] = 0.0f;
        if (s < S) {
          ms[s] = ld_cluster_f32(cluster_addr(msh + h, s));
          ls[s] = ld_cluster_f32(cluster_addr(lsum + h, s));
          if (ls[s] > 0.0f) M = fmaxf(M, ms[s]);
        }
      }
      float L = 0.0f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        ms[s] = (s < S && ls[s] > 0.0f) ? exp2f(ms[s] - M) : 0.0f;     // the split's weight
        L += ms[s] * ls[s];
      }
      const float inv = L > 0.0f ? 1.0f / L : 0.0f;
      for (int c = c_lo + t8; c < c_hi; c += 8) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          if (s < S && ms[s] > 0.0f) {
            const float4 v = ld_cluster_v4(cluster_addr(stage + h * kLatent + 4 * c, s));
            acc.x += ms[s] * v.x; acc.y += ms[s] * v.y; acc.z += ms[s] * v.z; acc.w += ms[s] * v.w;
          }
        }
        *reinterpret_cast<float4*>(p.out + (u.unit * H + h) * (int64_t)kLatent + 4 * c) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      }
      if (split == 0 && t8 == 0 && p.out_lse != nullptr)
        p.out_lse[u.unit * H + h] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    // no CTA may leave while another still reads its shared memory
    cluster_sync();
  }
  __syncthreads();
  tc::fence_after();
  if (warp == kLogitsWarp) tc::dealloc(tbase, kTmemCols);
}

// out[u][h] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s, splits in order; lse = (M + log2 L) ln 2.
__global__ void __launch_bounds__(128) combine_kernel(AttnParams p) {
  const int64_t row = blockIdx.x;                 // unit * H + h
  const int64_t unit = row / p.heads;
  const int h = (int)(row % p.heads);
  const int d = threadIdx.x * 4;
  float M = -INFINITY;
  for (int s = 0; s < p.splits; ++s) {
    const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + ((unit * p.splits + s) * p.heads + h) * 2);
    if (ml.y > 0.0f) M = fmaxf(M, ml.x);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.0f;
  if (M != -INFINITY) {
    for (int s = 0; s < p.splits; ++s) {
      const int64_t pr = (unit * p.splits + s) * p.heads + h;
      const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + pr * 2);
      if (!(ml.y > 0.0f)) continue;
      const float w = exp2f(ml.x - M);
      const float4 v = *reinterpret_cast<const float4*>(p.part_o + pr * kLatent + d);
      acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
      L += w * ml.y;
    }
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  *reinterpret_cast<float4*>(p.out + row * kLatent + d) =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (threadIdx.x == 0 && p.out_lse != nullptr) p.out_lse[row] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
}


}  // namespace

cudaError_t launch_attn(const AttnParams& p, cudaStream_t s) {
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
  ProfScope prof("sparse_attn", s);
  clear_stale_error();
  cudaError_t e = ensure_smem_limit(attn_tc_kernel, kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.splits, (unsigned)p.units);
  if (!p.cluster) {
    attn_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(p, map);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel, p, map);
}

int attn_max_clusters(int size) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> known;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(dev, size);
  auto it = known.find(key);
  if (it != known.end()) return it->second;
  int n = 0;
  if (ensure_smem_limit(attn_tc_kernel, kSmemBytes) == cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)size, 1, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  known[key] = n;
  return n;
}

cudaError_t launch_combine(const AttnParams& p, cudaStream_t s) {
  if (p.units == 0 || p.splits == 1 || p.cluster) return cudaSuccess;
  ProfScope prof("attn_combine", s);
  clear_stale_error();
  combine_kernel<<<(unsigned)(p.units * p.heads), 128, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace csa
