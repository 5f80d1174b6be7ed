// Deterministic Top-K over block scores: radix select on order-preserving 32-bit keys, ties to the
// lower block id, output in ascending block id padded with -1.
//
// Follows "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (card), Key ideas ("Top-K
// indices" over "blocks of 8"). The tie rule and output order are this library's readings.
//
// One CTA per query. Scores are mapped to keys that order like the floats (-0 and +0 collapse to one
// key); -inf marks a non-candidate. Four 8-bit histogram passes (most significant byte first) find the
// K-th largest key T and how many keys equal to T must be taken; a final pass in ascending id order
// takes every key > T and the first `need_eq` keys == T, placing each with a block-wide prefix count, so
// the result does not depend on thread scheduling.
#include "csa_internal.cuh"

namespace csa {
namespace {

constexpr int kTopkThreads = 1024;
constexpr uint32_t kNegInfKey = 0x007FFFFFu;   // key of -inf

__device__ __forceinline__ uint32_t order_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;                 // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive block scan of a count (< 65536 per call).
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < (kTopkThreads / 32) ? warp_sums[lane] : 0u;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    warp_sums[lane] = w;   // inclusive prefix over warps
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? warp_sums[warp - 1] : 0u;
  *total = warp_sums[kTopkThreads / 32 - 1];
  const uint32_t res = x + before;
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(TopkParams p) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t s_prefix, s_krem, s_ncand;
  griddep_wait();                                  // the scores come from the kernel before
  griddep_launch();

  const int64_t unit = blockIdx.x;
  const float* sc = p.scores + unit * p.score_stride;
  int32_t* out = p.out + unit * p.out_stride;
  const int tid = threadIdx.x;

  // pass 0: candidate count and histogram of the top byte
  for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0u;
  if (tid == 0) s_ncand = 0u;
  __syncthreads();
  uint32_t local = 0;
  for (int64_t i = tid; i < p.n; i += kTopkThreads) {
    const uint32_t key = order_key(__ldg(sc + i));
    if (key > kNegInfKey) {
      ++local;
      atomicAdd(&hist[key >> 24], 1u);
    }
  }
  atomicAdd(&s_ncand, local);
  __syncthreads();
  const uint32_t ncand = s_ncand;
  const uint32_t k = (uint32_t)p.k;

  uint32_t T = kNegInfKey + 1u, need_eq = 0u;   // take-all defaults
  const bool take_all = ncand <= k;
  if (!take_all) {
    uint32_t prefix = 0u, mask = 0u, krem = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (shift < 24) {
        for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0u;
        __syncthreads();
        for (int64_t i = tid; i < p.n; i += kTopkThreads) {
          const uint32_t key = order_key(__ldg(sc + i));
          if (key > kNegInfKey && (key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFFu], 1u);
        }
        __syncthreads();
      }
      if (tid == 0) {
        uint32_t cum = 0u;
        int bin = 255;
        for (; bin > 0; --bin) {
          if (cum + hist[bin] >= krem) break;
          cum += hist[bin];
        }
        s_krem = krem - cum;
        s_prefix = prefix | ((uint32_t)bin << shift);
      }
      __syncthreads();
      krem = s_krem;
      prefix = s_prefix;
      mask |= 0xFFu << shift;
      __syncthreads();
    }
    T = prefix;        // the K-th largest key
    need_eq = krem;    // how many keys equal to T are taken
  }

  // selection in ascending id order
  uint32_t taken_before = 0u, eq_before = 0u;
  for (int64_t base = 0; base < p.n; base += kTopkThreads) {
    const int64_t i = base + tid;
    uint32_t key = 0u;
    if (i < p.n) key = order_key(__ldg(sc + i));
    const bool cand = i < p.n && key > kNegInfKey;
    const bool gt = cand && (take_all ? true : key > T);
    const bool eq = cand && !take_all && key == T;
    uint32_t tot;
    const uint32_t eq_incl = block_scan(eq ? 1u : 0u, warp_sums, &tot);
    const uint32_t eq_rank = eq_before + eq_incl - (eq ? 1u : 0u);
    eq_before += tot;
    const bool take = gt || (eq && eq_rank < need_eq);
    const uint32_t take_incl = block_scan(take ? 1u : 0u, warp_sums, &tot);
    if (take) {
      const uint32_t pos = taken_before + take_incl - 1u;
      int32_t id = (int32_t)i;
      if (p.map_super != nullptr) {
        const int32_t g = p.map_super[unit * p.map_stride + i / kSuper];
        id = g * kSuper + (int32_t)(i % kSuper);
      }
      if (pos < k) out[pos] = id;
    }
    taken_before += tot;
  }
  for (uint32_t pos = taken_before + tid; pos < k; pos += kTopkThreads) out[pos] = -1;
}

// Register-resident variant for n <= 1024 * KPT: thread t holds the keys of ids [t KPT, t KPT + KPT), so
// thread order is id order. Each pass adds its digits to one of two shared histograms with plain atomics
// (on this hardware they beat warp-aggregated ones even when every key has the same digit) and clears the
// other for the next pass, so a pass needs two barriers; one warp finds the bin, and one block scan of
// packed (equal-count, greater-count) pairs places every selected id.
template <int KPT>
__global__ void __launch_bounds__(kTopkThreads, 1) topk_reg_kernel(TopkParams p) {
  __shared__ uint32_t hist[2][256];
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t s_prefix, s_krem, s_ncand;
  griddep_wait();                                  // the scores come from the kernel before
  griddep_launch();
  const int64_t unit = blockIdx.x;
  const float* sc = p.scores + unit * p.score_stride;
  int32_t* out = p.out + unit * p.out_stride;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 512; i += kTopkThreads) (&hist[0][0])[i] = 0u;

  uint32_t key[KPT];
  const int64_t id0 = (int64_t)tid * KPT;
  if (id0 + KPT <= p.n && (reinterpret_cast<uintptr_t>(sc) & 15u) == 0) {
#pragma unroll
    for (int i = 0; i < KPT / 4; ++i) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(sc + id0) + i);
      key[4 * i] = order_key(f.x);
      key[4 * i + 1] = order_key(f.y);
      key[4 * i + 2] = order_key(f.z);
      key[4 * i + 3] = order_key(f.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < KPT; ++i) key[i] = id0 + i < p.n ? order_key(__ldg(sc + id0 + i)) : 0u;   // 0: no candidate
  }
  __syncthreads();

  const uint32_t k = (uint32_t)p.k;
  uint32_t prefix = 0u, mask = 0u, krem = k, ncand = 0u;
  int cur = 0;
  for (int shift = 24; shift >= 0; shift -= 8, cur ^= 1) {
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      if (key[i] > kNegInfKey && (key[i] & mask) == prefix)
        atomicAdd(&hist[cur][(key[i] >> shift) & 0xFFu], 1u);
    }
    for (int i = tid; i < 256; i += kTopkThreads) hist[cur ^ 1][i] = 0u;   // the next pass's bins
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255 - 8 l .. 248 - 8 l (descending)
      uint32_t b[8], own = 0u;
#pragma unroll
      for (int i = 0; i < 8; ++i) { b[i] = hist[cur][255 - 8 * lane - i]; own += b[i]; }
      uint32_t incl = own;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
      if (shift == 24 && lane == 0) s_ncand = total;
      const uint32_t hit = __ballot_sync(0xffffffffu, incl >= krem);
      if (hit != 0u && lane == __ffs(hit) - 1) {
        // the first of this lane's bins where the running count reaches krem (the last one otherwise)
        uint32_t cum = incl - own, before = 0u;
        int sel = -1;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (sel < 0 && (cum + b[i] >= krem || i == 7)) { sel = i; before = cum; }
          cum += b[i];
        }
        s_krem = krem - before;
        s_prefix = prefix | ((uint32_t)(255 - 8 * lane - sel) << shift);
      }
      if (hit == 0u && lane == 0) { s_krem = 0u; s_prefix = prefix; }   // fewer candidates than k
    }
    __syncthreads();
    if (shift == 24) {
      ncand = s_ncand;
      if (ncand <= k) break;          // every candidate is taken
    }
    krem = s_krem;
    prefix = s_prefix;
    mask |= 0xFFu << shift;
  }
  const bool take_all = ncand <= k;
  const uint32_t T = take_all ? kNegInfKey : prefix;
  const uint32_t need_eq = take_all ? 0u : krem;

  uint32_t gt = 0u, eq = 0u;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    gt += key[i] > T ? 1u : 0u;
    eq += (!take_all && key[i] == T) ? 1u : 0u;
  }
  // exclusive block scan of (eq << 16 | gt); both totals stay below 2^16
  const uint32_t v = (eq << 16) | gt;
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_sums[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const uint32_t excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0u);
  const uint32_t tot = warp_sums[31];
  uint32_t eq_before = excl >> 16;
  uint32_t pos = (excl & 0xFFFFu) + (eq_before < need_eq ? eq_before : need_eq);
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    bool take = key[i] > T;
    if (!take_all && key[i] == T) {
      take = eq_before < need_eq;
      ++eq_before;
    }
    if (take) {
      const int64_t idx = id0 + i;
      int32_t id = (int32_t)idx;
      if (p.map_super != nullptr) {
        const int32_t g = p.map_super[unit * p.map_stride + idx / kSuper];
        id = g * kSuper + (int32_t)(idx % kSuper);
      }
      if (pos < k) out[pos] = id;
      ++pos;
    }
  }
  const uint32_t eq_tot = tot >> 16;
  const uint32_t taken = (tot & 0xFFFFu) + (eq_tot < need_eq ? eq_tot : need_eq);
  for (uint32_t q = taken + tid; q < k; q += kTopkThreads) out[q] = -1;
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, cudaStream_t s, bool pdl) {
  if (p.units == 0) return cudaSuccess;
  ProfScope prof("topk", s);
  clear_stale_error();
  const dim3 grid((unsigned)p.units), block(kTopkThreads);
  if (p.n <= 4 * kTopkThreads) return launch_ex(topk_reg_kernel<4>, grid, block, 0, s, pdl, p);
  if (p.n <= 8 * kTopkThreads) return launch_ex(topk_reg_kernel<8>, grid, block, 0, s, pdl, p);
  if (p.n <= 16 * kTopkThreads) return launch_ex(topk_reg_kernel<16>, grid, block, 0, s, pdl, p);
  return launch_ex(topk_kernel, grid, block, 0, s, pdl, p);
}

}  // namespace csa
