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

}  // namespace

cudaError_t launch_topk(const TopkParams& p, cudaStream_t s) {
  if (p.units == 0) return cudaSuccess;
  ProfScope prof("topk", s);
  clear_stale_error();
  topk_kernel<<<(unsigned)p.units, kTopkThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace csa
