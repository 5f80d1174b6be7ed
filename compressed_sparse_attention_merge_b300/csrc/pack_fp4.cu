// Pair-merge + FP4 quantiser + block-major store, and the super-block coarse-key sums.
//
// Follows "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression" (paper-digest), Core
// Mechanics ("Sequence: the Encoder merges 2 adjacent positions into 1 cache entry") and the FP4 global
// KV of "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (card), Key ideas. The numeric
// format (E2M1 codes, E4M3 scale per 16 elements, amax/6 or power-of-two scale) is this library's own and
// is stated in include/csa.h; every fp32 step uses an explicit round-to-nearest intrinsic so that the
// bytes do not depend on contraction or fast-math choices.
//
// One thread quantises one 16-element group: a warp covers 32 consecutive groups (a whole 512-d entry),
// so loads (2 x 32 B or 1 x 32 B per thread) and stores (8 code bytes + 1 scale byte per thread) are
// contiguous across the warp. The kernel is HBM-bound.
#include "csa_internal.cuh"

namespace csa {
namespace {

__device__ __forceinline__ void load16(const void* base, int dtype, int64_t elem_off, float* v) {
  if (dtype == CSA_DTYPE_BF16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + elem_off);
    uint4 a = __ldg(p), b = __ldg(p + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem_off);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float4 f = __ldg(p + i);
      v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
  }
}

__global__ void __launch_bounds__(256) pack_fp4_kernel(PackParams p) {
  const int groups = p.dim / kGroup;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = p.batch * p.n_new * groups;
  if (t >= total) return;
  const int g = (int)(t % groups);
  const int64_t i = (t / groups) % p.n_new;
  const int64_t b = t / ((int64_t)groups * p.n_new);

  const int64_t first = p.first_entry ? (int64_t)p.first_entry[b] : 0;
  if (first < 0 || first + p.n_new > p.max_entries) {
    if (i == 0 && g == 0) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_PACK, (uint32_t)b);
    return;
  }

  float m[16];
  const int64_t row0 = b * p.x_stride_b + (int64_t)g * kGroup;
  if (p.merge == 2) {
    float a[16], c[16];
    load16(p.x, p.x_dtype, row0 + (2 * i) * p.x_stride_t, a);
    load16(p.x, p.x_dtype, row0 + (2 * i + 1) * p.x_stride_t, c);
#pragma unroll
    for (int j = 0; j < 16; ++j) m[j] = __fmul_rn(__fadd_rn(a[j], c[j]), 0.5f);
  } else {
    load16(p.x, p.x_dtype, row0 + i * p.x_stride_t, m);
  }

  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(m[j]));
  const float sf = __fdiv_rn(amax, 6.0f);

  uint32_t sbyte = 0;
  float s = 0.0f;
  if (sf > 0.0f) {
    if (p.scale_rule == CSA_SCALE_AMAX) {
      sbyte = float_to_e4m3_satfinite(sf);
      s = e4m3_to_float(sbyte);
    } else {
      sbyte = pow2_scale(sf, &s);
    }
  }

  uint32_t lo = 0, hi = 0;
  if (s > 0.0f) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t c0 = e2m1_code(__fdiv_rn(m[2 * j], s));
      const uint32_t c1 = e2m1_code(__fdiv_rn(m[2 * j + 1], s));
      const uint32_t byte = c0 | (c1 << 4);
      if (j < 4) lo |= byte << (8 * j); else hi |= byte << (8 * (j - 4));
    }
  }

  const int64_t e = first + i;
  uint8_t* blk = p.cache + b * p.cache_stride_b + (e / kBlockEntries) * (int64_t)block_bytes(p.dim);
  const int slot = (int)(e % kBlockEntries);
  *reinterpret_cast<uint2*>(blk + slot * (p.dim / 2) + g * 8) = make_uint2(lo, hi);
  blk[kBlockEntries * (p.dim / 2) + slot * groups + g] = (uint8_t)sbyte;
}

// coarse_sum[b][g][d] = fp32 sum, ascending entry order, of the dequantised element d of entries
// [512 g, min(512 (g + 1), first + n_new)), for every super-block g touched by this call. One CTA per
// (super-block, sequence), one thread per element d: the super-block's packed bytes are staged through
// shared memory in chunks, each one bulk copy, and each thread then sums its element over the chunk's
// entries in ascending order.
constexpr int kCoarseStage = 36864;

__global__ void __launch_bounds__(1024) coarse_sum_kernel(PackParams p, int touched) {
  __shared__ __align__(16) uint8_t stage[kCoarseStage];
  __shared__ __align__(8) uint64_t bar;
  const int d = threadIdx.x;                     // blockDim.x == dim
  const int gl = blockIdx.x;
  const int64_t b = blockIdx.y;
  const int64_t first = p.first_entry ? (int64_t)p.first_entry[b] : 0;
  if (first < 0 || first + p.n_new > p.max_entries || p.n_new == 0) return;
  const int64_t end = first + p.n_new;
  const int64_t per_super = (int64_t)kSuper * kBlockEntries;
  const int64_t g = first / per_super + gl;
  if (gl >= touched || g * per_super >= end) return;
  const int64_t e_hi = (g + 1) * per_super < end ? (g + 1) * per_super : end;

  const int bb = block_bytes(p.dim);
  const int half = p.dim / 2, groups = p.dim / kGroup;
  const int chunk_blocks = kCoarseStage / bb < kSuper ? kCoarseStage / bb : kSuper;
  const uint8_t* seq = p.cache + b * p.cache_stride_b;
  if (d == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  float acc = 0.0f;
  uint32_t phase = 0;
  for (int64_t blk0 = g * kSuper; blk0 * kBlockEntries < e_hi; blk0 += chunk_blocks) {
    const int64_t n_e = e_hi - blk0 * kBlockEntries;
    const int nb = (int)((n_e + kBlockEntries - 1) / kBlockEntries < chunk_blocks
                             ? (n_e + kBlockEntries - 1) / kBlockEntries : chunk_blocks);
    __syncthreads();                             // the previous chunk has been read (and bar initialised)
    if (d == 0) {
      mbar_arrive_expect_tx(&bar, (uint32_t)(nb * bb));
      bulk_g2s(stage, seq + blk0 * bb, (uint32_t)(nb * bb), &bar);
    }
    if (!__syncthreads_and(mbar_wait(&bar, phase))) {
      // give up: report, let the copy land (bounded), leave without writing a sum
      if (d == 0) {
        report(p.hdr, CSA_ERR_TIMEOUT, KID_COARSE_SUM, (uint32_t)b);
        mbar_wait(&bar, phase);
      }
      return;
    }
    phase ^= 1u;
    const int ne = (int)(n_e < (int64_t)nb * kBlockEntries ? n_e : (int64_t)nb * kBlockEntries);
#pragma unroll 8
    for (int i = 0; i < ne; ++i) {
      const uint8_t* blk = stage + (i >> 3) * bb;
      const int slot = i & 7;
      // both nibbles of the byte to fp16 (exact), this thread's element, times the group scale (exact in
      // fp32), added in ascending entry order
      const uint32_t h2 = e2m1x2_to_f16x2(blk[slot * half + d / 2]);
      const float x = __half2float(__ushort_as_half((unsigned short)((d & 1) ? (h2 >> 16) : (h2 & 0xFFFFu))));
      const float sc = e4m3_to_float(blk[kBlockEntries * half + slot * groups + d / kGroup]);
      acc = __fadd_rn(acc, __fmul_rn(x, sc));
    }
  }
  p.coarse_sum[b * p.coarse_stride_b + g * p.dim + d] = acc;
}

}  // namespace

cudaError_t launch_pack(const PackParams& p, cudaStream_t s) {
  const int64_t total = p.batch * p.n_new * (p.dim / kGroup);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  ProfScope prof("pack_fp4", s);
  clear_stale_error();
  pack_fp4_kernel<<<(unsigned)blocks, threads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_coarse_sum(const PackParams& p, cudaStream_t s) {
  if (p.coarse_sum == nullptr || p.n_new == 0 || p.batch == 0) return cudaSuccess;
  const int64_t per_super = (int64_t)kSuper * kBlockEntries;
  const int touched = (int)((p.n_new + per_super - 1) / per_super) + 1;
  dim3 grid((unsigned)touched, (unsigned)p.batch);
  ProfScope prof("coarse_sum", s);
  clear_stale_error();
  coarse_sum_kernel<<<grid, p.dim, 0, s>>>(p, touched);
  return cudaGetLastError();
}

}  // namespace csa
