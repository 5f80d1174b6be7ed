// Pair-merge + FP4 quantiser + block-major store, and the super-block coarse-key sums.
//
// Follows "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression" (paper-digest), Core
// Mechanics ("Sequence: the Encoder merges 2 adjacent positions into 1 cache entry") and the FP4 global
// KV of "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (card), Key ideas. The numeric
// format (E2M1 codes, E4M3 scale per 16 elements, amax/6 or power-of-two scale) is this library's own and
// is stated in include/csa.h; every fp32 step uses an explicit round-to-nearest intrinsic so that the
// bytes do not depend on contraction or fast-math choices.
//
// Four threads (a quad) quantise one 16-element group, four elements each: the group maximum is taken with
// two shuffles inside the quad, each thread divides and encodes its own four elements and stores their two
// code bytes, and the quad's first thread stores the scale byte. A warp covers 8 consecutive groups, so
// loads and stores are contiguous across the warp.
#include "csa_internal.cuh"

namespace csa {
namespace {

__device__ __forceinline__ void load4(const void* base, int dtype, int64_t elem_off, float* v) {
  if (dtype == CSA_DTYPE_BF16) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + elem_off));
    v[0] = __uint_as_float(w.x << 16);
    v[1] = __uint_as_float(w.x & 0xFFFF0000u);
    v[2] = __uint_as_float(w.y << 16);
    v[3] = __uint_as_float(w.y & 0xFFFF0000u);
  } else {
    const float4 f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem_off));
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  }
}

__global__ void __launch_bounds__(256) pack_fp4_kernel(PackParams p) {
  const int groups = p.dim / kGroup;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t gt = t >> 2;                     // the group of this thread's quad
  const int j = (int)(t & 3);                    // elements 4 j .. 4 j + 3 of the group
  const int64_t total = p.batch * p.n_new * groups;
  if (gt >= total) return;                       // whole quads leave together
  const int g = (int)(gt % groups);
  const int64_t i = (gt / groups) % p.n_new;
  const int64_t b = gt / ((int64_t)groups * p.n_new);

  const int64_t first = p.first_entry ? (int64_t)p.first_entry[b] : 0;
  if (first < 0 || first + p.n_new > p.max_entries) {
    if (i == 0 && g == 0 && j == 0) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_PACK, (uint32_t)b);
    return;
  }

  float m[4];
  const int64_t el = b * p.x_stride_b + (int64_t)g * kGroup + 4 * j;
  if (p.merge == 2) {
    float a[4], c[4];
    load4(p.x, p.x_dtype, el + (2 * i) * p.x_stride_t, a);
    load4(p.x, p.x_dtype, el + (2 * i + 1) * p.x_stride_t, c);
#pragma unroll
    for (int k = 0; k < 4; ++k) m[k] = __fmul_rn(__fadd_rn(a[k], c[k]), 0.5f);
  } else {
    load4(p.x, p.x_dtype, el + i * p.x_stride_t, m);
  }

  float amax = fmaxf(fmaxf(fabsf(m[0]), fabsf(m[1])), fmaxf(fabsf(m[2]), fabsf(m[3])));
  const unsigned quad = 0xFu << (threadIdx.x & 28u);
  amax = fmaxf(amax, __shfl_xor_sync(quad, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(quad, amax, 2));
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

  uint32_t codes = 0;                            // two bytes: elements 4 j .. 4 j + 3, low nibble first
  if (s > 0.0f) {
#pragma unroll
    for (int k = 0; k < 4; ++k) codes |= e2m1_code(__fdiv_rn(m[k], s)) << (4 * k);
  }

  const int64_t e = first + i;
  uint8_t* blk = p.cache + b * p.cache_stride_b + (e / kBlockEntries) * (int64_t)block_bytes(p.dim);
  const int slot = (int)(e % kBlockEntries);
  *reinterpret_cast<uint16_t*>(blk + slot * (p.dim / 2) + g * 8 + 2 * j) = (uint16_t)codes;
  if (j == 0) blk[kBlockEntries * (p.dim / 2) + slot * groups + g] = (uint8_t)sbyte;
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
  const int64_t total = 4 * p.batch * p.n_new * (p.dim / kGroup);      // four threads per group
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
