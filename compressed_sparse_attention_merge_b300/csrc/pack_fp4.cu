// Pair-merge + FP4 quantiser + block-major store, and the super-block coarse-key sums.
//
// Follows "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression" (paper-digest), Core
// Mechanics ("Sequence: the Encoder merges 2 adjacent positions into 1 cache entry") and the FP4 global
// KV of "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (card), Key ideas. The numeric
// format (E2M1 codes, E4M3 scale per 16 elements, amax/6 or power-of-two scale) is this library's own and
// is stated in include/csa.h; every fp32 step uses an explicit round-to-nearest intrinsic so that the
// bytes do not depend on contraction or fast-math choices.
//
// TPG threads quantise one 16-element group, 16 / TPG elements each. With TPG = 4 (small calls, such as
// the per-step append) the group maximum is taken with two shuffles inside the quad and each thread
// divides and encodes four elements, which shortens the per-thread chain; with TPG = 1 (bulk calls) a
// thread takes a whole group with two 32-byte loads, which keeps the loads wide. Either way a warp's loads
// and stores are contiguous, and the first thread of a group stores its scale byte.
#include "csa_internal.cuh"

namespace csa {
namespace {

// n (4 or 16) consecutive elements from elem_off (a multiple of n) as fp32.
template <int n>
__device__ __forceinline__ void load_n(const void* base, int dtype, int64_t elem_off, float* v) {
  if (dtype == CSA_DTYPE_BF16) {
    uint32_t w[n / 2];
    if (n >= 8) {
      const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + elem_off);
#pragma unroll
      for (int i = 0; i < n / 8; ++i) {
        const uint4 x = __ldg(p + i);
        w[4 * i] = x.x; w[4 * i + 1] = x.y; w[4 * i + 2] = x.z; w[4 * i + 3] = x.w;
      }
    } else {
      const uint2 x = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + elem_off));
      w[0] = x.x; w[1] = x.y;
    }
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem_off);
#pragma unroll
    for (int i = 0; i < n / 4; ++i) {
      const float4 f = __ldg(p + i);
      v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
  }
}

// Thread t of a pack job: element slice j = t % TPG of group t / TPG.
template <int TPG>
__device__ __forceinline__ void pack_thread(const PackParams& p, int64_t t) {
  constexpr int EPT = kGroup / TPG;              // elements per thread
  const int groups = p.dim / kGroup;
  const int64_t gt = t / TPG;                    // this thread's group
  const int j = (int)(t % TPG);                  // elements EPT j .. EPT j + EPT - 1 of the group
  const int64_t total = p.batch * p.n_new * groups;
  if (gt >= total) return;                       // the threads of a group leave together
  const int g = (int)(gt % groups);
  const int64_t i = (gt / groups) % p.n_new;
  const int64_t b = gt / ((int64_t)groups * p.n_new);

  const int64_t first = p.first_entry ? (int64_t)p.first_entry[b] : 0;
  if (first < 0 || first + p.n_new > p.max_entries) {
    if (i == 0 && g == 0 && j == 0) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_PACK, (uint32_t)b);
    return;
  }

  float m[EPT];
  const int64_t el = b * p.x_stride_b + (int64_t)g * kGroup + EPT * j;
  if (p.merge == 2) {
    float a[EPT], c[EPT];
    load_n<EPT>(p.x, p.x_dtype, el + (2 * i) * p.x_stride_t, a);
    load_n<EPT>(p.x, p.x_dtype, el + (2 * i + 1) * p.x_stride_t, c);
#pragma unroll
    for (int k = 0; k < EPT; ++k) m[k] = __fmul_rn(__fadd_rn(a[k], c[k]), 0.5f);
  } else {
    load_n<EPT>(p.x, p.x_dtype, el + i * p.x_stride_t, m);
  }

  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < EPT; ++k) amax = fmaxf(amax, fabsf(m[k]));
  if (TPG == 4) {
    const unsigned quad = 0xFu << (threadIdx.x & 28u);
    amax = fmaxf(amax, __shfl_xor_sync(quad, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(quad, amax, 2));
  }
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

  uint32_t codes[EPT / 8 > 0 ? EPT / 8 : 1] = {};    // EPT / 2 code bytes, low nibble first
  if (s > 0.0f) {
#pragma unroll
    for (int k = 0; k < EPT; ++k) codes[k / 8] |= e2m1_code(__fdiv_rn(m[k], s)) << (4 * (k % 8));
  }

  const int64_t e = first + i;
  uint8_t* blk = p.cache + b * p.cache_stride_b + (e / kBlockEntries) * (int64_t)block_bytes(p.dim);
  const int slot = (int)(e % kBlockEntries);
  uint8_t* dst = blk + slot * (p.dim / 2) + g * 8 + (EPT / 2) * j;
  if (EPT == 16) *reinterpret_cast<uint2*>(dst) = make_uint2(codes[0], codes[EPT / 8 > 1 ? 1 : 0]);
  else *reinterpret_cast<uint16_t*>(dst) = (uint16_t)codes[0];
  if (j == 0) blk[kBlockEntries * (p.dim / 2) + slot * groups + g] = (uint8_t)sbyte;
}

template <int TPG>
__global__ void __launch_bounds__(256) pack_fp4_kernel(PackParams p) {
  griddep_wait();                                  // before any access: the cache may still be read before
  griddep_launch();
  pack_thread<TPG>(p, (int64_t)blockIdx.x * blockDim.x + threadIdx.x);
}

// Several jobs in one launch; each CTA belongs to one job (its CTA range in m.cta_begin).
template <int TPG>
__global__ void __launch_bounds__(256) pack_fp4_multi_kernel(const __grid_constant__ PackMulti m) {
  griddep_wait();                                  // before any access: the caches may still be read before
  griddep_launch();
  int j = 0;
  while (j + 1 < m.n && (int64_t)blockIdx.x >= m.cta_begin[j + 1]) ++j;
  pack_thread<TPG>(m.job[j], ((int64_t)blockIdx.x - m.cta_begin[j]) * blockDim.x + threadIdx.x);
}

// coarse_sum[b][g][d] = the exact sum, rounded once to fp32, of the dequantised element d of entries
// [512 g, min(512 (g + 1), first + n_new)), for every super-block g touched by this call. One CTA per
// (super-block, 32 columns, sequence): the super-block's packed bytes are staged through shared memory in
// chunks, each one bulk copy; the 32 warps take slices of the entries, each lane summing its column in int64
// fixed point (2^13 times a dequantised key is an integer), and the slices' sums are added and rounded at the
// end.
constexpr int kCoarseStage = 36864;

__global__ void __launch_bounds__(1024) coarse_sum_kernel(PackParams p, int touched) {
  __shared__ __align__(16) uint8_t stage[kCoarseStage];
  __shared__ long long part[1024];
  __shared__ __align__(8) uint64_t bar;
  griddep_wait();                                // before any access: the packed entries come from the kernel before
  griddep_launch();
  // thread = (column d, slice of the entries): a dequantised key is a multiple of 2^-13 below 2,688 in
  // magnitude, so 2^13 times it is an integer and the slices' int64 sums add up to the exact sum in any order,
  // rounded once to fp32 at the end
  // a CTA takes 32 columns of one super-block (grid.x = touched super-blocks x dim / 32): lane = column,
  // warp = slice of the entries
  const int ncg = p.dim / 32;
  const int d = (blockIdx.x % ncg) * 32 + (threadIdx.x & 31);
  const int sl = threadIdx.x >> 5;
  const int slices = blockDim.x >> 5;
  const int gl = blockIdx.x / ncg;
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
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  long long acc = 0;
  uint32_t phase = 0;
  for (int64_t blk0 = g * kSuper; blk0 * kBlockEntries < e_hi; blk0 += chunk_blocks) {
    const int64_t n_e = e_hi - blk0 * kBlockEntries;
    const int nb = (int)((n_e + kBlockEntries - 1) / kBlockEntries < chunk_blocks
                             ? (n_e + kBlockEntries - 1) / kBlockEntries : chunk_blocks);
    __syncthreads();                             // the previous chunk has been read (and bar initialised)
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(&bar, (uint32_t)(nb * bb));
      bulk_g2s(stage, seq + blk0 * bb, (uint32_t)(nb * bb), &bar);
    }
    if (!__syncthreads_and(mbar_wait(&bar, phase))) {
      // give up: report, let the copy land (bounded), leave without writing a sum
      if (threadIdx.x == 0) {
        report(p.hdr, CSA_ERR_TIMEOUT, KID_COARSE_SUM, (uint32_t)b);
        mbar_wait(&bar, phase);
      }
      return;
    }
    phase ^= 1u;
    const int ne = (int)(n_e < (int64_t)nb * kBlockEntries ? n_e : (int64_t)nb * kBlockEntries);
#pragma unroll 4
    for (int i = sl; i < ne; i += slices) {
      const uint8_t* blk = stage + (i >> 3) * bb;
      const int slot = i & 7;
      // 2^13 times the dequantised element, from the bits: the E2M1 magnitude in halves (0, 1, 2, 3, 4, 6, 8,
      // 12 for codes 0-7) times 2^12 times the E4M3 scale ((8 + m) 2^(e + 2) for exponent field e > 0, 8 m
      // for a subnormal), below 2^25
      const uint32_t code = ((uint32_t)blk[slot * half + d / 2] >> (4 * (d & 1))) & 0xFu;
      const int c2 = (int)((0xC8643210u >> (4 * (code & 7u))) & 0xFu);
      const uint32_t sb = blk[kBlockEntries * half + slot * groups + d / kGroup];
      const uint32_t e = (sb >> 3) & 0xFu, m = sb & 7u;
      const int s12 = e == 0u ? (int)(m << 3) : (int)((8u + m) << (e + 2u));
      const int v = c2 * s12;
      acc += (code & 8u) ? -(long long)v : (long long)v;
    }
  }
  part[threadIdx.x] = acc;
  __syncthreads();
  if (sl == 0) {
    long long sum = 0;
    for (int k = 0; k < slices; ++k) sum += part[k * 32 + (threadIdx.x & 31)];
    p.coarse_sum[b * p.coarse_stride_b + g * p.dim + d] = __fmul_rn(__ll2float_rn(sum), 1.0f / 8192.0f);
  }
}

}  // namespace

cudaError_t launch_pack(const PackParams& p, cudaStream_t s) {
  const int64_t groups = p.batch * p.n_new * (p.dim / kGroup);
  if (groups == 0) return cudaSuccess;
  const int threads = 256;
  ProfScope prof("pack_fp4", s);
  clear_stale_error();
  // a quad per group while the call is smaller than eight 256-thread CTAs on each of 148 SMs (the modes
  // write the same bytes; the choice only trades per-thread latency against load width)
  // (a programmatic dependent: the kernel waits before its first access)
  if (groups * 4 <= (int64_t)8 * threads * 148)
    return launch_ex(pack_fp4_kernel<4>, dim3((unsigned)((groups * 4 + threads - 1) / threads)), dim3(threads), 0, s,
                     true, p);
  return launch_ex(pack_fp4_kernel<1>, dim3((unsigned)((groups + threads - 1) / threads)), dim3(threads), 0, s, true, p);
}

cudaError_t launch_pack_multi(const PackParams* jobs, int n, cudaStream_t s) {
  const int threads = 256;
  int64_t total = 0;
  for (int j = 0; j < n; ++j) total += jobs[j].batch * jobs[j].n_new * (jobs[j].dim / kGroup);
  if (total == 0) return cudaSuccess;
  // the same per-group choice as launch_pack, taken on the jobs' total
  const int tpg = total * 4 <= (int64_t)8 * threads * 148 ? 4 : 1;
  PackMulti m{};
  int64_t ctas = 0;
  for (int j = 0; j < n; ++j) {
    const int64_t groups = jobs[j].batch * jobs[j].n_new * (jobs[j].dim / kGroup);
    if (groups == 0) continue;
    m.job[m.n] = jobs[j];
    m.cta_begin[m.n] = ctas;
    ctas += (groups * tpg + threads - 1) / threads;
    ++m.n;
  }
  m.cta_begin[m.n] = ctas;
  ProfScope prof("pack_fp4", s);
  clear_stale_error();
  if (tpg == 4) return launch_ex(pack_fp4_multi_kernel<4>, dim3((unsigned)ctas), dim3(threads), 0, s, true, m);
  return launch_ex(pack_fp4_multi_kernel<1>, dim3((unsigned)ctas), dim3(threads), 0, s, true, m);
}

cudaError_t launch_coarse_sum(const PackParams& p, cudaStream_t s) {
  if (p.coarse_sum == nullptr || p.n_new == 0 || p.batch == 0) return cudaSuccess;
  const int64_t per_super = (int64_t)kSuper * kBlockEntries;
  const int touched = (int)((p.n_new + per_super - 1) / per_super) + 1;
  // dim / 32 CTAs per touched super-block (dim is 64, 128 or 256), 1024 threads: 32 columns x 32 slices
  dim3 grid((unsigned)(touched * (p.dim / 32)), (unsigned)p.batch);
  ProfScope prof("coarse_sum", s);
  clear_stale_error();
  return launch_ex(coarse_sum_kernel, grid, dim3(1024u), 0, s, true, p, touched);
}

}  // namespace csa
