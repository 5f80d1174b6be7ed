// Sparse attention over selected FP4 cache blocks merged with the sliding window, split over the row
// list, plus the fixed-order log-sum-exp combine of the splits.
//
// Follows "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression" (paper-digest), Core
// Mechanics ("one 512-dim latent shares keys and values across all attention heads") and Terminology
// (sliding window of 128), and "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (card),
// Key ideas ("Every layer keeps its own query and sliding-window KV").
//
// Design. A CTA owns one query (all heads, 16 per head group, one warp quad per group) and a
// contiguous range of 64-row tiles of its row list: first the selected blocks (8 per tile), then the
// window (64 rows per tile). The raw FP4 blocks of the next tile are copied into shared memory with
// cp.async while the current tile is computed. A tile is dequantised once into a swizzled fp16 [64 x 512]
// tile (exact: E2M1 x E4M3 fits fp16) that serves as K for the logits and as V for the output; the
// window rows (bf16) are converted to fp16 on the way in. Logits and the P.V product run on mma.sync
// m16n8k16 (fp16 in, fp32 accumulate) with operands fetched by ldmatrix; the online softmax keeps the
// running max and sum per head in shared memory and rescales the fp32 output registers. Splits write
// unnormalised partials (o, m, l); the combine kernel merges them in split order.
#include "csa_internal.cuh"

namespace csa {
namespace {

constexpr int kTileRows = 64;
constexpr int kRowBytes = kLatent * 2;                    // fp16 row of the [64 x 512] tile
constexpr int kLatBlockBytes = block_bytes(kLatent);      // 2304
constexpr int kSsStride = kTileRows + 4;                  // fp32 logits row stride (floats)
constexpr int kPsStride = kTileRows * 2 + 16;             // fp16 probabilities row stride (bytes)
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint32_t swz(int row, int chunk) {     // byte offset in a [row][512] fp16 tile
  return (uint32_t)(row * kRowBytes + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" :: "r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// 8 bf16 -> 8 fp16 (packed in a uint4)
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
    __half2 h = __floats2half2_rn(lo, hi);
    o[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

struct UnitInfo {
  int64_t n_e, n_b, pos;
  bool prefill;
};

// Block id in slot j of block tile t, and whether it may be read.
__device__ __forceinline__ int64_t tile_block(const AttnParams& p, int64_t unit, int t, int j,
                                              const UnitInfo& ui, bool* ok) {
  const int slot = t * kBlockEntries + j;
  int64_t id = -1;
  if (slot < p.top_k) id = __ldg(p.idx + unit * p.top_k + slot);
  *ok = id >= 0 && id < ui.n_b;
  return id;
}

template <int HG>
struct Smem {
  static constexpr int H = 16 * HG;
  static constexpr int q_off = 0;
  static constexpr int kv_off = q_off + H * kRowBytes;
  static constexpr int raw_off = kv_off + kTileRows * kRowBytes;
  static constexpr int ss_off = raw_off + kBlockEntries * kLatBlockBytes;
  static constexpr int ps_off = ss_off + H * kSsStride * 4;
  static constexpr int stat_off = ps_off + H * kPsStride;
  static constexpr int rowv_off = stat_off + 3 * H * 4;
  static constexpr int bytes = rowv_off + kTileRows;
};

template <int HG>
__global__ void __launch_bounds__(128 * HG, 1) attn_kernel(AttnParams p) {
  using S = Smem<HG>;
  constexpr int H = S::H;
  constexpr int NT = 128 * HG;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* qs = smem + S::q_off;
  uint8_t* kv = smem + S::kv_off;
  uint8_t* raw = smem + S::raw_off;
  float* ss = reinterpret_cast<float*>(smem + S::ss_off);
  uint8_t* ps = smem + S::ps_off;
  float* m_run = reinterpret_cast<float*>(smem + S::stat_off);
  float* l_run = m_run + H;
  float* alpha = l_run + H;
  uint8_t* rowv = smem + S::rowv_off;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int split = blockIdx.x;
  const int64_t unit = blockIdx.y;
  const int64_t b = unit / p.n_query;

  UnitInfo ui;
  ui.n_e = __ldg(p.n_entries + b);
  if (ui.n_e < 0 || ui.n_e > p.max_entries) {
    if (tid == 0 && split == 0) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_ATTN, (uint32_t)b);
    ui.n_e = ui.n_e < 0 ? 0 : p.max_entries;
  }
  ui.n_b = (ui.n_e + kBlockEntries - 1) / kBlockEntries;
  ui.prefill = p.q_pos != nullptr;
  ui.pos = ui.prefill ? (int64_t)__ldg(p.q_pos + unit) : INT64_MAX;
  const int64_t nb_cap = (p.max_entries + kBlockEntries - 1) / kBlockEntries;

  const int nbt = (p.top_k + kBlockEntries - 1) / kBlockEntries;
  const int t0 = (int)((int64_t)split * p.tiles / p.splits);
  const int t1 = (int)((int64_t)(split + 1) * p.tiles / p.splits);
  const uint8_t* seq = p.cache + b * p.cache_stride_b;

  // ---- query rows -> fp16, swizzled
  const __nv_bfloat16* qg = p.q + unit * (int64_t)H * kLatent;
  for (int i = tid; i < H * 64; i += NT) {
    const int row = i >> 6, ch = i & 63;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(qg + row * kLatent + ch * 8));
    *reinterpret_cast<uint4*>(qs + swz(row, ch)) = bf16x8_to_f16x8(v);
  }
  for (int i = tid; i < H; i += NT) { m_run[i] = -INFINITY; l_run[i] = 0.0f; alpha[i] = 1.0f; }

  // raw copy of the 8 blocks of block tile t (valid ones only)
  auto issue = [&](int t) {
    for (int i = tid; i < kBlockEntries * (kLatBlockBytes / 16); i += NT) {
      const int j = i / (kLatBlockBytes / 16), ch = i % (kLatBlockBytes / 16);
      bool ok;
      const int64_t id = tile_block(p, unit, t, j, ui, &ok);
      if (ok) cp_async16(smem_u32(raw + j * kLatBlockBytes + ch * 16), seq + id * kLatBlockBytes + ch * 16);
      if (ch == 0 && (id < -1 || id >= nb_cap)) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_ATTN, (uint32_t)unit);
    }
    cp_async_commit();
  };
  if (t0 < t1 && t0 < nbt) issue(t0);

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  const int hg = warp >> 2, quarter = warp & 3;

  for (int t = t0; t < t1; ++t) {
    cp_async_wait_all();
    __syncthreads();                                                     // (A)
    if (t < nbt) {
      // ---- dequantise the 8 raw blocks: one 16-element group per thread step
      for (int i = tid; i < kTileRows * 32; i += NT) {
        const int row = i >> 5, grp = i & 31;
        const int j = row >> 3, slot = row & 7;
        bool ok;
        const int64_t id = tile_block(p, unit, t, j, ui, &ok);
        const int64_t e = id * kBlockEntries + slot;
        const bool valid = ok && e < ui.n_e && 2 * e + 1 <= ui.pos;
        uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
        if (valid) {
          const uint8_t* blk = raw + j * kLatBlockBytes;
          const uint2 cb = *reinterpret_cast<const uint2*>(blk + slot * (kLatent / 2) + grp * 8);
          const uint32_t sc = e4m3_to_f16x2_bcast(blk[kBlockEntries * (kLatent / 2) + slot * 32 + grp]);
          uint32_t h[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            h[k] = hmul2_u32(e2m1x2_to_f16x2((cb.x >> (8 * k)) & 0xFFu), sc);
            h[4 + k] = hmul2_u32(e2m1x2_to_f16x2((cb.y >> (8 * k)) & 0xFFu), sc);
          }
          w0 = make_uint4(h[0], h[1], h[2], h[3]);
          w1 = make_uint4(h[4], h[5], h[6], h[7]);
        }
        *reinterpret_cast<uint4*>(kv + swz(row, 2 * grp)) = w0;
        *reinterpret_cast<uint4*>(kv + swz(row, 2 * grp + 1)) = w1;
        if (grp == 0) rowv[row] = valid ? 1 : 0;
      }
    } else {
      // ---- window rows (bf16 -> fp16)
      const int s0 = (t - nbt) * kTileRows;
      for (int i = tid; i < kTileRows * 64; i += NT) {
        const int row = i >> 6, ch = i & 63;
        const int slot = s0 + row;
        bool valid = slot < p.window;
        int64_t src = slot;
        if (ui.prefill) {
          const int64_t first = __ldg(p.swa_first_pos + b);
          const int64_t tok = ui.pos - p.window + 1 + slot;
          valid = valid && tok >= first;
          src = tok - first;
        } else {
          valid = valid && slot < __ldg(p.swa_len + b);
        }
        if (valid && (src < 0 || src >= p.swa_rows)) {
          if (ch == 0) report(p.hdr, CSA_ERR_DEVICE_CHECK, KID_ATTN, (uint32_t)unit);
          valid = false;
        }
        uint4 v = make_uint4(0, 0, 0, 0);
        if (valid) {
          v = __ldg(reinterpret_cast<const uint4*>(p.swa + b * p.swa_stride_b + src * kLatent + ch * 8));
          v = bf16x8_to_f16x8(v);
        }
        *reinterpret_cast<uint4*>(kv + swz(row, ch)) = v;
        if (ch == 0) rowv[row] = valid ? 1 : 0;
      }
    }
    __syncthreads();                                                     // (B)
    if (t + 1 < t1 && t + 1 < nbt) issue(t + 1);

    // ---- logits: warp (hg, quarter) -> heads 16 hg.., rows 16 quarter..
    {
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int arow = 16 * hg + (lane & 15);
      const int brow = 16 * quarter + (lane & 7) + ((lane >> 4) << 3);
      const uint32_t qbase = smem_u32(qs), kbase = smem_u32(kv);
#pragma unroll 8
      for (int kk = 0; kk < 32; ++kk) {
        uint32_t a[4], bb[4];
        ldsm_x4(qbase + swz(arow, 2 * kk + (lane >> 4)), a);
        ldsm_x4(kbase + swz(brow, 2 * kk + ((lane >> 3) & 1)), bb);
        mma16816(acc[0], a, bb[0], bb[1]);
        mma16816(acc[1], a, bb[2], bb[3]);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int row = 16 * quarter + 8 * nt + 2 * c;
        const bool v0 = rowv[row], v1 = rowv[row + 1];
        const int h0 = 16 * hg + g;
        float* s0 = ss + h0 * kSsStride + row;
        float* s1 = ss + (h0 + 8) * kSsStride + row;
        s0[0] = v0 ? acc[nt][0] * p.scale_log2 : -INFINITY;
        s0[1] = v1 ? acc[nt][1] * p.scale_log2 : -INFINITY;
        s1[0] = v0 ? acc[nt][2] * p.scale_log2 : -INFINITY;
        s1[1] = v1 ? acc[nt][3] * p.scale_log2 : -INFINITY;
      }
    }
    __syncthreads();                                                     // (C)

    // ---- online softmax: 8 threads per head, 8 rows each
    {
      const int head = tid >> 3, part = tid & 7;
      const float m_old = m_run[head];
      const float4 x0 = *reinterpret_cast<const float4*>(ss + head * kSsStride + part * 8);
      const float4 x1 = *reinterpret_cast<const float4*>(ss + head * kSsStride + part * 8 + 4);
      float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      float mx = v[0];
#pragma unroll
      for (int i = 1; i < 8; ++i) mx = fmaxf(mx, v[i]);
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m_old, mx);
      const float m_use = m_new == -INFINITY ? 0.0f : m_new;
      float sum = 0.0f;
      uint32_t ph[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float p0 = exp2f(v[2 * i] - m_use), p1 = exp2f(v[2 * i + 1] - m_use);
        sum += p0 + p1;
        __half2 hh = __floats2half2_rn(p0, p1);
        ph[i] = *reinterpret_cast<uint32_t*>(&hh);
      }
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      *reinterpret_cast<uint4*>(ps + head * kPsStride + part * 16) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
      if (part == 0) {
        const float a = exp2f(m_old - m_use);
        alpha[head] = a;
        l_run[head] = l_run[head] * a + sum;
        m_run[head] = m_new;
      }
    }
    __syncthreads();                                                     // (D)

    // ---- o = alpha * o + P V: warp (hg, quarter) -> heads 16 hg.., d in [128 quarter, +128)
    {
      const float a0 = alpha[16 * hg + g], a1 = alpha[16 * hg + g + 8];
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        o[nt][0] *= a0; o[nt][1] *= a0; o[nt][2] *= a1; o[nt][3] *= a1;
      }
      const uint32_t pbase = smem_u32(ps), kbase = smem_u32(kv);
      const int prow = 16 * hg + (lane & 15);
      const int mi = lane >> 3;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4];
        ldsm_x4(pbase + prow * kPsStride + (2 * ks + (lane >> 4)) * 16, a);
        const int vrow = 16 * ks + (lane & 7) + (mi & 1) * 8;
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t bb[4];
          ldsm_x4_t(kbase + swz(vrow, 16 * quarter + 2 * np + (mi >> 1)), bb);
          mma16816(o[2 * np], a, bb[0], bb[1]);
          mma16816(o[2 * np + 1], a, bb[2], bb[3]);
        }
      }
    }
  }
  __syncthreads();

  // ---- epilogue
  const int h0 = 16 * hg + g, h1 = h0 + 8;
  const float l0 = l_run[h0], l1 = l_run[h1];
  if (p.splits == 1) {
    const float i0 = l0 > 0.0f ? 1.0f / l0 : 0.0f, i1 = l1 > 0.0f ? 1.0f / l1 : 0.0f;
    float* out0 = p.out + (unit * H + h0) * (int64_t)kLatent + 128 * quarter + 2 * c;
    float* out1 = p.out + (unit * H + h1) * (int64_t)kLatent + 128 * quarter + 2 * c;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      *reinterpret_cast<float2*>(out0 + 8 * nt) = make_float2(o[nt][0] * i0, o[nt][1] * i0);
      *reinterpret_cast<float2*>(out1 + 8 * nt) = make_float2(o[nt][2] * i1, o[nt][3] * i1);
    }
    if (p.out_lse != nullptr && quarter == 0 && c == 0) {
      p.out_lse[unit * H + h0] = l0 > 0.0f ? (m_run[h0] + log2f(l0)) * kLn2 : -INFINITY;
      p.out_lse[unit * H + h1] = l1 > 0.0f ? (m_run[h1] + log2f(l1)) * kLn2 : -INFINITY;
    }
  } else {
    const int64_t prow = (unit * p.splits + split) * H;
    float* out0 = p.part_o + (prow + h0) * kLatent + 128 * quarter + 2 * c;
    float* out1 = p.part_o + (prow + h1) * kLatent + 128 * quarter + 2 * c;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      *reinterpret_cast<float2*>(out0 + 8 * nt) = make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2*>(out1 + 8 * nt) = make_float2(o[nt][2], o[nt][3]);
    }
    if (quarter == 0 && c == 0) {
      *reinterpret_cast<float2*>(p.part_ml + (prow + h0) * 2) = make_float2(m_run[h0], l0);
      *reinterpret_cast<float2*>(p.part_ml + (prow + h1) * 2) = make_float2(m_run[h1], l1);
    }
  }
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

template <int HG>
cudaError_t launch_attn_t(const AttnParams& p, cudaStream_t s) {
  const int bytes = Smem<HG>::bytes;
  clear_stale_error();
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<HG>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.splits, (unsigned)p.units);
  attn_kernel<HG><<<grid, 128 * HG, bytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn(const AttnParams& p, cudaStream_t s) {
  if (p.units == 0) return cudaSuccess;
  ProfScope prof("sparse_attn", s);
  switch (p.heads) {
    case 16: return launch_attn_t<1>(p, s);
    case 32: return launch_attn_t<2>(p, s);
    case 48: return launch_attn_t<3>(p, s);
    case 64: return launch_attn_t<4>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine(const AttnParams& p, cudaStream_t s) {
  if (p.units == 0 || p.splits == 1) return cudaSuccess;
  ProfScope prof("attn_combine", s);
  clear_stale_error();
  combine_kernel<<<(unsigned)(p.units * p.heads), 128, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace csa
