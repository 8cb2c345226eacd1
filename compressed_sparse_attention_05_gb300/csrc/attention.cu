// Gathered sparse MQA attention over the selected compressed entries plus
// the FP8 sliding window.  "DeepSeek-V4.1 架构解析" §02 (fewer KV heads, attend
// over the Top-K) and §03 (FP4 main KV dequantised before the matmul; SWA
// kept in FP8, the last 128 raw tokens).  Head layout, key set and softmax:
// reading R11 of include/csa2.h.
//
// One CTA per (query token, group of 16 heads), 8 warps.  Per 64-key tile:
// gather + dequantise the keys into shared memory, S = Q K^T on tensor cores
// (m16n8k16, each warp 8 keys), online softmax in fp32 (exp2 domain), then
// O += P V with each warp owning an eighth of the value channels.  K = V: the
// same shared-memory tile feeds both products.
//
// Operands are fp16.  MXFP4 entries are converted by cvt.rn.f16x2.e2m1x2 and
// scaled in f16x2: e2m1 * e4m3 has at most 6 significant bits and lies in
// [2^-10, 2688], so the values are exactly the bf16 dequantised latent.  Q and
// the window rows are first rounded to bf16 (the operands the method
// specifies) and carried in fp16, which holds every bf16 value of magnitude
// in [2^-14, 65504] exactly; P is rounded to fp16 (11 significant bits).
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace csa2 {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kTK = 64;       // keys per tile
constexpr int kHG = 16;       // heads per CTA

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two E2M1 codes (one byte, even channel in the low nibble) -> f16x2, low half first.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(r) : "r"(byte));
  return r;
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// An fp32 value holding a bf16 value -> fp16 bits (exact inside the fp16 range).
__device__ __forceinline__ uint32_t f32_to_f16_bits(float f) {
  return (uint32_t)__half_as_ushort(__float2half_rn(f));
}

template <int D>
struct AttnSmem {
  static constexpr int QS = D + 8;     // row stride (elements) of Q and K tiles
  static constexpr int PS = kTK + 8;   // row stride of P
  uint16_t q[kHG * QS];
  uint16_t k[kTK * QS];
  float s[kHG * kTK];
  uint16_t p[kHG * PS];
  int64_t key_src[kTK];                // >= 0 main-KV slot; <= -2 window row (-2 - r); -1 none
  float m[kHG], l[kHG], alpha[kHG];
};

// Dequantise one 16-channel group of a key into 16 fp16 values in shared memory.
template <int D>
__device__ __forceinline__ void dequant_group(const AttnArgs& a, int b, int64_t src, int grp,
                                              uint16_t* dst) {
  uint32_t w[8];
  if (src >= 0) {
    const uint2 c = *reinterpret_cast<const uint2*>(a.kv_codes + src * (D / 2) + grp * 8);
    const float sc = e4m3_to_f32(a.kv_scales[src * (D / 16) + grp]);
    const uint32_t s2 = f32_to_f16_bits(sc) * 0x10001u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t word = i < 4 ? c.x : c.y;
      w[i] = hmul2_u32(e2m1x2_to_f16x2((word >> ((i & 3) * 8)) & 0xFFu), s2);  // exact
    }
  } else if (src <= -2) {
    const int64_t wr = (int64_t)b * a.swa_cap + (-2 - src);
    const uint4 c = *reinterpret_cast<const uint4*>(a.swa_codes + wr * D + grp * 16);
    const float sc = a.swa_scales[wr];
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t word = cw[i >> 1];
      const int sh = (i & 1) * 16;
      const float lo = bf16_bits_to_f32(f32_to_bf16_bits(e4m3_to_f32((word >> sh) & 0xFFu) * sc));
      const float hi = bf16_bits_to_f32(f32_to_bf16_bits(e4m3_to_f32((word >> (sh + 8)) & 0xFFu) * sc));
      w[i] = f32_to_f16_bits(lo) | (f32_to_f16_bits(hi) << 16);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = 0;
  }
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads)
k_sparse_attn(AttnArgs a, uint32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  AttnSmem<D>& sm = *reinterpret_cast<AttnSmem<D>*>(smem_raw);
  constexpr int QS = AttnSmem<D>::QS, PS = AttnSmem<D>::PS;
  constexpr int DW = D / kAttnWarps;   // value channels per warp
  constexpr int NT = DW / 8;           // 8-wide n-tiles per warp
  const int64_t row = blockIdx.y;
  const int hg = blockIdx.x;
  const int b = (int)(row / a.Tq);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;

  const int t = a.q_pos[row];
  const int nv = n_visible(a.n_entries[b], t);  // bounds the indices checked below
  int n_sel = a.cnt[row];
  if (n_sel < 0 || n_sel > a.K) {
    if (tid == 0) raise_status(status, CSA2_STATUS_BAD_COUNT);
    n_sel = n_sel < 0 ? 0 : a.K;
  }
  const int pos0 = a.swa_cap > 0 ? a.swa_pos0[b] : 0;
  const int w_lo = max(max(0, t - a.W + 1), pos0);
  const int w_hi = min(t, pos0 + a.swa_cap - 1);
  const int n_win = max(0, w_hi - w_lo + 1);
  const int n_keys = n_sel + n_win;

  // Q rows of this head group as fp16 (zero rows past Hq)
  for (int i = tid; i < kHG * (D / 8); i += kAttnThreads) {
    const int h = i / (D / 8), c8 = i % (D / 8);
    const int head = hg * kHG + h;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (head < a.Hq) {
      const uint4 qb = *reinterpret_cast<const uint4*>(a.Q + (row * a.Hq + head) * D + c8 * 8);
      const uint32_t qw[4] = {qb.x, qb.y, qb.z, qb.w};
      uint32_t ov[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ov[j] = f32_to_f16_bits(bf16_bits_to_f32(qw[j] & 0xFFFFu)) |
                (f32_to_f16_bits(bf16_bits_to_f32(qw[j] >> 16)) << 16);
      v = make_uint4(ov[0], ov[1], ov[2], ov[3]);
    }
    *reinterpret_cast<uint4*>(&sm.q[h * QS + c8 * 8]) = v;
  }
  if (tid < kHG) {
    sm.m[tid] = -INFINITY;
    sm.l[tid] = 0.f;
  }

  float o[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  const float sl2 = a.scale * 1.4426950408889634f;  // logits in log2 units

  for (int k0 = 0; k0 < n_keys; k0 += kTK) {
    // ---- key sources of this tile
    if (tid < kTK) {
      const int i = k0 + tid;
      int64_t src = -1;
      if (i < n_sel) {
        const int j = a.idx[row * a.K + i];
        if (j >= 0 && j < nv) src = entry_slot(a.page_table, a.max_pages, a.n_pages, b, j, status);
        else raise_status(status, CSA2_STATUS_BAD_INDEX);
      } else if (i < n_keys) {
        src = -2 - (int64_t)(w_lo + (i - n_sel) - pos0);
      }
      sm.key_src[tid] = src;
    }
    __syncthreads();
    // ---- gather + dequantise
    for (int i = tid; i < kTK * (D / 16); i += kAttnThreads) {
      const int kr = i / (D / 16), grp = i % (D / 16);
      dequant_group<D>(a, b, sm.key_src[kr], grp, &sm.k[kr * QS + grp * 16]);
    }
    __syncthreads();
    // ---- S = Q K^T : warp owns keys 8*warp .. +7
    {
      float s0[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t qa = smem_u32(&sm.q[(lane & 15) * QS + (lane >> 4) * 8]);
      // x4 over keys 8w..8w+7: matrices = 8-channel chunks 0..3 of a 32-channel step
      const uint32_t kb = smem_u32(&sm.k[(warp * 8 + (lane & 7)) * QS + (lane >> 3) * 8]);
#pragma unroll 4
      for (int ks = 0; ks < D / 32; ++ks) {
        uint32_t a0, a1, a2, a3, a4, a5, a6, a7, b0, b1, b2, b3;
        ldsm_x4(qa + ks * 64, a0, a1, a2, a3);
        ldsm_x4(qa + ks * 64 + 32, a4, a5, a6, a7);
        ldsm_x4(kb + ks * 64, b0, b1, b2, b3);
        mma_f16(s0, a0, a1, a2, a3, b0, b1);
        mma_f16(s0, a4, a5, a6, a7, b2, b3);
      }
      const int key0 = warp * 8 + 2 * t4;
      const bool v0 = sm.key_src[key0] != -1, v1 = sm.key_src[key0 + 1] != -1;
      sm.s[g * kTK + key0] = v0 ? s0[0] * sl2 : -INFINITY;
      sm.s[g * kTK + key0 + 1] = v1 ? s0[1] * sl2 : -INFINITY;
      sm.s[(g + 8) * kTK + key0] = v0 ? s0[2] * sl2 : -INFINITY;
      sm.s[(g + 8) * kTK + key0 + 1] = v1 ? s0[3] * sl2 : -INFINITY;
    }
    __syncthreads();
    // ---- online softmax: 16 threads per head, 4 keys each
    {
      const int h = tid >> 4, part = tid & 15;
      const float4 sv = *reinterpret_cast<const float4*>(&sm.s[h * kTK + part * 4]);
      float mx = fmaxf(fmaxf(sv.x, sv.y), fmaxf(sv.z, sv.w));
#pragma unroll
      for (int o2 = 1; o2 < 16; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
      const float m_old = sm.m[h];
      const float m_new = fmaxf(m_old, mx);
      const bool none = m_new == -INFINITY;
      const __half p0 = __float2half_rn(none ? 0.f : exp2f(sv.x - m_new));
      const __half p1 = __float2half_rn(none ? 0.f : exp2f(sv.y - m_new));
      const __half p2 = __float2half_rn(none ? 0.f : exp2f(sv.z - m_new));
      const __half p3 = __float2half_rn(none ? 0.f : exp2f(sv.w - m_new));
      // normalise by the rounded weights that the PV product uses
      float sum = __half2float(p0) + __half2float(p1) + __half2float(p2) + __half2float(p3);
      uint2 pw;
      pw.x = (uint32_t)__half_as_ushort(p0) | ((uint32_t)__half_as_ushort(p1) << 16);
      pw.y = (uint32_t)__half_as_ushort(p2) | ((uint32_t)__half_as_ushort(p3) << 16);
      *reinterpret_cast<uint2*>(&sm.p[h * PS + part * 4]) = pw;
#pragma unroll
      for (int o2 = 1; o2 < 16; o2 <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o2);
      __syncwarp();
      if (part == 0) {
        const float al = none ? 1.f : exp2f(m_old - m_new);
        sm.alpha[h] = al;
        sm.l[h] = sm.l[h] * al + sum;
        sm.m[h] = m_new;
      }
    }
    __syncthreads();
    // ---- O = O * alpha + P V : warp owns channels warp*DW .. +DW
    {
      const float al0 = sm.alpha[g], al1 = sm.alpha[g + 8];
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        o[i][0] *= al0; o[i][1] *= al0; o[i][2] *= al1; o[i][3] *= al1;
      }
      const uint32_t pa = smem_u32(&sm.p[(lane & 15) * PS + (lane >> 4) * 8]);
      const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
      for (int kk = 0; kk < kTK / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(pa + kk * 32, a0, a1, a2, a3);
        const uint32_t vb = smem_u32(&sm.k[(kk * 16 + (mi & 1) * 8 + r8) * QS + warp * DW + (mi >> 1) * 8]);
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + np * 32, b0, b1, b2, b3);
          mma_f16(o[2 * np], a0, a1, a2, a3, b0, b1);
          mma_f16(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
        if (NT & 1) {
          uint32_t b0, b1;
          ldsm_x2_t(smem_u32(&sm.k[(kk * 16 + (lane & 15)) * QS + warp * DW + (NT - 1) * 8]), b0, b1);
          mma_f16(o[NT - 1], a0, a1, a2, a3, b0, b1);
        }
      }
    }
    __syncthreads();
  }

  // ---- normalise and store
  const float l0 = sm.l[g], l1 = sm.l[g + 8];
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const int head0 = hg * kHG + g, head1 = head0 + 8;
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const int ch = warp * DW + i * 8 + 2 * t4;
    if (head0 < a.Hq)
      *reinterpret_cast<float2*>(a.O + (row * a.Hq + head0) * D + ch) = make_float2(o[i][0] * inv0, o[i][1] * inv0);
    if (head1 < a.Hq)
      *reinterpret_cast<float2*>(a.O + (row * a.Hq + head1) * D + ch) = make_float2(o[i][2] * inv1, o[i][3] * inv1);
  }
  if (a.lse && tid < kHG && hg * kHG + tid < a.Hq) {
    const float l = sm.l[tid];
    a.lse[row * a.Hq + hg * kHG + tid] = l > 0.f ? (sm.m[tid] + log2f(l)) * 0.6931471805599453f : -INFINITY;
  }
}

// ---- register-prefetch variant (d = 512) -------------------------------------------
// Same tiling and math as k_sparse_attn, with the gather latency taken off the
// critical path: every key's source (pool slot or window row) is resolved
// once at the start, and the packed bytes of tile t+1 (each thread: 8 groups
// of 16 channels) are loaded into registers while tile t runs its tensor-core
// phases.  90 KB of shared memory keeps two CTAs per SM.
__global__ void __launch_bounds__(kAttnThreads, 2)
k_sparse_attn_rp(AttnArgs a, uint32_t* status) {
  constexpr int D = 512;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  AttnSmem<D>& sm = *reinterpret_cast<AttnSmem<D>*>(smem_raw);
  int64_t* slots = reinterpret_cast<int64_t*>(smem_raw + sizeof(AttnSmem<D>));
  constexpr int QS = AttnSmem<D>::QS, PS = AttnSmem<D>::PS;
  constexpr int DW = D / kAttnWarps, NT = DW / 8;
  constexpr int kItems = kTK * (D / 16) / kAttnThreads;   // 8 groups per thread per tile
  const int64_t row = blockIdx.y;
  const int hg = blockIdx.x;
  const int b = (int)(row / a.Tq);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;

  const int t = a.q_pos[row];
  const int nv = n_visible(a.n_entries[b], t);
  int n_sel = a.cnt[row];
  if (n_sel < 0 || n_sel > a.K) {
    if (tid == 0) raise_status(status, CSA2_STATUS_BAD_COUNT);
    n_sel = n_sel < 0 ? 0 : a.K;
  }
  const int pos0 = a.swa_cap > 0 ? a.swa_pos0[b] : 0;
  const int w_lo = max(max(0, t - a.W + 1), pos0);
  const int w_hi = min(t, pos0 + a.swa_cap - 1);
  const int n_win = max(0, w_hi - w_lo + 1);
  const int n_keys = n_sel + n_win;
  const int n_tiles = (n_keys + kTK - 1) / kTK;

  for (int i = tid; i < n_keys; i += kAttnThreads) {
    int64_t sv;
    if (i < n_sel) {
      const int j = a.idx[row * a.K + i];
      sv = -1;
      if (j >= 0 && j < nv) sv = entry_slot(a.page_table, a.max_pages, a.n_pages, b, j, status);
      else raise_status(status, CSA2_STATUS_BAD_INDEX);
    } else {
      sv = -2 - (int64_t)(w_lo + (i - n_sel) - pos0);
    }
    slots[i] = sv;
  }
  for (int i = tid; i < kHG * (D / 8); i += kAttnThreads) {
    const int h = i / (D / 8), c8 = i % (D / 8);
    const int head = hg * kHG + h;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (head < a.Hq) {
      const uint4 qb = *reinterpret_cast<const uint4*>(a.Q + (row * a.Hq + head) * D + c8 * 8);
      const uint32_t qw[4] = {qb.x, qb.y, qb.z, qb.w};
      uint32_t ov[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ov[j] = f32_to_f16_bits(bf16_bits_to_f32(qw[j] & 0xFFFFu)) |
                (f32_to_f16_bits(bf16_bits_to_f32(qw[j] >> 16)) << 16);
      v = make_uint4(ov[0], ov[1], ov[2], ov[3]);
    }
    *reinterpret_cast<uint4*>(&sm.q[h * QS + c8 * 8]) = v;
  }
  if (tid < kHG) {
    sm.m[tid] = -INFINITY;
    sm.l[tid] = 0.f;
  }
  __syncthreads();

  // item u of this thread: key (tid / 32) + 8u of the tile, group tid % 32
  const int grp = tid & 31;
  uint4 raw[kItems];
  float rsc[kItems];
  auto prefetch = [&](int ti) {
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int kr = (tid >> 5) + 8 * u;
      const int i = ti * kTK + kr;
      const int64_t src = i < n_keys ? slots[i] : -1;
      if (src >= 0) {
        const uint2 c = *reinterpret_cast<const uint2*>(a.kv_codes + src * (D / 2) + grp * 8);
        raw[u] = make_uint4(c.x, c.y, a.kv_scales[src * (D / 16) + grp], 0);
      } else if (src <= -2) {
        const int64_t wr = (int64_t)b * a.swa_cap + (-2 - src);
        raw[u] = *reinterpret_cast<const uint4*>(a.swa_codes + wr * D + grp * 16);
        rsc[u] = a.swa_scales[wr];
      }
    }
  };

  float o[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  const float sl2 = a.scale * 1.4426950408889634f;
  if (n_tiles > 0) prefetch(0);

  for (int ti = 0; ti < n_tiles; ++ti) {
    // ---- dequantise the prefetched tile
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int kr = (tid >> 5) + 8 * u;
      const int i = ti * kTK + kr;
      const int64_t src = i < n_keys ? slots[i] : -1;
      uint32_t w[8];
      if (src >= 0) {
        const uint32_t s2 = f32_to_f16_bits(e4m3_to_f32(raw[u].z)) * 0x10001u;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t word = q < 4 ? raw[u].x : raw[u].y;
          w[q] = hmul2_u32(e2m1x2_to_f16x2((word >> ((q & 3) * 8)) & 0xFFu), s2);
        }
      } else if (src <= -2) {
        const uint32_t cw[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t word = cw[q >> 1];
          const int sh = (q & 1) * 16;
          const float lo = bf16_bits_to_f32(f32_to_bf16_bits(e4m3_to_f32((word >> sh) & 0xFFu) * rsc[u]));
          const float hi = bf16_bits_to_f32(f32_to_bf16_bits(e4m3_to_f32((word >> (sh + 8)) & 0xFFu) * rsc[u]));
          w[q] = f32_to_f16_bits(lo) | (f32_to_f16_bits(hi) << 16);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) w[q] = 0;
      }
      uint4* d4 = reinterpret_cast<uint4*>(&sm.k[kr * QS + grp * 16]);
      d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
      d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    __syncthreads();
    if (ti + 1 < n_tiles) prefetch(ti + 1);   // in flight during the phases below
    // ---- S = Q K^T : warp owns keys 8*warp .. +7 (four accumulators)
    {
      float sa[4][4] = {};
      const uint32_t qa = smem_u32(&sm.q[(lane & 15) * QS + (lane >> 4) * 8]);
      const uint32_t kb = smem_u32(&sm.k[(warp * 8 + (lane & 7)) * QS + (lane >> 3) * 8]);
#pragma unroll
      for (int ks = 0; ks < D / 32; ks += 2) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          uint32_t a0, a1, a2, a3, a4, a5, a6, a7, b0, b1, b2, b3;
          ldsm_x4(qa + (ks + u) * 64, a0, a1, a2, a3);
          ldsm_x4(qa + (ks + u) * 64 + 32, a4, a5, a6, a7);
          ldsm_x4(kb + (ks + u) * 64, b0, b1, b2, b3);
          mma_f16(sa[2 * u], a0, a1, a2, a3, b0, b1);
          mma_f16(sa[2 * u + 1], a4, a5, a6, a7, b2, b3);
        }
      }
      const int key0 = warp * 8 + 2 * t4;
      const int i0 = ti * kTK + key0;
      const bool v0 = i0 < n_keys && slots[i0] != -1, v1 = i0 + 1 < n_keys && slots[i0 + 1] != -1;
      float s0[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) s0[r] = (sa[0][r] + sa[1][r]) + (sa[2][r] + sa[3][r]);
      sm.s[g * kTK + key0] = v0 ? s0[0] * sl2 : -INFINITY;
      sm.s[g * kTK + key0 + 1] = v1 ? s0[1] * sl2 : -INFINITY;
      sm.s[(g + 8) * kTK + key0] = v0 ? s0[2] * sl2 : -INFINITY;
      sm.s[(g + 8) * kTK + key0 + 1] = v1 ? s0[3] * sl2 : -INFINITY;
    }
    __syncthreads();
    // ---- online softmax: 16 threads per head, 4 keys each
    {
      const int h = tid >> 4, part = tid & 15;
      const float4 sv = *reinterpret_cast<const float4*>(&sm.s[h * kTK + part * 4]);
      float mx = fmaxf(fmaxf(sv.x, sv.y), fmaxf(sv.z, sv.w));
#pragma unroll
      for (int o2 = 1; o2 < 16; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
      const float m_old = sm.m[h];
      const float m_new = fmaxf(m_old, mx);
      const bool none = m_new == -INFINITY;
      const __half p0 = __float2half_rn(none ? 0.f : exp2f(sv.x - m_new));
      const __half p1 = __float2half_rn(none ? 0.f : exp2f(sv.y - m_new));
      const __half p2 = __float2half_rn(none ? 0.f : exp2f(sv.z - m_new));
      const __half p3 = __float2half_rn(none ? 0.f : exp2f(sv.w - m_new));
      float sum = __half2float(p0) + __half2float(p1) + __half2float(p2) + __half2float(p3);
      uint2 pw;
      pw.x = (uint32_t)__half_as_ushort(p0) | ((uint32_t)__half_as_ushort(p1) << 16);
      pw.y = (uint32_t)__half_as_ushort(p2) | ((uint32_t)__half_as_ushort(p3) << 16);
      *reinterpret_cast<uint2*>(&sm.p[h * PS + part * 4]) = pw;
#pragma unroll
      for (int o2 = 1; o2 < 16; o2 <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o2);
      __syncwarp();
      if (part == 0) {
        const float al = none ? 1.f : exp2f(m_old - m_new);
        sm.alpha[h] = al;
        sm.l[h] = sm.l[h] * al + sum;
        sm.m[h] = m_new;
      }
    }
    __syncthreads();
    // ---- O = O * alpha + P V : warp owns channels warp*DW .. +DW
    {
      const float al0 = sm.alpha[g], al1 = sm.alpha[g + 8];
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        o[i][0] *= al0; o[i][1] *= al0; o[i][2] *= al1; o[i][3] *= al1;
      }
      const uint32_t pa = smem_u32(&sm.p[(lane & 15) * PS + (lane >> 4) * 8]);
      const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
      for (int kk = 0; kk < kTK / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(pa + kk * 32, a0, a1, a2, a3);
        const uint32_t vb = smem_u32(&sm.k[(kk * 16 + (mi & 1) * 8 + r8) * QS + warp * DW + (mi >> 1) * 8]);
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + np * 32, b0, b1, b2, b3);
          mma_f16(o[2 * np], a0, a1, a2, a3, b0, b1);
          mma_f16(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();
  }
  // ---- normalise and store
  const float l0 = sm.l[g], l1 = sm.l[g + 8];
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const int head0 = hg * kHG + g, head1 = head0 + 8;
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const int ch = warp * DW + i * 8 + 2 * t4;
    if (head0 < a.Hq)
      *reinterpret_cast<float2*>(a.O + (row * a.Hq + head0) * D + ch) = make_float2(o[i][0] * inv0, o[i][1] * inv0);
    if (head1 < a.Hq)
      *reinterpret_cast<float2*>(a.O + (row * a.Hq + head1) * D + ch) = make_float2(o[i][2] * inv1, o[i][3] * inv1);
  }
  if (a.lse && tid < kHG && hg * kHG + tid < a.Hq) {
    const float l = sm.l[tid];
    a.lse[row * a.Hq + hg * kHG + tid] = l > 0.f ? (sm.m[tid] + log2f(l)) * 0.6931471805599453f : -INFINITY;
  }
}

// ---- pipelined variant (d = 512) -------------------------------------------------------
// A ninth warp produces: it resolves the key sources of tile t+1 (indices ->
// page table -> pool slot, or a window row) and bulk-copies their packed
// bytes (256 B of E2M1 codes + 32 B of E4M3 scales per entry, or 512 B of FP8
// codes per window row) into a double-buffered staging area, completing on an
// mbarrier with the byte count.  The eight consumer warps dequantise tile t
// from staging into the fp16 tile, release the stage, and run S, softmax and
// PV as above, synchronising among themselves with a named barrier.
constexpr int kPipeConsumers = 8;
constexpr int kPipeThreads = (kPipeConsumers + 1) * 32;
constexpr int kStageCodes = 512;  // bytes per key of staged codes (window rows need d bytes)
constexpr int kStages = 3;        // staging depth (tiles in flight ahead of the consumers)
constexpr int kMaxKeys = 2048 + 1024;  // K + W upper bound: key sources resolved up front

struct PipeSmem {
  static constexpr int QS = 512 + 8, PS = kTK + 8;
  uint16_t q[kHG * QS];
  uint16_t k[kTK * QS];
  float s[kHG * kTK];
  uint16_t p[kHG * PS];
  uint8_t codes[kStages][kTK][kStageCodes];
  uint8_t scales[kStages][kTK][32];
  float wscale[kStages][kTK];
  int64_t key_src[kStages][kTK];
  uint64_t full[kStages], empty[kStages];
  float m[kHG], l[kHG], alpha[kHG];
  int abort;
};

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kPipeConsumers * 32) : "memory");
}
// Barrier among the consumer warps that also ANDs a predicate: every consumer
// gets the same answer, so they leave a loop together.
__device__ __forceinline__ bool consumer_vote_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kPipeConsumers * 32)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort) return false;
  }
  *abort = 1;
  return false;
}

__global__ void __launch_bounds__(kPipeThreads)
k_sparse_attn_pipe(AttnArgs a, uint32_t* status) {
  constexpr int D = 512;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  PipeSmem& sm = *reinterpret_cast<PipeSmem*>(smem_raw);
  constexpr int QS = PipeSmem::QS, PS = PipeSmem::PS;
  constexpr int DW = D / kPipeConsumers, NT = DW / 8;
  const int64_t row = blockIdx.y;
  const int hg = blockIdx.x;
  const int b = (int)(row / a.Tq);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int t = a.q_pos[row];
  const int nv = n_visible(a.n_entries[b], t);
  int n_sel = a.cnt[row];
  if (n_sel < 0 || n_sel > a.K) {
    if (tid == 0) raise_status(status, CSA2_STATUS_BAD_COUNT);
    n_sel = n_sel < 0 ? 0 : a.K;
  }
  const int pos0 = a.swa_cap > 0 ? a.swa_pos0[b] : 0;
  const int w_lo = max(max(0, t - a.W + 1), pos0);
  const int w_hi = min(t, pos0 + a.swa_cap - 1);
  const int n_win = max(0, w_hi - w_lo + 1);
  const int n_keys = n_sel + n_win;
  const int n_tiles = (n_keys + kTK - 1) / kTK;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(&sm.full[i], 1);
      tc::mbar_init(&sm.empty[i], 1);
    }
    sm.abort = 0;
    tc::mbar_fence_init();
  }
  if (tid < kHG) {
    sm.m[tid] = -INFINITY;
    sm.l[tid] = 0.f;
  }
  // resolve every key's source once, with all threads: index -> page table ->
  // pool slot for selected entries, window row for the rest (-1 = no key)
  int64_t* slots = reinterpret_cast<int64_t*>(smem_raw + sizeof(PipeSmem));
  for (int i = tid; i < n_keys; i += kPipeThreads) {
    int64_t sv = -1;
    if (i < n_sel) {
      const int j = a.idx[row * a.K + i];
      if (j >= 0 && j < nv) sv = entry_slot(a.page_table, a.max_pages, a.n_pages, b, j, status);
      else raise_status(status, CSA2_STATUS_BAD_INDEX);
    } else {
      sv = -2 - (int64_t)(w_lo + (i - n_sel) - pos0);
    }
    slots[i] = sv;
  }
  __syncthreads();
  volatile int* abort = &sm.abort;

  if (warp == kPipeConsumers) {
    // ---------------- producer
    int issued = 0;
    for (int ti = 0; ti < n_tiles; ++ti) {
      const int st = ti % kStages;
      // lane 0 waits for the stage; the warp follows its answer (warp-uniform exit)
      bool okw = true;
      if (ti >= kStages && lane == 0) okw = pipe_wait(&sm.empty[st], ((ti / kStages) - 1) & 1, abort);
      if (!__shfl_sync(0xffffffffu, okw, 0)) break;
      int64_t src[2];
      uint32_t bytes = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kr = lane * 2 + h;
        const int i = ti * kTK + kr;
        const int64_t sv = i < n_keys ? slots[i] : -1;
        if (sv >= 0) {
          bytes += 256 + 32;
        } else if (sv <= -2) {
          sm.wscale[st][kr] = a.swa_scales[(int64_t)b * a.swa_cap + (-2 - sv)];
          bytes += D;
        }
        src[h] = sv;
        sm.key_src[st][kr] = sv;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
      if (lane == 0) tc::mbar_arrive_expect_tx(&sm.full[st], bytes);
      __syncwarp();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kr = lane * 2 + h;
        if (src[h] >= 0) {
          tc::bulk_g2s(sm.codes[st][kr], a.kv_codes + src[h] * (D / 2), 256, &sm.full[st]);
          tc::bulk_g2s(sm.scales[st][kr], a.kv_scales + src[h] * (D / 16), 32, &sm.full[st]);
        } else if (src[h] <= -2) {
          tc::bulk_g2s(sm.codes[st][kr], a.swa_codes + ((int64_t)b * a.swa_cap + (-2 - src[h])) * D, D,
                       &sm.full[st]);
        }
      }
      issued = ti + 1;
    }
    // drain the copies still in flight before the CTA can exit
    if (lane == 0)
      for (int ti = max(0, issued - kStages); ti < issued; ++ti)
        for (uint32_t k2 = 0; k2 < (1u << 22); ++k2)
          if (tc::mbar_try_wait(&sm.full[ti % kStages], (ti / kStages) & 1)) break;
  } else {
    // ---------------- consumers
    const int g = lane >> 2, t4 = lane & 3;
    for (int i = tid; i < kHG * (D / 8); i += kPipeConsumers * 32) {
      const int h = i / (D / 8), c8 = i % (D / 8);
      const int head = hg * kHG + h;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (head < a.Hq) {
        const uint4 qb = *reinterpret_cast<const uint4*>(a.Q + (row * a.Hq + head) * D + c8 * 8);
        const uint32_t qw[4] = {qb.x, qb.y, qb.z, qb.w};
        uint32_t ov[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          ov[j] = f32_to_f16_bits(bf16_bits_to_f32(qw[j] & 0xFFFFu)) |
                  (f32_to_f16_bits(bf16_bits_to_f32(qw[j] >> 16)) << 16);
        v = make_uint4(ov[0], ov[1], ov[2], ov[3]);
      }
      *reinterpret_cast<uint4*>(&sm.q[h * QS + c8 * 8]) = v;
    }
    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    const float sl2 = a.scale * 1.4426950408889634f;

    for (int ti = 0; ti < n_tiles; ++ti) {
      const int st = ti % kStages;
      if (!consumer_vote_and(pipe_wait(&sm.full[st], (ti / kStages) & 1, abort))) break;
      // ---- dequantise the staged tile: item = (key, 16-channel group)
      for (int it = tid; it < kTK * (D / 16); it += kPipeConsumers * 32) {
        const int kr = it & (kTK - 1), grp = it / kTK;
        const int64_t src = sm.key_src[st][kr];
        uint32_t w[8];
        if (src >= 0) {
          const uint2 c = *reinterpret_cast<const uint2*>(&sm.codes[st][kr][grp * 8]);
          const uint32_t s2 = f32_to_f16_bits(e4m3_to_f32(sm.scales[st][kr][grp])) * 0x10001u;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t word = i < 4 ? c.x : c.y;
            w[i] = hmul2_u32(e2m1x2_to_f16x2((word >> ((i & 3) * 8)) & 0xFFu), s2);
          }
        } else if (src <= -2) {
          const uint4 c = *reinterpret_cast<const uint4*>(&sm.codes[st][kr][grp * 16]);
          const float sc = sm.wscale[st][kr];
          const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t word = cw[i >> 1];
            const int sh = (i & 1) * 16;
            const float lo = bf16_bits_to_f32(f32_to_bf16_bits(e4m3_to_f32((word >> sh) & 0xFFu) * sc));
            const float hi = bf16_bits_to_f32(f32_to_bf16_bits(e4m3_to_f32((word >> (sh + 8)) & 0xFFu) * sc));
            w[i] = f32_to_f16_bits(lo) | (f32_to_f16_bits(hi) << 16);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = 0;
        }
        uint4* d4 = reinterpret_cast<uint4*>(&sm.k[kr * QS + grp * 16]);
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
      consumer_sync();
      // ---- S = Q K^T : warp owns keys 8*warp .. +7; four independent
      // accumulators keep the tensor-core dependency chain short
      {
        float sa[4][4] = {};
        const uint32_t qa = smem_u32(&sm.q[(lane & 15) * QS + (lane >> 4) * 8]);
        const uint32_t kb = smem_u32(&sm.k[(warp * 8 + (lane & 7)) * QS + (lane >> 3) * 8]);
#pragma unroll
        for (int ks = 0; ks < D / 32; ks += 2) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            uint32_t a0, a1, a2, a3, a4, a5, a6, a7, b0, b1, b2, b3;
            ldsm_x4(qa + (ks + u) * 64, a0, a1, a2, a3);
            ldsm_x4(qa + (ks + u) * 64 + 32, a4, a5, a6, a7);
            ldsm_x4(kb + (ks + u) * 64, b0, b1, b2, b3);
            mma_f16(sa[2 * u], a0, a1, a2, a3, b0, b1);
            mma_f16(sa[2 * u + 1], a4, a5, a6, a7, b2, b3);
          }
        }
        float s0[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) s0[r] = (sa[0][r] + sa[1][r]) + (sa[2][r] + sa[3][r]);
        const int key0 = warp * 8 + 2 * t4;
        const bool v0 = sm.key_src[st][key0] != -1, v1 = sm.key_src[st][key0 + 1] != -1;
        sm.s[g * kTK + key0] = v0 ? s0[0] * sl2 : -INFINITY;
        sm.s[g * kTK + key0 + 1] = v1 ? s0[1] * sl2 : -INFINITY;
        sm.s[(g + 8) * kTK + key0] = v0 ? s0[2] * sl2 : -INFINITY;
        sm.s[(g + 8) * kTK + key0 + 1] = v1 ? s0[3] * sl2 : -INFINITY;
      }
      consumer_sync();
      // staging and key sources of this tile are no longer read: hand the stage back
      if (tid == 0) tc::mbar_arrive(&sm.empty[st]);
      // ---- online softmax: 16 threads per head, 4 keys each
      {
        const int h = tid >> 4, part = tid & 15;
        const float4 sv = *reinterpret_cast<const float4*>(&sm.s[h * kTK + part * 4]);
        float mx = fmaxf(fmaxf(sv.x, sv.y), fmaxf(sv.z, sv.w));
#pragma unroll
        for (int o2 = 1; o2 < 16; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        const float m_old = sm.m[h];
        const float m_new = fmaxf(m_old, mx);
        const bool none = m_new == -INFINITY;
        const __half p0 = __float2half_rn(none ? 0.f : exp2f(sv.x - m_new));
        const __half p1 = __float2half_rn(none ? 0.f : exp2f(sv.y - m_new));
        const __half p2 = __float2half_rn(none ? 0.f : exp2f(sv.z - m_new));
        const __half p3 = __float2half_rn(none ? 0.f : exp2f(sv.w - m_new));
        float sum = __half2float(p0) + __half2float(p1) + __half2float(p2) + __half2float(p3);
        uint2 pw;
        pw.x = (uint32_t)__half_as_ushort(p0) | ((uint32_t)__half_as_ushort(p1) << 16);
        pw.y = (uint32_t)__half_as_ushort(p2) | ((uint32_t)__half_as_ushort(p3) << 16);
        *reinterpret_cast<uint2*>(&sm.p[h * PS + part * 4]) = pw;
#pragma unroll
        for (int o2 = 1; o2 < 16; o2 <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o2);
        __syncwarp();
        if (part == 0) {
          const float al = none ? 1.f : exp2f(m_old - m_new);
          sm.alpha[h] = al;
          sm.l[h] = sm.l[h] * al + sum;
          sm.m[h] = m_new;
        }
      }
      consumer_sync();
      // ---- O = O * alpha + P V : warp owns channels warp*DW .. +DW
      {
        const float al0 = sm.alpha[g], al1 = sm.alpha[g + 8];
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          o[i][0] *= al0; o[i][1] *= al0; o[i][2] *= al1; o[i][3] *= al1;
        }
        const uint32_t pa = smem_u32(&sm.p[(lane & 15) * PS + (lane >> 4) * 8]);
        const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
        for (int kk = 0; kk < kTK / 16; ++kk) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(pa + kk * 32, a0, a1, a2, a3);
          const uint32_t vb = smem_u32(&sm.k[(kk * 16 + (mi & 1) * 8 + r8) * QS + warp * DW + (mi >> 1) * 8]);
#pragma unroll
          for (int np = 0; np < NT / 2; ++np) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vb + np * 32, b0, b1, b2, b3);
            mma_f16(o[2 * np], a0, a1, a2, a3, b0, b1);
            mma_f16(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
          }
        }
      }
      consumer_sync();
    }
    // ---- normalise and store
    const float l0 = sm.l[g], l1 = sm.l[g + 8];
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const int head0 = hg * kHG + g, head1 = head0 + 8;
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int ch = warp * DW + i * 8 + 2 * t4;
      if (head0 < a.Hq)
        *reinterpret_cast<float2*>(a.O + (row * a.Hq + head0) * D + ch) = make_float2(o[i][0] * inv0, o[i][1] * inv0);
      if (head1 < a.Hq)
        *reinterpret_cast<float2*>(a.O + (row * a.Hq + head1) * D + ch) = make_float2(o[i][2] * inv1, o[i][3] * inv1);
    }
    if (a.lse && tid < kHG && hg * kHG + tid < a.Hq) {
      const float l = sm.l[tid];
      a.lse[row * a.Hq + hg * kHG + tid] = l > 0.f ? (sm.m[tid] + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
  }
  __syncthreads();
  if (tid == 0 && sm.abort) raise_status(status, CSA2_STATUS_TIMEOUT);
}

template <int D>
static cudaError_t launch_attn_d(const AttnArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(AttnSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(k_sparse_attn<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Hq + kHG - 1) / kHG, (unsigned)((int64_t)a.B * a.Tq));
  k_sparse_attn<D><<<grid, kAttnThreads, smem, s>>>(a, status_word());
  return counted(cudaGetLastError());
}

cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t s) {
  if ((int64_t)a.B * a.Tq == 0) return cudaSuccess;
  if (sparse_attn_tc_supported(a)) return launch_sparse_attn_tc(a, s);
  const int64_t ctas = (int64_t)((a.Hq + kHG - 1) / kHG) * a.B * a.Tq;
  if (a.d == 512 && a.K + a.W <= kMaxKeys && ctas <= 152) {
    // few CTAs (decode): the producer-warp pipeline hides more latency per CTA
    const size_t smem = sizeof(PipeSmem) + (size_t)(a.K + a.W) * sizeof(int64_t);
    cudaError_t e = cudaFuncSetAttribute(k_sparse_attn_pipe, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.Hq + kHG - 1) / kHG, (unsigned)((int64_t)a.B * a.Tq));
    k_sparse_attn_pipe<<<grid, kPipeThreads, smem, s>>>(a, status_word());
    return counted(cudaGetLastError());
  }
  if (a.d == 512 && a.K + a.W <= kMaxKeys) {
    const size_t smem = sizeof(AttnSmem<512>) + (size_t)(a.K + a.W) * sizeof(int64_t);
    cudaError_t e = cudaFuncSetAttribute(k_sparse_attn_rp, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.Hq + kHG - 1) / kHG, (unsigned)((int64_t)a.B * a.Tq));
    k_sparse_attn_rp<<<grid, kAttnThreads, smem, s>>>(a, status_word());
    return counted(cudaGetLastError());
  }
  return launch_attn_d<64>(a, s);
}

}  // namespace csa2
