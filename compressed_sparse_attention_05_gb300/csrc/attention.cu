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
// This kernel serves d = 64 (the small latent of the parity workload); d = 512
// runs on the tensor-memory kernel of attention_tc.cu.
//
// Operands are fp16.  MXFP4 entries are converted by cvt.rn.f16x2.e2m1x2 and
// scaled in f16x2: e2m1 * e4m3 has at most 6 significant bits and lies in
// [2^-10, 2688], so the values are exactly the bf16 dequantised latent.  Q and
// the window rows are bf16 values (the operands the method specifies) carried
// in fp16 after a power-of-two scaling that changes no significand bit: each
// head of Q by 2^-e_h (largest magnitude in [2^14, 2^15), logits multiplied
// back), a window row whose scale lies outside [2^-8, 2^7] by 2^-f (logits
// multiplied back by 2^f, softmax weight carried as 2^f p, normaliser adding
// p).  P is rounded to fp16 (11 significant bits) for the PV product; the
// normaliser sums the unrounded fp32 weights (relative difference <= 2^-11).
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
  float sl2h[kHG];                     // logit multiplier per head: scale * log2(e) * 2^e_h
  int qexp[kHG];                       // largest bf16 exponent field per head, then e_h
  int kexp[kTK];                       // exponent f of a window row's scale (0: none)
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
    const float sw = a.swa_scales[wr];
    const float sc = sw * pow2i(-window_exp(sw));
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

  // Q rows of this head group: bf16 bits first, with each head's largest exponent field
  if (tid < kHG) {
    sm.m[tid] = -INFINITY;
    sm.l[tid] = 0.f;
    sm.qexp[tid] = 0;
  }
  __syncthreads();
  for (int i = tid; i < kHG * (D / 8); i += kAttnThreads) {
    const int h = i / (D / 8), c8 = i % (D / 8);
    const int head = hg * kHG + h;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (head < a.Hq) v = *reinterpret_cast<const uint4*>(a.Q + (row * a.Hq + head) * D + c8 * 8);
    const uint32_t qw[4] = {v.x, v.y, v.z, v.w};
    int e = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) e = max(e, (int)max((qw[j] >> 7) & 0xFFu, (qw[j] >> 23) & 0xFFu));
    if (e) atomicMax(&sm.qexp[h], e);
    *reinterpret_cast<uint4*>(&sm.q[h * QS + c8 * 8]) = v;
  }
  __syncthreads();
  if (tid < kHG) {
    const int eh = q_head_exp(sm.qexp[tid]);
    sm.qexp[tid] = eh;
    sm.sl2h[tid] = a.scale * 1.4426950408889634f * pow2i(eh);
  }
  __syncthreads();
  // -> fp16, head h scaled by 2^-e_h (exact)
  for (int i = tid; i < kHG * (D / 8); i += kAttnThreads) {
    const int h = i / (D / 8), c8 = i % (D / 8);
    const float qs = pow2i(-sm.qexp[h]);
    uint4* p = reinterpret_cast<uint4*>(&sm.q[h * QS + c8 * 8]);
    const uint4 v = *p;
    const uint32_t qw[4] = {v.x, v.y, v.z, v.w};
    uint32_t ov[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      ov[j] = f32_to_f16_bits(bf16_bits_to_f32(qw[j] & 0xFFFFu) * qs) |
              (f32_to_f16_bits(bf16_bits_to_f32(qw[j] >> 16) * qs) << 16);
    *p = make_uint4(ov[0], ov[1], ov[2], ov[3]);
  }

  float o[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

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
      sm.kexp[tid] = src <= -2 ? window_exp(a.swa_scales[(int64_t)b * a.swa_cap + (-2 - src)]) : 0;
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
      // logits in log2 units, as the PV product carries them: y = x + f for a rescaled
      // window row (x times 2^f), y = x otherwise
      const int key0 = warp * 8 + 2 * t4;
      const bool v0 = sm.key_src[key0] != -1, v1 = sm.key_src[key0 + 1] != -1;
      const int f0 = sm.kexp[key0], f1 = sm.kexp[key0 + 1];
      const float m0 = sm.sl2h[g], m1 = sm.sl2h[g + 8];
      auto y = [](float x, int f) { return f ? x * pow2i(f) + (float)f : x; };
      sm.s[g * kTK + key0] = v0 ? y(s0[0] * m0, f0) : -INFINITY;
      sm.s[g * kTK + key0 + 1] = v1 ? y(s0[1] * m0, f1) : -INFINITY;
      sm.s[(g + 8) * kTK + key0] = v0 ? y(s0[2] * m1, f0) : -INFINITY;
      sm.s[(g + 8) * kTK + key0 + 1] = v1 ? y(s0[3] * m1, f1) : -INFINITY;
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
      const float e0 = none ? 0.f : exp2f(sv.x - m_new), e1 = none ? 0.f : exp2f(sv.y - m_new);
      const float e2 = none ? 0.f : exp2f(sv.z - m_new), e3 = none ? 0.f : exp2f(sv.w - m_new);
      const __half p0 = __float2half_rn(e0), p1 = __float2half_rn(e1);
      const __half p2 = __float2half_rn(e2), p3 = __float2half_rn(e3);
      // the normaliser sums the fp32 weights (2^f p of a rescaled window row counts as
      // p): a weight carried as 2^f p with f < 0 may underflow fp16 in the PV product,
      // where its row's values are negligible, but must still count in the normaliser
      const int4 fq = *reinterpret_cast<const int4*>(&sm.kexp[part * 4]);
      float sum = e0 * pow2i(-fq.x) + e1 * pow2i(-fq.y) + e2 * pow2i(-fq.z) + e3 * pow2i(-fq.w);
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
  if (a.d != 64) return cudaErrorInvalidValue;   // d = 512 always takes the tensor-memory kernel
  return launch_attn_d<64>(a, s);
}

}  // namespace csa2
