// Packing kernels: MXFP4 main KV (with RMSNorm + RoPE in front), FP8 window.
//
// Formats follow "DeepSeek-V4.1 架构解析" §03: E2M1 values with one E4M3 scale
// per 16 channels and no global scale, quantised after RoPE; the sliding
// window stays FP8.  Rounding rules: readings R2-R5 of include/csa2.h.
// Bandwidth-bound: every kernel reads and writes each byte once with 16-byte
// (or 8-byte) accesses.  Built without fast-math: the divisions that decide a
// code are IEEE fp32 divisions, as the bit-exact contract requires.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace csa2 {

// One thread per 16-channel group of a contiguous fp32 array.
__global__ void k_pack_mxfp4(const float* __restrict__ x, int64_t n_groups,
                             uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= n_groups) return;
  const float4* src = reinterpret_cast<const float4*>(x + g * 16);
  float v[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 f = src[i];
    v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
  }
  Mxfp4Group p = pack_group16(v);
  reinterpret_cast<uint2*>(codes)[g] = p.codes;
  scales[g] = (uint8_t)p.scale;
}

__global__ void k_unpack_mxfp4(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                               int64_t n_groups, uint16_t* __restrict__ out) {
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= n_groups) return;
  const uint2 c = reinterpret_cast<const uint2*>(codes)[g];
  const float s = e4m3_to_f32(scales[g]);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t word = i < 4 ? c.x : c.y;
    const int sh = (i & 3) * 8;
    const uint32_t lo = (word >> sh) & 0xFu, hi = (word >> (sh + 4)) & 0xFu;
    // e2m1 * e4m3 has at most 6 significant bits: the product is exact and
    // its bf16 pattern is the top half of the fp32 pattern
    const float a = bf16_bits_to_f32(e2m1_to_bf16_bits(lo)) * s;
    const float b = bf16_bits_to_f32(e2m1_to_bf16_bits(hi)) * s;
    w[i] = (__float_as_uint(a) >> 16) | (__float_as_uint(b) & 0xFFFF0000u);
  }
  uint4* dst = reinterpret_cast<uint4*>(out + g * 16);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// One warp per row of d channels: scale = amax / 448, codes = E4M3(x / scale).
__device__ __forceinline__ void fp8_row(const float* __restrict__ x, int d, uint8_t* __restrict__ codes,
                                        float* scale_out, int lane) {
  float amax = 0.f;
  for (int c = lane * 4; c < d; c += 128) {
    float4 f = *reinterpret_cast<const float4*>(x + c);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
  }
  amax = warp_max(amax);
  const float s = amax / 448.0f;
  for (int c = lane * 4; c < d; c += 128) {
    float4 f = *reinterpret_cast<const float4*>(x + c);
    uint32_t w = 0;
    if (s != 0.f) {
      w = f32_to_e4m3(f.x / s) | (f32_to_e4m3(f.y / s) << 8) | (f32_to_e4m3(f.z / s) << 16) |
          (f32_to_e4m3(f.w / s) << 24);
    }
    *reinterpret_cast<uint32_t*>(codes + c) = w;
  }
  if (lane == 0) *scale_out = s;
}

__global__ void k_pack_fp8(const float* __restrict__ x, int64_t n_rows, int d,
                           uint8_t* __restrict__ codes, float* __restrict__ scales) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (row >= n_rows) return;
  fp8_row(x + row * d, d, codes + row * d, scales + row, threadIdx.x & 31);
}

__global__ void k_pack_fp8_window(const float* __restrict__ x, int B, int Tq, int d,
                                  const int32_t* __restrict__ q_pos, const int32_t* __restrict__ pos0,
                                  int swa_cap, uint8_t* __restrict__ codes,
                                  float* __restrict__ scales, uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (row >= (int64_t)B * Tq) return;
  const int b = (int)(row / Tq);
  const int64_t wr = (int64_t)q_pos[row] - pos0[b];
  if (wr < 0 || wr >= swa_cap) {
    if ((threadIdx.x & 31) == 0) raise_status(status, CSA2_STATUS_BAD_COUNT);
    return;
  }
  const int64_t dst = (int64_t)b * swa_cap + wr;
  fp8_row(x + row * d, d, codes + dst * d, scales + dst, threadIdx.x & 31);
}

// RMSNorm + RoPE of one latent row held by a warp.
//
// RoPE angles: the position p reaches ~4M (entry positions 4e + 3 of a 1M-entry
// cache, or raw token positions), so the angle p * theta_i can be ~4e6 rad.
// The rotation of frequency i is kept as turns per position, g_i =
// frac(theta_i / 2 pi) in 0.64 fixed point (host, fp64); p * g_i mod 2^64 in
// integer arithmetic is then the angle's fraction of a turn (error <= p *
// 2^-53 turns, like the fp64 product p * theta_i), and fp64 sincospi of that
// fraction and an fp64 rotation give the rotated channels rounded once to
// fp32, as an fp64 RoPE does: an fp32 rotation moves values across the FP4 /
// FP8 rounding boundaries now and then.  fp64 is slow on this GPU, so the
// pairs are spread over the lanes: one angle and one pair per lane.
constexpr int kNrpWarps = 4;
struct RopeTurns {
  uint64_t g[256];   // r/2 <= 256 frequencies
};

// Lane l holds channels 16l .. 16l+15 of the row in v (has = 16l < d; d <= 512).
// On return v holds the normalised, rotated channels and buf (the warp's row
// buffer, d floats) the whole row.
__device__ __forceinline__ void norm_rope_row(float (&v)[16], bool has, int d, int r,
                                              const float* __restrict__ gamma, float eps, uint64_t pos,
                                              const RopeTurns& rope, float* buf, int lane) {
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < 16; ++c) ss += v[c] * v[c];
  ss = warp_sum(ss);
  const float inv = 1.0f / sqrtf(ss / (float)d + eps);
  if (has) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      v[c] = v[c] * inv * gamma[lane * 16 + c];
      buf[lane * 16 + c] = v[c];
    }
  }
  __syncwarp();
  // rotate-half RoPE on channels [d - r, d): lane l rotates pair
  // (d - r + l, d - r/2 + l) of each round of 32 pairs in the row buffer, then
  // the channels' owners read them back
  const int half = r / 2;
  for (int k0 = 0; k0 < half; k0 += 32) {
    const int pi = k0 + lane;
    if (pi < half) {
      double sn, cs;
      const uint64_t turns = pos * rope.g[pi];                    // fraction of a turn, mod 2^64
      sincospi((double)(int64_t)turns * 0x1p-63, &sn, &cs);       // angle / pi in [-1, 1)
      const double x1 = (double)buf[d - r + pi], x2 = (double)buf[d - half + pi];
      buf[d - r + pi] = (float)(x1 * cs - x2 * sn);
      buf[d - half + pi] = (float)(x1 * sn + x2 * cs);
    }
  }
  __syncwarp();
  if (has && r > 0) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int ch = lane * 16 + c;
      if (ch >= d - r) v[c] = buf[ch];
    }
  }
}

// Lane l's 16 channels of latent row m: the split-K partials summed in a fixed
// order (deterministic).
__device__ __forceinline__ void load_latent(const LatentSource& src, int64_t m, bool has, int lane,
                                            float (&v)[16]) {
#pragma unroll
  for (int c = 0; c < 16; ++c) v[c] = 0.f;
  if (!has) return;
  for (int sp = 0; sp < src.n_split; ++sp) {
    const float4* p = reinterpret_cast<const float4*>(src.base + sp * src.split_stride + m * src.row_stride +
                                                      lane * 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4 f = p[q];
      v[4 * q] += f.x; v[4 * q + 1] += f.y; v[4 * q + 2] += f.z; v[4 * q + 3] += f.w;
    }
  }
}

// RMSNorm + RoPE (at the entry position 4e + 3) + MXFP4 pack + paged store of
// entry m (sequence m / n_max, its entry m % n_max), one warp.  Lane l owns
// channels 16l .. 16l+15 (one MXFP4 group).
__device__ __forceinline__ void norm_rope_pack_entry(const LatentSource& src, int64_t m, int n_max, int d, int r,
                                                     const float* __restrict__ gamma, float eps,
                                                     const int32_t* __restrict__ first_entry,
                                                     const int32_t* __restrict__ n_rows,
                                                     const int32_t* __restrict__ page_table, int max_pages,
                                                     int64_t n_pages, uint8_t* __restrict__ kv_codes,
                                                     uint8_t* __restrict__ kv_scales, const float* idx_src,
                                                     int64_t idx_row_stride, int Di, int idx_dtype, void* idx_k,
                                                     int kv_fp8, const RopeTurns& rope, float* row, int lane,
                                                     uint32_t* status) {
  const int b = (int)(m / n_max), i = (int)(m % n_max);
  if (n_rows && i >= n_rows[b]) return;
  const int e = first_entry[b] + i;
  const int64_t slot = entry_slot(page_table, max_pages, n_pages, b, e, status);
  if (slot < 0) return;

  const bool has = lane < d / 16;
  float v[16];
  load_latent(src, m, has, lane, v);
  norm_rope_row(v, has, d, r, gamma, eps, 4ull * (uint64_t)e + 3ull, rope, row, lane);
  if (kv_fp8) {   // the FP8 main-KV format: R5's row rule, one fp32 scale per entry
    __syncwarp();
    fp8_row(row, d, kv_codes + slot * d, reinterpret_cast<float*>(kv_scales) + slot, lane);
  } else if (has) {
    Mxfp4Group g = pack_group16(v);
    reinterpret_cast<uint2*>(kv_codes + slot * (d / 2))[lane] = g.codes;
    kv_scales[slot * (d / 16) + lane] = (uint8_t)g.scale;
  }
  // indexer key of the entry (compression epilogue): sum the split partials
  if (idx_k) {
    for (int c = lane; c < Di; c += 32) {
      float acc = 0.f;
      for (int sp = 0; sp < src.n_split; ++sp)
        acc += idx_src[sp * src.split_stride + m * idx_row_stride + c];
      if (idx_dtype == CSA2_BF16)
        reinterpret_cast<uint16_t*>(idx_k)[slot * Di + c] = (uint16_t)f32_to_bf16_bits(acc);
      else
        reinterpret_cast<float*>(idx_k)[slot * Di + c] = acc;
    }
  }
}

__global__ void __launch_bounds__(kNrpWarps * 32)
k_norm_rope_pack(LatentSource src, int B, int n_max, int d, int r, const float* __restrict__ gamma,
                 float eps, const int32_t* __restrict__ first_entry,
                 const int32_t* __restrict__ n_rows, const int32_t* __restrict__ page_table,
                 int max_pages, int64_t n_pages, uint8_t* __restrict__ kv_codes,
                 uint8_t* __restrict__ kv_scales, const float* idx_src, int64_t idx_row_stride,
                 int Di, int idx_dtype, void* idx_k, int kv_fp8, const __grid_constant__ RopeTurns rope,
                 uint32_t* status) {
  __shared__ __align__(16) float row_buf[kNrpWarps][512];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * kNrpWarps + warp;
  if (m >= (int64_t)B * n_max) return;
  norm_rope_pack_entry(src, m, n_max, d, r, gamma, eps, first_entry, n_rows, page_table, max_pages, n_pages, kv_codes,
                       kv_scales, idx_src, idx_row_stride, Di, idx_dtype, idx_k, kv_fp8, rope, row_buf[warp], lane,
                       status);
}

// The same for several layers at once (grid.y = layer): every layer's latent
// and index-key columns lie at a fixed stride in one GEMM output, its gamma at
// a fixed stride, and its cache where its own pointers say.
__global__ void __launch_bounds__(kNrpWarps * 32)
k_norm_rope_pack_layers(LatentSource src, int B, int n_max, int d, int r, const float* __restrict__ gamma,
                        float eps, const int32_t* __restrict__ first_entry, int max_pages, const float* idx_src,
                        int64_t idx_row_stride, int Di, int idx_dtype, int kv_fp8,
                        const __grid_constant__ PackLayers layers, const __grid_constant__ RopeTurns rope,
                        uint32_t* status) {
  __shared__ __align__(16) float row_buf[kNrpWarps][512];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * kNrpWarps + warp;
  if (m >= (int64_t)B * n_max) return;
  const int l = (int)blockIdx.y;
  const PackLayer& c = layers.l[l];
  LatentSource ls = src;
  ls.base += l * layers.col_stride;
  norm_rope_pack_entry(ls, m, n_max, d, r, gamma + l * layers.gamma_stride, eps, first_entry, nullptr, c.page_table,
                       max_pages, c.n_pages, c.kv_codes, c.kv_scales, idx_src ? idx_src + l * layers.col_stride : nullptr,
                       idx_row_stride, Di, idx_dtype, c.idx_k, kv_fp8, rope, row_buf[warp], lane, status);
}

// Window rows of replayed tokens (SWA Bounded Replay, reading R13): one warp
// per token sums its projection's split partials, applies RMSNorm and RoPE at
// the token's own raw position and packs the row to FP8 (R5) into window row
// tok_pos0[b] + i - win_pos0[b]; a row outside the buffer is skipped and
// flagged.
__global__ void __launch_bounds__(kNrpWarps * 32)
k_norm_rope_fp8_window(LatentSource src, int B, int n_tok, int d, int r, const float* __restrict__ gamma,
                       float eps, const int32_t* __restrict__ tok_pos0, const int32_t* __restrict__ win_pos0,
                       int swa_cap, uint8_t* __restrict__ codes, float* __restrict__ scales,
                       const __grid_constant__ RopeTurns rope, uint32_t* status) {
  __shared__ __align__(16) float row_buf[kNrpWarps][512];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * kNrpWarps + warp;
  if (m >= (int64_t)B * n_tok) return;
  const int b = (int)(m / n_tok), i = (int)(m % n_tok);
  const int64_t p = (int64_t)tok_pos0[b] + i;
  const int64_t wr = p - win_pos0[b];
  if (p < 0 || wr < 0 || wr >= swa_cap) {
    if (lane == 0) raise_status(status, CSA2_STATUS_BAD_COUNT);
    return;
  }
  const bool has = lane < d / 16;
  float v[16];
  load_latent(src, m, has, lane, v);
  norm_rope_row(v, has, d, r, gamma, eps, (uint64_t)p, rope, row_buf[warp], lane);
  __syncwarp();
  const int64_t dst = (int64_t)b * swa_cap + wr;
  fp8_row(row_buf[warp], d, codes + dst * d, scales + dst, lane);
}

static inline unsigned grid_for(int64_t n, int per_block) {
  return (unsigned)((n + per_block - 1) / per_block);
}

cudaError_t launch_pack_mxfp4(const float* x, int64_t n_rows, int d, uint8_t* codes,
                              uint8_t* scales, cudaStream_t s) {
  const int64_t n = n_rows * (d / 16);
  if (n == 0) return cudaSuccess;
  k_pack_mxfp4<<<grid_for(n, 256), 256, 0, s>>>(x, n, codes, scales);
  return counted(cudaGetLastError());
}

cudaError_t launch_unpack_mxfp4(const uint8_t* codes, const uint8_t* scales, int64_t n_rows,
                                int d, uint16_t* out, cudaStream_t s) {
  const int64_t n = n_rows * (d / 16);
  if (n == 0) return cudaSuccess;
  k_unpack_mxfp4<<<grid_for(n, 256), 256, 0, s>>>(codes, scales, n, out);
  return counted(cudaGetLastError());
}

cudaError_t launch_pack_fp8(const float* x, int64_t n_rows, int d, uint8_t* codes,
                            float* scales, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  k_pack_fp8<<<grid_for(n_rows, 8), 256, 0, s>>>(x, n_rows, d, codes, scales);
  return counted(cudaGetLastError());
}

cudaError_t launch_pack_fp8_window(const float* x, int B, int Tq, int d, const int32_t* q_pos,
                                   const int32_t* pos0, int swa_cap, uint8_t* codes,
                                   float* scales, cudaStream_t s) {
  const int64_t rows = (int64_t)B * Tq;
  if (rows == 0) return cudaSuccess;
  return launch_step(k_pack_fp8_window, dim3(grid_for(rows, 8)), dim3(256), 0, s, x, B, Tq, d, q_pos, pos0, swa_cap,
                     codes, scales, status_word());
}

// theta_i = base^(-2i/r) radians per position, as 0.64 fixed-point turns (host, fp64).
static RopeTurns rope_turns(int r, float rope_base) {
  RopeTurns rope = {};
  for (int i = 0; i < r / 2; ++i) {
    const double f = std::pow((double)rope_base, -2.0 * i / (double)r) / (2.0 * 3.14159265358979323846);
    const double frac = std::ldexp(f - std::floor(f), 64);
    rope.g[i] = frac >= 18446744073709551616.0 ? 0ull : (uint64_t)frac;
  }
  return rope;
}

cudaError_t launch_norm_rope_pack(LatentSource src, int B, int n_max, int d, int r,
                                  const float* gamma, float eps, float rope_base,
                                  const int32_t* first_entry, const int32_t* n_rows,
                                  const int32_t* page_table, int max_pages, int64_t n_pages,
                                  uint8_t* kv_codes, uint8_t* kv_scales, const float* idx_src,
                                  int64_t idx_row_stride, int Di, int idx_dtype, void* idx_k,
                                  cudaStream_t s, int kv_fp8) {
  const int64_t rows = (int64_t)B * n_max;
  if (rows == 0) return cudaSuccess;
  if (r < 0 || r / 2 > 256 || (kv_fp8 && d != 512)) return cudaErrorInvalidValue;
  const RopeTurns rope = rope_turns(r, rope_base);
  return launch_step(k_norm_rope_pack, dim3(grid_for(rows, kNrpWarps)), dim3(kNrpWarps * 32), 0, s,
      src, B, n_max, d, r, gamma, eps, first_entry, n_rows, page_table, max_pages,
      n_pages, kv_codes, kv_scales, idx_src, idx_row_stride, Di, idx_dtype, idx_k, kv_fp8, rope, status_word());
}

cudaError_t launch_norm_rope_pack_layers(LatentSource src, int B, int n_max, int d, int r, const float* gamma,
                                         float eps, float rope_base, const int32_t* first_entry, int max_pages,
                                         const float* idx_src, int64_t idx_row_stride, int Di, int idx_dtype,
                                         int kv_fp8, const PackLayers& layers, int n_layers, cudaStream_t s) {
  const int64_t rows = (int64_t)B * n_max;
  if (rows == 0 || n_layers == 0) return cudaSuccess;
  if (r < 0 || r / 2 > 256 || (kv_fp8 && d != 512) || n_layers > kPackLayersMax) return cudaErrorInvalidValue;
  const RopeTurns rope = rope_turns(r, rope_base);
  return launch_step(k_norm_rope_pack_layers, dim3(grid_for(rows, kNrpWarps), (unsigned)n_layers),
                     dim3(kNrpWarps * 32), 0, s, src, B, n_max, d, r, gamma, eps, first_entry, max_pages, idx_src,
                     idx_row_stride, Di, idx_dtype, kv_fp8, layers, rope, status_word());
}

cudaError_t launch_norm_rope_fp8_window(LatentSource src, int B, int n_tok, int d, int r,
                                        const float* gamma, float eps, float rope_base,
                                        const int32_t* tok_pos0, const int32_t* win_pos0, int swa_cap,
                                        uint8_t* codes, float* scales, cudaStream_t s) {
  const int64_t rows = (int64_t)B * n_tok;
  if (rows == 0) return cudaSuccess;
  if (r < 0 || r / 2 > 256 || d > 512 || d % 16 != 0) return cudaErrorInvalidValue;
  const RopeTurns rope = rope_turns(r, rope_base);
  return launch_step(k_norm_rope_fp8_window, dim3(grid_for(rows, kNrpWarps)), dim3(kNrpWarps * 32), 0, s,
                     src, B, n_tok, d, r, gamma, eps, tok_pos0, win_pos0, swa_cap, codes, scales, rope,
                     status_word());
}

}  // namespace csa2
