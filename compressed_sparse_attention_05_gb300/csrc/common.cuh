// Shared device helpers of the CSA2 kernels: number formats, bf16 bits,
// warp reductions, and the launch-side plumbing (status word, errors).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/csa2.h"

namespace csa2 {

constexpr int kPage = 64;  // compressed entries per KV page

// ---------------------------------------------------------------------------
// E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinity)

// Value of an E4M3 code.  Exponent field 0 is subnormal: m * 2^-9.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  const uint32_t e = (c >> 3) & 0xFu, m = c & 7u;
  float mag = (e == 0) ? (float)m * 0.001953125f
                       : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return __uint_as_float(__float_as_uint(mag) | ((c & 0x80u) << 24));
}

// Round-to-nearest-even, satfinite E4M3 code of an fp32 value (hardware cvt;
// both halves of the packed result hold the same conversion).
__device__ __forceinline__ uint32_t f32_to_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(x));
  return r & 0xFFu;
}

// Round-to-nearest-even, satfinite E2M1 code of an fp32 value.  Magnitudes
// 0, .5, 1, 1.5, 2, 3, 4, 6 have codes 0..7; a midpoint goes to the even
// code; the sign bit is kept (so small negatives give code 0x8).
__device__ __forceinline__ uint32_t f32_to_e2m1(float v) {
  const float a = fabsf(v);
  uint32_t c;
  if (a <= 0.25f) c = 0;
  else if (a < 0.75f) c = 1;
  else if (a <= 1.25f) c = 2;
  else if (a < 1.75f) c = 3;
  else if (a <= 2.5f) c = 4;
  else if (a < 3.5f) c = 5;
  else if (a <= 5.0f) c = 6;
  else c = 7;
  return c | ((__float_as_uint(v) >> 28) & 8u);
}

// bf16 bit pattern of the E2M1 code c (exact: at most 2 significant bits).
__device__ __forceinline__ uint32_t e2m1_to_bf16_bits(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  uint32_t mag;
  if (e == 0) mag = m ? (126u << 7) : 0u;            // 0.5 or 0
  else mag = ((e + 126u) << 7) | (m << 6);           // 2^(e-1) * (1 + m/2)
  return mag | ((c & 8u) << 12);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// Round-to-nearest-even fp32 -> bf16 bits (finite inputs).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return u >> 16;
}

// ---------------------------------------------------------------------------
// fp16 attention operands (reading R11): powers of two that bring bf16 values
// into fp16's range without touching a significand bit

// 2^e as an fp32 value (e in [-126, 127]).
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }

// Exponent f of a window row's dequantisation scale s: 0 while the row's
// values bf16(e4m3 * s) are exact in fp16 (s in [2^-8, 2^7]: magnitudes in
// [2^-17, 65504], every bf16 bit above 2^-24), else floor(log2 s) clamped to
// [-100, 100]; the row is then dequantised with s * 2^-f (in [1, 2)), its
// logits are multiplied by 2^f and its softmax weight p is carried as 2^f p.
__device__ __forceinline__ int window_exp(float s) {
  if (!(s > 0.f) || (s >= 0.00390625f && s <= 128.f)) return 0;
  const int e = (int)((__float_as_uint(s) >> 23) & 0xFFu) - 127;
  return e < -100 ? -100 : (e > 100 ? 100 : e);
}

// Exponent e_h that scales a head of Q (largest bf16 exponent field eb, 0 for
// an all-zero head) so that its largest magnitude lies in [2^14, 2^15).
__device__ __forceinline__ int q_head_exp(int eb) {
  return eb ? (eb - 141 < -110 ? -110 : (eb - 141 > 110 ? 110 : eb - 141)) : 0;
}

// ---------------------------------------------------------------------------
// MXFP4 group of 16 channels (scale = E4M3(amax / 6), codes = E2M1(x / scale))

struct Mxfp4Group {
  uint2 codes;    // 16 nibbles, channel 2i in the low nibble of byte i
  uint32_t scale; // E4M3 code
};

__device__ __forceinline__ Mxfp4Group pack_group16(const float (&x)[16]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  Mxfp4Group g;
  g.scale = f32_to_e4m3(amax / 6.0f);            // IEEE division (no fast-math)
  const float s = e4m3_to_f32(g.scale);
  uint32_t lo = 0, hi = 0;
  if (s != 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) lo |= f32_to_e2m1(x[i] / s) << (4 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i) hi |= f32_to_e2m1(x[8 + i] / s) << (4 * i);
  }
  g.codes = make_uint2(lo, hi);
  return g;
}

// ---------------------------------------------------------------------------
// warp helpers

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Visible entries of the token at raw position t: j < min(n_entries, (t+1)/4).
__device__ __forceinline__ int n_visible(int n_entries, int t) {
  int v = (t + 1) >> 2;
  if (t < 0) v = 0;
  return v < n_entries ? v : n_entries;
}

// Programmatic dependent launch: the kernels of a layer step are launched so
// that the next one may start its independent prologue while this one runs.
// pdl_trigger lets the next kernel launch; pdl_wait blocks until the previous
// kernel has completed and its writes are visible (a no-op when the launch
// carried no dependency).  Every kernel launched with launch_step calls
// pdl_wait before it reads anything an earlier kernel of the step wrote.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// Physical page of entry j of sequence b, or -1 (and a status bit) if the
// page-table entry is out of range.
__device__ __forceinline__ int64_t entry_slot(const int32_t* page_table, int max_pages,
                                              int64_t n_pages, int b, int j,
                                              uint32_t* status) {
  const int lp = j >> 6;
  if (j < 0 || lp >= max_pages) {
    raise_status(status, CSA2_STATUS_BAD_INDEX);
    return -1;
  }
  const int p = page_table[(int64_t)b * max_pages + lp];
  if (p < 0 || p >= n_pages) {
    raise_status(status, CSA2_STATUS_BAD_PAGE);
    return -1;
  }
  return (int64_t)p * kPage + (j & (kPage - 1));
}

}  // namespace csa2
