// Gathered sparse MQA attention on the fifth-generation tensor cores
// (tcgen05, accumulators in tensor memory).  "DeepSeek-V4.1 架构解析" §02
// (one shared latent KV head, attention over the Top-K selection) and §03
// (FP4 main KV dequantised before the matmul; FP8 sliding window of the last
// 128 tokens).  Same result as the legacy kernels of attention.cu: head
// layout, key set and softmax follow reading R11 of include/csa2.h.
//
// Shapes: d = 512, up to 128 query heads (one CTA per group of 64), up to
// 3,072 keys per token (K <= 2,048 plus W <= 1,024).  The
// token's key list (selected entries, then window rows) is cut into chunks
// of 128 keys.  Swapped operands put the 128 keys of a chunk, not the 64
// heads, on the MMA's M side:
//   S^T [128 keys x 64 heads]  = K_chunk [128 x 512] . Q^T      (32 MMAs, k = 16 dims)
//   O^T [512 dims x 64 heads] += V_chunk^T [512 x 128] . P^T    (4 M-tiles x 8 MMAs, k = 16 keys)
// K = V, so one dequantised shared-memory tile serves as the K-major A
// operand of the first product and as the MN-major A operand of the second.
// S^T takes 64 tensor-memory columns and O^T four M-tiles of 64.  PV runs
// tile by tile with a commit per tile, so that the next chunk's slice of the
// K tile is rewritten as soon as the tile that read it is done.
//
// A CTA (16 worker warps and one MMA warp) owns one token (all heads) and a contiguous run of its
// chunks.  Per chunk: the threads dequantise the tile in four 128-dim slices
// (thread = one key x 32 dims of every slice, a warp = 8 whole keys); each
// warp announces a written slice on an mbarrier and
// the MMA warp issues the slice's eight S MMAs once all warps have, so
// dequantisation overlaps the tensor core.  (An MMA issue blocks the issuing
// thread while the tensor pipe is full, hence a warp of its own.)  The next
// chunk's bytes are requested together once the tile is written (loads spread
// over the slices stall the slices that follow them).  Softmax (thread = one key x 16 heads): the reference maximum of a
// head only moves when a score exceeds it by more than 2^8 (then O^T is
// rescaled in tensor memory), so P = exp2(s - m) <= 256 fits fp16 and most
// chunks need no maximum reduction at all; row sums stay per thread until
// the end of the token.
//
// Few tokens (decode): a token's keys are spread evenly over a cluster of up
// to 8 CTAs; each CTA finishes a partial (m, l, O) and the cluster merges
// them through distributed shared memory, without global scratch: every rank
// owns a slice of the heads and sums the ranks' scaled partials of those heads
// in rank order.
//
// Operands are fp16.  MXFP4 values (<= 6 significant bits, in [2^-10, 2688])
// are exact.  bf16 values outside fp16's range are brought into it by powers
// of two, which change no bit of a significand: each head of Q is scaled by
// 2^-e_h so that its largest magnitude lies in [2^14, 2^15) (and its logits
// are multiplied back by 2^e_h), and a window row whose per-token scale lies
// outside [2^-8, 2^7] is dequantised with the scale 2^-f s (s' in [1, 2)), its
// logits multiplied back by 2^f and its softmax weight carried as 2^f p in the
// PV product (the reference maximum then follows the largest 2^f p, and the
// normaliser adds p itself).  Main-KV entries in the FP8 format (the V4-style
// layout kept for the A/B against MXFP4: E4M3 row + fp32 scale, one 32-byte
// run of codes per thread and slice) go through the window rows' path: code x
// scale rounded to bf16, the same power-of-two treatment; the kernel is
// instantiated once per format.  P is rounded to fp16 for the PV product; the
// normaliser sums the unrounded fp32 P (relative difference <= 2^-11).
// Accumulation is fp32.
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace csa2 {
namespace {

constexpr int kD = 512;          // latent width (keys = values)
constexpr int kHeads = 64;       // N of both products; fewer heads are zero-padded
constexpr int kChunk = 128;      // keys per chunk (M of the score product)
constexpr int kMaxChunks = 24;   // keys per token <= 3,072 (K <= 2,048 plus W <= 1,024)
constexpr int kMaxSplit = 8;     // CTAs per token in the cluster path (largest portable cluster)
constexpr int kWorkers = 512;             // 16 warps: dequantisation and softmax
constexpr int kThreads = kWorkers + 32;   // + one warp that allocates tensor memory and issues the MMAs
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;     // S^T: 64 columns
constexpr uint32_t kColO = 256;   // O^T: four M-tiles of 64 columns
constexpr float kRescaleLog2 = 8.f;  // move a head's reference maximum only beyond this growth

// Byte offsets inside the operand tiles (no-swizzle canonical layout: core
// matrices of 8 rows x 16 bytes).
//   Q  [head][dim]: (h/8)*8192 + (d/8)*128 + (h%8)*16 + (d%8)*2
//   K  [key][dim]:  (k/8)*8192 + (d/8)*128 + (k%8)*16 + (d%8)*2
//   P  [key][head]: (k/8)*1024 + (h/8)*128 + (k%8)*16 + (h%8)*2
struct TcSmem {
  uint16_t q[kHeads * kD];
  uint16_t k[kChunk * kD];             // becomes the fp32 partial O [64][512] in the cluster merge
  uint16_t p[kChunk * kHeads];
  int32_t slot[kMaxChunks * kChunk];   // >= 0 main-KV slot; <= -2 window row (-2 - row); -1 none
  int8_t kexp[kMaxChunks * kChunk];    // window row: exponent f of its dequantisation scale (0: none)
  float red[4][kHeads];                // per lane-quarter partial max / sum
  float sl2h[kHeads];                  // logit multiplier of each head: softmax scale * log2(e) * 2^e_h
  int qexp[kHeads];                    // largest bf16 exponent field of each head of Q
  float m_ref[kHeads];                 // reference maximum (log2 domain) of each head
  float m_thr[kHeads];                 // m_ref + 2^8 growth allowance
  float m_exp[kHeads];                 // m_ref, or 0 while the head has seen no key
  float alpha[kHeads], l_run[kHeads], fac[kHeads];
  uint64_t k_ready[4];   // workers -> MMA warp: slice of the K tile written (one arrival per warp)
  uint64_t p_ready;      // workers -> MMA warp: P written, O^T rescaled
  uint64_t bar_s;        // MMA commit: S^T complete
  uint64_t bar_pv[4];    // MMA commit: PV M-tile complete (its K slice is free again)
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
// Two E2M1 codes (one byte, even channel in the low nibble) -> f16x2, low half first.
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(r) : "r"(byte));
  return r;
}
// Two E4M3 codes (low 16 bits, first code in the low byte) -> f16x2, low half first (exact).
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t pair) {
  uint32_t r;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(r) : "r"(pair));
  return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// (lo, hi) fp32 -> f16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t f32x2_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// (lo, hi) fp32 -> bf16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t f32x2_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float f16_lo(uint32_t h2) { return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))); }
__device__ __forceinline__ float f16_hi(uint32_t h2) { return __half2float(__ushort_as_half((unsigned short)(h2 >> 16))); }
// Two window codes -> f16x2 of bf16(fp32(e4m3 * scale)) (the window operand).
__device__ __forceinline__ uint32_t win2_f16x2(uint32_t pair, float sc) {
  const uint32_t e = e4m3x2_f16x2(pair);
  const uint32_t bf = f32x2_bf16x2(f16_lo(e) * sc, f16_hi(e) * sc);
  return f32x2_f16x2(__uint_as_float(bf << 16), __uint_as_float(bf & 0xFFFF0000u));
}
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Reduction (max or sum) over the 32 lanes of each of 16 columns; lane L
// ends with column L & 15.  v is consumed.
template <bool kMax>
__device__ __forceinline__ float reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float o = __shfl_xor_sync(0xffffffffu, v[j], 16);
    v[j] = kMax ? fmaxf(v[j], o) : v[j] + o;
  }
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int j = 0; j < w; ++j) {
      const float send = upper ? v[j] : v[j + w];
      const float keep = upper ? v[j + w] : v[j];
      const float got = __shfl_xor_sync(0xffffffffu, send, w);
      v[j] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

// ---- distributed shared memory (cluster merge) ------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_cluster(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Barrier / vote among the worker warps only (the MMA warp never joins).
__device__ __forceinline__ void workers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kWorkers) : "memory");
}
__device__ __forceinline__ bool workers_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kWorkers)
      : "memory");
  return r != 0;
}

// Packed bytes of one key for the thread's 32 dims (128*sl + 32*qd ..) of each
// slice sl, held in registers from the moment they are requested until the slice
// is stored, so that the gather of the next chunk overlaps this chunk's products.
struct KeyBytes {
  uint4 v[4];
};
// Loads that the compiler keeps where they are written (volatile): a plain load
// may be moved down to its first use, which would turn the prefetch into a stall.
__device__ __forceinline__ uint4 ld_gather16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_gather8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_gather4f(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
// MXFP4 scales of a key: quarter qd loads bytes 8*qd .. +7 (the groups of slice qd)
__device__ __forceinline__ uint2 load_scales(const AttnArgs& a, int32_t src, int qd) {
  return src >= 0 ? ld_gather8(a.kv_scales + (int64_t)src * (kD / 16) + 8 * qd) : make_uint2(0, 0);
}
// A key stored as an FP8 row: a window row, or a main-KV entry in the FP8 format.
template <bool kFp8>
__device__ __forceinline__ bool fp8_row_key(int32_t src) {
  return src <= -2 || (kFp8 && src >= 0);
}

// Packed bytes of slice SL of a key for the thread's 32 dims.  MXFP4 entry:
// 16 bytes, in v[SL] (all four slices are requested together).  FP8 row: 32
// bytes, in v[2 (SL & 1)] and the next (slices 0 and 1 are requested together,
// slices 2 and 3 reuse their registers once 0 and 1 are stored).
template <int SL, bool kFp8>
__device__ __forceinline__ void load_slice(const AttnArgs& a, int32_t src, int qd, KeyBytes& kb) {
  if (src == -1) return;
  if (fp8_row_key<kFp8>(src)) {
    const uint8_t* p = (src <= -2 ? a.swa_codes + (-2 - (int64_t)src) * kD : a.kv_codes + (int64_t)src * kD) +
                       32 * qd + 128 * SL;
    kb.v[2 * (SL & 1)] = ld_gather16(p);
    kb.v[2 * (SL & 1) + 1] = ld_gather16(p + 16);
  } else {
    kb.v[SL] = ld_gather16(a.kv_codes + (int64_t)src * (kD / 2) + 16 * qd + 64 * SL);
  }
}
// Dequantisation scale of an FP8 row (a window row, or a main-KV entry in the FP8
// format), times 2^-f (see window_exp); 0 for an MXFP4 entry or no key.
template <bool kFp8>
__device__ __forceinline__ float load_wscale(const AttnArgs& a, int32_t src) {
  float sw;
  if (src <= -2) sw = ld_gather4f(a.swa_scales + (-2 - (int64_t)src));
  else if (kFp8 && src >= 0) sw = ld_gather4f(reinterpret_cast<const float*>(a.kv_scales) + src);
  else return 0.f;
  return sw * pow2i(-window_exp(sw));
}
// Exponent f of a key's FP8 scale (0 for MXFP4 entries and missing keys).
template <bool kFp8>
__device__ __forceinline__ int key_exp(const AttnArgs& a, int32_t src) {
  if (src <= -2) return window_exp(__ldg(a.swa_scales + (-2 - (int64_t)src)));
  if (kFp8 && src >= 0) return window_exp(__ldg(reinterpret_cast<const float*>(a.kv_scales) + src));
  return 0;
}

// 32 E4M3 codes (c0: dims 0-15, c1: 16-31) times the (2^-f scaled) row scale,
// rounded to bf16 as the operand rule says, into 4 core-matrix rows of fp16.
__device__ __forceinline__ void store_fp8_dims(uint4 c0, uint4 c1, float sc, unsigned char* dst) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 c = j < 2 ? c0 : c1;
    const uint32_t w0 = word_of(c, (j & 1) * 2), w1 = word_of(c, (j & 1) * 2 + 1);
    uint4 o;
    o.x = win2_f16x2(w0 & 0xFFFFu, sc);
    o.y = win2_f16x2(w0 >> 16, sc);
    o.z = win2_f16x2(w1 & 0xFFFFu, sc);
    o.w = win2_f16x2(w1 >> 16, sc);
    *reinterpret_cast<uint4*>(dst + j * 128) = o;
  }
}

// Dequantise the thread's 32 dims of slice SL into the K tile (4 core-matrix rows).
template <int SL, bool kFp8>
__device__ __forceinline__ void store_slice(const AttnArgs& a, const KeyBytes& kb, uint32_t sc_pair, int32_t src,
                                            float wsc, int key, int qd, unsigned char* ktile) {
  unsigned char* dst = ktile + (key >> 3) * 8192 + (16 * SL + 4 * qd) * 128 + (key & 7) * 16;
  if (fp8_row_key<kFp8>(src)) {
    store_fp8_dims(kb.v[2 * (SL & 1)], kb.v[2 * (SL & 1) + 1], wsc, dst);
  } else if (src >= 0) {
    const uint32_t s = e4m3x2_f16x2(sc_pair);
    const uint32_t g0 = prmt(s, s, 0x1010u), g1 = prmt(s, s, 0x3232u);   // (scale, scale) of each group
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t w = word_of(kb.v[SL], j);
      const uint32_t s2 = j < 2 ? g0 : g1;
      uint4 o;
      o.x = hmul2(e2m1x2_f16x2(w & 0xFFu), s2);   // exact: <= 6 significant bits
      o.y = hmul2(e2m1x2_f16x2((w >> 8) & 0xFFu), s2);
      o.z = hmul2(e2m1x2_f16x2((w >> 16) & 0xFFu), s2);
      o.w = hmul2(e2m1x2_f16x2(w >> 24), s2);
      *reinterpret_cast<uint4*>(dst + j * 128) = o;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(dst + j * 128) = make_uint4(0, 0, 0, 0);
  }
}

// Resolves key kk of a CTA's key list -- sel_cap selection slots (slots sel_off ..
// of the token's Top-K, the first n_sel of which hold selected entries), then
// window rows from raw position w_first -- to a main-KV slot (page table) or a
// window row, or -1 past the list [.., kk_end) or in an unused selection slot.
// The index load does not wait for n_sel when sel_cap is fixed (the cluster path).
__device__ __forceinline__ int32_t key_source(const AttnArgs& a, int64_t row, int b, int kk, int n_sel, int sel_off,
                                              int sel_cap, int kk_end, int nv, int w_first, int pos0, bool report,
                                              uint32_t* status) {
  if (kk >= kk_end) return -1;
  if (kk < sel_cap) {
    const int j = __ldg(a.idx + row * a.K + sel_off + kk);
    if (sel_off + kk >= n_sel) return -1;
    if (j < 0 || j >= nv || (j >> 6) >= a.max_pages) {
      if (report) raise_status(status, CSA2_STATUS_BAD_INDEX);
      return -1;
    }
    const int p = __ldg(a.page_table + (int64_t)b * a.max_pages + (j >> 6));
    if (p < 0 || p >= a.n_pages) {
      if (report) raise_status(status, CSA2_STATUS_BAD_PAGE);
      return -1;
    }
    return p * kPage + (j & (kPage - 1));
  }
  return (int32_t)(-2 - ((int64_t)b * a.swa_cap + (w_first + (kk - sel_cap) - pos0)));
}

// Scores of the thread's key for heads 16*hg .. +15 in the log2 domain, as
// the PV product carries them: y = x + f with x = S^T * scale * log2(e) (the
// head's and the key's powers of two undone), or -inf for a missing key.
__device__ __forceinline__ void load_scores(uint32_t tm, int hg, uint32_t lane_q, bool valid, const float* sl2h,
                                            int fk, float (&x)[16]) {
  tc::tmem_ld16(tm + kColS + 16 * hg + lane_q, x);
  tc::tmem_wait_ld();
  const float4* m4 = reinterpret_cast<const float4*>(sl2h + 16 * hg);
#pragma unroll
  for (int j4 = 0; j4 < 4; ++j4) {
    const float4 m = m4[j4];
    x[4 * j4] *= m.x; x[4 * j4 + 1] *= m.y; x[4 * j4 + 2] *= m.z; x[4 * j4 + 3] *= m.w;
  }
  if (fk != 0) {   // a rescaled window row: logits times 2^f, weights carried as 2^f p
    const float kf = pow2i(fk), ff = (float)fk;
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = x[j] * kf + ff;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) x[j] = valid ? x[j] : -INFINITY;
}

// Bounded wait of a whole warp; on time-out the CTA's abort flag is raised.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  bool ok = false;
  for (uint32_t i = 0; i < (1u << 21); ++i) {   // <= 2^21 suspensions of <= 1 us
    if (tc::mbar_try_wait_sleep(bar, parity, 1000)) {
      ok = true;
      break;
    }
    if ((i & 63) == 63 && *abort) break;
  }
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) *abort = 1;
  return ok;
}



template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
k_sparse_attn_tc(AttnArgs a, uint32_t* status, int n_split) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  TcSmem& sm = *reinterpret_cast<TcSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool mma_warp = warp == kWorkers / 32;
  const int64_t row = blockIdx.x / n_split;
  const int rank = (int)(blockIdx.x % n_split);
  const int b = (int)(row / a.Tq);
  const int hb = kHeads * (int)blockIdx.y;   // first head of this CTA's group of 64
  // dequantisation: one key, 32 dims of each slice.  A warp holds 8 whole keys
  // (coalesced loads); lanes 8q .. 8q+7 hold quarter q of the 8 keys, so each
  // 8-lane phase of a 16-byte store covers 8 distinct bank groups.
  const int key = ((warp & 15) << 3) | (lane & 7), qd = (lane >> 3) & 3;
  const int q4 = warp & 3, hg = (warp >> 2) & 3;             // softmax: key 32*q4 + lane (= key), heads 16*hg ..
  volatile int* abort = &sm.abort;

  pdl_trigger();
  // ---- before the previous kernel of the step is done: the token's own inputs
  // (scalars, Q rows), barriers, tensor memory and the Q operand
  const int t = a.q_pos[row];
  const int n_ent = a.n_entries[b];
  const int pos0 = a.swa_cap > 0 ? a.swa_pos0[b] : 0;
  uint4 qv[8];   // unit = (head, 8 dims); 8 heads of a unit group share a core matrix
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int u = tid + kWorkers * r;
    const int h = ((u >> 9) << 3) | (u & 7), c8 = (u >> 3) & 63;
    qv[r] = (!mma_warp && hb + h < a.Hq) ? __ldg(reinterpret_cast<const uint4*>(a.Q + (row * a.Hq + hb + h) * kD + c8 * 8))
                                    : make_uint4(0, 0, 0, 0);
  }
  if (tid == 0) {
    tc::mbar_init(&sm.bar_s, 1);
    tc::mbar_init(&sm.p_ready, kWorkers / 32);
    for (int i = 0; i < 4; ++i) {
      tc::mbar_init(&sm.bar_pv[i], 1);
      tc::mbar_init(&sm.k_ready[i], kWorkers / 32);
    }
    sm.abort = 0;
    tc::mbar_fence_init();
  }
  if (mma_warp) tc::tmem_alloc(&sm.tmem, kTmemCols);
  if (tid < kHeads) {
    sm.m_ref[tid] = -INFINITY;
    sm.m_thr[tid] = -INFINITY;
    sm.m_exp[tid] = 0.f;
    sm.qexp[tid] = 0;
  }
  __syncthreads();
  // largest bf16 exponent field of each head (lanes L, L^8, L^16, L^24 share a head)
  if (!mma_warp) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      uint32_t e = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w = word_of(qv[r], j);
        e = max(e, max((w >> 7) & 0xFFu, (w >> 23) & 0xFFu));
      }
      e = max(e, __shfl_xor_sync(0xffffffffu, e, 8));
      e = max(e, __shfl_xor_sync(0xffffffffu, e, 16));
      if (lane < 8 && e) atomicMax(&sm.qexp[8 * r + lane], (int)e);
    }
  }
  __syncthreads();
  // per head: 2^-e_h brings the largest magnitude into [2^14, 2^15) (e_h in [-110, 110])
  if (tid < kHeads) {
    const int eh = q_head_exp(sm.qexp[tid]);
    sm.qexp[tid] = eh;
    sm.sl2h[tid] = a.scale * 1.4426950408889634f * pow2i(eh);
  }
  __syncthreads();
  // Q (bf16) -> fp16 B operand, head h scaled by 2^-e_h (exact)
  if (!mma_warp) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int u = tid + kWorkers * r;
      const int h = ((u >> 9) << 3) | (u & 7), c8 = (u >> 3) & 63;
      const float qs = pow2i(-sm.qexp[h]);
      uint32_t ov[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w = word_of(qv[r], j);
        ov[j] = f32x2_f16x2(__uint_as_float(w << 16) * qs, __uint_as_float(w & 0xFFFF0000u) * qs);
      }
      *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(sm.q) + (h >> 3) * 8192 + c8 * 128 + (h & 7) * 16) =
          make_uint4(ov[0], ov[1], ov[2], ov[3]);
    }
  }
  // the window rows of the token: raw positions max(0, t-W+1, pos0) .. min(t, last row held)
  const int w_lo = max(max(0, t - a.W + 1), pos0);
  const int w_hi = min(t, pos0 + a.swa_cap - 1);
  const int n_win = max(0, w_hi - w_lo + 1);
  // ---- the selection (and the window rows) come from earlier kernels of the step
  pdl_wait();
  int n_sel = a.cnt[row];
  const int nv = n_visible(n_ent, t);
  if (n_sel < 0 || n_sel > a.K) {
    if (tid == 0 && rank == 0) raise_status(status, CSA2_STATUS_BAD_COUNT);
    n_sel = n_sel < 0 ? 0 : a.K;
  }
  // the key list.  One CTA per token: its n_sel selected entries, then its window
  // rows.  A cluster: rank r takes an equal share of the K selection slots (unused
  // ones empty, so that the index loads need not wait for the count) and an equal
  // share of the window rows.
  int sel_off = 0, sel_cap = n_sel, w_first = w_lo, n_mine = n_sel + n_win;
  if (n_split > 1) {
    sel_off = (int)((int64_t)a.K * rank / n_split);
    sel_cap = (int)((int64_t)a.K * (rank + 1) / n_split) - sel_off;
    const int u0 = (int)((int64_t)n_win * rank / n_split), u1 = (int)((int64_t)n_win * (rank + 1) / n_split);
    w_first = w_lo + u0;
    n_mine = sel_cap + (u1 - u0);
  }
  const int kb0 = 0, kb1 = n_mine;
  const int n_my = (kb1 - kb0 + kChunk - 1) / kChunk;   // chunks of kChunk keys, <= kMaxChunks

  // ---- key sources.  Every worker resolves its key in the first chunk; the
  // key's later chunks are shared out among its four threads.
  int32_t cur_src = -1;
  if (!mma_warp && n_my > 0) {
    cur_src = key_source(a, row, b, kb0 + key, n_sel, sel_off, sel_cap, kb1, nv, w_first, pos0, qd == 0, status);
    if (qd == 0) {
      sm.slot[key] = cur_src;
      sm.kexp[key] = (int8_t)key_exp<kFp8>(a, cur_src);
    }
    for (int c = qd + 1; c < n_my; c += 4) {
      const int32_t src =
          key_source(a, row, b, kb0 + c * kChunk + key, n_sel, sel_off, sel_cap, kb1, nv, w_first, pos0, true,
                     status);
      sm.slot[c * kChunk + key] = src;
      sm.kexp[c * kChunk + key] = (int8_t)key_exp<kFp8>(a, src);
    }
  }
  // ---- the first chunk's packed bytes
  float cur_wsc = 0.f;
  uint2 cur_sc = make_uint2(0, 0);
  KeyBytes kb;
  if (!mma_warp && n_my > 0) {
    load_slice<0, kFp8>(a, cur_src, qd, kb);
    load_slice<1, kFp8>(a, cur_src, qd, kb);
    if (!fp8_row_key<kFp8>(cur_src)) {
      load_slice<2, kFp8>(a, cur_src, qd, kb);
      load_slice<3, kFp8>(a, cur_src, qd, kb);
      cur_sc = load_scales(a, cur_src, qd);
    }
    cur_wsc = load_wscale<kFp8>(a, cur_src);
  }
  tc::fence_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = sm.tmem;

  if (mma_warp) {
    // ================= MMA issue (one thread; an MMA issue blocks while the tensor pipe is busy) ====
    if (lane == 0) {
      constexpr uint32_t kIdS = tc::idesc_f16(128, kHeads, 0, 0, 0);   // K-major A and B
      constexpr uint32_t kIdO = tc::idesc_f16(128, kHeads, 0, 1, 1);   // MN-major A and B
      const uint64_t dk_s = tc::smem_desc(tc::smem_addr(sm.k), 128, 8192);
      const uint64_t dq_s = tc::smem_desc(tc::smem_addr(sm.q), 128, 8192);
      const uint64_t dk_o = tc::smem_desc(tc::smem_addr(sm.k), 8192, 128);
      const uint64_t dp_o = tc::smem_desc(tc::smem_addr(sm.p), 1024, 128);
      for (int it = 0; it < n_my; ++it) {
        bool ok = true;
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
          ok = ok && tc::mbar_wait(&sm.k_ready[sl], it & 1, 1u << 22);
          if (!ok) break;
          tc::tc_fence_after();
#pragma unroll
          for (int ks = 8 * sl; ks < 8 * sl + 8; ++ks)   // descriptor addresses advance in 16-byte units
            tc::mma_f16(tm + kColS, dk_s + (uint64_t)(ks * 16), dq_s + (uint64_t)(ks * 16), kIdS, ks > 0);
        }
        if (!ok) { *abort = 1; break; }
        tc::mma_commit(&sm.bar_s);
        if (!tc::mbar_wait(&sm.p_ready, it & 1, 1u << 22)) { *abort = 1; break; }
        tc::tc_fence_after();
        // PV over the chunk's keys only (a short last chunk skips its empty 16-key steps)
        const int ksteps = (min(kChunk, kb1 - kb0 - kChunk * it) + 15) / 16;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {   // tile by tile: a finished tile frees its K slice for the next chunk
          for (int kk = 0; kk < ksteps; ++kk)
            tc::mma_f16(tm + kColO + 64 * mt, dk_o + (uint64_t)(mt * 128 + kk * 1024), dp_o + (uint64_t)(kk * 128),
                        kIdO, (it > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(&sm.bar_pv[mt]);
        }
      }
    }
    __syncwarp();
  } else {
    // ================= workers: dequantisation and softmax =================
    unsigned char* ktile = reinterpret_cast<unsigned char*>(sm.k);
    const uint32_t lane_q = (uint32_t)(32 * q4) << 16;
    const int kc = 32 * q4 + lane;   // the softmax thread's key
    float lsum[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) lsum[j] = 0.f;

    for (int it = 0; it < n_my; ++it) {
      const int32_t nxt_src = it + 1 < n_my ? sm.slot[(it + 1) * kChunk + key] : -1;
      bool wok = true;
      // ---- dequantise slice by slice; refill each slice's registers with the next chunk
#define CSA2_SLICE(SL)                                                                   \
  {                                                                                      \
    if (it > 0) wok = wok && warp_wait(&sm.bar_pv[SL], (it - 1) & 1, abort);             \
    {                                                                                    \
      /* the slice's two group scales were loaded by quarter SL of the key */            \
      const uint32_t w0 = __shfl_sync(0xffffffffu, cur_sc.x, (lane & 7) | (SL << 3));    \
      const uint32_t w1 = __shfl_sync(0xffffffffu, cur_sc.y, (lane & 7) | (SL << 3));    \
      const uint32_t pr = ((qd >> 1) ? w1 : w0) >> (16 * (qd & 1));                      \
      if (wok) store_slice<SL, kFp8>(a, kb, pr & 0xFFFFu, cur_src, cur_wsc, key, qd, ktile); \
      /* FP8 rows: slices 2 and 3 of this chunk reuse the registers of 0 and 1 */        \
      if (SL < 2 && fp8_row_key<kFp8>(cur_src)) load_slice<(SL + 2) & 3, kFp8>(a, cur_src, qd, kb); \
    }                                                                                    \
    tc::fence_async_smem();                                                              \
    __syncwarp();                                                                        \
    if (lane == 0) tc::mbar_arrive(&sm.k_ready[SL]);                                     \
  }
      CSA2_SLICE(0)
      CSA2_SLICE(1)
      CSA2_SLICE(2)
      CSA2_SLICE(3)
#undef CSA2_SLICE
      // the next chunk's bytes, requested together once this chunk's tile is written
      if (it + 1 < n_my) {
        load_slice<0, kFp8>(a, nxt_src, qd, kb);
        load_slice<1, kFp8>(a, nxt_src, qd, kb);
        if (!fp8_row_key<kFp8>(nxt_src)) {
          load_slice<2, kFp8>(a, nxt_src, qd, kb);
          load_slice<3, kFp8>(a, nxt_src, qd, kb);
        }
      }
      const bool valid = sm.slot[it * kChunk + kc] != -1;   // the softmax thread's key
      const int fk = sm.kexp[it * kChunk + kc];
      cur_src = nxt_src;
      cur_wsc = load_wscale<kFp8>(a, nxt_src);
      if (!kFp8) cur_sc = load_scales(a, nxt_src, qd);

      // ---- softmax of the chunk: this thread's key, heads 16*hg .. +15
      wok = wok && warp_wait(&sm.bar_s, it & 1, abort);
      tc::tc_fence_after();
      float x[16];
      bool above = false;
      if (wok) {
        load_scores(tm, hg, lane_q, valid, sm.sl2h, fk, x);
        const float4* thr = reinterpret_cast<const float4*>(&sm.m_thr[16 * hg]);
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          const float4 th = thr[j4];
          above |= (x[4 * j4] > th.x) | (x[4 * j4 + 1] > th.y) | (x[4 * j4 + 2] > th.z) | (x[4 * j4 + 3] > th.w);
        }
      }
      // one vote per chunk: did a score outgrow its head's reference, or has a
      // wait failed?  (The flag is read before the vote, so all workers agree.)
      const bool seen_abort = *abort != 0;
      if (workers_or(above || seen_abort)) {
        if (workers_or(seen_abort)) break;
        // reduce the chunk's maxima (x is consumed, then summed again from tensor memory)
        const float mx = reduce16<true>(x, lane);
        if (lane < 16) sm.red[q4][16 * hg + lane] = mx;
        load_scores(tm, hg, lane_q, valid, sm.sl2h, fk, x);
        workers_sync();
        int need = 0;
        if (tid < kHeads) {
          const float mloc = fmaxf(fmaxf(sm.red[0][tid], sm.red[1][tid]), fmaxf(sm.red[2][tid], sm.red[3][tid]));
          const float mo = sm.m_ref[tid];
          float al = 1.f;
          if (mloc > mo + kRescaleLog2 || (mo == -INFINITY && mloc > -INFINITY)) {
            if (mo != -INFINITY) {   // the head holds keys already: rescale them
              al = ex2(mo - mloc);
              need = 1;
            }
            sm.m_ref[tid] = mloc;
            sm.m_thr[tid] = mloc + kRescaleLog2;
            sm.m_exp[tid] = mloc;
          }
          sm.alpha[tid] = al;
        }
        if (workers_or(need)) {
          // O^T *= alpha (per head = column): warp 4*mt + q4 takes M-tile mt, its lane quarter
          const int mt = warp >> 2;
#pragma unroll 1
          for (int c = 0; c < kHeads; c += 16) {
            const uint32_t ta = tm + kColO + 64 * mt + c + lane_q;
            float o[16];
            tc::tmem_ld16(ta, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] *= sm.alpha[c + j];
            tc::tmem_st16(ta, o);
          }
          tc::tmem_wait_st();
#pragma unroll
          for (int j = 0; j < 16; ++j) lsum[j] *= sm.alpha[16 * hg + j];
        }
      }
      // P = exp2(s - m_ref) in fp16 (the MN-major B operand of the PV product)
      {
        uint32_t pk[8];
        const float pf = pow2i(-fk);   // the normaliser adds p = 2^-f (2^f p)
        const float4* me = reinterpret_cast<const float4*>(&sm.m_exp[16 * hg]);
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          const float4 m4 = me[j4];
          const float p0 = ex2(x[4 * j4] - m4.x), p1 = ex2(x[4 * j4 + 1] - m4.y);
          const float p2 = ex2(x[4 * j4 + 2] - m4.z), p3 = ex2(x[4 * j4 + 3] - m4.w);
          lsum[4 * j4] += p0 * pf;
          lsum[4 * j4 + 1] += p1 * pf;
          lsum[4 * j4 + 2] += p2 * pf;
          lsum[4 * j4 + 3] += p3 * pf;
          pk[2 * j4] = f32x2_f16x2(p0, p1);
          pk[2 * j4 + 1] = f32x2_f16x2(p2, p3);
        }
        unsigned char* pdst =
            reinterpret_cast<unsigned char*>(sm.p) + (kc >> 3) * 1024 + (2 * hg) * 128 + (kc & 7) * 16;
        *reinterpret_cast<uint4*>(pdst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(pdst + 128) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
      tc::fence_async_smem();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.p_ready);
    }
    // all PV products of the CTA are complete once the last commit has arrived
    if (!*abort && n_my > 0) warp_wait(&sm.bar_pv[3], (n_my - 1) & 1, abort);
    tc::tc_fence_after();
    // row sums over the 128 keys: warp, then lane quarters
    const float s = reduce16<false>(lsum, lane);
    if (lane < 16) sm.red[q4][16 * hg + lane] = s;
  }
  __syncthreads();
  const bool ok = *abort == 0;
  const bool have_o = ok && n_my > 0;
  if (tid < kHeads) sm.l_run[tid] = (sm.red[0][tid] + sm.red[1][tid]) + (sm.red[2][tid] + sm.red[3][tid]);
  __syncthreads();
  const int mt = (warp >> 2) & 3;   // epilogue (workers): warp takes M-tile mt, dims 128*mt + 32*q4 + lane

  if (n_split == 1) {
    if (tid < kHeads) sm.fac[tid] = sm.l_run[tid] > 0.f ? 1.f / sm.l_run[tid] : 0.f;
    if (a.lse && tid < kHeads && hb + tid < a.Hq) {
      const float l = sm.l_run[tid];
      a.lse[row * a.Hq + hb + tid] = l > 0.f ? (sm.m_ref[tid] + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    if (!mma_warp) {
      for (int c = 0; c < kHeads; c += 16) {
        float o[16];
        if (have_o) {
          tc::tmem_ld16(tm + kColO + 64 * mt + c + ((uint32_t)(32 * q4) << 16), o);
          tc::tmem_wait_ld();
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int h = c + j;
          if (hb + h < a.Hq) a.O[(row * a.Hq + hb + h) * kD + 128 * mt + 32 * q4 + lane] = have_o ? o[j] * sm.fac[h] : 0.f;
        }
      }
    }
  } else {
    // ---- merge the cluster's partials with one exchange.  Every rank publishes its
    // (m, l) and its unscaled partial O in its own shared memory, [head][dim] (a
    // warp's remote reads below are then contiguous); after one cluster barrier
    // rank r sums heads [own(r), own(r+1)) over the ranks in rank order, each rank's
    // partial scaled by 2^(m_q - M) / L.
    const int crank = (int)cluster_rank();
    float* part = reinterpret_cast<float*>(sm.k);   // every MMA that read the K tile is complete
    if (!mma_warp) {
      const int dim = 128 * mt + 32 * q4 + lane;
      for (int c = 0; c < kHeads; c += 16) {
        float o[16];
        if (have_o) {
          tc::tmem_ld16(tm + kColO + 64 * mt + c + ((uint32_t)(32 * q4) << 16), o);
          tc::tmem_wait_ld();
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) part[(c + j) * kD + dim] = have_o ? o[j] : 0.f;
      }
    }
    cluster_sync();   // every rank's (m, l) and partial O are published
    const int h0 = kHeads * crank / n_split, h1 = kHeads * (crank + 1) / n_split;
    float* facq = reinterpret_cast<float*>(sm.q);    // [rank][head]: the Q tile is no longer read
    if (tid < kHeads) {
      // every rank's (m, l) of this head; the loads are independent (unrolled, predicated)
      const uint32_t am = tc::smem_addr(&sm.m_ref[tid]), al = tc::smem_addr(&sm.l_run[tid]);
      float mq[kMaxSplit], lq[kMaxSplit];
#pragma unroll
      for (int q = 0; q < kMaxSplit; ++q) {
        mq[q] = q < n_split ? ld_cluster(map_to_rank(am, q)) : -INFINITY;
        lq[q] = q < n_split ? ld_cluster(map_to_rank(al, q)) : 0.f;
      }
      float M = -INFINITY;
#pragma unroll
      for (int q = 0; q < kMaxSplit; ++q) M = fmaxf(M, mq[q]);
      float L = 0.f;
#pragma unroll
      for (int q = 0; q < kMaxSplit; ++q)
        if (mq[q] != -INFINITY) L += lq[q] * ex2(mq[q] - M);
#pragma unroll
      for (int q = 0; q < kMaxSplit; ++q)
        if (q < n_split) facq[q * kHeads + tid] = (mq[q] == -INFINITY || L <= 0.f) ? 0.f : ex2(mq[q] - M) / L;
      if (crank == 0 && a.lse && hb + tid < a.Hq)
        a.lse[row * a.Hq + hb + tid] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    // this rank's heads, 4 dims per element; every rank's value of two elements in flight
    const uint32_t pbase = tc::smem_addr(part);
    const int n4 = (h1 - h0) * (kD / 4);
    for (int e0 = tid; e0 < n4; e0 += 2 * kThreads) {
      float4 r[2][kMaxSplit];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int e = e0 + u * kThreads;
#pragma unroll
        for (int q = 0; q < kMaxSplit; ++q)
          r[u][q] = (q < n_split && e < n4) ? ld_cluster4(map_to_rank(pbase + 16u * (uint32_t)(h0 * (kD / 4) + e), q))
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int e = e0 + u * kThreads;
        if (e >= n4) continue;
        const int h = h0 + e / (kD / 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < kMaxSplit; ++q) {
          if (q >= n_split) break;
          const float f = facq[q * kHeads + h];
          acc.x += r[u][q].x * f; acc.y += r[u][q].y * f; acc.z += r[u][q].z * f; acc.w += r[u][q].w * f;
        }
        if (hb + h < a.Hq) *reinterpret_cast<float4*>(a.O + (row * a.Hq + hb + h) * kD + (e % (kD / 4)) * 4) = acc;
      }
    }
    cluster_sync();   // no CTA leaves while another still reads its shared memory
  }
  tc::tc_fence_before();
  __syncthreads();
  if (mma_warp) tc::tmem_dealloc(tm, kTmemCols);
  if (tid == 0 && !ok) raise_status(status, CSA2_STATUS_TIMEOUT);
}

}  // namespace

bool sparse_attn_tc_supported(const AttnArgs& a) {
  return a.d == kD && a.Hq >= 1 && a.Hq <= 2 * kHeads && a.K >= 0 && a.W >= 0 &&
         (int64_t)a.K + a.W <= (int64_t)kMaxChunks * kChunk && a.n_pages * kPage < ((int64_t)1 << 31) &&
         (int64_t)a.B * a.swa_cap < ((int64_t)1 << 31) - 2;
}

cudaError_t launch_sparse_attn_tc(const AttnArgs& a, cudaStream_t s) {
  const int64_t rows = (int64_t)a.B * a.Tq;
  if (rows == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int max_chunks = (int)((a.K + a.W + kChunk - 1) / kChunk);
  int n_split = 1;
  if (rows < sms && max_chunks > 1)
    n_split = (int)std::max<int64_t>(1, std::min<int64_t>(std::min(max_chunks, kMaxSplit), sms / rows));
  const size_t smem = sizeof(TcSmem);
  auto kernel = a.kv_fp8 ? k_sparse_attn_tc<true> : k_sparse_attn_tc<false>;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (rows * n_split >= ((int64_t)1 << 31)) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(rows * n_split), (unsigned)((a.Hq + kHeads - 1) / kHeads));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_trigger / pdl_wait
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)n_split;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = n_split > 1 ? 2 : 1;
  return counted(cudaLaunchKernelEx(&cfg, kernel, a, status_word(), n_split));
}

}  // namespace csa2
