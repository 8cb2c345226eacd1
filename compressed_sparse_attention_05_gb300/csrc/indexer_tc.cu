// Sparse-indexer scores of many query tokens at once (prefill chunks) on the
// fifth-generation tensor cores.  "DeepSeek-V4.1 架构解析" §02: every query
// scores every causally visible compressed entry, s_j = sum_h w_h ReLU(q_h . k_j)
// (score form: reading R6 of include/csa2.h).
//
// With thousands of query tokens over the same pages this is a GEMM:
//   C [128 entries x (32 queries x 8 heads)] = K_tile [128 x 128] . Q_block^T
// per 128-entry tile (two 64-entry pages), K = 128 dims in eight k = 16 MMAs of
// N = 256.  The key pages are row-major in HBM, so a tensor-map TMA copy
// (128-byte swizzle) writes each page as the K-major A operand; the 32-query
// block is the K-major B operand, written once per CTA.  C goes to one of two
// 256-column tensor-memory accumulators, so the epilogue of a tile (ReLU,
// weighted head sum, causal mask, coalesced score stores, optional 8-entry
// block maxima) overlaps the MMAs of the next.
//
// Roles: warp 0 streams the key tiles (page ids read 32 at a time, three
// 32 KB stages), warp 1 allocates tensor memory and issues the MMAs, warps
// 2..17 are the epilogue (warp w reads lane quarter w % 4 and queries
// 8 * ((w - 2) / 4) .. +7 of the block).
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tma.cuh"

namespace csa2 {
namespace {

constexpr int kQB = 32;                     // query tokens per CTA
constexpr int kGHi = 8;                     // indexer heads
constexpr int kGDi = 128;                   // indexer key width (bf16)
constexpr int kGN = kQB * kGHi;             // MMA N = 256
constexpr int kGTile = 128;                 // entries per tile
constexpr int kGStages = 3;
constexpr int kGTileBytes = kGTile * kGDi * 2;   // 32 KB
constexpr int kGEpiWarps = 16;
constexpr int kGThreads = (2 + kGEpiWarps) * 32;
constexpr uint32_t kGTmemCols = 2 * kGN;    // two accumulators

struct GemmSmem {
  unsigned char ring[kGStages][kGTileBytes];   // 128-byte-swizzled K-major tiles (1024-aligned)
  uint16_t q[kGN * kGDi];                      // B operand, no swizzle: (n/8)*2048 + (d/8)*128 + (n%8)*16 + (d%8)*2
  float w[kGN];                                // head weights of the block's queries
  int nv[kQB];                                 // visible entries of each query
  uint64_t full[kGStages], empty[kGStages], acc_full[2], acc_empty[2];
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ bool role_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort) return false;
  }
  *abort = 1;
  return false;
}

__global__ void __launch_bounds__(kGThreads, 1)
k_index_scores_gemm(IndexerArgs a, const __grid_constant__ CUtensorMap kmap, int tiles_per_cta,
                    float* __restrict__ scores, int64_t stride, float* __restrict__ blockmax, int64_t bm_stride,
                    uint32_t* status) {
  extern __shared__ unsigned char smem_raw[];
  pdl_trigger();
  pdl_wait();
  const uint32_t pad = (1024u - (tc::smem_addr(smem_raw) & 1023u)) & 1023u;
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(smem_raw + pad);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z;
  const int i0 = blockIdx.y * kQB;                 // first query row of the block
  const int nq = min(kQB, a.Tq - i0);
  const int64_t row0 = (int64_t)b * a.Tq + i0;
  const int n_ent = min(a.n_entries[b], a.max_entries);

  // ---- set-up: visible counts, the query block (B operand) and its weights
  if (tid < kQB) sm.nv[tid] = tid < nq ? n_visible(n_ent, a.q_pos[row0 + tid]) : 0;
  for (int u = tid; u < kGN * (kGDi / 8); u += kGThreads) {
    const int n = u >> 4, c8 = u & 15;             // n = query * 8 + head
    const int qq = n >> 3;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (qq < nq) v = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) +
                                                          ((row0 + qq) * kGHi + (n & 7)) * kGDi + c8 * 8));
    *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(sm.q) + (n >> 3) * 2048 + c8 * 128 + (n & 7) * 16) = v;
  }
  for (int n = tid; n < kGN; n += kGThreads) sm.w[n] = (n >> 3) < nq ? a.w[(row0 + (n >> 3)) * kGHi + (n & 7)] : 0.f;
  if (tid == 0) {
    for (int s = 0; s < kGStages; ++s) {
      tc::mbar_init(&sm.full[s], 1);
      tc::mbar_init(&sm.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sm.acc_full[i], 1);
      tc::mbar_init(&sm.acc_empty[i], kGEpiWarps);
    }
    sm.abort = 0;
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(&sm.tmem, kGTmemCols);
  tc::fence_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = sm.tmem;
  volatile int* abort = &sm.abort;

  // the CTA's tiles: [t0, t1) of the block's visible range
  int max_nv = 0;
  for (int i = 0; i < kQB; ++i) max_nv = max(max_nv, sm.nv[i]);
  const int n_tiles = (max_nv + kGTile - 1) / kGTile;
  const int t0 = blockIdx.x * tiles_per_cta, t1 = min(n_tiles, t0 + tiles_per_cta);
  const int my = max(0, t1 - t0);

  if (warp == 0) {
    // ================= producer: two pages per tile, page ids 32 at a time =================
    const int64_t pt_row = (int64_t)b * a.max_pages;
    const int p_lo = 2 * t0, p_hi = min(2 * t1, (max_nv + kPage - 1) / kPage);
    auto page_id = [&](int lp) -> int {
      return (lp < p_hi && lp < a.max_pages) ? __ldg(a.page_table + pt_row + lp) : -1;
    };
    int cur = page_id(p_lo + lane), nxt = page_id(p_lo + 32 + lane);
    int issued = 0;
    for (int i = 0; i < my; ++i) {
      const int st = i % kGStages;
      int pg[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int k = 2 * i + h;                       // page index relative to p_lo
        if (k > 0 && (k & 31) == 0) {
          cur = nxt;
          nxt = page_id(p_lo + k + 32 + lane);
        }
        pg[h] = __shfl_sync(0xffffffffu, cur, k & 31);
      }
      bool ok = true;
      if (lane == 0) {
        if (i >= kGStages && !role_wait(&sm.empty[st], ((i / kGStages) - 1) & 1, abort)) {
          ok = false;
        } else {
          uint32_t bytes = 0;
          for (int h = 0; h < 2; ++h) {
            const int lp = 2 * (t0 + i) + h;
            const bool in_range = lp < p_hi;
            const bool good = in_range && pg[h] >= 0 && pg[h] < a.n_pages;
            if (in_range && !good) raise_status(status, CSA2_STATUS_BAD_PAGE);
            pg[h] = good ? pg[h] : -1;
            if (good) bytes += 2 * 8192;
          }
          tc::mbar_arrive_expect_tx(&sm.full[st], bytes);
          for (int h = 0; h < 2; ++h)
            if (pg[h] >= 0)
              for (int kb = 0; kb < 2; ++kb)   // dims 64*kb .. +63 of the page's 64 rows
                tma::load_2d(sm.ring[st] + kb * 16384 + h * 8192, &kmap, 64 * kb, pg[h] * kPage, &sm.full[st]);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      issued = i + 1;
    }
    if (lane == 0)   // every issued copy lands before the CTA can exit
      for (int i = max(0, issued - kGStages); i < issued; ++i)
        for (uint32_t k = 0; k < (1u << 22); ++k)
          if (tc::mbar_try_wait(&sm.full[i % kGStages], (i / kGStages) & 1)) break;
  } else if (warp == 1) {
    // ================= MMA issue =================
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_f16(128, kGN, 1, 0, 0);   // bf16, K-major A and B
      const uint64_t dq = tc::smem_desc(tc::smem_addr(sm.q), 128, 2048);
      for (int i = 0; i < my; ++i) {
        const int st = i % kGStages, buf = i & 1;
        if (!role_wait(&sm.full[st], (i / kGStages) & 1, abort)) break;
        if (i >= 2 && !role_wait(&sm.acc_empty[buf], ((i >> 1) - 1) & 1, abort)) break;
        tc::tc_fence_after();
        const uint32_t a0 = tc::smem_addr(sm.ring[st]);
#pragma unroll
        for (int ks = 0; ks < kGDi / 16; ++ks) {
          const uint64_t ad = tc::smem_desc(a0 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024) | ((uint64_t)2 << 61);
          tc::mma_f16(tm + buf * kGN, ad, dq + (uint64_t)(ks * 16), idesc, ks > 0);
        }
        tc::mma_commit(&sm.empty[st]);
        tc::mma_commit(&sm.acc_full[buf]);
      }
    }
    __syncwarp();
  } else {
    // ================= epilogue =================
    const int ew = warp - 2;
    const int qtr = warp & 3;                 // tensor-memory lane quarter of this warp
    const int qg = ew >> 2;                   // queries 8*qg .. 8*qg+7
    for (int i = 0; i < my; ++i) {
      const int buf = i & 1;
      if (!__all_sync(0xffffffffu, role_wait(&sm.acc_full[buf], (i >> 1) & 1, abort))) break;
      tc::tc_fence_after();
      const int e = (t0 + i) * kGTile + 32 * qtr + lane;
#pragma unroll
      for (int c = 0; c < 4; ++c) {           // two queries per 16 columns
        float v[16];
        tc::tmem_ld16(tm + buf * kGN + 64 * qg + 16 * c + ((uint32_t)(32 * qtr) << 16), v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int qq = 8 * qg + 2 * c + u;
          const float4 w0 = *reinterpret_cast<const float4*>(&sm.w[qq * 8]);
          const float4 w1 = *reinterpret_cast<const float4*>(&sm.w[qq * 8 + 4]);
          const float* x = v + 8 * u;
          float s = w0.x * fmaxf(x[0], 0.f);
          s = fmaf(w0.y, fmaxf(x[1], 0.f), s);
          s = fmaf(w0.z, fmaxf(x[2], 0.f), s);
          s = fmaf(w0.w, fmaxf(x[3], 0.f), s);
          s = fmaf(w1.x, fmaxf(x[4], 0.f), s);
          s = fmaf(w1.y, fmaxf(x[5], 0.f), s);
          s = fmaf(w1.z, fmaxf(x[6], 0.f), s);
          s = fmaf(w1.w, fmaxf(x[7], 0.f), s);
          const int nvq = sm.nv[qq];
          const bool vis = e < nvq;   // (a bad page raised CSA2_STATUS_BAD_PAGE; its scores are not meaningful)
          if (vis) scores[(row0 + qq) * stride + e] = s;
          if (blockmax) {   // maxima of 8 consecutive entries = 8 consecutive lanes
            float m = vis ? s : -INFINITY;
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            if ((lane & 7) == 0 && e < nvq && qq < nq) blockmax[(row0 + qq) * bm_stride + e / 8] = m;
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.acc_empty[buf]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tm, kGTmemCols);
  if (tid == 0 && *abort) raise_status(status, CSA2_STATUS_TIMEOUT);
}

}  // namespace

bool index_scores_gemm_supported(const IndexerArgs& a) {
  return a.dtype == CSA2_BF16 && a.Hi == kGHi && a.Di == kGDi && a.Tq >= kQB && a.n_pages > 0 &&
         a.n_pages * kPage < ((int64_t)1 << 31) && tensor_map_encoder() != nullptr;
}

cudaError_t launch_index_scores_gemm(const IndexerArgs& a, float* scores, int64_t stride, float* blockmax,
                                     int64_t bm_stride, int max_entries, cudaStream_t s) {
  // the key pool as a 2-D tensor: rows = n_pages * 64 entries of 128 bf16 (256 B)
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)kGDi, (cuuint64_t)a.n_pages * kPage};
  const cuuint64_t strides[1] = {(cuuint64_t)kGDi * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kPage};
  const cuuint32_t estr[2] = {1, 1};
  if (tensor_map_encoder()(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.k), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int q_blocks = (a.Tq + kQB - 1) / kQB;
  const int max_tiles = (max_entries + kGTile - 1) / kGTile;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // split the entries only as far as it takes to fill the SMs once
  const int64_t blocks = (int64_t)q_blocks * a.B;
  int splits = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, sms / std::max<int64_t>(1, blocks)));
  const int tiles_per_cta = std::max(1, (max_tiles + splits - 1) / splits);
  splits = std::max(1, (max_tiles + tiles_per_cta - 1) / tiles_per_cta);
  const size_t smem = sizeof(GemmSmem) + 1024;
  e = cudaFuncSetAttribute(k_index_scores_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(splits, q_blocks, a.B);
  return launch_step(k_index_scores_gemm, grid, dim3(kGThreads), smem, s, a, map, tiles_per_cta, scores, stride,
                     blockmax, bm_stride, status_word());
}

}  // namespace csa2
