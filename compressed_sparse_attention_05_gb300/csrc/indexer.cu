// Sparse-indexer scoring: s_j = sum_h w_h * ReLU(q_h . k_j) for every
// causally visible compressed entry (Full) or for the pooled positions only
// (Reindex).  "DeepSeek-V4.1 架构解析" §02: the indexer scores every visible
// entry and keeps a Top-512; Reindex layers rescore the shared indexer keys
// with their own query, inside the 2,048 x 8 pool.  Score form: reading R6.
//
// Decode is bound by HBM: every visible key (Di bf16) is read exactly once.
// The bf16 path runs on tensor cores (m16n8k16, fp32 accumulate), entries as
// the M dimension and heads as N, so the ALU stays far below the 8 FLOP/B the
// scan needs.  Each thread loads its A fragments straight from the paged key
// rows with 16-byte loads: the head dimension is visited in a permuted order
// (the same permutation for q and k, so the dot products are unchanged) that
// makes every warp load instruction touch 16 full 32-byte sectors.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace csa2 {

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Visible positions (0..8) of pooled block `blk` when nv entries are visible.
__device__ __forceinline__ int visible_in_block(int nv, int32_t blk) {
  const int64_t v = (int64_t)nv - 8LL * blk;
  return v <= 0 ? 0 : (v >= 8 ? 8 : (int)v);
}

constexpr int kIdxWarps = 8;          // warps per CTA
constexpr int kIdxTilesPerWarp = 4;   // 16-entry tiles per warp
constexpr int kIdxChunk = kIdxWarps * kIdxTilesPerWarp * 16;  // entries per CTA

// Scores of one 16-entry tile for one query from A fragments already in
// registers.  Returns (via out_g, out_g8) the scores of entries g and g+8.
template <int NCH, int NT>
__device__ __forceinline__ void tile_scores(const uint4 (&ka)[NCH], const uint4 (&kb)[NCH],
                                            const uint4 (&qf)[NT][NCH], const float (&wv)[NT][2],
                                            float& out_g, float& out_g8) {
  float acc_g = 0.f, acc_g8 = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      mma_bf16_16816(d, ka[c].x, kb[c].x, ka[c].y, kb[c].y, qf[nt][c].x, qf[nt][c].y);
      mma_bf16_16816(d, ka[c].z, kb[c].z, ka[c].w, kb[c].w, qf[nt][c].z, qf[nt][c].w);
    }
    acc_g += wv[nt][0] * fmaxf(d[0], 0.f) + wv[nt][1] * fmaxf(d[1], 0.f);
    acc_g8 += wv[nt][0] * fmaxf(d[2], 0.f) + wv[nt][1] * fmaxf(d[3], 0.f);
  }
  acc_g += __shfl_xor_sync(0xffffffffu, acc_g, 1);
  acc_g += __shfl_xor_sync(0xffffffffu, acc_g, 2);
  acc_g8 += __shfl_xor_sync(0xffffffffu, acc_g8, 1);
  acc_g8 += __shfl_xor_sync(0xffffffffu, acc_g8, 2);
  out_g = acc_g;
  out_g8 = acc_g8;
}

// Query fragments of head group nt for the thread (g, t): heads 8nt + g,
// dims 32c + 8t .. +7 (zero for heads >= Hi).
template <int NCH, int NT>
__device__ __forceinline__ void load_query(const uint16_t* __restrict__ q, const float* __restrict__ w,
                                           int Hi, int Di, int lane, uint4 (&qf)[NT][NCH],
                                           float (&wv)[NT][2]) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = nt * 8 + g;
#pragma unroll
    for (int c = 0; c < NCH; ++c)
      qf[nt][c] = h < Hi ? *reinterpret_cast<const uint4*>(q + (int64_t)h * Di + 32 * c + 8 * t)
                         : make_uint4(0, 0, 0, 0);
    const int h0 = nt * 8 + 2 * t;
    wv[nt][0] = h0 < Hi ? w[h0] : 0.f;
    wv[nt][1] = h0 + 1 < Hi ? w[h0 + 1] : 0.f;
  }
}

// Order-preserving key of an fp32 score (-0 folded into +0); its top 11 bits
// index the per-row histogram the Top-K kernel starts from.
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) == 0) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
constexpr int kHistBins = 2048;
constexpr int kHistMaxQG = 8;   // query rows per CTA when a histogram is built

// Full mode.  grid = (entry chunks, query groups, B); a CTA scores one chunk
// of kIdxChunk entries of sequence b against QG consecutive query tokens.
// Each warp walks its 16-entry tiles with the next tile's key fragments in
// flight while the current one is on the tensor cores.
template <int NCH, int NT>
__global__ void __launch_bounds__(kIdxWarps * 32)
k_index_scores_mma(IndexerArgs a, int QG, float* __restrict__ scores, int64_t stride,
                   float* __restrict__ blockmax, int64_t bm_stride, uint32_t* __restrict__ hist,
                   uint32_t* status) {
  extern __shared__ uint32_t shist[];   // [QG][kHistBins] when hist != nullptr
  const int b = blockIdx.z;
  const int i0 = blockIdx.y * QG;
  const int i1 = min(a.Tq, i0 + QG);
  const int n_ent = min(a.n_entries[b], a.max_entries);
  int max_vis = 0;
  for (int i = i0; i < i1; ++i) max_vis = max(max_vis, n_visible(n_ent, a.q_pos[(int64_t)b * a.Tq + i]));
  const int chunk0 = blockIdx.x * kIdxChunk;
  if (chunk0 >= max_vis) return;
  if (hist) {
    for (int i = threadIdx.x; i < (i1 - i0) * kHistBins; i += blockDim.x) shist[i] = 0;
    __syncthreads();
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const uint16_t* kbase = reinterpret_cast<const uint16_t*>(a.k);
  const int tile0 = chunk0 + warp * kIdxTilesPerWarp * 16;
  uint4 ka[2][NCH], kb[2][NCH];
  auto load_tile = [&](int e0, uint4 (&ra)[NCH], uint4 (&rb)[NCH]) -> bool {
    const int64_t slot0 = entry_slot(a.page_table, a.max_pages, a.n_pages, b, e0, status);
    if (slot0 < 0) return false;
    const uint16_t* rg = kbase + (slot0 + g) * a.Di + 8 * t;
    const uint16_t* rg8 = kbase + (slot0 + g + 8) * a.Di + 8 * t;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      ra[c] = __ldg(reinterpret_cast<const uint4*>(rg + 32 * c));
      rb[c] = __ldg(reinterpret_cast<const uint4*>(rg8 + 32 * c));
    }
    return true;
  };
  bool ok_cur = tile0 < max_vis && load_tile(tile0, ka[0], kb[0]);
#pragma unroll
  for (int tt = 0; tt < kIdxTilesPerWarp; ++tt) {
    const int cur = tt & 1;
    const int e0 = tile0 + tt * 16;
    if (e0 >= max_vis) break;
    bool ok_next = false;
    if (tt + 1 < kIdxTilesPerWarp && e0 + 16 < max_vis) ok_next = load_tile(e0 + 16, ka[cur ^ 1], kb[cur ^ 1]);
    if (ok_cur) {
      for (int i = i0; i < i1; ++i) {
        const int64_t row = (int64_t)b * a.Tq + i;
        const int nv = n_visible(n_ent, a.q_pos[row]);
        if (e0 >= nv) continue;
        uint4 qf[NT][NCH];
        float wv[NT][2];
        load_query<NCH, NT>(reinterpret_cast<const uint16_t*>(a.q) + row * a.Hi * a.Di, a.w + row * a.Hi,
                            a.Hi, a.Di, lane, qf, wv);
        float sg, sg8;
        tile_scores<NCH, NT>(ka[cur], kb[cur], qf, wv, sg, sg8);
        const bool vg = e0 + g < nv, vg8 = e0 + g + 8 < nv;
        if (t == 0 && vg) scores[row * stride + e0 + g] = sg;
        if (t == 1 && vg8) scores[row * stride + e0 + g + 8] = sg8;
        if (hist) {
          // lanes t == 0 carry entry g, lanes t == 1 entry g + 8
          const bool has = (t == 0 && vg) || (t == 1 && vg8);
          if (has) atomicAdd(&shist[(i - i0) * kHistBins + (score_key(t == 0 ? sg : sg8) >> 21)], 1u);
        }
        if (blockmax) {
          float m0 = vg ? sg : -INFINITY, m1 = vg8 ? sg8 : -INFINITY;
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
            m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
          }
          if (lane == 0) blockmax[row * bm_stride + e0 / 8] = m0;
          if (lane == 1 && e0 + 8 < nv) blockmax[row * bm_stride + e0 / 8 + 1] = m1;
        }
      }
    }
    ok_cur = ok_next;
  }
  if (hist) {
    __syncthreads();
    for (int i = threadIdx.x; i < (i1 - i0) * kHistBins; i += blockDim.x) {
      const uint32_t c = shist[i];
      if (c) atomicAdd(&hist[((int64_t)b * a.Tq + i0 + i / kHistBins) * kHistBins + (i % kHistBins)], c);
    }
  }
}

// ---- page-streaming scan (Full mode, bf16 keys, Di = 128) ---------------------------
// One lane of a producer warp streams whole key pages (64 entries x 256 B =
// 16 KB, contiguous in the pool) into a ring of shared-memory stages with
// cp.async.bulk; each stage completes on an mbarrier with its byte count.
// Four consumer warps take 16 entries each per page and run the same tensor-
// core scoring as above from shared memory, then release the stage.  Many
// pages per SM stay in flight, which is what an HBM-bound scan needs.
// Every wait is bounded; on a timeout the CTA raises CSA2_STATUS_TIMEOUT,
// drains the copies it issued and exits.
constexpr int kScanStages = 3;   // 4 CTAs per SM: the scoring warps, not the copies, set the pace
constexpr int kScanConsumers = 4;
constexpr int kScanThreads = (kScanConsumers + 1) * 32;
constexpr int kPageBytes = kPage * 128 * 2;

struct ScanShared {
  uint64_t full[kScanStages];
  uint64_t empty[kScanStages];
  int valid[kScanStages];
  int abort;
};

// Waits for `parity` on `bar` while no other role has aborted.
__device__ __forceinline__ bool scan_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (uint32_t i = 0; i < (1u << 21); ++i) {   // <= 2^21 suspensions of <= 1 us
    if (tc::mbar_try_wait_sleep(bar, parity, 1000)) return true;
    if ((i & 255) == 255 && *abort) return false;
  }
  *abort = 1;
  return false;
}

// Pages of a single-query row b: ceil(visible / 64).
__device__ __forceinline__ int row_pages(const IndexerArgs& a, int b) {
  const int nv = n_visible(min(a.n_entries[b], a.max_entries), a.q_pos[(int64_t)b * a.Tq]);
  return (nv + kPage - 1) / kPage;
}

// Balanced single-wave partition when every row has one query (Tq == 1):
// with P pages in all and S CTA slots, every row gets ceil(pages_b / ppc)
// CTAs of ppc = ceil(P / (S - B)) pages, so the grid never exceeds S and no
// CTA spans two rows.  Each CTA derives its (row, page range) itself; every
// warp computes it with its lanes on 32 rows at a time (warp sums and a
// prefix scan), so the set-up costs one round of loads, not one per row.
__device__ __forceinline__ bool flat_assign(const IndexerArgs& a, int slots, int& b_out, int& p0, int& p1) {
  const int lane = threadIdx.x & 31;
  int64_t total = 0;
  for (int base = 0; base < a.B; base += 32) {
    const int b = base + lane;
    int pb = b < a.B ? row_pages(a, b) : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pb += __shfl_xor_sync(0xffffffffu, pb, o);
    total += pb;
  }
  const int denom = max(1, slots - a.B);
  int64_t ppc64 = (total + denom - 1) / denom;
  const int ppc = ppc64 < 1 ? 1 : (int)ppc64;
  int c = blockIdx.x;
  for (int base = 0; base < a.B; base += 32) {
    const int b = base + lane;
    const int pb = b < a.B ? row_pages(a, b) : 0;
    const int nc = (pb + ppc - 1) / ppc;
    int incl = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = incl - nc;
    const int tot = __shfl_sync(0xffffffffu, incl, 31);
    if (c < tot) {
      const int owner = __ffs(__ballot_sync(0xffffffffu, c >= excl && c < incl)) - 1;
      b_out = base + owner;
      p0 = (c - __shfl_sync(0xffffffffu, excl, owner)) * ppc;
      p1 = min(__shfl_sync(0xffffffffu, pb, owner), p0 + ppc);
      return p0 < p1;
    }
    c -= tot;
  }
  return false;
}

template <int NT>
__global__ void __launch_bounds__(kScanThreads)
k_index_scan_pages(IndexerArgs a, int QG, int pages_per_cta, int flat_slots, float* __restrict__ scores,
                   int64_t stride, float* __restrict__ blockmax, int64_t bm_stride, uint32_t* __restrict__ hist,
                   uint32_t* __restrict__ bm_hist, uint32_t* status) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ ScanShared ss;
  pdl_trigger();
  unsigned char* ring = smem_raw;                                   // kScanStages pages
  uint32_t* shist = reinterpret_cast<uint32_t*>(smem_raw + kScanStages * kPageBytes);
  // block-maxima histogram of the (one) query row, after the score histogram
  uint32_t* sbm = shist + (hist ? kHistBins : 0);
  int b, p0, p1, i0, i1;
  if (flat_slots > 0) {          // one query per row
    if (!flat_assign(a, flat_slots, b, p0, p1)) return;
    i0 = 0;
    i1 = 1;
  } else {
    b = blockIdx.z;
    i0 = blockIdx.y * QG;
    i1 = min(a.Tq, i0 + QG);
    const int n_ent_b = min(a.n_entries[b], a.max_entries);
    int max_vis = 0;
    for (int i = i0; i < i1; ++i) max_vis = max(max_vis, n_visible(n_ent_b, a.q_pos[(int64_t)b * a.Tq + i]));
    p0 = blockIdx.x * pages_per_cta;
    p1 = min((max_vis + kPage - 1) / kPage, p0 + pages_per_cta);
    if (p0 >= p1) return;
  }
  const int n_ent = min(a.n_entries[b], a.max_entries);
  const int n_pages = p1 - p0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kScanStages; ++s) {
      tc::mbar_init(&ss.full[s], 1);
      tc::mbar_init(&ss.empty[s], kScanConsumers);
    }
    ss.abort = 0;
    tc::mbar_fence_init();
  }
  if (hist)
    for (int i = threadIdx.x; i < (i1 - i0) * kHistBins; i += blockDim.x) shist[i] = 0;
  if (bm_hist)   // one query row per CTA on this path (checked by the launcher)
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) sbm[i] = 0;
  __syncthreads();
  // The set-up above reads inputs only (counts, positions); the keys (new entries
  // of a compressing step), the scores and the histograms belong to earlier kernels.
  pdl_wait();
  volatile int* abort = &ss.abort;

  if (warp == kScanConsumers) {
    // ---- producer warp: the page ids come 32 at a time, one batch ahead, so
    // that no page copy waits for its page-table read; lane 0 issues the copies
    const int64_t pt_row = (int64_t)b * a.max_pages;
    auto page_id = [&](int lp) -> int {
      return (lp < p1 && lp < a.max_pages) ? __ldg(a.page_table + pt_row + lp) : -1;
    };
    int cur = page_id(p0 + lane), nxt = page_id(p0 + 32 + lane);
    int issued = 0;
    const uint64_t stream_policy = tc::l2_evict_first_policy();   // keys are read once
    for (int i = 0; i < n_pages; ++i) {
      if (i > 0 && (i & 31) == 0) {
        cur = nxt;
        nxt = page_id(p0 + i + 32 + lane);
      }
      const int pg = __shfl_sync(0xffffffffu, cur, i & 31);
      const int st = i % kScanStages;
      bool ok = true;
      if (lane == 0) {
        if (i >= kScanStages && !scan_wait(&ss.empty[st], ((i / kScanStages) - 1) & 1, abort)) {
          ok = false;
        } else if (pg < 0 || pg >= a.n_pages) {
          raise_status(status, CSA2_STATUS_BAD_PAGE);
          ss.valid[st] = 0;
          tc::mbar_arrive(&ss.full[st]);
        } else {
          ss.valid[st] = 1;
          tc::mbar_arrive_expect_tx(&ss.full[st], kPageBytes);
          tc::bulk_g2s_hint(ring + st * kPageBytes,
                            reinterpret_cast<const unsigned char*>(a.k) + (int64_t)pg * kPageBytes, kPageBytes,
                            &ss.full[st], stream_policy);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      issued = i + 1;
    }
    // drain: every issued copy must have landed before the CTA exits
    if (lane == 0)
      for (int i = max(0, issued - kScanStages); i < issued; ++i) {
        const int st = i % kScanStages;
        for (uint32_t k = 0; k < (1u << 22); ++k)
          if (tc::mbar_try_wait(&ss.full[st], (i / kScanStages) & 1)) break;
      }
  } else {
    // ---- consumers: warp w owns entries 16w .. 16w+15 of every page
    const int g = lane >> 2, t = lane & 3;
    uint4 qf1[NT][4];      // the query of a single-query CTA, loaded once
    float wv1[NT][2];
    if (i1 - i0 == 1) {
      const int64_t row = (int64_t)b * a.Tq + i0;
      load_query<4, NT>(reinterpret_cast<const uint16_t*>(a.q) + row * a.Hi * a.Di, a.w + row * a.Hi, a.Hi, a.Di,
                        lane, qf1, wv1);
    }
    for (int i = 0; i < n_pages; ++i) {
      const int st = i % kScanStages;
      // warp-uniform exit: the warp's shuffles below need every lane
      if (!__all_sync(0xffffffffu, scan_wait(&ss.full[st], (i / kScanStages) & 1, abort))) break;
      if (ss.valid[st]) {
        const unsigned char* pg = ring + st * kPageBytes + (warp * 16) * 256 + 16 * t;
        uint4 ka[4], kb[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          ka[c] = *reinterpret_cast<const uint4*>(pg + g * 256 + 64 * c);
          kb[c] = *reinterpret_cast<const uint4*>(pg + (g + 8) * 256 + 64 * c);
        }
        const int e0 = (p0 + i) * kPage + warp * 16;
        for (int qi = i0; qi < i1; ++qi) {
          const int64_t row = (int64_t)b * a.Tq + qi;
          const int nv = n_visible(n_ent, a.q_pos[row]);
          if (e0 >= nv) continue;
          float sg, sg8;
          if (i1 - i0 == 1) {
            tile_scores<4, NT>(ka, kb, qf1, wv1, sg, sg8);
          } else {
            uint4 qf[NT][4];
            float wv[NT][2];
            load_query<4, NT>(reinterpret_cast<const uint16_t*>(a.q) + row * a.Hi * a.Di, a.w + row * a.Hi, a.Hi,
                              a.Di, lane, qf, wv);
            tile_scores<4, NT>(ka, kb, qf, wv, sg, sg8);
          }
          const bool vg = e0 + g < nv, vg8 = e0 + g + 8 < nv;
          if (t == 0 && vg) scores[row * stride + e0 + g] = sg;
          if (t == 1 && vg8) scores[row * stride + e0 + g + 8] = sg8;
          if (hist) {
            const bool has = (t == 0 && vg) || (t == 1 && vg8);
            if (has) atomicAdd(&shist[(qi - i0) * kHistBins + (score_key(t == 0 ? sg : sg8) >> 21)], 1u);
          }
          if (blockmax) {
            float m0 = vg ? sg : -INFINITY, m1 = vg8 ? sg8 : -INFINITY;
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
              m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
              m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
            }
            if (lane == 0) blockmax[row * bm_stride + e0 / 8] = m0;
            if (lane == 1 && e0 + 8 < nv) blockmax[row * bm_stride + e0 / 8 + 1] = m1;
            if (bm_hist) {   // the blocks with a visible entry, as for the scores
              if (lane == 0 && e0 < nv) atomicAdd(&sbm[score_key(m0) >> 21], 1u);
              if (lane == 1 && e0 + 8 < nv) atomicAdd(&sbm[score_key(m1) >> 21], 1u);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&ss.empty[st]);
    }
  }
  __syncthreads();
  if (*abort && threadIdx.x == 0) raise_status(status, CSA2_STATUS_TIMEOUT);
  if (hist) {
    for (int i = threadIdx.x; i < (i1 - i0) * kHistBins; i += blockDim.x) {
      const uint32_t c = shist[i];
      if (c) atomicAdd(&hist[((int64_t)b * a.Tq + i0 + i / kHistBins) * kHistBins + (i % kHistBins)], c);
    }
  }
  if (bm_hist) {
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) {
      const uint32_t c = sbm[i];
      if (c) atomicAdd(&bm_hist[((int64_t)b * a.Tq + i0) * kHistBins + i], c);
    }
  }
}

// Zeroes a histogram buffer as a step kernel (a memset node would end the chain of
// programmatic launches: the scan's prologue could not overlap it).
__global__ void k_zero_u32x4(uint4* __restrict__ p, int64_t n4) {
  pdl_trigger();
  pdl_wait();   // an earlier kernel may still read the buffer
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x)
    p[i] = make_uint4(0, 0, 0, 0);
}

cudaError_t launch_zero_u32(uint32_t* p, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if ((reinterpret_cast<uintptr_t>(p) & 15) != 0 || n % 4 != 0) return cudaMemsetAsync(p, 0, (size_t)n * 4, s);
  const int64_t n4 = n / 4;
  const int64_t blocks = std::min<int64_t>((n4 + 255) / 256, 1024);
  return launch_step(k_zero_u32x4, dim3((unsigned)blocks), dim3(256), 0, s, reinterpret_cast<uint4*>(p), n4);
}

static int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  }
  return n;
}

template <int NT>
static cudaError_t launch_scan_pages(const IndexerArgs& a, float* scores, int64_t stride, float* blockmax,
                                     int64_t bm_stride, int max_entries, uint32_t* hist, uint32_t* bm_hist,
                                     cudaStream_t s) {
  const int QG = a.Tq >= kHistMaxQG ? kHistMaxQG : a.Tq;
  const int q_groups = (a.Tq + QG - 1) / QG;
  const int max_pages_vis = (max_entries + kPage - 1) / kPage;
  // about two CTAs per SM over the whole grid
  const int64_t want = 2LL * num_sms();
  int per_seq = (int)((want + (int64_t)a.B * q_groups - 1) / ((int64_t)a.B * q_groups));
  per_seq = per_seq < 1 ? 1 : per_seq;
  int ppc = (max_pages_vis + per_seq - 1) / per_seq;
  ppc = ppc < 1 ? 1 : ppc;
  if (a.Tq != 1 || !blockmax) bm_hist = nullptr;   // one query row per CTA only
  const size_t smem = (size_t)kScanStages * kPageBytes + (hist ? (size_t)QG * kHistBins * 4 : 0) +
                      (bm_hist ? (size_t)kHistBins * 4 : 0);
  cudaError_t e = cudaFuncSetAttribute(k_index_scan_pages<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (a.Tq == 1) {
    // CTA slots resident at once (shared memory bounds the CTAs per SM)
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_index_scan_pages<NT>, kScanThreads, smem);
    if (e != cudaSuccess || per_sm < 1) per_sm = 1;
    const int slots = per_sm * num_sms();
    const int grid = slots > a.B ? slots : a.B + 1;
    return launch_step(k_index_scan_pages<NT>, dim3(grid), dim3(kScanThreads), smem, s, a, 1, 0, grid, scores, stride,
                       blockmax, bm_stride, hist, bm_hist, status_word());
  }
  dim3 grid((max_pages_vis + ppc - 1) / ppc, q_groups, a.B);
  return launch_step(k_index_scan_pages<NT>, grid, dim3(kScanThreads), smem, s, a, QG, ppc, 0, scores, stride,
                     blockmax, bm_stride, hist, bm_hist, status_word());
}

// Histogram of already-written scores (the generic scoring path).
__global__ void k_score_hist(const float* __restrict__ scores, int64_t stride, IndexerArgs a,
                             uint32_t* __restrict__ hist) {
  const int64_t row = blockIdx.y;
  const int b = (int)(row / a.Tq);
  const int nv = n_visible(min(a.n_entries[b], a.max_entries), a.q_pos[row]);
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const bool has = j < nv;
  const uint32_t bin = has ? score_key(scores[row * stride + j]) >> 21 : 0xFFFFFFFFu;
  const uint32_t peers = __match_any_sync(0xffffffffu, bin);
  if (has && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[row * kHistBins + bin], __popc(peers));
}

// Reindex.  grid = (pool-block pairs / kIdxWarps, rows): warp w scores the
// two pooled blocks 2p, 2p+1 (16 positions = one tile; rows g -> block 2p,
// rows g+8 -> block 2p+1) into compact columns 8*slot + e.
template <int NCH, int NT>
__global__ void __launch_bounds__(kIdxWarps * 32)
k_index_scores_pool_mma(IndexerArgs a, const int32_t* __restrict__ pool,
                        const int32_t* __restrict__ pool_cnt, int n_pool,
                        float* __restrict__ scores, int64_t stride, int32_t* __restrict__ n_valid,
                        uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int64_t row = blockIdx.y;
  const int b = (int)(row / a.Tq);
  const int nv = n_visible(min(a.n_entries[b], a.max_entries), a.q_pos[row]);
  const int pc = min(max(pool_cnt[row], 0), n_pool);
  const int32_t* prow = pool + row * n_pool;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  if (blockIdx.x == 0 && warp == 0) {
    int cnt = 0;
    for (int p = lane; p < pc; p += 32) cnt += visible_in_block(nv, prow[p]);
    cnt = (int)warp_sum((float)cnt);
    if (lane == 0) n_valid[row] = cnt;
  }
  const int pair = blockIdx.x * kIdxWarps + warp;
  const int p0 = 2 * pair;
  if (p0 >= pc) return;
  const int64_t blk0 = prow[p0];
  const int64_t blk1 = p0 + 1 < pc ? prow[p0 + 1] : -1;
  const int64_t e_g = 8 * blk0 + g;
  const int64_t e_g8 = blk1 >= 0 ? 8 * blk1 + g : -1;
  const bool vg = blk0 >= 0 && e_g < nv;
  const bool vg8 = e_g8 >= 0 && e_g8 < nv;
  if ((blk0 < 0 || 8 * blk0 >= nv) && lane == 0) raise_status(status, CSA2_STATUS_BAD_INDEX);
  const int64_t sg_slot = vg ? entry_slot(a.page_table, a.max_pages, a.n_pages, b, (int)e_g, status) : -1;
  const int64_t sg8_slot = vg8 ? entry_slot(a.page_table, a.max_pages, a.n_pages, b, (int)e_g8, status) : -1;
  const uint16_t* kbase = reinterpret_cast<const uint16_t*>(a.k);
  uint4 ka[NCH], kb[NCH];
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    ka[c] = sg_slot >= 0 ? __ldg(reinterpret_cast<const uint4*>(kbase + sg_slot * a.Di + 8 * t + 32 * c))
                         : make_uint4(0, 0, 0, 0);
    kb[c] = sg8_slot >= 0 ? __ldg(reinterpret_cast<const uint4*>(kbase + sg8_slot * a.Di + 8 * t + 32 * c))
                          : make_uint4(0, 0, 0, 0);
  }
  uint4 qf[NT][NCH];
  float wv[NT][2];
  load_query<NCH, NT>(reinterpret_cast<const uint16_t*>(a.q) + row * a.Hi * a.Di, a.w + row * a.Hi, a.Hi,
                      a.Di, lane, qf, wv);
  float s0, s1;
  tile_scores<NCH, NT>(ka, kb, qf, wv, s0, s1);
  if (t == 0 && vg) scores[row * stride + 8 * p0 + g] = s0;
  if (t == 1 && vg8) scores[row * stride + 8 * (p0 + 1) + g] = s1;
}

// Reindex over many query tokens: the pooled positions' scores gathered from a
// row of scores of every visible entry (the tensor-core GEMM's output) into
// compact columns 8*slot + e of the same row, with the pool scorer's count of
// visible positions and its check of the pool.  One CTA per row; every value
// is read before any is written, so the pool's order does not matter.
constexpr int kCompactThreads = 1024;
constexpr int kCompactPer = 32;   // 8 x 4,096 pooled positions at most
__global__ void __launch_bounds__(kCompactThreads, 1)
k_pool_compact(IndexerArgs a, const int32_t* __restrict__ pool, const int32_t* __restrict__ pool_cnt, int n_pool,
               float* __restrict__ scores, int64_t stride, int32_t* __restrict__ n_valid, uint32_t* status) {
  __shared__ int s_cnt[kCompactThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const int b = (int)(row / a.Tq);
  const int nv = n_visible(min(a.n_entries[b], a.max_entries), a.q_pos[row]);
  const int pc = min(max(pool_cnt[row], 0), n_pool);
  const int32_t* prow = pool + row * n_pool;
  float* srow = scores + row * stride;
  const int tid = threadIdx.x;
  float v[kCompactPer];
  uint32_t keep = 0;   // bit k: value k is written back
  int cnt = 0;
#pragma unroll
  for (int k = 0; k < kCompactPer; ++k) {
    const int c = tid + kCompactThreads * k;
    v[k] = 0.f;
    if (c < 8 * pc) {
      const int32_t blk = prow[c >> 3];
      const int64_t e = 8LL * blk + (c & 7);
      if (blk >= 0 && e < nv) {
        v[k] = srow[e];
        keep |= 1u << k;
      }
      cnt += (c & 7) < visible_in_block(nv, blk) ? 1 : 0;
      if ((c & 7) == 0 && (blk < 0 || 8LL * blk >= nv)) raise_status(status, CSA2_STATUS_BAD_INDEX);
    }
  }
  cnt = (int)warp_sum((float)cnt);
  if ((tid & 31) == 0) s_cnt[tid >> 5] = cnt;
  __syncthreads();   // (also: every read of the row is done before the writes below)
  if (tid < 32) {
    int t = s_cnt[tid];
    t = (int)warp_sum((float)t);
    if (tid == 0) n_valid[row] = t;
  }
#pragma unroll
  for (int k = 0; k < kCompactPer; ++k)
    if ((keep >> k) & 1u) srow[tid + kCompactThreads * k] = v[k];
}

cudaError_t launch_pool_compact(const IndexerArgs& a, const int32_t* pool, const int32_t* pool_cnt, int n_pool,
                                float* scores, int64_t stride, int32_t* n_valid, cudaStream_t s) {
  const int64_t rows = (int64_t)a.B * a.Tq;
  if (rows == 0) return cudaSuccess;
  if (n_pool > kCompactThreads * kCompactPer / 8) return cudaErrorInvalidValue;
  return launch_step(k_pool_compact, dim3((unsigned)rows), dim3(kCompactThreads), 0, s, a, pool, pool_cnt, n_pool,
                     scores, stride, n_valid, status_word());
}

// Generic path (fp32 keys, or shapes the tensor-core path does not take):
// one thread per (query, entry), query staged in shared memory.
template <typename T>
__device__ __forceinline__ float load_as_f32(const T* p, int64_t i);
template <>
__device__ __forceinline__ float load_as_f32<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float load_as_f32<uint16_t>(const uint16_t* p, int64_t i) {
  return bf16_bits_to_f32(p[i]);
}

template <typename T>
__global__ void k_index_scores_generic(IndexerArgs a, const int32_t* __restrict__ pool,
                                       const int32_t* __restrict__ pool_cnt, int n_pool,
                                       float* __restrict__ scores, int64_t stride,
                                       int32_t* __restrict__ n_valid, uint32_t* status) {
  extern __shared__ float sq[];  // [Hi][Di] then w[Hi]
  const int64_t row = blockIdx.y;
  const int b = (int)(row / a.Tq);
  const int nv = n_visible(min(a.n_entries[b], a.max_entries), a.q_pos[row]);
  const T* q = reinterpret_cast<const T*>(a.q) + row * a.Hi * a.Di;
  for (int i = threadIdx.x; i < a.Hi * a.Di; i += blockDim.x) sq[i] = load_as_f32<T>(q, i);
  for (int i = threadIdx.x; i < a.Hi; i += blockDim.x) sq[a.Hi * a.Di + i] = a.w[row * a.Hi + i];
  __syncthreads();
  const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int e;
  if (pool) {
    const int pc = min(max(pool_cnt[row], 0), n_pool);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      int cnt = 0;
      for (int p = 0; p < pc; ++p) cnt += visible_in_block(nv, pool[row * n_pool + p]);
      n_valid[row] = cnt;
    }
    if (c >= 8 * (int64_t)pc) return;
    const int64_t ee = 8LL * pool[row * n_pool + c / 8] + (c % 8);
    e = (ee < 0 || ee >= nv) ? -1 : (int)ee;
  } else {
    e = (int)c;
  }
  if (e < 0 || e >= nv || c >= stride) return;
  const int64_t slot = entry_slot(a.page_table, a.max_pages, a.n_pages, b, e, status);
  if (slot < 0) return;
  const T* k = reinterpret_cast<const T*>(a.k) + slot * a.Di;
  float s = 0.f;
  for (int h = 0; h < a.Hi; ++h) {
    float dot = 0.f;
    for (int i = 0; i < a.Di; ++i) dot = fmaf(sq[h * a.Di + i], load_as_f32<T>(k, i), dot);
    s += sq[a.Hi * a.Di + h] * fmaxf(dot, 0.f);
  }
  scores[row * stride + c] = s;
}

static bool mma_path(const IndexerArgs& a) {
  return a.dtype == CSA2_BF16 && (a.Di == 32 || a.Di == 64 || a.Di == 128) && a.Hi <= 16;
}

template <int NCH, int NT>
static cudaError_t launch_full_mma(const IndexerArgs& a, float* scores, int64_t stride,
                                   float* blockmax, int64_t bm_stride, int max_entries, uint32_t* hist,
                                   cudaStream_t s) {
  const int qg_max = hist ? kHistMaxQG : 16;
  const int QG = a.Tq >= qg_max ? qg_max : a.Tq;
  const size_t smem = hist ? (size_t)QG * kHistBins * sizeof(uint32_t) : 0;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_index_scores_mma<NCH, NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((max_entries + kIdxChunk - 1) / kIdxChunk, (a.Tq + QG - 1) / QG, a.B);
  k_index_scores_mma<NCH, NT><<<grid, kIdxWarps * 32, smem, s>>>(a, QG, scores, stride, blockmax,
                                                                 bm_stride, hist, status_word());
  return counted(cudaGetLastError());
}

template <int NCH, int NT>
static cudaError_t launch_pool_mma(const IndexerArgs& a, const int32_t* pool, const int32_t* pool_cnt,
                                   int n_pool, float* scores, int64_t stride, int32_t* n_valid,
                                   cudaStream_t s) {
  const int pairs = (n_pool + 1) / 2;
  dim3 grid((pairs + kIdxWarps - 1) / kIdxWarps, a.B * a.Tq);
  return launch_step(k_index_scores_pool_mma<NCH, NT>, grid, dim3(kIdxWarps * 32), 0, s, a, pool, pool_cnt, n_pool,
                     scores, stride, n_valid, status_word());
}

#define CSA2_DISPATCH_MMA(FN, ...)                                  \
  do {                                                              \
    const int nt = a.Hi > 8 ? 2 : 1;                                \
    if (a.Di == 128) return nt == 1 ? FN<4, 1>(__VA_ARGS__) : FN<4, 2>(__VA_ARGS__); \
    if (a.Di == 64) return nt == 1 ? FN<2, 1>(__VA_ARGS__) : FN<2, 2>(__VA_ARGS__);  \
    return nt == 1 ? FN<1, 1>(__VA_ARGS__) : FN<1, 2>(__VA_ARGS__);                  \
  } while (0)

cudaError_t launch_index_scores(const IndexerArgs& a, float* scores, int64_t stride, float* blockmax,
                                int64_t bm_stride, int block, int max_entries, uint32_t* hist, cudaStream_t s,
                                uint32_t* bm_hist, bool* bm_hist_built) {
  if (bm_hist_built) *bm_hist_built = false;
  if ((int64_t)a.B * a.Tq == 0 || max_entries == 0) return cudaSuccess;
  if (block == 8 && index_scores_gemm_supported(a)) {
    cudaError_t e = launch_index_scores_gemm(a, scores, stride, blockmax, bm_stride, max_entries, s);
    if (e != cudaSuccess || !hist) return e;
    dim3 hg((max_entries + 255) / 256, a.B * a.Tq);
    k_score_hist<<<hg, 256, 0, s>>>(scores, stride, a, hist);
    return counted(cudaGetLastError());
  }
  if (mma_path(a) && block == 8 && a.Di == 128) {
    if (bm_hist_built) *bm_hist_built = bm_hist && a.Tq == 1 && blockmax;
    if (a.Hi > 8) return launch_scan_pages<2>(a, scores, stride, blockmax, bm_stride, max_entries, hist, bm_hist, s);
    return launch_scan_pages<1>(a, scores, stride, blockmax, bm_stride, max_entries, hist, bm_hist, s);
  }
  if (mma_path(a) && block == 8) {
    CSA2_DISPATCH_MMA(launch_full_mma, a, scores, stride, blockmax, bm_stride, max_entries, hist, s);
  }
  dim3 grid((max_entries + 255) / 256, a.B * a.Tq);
  const size_t smem = (size_t)(a.Hi * a.Di + a.Hi) * sizeof(float);
  if (a.dtype == CSA2_BF16)
    k_index_scores_generic<uint16_t><<<grid, 256, smem, s>>>(a, nullptr, nullptr, 0, scores, stride,
                                                              nullptr, status_word());
  else
    k_index_scores_generic<float><<<grid, 256, smem, s>>>(a, nullptr, nullptr, 0, scores, stride,
                                                           nullptr, status_word());
  cudaError_t e = counted(cudaGetLastError());
  if (e != cudaSuccess) return e;
  if (hist) {
    dim3 hg((max_entries + 255) / 256, a.B * a.Tq);
    k_score_hist<<<hg, 256, 0, s>>>(scores, stride, a, hist);
    e = counted(cudaGetLastError());
    if (e != cudaSuccess) return e;
  }
  if (!blockmax) return cudaSuccess;
  ValidSpec v{nullptr, a.n_entries, a.q_pos, a.Tq, 1, a.max_entries};
  return launch_block_max(scores, (int64_t)a.B * a.Tq, stride, v, block, blockmax, bm_stride, s);
}

cudaError_t launch_index_scores_pool(const IndexerArgs& a, const int32_t* pool, const int32_t* pool_cnt,
                                     int n_pool, int block, float* scores, int64_t stride,
                                     int32_t* n_valid, cudaStream_t s) {
  if ((int64_t)a.B * a.Tq == 0) return cudaSuccess;
  if (mma_path(a) && block == 8) {
    CSA2_DISPATCH_MMA(launch_pool_mma, a, pool, pool_cnt, n_pool, scores, stride, n_valid, s);
  }
  dim3 grid((unsigned)((8 * (int64_t)n_pool + 255) / 256), a.B * a.Tq);
  const size_t smem = (size_t)(a.Hi * a.Di + a.Hi) * sizeof(float);
  if (a.dtype == CSA2_BF16)
    k_index_scores_generic<uint16_t><<<grid, 256, smem, s>>>(a, pool, pool_cnt, n_pool, scores,
                                                              stride, n_valid, status_word());
  else
    k_index_scores_generic<float><<<grid, 256, smem, s>>>(a, pool, pool_cnt, n_pool, scores, stride,
                                                           n_valid, status_word());
  return counted(cudaGetLastError());
}

}  // namespace csa2
