// Top-K selection (radix select) and block maxima for the hierarchical pool.
//
// "DeepSeek-V4.1 架构解析" §02: each query keeps the Top-512 entries by index
// score; the hierarchical indexer keeps the 2,048 blocks of 8 with the largest
// block-max score.  Tie and ordering rules: readings R8-R9 of include/csa2.h.
//
// One CTA per row.  Scores map to order-preserving 32-bit keys (-0 folded into
// +0); four 8-bit radix passes find the exact K-th key T and how many of the
// entries equal to T are taken; a last pass in index order writes the
// selection ascending, taking equal keys from the lowest index up.  Every
// pass reads the row once with coalesced loads; histogram updates are
// aggregated per warp with match.any so equal digits cost one shared atomic.
#include "common.cuh"
#include "internal.h"

namespace csa2 {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) == 0) u = 0;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int row_valid(const ValidSpec& v, int64_t row, int64_t stride) {
  int64_t n;
  if (v.n_valid) {
    n = v.n_valid[row];
  } else if (v.n_entries) {
    const int b = (int)(row / v.Tq);
    int ne = v.n_entries[b];
    if (v.max_n > 0 && ne > v.max_n) ne = (int)v.max_n;
    n = n_visible(ne, v.q_pos[row]);
    if (v.divisor > 1) n = (n + v.divisor - 1) / v.divisor;
  } else {
    n = stride;
  }
  return (int)(n < 0 ? 0 : (n > stride ? stride : n));
}

__device__ __forceinline__ int32_t remap_index(const Remap& r, int64_t row, int c) {
  if (!r.pool) return c;
  return r.pool[row * r.pool_stride + c / r.block] * r.block + c % r.block;
}

// Exclusive block-wide prefix sum of one int per thread (kTopkThreads threads).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kTopkWarps ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kTopkWarps) warp_tot[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const int before = warp ? warp_tot[warp - 1] : 0;
  total = warp_tot[kTopkWarps - 1];
  __syncthreads();
  return before + x - v;
}

__global__ void __launch_bounds__(kTopkThreads)
k_topk(const float* __restrict__ scores, int64_t stride, ValidSpec v, int k,
       int32_t* __restrict__ out_idx, int32_t* __restrict__ out_cnt, Remap remap) {
  __shared__ uint32_t hist[kTopkWarps][256];
  __shared__ int warp_tot[kTopkWarps];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_need;
  const int64_t row = blockIdx.x;
  const float* s = scores + row * stride;
  const int n = row_valid(v, row, stride);
  const int kk = min(k, n);
  int32_t* out = out_idx + row * (int64_t)k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int j = kk + tid; j < k; j += kTopkThreads) out[j] = -1;
  if (tid == 0) out_cnt[row] = kk;
  if (kk == 0) return;
  if (kk == n) {  // everything visible is selected
    for (int j = tid; j < n; j += kTopkThreads) out[j] = remap_index(remap, row, j);
    return;
  }

  uint32_t prefix = 0, mask = 0;
  int need = kk;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < kTopkWarps * 256; i += kTopkThreads) (&hist[0][0])[i] = 0;
    __syncthreads();
    for (int j0 = 0; j0 < n; j0 += kTopkThreads) {
      const int j = j0 + tid;
      uint32_t digit = 256;  // 256 = not counted
      if (j < n) {
        const uint32_t key = order_key(s[j]);
        if ((key & mask) == prefix) digit = (key >> shift) & 0xFFu;
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, digit);
      if (digit < 256 && lane == __ffs(peers) - 1) atomicAdd(&hist[warp][digit], __popc(peers));
    }
    __syncthreads();
    if (tid < 256) {
      uint32_t c = 0;
#pragma unroll 8
      for (int w = 0; w < kTopkWarps; ++w) c += hist[w][tid];
      hist[0][tid] = c;
    }
    __syncthreads();
    if (tid == 0) {
      int cum = 0;
      for (int dg = 255; dg >= 0; --dg) {
        const int c = (int)hist[0][dg];
        if (cum + c >= need) {
          sh_prefix = prefix | ((uint32_t)dg << shift);
          sh_need = need - cum;
          break;
        }
        cum += c;
      }
    }
    __syncthreads();
    prefix = sh_prefix;
    need = sh_need;
    mask |= 0xFFu << shift;
  }
  const uint32_t T = prefix;  // the K-th largest key; `need` of the keys == T are taken

  // index-ordered output: thread tid owns columns [lo, hi)
  const int chunk = (n + kTopkThreads - 1) / kTopkThreads;
  const int lo = min(n, tid * chunk), hi = min(n, lo + chunk);
  int gt = 0, eq = 0;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = order_key(s[j]);
    gt += key > T;
    eq += key == T;
  }
  int tot;
  const int gt_before = block_exclusive_scan(gt, warp_tot, tot);
  const int eq_before = block_exclusive_scan(eq, warp_tot, tot);
  int pos = gt_before + min(eq_before, need);
  int eq_seen = eq_before;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = order_key(s[j]);
    if (key > T) {
      out[pos++] = remap_index(remap, row, j);
    } else if (key == T) {
      if (eq_seen < need) out[pos++] = remap_index(remap, row, j);
      ++eq_seen;
    }
  }
}

// Block maxima: out[row][b] = max of scores[row][8b .. 8b+7] over the valid
// columns, for b < ceil(n_valid / block).
__global__ void k_block_max(const float* __restrict__ scores, int64_t stride, ValidSpec v, int block,
                            float* __restrict__ out, int64_t out_stride) {
  const int64_t row = blockIdx.y;
  const int n = row_valid(v, row, stride);
  const int nb = (n + block - 1) / block;
  const int bidx = blockIdx.x * blockDim.x + threadIdx.x;
  if (bidx >= nb) return;
  const float* s = scores + row * stride + (int64_t)bidx * block;
  const int m = min(block, n - bidx * block);
  float mx = s[0];
  for (int i = 1; i < m; ++i) mx = fmaxf(mx, s[i]);
  out[row * out_stride + bidx] = mx;
}

cudaError_t launch_topk(const float* scores, int64_t rows, int64_t stride, ValidSpec v, int k,
                        int32_t* out_idx, int32_t* out_cnt, Remap remap, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  k_topk<<<(unsigned)rows, kTopkThreads, 0, s>>>(scores, stride, v, k, out_idx, out_cnt, remap);
  return counted(cudaGetLastError());
}

cudaError_t launch_block_max(const float* scores, int64_t rows, int64_t stride, ValidSpec v, int block,
                             float* out, int64_t out_stride, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int64_t nb = (stride + block - 1) / block;
  dim3 grid((unsigned)((nb + 255) / 256), (unsigned)rows);
  k_block_max<<<grid, 256, 0, s>>>(scores, stride, v, block, out, out_stride);
  return counted(cudaGetLastError());
}

}  // namespace csa2
