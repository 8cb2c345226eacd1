// Top-K selection and block maxima for the hierarchical pool.
//
// "DeepSeek-V4.1 架构解析" §02: each query keeps the Top-512 entries by index
// score; the hierarchical indexer keeps the 2,048 blocks of 8 with the largest
// block-max score.  Tie and ordering rules: readings R8-R9 of include/csa2.h.
//
// One CTA per row.  Scores map to order-preserving 32-bit keys (-0 folded into
// +0).  A 2048-bin histogram of the top 11 key bits (built by the scoring
// kernel while it writes the scores, or here in one pass) locates the bin
// that holds the K-th key; one pass over the row then keeps every entry of a
// higher bin and copies the entries of that bin into shared memory, where the
// exact K-th key and its tie count are found by radix passes over the few
// candidates.  The selection is sorted by index in shared memory and written
// ascending.  When the threshold bin is too full for shared memory (e.g. many
// equal scores), a radix select over the whole row finishes from the 11-bit
// prefix instead.  Warp-aggregated (match.any / ballot) shared atomics keep
// equal digits from serialising.
#include "common.cuh"
#include "internal.h"

namespace csa2 {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kCandCap = 4096;      // candidates of the threshold bin kept in smem
constexpr int kBatch = 8;           // row elements loaded per thread before they are used

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) == 0) u = 0;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The float whose order_key is `key` (key > 0).
__device__ __forceinline__ float key_float(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

__device__ __forceinline__ int row_valid(const ValidSpec& v, int64_t row, int64_t stride) {
  int64_t n;
  if (v.n_valid) {
    n = v.n_valid[row];
    if (v.divisor > 1) n = (n + v.divisor - 1) / v.divisor;
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

// Exclusive block-wide prefix sum of one int per thread (NT threads).
template <int NT>
__device__ __forceinline__ int block_exclusive_scan_t(int v, int* warp_tot) {
  constexpr int NW = NT / 32;
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
    int w = lane < NW ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NW) warp_tot[lane] = w;
  }
  __syncthreads();
  const int before = warp ? warp_tot[warp - 1] : 0;
  __syncthreads();
  return before + x - v;
}

// Shared-memory reductions without a returned value (red.shared: the issuing
// thread does not wait for them).
__device__ __forceinline__ void red_add_shared(uint32_t* p, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(p)), "r"(v) : "memory");
}
__device__ __forceinline__ void red_or_shared(uint32_t* p, uint32_t v) {
  asm volatile("red.shared.or.b32 [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(p)), "r"(v) : "memory");
}

// Adds `digit` (< nbins, or >= nbins for "none") to a shared histogram: one
// shared reduction per lane (match.any aggregation costs more than the rare
// serialisation of equal digits).
__device__ __forceinline__ void warp_hist_add(uint32_t* hist, uint32_t digit, uint32_t nbins) {
  if (digit < nbins) red_add_shared(&hist[digit], 1u);
}

// Slot in a shared list for every lane with `take` (one atomic per warp); -1
// for lanes that take nothing or when the list is full.
__device__ __forceinline__ int warp_slot(int* counter, bool take, int cap) {
  const uint32_t m = __ballot_sync(0xffffffffu, take);
  if (!m) return -1;
  const int lane = threadIdx.x & 31;
  int base = 0;
  if (lane == __ffs(m) - 1) base = atomicAdd(counter, __popc(m));
  base = __shfl_sync(0xffffffffu, base, __ffs(m) - 1);
  const int pos = base + __popc(m & ((1u << lane) - 1));
  return (take && pos < cap) ? pos : -1;
}

// Finds, scanning digits from the top, the digit holding the need-th largest
// element of a `bins`-bin histogram; *above receives the count in higher bins.
template <int NT>
__device__ __forceinline__ int find_digit_t(const uint32_t* hist, int bins, int need, int* warp_tot, int* above) {
  __shared__ int s_digit, s_above;
  const int per = (bins + NT - 1) / NT;
  const int hi = bins - (int)threadIdx.x * per;   // thread t owns [hi - per, hi), highest first
  const int lo = max(0, hi - per);
  int c = 0;
  for (int d = lo; d < hi; ++d) c += hist[d];
  if (threadIdx.x == 0) { s_digit = 0; s_above = 0; }
  const int before = block_exclusive_scan_t<NT>(c, warp_tot);
  if (before < need && before + c >= need) {
    int cum = before;
    for (int d = hi - 1; d >= lo; --d) {
      const int h = (int)hist[d];
      if (cum + h >= need) {
        s_digit = d;
        s_above = cum;
        break;
      }
      cum += h;
    }
  }
  __syncthreads();
  *above = s_above;
  return s_digit;
}

constexpr int kBitmapMax = 1 << 18;            // rows up to 262,144 entries use bitmaps
constexpr int kBitmapWords = kBitmapMax / 32;

struct TopkSmem {
  uint32_t hist[2048];
  uint32_t hist2[256];
  int warp_tot[kTopkWarps];
  int nC;
  uint32_t ckey[kCandCap];        // candidate keys of the threshold bin
  int32_t cidx[kCandCap];         // and their indices
  uint32_t sel_bits[kBitmapWords];  // selected entries, one bit per index
  uint32_t tie_bits[kBitmapWords];  // entries equal to the K-th key
};

// The exact K-th key among keys[0 .. nC) by one warp: three 7-bit radix
// passes below the 11-bit bin, with warp shuffles instead of block barriers
// (few candidates).  *T_out = the K-th key, *need_out = entries equal to it
// to take.
template <class Sm>
__device__ void warp_radix_threshold(Sm& sm, const uint32_t* keys, int nC, int bstar, int need, uint32_t* T_out,
                                     int* need_out) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = (uint32_t)bstar << 21, mask = 0xFFE00000u;
  for (int p = 0; p < 3; ++p) {
    const int sh = 14 - 7 * p;
    for (int i = lane; i < 128; i += 32) sm.hist2[i] = 0;
    __syncwarp();
    for (int i = lane; i < nC; i += 32) {
      const uint32_t key = keys[i];
      if ((key & mask) == prefix) red_add_shared(&sm.hist2[(key >> sh) & 127u], 1u);
    }
    __syncwarp();
    // lane L owns digits 127 - 4L .. 124 - 4L, highest first
    uint32_t h[4];
    int c = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      h[q] = sm.hist2[127 - 4 * lane - q];
      c += (int)h[q];
    }
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int before = incl - c;
    const uint32_t hit = __ballot_sync(0xffffffffu, before < need && incl >= need);
    const int L = hit ? __ffs(hit) - 1 : 0;   // the matching candidates always hold >= need entries
    int dg = 0, ab = 0;
    if (lane == L) {
      int cum = before;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (cum + (int)h[q] >= need) {
          dg = 127 - 4 * lane - q;
          ab = cum;
          break;
        }
        cum += (int)h[q];
      }
    }
    dg = __shfl_sync(0xffffffffu, dg, L);
    ab = __shfl_sync(0xffffffffu, ab, L);
    need -= ab;
    prefix |= (uint32_t)dg << sh;
    mask |= 127u << sh;
    __syncwarp();   // every lane has read hist2 before the next pass clears it
  }
  *T_out = prefix;
  *need_out = need;
}

// Index-ordered output of the selection: sel_bits holds every selected entry
// but the ties, tie_bits the entries equal to the K-th key, of which the
// `need` lowest-index ones are taken.
template <int NT, class Sm>
__device__ void write_selection(Sm& sm, int words, int kk, int need, int32_t* __restrict__ out, const Remap& remap,
                                int64_t row) {
  const int tid = threadIdx.x;
  // index-ordered output: thread tid owns words [w0, w1)
  const int per = (words + NT - 1) / NT;
  const int w0 = min(words, tid * per), w1 = min(words, w0 + per);
  int ties = 0;
  for (int w = w0; w < w1; ++w) ties += __popc(sm.tie_bits[w]);
  int ties_before = block_exclusive_scan_t<NT>(ties, sm.warp_tot);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) {
    uint32_t tb = sm.tie_bits[w];
    while (tb && ties_before < need) {      // lowest indices first
      const uint32_t low = tb & (0u - tb);
      sm.sel_bits[w] |= low;
      tb ^= low;
      ++ties_before;
    }
    cnt += __popc(sm.sel_bits[w]);
  }
  int pos = block_exclusive_scan_t<NT>(cnt, sm.warp_tot);
  for (int w = w0; w < w1; ++w) {
    uint32_t sb = sm.sel_bits[w];
    while (sb) {
      const int bit = __ffs(sb) - 1;
      sb &= sb - 1;
      if (pos < kk) out[pos] = remap_index(remap, row, w * 32 + bit);
      ++pos;
    }
  }
}

// Selection from the candidates of the threshold bin: the sel bitmap already
// holds every entry of a higher bin; find the exact K-th key among the
// candidates, mark the candidates above it and the `need` lowest-index ties,
// and write the selection in index order.
template <int NT, class Sm, bool kWarpRadix = false>
__device__ void finish_from_candidates(Sm& sm, int n, int kk, int bstar, int need, int nC,
                                       int32_t* __restrict__ out, const Remap& remap, int64_t row) {
  const int tid = threadIdx.x;
  const int words = (n + 31) / 32;
  uint32_t prefix = (uint32_t)bstar << 21, mask = 0xFFE00000u;
  if (kWarpRadix) {
    __shared__ uint32_t s_T;
    __shared__ int s_need;
    if (tid < 32) {
      uint32_t t;
      int nd;
      warp_radix_threshold(sm, sm.ckey, nC, bstar, need, &t, &nd);
      if (tid == 0) {
        s_T = t;
        s_need = nd;
      }
    }
    __syncthreads();
    prefix = s_T;
    need = s_need;
  }
  for (int p = 0; p < (kWarpRadix ? 0 : 3); ++p) {   // 3 radix passes of 7 bits over the candidates
    const int sh = 14 - 7 * p;
    const uint32_t nb = 128;
    for (int i = tid; i < (int)nb; i += NT) sm.hist2[i] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < nC; i0 += NT) {
      const int i = i0 + tid;
      uint32_t dg = 0xFFFFFFFFu;
      if (i < nC) {
        const uint32_t key = sm.ckey[i];
        if ((key & mask) == prefix) dg = (key >> sh) & (nb - 1);
      }
      warp_hist_add(sm.hist2, dg, nb);
    }
    __syncthreads();
    int ab;
    const int dg = find_digit_t<NT>(sm.hist2, (int)nb, need, sm.warp_tot, &ab);
    need -= ab;
    prefix |= (uint32_t)dg << sh;
    mask |= (nb - 1) << sh;
  }
  const uint32_t T = prefix;             // exact K-th key; `need` entries equal to T are taken
  for (int i = tid; i < nC; i += NT) {
    const uint32_t key = sm.ckey[i];
    const int32_t j = sm.cidx[i];
    if (key > T) red_or_shared(&sm.sel_bits[j >> 5], 1u << (j & 31));
    else if (key == T) red_or_shared(&sm.tie_bits[j >> 5], 1u << (j & 31));
  }
  __syncthreads();
  write_selection<NT>(sm, words, kk, need, out, remap, row);
}

// Crowded threshold bin: radix select over the whole row from the 11-bit
// prefix, then an index-ordered pass writes the selection.
template <int NT, class Sm>
__device__ void radix_whole_row(Sm& sm, const float* __restrict__ s, int n, int kk, int bstar, int need,
                                int32_t* __restrict__ out, const Remap& remap, int64_t row) {
  const int tid = threadIdx.x;
  uint32_t prefix = (uint32_t)bstar << 21, mask = 0xFFE00000u;
  for (int p = 0; p < 3; ++p) {
    const int sh = p == 0 ? 13 : (p == 1 ? 5 : 0);
    const uint32_t nb = p == 2 ? 32u : 256u;
    for (int i = tid; i < (int)nb; i += NT) sm.hist2[i] = 0;
    __syncthreads();
    for (int j0 = 0; j0 < n; j0 += NT) {
      const int j = j0 + tid;
      uint32_t dg = 0xFFFFFFFFu;
      if (j < n) {
        const uint32_t key = order_key(s[j]);
        if ((key & mask) == prefix) dg = (key >> sh) & (nb - 1);
      }
      warp_hist_add(sm.hist2, dg, nb);
    }
    __syncthreads();
    int ab;
    const int dg = find_digit_t<NT>(sm.hist2, (int)nb, need, sm.warp_tot, &ab);
    need -= ab;
    prefix |= (uint32_t)dg << sh;
    mask |= (nb - 1) << sh;
  }
  const uint32_t T = prefix;
  const int chunk = (n + NT - 1) / NT;
  const int lo = min(n, tid * chunk), hi = min(n, lo + chunk);
  int gt = 0, eq = 0;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = order_key(s[j]);
    gt += key > T;
    eq += key == T;
  }
  const int gt_before = block_exclusive_scan_t<NT>(gt, sm.warp_tot);
  const int eq_before = block_exclusive_scan_t<NT>(eq, sm.warp_tot);
  int pos = gt_before + min(eq_before, need);
  int eq_seen = eq_before;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = order_key(s[j]);
    if (key > T) {
      if (pos < kk) out[pos] = remap_index(remap, row, j);
      ++pos;
    } else if (key == T) {
      if (eq_seen < need) {
        if (pos < kk) out[pos] = remap_index(remap, row, j);
        ++pos;
      }
      ++eq_seen;
    }
  }
}

// Loads (or builds) the 2048-bin key histogram of a row into shared memory
// and locates the threshold bin.
template <int NT>
__device__ __forceinline__ void locate_bin(uint32_t* shist, int* warp_tot, const float* __restrict__ s, int n,
                                           int kk, const uint32_t* __restrict__ hist_row, int* bstar, int* above) {
  const int tid = threadIdx.x;
  if (hist_row) {
    for (int i = tid; i < 2048; i += NT) shist[i] = hist_row[i];
  } else {
    for (int i = tid; i < 2048; i += NT) shist[i] = 0;
    __syncthreads();
    for (int j0 = 0; j0 < n; j0 += NT * kBatch) {
      float v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {   // independent loads first
        const int j = j0 + u * NT + tid;
        v[u] = j < n ? s[j] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = j0 + u * NT + tid;
        warp_hist_add(shist, j < n ? order_key(v[u]) >> 21 : 0xFFFFFFFFu, 2048);
      }
    }
  }
  __syncthreads();
  *bstar = find_digit_t<NT>(shist, 2048, kk, warp_tot, above);
}

// kB row elements per thread are loaded before any is used; kMinBlocks CTAs
// (rows) per SM.  Few rows: <32, 1> (one round trip for a 32K-entry row);
// many rows: <8, 2> (two rows per SM, <= 32 registers).
template <int kB, int kMinBlocks>
__global__ void __launch_bounds__(kTopkThreads, kMinBlocks)
k_topk(const float* __restrict__ scores, int64_t stride, ValidSpec v, int k, int32_t* __restrict__ out_idx,
       int32_t* __restrict__ out_cnt, Remap remap, const uint32_t* __restrict__ hist_in, int64_t hist_stride) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(smem_raw);
  const int64_t row = blockIdx.x;
  const float* s = scores + row * stride;
  const int n = row_valid(v, row, stride);
  const int kk = min(k, n);
  int32_t* out = out_idx + row * (int64_t)k;
  const int tid = threadIdx.x, lane = tid & 31;

  for (int j = kk + tid; j < k; j += kTopkThreads) out[j] = -1;
  if (tid == 0) out_cnt[row] = kk;
  if (kk == 0) return;
  if (kk == n) {  // everything visible is selected
    for (int j = tid; j < n; j += kTopkThreads) out[j] = remap_index(remap, row, j);
    return;
  }
  if (tid == 0) sm.nC = 0;
  int bstar, above;
  locate_bin<kTopkThreads>(sm.hist, sm.warp_tot, s, n, kk, hist_in ? hist_in + row * hist_stride : nullptr,
                           &bstar, &above);
  const int need = kk - above;           // entries of bin bstar to take
  const int n_bin = (int)sm.hist[bstar];
  if (n_bin > kCandCap || n > kBitmapMax) {
    radix_whole_row<kTopkThreads>(sm, s, n, kk, bstar, need, out, remap, row);
    return;
  }
  const int words = (n + 31) / 32;
  for (int i = tid; i < words; i += kTopkThreads) sm.tie_bits[i] = 0;
  // one pass: higher bins -> selection bitmap; bin bstar -> candidate list
  // (lanes of a warp cover one aligned 32-entry word, so the ballot is the
  // word); a batch's candidates are appended with one atomic per warp
  for (int j0 = 0; j0 < n; j0 += kTopkThreads * kB) {
    float vv[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) {   // independent loads first
      const int j = j0 + u * kTopkThreads + tid;
      vv[u] = j < n ? s[j] : 0.f;
    }
    uint32_t cmask = 0;
    int ccount = 0;
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int j = j0 + u * kTopkThreads + tid;
      uint32_t bin = 0;
      if (j < n) bin = order_key(vv[u]) >> 21;
      const uint32_t word = __ballot_sync(0xffffffffu, j < n && bin > (uint32_t)bstar);
      if (lane == 0 && j < n) sm.sel_bits[j >> 5] = word;
      if (j < n && bin == (uint32_t)bstar) {
        cmask |= 1u << u;
        ++ccount;
      }
    }
    int incl = ccount;   // warp prefix sum of the candidate counts
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int wtot = __shfl_sync(0xffffffffu, incl, 31);
    if (wtot) {
      int base = 0;
      if (lane == 31) base = atomicAdd(&sm.nC, wtot);
      base = __shfl_sync(0xffffffffu, base, 31);
      int pos = base + incl - ccount;
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        if ((cmask >> u) & 1u) {
          if (pos < kCandCap) {
            sm.ckey[pos] = order_key(vv[u]);
            sm.cidx[pos] = j0 + u * kTopkThreads + tid;
          }
          ++pos;
        }
      }
    }
  }
  __syncthreads();
  finish_from_candidates<kTopkThreads, TopkSmem, true>(sm, n, kk, bstar, need, min(sm.nC, kCandCap), out, remap, row);
}

// ---- one row per CTA, histogram given or row in registers ----------------------------
// When the scoring kernel built the row's histogram (decode) the threshold bin
// is known before the row is read: the row's first loads are issued first and
// the bin is located while they are in flight.  Without one, a row of at most
// 32,768 entries is held in registers whole (32 entries per thread) and its
// histogram built from them.  Every entry is then compared as a float with the
// bin's edges: above the bin -> selection bit, inside -> candidate; the finish
// is k_topk's.
constexpr int kHistBatch = 32;   // row elements per thread in flight

template <bool kVec>
__device__ __forceinline__ int hb_index(int j0, int tid, int u) {
  return kVec ? j0 + 4 * ((u >> 2) * kTopkThreads + tid) + (u & 3) : j0 + u * kTopkThreads + tid;
}
template <bool kVec>
__device__ __forceinline__ void load_hb(const float* __restrict__ s, int n, int j0, int tid, float (&x)[kHistBatch]) {
  if (kVec) {
#pragma unroll
    for (int u = 0; u < kHistBatch / 4; ++u) {
      const int j = hb_index<true>(j0, tid, 4 * u);
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j + 3 < n) {
        f = *reinterpret_cast<const float4*>(s + j);
      } else if (j < n) {
        f.x = s[j];
        if (j + 1 < n) f.y = s[j + 1];
        if (j + 2 < n) f.z = s[j + 2];
      }
      x[4 * u] = f.x; x[4 * u + 1] = f.y; x[4 * u + 2] = f.z; x[4 * u + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int u = 0; u < kHistBatch; ++u) {
      const int j = hb_index<false>(j0, tid, u);
      x[u] = j < n ? s[j] : 0.f;
    }
  }
}

template <bool kVec>
__global__ void __launch_bounds__(kTopkThreads, 1)
k_topk_hist(const float* __restrict__ scores, int64_t stride, ValidSpec v, int k, int32_t* __restrict__ out_idx,
            int32_t* __restrict__ out_cnt, Remap remap, const uint32_t* __restrict__ hist_in, int64_t hist_stride,
            uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(smem_raw);
  const int64_t row = blockIdx.x;
  const float* s = scores + row * stride;
  int n = row_valid(v, row, stride);   // <= kBitmapMax, or <= the register capacity without hist_in
  if (!hist_in && n > kTopkThreads * kHistBatch) {   // the launcher's bound on the valid counts was wrong
    if (threadIdx.x == 0) raise_status(status, CSA2_STATUS_BAD_COUNT);
    n = kTopkThreads * kHistBatch;
  }
  const int kk = min(k, n);
  int32_t* out = out_idx + row * (int64_t)k;
  const int tid = threadIdx.x, lane = tid & 31;

  for (int j = kk + tid; j < k; j += kTopkThreads) out[j] = -1;
  if (tid == 0) out_cnt[row] = kk;
  if (kk == 0) return;
  if (kk == n) {
    for (int j = tid; j < n; j += kTopkThreads) out[j] = remap_index(remap, row, j);
    return;
  }
  float x[kHistBatch];
  load_hb<kVec>(s, n, 0, tid, x);   // in flight while the bin is located
  const int words = (n + 31) / 32;
  for (int i = tid; i < words; i += kTopkThreads) {
    sm.sel_bits[i] = 0;
    sm.tie_bits[i] = 0;
  }
  if (tid == 0) sm.nC = 0;
  if (hist_in) {
    for (int i = tid; i < 2048; i += kTopkThreads) sm.hist[i] = hist_in[row * hist_stride + i];
  } else {   // n <= kTopkThreads * kHistBatch (checked by the launcher): the whole row is in x
    for (int i = tid; i < 2048; i += kTopkThreads) sm.hist[i] = 0;
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kHistBatch; ++u)
      warp_hist_add(sm.hist, hb_index<kVec>(0, tid, u) < n ? order_key(x[u]) >> 21 : 0xFFFFFFFFu, 2048);
  }
  __syncthreads();
  int above;
  const int bstar = find_digit_t<kTopkThreads>(sm.hist, 2048, kk, sm.warp_tot, &above);
  const int need = kk - above;
  if ((int)sm.hist[bstar] > kCandCap) {
    radix_whole_row<kTopkThreads>(sm, s, n, kk, bstar, need, out, remap, row);
    return;
  }
  const float f_lo = bstar == 0 ? -INFINITY : key_float((uint32_t)bstar << 21);
  const float f_hi = bstar == 2047 ? __uint_as_float(0x7FFFFFFFu) : key_float((uint32_t)(bstar + 1) << 21);   // NaN: none above
  for (int j0 = 0; j0 < n; j0 += kTopkThreads * kHistBatch) {
    if (j0 > 0) load_hb<kVec>(s, n, j0, tid, x);
    uint32_t cm = 0;
#pragma unroll
    for (int u = 0; u < kHistBatch; ++u) {
      const int j = hb_index<kVec>(j0, tid, u);
      if (j < n) {
        if (x[u] >= f_hi) red_or_shared(&sm.sel_bits[j >> 5], 1u << (j & 31));
        else if (x[u] >= f_lo) cm |= 1u << u;
      }
    }
    const int c = __popc(cm);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int wtot = __shfl_sync(0xffffffffu, incl, 31);
    if (wtot) {
      int base = 0;
      if (lane == 31) base = atomicAdd(&sm.nC, wtot);
      base = __shfl_sync(0xffffffffu, base, 31);
      int pos = base + incl - c;
#pragma unroll
      for (int u = 0; u < kHistBatch; ++u) {
        if ((cm >> u) & 1u) {
          if (pos < kCandCap) {
            sm.ckey[pos] = order_key(x[u]);
            sm.cidx[pos] = hb_index<kVec>(j0, tid, u);
          }
          ++pos;
        }
      }
    }
  }
  __syncthreads();
  finish_from_candidates<kTopkThreads, TopkSmem, true>(sm, n, kk, bstar, need, min(sm.nC, kCandCap), out, remap, row);
}

// ---- few rows with a given histogram, each spread over a cluster -------------------------
// Decode: 32 rows of 32,768 scores would keep 32 SMs busy.  A cluster of
// kTopkRanks CTAs takes one row, rank r a contiguous quarter of it.  Every
// rank locates the threshold bin from the row's histogram while its quarter
// loads, counts its entries above the bin and sends the bin's candidates
// (key, index) and that count to every rank of the cluster (distributed
// shared-memory stores, then one cluster barrier).  From then on each rank
// works alone on identical data: the exact K-th key among all candidates (two
// radix passes of 11 and 10 bits), the ties taken (the lowest indices), every
// rank's selected count and so its own output offset; it then writes its
// quarter's selection in index order.  The ranks' outputs are contiguous runs
// of one ascending list.
constexpr int kTopkRanks = 4;
constexpr int kClThreads = 1024;                             // threads per rank
constexpr int kClPer = 8;                                    // contiguous entries per thread
constexpr int kClusterMaxN = kTopkRanks * kClThreads * kClPer;
constexpr int kClusterCap = 2048;   // candidates of the threshold bin, all ranks together

struct TopkClusterSmem {
  uint32_t hist[2048];
  uint32_t hist2[2048];
  int warp_tot[kTopkWarps];
  int n_above[kTopkRanks];   // entries above the bin in rank r's quarter (sent by rank r)
  int n_cand[kTopkRanks];    // candidates of rank r's quarter (sent by rank r)
  int local_above, local_cand, tie_idx, bstar, need, n_tie, off;
  uint32_t T;
  uint2 cand[kTopkRanks][kClusterCap];   // (key, index); segment r filled by rank r
};

__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_map(const void* p, uint32_t rank) {   // this CTA's address in `rank`
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
  return r;
}
// Split cluster barrier: arrive early (no ordering), wait before the first
// remote store (every CTA of the cluster has then started).
__device__ __forceinline__ void cl_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cl_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void cl_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cl_st(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cl_st2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

// One warp: the digit of a BINS-bin histogram (BINS = 64 m) that holds the
// need-th largest element, and the count in the digits above it.  Two levels of
// warp scans: lane l first sums the BINS/32 digits of chunk l (chunk 0 = the
// highest digits), then the chunk that holds the element is split over the lanes
// two digits each.  No block barrier.
template <int BINS>
__device__ __forceinline__ int warp_find_digit(const uint32_t* hist, int need, int* above_out) {
  constexpr int PER = BINS / 32;
  const int lane = threadIdx.x & 31;
  const int hi = BINS - PER * lane;   // lane's chunk: digits [hi - PER, hi)
  const uint4* h4 = reinterpret_cast<const uint4*>(hist + hi - PER);
  int c = 0;
#pragma unroll
  for (int q = 0; q < PER / 4; ++q) {
    const uint4 w = h4[q];
    c += (int)(w.x + w.y + w.z + w.w);
  }
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  uint32_t hit = __ballot_sync(0xffffffffu, incl - c < need && incl >= need);
  const int L = hit ? __ffs(hit) - 1 : 31;
  int cum = __shfl_sync(0xffffffffu, incl - c, L);   // elements above chunk L
  // chunk L, highest digits first: lane l takes digits top - 2l and top - 2l - 1
  const int top = BINS - PER * L - 1 - 2 * lane;
  const int ha = 2 * lane < PER ? (int)hist[top] : 0;
  const int hb = 2 * lane + 1 < PER ? (int)hist[top - 1] : 0;
  int c2 = ha + hb, incl2 = c2;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl2, o);
    if (lane >= o) incl2 += t;
  }
  const int before = cum + incl2 - c2;
  hit = __ballot_sync(0xffffffffu, before < need && before + c2 >= need);
  const int L2 = hit ? __ffs(hit) - 1 : 0;
  const int first = before + ha >= need;   // the element lies in the higher of the two digits
  const int dg = __shfl_sync(0xffffffffu, first ? top : top - 1, L2);
  *above_out = __shfl_sync(0xffffffffu, first ? before : before + ha, L2);
  return dg;
}

template <bool kVec>
__global__ void __launch_bounds__(kClThreads, 1)
k_topk_cluster(const float* __restrict__ scores, int64_t stride, ValidSpec v, int k, int32_t* __restrict__ out_idx,
               int32_t* __restrict__ out_cnt, Remap remap, const uint32_t* __restrict__ hist_in,
               int64_t hist_stride) {
  constexpr int NT = kClThreads;
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkClusterSmem& sm = *reinterpret_cast<TopkClusterSmem*>(smem_raw);
  const uint32_t rank = cl_rank();
  const int64_t row = blockIdx.x / kTopkRanks;
  const float* s = scores + row * stride;
  const int n = row_valid(v, row, stride);   // <= stride <= kClusterMaxN (checked by the launcher)
  const int kk = min(k, n);
  int32_t* out = out_idx + row * (int64_t)k;
  const int tid = threadIdx.x, lane = tid & 31;
  // every rank takes the same early exits: they depend on the row only
  if (rank == 0) {
    for (int j = kk + tid; j < k; j += NT) out[j] = -1;
    if (tid == 0) out_cnt[row] = kk;
  }
  if (kk == 0) return;
  if (kk == n) {
    if (rank == 0)
      for (int j = tid; j < n; j += NT) out[j] = remap_index(remap, row, j);
    return;
  }
  // this rank's quarter of the row (a multiple of 4 entries: float4 aligned); thread
  // tid holds the kClPer entries j0 .. j0 + kClPer - 1 (index order = thread order)
  const int part = ((n + 4 * kTopkRanks - 1) / (4 * kTopkRanks)) * 4;
  const int q0 = min(n, (int)rank * part), q1 = min(n, q0 + part);
  const int j0 = q0 + kClPer * tid;
  float x[kClPer];
#pragma unroll
  for (int u = 0; u < kClPer; u += 4) {
    const int j = j0 + u;
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (kVec && j + 3 < q1) {
      f = *reinterpret_cast<const float4*>(s + j);
    } else if (j < q1) {
      f.x = s[j];
      if (j + 1 < q1) f.y = s[j + 1];
      if (j + 2 < q1) f.z = s[j + 2];
      if (j + 3 < q1) f.w = s[j + 3];
    }
    x[u] = f.x; x[u + 1] = f.y; x[u + 2] = f.z; x[u + 3] = f.w;
  }
  for (int i = tid; i < 2048; i += NT) sm.hist[i] = hist_in[row * hist_stride + i];
  if (tid == 0) {
    sm.local_above = 0;
    sm.local_cand = 0;
    sm.tie_idx = 0x7FFFFFFF;
  }
  __syncthreads();
  if (tid < 32) {
    int ab;
    const int d = warp_find_digit<2048>(sm.hist, kk, &ab);
    if (tid == 0) {
      sm.bstar = d;
      sm.need = kk - ab;
    }
  }
  __syncthreads();
  const int bstar = sm.bstar;
  int need = sm.need;
  if ((int)sm.hist[bstar] > kClusterCap) {   // crowded bin (same decision on every rank)
    if (rank == 0) radix_whole_row<NT>(sm, s, n, kk, bstar, need, out, remap, row);
    return;
  }
  cl_arrive_relaxed();

  // ---- classify the quarter: above the bin, or a candidate of the bin
  int my_above = 0;
  uint32_t cm = 0;
#pragma unroll
  for (int u = 0; u < kClPer; ++u) {
    if (j0 + u < q1) {
      const int bin = (int)(order_key(x[u]) >> 21);
      my_above += bin > bstar;
      if (bin == bstar) cm |= 1u << u;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) my_above += __shfl_xor_sync(0xffffffffu, my_above, o);
  if (lane == 0 && my_above) atomicAdd(&sm.local_above, my_above);
  const int c = __popc(cm);
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const int wtot = __shfl_sync(0xffffffffu, incl, 31);
  int base = 0;
  if (lane == 31 && wtot) base = atomicAdd(&sm.local_cand, wtot);
  int pos = __shfl_sync(0xffffffffu, base, 31) + incl - c;
  cl_wait();   // every CTA of the cluster has started: its shared memory may be written
#pragma unroll
  for (int u = 0; u < kClPer; ++u) {
    if ((cm >> u) & 1u) {
      if (pos < kClusterCap) {
#pragma unroll
        for (int r = 0; r < kTopkRanks; ++r)
          cl_st2(cl_map(&sm.cand[rank][pos], (uint32_t)r), order_key(x[u]), (uint32_t)(j0 + u));
      }
      ++pos;
    }
  }
  __syncthreads();
  if (tid < kTopkRanks) {
    cl_st(cl_map(&sm.n_above[rank], (uint32_t)tid), (uint32_t)sm.local_above);
    cl_st(cl_map(&sm.n_cand[rank], (uint32_t)tid), (uint32_t)min(sm.local_cand, kClusterCap));
  }
  cl_sync();   // every rank's counts and candidates are in every rank

  // ---- the exact K-th key T among the candidates: bits 20..10, then 9..0 (block-wide
  // histograms, one warp locates the digit), the ties taken and this rank's offset
  for (int i = tid; i < 2048; i += NT) sm.hist2[i] = 0;
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kTopkRanks; ++r)
    for (int i = tid; i < sm.n_cand[r]; i += NT) red_add_shared(&sm.hist2[(sm.cand[r][i].x >> 10) & 2047u], 1u);
  __syncthreads();
  if (tid < 32) {
    int ab;
    const int d1 = warp_find_digit<2048>(sm.hist2, need, &ab);
    if (tid == 0) {
      sm.T = ((uint32_t)bstar << 11) | (uint32_t)d1;   // key >> 10 of the K-th key
      sm.need = need - ab;
    }
  }
  __syncthreads();
  const uint32_t hi21 = sm.T;
  need = sm.need;
  for (int i = tid; i < 1024; i += NT) sm.hist2[i] = 0;
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kTopkRanks; ++r)
    for (int i = tid; i < sm.n_cand[r]; i += NT) {
      const uint32_t key = sm.cand[r][i].x;
      if ((key >> 10) == hi21) red_add_shared(&sm.hist2[key & 1023u], 1u);
    }
  __syncthreads();
  if (tid < 32) {
    int ab;
    const int d2 = warp_find_digit<1024>(sm.hist2, need, &ab);
    if (tid == 0) {
      sm.T = (hi21 << 10) | (uint32_t)d2;
      sm.need = need - ab;                  // entries equal to T that are taken (>= 1)
      sm.n_tie = (int)sm.hist2[d2];
      int off = 0;
      for (int r = 0; r < (int)rank; ++r) off += sm.n_above[r];
      sm.off = off;
    }
  }
  __syncthreads();
  const uint32_t T = sm.T;
  need = sm.need;
  if (need < sm.n_tie) {
    // ties by lower index: the need-th smallest index among the entries equal to T
    // (rare: scores exactly equal to the K-th)
#pragma unroll
    for (int r = 0; r < kTopkRanks; ++r)
      for (int i = tid; i < sm.n_cand[r]; i += NT) {
        const uint2 ci = sm.cand[r][i];
        if (ci.x != T) continue;
        int smaller = 0;
        for (int r2 = 0; r2 < kTopkRanks; ++r2)
          for (int i2 = 0; i2 < sm.n_cand[r2]; ++i2) {
            const uint2 c2 = sm.cand[r2][i2];
            smaller += c2.x == T && (int)c2.y < (int)ci.y;
          }
        if (smaller == need - 1) sm.tie_idx = (int)ci.y;
      }
    __syncthreads();
  }
  const int tie_idx = sm.tie_idx;   // 0x7FFFFFFF when every tie is taken
  {
    // selected candidates of the ranks before this one
    int before = 0;
    for (int r = 0; r < (int)rank; ++r)
      for (int i = tid; i < sm.n_cand[r]; i += NT) {
        const uint2 ci = sm.cand[r][i];
        before += ci.x > T || (ci.x == T && (int)ci.y <= tie_idx);
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
    if (lane == 0 && before) atomicAdd(&sm.off, before);
  }
  __syncthreads();
  const int off = sm.off;

  // ---- this quarter's selection in index order
  uint32_t sel = 0;
#pragma unroll
  for (int u = 0; u < kClPer; ++u) {
    if (j0 + u < q1) {
      const uint32_t key = order_key(x[u]);
      if ((key >> 21) > (uint32_t)bstar || (((cm >> u) & 1u) && (key > T || (key == T && j0 + u <= tie_idx))))
        sel |= 1u << u;
    }
  }
  int p = off + block_exclusive_scan_t<NT>(__popc(sel), sm.warp_tot);
  while (sel) {
    const int u = __ffs(sel) - 1;
    sel &= sel - 1;
    if (p < kk) out[p] = remap_index(remap, row, j0 + u);
    ++p;
  }
}

// ---- many short rows (prefill: one row per query token) ------------------------------
// Rows of at most 32,768 entries, many more rows than SMs: a 256-thread CTA
// per row, six rows per SM, and few instructions per entry.  A sample of the
// row (64 spread runs of 16 entries) gives a lower bound for the K-th key: the
// bin of the sample's r-th largest key, r = 1.5 times the sample's expected
// share of the Top-K plus 8.  One pass over the row then compares every entry with
// that bound as a float and keeps only the entries at or above it (their
// keys, indices and 2048-bin histogram) in shared memory; the exact
// selection (threshold bin, radix passes, ties by lower index, index-ordered
// output) runs over those candidates.  When the bound was too high (fewer
// than K candidates) or too low (more than fit), the row is selected by radix
// passes over the whole row instead.
constexpr int kShortThreads = 256;
constexpr int kShortMaxN = 32768;
constexpr int kShortCap = 2048;     // candidates kept in shared memory
constexpr int kShortBatch = 8;      // row elements per thread loaded before any is used
constexpr int kSample = 1024;       // 64 runs of 16 entries

struct TopkShortSmem {
  uint32_t hist[2048];
  uint32_t hist2[256];
  int warp_tot[kShortThreads / 32];
  int nC, nB;
  uint32_t ckey[kShortCap];
  int32_t cidx[kShortCap];
  uint32_t sel_bits[kShortMaxN / 32];
  uint32_t tie_bits[kShortMaxN / 32];
};

// Element u of the thread's batch: with kVec, four consecutive entries per float4.
template <bool kVec>
__device__ __forceinline__ int batch_index(int j0, int tid, int u) {
  return kVec ? j0 + 4 * ((u >> 2) * kShortThreads + tid) + (u & 3) : j0 + u * kShortThreads + tid;
}
template <bool kVec>
__device__ __forceinline__ void load_batch(const float* __restrict__ s, int n, int j0, int tid,
                                           float (&x)[kShortBatch]) {
  if (kVec) {
#pragma unroll
    for (int u = 0; u < kShortBatch / 4; ++u) {
      const int j = batch_index<true>(j0, tid, 4 * u);
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j + 3 < n) {
        f = *reinterpret_cast<const float4*>(s + j);
      } else if (j < n) {
        f.x = s[j];
        if (j + 1 < n) f.y = s[j + 1];
        if (j + 2 < n) f.z = s[j + 2];
      }
      x[4 * u] = f.x; x[4 * u + 1] = f.y; x[4 * u + 2] = f.z; x[4 * u + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int u = 0; u < kShortBatch; ++u) {
      const int j = batch_index<false>(j0, tid, u);
      x[u] = j < n ? s[j] : 0.f;
    }
  }
}

// Appends the batch's entries at or above f_lo (all of them with take_all) to
// the candidates (one atomic per warp) and adds their keys to the histogram.
template <bool kVec>
__device__ __forceinline__ void collect_batch(TopkShortSmem& sm, const float (&x)[kShortBatch], int j0, int n,
                                              bool take_all, float f_lo, int tid) {
  const int lane = tid & 31;
  uint32_t cm = 0;
#pragma unroll
  for (int u = 0; u < kShortBatch; ++u)
    if (batch_index<kVec>(j0, tid, u) < n && (take_all || x[u] >= f_lo)) cm |= 1u << u;
  const int c = __popc(cm);
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const int wtot = __shfl_sync(0xffffffffu, incl, 31);
  if (wtot) {
    int base = 0;
    if (lane == 31) base = atomicAdd(&sm.nC, wtot);
    base = __shfl_sync(0xffffffffu, base, 31);
    int pos = base + incl - c;
#pragma unroll
    for (int u = 0; u < kShortBatch; ++u) {
      if ((cm >> u) & 1u) {
        const uint32_t key = order_key(x[u]);
        if (pos < kShortCap) {
          sm.ckey[pos] = key;
          sm.cidx[pos] = batch_index<kVec>(j0, tid, u);
        }
        warp_hist_add(sm.hist, key >> 21, 2048);
        ++pos;
      }
    }
  }
}

template <bool kVec>
__global__ void __launch_bounds__(kShortThreads, 6)
k_topk_short(const float* __restrict__ scores, int64_t stride, ValidSpec v, int k, int32_t* __restrict__ out_idx,
             int32_t* __restrict__ out_cnt, Remap remap) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkShortSmem& sm = *reinterpret_cast<TopkShortSmem*>(smem_raw);
  constexpr int NT = kShortThreads;
  constexpr int kStep = kShortBatch * NT;   // entries per batch
  const int64_t row = blockIdx.x;
  const float* s = scores + row * stride;
  const int n = row_valid(v, row, stride);   // <= stride <= kShortMaxN (checked by the launcher)
  const int kk = min(k, n);
  int32_t* out = out_idx + row * (int64_t)k;
  const int tid = threadIdx.x;

  for (int j = kk + tid; j < k; j += NT) out[j] = -1;
  if (tid == 0) out_cnt[row] = kk;
  if (kk == 0) return;
  if (kk == n) {
    for (int j = tid; j < n; j += NT) out[j] = remap_index(remap, row, j);
    return;
  }
  const int words = (n + 31) / 32;
  for (int i = tid; i < words; i += NT) {
    sm.sel_bits[i] = 0;
    sm.tie_bits[i] = 0;
  }
  for (int i = tid; i < 2048; i += NT) sm.hist[i] = 0;
  if (tid == 0) sm.nC = 0;
  __syncthreads();

  // the first batch of the row is requested before the sample is analysed
  float x0[kShortBatch];
  load_batch<kVec>(s, n, 0, tid, x0);
  // ---- lower bound of the K-th key from the sample (rows longer than 2 x the sample)
  bool take_all = true;
  float f_lo = 0.f;
  if (n > 2 * kSample) {
    const int run = tid >> 2;   // 64 runs of 16 entries, thread = 4 of them
    const int j = ((int)(((int64_t)run * (n - 16)) / 63) & ~3) + 4 * (tid & 3);
    float x[4];
    if (kVec) {
      const float4 f = *reinterpret_cast<const float4*>(s + j);
      x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) x[u] = s[j + u];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) warp_hist_add(sm.hist, order_key(x[u]) >> 21, 2048);
    __syncthreads();
    const int r = min(kSample, (int)((3LL * kk * kSample + 2 * n - 1) / (2 * n)) + 8);   // 1.5 x the expected share
    int ab;
    const int b_lo = find_digit_t<NT>(sm.hist, 2048, r, sm.warp_tot, &ab);
    if (b_lo > 0) {
      take_all = false;
      f_lo = key_float((uint32_t)b_lo << 21);
    }
    for (int i = tid; i < 2048; i += NT) sm.hist[i] = 0;
    __syncthreads();
  }

  // ---- one pass: entries at or above the bound -> candidates and their histogram;
  // the next batch is requested before the current one is collected
  for (int j0 = 0; j0 < n; j0 += kStep) {
    float x1[kShortBatch];
    if (j0 + kStep < n) load_batch<kVec>(s, n, j0 + kStep, tid, x1);
    collect_batch<kVec>(sm, x0, j0, n, take_all, f_lo, tid);
#pragma unroll
    for (int u = 0; u < kShortBatch; ++u) x0[u] = x1[u];
  }
  __syncthreads();
  const int nC = sm.nC;
  int above;
  if (nC >= kk && nC <= kShortCap) {   // the candidates hold the Top-K
    const int bstar = find_digit_t<NT>(sm.hist, 2048, kk, sm.warp_tot, &above);
    // higher bins -> selected; the threshold bin's candidates -> a short list
    // (keys in hist[0 .. 1024), indices in hist[1024 ..): the histogram is done)
    if (tid == 0) sm.nB = 0;
    __syncthreads();
    for (int i0 = 0; i0 < nC; i0 += NT) {
      const int i = i0 + tid;
      uint32_t key = 0;
      int32_t j = 0;
      if (i < nC) {
        key = sm.ckey[i];
        j = sm.cidx[i];
        if ((key >> 21) > (uint32_t)bstar) red_or_shared(&sm.sel_bits[j >> 5], 1u << (j & 31));
      }
      const int slot = warp_slot(&sm.nB, i < nC && (key >> 21) == (uint32_t)bstar, 1024);
      if (slot >= 0) {
        sm.hist[slot] = key;
        sm.hist[1024 + slot] = (uint32_t)j;
      }
    }
    __syncthreads();
    const int nB = sm.nB;
    if (nB > 1024) {   // crowded threshold bin: block-wide radix passes over all candidates
      finish_from_candidates<NT>(sm, n, kk, bstar, kk - above, nC, out, remap, row);
      return;
    }
    __shared__ uint32_t s_T;
    __shared__ int s_need;
    if (tid < 32) {
      uint32_t t;
      int nd;
      warp_radix_threshold(sm, sm.hist, nB, bstar, kk - above, &t, &nd);
      if (tid == 0) {
        s_T = t;
        s_need = nd;
      }
    }
    __syncthreads();
    const uint32_t T = s_T;
    for (int i = tid; i < nB; i += NT) {
      const uint32_t key = sm.hist[i];
      const int32_t j = (int32_t)sm.hist[1024 + i];
      if (key > T) red_or_shared(&sm.sel_bits[j >> 5], 1u << (j & 31));
      else if (key == T) red_or_shared(&sm.tie_bits[j >> 5], 1u << (j & 31));
    }
    __syncthreads();
    write_selection<NT>(sm, words, kk, s_need, out, remap, row);
    return;
  }
  // the bound missed: the whole row's histogram, then radix passes over the row
  for (int i = tid; i < 2048; i += NT) sm.hist[i] = 0;
  __syncthreads();
  for (int j0 = 0; j0 < n; j0 += kStep) {
    float x[kShortBatch];
    load_batch<kVec>(s, n, j0, tid, x);
#pragma unroll
    for (int u = 0; u < kShortBatch; ++u)
      warp_hist_add(sm.hist, batch_index<kVec>(j0, tid, u) < n ? order_key(x[u]) >> 21 : 0xFFFFFFFFu, 2048);
  }
  __syncthreads();
  const int bstar = find_digit_t<NT>(sm.hist, 2048, kk, sm.warp_tot, &above);
  radix_whole_row<NT>(sm, s, n, kk, bstar, kk - above, out, remap, row);
}

// ---- split Top-K: few, long rows ---------------------------------------------------
// The collection pass of k_topk spread over many CTAs per row: every CTA
// locates the threshold bin from the row histogram itself, then for its chunk
// of 4,096 entries writes the selection-bitmap words of the higher bins and
// appends the threshold bin's candidates to a per-row list in scratch.  One
// CTA per row then finishes from the candidates (k_topk_finish).
constexpr int kCollectThreads = 256;
constexpr int kCollectChunk = 4096;

__global__ void __launch_bounds__(kCollectThreads)
k_topk_collect(const float* __restrict__ scores, int64_t stride, ValidSpec v, int k,
               const uint32_t* __restrict__ hist_in, int64_t hist_stride, uint32_t* __restrict__ sel_words,
               int64_t words_stride, uint32_t* __restrict__ cand_key, int32_t* __restrict__ cand_idx,
               int32_t* __restrict__ cand_count) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t shist[2048];
  __shared__ int warp_tot[kCollectThreads / 32];
  constexpr int kPer = kCollectChunk / kCollectThreads;   // 16 entries per thread
  const int64_t row = blockIdx.y;
  const float* s = scores + row * stride;
  const int n = row_valid(v, row, stride);
  const int kk = min(k, n);
  const int c0 = blockIdx.x * kCollectChunk;
  if (kk == 0 || kk == n || c0 >= n || n > kBitmapMax) return;
  const int c1 = min(n, c0 + kCollectChunk);
  const int tid = threadIdx.x, lane = tid & 31;
  // the chunk's loads are in flight while the threshold bin is located
  float vv[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int j = c0 + u * kCollectThreads + tid;
    vv[u] = j < c1 ? s[j] : 0.f;
  }
  int bstar, above;
  locate_bin<kCollectThreads>(shist, warp_tot, s, n, kk, hist_in + row * hist_stride, &bstar, &above);
  if ((int)shist[bstar] > kCandCap) return;       // the finish kernel takes the whole-row path
  // the bin's edges as floats: above -> selection word bit, inside -> candidate
  const float f_lo = bstar == 0 ? -INFINITY : key_float((uint32_t)bstar << 21);
  const float f_hi = bstar == 2047 ? __uint_as_float(0x7FFFFFFFu) : key_float((uint32_t)(bstar + 1) << 21);
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int j = c0 + u * kCollectThreads + tid;   // a warp covers one aligned 32-entry word
    const bool in = j < c1;
    const bool sel = in && vv[u] >= f_hi;
    const uint32_t word = __ballot_sync(0xffffffffu, sel);
    if (lane == 0 && in) sel_words[row * words_stride + (j >> 5)] = word;
    const bool cand = in && !sel && vv[u] >= f_lo;
    const uint32_t m = __ballot_sync(0xffffffffu, cand);
    if (m) {
      int base = 0;
      if (lane == __ffs(m) - 1) base = atomicAdd(&cand_count[row], __popc(m));
      base = __shfl_sync(0xffffffffu, base, __ffs(m) - 1);
      const int pos = base + __popc(m & ((1u << lane) - 1));
      if (cand && pos < kCandCap) {
        cand_key[row * kCandCap + pos] = order_key(vv[u]);
        cand_idx[row * kCandCap + pos] = j;
      }
    }
  }
}

__global__ void __launch_bounds__(kTopkThreads)
k_topk_finish(const float* __restrict__ scores, int64_t stride, ValidSpec v, int k, int32_t* __restrict__ out_idx,
              int32_t* __restrict__ out_cnt, Remap remap, const uint32_t* __restrict__ hist_in, int64_t hist_stride,
              const uint32_t* __restrict__ sel_words, int64_t words_stride, const uint32_t* __restrict__ cand_key,
              const int32_t* __restrict__ cand_idx, const int32_t* __restrict__ cand_count) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(smem_raw);
  const int64_t row = blockIdx.x;
  const float* s = scores + row * stride;
  const int n = row_valid(v, row, stride);
  const int kk = min(k, n);
  int32_t* out = out_idx + row * (int64_t)k;
  const int tid = threadIdx.x;
  for (int j = kk + tid; j < k; j += kTopkThreads) out[j] = -1;
  if (tid == 0) out_cnt[row] = kk;
  if (kk == 0) return;
  if (kk == n) {
    for (int j = tid; j < n; j += kTopkThreads) out[j] = remap_index(remap, row, j);
    return;
  }
  int bstar, above;
  locate_bin<kTopkThreads>(sm.hist, sm.warp_tot, s, n, kk, hist_in + row * hist_stride, &bstar, &above);
  const int need = kk - above;
  if ((int)sm.hist[bstar] > kCandCap || n > kBitmapMax) {
    radix_whole_row<kTopkThreads>(sm, s, n, kk, bstar, need, out, remap, row);
    return;
  }
  const int words = (n + 31) / 32;
  const int nC = min(cand_count[row], kCandCap);
  for (int i = tid; i < words; i += kTopkThreads) {
    sm.sel_bits[i] = sel_words[row * words_stride + i];
    sm.tie_bits[i] = 0;
  }
  for (int i = tid; i < nC; i += kTopkThreads) {
    sm.ckey[i] = cand_key[row * kCandCap + i];
    sm.cidx[i] = cand_idx[row * kCandCap + i];
  }
  __syncthreads();
  finish_from_candidates<kTopkThreads, TopkSmem, true>(sm, n, kk, bstar, need, nC, out, remap, row);
}

// 2048-bin key histograms of given score rows (for the split path on a given array).
__global__ void __launch_bounds__(kCollectThreads)
k_row_hist(const float* __restrict__ scores, int64_t stride, ValidSpec v, uint32_t* __restrict__ hist) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t sh[2048];
  const int64_t row = blockIdx.y;
  const int n = row_valid(v, row, stride);
  const int c0 = blockIdx.x * kCollectChunk;
  if (c0 >= n) return;
  const int c1 = min(n, c0 + kCollectChunk);
  for (int i = threadIdx.x; i < 2048; i += kCollectThreads) sh[i] = 0;
  __syncthreads();
  const float* s = scores + row * stride;
  for (int j0 = c0; j0 < c1; j0 += kCollectThreads * kBatch) {
    float vv[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = j0 + u * kCollectThreads + threadIdx.x;
      vv[u] = j < c1 ? s[j] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = j0 + u * kCollectThreads + threadIdx.x;
      warp_hist_add(sh, j < c1 ? order_key(vv[u]) >> 21 : 0xFFFFFFFFu, 2048);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 2048; i += kCollectThreads)
    if (sh[i]) atomicAdd(&hist[row * 2048 + i], sh[i]);
}

cudaError_t launch_row_hist(const float* scores, int64_t rows, int64_t stride, ValidSpec v, uint32_t* hist,
                            cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(hist, 0, (size_t)rows * 2048 * 4, s);
  if (e != cudaSuccess) return e;
  dim3 g((unsigned)((stride + kCollectChunk - 1) / kCollectChunk), (unsigned)rows);
  return launch_step(k_row_hist, g, dim3(kCollectThreads), 0, s, scores, stride, v, hist);
}

size_t topk_split_scratch_bytes(int64_t rows, int64_t stride) {
  const int64_t words = (stride + 31) / 32;
  return (size_t)rows * (words * 4 + (int64_t)kCandCap * 8 + 16);
}

cudaError_t launch_topk_split(const float* scores, int64_t rows, int64_t stride, ValidSpec v, int k,
                              int32_t* out_idx, int32_t* out_cnt, Remap remap, const uint32_t* hist,
                              int64_t hist_stride, void* scratch, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int64_t words = (stride + 31) / 32;
  char* p = static_cast<char*>(scratch);
  uint32_t* cand_key = reinterpret_cast<uint32_t*>(p);
  int32_t* cand_idx = reinterpret_cast<int32_t*>(p + (size_t)rows * kCandCap * 4);
  int32_t* cand_count = reinterpret_cast<int32_t*>(p + (size_t)rows * kCandCap * 8);
  uint32_t* sel_words = reinterpret_cast<uint32_t*>(p + (size_t)rows * kCandCap * 8 + (size_t)rows * 16);
  cudaError_t e = cudaMemsetAsync(cand_count, 0, (size_t)rows * 16, s);
  if (e != cudaSuccess) return e;
  dim3 g1((unsigned)((stride + kCollectChunk - 1) / kCollectChunk), (unsigned)rows);
  e = launch_step(k_topk_collect, g1, dim3(kCollectThreads), 0, s, scores, stride, v, k, hist, hist_stride,
                  sel_words, words, cand_key, cand_idx, cand_count);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(TopkSmem);
  e = cudaFuncSetAttribute(k_topk_finish, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_step(k_topk_finish, dim3((unsigned)rows), dim3(kTopkThreads), smem, s, scores, stride, v, k, out_idx,
                     out_cnt, remap, hist, hist_stride, sel_words, words, cand_key, cand_idx, cand_count);
}

// Block maxima: out[row][b] = max of scores[row][8b .. 8b+7] over the valid
// columns, for b < ceil(n_valid / block).
__global__ void k_block_max(const float* __restrict__ scores, int64_t stride, ValidSpec v, int block,
                            float* __restrict__ out, int64_t out_stride) {
  pdl_trigger();
  pdl_wait();
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
                        int32_t* out_idx, int32_t* out_cnt, Remap remap, const uint32_t* hist,
                        int64_t hist_stride, cudaStream_t s, int64_t max_n) {
  if (rows == 0) return cudaSuccess;
  const int64_t span = (max_n > 0 && max_n < stride) ? max_n : stride;   // longest valid row
  const size_t smem = sizeof(TopkSmem);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (rows >= 2 * (int64_t)sms && stride <= kShortMaxN) {   // many short rows
    const size_t ssm = sizeof(TopkShortSmem);
    const bool vec = (reinterpret_cast<uintptr_t>(scores) & 15) == 0 && stride % 4 == 0;
    if (vec) {
      e = cudaFuncSetAttribute(k_topk_short<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
      if (e != cudaSuccess) return e;
      return launch_step(k_topk_short<true>, dim3((unsigned)rows), dim3(kShortThreads), ssm, s, scores, stride, v, k,
                         out_idx, out_cnt, remap);
    }
    e = cudaFuncSetAttribute(k_topk_short<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
    if (e != cudaSuccess) return e;
    return launch_step(k_topk_short<false>, dim3((unsigned)rows), dim3(kShortThreads), ssm, s, scores, stride, v, k,
                       out_idx, out_cnt, remap);
  }
  if (hist && rows * kTopkRanks <= sms && span <= kClusterMaxN && span > kTopkThreads * 8 &&
      k <= kClusterCap / kTopkRanks) {
    // a cluster per row (few rows with a histogram, K <= 512: decode).  A larger K (the block
    // pool's 2,048 blocks) crowds the threshold bin past the cluster's candidate store, and
    // one CTA per row (k_topk_hist, below) is faster there: 29 against 55 us for 8 rows.
    const bool vec = (reinterpret_cast<uintptr_t>(scores) & 15) == 0 && stride % 4 == 0;
    const size_t csm = sizeof(TopkClusterSmem);
    auto kern = vec ? k_topk_cluster<true> : k_topk_cluster<false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csm);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows * kTopkRanks));
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = csm;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = kTopkRanks;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return counted(cudaLaunchKernelEx(&cfg, kern, scores, stride, v, k, out_idx, out_cnt, remap, hist, hist_stride));
  }
  if (rows <= sms && (hist ? span <= kBitmapMax : span <= (int64_t)kTopkThreads * kHistBatch)) {
    const bool vec = (reinterpret_cast<uintptr_t>(scores) & 15) == 0 && stride % 4 == 0;
    if (vec) {
      e = cudaFuncSetAttribute(k_topk_hist<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      return launch_step(k_topk_hist<true>, dim3((unsigned)rows), dim3(kTopkThreads), smem, s, scores, stride, v, k,
                         out_idx, out_cnt, remap, hist, hist_stride, status_word());
    }
    e = cudaFuncSetAttribute(k_topk_hist<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_step(k_topk_hist<false>, dim3((unsigned)rows), dim3(kTopkThreads), smem, s, scores, stride, v, k,
                       out_idx, out_cnt, remap, hist, hist_stride, status_word());
  }
  if (rows <= sms) {   // one wave of rows: latency counts, occupancy does not
    e = cudaFuncSetAttribute(k_topk<32, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_step(k_topk<32, 1>, dim3((unsigned)rows), dim3(kTopkThreads), smem, s, scores, stride, v, k,
                       out_idx, out_cnt, remap, hist, hist_stride);
  }
  e = cudaFuncSetAttribute(k_topk<8, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_step(k_topk<8, 2>, dim3((unsigned)rows), dim3(kTopkThreads), smem, s, scores, stride, v, k, out_idx,
                     out_cnt, remap, hist, hist_stride);
}

cudaError_t launch_block_max(const float* scores, int64_t rows, int64_t stride, ValidSpec v, int block,
                             float* out, int64_t out_stride, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int64_t nb = (stride + block - 1) / block;
  dim3 grid((unsigned)((nb + 255) / 256), (unsigned)rows);
  return launch_step(k_block_max, grid, dim3(256), 0, s, scores, stride, v, block, out, out_stride);
}

}  // namespace csa2
