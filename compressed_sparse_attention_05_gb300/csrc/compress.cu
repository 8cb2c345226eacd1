// 4:1 sequence compression: every 4 consecutive new tokens become one KV
// entry through a learned linear map ("DeepSeek-V4.1 架构解析" §02; DeepSeek V4
// review §2.1-§2.2), reading R1: c_j = W [h_4j; h_4j+1; h_4j+2; h_4j+3].
// The same GEMM with one token per row projects the replayed tokens onto
// their window rows (SWA Bounded Replay, §03; reading R13).
//
// The g-token concatenation (g = 4, or 1 for window rows) is a plain view of
// the row-major hidden states (row j of A starts at token g j), so A needs no
// gather.  The GEMM computes
// [W; W_idx] (d + Di output channels) in one pass over A and writes split-K
// fp32 partials; the epilogue kernel (pack.cu) sums the splits in a fixed
// order, applies RMSNorm + RoPE + MXFP4 and stores the paged entry and its
// indexer key.  The main kernel runs on the fifth-generation tensor cores
// (tcgen05, TMA-fed); an mma.sync kernel (m16n8k16 bf16, fp32 accumulate,
// 128x128x32 CTA tiles, cp.async double buffering) takes the shapes it does
// not (d not a multiple of 128, H not a multiple of 16).
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tma.cuh"

namespace csa2 {

constexpr int kGM = 128, kGN = 128, kGK = 32;
constexpr int kGThreads = 256;
constexpr int kGS = kGK + 8;  // smem row stride (elements): 80 B, conflict-free ldmatrix

__device__ __forceinline__ uint32_t g_smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // zero-fill when invalid
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n"); }

__device__ __forceinline__ void g_ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void g_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                      uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// grid = (N tiles, M tiles, splits).  8 warps as 2 (M) x 4 (N), warp tile 64 x 32.
__global__ void __launch_bounds__(kGThreads)
k_compress_gemm(const uint16_t* __restrict__ hidden, int G, int T, int H, const uint16_t* __restrict__ W,
                int d, const uint16_t* __restrict__ W_idx, int Di, int M, float* __restrict__ partials,
                int tok_per_row) {
  __shared__ __align__(16) uint16_t sa[2][kGM * kGS];
  __shared__ __align__(16) uint16_t sb[2][kGN * kGS];
  const int N = d + Di;
  const int64_t Kd = (int64_t)tok_per_row * H;
  const int m0 = blockIdx.y * kGM, n0 = blockIdx.x * kGN;
  // split blockIdx.z of gridDim.z takes K steps [st0, st1)
  const int steps = (int)(Kd / kGK);
  const int st0 = (int)((int64_t)blockIdx.z * steps / gridDim.z), st1 = (int)((int64_t)(blockIdx.z + 1) * steps / gridDim.z);
  const int kbeg = st0 * kGK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 2, wn = warp & 3;

  // each thread copies 2 x 16 B of A and of B per stage
  const uint16_t* a_src[2];
  const uint16_t* b_src[2];
  bool a_ok[2], b_ok[2];
  int ld_row[2], ld_col[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int c = tid + i * kGThreads;     // 0..511
    ld_row[i] = c >> 2;                    // 0..127
    ld_col[i] = (c & 3) * 8;               // 0, 8, 16, 24
    const int m = m0 + ld_row[i];
    a_ok[i] = m < M;
    const int mm = a_ok[i] ? m : 0;
    a_src[i] = hidden + ((int64_t)(mm / G) * T + (int64_t)tok_per_row * (mm % G)) * H;
    const int n = n0 + ld_row[i];
    b_ok[i] = n < N;
    b_src[i] = n < d ? W + (int64_t)n * Kd : W_idx + (int64_t)((b_ok[i] ? n : d) - d) * Kd;
    if (!b_ok[i]) b_src[i] = W;
  }
  auto load_stage = [&](int st, int k0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      cp_async16(g_smem_u32(&sa[st][ld_row[i] * kGS + ld_col[i]]), a_src[i] + k0 + ld_col[i], a_ok[i]);
      cp_async16(g_smem_u32(&sb[st][ld_row[i] * kGS + ld_col[i]]), b_src[i] + k0 + ld_col[i], b_ok[i]);
    }
    cp_async_commit();
  };

  float acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;

  const int n_iter = st1 - st0;
  if (n_iter > 0) load_stage(0, kbeg);
  for (int it = 0; it < n_iter; ++it) {
    const int st = it & 1;
    cp_async_wait_all();
    __syncthreads();
    if (it + 1 < n_iter) load_stage(st ^ 1, kbeg + (it + 1) * kGK);
#pragma unroll
    for (int ks = 0; ks < kGK / 16; ++ks) {
      uint32_t af[4][4];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int r = wm * 64 + mt * 16 + (lane & 15);
        g_ldsm_x4(g_smem_u32(&sa[st][r * kGS + ks * 16 + (lane >> 4) * 8]), af[mt][0], af[mt][1],
                  af[mt][2], af[mt][3]);
      }
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int mi = lane >> 3, r8 = lane & 7;
        const int r = wn * 32 + np * 16 + (mi >> 1) * 8 + r8;
        uint32_t b0, b1, b2, b3;
        g_ldsm_x4(g_smem_u32(&sb[st][r * kGS + ks * 16 + (mi & 1) * 8]), b0, b1, b2, b3);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          g_mma(acc[mt][2 * np], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1);
          g_mma(acc[mt][2 * np + 1], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b2, b3);
        }
      }
    }
    __syncthreads();
  }
  float* out = partials + (int64_t)blockIdx.z * M * N;
  const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int m = m0 + wm * 64 + mt * 16 + g;
      const int n = n0 + wn * 32 + nt * 8 + 2 * t4;
      if (n < N) {
        if (m < M) *reinterpret_cast<float2*>(out + (int64_t)m * N + n) = make_float2(acc[mt][nt][0], acc[mt][nt][1]);
        if (m + 8 < M)
          *reinterpret_cast<float2*>(out + (int64_t)(m + 8) * N + n) = make_float2(acc[mt][nt][2], acc[mt][nt][3]);
      }
    }
}

// ---- tcgen05 + TMA path -------------------------------------------------------------
// CTA tile 128 entries x 256 output channels; K in 64-wide stages of 48 KB
// (A then B, both 128-byte-swizzled K-major) in a 4-stage ring filled by
// tensor-map copies: A is the hidden states seen as [B][G][gH] (row j of
// batch b starts at token g j), B is W or W_idx (W_idx tiles hold Di rows;
// the tile's other columns are never stored).  Warp 0 issues the copies,
// warp 1 the MMAs (M = 128, N = 256, K = 16) into a 256-column fp32
// accumulator in tensor memory, warps 2..5 write the fp32 partial sums.
// Split K: grid.z = B x n_split, split s takes stages [s n / n_split,
// (s + 1) n / n_split).  Every wait is bounded.
//
// kMc > 1: the kMc CTAs of a cluster take consecutive M tiles of the same N
// tile; each copies 1/kMc of the B tile and multicasts it to all of them, so
// that a CTA reads 16 KB + 32/kMc KB per stage from L2 instead of 48 KB.  A
// stage is refilled only once every CTA of the cluster has released it (each
// CTA's MMA commit arrives on the stage's empty barrier of all of them).
constexpr int kTmM = 128, kTmN = 256, kTmK = 64, kTmStages = 4;
constexpr int kTmABytes = kTmM * kTmK * 2;                 // 16 KB
constexpr int kTmStageBytes = kTmABytes + kTmN * kTmK * 2;   // 48 KB
constexpr int kTmEpiWarps = 4;
constexpr int kTmThreads = (2 + kTmEpiWarps) * 32;
constexpr int kTmSmsTarget = 152;   // splits fill this many SMs once (the GPU's SM count)

struct CompressSmem {
  unsigned char ring[kTmStages][kTmStageBytes];
  uint64_t full[kTmStages], empty[kTmStages], acc_full;
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort) return false;
  }
  *abort = 1;
  return false;
}

template <int kMc>
__global__ void __launch_bounds__(kTmThreads, 1)
k_compress_gemm_tma(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap wmap,
                    const __grid_constant__ CUtensorMap imap, int G, int d, int Di, int N, int M, int n_stages,
                    int n_split, float* __restrict__ partials, uint32_t* status) {
  extern __shared__ unsigned char smem_raw[];
  pdl_trigger();
  pdl_wait();
  const uint32_t pad = (1024u - (tc::smem_addr(smem_raw) & 1023u)) & 1023u;
  CompressSmem& sm = *reinterpret_cast<CompressSmem*>(smem_raw + pad);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * kTmN, j0 = blockIdx.y * kTmM;
  const int b = blockIdx.z / n_split, split = blockIdx.z % n_split;
  const int s0 = (int)((int64_t)split * n_stages / n_split);
  const int my = (int)((int64_t)(split + 1) * n_stages / n_split) - s0;

  if (tid == 0) {
    for (int i = 0; i < kTmStages; ++i) {
      tc::mbar_init(&sm.full[i], 1);
      tc::mbar_init(&sm.empty[i], kMc);
    }
    tc::mbar_init(&sm.acc_full, 1);
    sm.abort = 0;
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(&sm.tmem, kTmN);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (kMc > 1) tc::cluster_barrier();   // every CTA's barriers exist before a peer copies or arrives into them
  const uint32_t crank = kMc > 1 ? tc::cluster_ctarank() : 0;
  constexpr uint16_t kMask = (uint16_t)((1u << kMc) - 1);
  constexpr int kBRows = kTmN / kMc;   // B rows this CTA copies (kMc > 1)
  const uint32_t tm = sm.tmem;
  volatile int* abort = &sm.abort;

  if (warp == 0) {
    // ================= producer =================
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < my; ++i) {
        const int st = i % kTmStages;
        if (i >= kTmStages && !wait_or_abort(&sm.empty[st], ((i / kTmStages) - 1) & 1, abort)) break;
        const int kx = (s0 + i) * kTmK;
        if (kMc > 1) {
          // the B tile's rows held by W (or W_idx) in parts of kBRows; the parts past them are not copied
          const int rows = n0 < d ? min(kTmN, d - n0) : Di;
          const int parts = (rows + kBRows - 1) / kBRows;
          tc::mbar_arrive_expect_tx(&sm.full[st], (uint32_t)(kTmABytes + parts * kBRows * kTmK * 2));
          tma::load_3d(sm.ring[st], &amap, kx, j0, b, &sm.full[st]);
          if ((int)crank < parts) {
            unsigned char* bdst = sm.ring[st] + kTmABytes + crank * (kBRows * kTmK * 2);
            if (n0 < d) tma::load_2d_mc(bdst, &wmap, kx, n0 + (int)crank * kBRows, &sm.full[st], kMask);
            else tma::load_2d_mc(bdst, &imap, kx, n0 - d + (int)crank * kBRows, &sm.full[st], kMask);
          }
        } else {
          tc::mbar_arrive_expect_tx(&sm.full[st], (uint32_t)(kTmABytes + (n0 < d ? kTmN : Di) * kTmK * 2));
          tma::load_3d(sm.ring[st], &amap, kx, j0, b, &sm.full[st]);
          if (n0 < d) tma::load_2d(sm.ring[st] + kTmABytes, &wmap, kx, n0, &sm.full[st]);
          else tma::load_2d(sm.ring[st] + kTmABytes, &imap, kx, n0 - d, &sm.full[st]);
        }
        issued = i + 1;
      }
      for (int i = max(0, issued - kTmStages); i < issued; ++i)   // every issued copy lands before exit
        for (uint32_t k = 0; k < (1u << 22); ++k)
          if (tc::mbar_try_wait(&sm.full[i % kTmStages], (i / kTmStages) & 1)) break;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issue =================
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_f16(kTmM, kTmN, 1, 0, 0);   // bf16, K-major A and B
      for (int i = 0; i < my; ++i) {
        const int st = i % kTmStages;
        if (!wait_or_abort(&sm.full[st], (i / kTmStages) & 1, abort)) break;
        tc::tc_fence_after();
        const uint32_t sa = tc::smem_addr(sm.ring[st]), sb = sa + kTmABytes;
#pragma unroll
        for (int ks = 0; ks < kTmK / 16; ++ks) {
          const uint64_t ad = tc::smem_desc(sa + ks * 32, 16, 1024) | ((uint64_t)2 << 61);
          const uint64_t bd = tc::smem_desc(sb + ks * 32, 16, 1024) | ((uint64_t)2 << 61);
          tc::mma_f16(tm, ad, bd, idesc, (i > 0 || ks > 0) ? 1u : 0u);
        }
        if (kMc > 1) tc::mma_commit_mc(&sm.empty[st], kMask);   // the stage is free in this CTA
        else tc::mma_commit(&sm.empty[st]);
      }
      tc::mma_commit(&sm.acc_full);   // arrives once every MMA issued above is complete
    }
    __syncwarp();
  } else {
    // ================= epilogue: warp w reads lane quarter w % 4 =================
    const int q = warp & 3;
    const bool ok = __all_sync(0xffffffffu, wait_or_abort(&sm.acc_full, 0, abort));
    tc::tc_fence_after();
    if (ok && !*abort && my > 0) {
      const int j = j0 + 32 * q + lane;
      float* out = partials + ((int64_t)split * M + (int64_t)b * G + j) * N + n0;
#pragma unroll 1
      for (int c = 0; c < kTmN; c += 16) {
        float v[16];
        tc::tmem_ld16(tm + ((uint32_t)(32 * q) << 16) + c, v);
        tc::tmem_wait_ld();
        if (j < G) {
#pragma unroll
          for (int u = 0; u < 16; u += 4)
            if (n0 + c + u < N) *reinterpret_cast<float4*>(out + c + u) = make_float4(v[u], v[u + 1], v[u + 2], v[u + 3]);
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (kMc > 1) tc::cluster_barrier();   // no copy or commit of a peer still targets this CTA
  if (warp == 1) tc::tmem_dealloc(tm, kTmN);
  if (tid == 0 && *abort) raise_status(status, CSA2_STATUS_TIMEOUT);
}

// W_idx tiles start on a tile (d a multiple of 256); without W_idx any d >= 256 with
// 16-byte rows of output works (the last tile's rows past d are zero-filled).  The
// K stages tile g H exactly.
static bool tma_compress_ok(int T, int H, int d, int Di, int g) {
  return (Di ? d % kTmN == 0 : (d >= kTmN && d % 4 == 0)) && H % 16 == 0 && (g * H) % kTmK == 0 && T >= g &&
         Di % 4 == 0 && Di <= kTmN && tensor_map_encoder() != nullptr;
}

// Split K only as far as it takes to fill the SMs once.
static int compress_splits(int B, int G, int N, int Kd) {
  const int64_t tiles = (int64_t)B * ((G + kTmM - 1) / kTmM) * ((N + kTmN - 1) / kTmN);
  const int64_t s = std::max<int64_t>(1, kTmSmsTarget / std::max<int64_t>(1, tiles));
  return (int)std::min<int64_t>(s, std::max(1, Kd / kTmK));
}

size_t compress_partials_bytes(int B, int T, int H, int d, int Di, int* n_split_out, int g) {
  const int G = T / g, M = B * G, N = d + Di, Kd = g * H;
  const int sp = compress_splits(B, G, N, Kd);
  if (n_split_out) *n_split_out = sp;
  return (size_t)sp * M * N * sizeof(float);
}

cudaError_t launch_compress_gemm(const uint16_t* hidden, int B, int T, int H, const uint16_t* W, int d,
                                 const uint16_t* W_idx, int Di, float* partials, int n_split,
                                 cudaStream_t s, int g) {
  const int G = T / g, M = B * G, N = d + (W_idx ? Di : 0), Kd = g * H;
  if (M == 0) return cudaSuccess;
  if (tma_compress_ok(T, H, d, W_idx ? Di : 0, g)) {
    // A: [B][G][gH] view of the hidden states; W: [d][gH]; W_idx: [Di][gH]
    CUtensorMap amap, wmap, imap;
    const cuuint32_t estr[3] = {1, 1, 1};
    const cuuint64_t adims[3] = {(cuuint64_t)Kd, (cuuint64_t)G, (cuuint64_t)B};
    const cuuint64_t astr[2] = {(cuuint64_t)Kd * 2, (cuuint64_t)T * H * 2};
    const cuuint32_t abox[3] = {kTmK, kTmM, 1};
    const cuuint64_t wdims[2] = {(cuuint64_t)Kd, (cuuint64_t)d};
    const cuuint64_t wstr[1] = {(cuuint64_t)Kd * 2};
    // clusters of mc CTAs along M share each B tile (each copies and multicasts 1/mc of it)
    const int m_tiles = (G + kTmM - 1) / kTmM;
    const int mc = m_tiles % 4 == 0 ? 4 : (m_tiles % 2 == 0 ? 2 : 1);
    const cuuint32_t wbox[2] = {kTmK, (cuuint32_t)(kTmN / mc)};
    const cuuint64_t idims[2] = {(cuuint64_t)Kd, (cuuint64_t)(W_idx ? Di : d)};
    const cuuint32_t ibox[2] = {kTmK, (cuuint32_t)(mc > 1 ? kTmN / mc : (W_idx ? Di : kTmN))};
    EncodeTiled enc = tensor_map_encoder();
    if (enc(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(hidden), adims, astr, abox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(W), wdims, wstr, wbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&imap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(W_idx ? W_idx : W), idims, wstr, ibox,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    const size_t smem = sizeof(CompressSmem) + 1024;
    auto kernel = mc == 4 ? k_compress_gemm_tma<4> : (mc == 2 ? k_compress_gemm_tma<2> : k_compress_gemm_tma<1>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + kTmN - 1) / kTmN, m_tiles, B * n_split);
    cfg.blockDim = dim3(kTmThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = 1;
    at[1].val.clusterDim.y = (unsigned)mc;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = mc > 1 ? 2 : 1;
    return counted(cudaLaunchKernelEx(&cfg, kernel, amap, wmap, imap, G, d, W_idx ? Di : 0, N, M, Kd / kTmK, n_split,
                                      partials, status_word()));
  }
  dim3 grid((N + kGN - 1) / kGN, (M + kGM - 1) / kGM, n_split);
  k_compress_gemm<<<grid, kGThreads, 0, s>>>(hidden, G, T, H, W, d, W_idx, W_idx ? Di : 0, M, partials, g);
  return counted(cudaGetLastError());
}

}  // namespace csa2
