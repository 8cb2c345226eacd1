// 4:1 sequence compression: every 4 consecutive new tokens become one KV
// entry through a learned linear map ("DeepSeek-V4.1 架构解析" §02; DeepSeek V4
// review §2.1-§2.2), reading R1: c_j = W [h_4j; h_4j+1; h_4j+2; h_4j+3].
//
// The 4-token concatenation is a plain view of the row-major hidden states
// (row j of A starts at token 4j), so A needs no gather.  The GEMM computes
// [W; W_idx] (d + Di output channels) in one pass over A and writes split-K
// fp32 partials; the epilogue kernel (pack.cu) sums the splits in a fixed
// order, applies RMSNorm + RoPE + MXFP4 and stores the paged entry and its
// indexer key.  Tensor cores: m16n8k16 bf16, fp32 accumulate, 128x128x32
// CTA tiles, cp.async double buffering.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

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
                int d, const uint16_t* __restrict__ W_idx, int Di, int M, int k_per_split,
                float* __restrict__ partials) {
  __shared__ __align__(16) uint16_t sa[2][kGM * kGS];
  __shared__ __align__(16) uint16_t sb[2][kGN * kGS];
  const int N = d + Di;
  const int64_t Kd = 4LL * H;
  const int m0 = blockIdx.y * kGM, n0 = blockIdx.x * kGN;
  const int kbeg = blockIdx.z * k_per_split;
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
    a_src[i] = hidden + ((int64_t)(mm / G) * T + 4LL * (mm % G)) * H;
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

  const int n_iter = k_per_split / kGK;
  load_stage(0, kbeg);
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

// ---- tcgen05 path ----------------------------------------------------------------
// CTA tile 128 (M) x 128 (N) x 64 (K) per stage, 4-stage ring of operands in the
// 128-byte-swizzled K-major layout (8-row atoms of 1024 B, 16-byte chunk index
// XOR row % 8) written by cp.async; thread 0 issues tcgen05.mma (M=128, N=128,
// K=16) into a 128-column fp32 TMEM accumulator and commits each stage to an
// mbarrier that frees its buffers.  Every wait is bounded.
constexpr int kTcM = 128, kTcN = 128, kTcK = 64, kTcStages = 4, kTcThreads = 128;
constexpr int kTcStageBytes = (kTcM + kTcN) * kTcK * 2;   // 32 KB

__global__ void __launch_bounds__(kTcThreads)
k_compress_gemm_tc(const uint16_t* __restrict__ hidden, int G, int T, int H, const uint16_t* __restrict__ W,
                   int d, const uint16_t* __restrict__ W_idx, int Di, int M, int k_per_split,
                   float* __restrict__ partials, uint32_t* status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t bar_free[kTcStages];
  __shared__ uint64_t bar_done;
  __shared__ uint32_t tmem_slot;
  pdl_trigger();
  pdl_wait();
  const uint32_t pad = (1024u - (tc::smem_addr(smem_raw) & 1023u)) & 1023u;
  unsigned char* ring = smem_raw + pad;
  const int N = d + Di;
  const int64_t Kd = 4LL * H;
  const int m0 = blockIdx.y * kTcM, n0 = blockIdx.x * kTcN;
  const int kbeg = blockIdx.z * k_per_split;
  const int n_iter = k_per_split / kTcK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < kTcStages; ++i) tc::mbar_init(&bar_free[i], 1);
    tc::mbar_init(&bar_done, 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, kTcN);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // row sources: this thread copies rows (tid / 8) + 16 i, 16-byte chunk tid % 8
  const int c16 = tid & 7;
  auto stage_ptr = [&](int st) { return ring + st * kTcStageBytes; };
  auto issue_loads = [&](int st, int k0) {
    unsigned char* sa = stage_ptr(st);
    unsigned char* sb = sa + kTcM * kTcK * 2;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = (tid >> 3) + 16 * i;
      const uint32_t off = (r >> 3) * 1024 + (r & 7) * 128 + ((c16 ^ (r & 7)) << 4);
      const int m = m0 + r;
      const bool okA = m < M;
      const int mm = okA ? m : 0;
      const uint16_t* ga = hidden + ((int64_t)(mm / G) * T + 4LL * (mm % G)) * H + k0 + c16 * 8;
      const int n = n0 + r;
      const bool okB = n < N;
      const uint16_t* gb = !okB ? W : (n < d ? W + (int64_t)n * Kd : W_idx + (int64_t)(n - d) * Kd);
      gb += okB ? k0 + c16 * 8 : 0;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(tc::smem_addr(sa + off)), "l"(ga),
                   "r"(okA ? 16 : 0));
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(tc::smem_addr(sb + off)), "l"(gb),
                   "r"(okB ? 16 : 0));
    }
    asm volatile("cp.async.commit_group;\n");
  };

  constexpr uint32_t idesc = tc::idesc_f16(kTcM, kTcN, 1, 0, 0);
  bool ok = true;
  // prologue: stages 0 .. S-2
  for (int i = 0; i < kTcStages - 1; ++i) {
    if (i < n_iter) issue_loads(i, kbeg + i * kTcK);
    else asm volatile("cp.async.commit_group;\n");
  }
  for (int it = 0; it < n_iter; ++it) {
    // refill the stage that chunk it + S - 1 goes to, once its previous MMA is done;
    // the block votes so that every thread takes the same branch after a timeout
    const int nxt = it + kTcStages - 1;
    bool okw = true;
    if (nxt < n_iter && nxt >= kTcStages) okw = tc::mbar_wait(&bar_free[nxt % kTcStages], ((nxt / kTcStages) - 1) & 1);
    ok = __syncthreads_and(okw) != 0;
    if (!ok) break;
    if (nxt < n_iter) issue_loads(nxt % kTcStages, kbeg + nxt * kTcK);
    else asm volatile("cp.async.commit_group;\n");
    asm volatile("cp.async.wait_group %0;\n" ::"n"(kTcStages - 1));
    tc::fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::tc_fence_after();
      const int st = it % kTcStages;
      const uint32_t sa = tc::smem_addr(stage_ptr(st));
      const uint32_t sb = sa + kTcM * kTcK * 2;
#pragma unroll
      for (int ks = 0; ks < kTcK / 16; ++ks) {
        const uint64_t ad = tc::smem_desc(sa + ks * 32, 16, 1024) | ((uint64_t)2 << 61);
        const uint64_t bd = tc::smem_desc(sb + ks * 32, 16, 1024) | ((uint64_t)2 << 61);
        tc::mma_f16(tmem, ad, bd, idesc, (it > 0 || ks > 0) ? 1u : 0u);
      }
      tc::mma_commit(&bar_free[st]);
      if (it == n_iter - 1) tc::mma_commit(&bar_done);
    }
  }
  asm volatile("cp.async.wait_group 0;\n");
  if (ok && n_iter > 0) ok = __syncthreads_and(tc::mbar_wait(&bar_done, 0)) != 0;
  if (!ok && tid == 0) raise_status(status, CSA2_STATUS_TIMEOUT);
  tc::tc_fence_after();
  if (ok && n_iter > 0) {
    // epilogue: lane (32 warp + lane) holds row m0 + 32 warp + lane
    const int m = m0 + warp * 32 + lane;
    float* out = partials + (int64_t)blockIdx.z * M * N + (int64_t)m * N + n0;
#pragma unroll 1
    for (int c = 0; c < kTcN; c += 16) {
      float v[16];
      tc::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c, v);
      tc::tmem_wait_ld();
      if (m < M) {
#pragma unroll
        for (int q = 0; q < 16; q += 4)
          if (n0 + c + q < N) *reinterpret_cast<float4*>(out + c + q) = make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTcN);
}

// The tensor-memory GEMM is used once its operand layout has been checked on
// the GPU; the mma.sync kernel stays for shapes it does not take.
constexpr bool kUseTcCompress = true;

static int compress_splits(int M, int N, int Kd) {
  const int tiles = ((M + kGM - 1) / kGM) * ((N + kGN - 1) / kGN);
  int splits = 1;
  // aim for about one wave of 152 SMs while each split keeps >= 1024 of K
  // (a multiple of the 64-wide K stage of both kernels)
  while (tiles * splits < 152 && Kd / (splits * 2) >= 1024 && (Kd / (splits * 2)) % 64 == 0) splits *= 2;
  return splits;
}

size_t compress_partials_bytes(int B, int T, int H, int d, int Di, int* n_split_out) {
  const int M = B * (T / 4), N = d + Di, Kd = 4 * H;
  const int sp = compress_splits(M, N, Kd);
  if (n_split_out) *n_split_out = sp;
  return (size_t)sp * M * N * sizeof(float);
}

cudaError_t launch_compress_gemm(const uint16_t* hidden, int B, int T, int H, const uint16_t* W, int d,
                                 const uint16_t* W_idx, int Di, float* partials, int n_split,
                                 cudaStream_t s) {
  const int G = T / 4, M = B * G, N = d + (W_idx ? Di : 0), Kd = 4 * H;
  if (M == 0) return cudaSuccess;
  dim3 grid((N + kGN - 1) / kGN, (M + kGM - 1) / kGM, n_split);
  if (kUseTcCompress && (Kd / n_split) % kTcK == 0) {
    const size_t smem = kTcStages * kTcStageBytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(k_compress_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_step(k_compress_gemm_tc, grid, dim3(kTcThreads), smem, s, hidden, G, T, H, W, d, W_idx,
                       W_idx ? Di : 0, M, Kd / n_split, partials, status_word());
  }
  k_compress_gemm<<<grid, kGThreads, 0, s>>>(hidden, G, T, H, W, d, W_idx, W_idx ? Di : 0, M,
                                             Kd / n_split, partials);
  return counted(cudaGetLastError());
}

}  // namespace csa2
