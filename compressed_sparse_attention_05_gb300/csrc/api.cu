// C ABI of the CSA2 layer step (include/csa2.h): host-side validation,
// workspace carving and the order in which one layer step launches its
// kernels.  Nothing here allocates device memory or synchronises a stream
// (except csa2_get_status, which reads the status word back).
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace csa2 {

__device__ uint32_t g_status_word;

static thread_local char g_err[512];

// NVTX range over one entry point (its validation and kernel launches), so that a
// profiler timeline groups each launch under the call that made it.  Costs a
// function call when no tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

static int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

static int cuda_fail(cudaError_t e, const char* what) {
  return fail(CSA2_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Unique id of the calling thread's current CUDA context (0 if there is none).
// Module globals (the status word, the no-allocation scratch) get a new
// device address whenever the context is re-created (cudaDeviceReset), so
// their cached addresses are keyed on this id rather than on the device
// ordinal.  The driver calls are reached through the runtime (no libcuda link).
static unsigned long long current_context_id() {
  using GetCurrent = int (*)(void**);
  using GetId = int (*)(void*, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != 0 || !ctx || get_id(ctx, &id) != 0) return 0;
  return id;
}

void* symbol_address_cached(const void* symbol, cudaError_t* err) {
  static std::mutex mu;
  struct Entry {
    unsigned long long ctx;
    const void* symbol;
    void* addr;
  };
  static Entry cache[128];
  static int n = 0;
  *err = cudaSuccess;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (ctx)
    for (int i = 0; i < n; ++i)
      if (cache[i].ctx == ctx && cache[i].symbol == symbol) return cache[i].addr;
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, symbol);
  if (*err != cudaSuccess) return nullptr;
  if (ctx) {
    const int slot = n < 128 ? n++ : (int)(ctx % 128);
    cache[slot] = Entry{ctx, symbol, p};
  }
  return p;
}

uint32_t* status_word() {
  cudaError_t e;
  return static_cast<uint32_t*>(symbol_address_cached(reinterpret_cast<const void*>(&g_status_word), &e));
}

static std::atomic<uint64_t> g_launches{0};

cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

#define REQUIRE(cond, ...)                                   \
  do {                                                       \
    if (!(cond)) return fail(CSA2_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)
#define REQUIRE_PTR(p)                                                              \
  do {                                                                              \
    if (!(p)) return fail(CSA2_ERR_INVALID_ARG, "%s must not be NULL", #p);         \
    if (!aligned16(p)) return fail(CSA2_ERR_INVALID_ARG, "%s must be 16-byte aligned", #p); \
  } while (0)
// int32 index / count / position arrays are read element-wise: 4-byte alignment
#define REQUIRE_IPTR(p)                                                             \
  do {                                                                              \
    if (!(p)) return fail(CSA2_ERR_INVALID_ARG, "%s must not be NULL", #p);         \
    if (reinterpret_cast<uintptr_t>(p) & 3u)                                        \
      return fail(CSA2_ERR_INVALID_ARG, "%s must be 4-byte aligned", #p);           \
  } while (0)
#define LAUNCH(expr, what)                          \
  do {                                              \
    cudaError_t e_ = (expr);                        \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

static int check_dims(const csa2_dims* dm, bool need_indexer, bool need_attn) {
  REQUIRE(dm, "dims must not be NULL");
  REQUIRE(dm->B >= 0 && dm->Tq >= 0, "B and Tq must be >= 0");
  REQUIRE(dm->max_pages >= 1, "max_pages must be >= 1");
  if (need_indexer) {
    REQUIRE(dm->Hi >= 1 && dm->Hi <= 16, "Hi must be in 1..16 (got %d)", dm->Hi);
    REQUIRE(dm->Di == 32 || dm->Di == 64 || dm->Di == 128, "Di must be 32, 64 or 128 (got %d)", dm->Di);
    REQUIRE(dm->idx_dtype == CSA2_BF16 || dm->idx_dtype == CSA2_F32, "idx_dtype must be CSA2_BF16 or CSA2_F32");
    REQUIRE(dm->K >= 1 && dm->K <= 2048, "K must be in 1..2048 (got %d)", dm->K);
  }
  REQUIRE(dm->kv_format == CSA2_KV_MXFP4 || dm->kv_format == CSA2_KV_FP8, "kv_format must be CSA2_KV_MXFP4 or CSA2_KV_FP8");
  if (dm->kv_format == CSA2_KV_FP8 && dm->d != 512)
    return fail(CSA2_ERR_UNSUPPORTED, "the FP8 main-KV format needs d = 512 (got %d)", dm->d);
  if (need_attn) {
    if (dm->d != 64 && dm->d != 512) return fail(CSA2_ERR_UNSUPPORTED, "d must be 64 or 512 (got %d)", dm->d);
    REQUIRE(dm->Hq >= 1 && dm->Hq <= 128, "Hq must be in 1..128 (got %d)", dm->Hq);
    REQUIRE(dm->K >= 1 && dm->K <= 2048, "K must be in 1..2048 (got %d)", dm->K);
    REQUIRE(dm->W >= 0 && dm->W <= 1024, "W must be in 0..1024 (got %d)", dm->W);
    REQUIRE(dm->swa_cap >= 0, "swa_cap must be >= 0");
  }
  return CSA2_OK;
}

static int check_cache(const csa2_cache* c, bool need_kv, bool need_idx) {
  REQUIRE(c, "cache must not be NULL");
  REQUIRE_IPTR(c->page_table);
  REQUIRE_IPTR(c->n_entries);
  REQUIRE(c->n_pages >= 1, "cache.n_pages must be >= 1");
  if (need_kv) {
    REQUIRE_PTR(c->kv_codes);
    REQUIRE_PTR(c->kv_scales);
  }
  if (need_idx) REQUIRE_PTR(c->idx_k);
  return CSA2_OK;
}

static IndexerArgs indexer_args(const csa2_dims* dm, const csa2_cache* c, const void* q, const float* w,
                                const int32_t* q_pos) {
  IndexerArgs a;
  a.q = q; a.w = w; a.k = c->idx_k; a.page_table = c->page_table; a.n_entries = c->n_entries;
  a.q_pos = q_pos; a.B = dm->B; a.Tq = dm->Tq; a.Hi = dm->Hi; a.Di = dm->Di; a.dtype = dm->idx_dtype;
  a.max_pages = dm->max_pages; a.n_pages = c->n_pages;
  a.max_entries = 0x7fffffff;
  return a;
}

// Workspace of csa2_index_topk: scores, block maxima, valid counts.
constexpr int kHistBins = 2048;  // score-key histogram bins per row (top 11 key bits)

// Long rows take the split Top-K (many CTAs per row): measured on the
// 1M-context group (8 rows of 262,144 entries) it saves ~30 us per step; on
// 32 rows of 32,768 entries the single-CTA rows are faster.  A batch whose
// longest row reaches 2^17 entries splits whatever its row count (one CTA per
// row would leave that row's scan of ~128K+ scores on one SM).
constexpr int64_t kSplitTopkMaxRows = 16;
constexpr int kSplitTopkMinEntries = 1 << 16;
constexpr int kSplitTopkAlwaysEntries = 1 << 17;
static bool use_split_topk(int64_t rows, int32_t max_entries) {
  return (rows <= kSplitTopkMaxRows && max_entries >= kSplitTopkMinEntries) || max_entries >= kSplitTopkAlwaysEntries;
}

struct IndexWs {
  size_t scores_off, bm_off, nvalid_off, hist_off, bmhist_off, split_off, total;
  int64_t s_stride, bm_stride;
};
static IndexWs index_ws_layout(const csa2_dims* dm, int32_t max_entries) {
  IndexWs L;
  const int64_t rows = (int64_t)dm->B * dm->Tq;
  const int64_t pool_pos = (int64_t)dm->n_pool_blocks * dm->pool_block;
  L.s_stride = (int64_t)round_up((size_t)(max_entries > pool_pos ? max_entries : pool_pos), 4);
  if (L.s_stride < 4) L.s_stride = 4;
  const int blk = dm->pool_block > 0 ? dm->pool_block : 8;
  L.bm_stride = (int64_t)round_up((size_t)((max_entries + blk - 1) / blk), 4);
  if (L.bm_stride < 4) L.bm_stride = 4;
  L.scores_off = 0;
  L.bm_off = round_up(L.scores_off + (size_t)(rows * L.s_stride) * 4, 256);
  L.nvalid_off = round_up(L.bm_off + (size_t)(rows * L.bm_stride) * 4, 256);
  L.hist_off = round_up(L.nvalid_off + (size_t)rows * 4, 256);
  L.bmhist_off = round_up(L.hist_off + (size_t)rows * kHistBins * 4, 256);
  L.split_off = round_up(L.bmhist_off + (dm->n_pool_blocks > 0 ? (size_t)rows * kHistBins * 4 : 0), 256);
  const size_t split = use_split_topk(rows, max_entries) ? topk_split_scratch_bytes(rows, L.s_stride) : 0;
  L.total = round_up(L.split_off + split, 256);
  return L;
}

}  // namespace csa2

using namespace csa2;

extern "C" {

int csa2_abi_version(void) { return CSA2_ABI_VERSION; }

uint64_t csa2_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* csa2_last_error(void) { return g_err; }

int csa2_get_status(uint32_t* bits, void* stream) {
  REQUIRE(bits, "bits must not be NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* w = status_word();
  if (!w) return fail(CSA2_ERR_CUDA, "status word unavailable");
  uint32_t host = 0;
  LAUNCH(cudaMemcpyAsync(&host, w, sizeof(uint32_t), cudaMemcpyDeviceToHost, s), "read status");
  LAUNCH(cudaMemsetAsync(w, 0, sizeof(uint32_t), s), "clear status");
  LAUNCH(cudaStreamSynchronize(s), "sync status");
  *bits = host;
  return CSA2_OK;
}

int csa2_pack_mxfp4_f32(const float* x, int64_t n_rows, int32_t d, uint8_t* codes, uint8_t* scales,
                        void* stream) {
  NvtxRange nvtx_("csa2_pack_mxfp4_f32");
  g_err[0] = 0;
  REQUIRE(n_rows >= 0, "n_rows must be >= 0");
  REQUIRE(d > 0 && d % 16 == 0 && d <= 4096, "d must be a multiple of 16 in 16..4096 (got %d)", d);
  if (n_rows == 0) return CSA2_OK;
  REQUIRE_PTR(x); REQUIRE_PTR(codes); REQUIRE(scales, "scales must not be NULL");
  LAUNCH(launch_pack_mxfp4(x, n_rows, d, codes, scales, static_cast<cudaStream_t>(stream)), "pack_mxfp4");
  return CSA2_OK;
}

int csa2_unpack_mxfp4_bf16(const uint8_t* codes, const uint8_t* scales, int64_t n_rows, int32_t d,
                           uint16_t* out, void* stream) {
  NvtxRange nvtx_("csa2_unpack_mxfp4_bf16");
  g_err[0] = 0;
  REQUIRE(n_rows >= 0, "n_rows must be >= 0");
  REQUIRE(d > 0 && d % 16 == 0 && d <= 4096, "d must be a multiple of 16 in 16..4096 (got %d)", d);
  if (n_rows == 0) return CSA2_OK;
  REQUIRE_PTR(codes); REQUIRE(scales, "scales must not be NULL"); REQUIRE_PTR(out);
  LAUNCH(launch_unpack_mxfp4(codes, scales, n_rows, d, out, static_cast<cudaStream_t>(stream)), "unpack_mxfp4");
  return CSA2_OK;
}

int csa2_pack_swa_fp8(const float* x, int64_t n_rows, int32_t d, uint8_t* codes, float* scales,
                      void* stream) {
  NvtxRange nvtx_("csa2_pack_swa_fp8");
  g_err[0] = 0;
  REQUIRE(n_rows >= 0, "n_rows must be >= 0");
  REQUIRE(d > 0 && d % 16 == 0 && d <= 4096, "d must be a multiple of 16 in 16..4096 (got %d)", d);
  if (n_rows == 0) return CSA2_OK;
  REQUIRE_PTR(x); REQUIRE_PTR(codes); REQUIRE(scales, "scales must not be NULL");
  LAUNCH(launch_pack_fp8(x, n_rows, d, codes, scales, static_cast<cudaStream_t>(stream)), "pack_fp8");
  return CSA2_OK;
}

int csa2_norm_rope_pack(const float* latent, int32_t B, int32_t n_max, int32_t d, int32_t r,
                        const float* gamma, float eps, float rope_base, const int32_t* first_entry,
                        const int32_t* n_rows, const int32_t* page_table, int32_t max_pages,
                        int64_t n_pages, uint8_t* kv_codes, uint8_t* kv_scales, void* stream) {
  NvtxRange nvtx_("csa2_norm_rope_pack");
  g_err[0] = 0;
  REQUIRE(B >= 0 && n_max >= 0, "B and n_max must be >= 0");
  if (d != 64 && d != 512) return fail(CSA2_ERR_UNSUPPORTED, "d must be 64 or 512 (got %d)", d);
  REQUIRE(r >= 0 && r <= d && r % 2 == 0, "r must be even and in 0..d (got %d)", r);
  REQUIRE(eps >= 0.f, "eps must be >= 0");
  if ((int64_t)B * n_max == 0) return CSA2_OK;
  REQUIRE_PTR(latent); REQUIRE_PTR(gamma); REQUIRE_IPTR(first_entry); REQUIRE_IPTR(n_rows);
  REQUIRE_IPTR(page_table); REQUIRE_PTR(kv_codes); REQUIRE_PTR(kv_scales);
  REQUIRE(max_pages >= 1 && n_pages >= 1, "max_pages and n_pages must be >= 1");
  LatentSource src{latent, d, 0, 1};
  LAUNCH(launch_norm_rope_pack(src, B, n_max, d, r, gamma, eps, rope_base, first_entry, n_rows, page_table,
                               max_pages, n_pages, kv_codes, kv_scales, nullptr, 0, 0, 0, nullptr,
                               static_cast<cudaStream_t>(stream)),
         "norm_rope_pack");
  return CSA2_OK;
}

int csa2_norm_rope_pack_fp8(const float* latent, int32_t B, int32_t n_max, int32_t d, int32_t r,
                            const float* gamma, float eps, float rope_base, const int32_t* first_entry,
                            const int32_t* n_rows, const int32_t* page_table, int32_t max_pages,
                            int64_t n_pages, uint8_t* kv_codes, float* kv_scales, void* stream) {
  NvtxRange nvtx_("csa2_norm_rope_pack_fp8");
  g_err[0] = 0;
  REQUIRE(B >= 0 && n_max >= 0, "B and n_max must be >= 0");
  if (d != 512) return fail(CSA2_ERR_UNSUPPORTED, "the FP8 main-KV format needs d = 512 (got %d)", d);
  REQUIRE(r >= 0 && r <= d && r % 2 == 0, "r must be even and in 0..d (got %d)", r);
  REQUIRE(eps >= 0.f, "eps must be >= 0");
  if ((int64_t)B * n_max == 0) return CSA2_OK;
  REQUIRE_PTR(latent); REQUIRE_PTR(gamma); REQUIRE_IPTR(first_entry); REQUIRE_IPTR(n_rows);
  REQUIRE_IPTR(page_table); REQUIRE_PTR(kv_codes); REQUIRE_PTR(kv_scales);
  REQUIRE(max_pages >= 1 && n_pages >= 1, "max_pages and n_pages must be >= 1");
  LatentSource src{latent, d, 0, 1};
  LAUNCH(launch_norm_rope_pack(src, B, n_max, d, r, gamma, eps, rope_base, first_entry, n_rows, page_table,
                               max_pages, n_pages, kv_codes, reinterpret_cast<uint8_t*>(kv_scales), nullptr, 0, 0, 0,
                               nullptr, static_cast<cudaStream_t>(stream), 1),
         "norm_rope_pack_fp8");
  return CSA2_OK;
}

size_t csa2_compress_workspace_size(int32_t B, int32_t T, int32_t H, int32_t d, int32_t Di) {
  if (B <= 0 || T < 4 || H <= 0 || d <= 0) return 0;
  return compress_partials_bytes(B, T, H, d, Di > 0 ? Di : 0, nullptr);
}

// The layers' outputs are one GEMM of N = L (d + Di) channels when every layer's block
// starts on a 128-channel tile (the TMA-fed GEMM); otherwise one call per layer.
static bool layers_grouped(int32_t H, int32_t d, int32_t Di) {
  return d % 128 == 0 && (d + Di) % 128 == 0 && H % 16 == 0;
}

size_t csa2_compress_layers_workspace_size(int32_t B, int32_t T, int32_t H, int32_t L, int32_t d, int32_t Di) {
  if (B <= 0 || T < 4 || H <= 0 || d <= 0 || L <= 0) return 0;
  if (!layers_grouped(H, d, Di)) return compress_partials_bytes(B, T, H, d, Di > 0 ? Di : 0, nullptr);
  return compress_partials_bytes(B, T, H, L * (d + Di), 0, nullptr);
}

int csa2_compress_pack(const uint16_t* hidden, int32_t B, int32_t T, int32_t H, const uint16_t* W,
                       const float* gamma, float eps, float rope_base, const uint16_t* W_idx,
                       const int32_t* first_entry, const csa2_dims* dm, const csa2_cache* c, void* ws,
                       size_t ws_bytes, void* stream) {
  NvtxRange nvtx_("csa2_compress_pack");
  g_err[0] = 0;
  int rc = check_dims(dm, false, false);
  if (rc) return rc;
  if (dm->d != 64 && dm->d != 512) return fail(CSA2_ERR_UNSUPPORTED, "d must be 64 or 512 (got %d)", dm->d);
  REQUIRE(B == dm->B, "B (%d) must equal dims.B (%d)", B, dm->B);
  REQUIRE(T >= 0 && H > 0, "T must be >= 0 and H > 0");
  REQUIRE(H % 64 == 0, "H must be a multiple of 64 (got %d)", H);
  REQUIRE(dm->r >= 0 && dm->r <= dm->d && dm->r % 2 == 0, "r must be even and in 0..d");
  if (B == 0 || T < 4) return CSA2_OK;
  REQUIRE_PTR(hidden); REQUIRE_PTR(W); REQUIRE_PTR(gamma); REQUIRE_IPTR(first_entry);
  rc = check_cache(c, true, W_idx != nullptr);
  if (rc) return rc;
  if (W_idx) {
    REQUIRE(aligned16(W_idx), "W_idx must be 16-byte aligned");
    REQUIRE(dm->Di == 32 || dm->Di == 64 || dm->Di == 128, "Di must be 32, 64 or 128");
    REQUIRE(dm->idx_dtype == CSA2_BF16 || dm->idx_dtype == CSA2_F32, "bad idx_dtype");
  }
  const int Di = W_idx ? dm->Di : 0;
  int n_split = 1;
  const size_t need = compress_partials_bytes(B, T, H, dm->d, Di, &n_split);
  if (!ws || ws_bytes < need) return fail(CSA2_ERR_WORKSPACE, "compress needs %zu workspace bytes (got %zu)", need, ws_bytes);
  REQUIRE(aligned16(ws), "ws must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* part = static_cast<float*>(ws);
  LAUNCH(launch_compress_gemm(hidden, B, T, H, W, dm->d, W_idx, Di, part, n_split, s), "compress_gemm");
  const int G = T / 4, N = dm->d + Di;
  LatentSource src{part, N, (int64_t)B * G * N, n_split};
  LAUNCH(launch_norm_rope_pack(src, B, G, dm->d, dm->r, gamma, eps, rope_base, first_entry, nullptr,
                               c->page_table, dm->max_pages, c->n_pages, c->kv_codes, c->kv_scales,
                               W_idx ? part + dm->d : nullptr, N, Di, dm->idx_dtype, W_idx ? c->idx_k : nullptr, s,
                               dm->kv_format == CSA2_KV_FP8),
         "compress_epilogue");
  return CSA2_OK;
}

int csa2_compress_layers(const uint16_t* hidden, int32_t B, int32_t T, int32_t H, int32_t L,
                         const uint16_t* W_all, int32_t Di, const float* gamma_all, float eps, float rope_base,
                         const int32_t* first_entry, const csa2_dims* dm, const csa2_cache* caches, void* ws,
                         size_t ws_bytes, void* stream) {
  NvtxRange nvtx_("csa2_compress_layers");
  g_err[0] = 0;
  int rc = check_dims(dm, false, false);
  if (rc) return rc;
  if (dm->d != 64 && dm->d != 512) return fail(CSA2_ERR_UNSUPPORTED, "d must be 64 or 512 (got %d)", dm->d);
  REQUIRE(L >= 1 && L <= 4096, "L must be in 1..4096 (got %d)", L);
  REQUIRE(B == dm->B, "B (%d) must equal dims.B (%d)", B, dm->B);
  REQUIRE(T >= 0 && H > 0, "T must be >= 0 and H > 0");
  REQUIRE(H % 64 == 0, "H must be a multiple of 64 (got %d)", H);
  REQUIRE(Di == 0 || Di == dm->Di, "Di must be 0 or dims.Di (got %d)", Di);
  REQUIRE(dm->r >= 0 && dm->r <= dm->d && dm->r % 2 == 0, "r must be even and in 0..d");
  if (B == 0 || T < 4) return CSA2_OK;
  REQUIRE_PTR(hidden); REQUIRE_PTR(W_all); REQUIRE_PTR(gamma_all); REQUIRE_IPTR(first_entry);
  REQUIRE(caches, "caches must not be NULL");
  if (Di) {
    REQUIRE(Di == 32 || Di == 64 || Di == 128, "Di must be 32, 64 or 128");
    REQUIRE(dm->idx_dtype == CSA2_BF16 || dm->idx_dtype == CSA2_F32, "bad idx_dtype");
  }
  for (int l = 0; l < L; ++l) {
    rc = check_cache(&caches[l], true, Di > 0);
    if (rc) return rc;
  }
  const int d = dm->d, G = T / 4, Nl = d + Di;
  const int64_t wl_elems = (int64_t)Nl * 4 * H;   // one layer's stacked weights
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t need = csa2_compress_layers_workspace_size(B, T, H, L, d, Di);
  if (!ws || ws_bytes < need) return fail(CSA2_ERR_WORKSPACE, "compress_layers needs %zu workspace bytes (got %zu)", need, ws_bytes);
  REQUIRE(aligned16(ws), "ws must be 16-byte aligned");
  if (!layers_grouped(H, d, Di)) {   // one compression per layer
    for (int l = 0; l < L; ++l) {
      rc = csa2_compress_pack(hidden, B, T, H, W_all + l * wl_elems, gamma_all + (int64_t)l * d, eps, rope_base,
                              Di ? W_all + l * wl_elems + (int64_t)d * 4 * H : nullptr, first_entry, dm, &caches[l],
                              ws, ws_bytes, stream);
      if (rc) return rc;
    }
    return CSA2_OK;
  }
  // one GEMM: the stacked weights are one [L (d + Di)][4H] operand
  const int N = L * Nl;
  int n_split = 1;
  compress_partials_bytes(B, T, H, N, 0, &n_split);
  float* part = static_cast<float*>(ws);
  LAUNCH(launch_compress_gemm(hidden, B, T, H, W_all, N, nullptr, 0, part, n_split, s), "compress_layers_gemm");
  // every layer's RMSNorm / RoPE / pack in one launch per kPackLayersMax layers
  for (int l0 = 0; l0 < L; l0 += kPackLayersMax) {
    const int nl = std::min(L - l0, kPackLayersMax);
    PackLayers pl = {};
    pl.col_stride = Nl;
    pl.gamma_stride = d;
    for (int l = 0; l < nl; ++l) {
      const csa2_cache* c = &caches[l0 + l];
      pl.l[l] = PackLayer{c->page_table, c->n_pages, c->kv_codes, c->kv_scales, Di ? c->idx_k : nullptr};
    }
    LatentSource src{part + (int64_t)l0 * Nl, N, (int64_t)B * G * N, n_split};
    LAUNCH(launch_norm_rope_pack_layers(src, B, G, d, dm->r, gamma_all + (int64_t)l0 * d, eps, rope_base,
                                        first_entry, dm->max_pages, Di ? part + (int64_t)l0 * Nl + d : nullptr, N, Di,
                                        dm->idx_dtype, dm->kv_format == CSA2_KV_FP8, pl, nl, s),
           "compress_layers_epilogue");
  }
  return CSA2_OK;
}

size_t csa2_swa_replay_workspace_size(int32_t B, int32_t n_tok, int32_t H, int32_t d) {
  if (B <= 0 || n_tok <= 0 || H <= 0 || d <= 0) return 0;
  return compress_partials_bytes(B, n_tok, H, d, 0, nullptr, 1);
}

int csa2_swa_replay(const uint16_t* hidden, int32_t B, int32_t n_tok, int32_t H, const uint16_t* W_swa,
                    const float* gamma, float eps, float rope_base, const int32_t* tok_pos0, const csa2_dims* dm,
                    const csa2_window* win, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx_("csa2_swa_replay");
  g_err[0] = 0;
  int rc = check_dims(dm, false, false);
  if (rc) return rc;
  if (dm->d != 64 && dm->d != 512) return fail(CSA2_ERR_UNSUPPORTED, "d must be 64 or 512 (got %d)", dm->d);
  REQUIRE(B == dm->B, "B (%d) must equal dims.B (%d)", B, dm->B);
  REQUIRE(n_tok >= 0 && H > 0, "n_tok must be >= 0 and H > 0");
  REQUIRE(H % 64 == 0, "H must be a multiple of 64 (got %d)", H);
  REQUIRE(dm->r >= 0 && dm->r <= dm->d && dm->r % 2 == 0, "r must be even and in 0..d");
  REQUIRE(eps >= 0.f, "eps must be >= 0");
  if (B == 0 || n_tok == 0) return CSA2_OK;
  REQUIRE_PTR(hidden); REQUIRE_PTR(W_swa); REQUIRE_PTR(gamma); REQUIRE_IPTR(tok_pos0);
  REQUIRE(win, "window must not be NULL");
  REQUIRE_PTR(win->codes); REQUIRE_PTR(win->scales); REQUIRE_IPTR(win->pos0);
  REQUIRE(dm->swa_cap >= 1, "dims.swa_cap must be >= 1 (got %d)", dm->swa_cap);
  int n_split = 1;
  const size_t need = compress_partials_bytes(B, n_tok, H, dm->d, 0, &n_split, 1);
  if (!ws || ws_bytes < need) return fail(CSA2_ERR_WORKSPACE, "swa_replay needs %zu workspace bytes (got %zu)", need, ws_bytes);
  REQUIRE(aligned16(ws), "ws must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* part = static_cast<float*>(ws);
  // one token per GEMM row: c_t = W_swa h_t, split-K fp32 partials
  LAUNCH(launch_compress_gemm(hidden, B, n_tok, H, W_swa, dm->d, nullptr, 0, part, n_split, s, 1), "swa_replay_gemm");
  LatentSource src{part, dm->d, (int64_t)B * n_tok * dm->d, n_split};
  LAUNCH(launch_norm_rope_fp8_window(src, B, n_tok, dm->d, dm->r, gamma, eps, rope_base, tok_pos0, win->pos0,
                                     dm->swa_cap, win->codes, win->scales, s),
         "swa_replay_epilogue");
  return CSA2_OK;
}

int csa2_index_scores(const csa2_dims* dm, const csa2_cache* c, const void* idx_q, const float* w,
                      const int32_t* q_pos, float* scores, int64_t score_stride, float* blockmax,
                      int64_t bm_stride, void* stream) {
  NvtxRange nvtx_("csa2_index_scores");
  g_err[0] = 0;
  int rc = check_dims(dm, true, false);
  if (rc) return rc;
  if ((int64_t)dm->B * dm->Tq == 0) return CSA2_OK;
  rc = check_cache(c, false, true);
  if (rc) return rc;
  REQUIRE_PTR(idx_q); REQUIRE_PTR(w); REQUIRE_IPTR(q_pos); REQUIRE_PTR(scores);
  REQUIRE(score_stride >= 1 && score_stride < (1LL << 31), "score_stride out of range");
  if (blockmax) {
    REQUIRE(dm->pool_block == 8, "pool_block must be 8");
    REQUIRE(bm_stride >= (score_stride + 7) / 8, "bm_stride must be >= ceil(score_stride / 8)");
  }
  IndexerArgs a = indexer_args(dm, c, idx_q, w, q_pos);
  a.max_entries = (int)score_stride;
  LAUNCH(launch_index_scores(a, scores, score_stride, blockmax, bm_stride, 8, (int)score_stride, nullptr,
                             static_cast<cudaStream_t>(stream)),
         "index_scores");
  return CSA2_OK;
}

size_t csa2_topk_workspace_size(int64_t rows, int64_t stride, int32_t k) {
  (void)k;
  if (rows <= 0 || stride <= 0) return 0;
  return round_up((size_t)rows * kHistBins * 4, 256) + topk_split_scratch_bytes(rows, stride);
}

int csa2_topk_f32(const float* scores, int64_t rows, int64_t stride, const int32_t* n_valid, int32_t k,
                  int32_t* out_idx, int32_t* out_cnt, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx_("csa2_topk_f32");
  (void)ws; (void)ws_bytes;
  g_err[0] = 0;
  REQUIRE(rows >= 0 && rows < (1LL << 31), "rows out of range");
  REQUIRE(stride >= 1 && stride < (1LL << 31), "stride out of range");
  REQUIRE(k >= 1 && k <= 4096, "k must be in 1..4096 (got %d)", k);
  if (rows == 0) return CSA2_OK;
  REQUIRE_PTR(scores); REQUIRE_IPTR(out_idx); REQUIRE_IPTR(out_cnt);
  if (n_valid) REQUIRE_IPTR(n_valid);
  ValidSpec v{n_valid, nullptr, nullptr, 1, 1, 0};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t need = csa2_topk_workspace_size(rows, stride, k);
  if (ws && ws_bytes >= need) {   // many CTAs per row
    REQUIRE(aligned16(ws), "ws must be 16-byte aligned");
    uint32_t* hist = static_cast<uint32_t*>(ws);
    char* split = static_cast<char*>(ws) + round_up((size_t)rows * kHistBins * 4, 256);
    LAUNCH(launch_row_hist(scores, rows, stride, v, hist, s), "row_hist");
    if (stride <= 32768) {   // rows the one-pass kernels take whole (a cluster or a CTA per row)
      LAUNCH(launch_topk(scores, rows, stride, v, k, out_idx, out_cnt, Remap{nullptr, 0, 8}, hist, kHistBins, s),
             "topk");
      return CSA2_OK;
    }
    LAUNCH(launch_topk_split(scores, rows, stride, v, k, out_idx, out_cnt, Remap{nullptr, 0, 8}, hist, kHistBins,
                             split, s),
           "topk_split");
    return CSA2_OK;
  }
  LAUNCH(launch_topk(scores, rows, stride, v, k, out_idx, out_cnt, Remap{nullptr, 0, 8}, nullptr, 0, s), "topk");
  return CSA2_OK;
}

int csa2_block_pool_f32(const float* scores, int64_t rows, int64_t stride, const int32_t* n_valid,
                        int32_t block, int32_t n_pool_blocks, int32_t* out_pool, int32_t* out_pool_cnt,
                        float* out_blockmax, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx_("csa2_block_pool_f32");
  g_err[0] = 0;
  REQUIRE(rows >= 0 && rows < (1LL << 31), "rows out of range");
  REQUIRE(stride >= 1 && stride < (1LL << 31), "stride out of range");
  REQUIRE(block >= 1 && block <= 64, "block must be in 1..64");
  REQUIRE(n_pool_blocks >= 1 && n_pool_blocks <= 4096, "n_pool_blocks must be in 1..4096");
  if (rows == 0) return CSA2_OK;
  REQUIRE_PTR(scores); REQUIRE_IPTR(n_valid); REQUIRE_IPTR(out_pool); REQUIRE_IPTR(out_pool_cnt);
  const int64_t nb = (stride + block - 1) / block;
  float* bm = out_blockmax;
  int64_t bm_stride = nb;
  if (!bm) {
    const size_t need = (size_t)(rows * nb) * sizeof(float);
    if (!ws || ws_bytes < need) return fail(CSA2_ERR_WORKSPACE, "block_pool needs %zu workspace bytes", need);
    bm = static_cast<float*>(ws);
  } else {
    REQUIRE(aligned16(bm), "out_blockmax must be 16-byte aligned");
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ValidSpec ve{n_valid, nullptr, nullptr, 1, 1, 0};
  LAUNCH(launch_block_max(scores, rows, stride, ve, block, bm, bm_stride, s), "block_max");
  // valid blocks per row: ceil(n_valid / block)
  ValidSpec vd{n_valid, nullptr, nullptr, 1, block, 0};
  LAUNCH(launch_topk(bm, rows, bm_stride, vd, n_pool_blocks, out_pool, out_pool_cnt, Remap{nullptr, 0, 8},
                     nullptr, 0, s),
         "block_pool_topk");
  return CSA2_OK;
}

size_t csa2_index_topk_workspace_size(const csa2_dims* dm, int32_t max_entries) {
  if (!dm || max_entries < 0) return 0;
  return index_ws_layout(dm, max_entries).total;
}

static int index_topk_impl(const csa2_dims* dm, const csa2_cache* c, const void* idx_q, const float* w,
                           const int32_t* q_pos, const int32_t* pool, const int32_t* pool_cnt,
                           int32_t* out_idx, int32_t* out_cnt, int32_t* out_pool, int32_t* out_pool_cnt,
                           int32_t max_entries, void* ws, size_t ws_bytes, cudaStream_t s) {
  int rc = check_dims(dm, true, false);
  if (rc) return rc;
  const int64_t rows = (int64_t)dm->B * dm->Tq;
  if (rows == 0) return CSA2_OK;
  rc = check_cache(c, false, true);
  if (rc) return rc;
  REQUIRE_PTR(idx_q); REQUIRE_PTR(w); REQUIRE_IPTR(q_pos); REQUIRE_IPTR(out_idx); REQUIRE_IPTR(out_cnt);
  REQUIRE(max_entries >= 0, "max_entries must be >= 0");
  const bool reindex = pool != nullptr;
  if (reindex || out_pool) {
    REQUIRE(dm->pool_block == 8, "pool_block must be 8 (got %d)", dm->pool_block);
    REQUIRE(dm->n_pool_blocks >= 1 && dm->n_pool_blocks <= 4096, "n_pool_blocks must be in 1..4096");
  }
  if (reindex) { REQUIRE_IPTR(pool); REQUIRE_IPTR(pool_cnt); }
  if (out_pool) { REQUIRE_IPTR(out_pool); REQUIRE_IPTR(out_pool_cnt); }
  const IndexWs L = index_ws_layout(dm, max_entries);
  if (!ws || ws_bytes < L.total) return fail(CSA2_ERR_WORKSPACE, "index_topk needs %zu workspace bytes (got %zu)", L.total, ws_bytes);
  REQUIRE(aligned16(ws), "ws must be 16-byte aligned");
  char* base = static_cast<char*>(ws);
  float* scores = reinterpret_cast<float*>(base + L.scores_off);
  float* bm = reinterpret_cast<float*>(base + L.bm_off);
  int32_t* nvalid = reinterpret_cast<int32_t*>(base + L.nvalid_off);
  uint32_t* hist = reinterpret_cast<uint32_t*>(base + L.hist_off);
  uint32_t* bm_hist = (out_pool && dm->n_pool_blocks > 0) ? reinterpret_cast<uint32_t*>(base + L.bmhist_off) : nullptr;
  IndexerArgs a = indexer_args(dm, c, idx_q, w, q_pos);
  a.max_entries = max_entries;
  if (!reindex) {
    // the many-query GEMM path builds no histogram: the Top-K kernel then builds each row's
    if (index_scores_gemm_supported(a)) hist = nullptr;
    if (hist) LAUNCH(launch_zero_u32(hist, rows * kHistBins, s), "zero histogram");
    if (!hist) bm_hist = nullptr;
    if (bm_hist) LAUNCH(launch_zero_u32(bm_hist, rows * kHistBins, s), "zero histogram");
    bool bm_built = false;
    LAUNCH(launch_index_scores(a, scores, L.s_stride, out_pool ? bm : nullptr, L.bm_stride, 8, max_entries, hist, s,
                               bm_hist, &bm_built),
           "index_scores");
    ValidSpec v{nullptr, c->n_entries, q_pos, dm->Tq, 1, max_entries};
    if (hist && use_split_topk(rows, max_entries))
      LAUNCH(launch_topk_split(scores, rows, L.s_stride, v, dm->K, out_idx, out_cnt, Remap{nullptr, 0, 8}, hist,
                               kHistBins, base + L.split_off, s),
             "topk");
    else
      LAUNCH(launch_topk(scores, rows, L.s_stride, v, dm->K, out_idx, out_cnt, Remap{nullptr, 0, 8}, hist,
                         hist ? kHistBins : 0, s),
             "topk");
    if (out_pool) {
      ValidSpec vb{nullptr, c->n_entries, q_pos, dm->Tq, 8, max_entries};
      LAUNCH(launch_topk(bm, rows, L.bm_stride, vb, dm->n_pool_blocks, out_pool, out_pool_cnt,
                         Remap{nullptr, 0, 8}, bm_built ? bm_hist : nullptr, bm_built ? kHistBins : 0, s),
             "block_pool");
    }
  } else {
    const int64_t pool_pos = (int64_t)dm->n_pool_blocks * 8;
    if (index_scores_gemm_supported(a) && max_entries > 0 && 4 * pool_pos >= max_entries) {
      // many query tokens over a pool that covers a good share of the entries: score
      // every visible entry on the tensor cores (the same score per position, R10),
      // then keep the pooled positions' scores
      LAUNCH(launch_index_scores_gemm(a, scores, L.s_stride, nullptr, 0, max_entries, s), "index_scores_gemm");
      LAUNCH(launch_pool_compact(a, pool, pool_cnt, dm->n_pool_blocks, scores, L.s_stride, nvalid, s),
             "pool_compact");
    } else {
      LAUNCH(launch_index_scores_pool(a, pool, pool_cnt, dm->n_pool_blocks, 8, scores, L.s_stride, nvalid, s),
             "index_scores_pool");
    }
    ValidSpec v{nvalid, nullptr, nullptr, 1, 1, 0};
    LAUNCH(launch_topk(scores, rows, L.s_stride, v, dm->K, out_idx, out_cnt,
                       Remap{pool, dm->n_pool_blocks, 8}, nullptr, 0, s, (int64_t)dm->n_pool_blocks * 8),
           "reindex_topk");
  }
  return CSA2_OK;
}

}  // extern "C"

namespace csa2 {
int index_topk_into(const csa2_dims* dm, const csa2_cache* c, const void* idx_q, const float* w,
                    const int32_t* q_pos, const int32_t* pool, const int32_t* pool_cnt, int32_t* out_idx,
                    int32_t* out_cnt, int32_t* out_pool, int32_t* out_pool_cnt, int32_t max_entries, void* ws,
                    size_t ws_bytes, cudaStream_t s) {
  g_err[0] = 0;
  return index_topk_impl(dm, c, idx_q, w, q_pos, pool, pool_cnt, out_idx, out_cnt, out_pool, out_pool_cnt,
                         max_entries, ws, ws_bytes, s);
}
int report_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace csa2

extern "C" {

int csa2_index_topk(const csa2_dims* dm, const csa2_cache* c, const void* idx_q, const float* w,
                    const int32_t* q_pos, const int32_t* pool, const int32_t* pool_cnt, int32_t* out_idx,
                    int32_t* out_cnt, int32_t* out_pool, int32_t* out_pool_cnt, int32_t max_entries,
                    void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx_("csa2_index_topk");
  g_err[0] = 0;
  return index_topk_impl(dm, c, idx_q, w, q_pos, pool, pool_cnt, out_idx, out_cnt, out_pool, out_pool_cnt,
                         max_entries, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

static int attn_impl(const csa2_dims* dm, const csa2_cache* c, const csa2_window* win, const uint16_t* Q,
                     const int32_t* q_pos, const int32_t* idx, const int32_t* cnt, float softmax_scale,
                     float* O, float* lse, cudaStream_t s) {
  int rc = check_dims(dm, false, true);
  if (rc) return rc;
  if ((int64_t)dm->B * dm->Tq == 0) return CSA2_OK;
  rc = check_cache(c, true, false);
  if (rc) return rc;
  REQUIRE(win, "window must not be NULL");
  REQUIRE_PTR(Q); REQUIRE_IPTR(q_pos); REQUIRE_IPTR(idx); REQUIRE_IPTR(cnt); REQUIRE_PTR(O);
  if (lse) REQUIRE(aligned16(lse), "lse must be 16-byte aligned");
  if (dm->swa_cap > 0 && dm->W > 0) {
    REQUIRE_PTR(win->codes); REQUIRE_PTR(win->scales); REQUIRE_IPTR(win->pos0);
  }
  AttnArgs a;
  a.Q = Q; a.kv_codes = c->kv_codes; a.kv_scales = c->kv_scales; a.page_table = c->page_table;
  a.n_pages = c->n_pages; a.max_pages = dm->max_pages; a.idx = idx; a.cnt = cnt; a.q_pos = q_pos;
  a.n_entries = c->n_entries; a.swa_codes = win->codes; a.swa_scales = win->scales; a.swa_pos0 = win->pos0;
  a.swa_cap = (dm->W > 0) ? dm->swa_cap : 0; a.W = dm->W; a.B = dm->B; a.Tq = dm->Tq; a.Hq = dm->Hq;
  a.d = dm->d; a.K = dm->K; a.scale = softmax_scale; a.O = O; a.lse = lse;
  a.kv_fp8 = dm->kv_format == CSA2_KV_FP8;
  LAUNCH(launch_sparse_attn(a, s), "sparse_attn");
  return CSA2_OK;
}

int csa2_sparse_attn(const csa2_dims* dm, const csa2_cache* c, const csa2_window* win, const uint16_t* Q,
                     const int32_t* q_pos, const int32_t* idx, const int32_t* cnt, float softmax_scale,
                     float* O, float* lse, void* stream) {
  NvtxRange nvtx_("csa2_sparse_attn");
  g_err[0] = 0;
  return attn_impl(dm, c, win, Q, q_pos, idx, cnt, softmax_scale, O, lse, static_cast<cudaStream_t>(stream));
}

size_t csa2_layer_workspace_size(const csa2_layer_args* a) {
  if (!a) return 0;
  size_t need = 0;
  if (a->mode != CSA2_MODE_REUSE) need = index_ws_layout(&a->dims, a->max_entries).total;
  if (a->mode == CSA2_MODE_FULL && a->hidden) {
    const size_t cw = csa2_compress_workspace_size(a->dims.B, a->T, a->H, a->dims.d, a->W_idx ? a->dims.Di : 0);
    if (cw > need) need = cw;
  }
  return need;
}

int csa2_layer(const csa2_layer_args* a, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx_("csa2_layer");
  g_err[0] = 0;
  REQUIRE(a, "args must not be NULL");
  REQUIRE(a->mode == CSA2_MODE_FULL || a->mode == CSA2_MODE_REINDEX || a->mode == CSA2_MODE_REUSE,
          "unknown mode %d", a->mode);
  const csa2_dims* dm = &a->dims;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int rc = check_dims(dm, a->mode != CSA2_MODE_REUSE, true);
  if (rc) return rc;
  const int64_t rows = (int64_t)dm->B * dm->Tq;
  if (rows == 0) return CSA2_OK;
  REQUIRE_IPTR(a->q_pos); REQUIRE_IPTR(a->idx_out); REQUIRE_IPTR(a->cnt_out);
  if (a->mode == CSA2_MODE_REUSE) { REQUIRE_IPTR(a->idx_in); REQUIRE_IPTR(a->cnt_in); }
  if (a->mode == CSA2_MODE_REINDEX) { REQUIRE_IPTR(a->pool); REQUIRE_IPTR(a->pool_cnt); }
  if (a->mode == CSA2_MODE_FULL && a->hierarchical) { REQUIRE_IPTR(a->pool); REQUIRE_IPTR(a->pool_cnt); }
  const size_t need = csa2_layer_workspace_size(a);
  if (need && (!ws || ws_bytes < need)) return fail(CSA2_ERR_WORKSPACE, "layer needs %zu workspace bytes (got %zu)", need, ws_bytes);
  // 1. compression of the new tokens (Full only)
  if (a->mode == CSA2_MODE_FULL && a->hidden) {
    rc = csa2_compress_pack(a->hidden, dm->B, a->T, a->H, a->W_c, a->gamma, a->eps, a->rope_base, a->W_idx,
                            a->first_entry, dm, &a->cache, ws, ws_bytes, stream);
    if (rc) return rc;
  }
  // 2. window rows of the query tokens
  if (a->swa_new) {
    REQUIRE_PTR(a->swa_new); REQUIRE_PTR(a->window.codes); REQUIRE_PTR(a->window.scales);
    REQUIRE_IPTR(a->window.pos0);
    LAUNCH(launch_pack_fp8_window(a->swa_new, dm->B, dm->Tq, dm->d, a->q_pos, a->window.pos0, dm->swa_cap,
                                  a->window.codes, a->window.scales, s),
           "pack_window");
  }
  // 3. indices
  const int32_t* idx = a->idx_out;
  const int32_t* cnt = a->cnt_out;
  if (a->mode == CSA2_MODE_FULL) {
    rc = index_topk_impl(dm, &a->cache, a->idx_q, a->idx_w, a->q_pos, nullptr, nullptr, a->idx_out, a->cnt_out,
                         a->hierarchical ? a->pool : nullptr, a->hierarchical ? a->pool_cnt : nullptr,
                         a->max_entries, ws, ws_bytes, s);
    if (rc) return rc;
  } else if (a->mode == CSA2_MODE_REINDEX) {
    rc = index_topk_impl(dm, &a->cache, a->idx_q, a->idx_w, a->q_pos, a->pool, a->pool_cnt, a->idx_out,
                         a->cnt_out, nullptr, nullptr, a->max_entries, ws, ws_bytes, s);
    if (rc) return rc;
  } else {
    if (a->idx_out != a->idx_in)
      LAUNCH(cudaMemcpyAsync(a->idx_out, a->idx_in, (size_t)rows * dm->K * sizeof(int32_t), cudaMemcpyDeviceToDevice, s),
             "reuse idx copy");
    if (a->cnt_out != a->cnt_in)
      LAUNCH(cudaMemcpyAsync(a->cnt_out, a->cnt_in, (size_t)rows * sizeof(int32_t), cudaMemcpyDeviceToDevice, s),
             "reuse cnt copy");
    idx = a->idx_in;
    cnt = a->cnt_in;
  }
  // 4. attention
  return attn_impl(dm, &a->cache, &a->window, a->Q, a->q_pos, idx, cnt, a->softmax_scale, a->O, a->lse, s);
}

}  // extern "C"
