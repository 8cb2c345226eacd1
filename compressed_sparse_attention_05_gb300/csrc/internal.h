// Launchers shared between the kernel translation units and the C-ABI layer
// (api.cu).  Arguments are validated by the caller; launchers only launch.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/csa2.h"

namespace csa2 {

// csa2_index_topk with caller-chosen scratch (used by the no-allocation entry point).
int index_topk_into(const csa2_dims* dm, const csa2_cache* c, const void* idx_q, const float* w,
                    const int32_t* q_pos, const int32_t* pool, const int32_t* pool_cnt, int32_t* out_idx,
                    int32_t* out_cnt, int32_t* out_pool, int32_t* out_pool_cnt, int32_t max_entries, void* ws,
                    size_t ws_bytes, cudaStream_t s);
// Records `msg` as the calling thread's last error and returns `code`.
int report_error(int code, const char* msg);

// Device status word of the current device (see csa2_get_status).
uint32_t* status_word();

// Device address of a module global in the calling thread's current context,
// looked up with cudaGetSymbolAddress once per (context, symbol) and cached.
// A context re-created by cudaDeviceReset gets a new id, hence a new lookup.
void* symbol_address_cached(const void* symbol, cudaError_t* err);

// Counts one kernel launch (csa2_launch_count) and returns the launch status.
cudaError_t counted(cudaError_t launch_status);

// Launches a step kernel with programmatic stream serialisation (see
// pdl_trigger / pdl_wait in common.cuh) and counts it.
template <typename... KArgs, typename... Args>
cudaError_t launch_step(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                        Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return counted(cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...));
}

// Zeroes n uint32 (a step kernel; falls back to a memset for unaligned buffers).
cudaError_t launch_zero_u32(uint32_t* p, int64_t n, cudaStream_t s);

// ---- pack.cu ----------------------------------------------------------------
cudaError_t launch_pack_mxfp4(const float* x, int64_t n_rows, int d, uint8_t* codes,
                              uint8_t* scales, cudaStream_t s);
cudaError_t launch_unpack_mxfp4(const uint8_t* codes, const uint8_t* scales, int64_t n_rows,
                                int d, uint16_t* out, cudaStream_t s);
cudaError_t launch_pack_fp8(const float* x, int64_t n_rows, int d, uint8_t* codes,
                            float* scales, cudaStream_t s);
// Window rows of query tokens: row (b, i) of x [B][Tq][d] goes to window row
// q_pos[b][i] - pos0[b] of sequence b.
cudaError_t launch_pack_fp8_window(const float* x, int B, int Tq, int d, const int32_t* q_pos,
                                   const int32_t* pos0, int swa_cap, uint8_t* codes,
                                   float* scales, cudaStream_t s);

// Row source of the norm/rope/pack epilogue: either a plain fp32 latent
// [B][n_max][d] or n_split fp32 partial sums [n_split][M][ld] (compression).
struct LatentSource {
  const float* base;
  int64_t row_stride;    // elements between consecutive rows
  int64_t split_stride;  // elements between split-K partials (0: one split)
  int n_split;
};
// Per-layer caches of launch_norm_rope_pack_layers (at most kPackLayersMax layers per launch).
constexpr int kPackLayersMax = 64;
struct PackLayer {
  const int32_t* page_table;
  int64_t n_pages;
  uint8_t* kv_codes;
  uint8_t* kv_scales;
  void* idx_k;
};
struct PackLayers {
  int64_t col_stride;     // GEMM output columns between consecutive layers
  int64_t gamma_stride;   // gamma elements between consecutive layers
  PackLayer l[kPackLayersMax];
};
cudaError_t launch_norm_rope_pack_layers(LatentSource src, int B, int n_max, int d, int r, const float* gamma,
                                         float eps, float rope_base, const int32_t* first_entry, int max_pages,
                                         const float* idx_src, int64_t idx_row_stride, int Di, int idx_dtype,
                                         int kv_fp8, const PackLayers& layers, int n_layers, cudaStream_t s);
cudaError_t launch_norm_rope_pack(LatentSource src, int B, int n_max, int d, int r,
                                  const float* gamma, float eps, float rope_base,
                                  const int32_t* first_entry, const int32_t* n_rows,
                                  const int32_t* page_table, int max_pages, int64_t n_pages,
                                  uint8_t* kv_codes, uint8_t* kv_scales,
                                  // optional indexer-key epilogue (compression)
                                  const float* idx_src, int64_t idx_row_stride, int Di,
                                  int idx_dtype, void* idx_k, cudaStream_t s,
                                  // 1: FP8 main-KV rows (E4M3 codes [d], fp32 scale per entry)
                                  int kv_fp8 = 0);
// Window rows rebuilt from replayed tokens: row i of sequence b (latent = the
// split sum of src row b * n_tok + i) gets RMSNorm, RoPE at raw position
// tok_pos0[b] + i and the FP8 pack, into window row tok_pos0[b] + i - win_pos0[b].
cudaError_t launch_norm_rope_fp8_window(LatentSource src, int B, int n_tok, int d, int r,
                                        const float* gamma, float eps, float rope_base,
                                        const int32_t* tok_pos0, const int32_t* win_pos0, int swa_cap,
                                        uint8_t* codes, float* scales, cudaStream_t s);

// ---- compress.cu --------------------------------------------------------------
// C[split][m][n] = sum over the split's K-range of A[m][:] * Bw[n][:], where
// A rows are the g-token groups of hidden (g = 4: compression; g = 1: one
// token per row, the window-row projection) and Bw = [W; W_idx] (n < d: W).
size_t compress_partials_bytes(int B, int T, int H, int d, int Di, int* n_split_out, int g = 4);
cudaError_t launch_compress_gemm(const uint16_t* hidden, int B, int T, int H,
                                 const uint16_t* W, int d, const uint16_t* W_idx, int Di,
                                 float* partials, int n_split, cudaStream_t s, int g = 4);

// ---- indexer.cu ---------------------------------------------------------------
struct IndexerArgs {
  const void* q;      // [rows][Hi][Di]
  const float* w;     // [rows][Hi]
  const void* k;      // [n_pages][64][Di]
  const int32_t* page_table;
  const int32_t* n_entries;  // [B]
  const int32_t* q_pos;      // [rows]
  int B, Tq, Hi, Di, dtype, max_pages;
  int64_t n_pages;
  int max_entries;           // visible counts are clamped to this (buffer bound)
};
// Full: scores[row][j] for visible j; blockmax (nullable) per `block` entries;
// hist (nullable, zeroed by the caller): per-row 2048-bin key histogram for launch_topk.
// bm_hist (nullable, zeroed by the caller): the same for the block maxima, built only
// by the one-query-per-row page scan; *bm_hist_built says whether it was.
cudaError_t launch_index_scores(const IndexerArgs& a, float* scores, int64_t stride,
                                float* blockmax, int64_t bm_stride, int block, int max_entries,
                                uint32_t* hist, cudaStream_t s, uint32_t* bm_hist = nullptr,
                                bool* bm_hist_built = nullptr);
// ---- indexer_tc.cu: many query tokens per sequence (prefill) as a tcgen05 GEMM
// (bf16 keys, Hi = 8, Di = 128, Tq >= 32).  Scores and block maxima as above;
// builds no histogram (the Top-K kernel builds its own).
// Reindex from full score rows: the pooled positions' scores gathered into compact
// columns 8*slot + e of the same rows (in place), and the visible count per row.
cudaError_t launch_pool_compact(const IndexerArgs& a, const int32_t* pool, const int32_t* pool_cnt, int n_pool,
                                float* scores, int64_t stride, int32_t* n_valid, cudaStream_t s);
bool index_scores_gemm_supported(const IndexerArgs& a);
cudaError_t launch_index_scores_gemm(const IndexerArgs& a, float* scores, int64_t stride, float* blockmax,
                                     int64_t bm_stride, int max_entries, cudaStream_t s);
// Reindex: compact scores[row][p*block + e] of the pooled blocks' visible
// positions; n_valid[row] receives the compact count.
cudaError_t launch_index_scores_pool(const IndexerArgs& a, const int32_t* pool,
                                     const int32_t* pool_cnt, int n_pool, int block,
                                     float* scores, int64_t stride, int32_t* n_valid,
                                     cudaStream_t s);

// ---- topk.cu --------------------------------------------------------------------
// Number of valid columns of a row: n_valid[row] if given, else derived from
// (n_entries[row / Tq], q_pos[row]) and divided (rounding up) by `divisor`,
// else `stride`.
struct ValidSpec {
  const int32_t* n_valid;
  const int32_t* n_entries;
  const int32_t* q_pos;
  int Tq;
  int divisor;
  int64_t max_n;   // > 0: entry counts derived from n_entries are clamped to it first
};
// Optional index remap for Reindex: out = pool[row][c / block] * block + c % block.
struct Remap {
  const int32_t* pool;
  int64_t pool_stride;
  int block;
};
// hist (nullable): per-row 2048-bin histogram of the top 11 bits of the
// order-preserving score keys of the valid columns (built by the scoring kernel).
// max_n (> 0): a bound on every row's valid count below the stride (the row
// is then read as if it were that long; valid counts above it are reported
// as CSA2_STATUS_BAD_COUNT and clamped).
cudaError_t launch_topk(const float* scores, int64_t rows, int64_t stride, ValidSpec v, int k,
                        int32_t* out_idx, int32_t* out_cnt, Remap remap, const uint32_t* hist,
                        int64_t hist_stride, cudaStream_t s, int64_t max_n = 0);
// Split Top-K for few rows: many CTAs per row collect, one CTA per row
// finishes.  Needs the row histograms and topk_split_scratch_bytes of scratch.
size_t topk_split_scratch_bytes(int64_t rows, int64_t stride);
// Per-row 2048-bin histograms of the top 11 key bits of given scores (zeroed first).
cudaError_t launch_row_hist(const float* scores, int64_t rows, int64_t stride, ValidSpec v, uint32_t* hist,
                            cudaStream_t s);
cudaError_t launch_topk_split(const float* scores, int64_t rows, int64_t stride, ValidSpec v, int k,
                              int32_t* out_idx, int32_t* out_cnt, Remap remap, const uint32_t* hist,
                              int64_t hist_stride, void* scratch, cudaStream_t s);
// Block maxima of the valid columns: out[row][b] = max(scores[row][block*b ..]).
cudaError_t launch_block_max(const float* scores, int64_t rows, int64_t stride, ValidSpec v,
                             int block, float* out, int64_t out_stride, cudaStream_t s);

// ---- attention.cu -------------------------------------------------------------
struct AttnArgs {
  const uint16_t* Q;          // [rows][Hq][d] bf16
  const uint8_t* kv_codes;
  const uint8_t* kv_scales;
  const int32_t* page_table;
  int64_t n_pages;
  int max_pages;
  const int32_t* idx;         // [rows][K]
  const int32_t* cnt;         // [rows]
  const int32_t* q_pos;       // [rows]
  const int32_t* n_entries;   // [B]
  const uint8_t* swa_codes;   // [B][swa_cap][d]
  const float* swa_scales;    // [B][swa_cap]
  const int32_t* swa_pos0;    // [B]
  int swa_cap, W;
  int B, Tq, Hq, d, K;
  float scale;
  float* O;                   // [rows][Hq][d]
  float* lse;                 // [rows][Hq] or null
  int kv_fp8;                 // main KV as FP8 rows (E4M3 [d] + fp32 scale per entry)
};
cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t s);
// ---- attention_tc.cu: tcgen05 kernel for d = 512 (every Hq and K + W the ABI admits)
bool sparse_attn_tc_supported(const AttnArgs& a);
cudaError_t launch_sparse_attn_tc(const AttnArgs& a, cudaStream_t s);

}  // namespace csa2
