/*
 * csa2.h -- C ABI of the CSA2 compressed-sparse-attention layer step (sm_103a).
 *
 * What the step computes follows "DeepSeek-V4.1 架构解析" (DeepSeek-V4.1
 * architecture analysis, blog.yuzhonghai.cloud), §02 "CSA2" and §03
 * "precision and state rebuild", with the 4:1 ratio also given by the
 * DeepSeek V4 review (wmrh.cn), §2.1-§2.2.  Where the pages leave a step open
 * this header fixes one reading; every such reading is marked READING.
 *
 * ---------------------------------------------------------------------------
 * Conventions (all entry points)
 *   - Every tensor pointer is caller-owned DEVICE memory unless stated.  The
 *     library allocates nothing and never synchronises the stream.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Every call returns CSA2_OK or an error code.  Arguments are validated on
 *     the host before anything is launched; on error nothing is launched and
 *     csa2_last_error() returns a message (thread-local, valid until the
 *     calling thread's next call).
 *   - Values held in device memory (page-table entries, entry counts, token
 *     positions, indices) cannot be checked on the host without a sync.  The
 *     kernels check them and skip an out-of-range access instead of making it;
 *     they then raise a flag in a device status word, which
 *     csa2_get_status() reads (and clears) after the caller syncs.
 *   - bf16 tensors are passed as uint16_t* (IEEE bfloat16 bit patterns).
 *   - All row-major; innermost dimension last.  Device pointers must be
 *     16-byte aligned.
 *
 * Shapes (names follow the pages):
 *   B   sequences;  Tq query tokens per sequence (1 for decode)
 *   d   latent width (64 or 512); r rotated channels at its end (even, <= d)
 *   Hq  attention query heads (1 .. 128; 64 in the pages' model)
 *   Hi, Di  indexer heads and head width (Hi <= 16, Di in {32, 64, 128})
 *   K   Top-K (1 .. 2048; 512 in the pages' model)
 *   W   sliding-window length in raw tokens (1 .. 1024; 128 in the pages)
 *
 * Data layout in HBM:
 *   KV page pool:    64 compressed entries per page.
 *     kv_codes  uint8 [n_pages][64][d/2]   E2M1 codes, channel 2i in the low
 *                                          nibble of byte i, 2i+1 in the high
 *     kv_scales uint8 [n_pages][64][d/16]  E4M3 scale codes, one per 16 channels
 *   (dims.kv_format = CSA2_KV_FP8, the V4-style main KV kept for comparison:
 *     kv_codes  uint8 [n_pages][64][d]     E4M3 codes
 *     kv_scales fp32  [n_pages][64]        one scale per entry, R5's rule;
 *     516 bytes per 512-d entry against MXFP4's 288.)
 *     idx_k     [n_pages][64][Di]          indexer keys (bf16 or fp32)
 *   page_table int32 [B][max_pages]: physical page of logical page p of
 *     sequence b; entry j of sequence b lives in page page_table[b][j/64],
 *     slot j%64.
 *   Window buffers:  swa_codes uint8 [B][swa_cap][d] (E4M3),
 *     swa_scales fp32 [B][swa_cap]; row i of sequence b is raw token
 *     swa_pos0[b] + i.
 *
 * READINGS fixed by this library (the pages leave these open):
 *   R1 compression: c_j = W * [h_4j; h_4j+1; h_4j+2; h_4j+3] (token-major
 *      concatenation, no bias); W is bf16 [d][4H]; a partial group makes no
 *      entry.
 *   R2 RMSNorm over all d channels: x = c / sqrt(mean(c^2) + eps) * gamma.
 *   R3 RoPE on the last r channels, rotate-half pairs (i, i + r/2),
 *      angle = p * base^(-2i/r), at p = 4j+3 (the entry's last token).
 *   R4 MXFP4: per 16 channels, scale = E4M3_rne_satfinite(amax / 6), codes =
 *      E2M1_rne_satfinite(x / scale) (fp32 IEEE division; ties to the even
 *      code; the sign bit is kept, so -0 is code 0x8); a scale that rounds
 *      to 0 makes all 16 codes +0.  Dequantised values e2m1 * e4m3 are exact
 *      in bf16 and in fp16.
 *   R5 FP8 window: per raw token, scale = amax / 448 (fp32, stored fp32),
 *      codes = E4M3_rne_satfinite(x / scale); scale 0 gives zero codes; the
 *      attention operand is bf16_rne(fp32(e4m3 * scale)).
 *   R6 index score s_j = sum_h w_h * ReLU(q_h . k_j), fp32 accumulation.
 *   R7 causality: entry j is visible to the token at raw position t iff
 *      4j + 3 <= t, i.e. j < min(n_entries, floor((t+1)/4)).
 *   R8 Top-K: the K highest scores (equal scores -> lower index; scores that
 *      are zero compare equal whatever their sign; NaN scores are not
 *      supported); if fewer than K entries are visible, all of them.  Output
 *      is the set in ascending index order, padded with -1, plus its count.
 *   R9 block pool: block b = entries 8b..8b+7; block score = max over its
 *      visible entries; the n_pool_blocks (2048) best blocks by (score desc,
 *      id asc), all visible blocks if fewer; output ascending, -1 padded.
 *   R10 Reindex scores the visible positions of the pooled blocks with its
 *      own indexer query against the shared indexer keys and keeps the Top-K
 *      (ties -> lower entry index).  Reuse copies the indices unchanged.
 *   R11 attention: K = V = the dequantised latent (one shared KV head); one
 *      softmax over {selected entries} U {window rows at raw positions
 *      max(0, t-W+1) .. t that the window buffer holds}, logits
 *      q . k * softmax_scale (1/sqrt(d) in the pages' model), no sink; a
 *      key in both sets counts twice.  O is fp32, lse (natural log) optional.
 *      Operand range: the products run on fp16 tensor-core operands with fp32
 *      accumulation.  Every bf16 value keeps all its bits there: each head of
 *      Q is scaled by a power of two that puts its largest magnitude in
 *      [2^14, 2^15) (values below 2^-31 of that largest one lose bits), and a
 *      window row whose scale lies outside [2^-8, 2^7] is dequantised with
 *      the scale times 2^-f (f = floor(log2 scale), clamped to [-100, 100]),
 *      its logits and softmax weights corrected by the same power.  MXFP4
 *      values (<= 2688 in magnitude, >= 2^-10) need none.  Logits must stay
 *      finite in fp32.
 *   R12 the indexer key of a new entry (Full layer with compression) is
 *      W_idx * [h_4j; ..; h_4j+3], rounded to the indexer dtype.
 *   R13 SWA Bounded Replay (csa2_swa_replay): a rebuilt window row is the
 *      replayed token's own latent RoPE_t(RMSNorm(W_swa h_t)) at its raw
 *      position t, packed as R5; the rebuilt window starts at the first
 *      replayed token.
 * ---------------------------------------------------------------------------
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define CSA2_OK 0
#define CSA2_ERR_INVALID_ARG 1 /* a pointer, size or alignment is wrong      */
#define CSA2_ERR_UNSUPPORTED 2 /* a valid shape this build has no kernel for */
#define CSA2_ERR_CUDA 3        /* a launch failed; see csa2_last_error()     */
#define CSA2_ERR_WORKSPACE 4   /* workspace NULL or smaller than required    */
#define CSA2_ERR_DEVICE_DATA 5 /* csa2_get_status: a kernel met bad device data */

/* element types of the indexer query / key */
#define CSA2_F32 0
#define CSA2_BF16 1

/* main-KV formats (dims.kv_format) */
#define CSA2_KV_MXFP4 0 /* E2M1 codes + E4M3 scale per 16 channels (V4.1, the pages' format) */
#define CSA2_KV_FP8 1   /* E4M3 codes + fp32 scale per entry (V4-style, for the A/B)       */

/* layer modes (static per layer) */
#define CSA2_MODE_FULL 0    /* compute KV (optional), score all, Top-K   */
#define CSA2_MODE_REINDEX 1 /* rescore the Full layer's pool, Top-K      */
#define CSA2_MODE_REUSE 2   /* take the previous layer's indices         */

/* status-word bits set by kernels that met bad device-resident data */
#define CSA2_STATUS_BAD_PAGE 1u     /* page-table entry outside [0, n_pages)  */
#define CSA2_STATUS_BAD_INDEX 2u    /* an index outside the visible entries   */
#define CSA2_STATUS_BAD_COUNT 4u    /* a count or position out of range       */
#define CSA2_STATUS_TIMEOUT 8u      /* a bounded on-chip wait gave up; outputs of that launch are invalid */

/* ABI version of this header (bumped on any incompatible change). */
#define CSA2_ABI_VERSION 2

int csa2_abi_version(void);

/* Number of kernels this library has launched in this process (all devices,
 * all threads).  Used to count launches inside a timed region. */
uint64_t csa2_launch_count(void);

/* Message of the last error of the calling thread ("" if none). */
const char* csa2_last_error(void);

/* Reads and clears the device status word (CSA2_STATUS_* bits) for the
 * current device.  Blocks until the stream's prior work is done.  Returns
 * CSA2_OK, or CSA2_ERR_CUDA if the copy failed; *bits receives the flags. */
int csa2_get_status(uint32_t* bits, void* stream);

/* Shapes shared by the entry points. */
typedef struct csa2_dims {
  int32_t B;             /* sequences                                      */
  int32_t Tq;            /* query tokens per sequence                      */
  int32_t d;             /* latent width: 64 or 512                        */
  int32_t r;             /* rotated channels at the end of the latent      */
  int32_t Hq;            /* attention query heads                          */
  int32_t Hi;            /* indexer heads                                  */
  int32_t Di;            /* indexer head width                             */
  int32_t idx_dtype;     /* CSA2_BF16 or CSA2_F32 (indexer q and k)        */
  int32_t K;             /* Top-K                                          */
  int32_t W;             /* window length in raw tokens                    */
  int32_t max_pages;     /* row length of the page table                   */
  int32_t n_pool_blocks; /* hierarchical pool: blocks kept (2048)          */
  int32_t pool_block;    /* hierarchical pool: entries per block (8)       */
  int32_t swa_cap;       /* rows per sequence in the window buffers        */
  int32_t kv_format;     /* CSA2_KV_MXFP4 (0) or CSA2_KV_FP8 (FP8 needs d = 512) */
} csa2_dims;

/* The shared compressed cache of one layer group. */
typedef struct csa2_cache {
  uint8_t* kv_codes;         /* [n_pages][64][d/2] (FP8: [n_pages][64][d])   */
  uint8_t* kv_scales;        /* [n_pages][64][d/16] (FP8: fp32 [n_pages][64]) */
  void* idx_k;               /* [n_pages][64][Di], idx_dtype                 */
  const int32_t* page_table; /* [B][max_pages]                               */
  const int32_t* n_entries;  /* [B] entries present (device)                 */
  int64_t n_pages;           /* physical pages in the pool                   */
} csa2_cache;

/* The sliding window of one layer. */
typedef struct csa2_window {
  uint8_t* codes;            /* [B][swa_cap][d] E4M3                         */
  float* scales;             /* [B][swa_cap]                                 */
  const int32_t* pos0;       /* [B] raw position of row 0 (device)           */
} csa2_window;

/* ---- a3: MXFP4 pack of a given fp32 array (bit-exact contract, R4) -------
 * x fp32 [n_rows][d] -> codes uint8 [n_rows][d/2], scales uint8 [n_rows][d/16].
 * d: multiple of 16, <= 4096.  n_rows may be 0 (no launch). */
int csa2_pack_mxfp4_f32(const float* x, int64_t n_rows, int32_t d, uint8_t* codes,
                        uint8_t* scales, void* stream);

/* Dequantise MXFP4 rows to bf16 (exact, R4).  out uint16 [n_rows][d]. */
int csa2_unpack_mxfp4_bf16(const uint8_t* codes, const uint8_t* scales, int64_t n_rows,
                           int32_t d, uint16_t* out, void* stream);

/* ---- a10: FP8 window pack (bit-exact contract, R5) ------------------------
 * x fp32 [n_rows][d] -> codes uint8 [n_rows][d], scales fp32 [n_rows].
 * d: multiple of 16, <= 4096. */
int csa2_pack_swa_fp8(const float* x, int64_t n_rows, int32_t d, uint8_t* codes,
                      float* scales, void* stream);

/* ---- a2+a3 on a given latent: RMSNorm, RoPE, MXFP4, paged store ----------
 * latent fp32 [B][n_max][d]; rows i < n_rows[b] of sequence b become entries
 * first_entry[b] + i (R2, R3 at position 4(first_entry[b]+i)+3, R4) and are
 * written into the page pool through page_table.  gamma fp32 [d].
 * first_entry, n_rows: int32 [B], device.  d in {64, 512}; r even, <= d. */
int csa2_norm_rope_pack(const float* latent, int32_t B, int32_t n_max, int32_t d, int32_t r,
                        const float* gamma, float eps, float rope_base,
                        const int32_t* first_entry, const int32_t* n_rows,
                        const int32_t* page_table, int32_t max_pages, int64_t n_pages,
                        uint8_t* kv_codes, uint8_t* kv_scales, void* stream);

/* The same for the FP8 main-KV format (dims.kv_format = CSA2_KV_FP8): after
 * RMSNorm and RoPE each entry row is packed by R5's rule (scale = amax / 448,
 * stored fp32; codes = E4M3_rne_satfinite(x / scale)) into kv_codes uint8
 * [n_pages][64][d] and kv_scales fp32 [n_pages][64].  The V4 review and the
 * V4.1 analysis (§03) describe V4's main KV as FP8; this format exists to
 * compare the two on the same path.  d = 512 only. */
int csa2_norm_rope_pack_fp8(const float* latent, int32_t B, int32_t n_max, int32_t d, int32_t r,
                            const float* gamma, float eps, float rope_base,
                            const int32_t* first_entry, const int32_t* n_rows,
                            const int32_t* page_table, int32_t max_pages, int64_t n_pages,
                            uint8_t* kv_codes, float* kv_scales, void* stream);

/* ---- a1-a4: compress new tokens into the paged cache ----------------------
 * hidden bf16 [B][T][H] (the new tokens of every sequence, token 0 at raw
 * position 4*first_entry[b]); W bf16 [d][4H]; gamma fp32 [d]; W_idx bf16
 * [Di][4H] or NULL; idx_k receives the new indexer keys (R12) when W_idx is
 * given.  Entries first_entry[b] .. first_entry[b] + T/4 - 1 are written.
 * Needs csa2_compress_workspace_size() bytes of workspace.
 * H: multiple of 64 (so 4H is a multiple of 256); d in {64, 512}. */
size_t csa2_compress_workspace_size(int32_t B, int32_t T, int32_t H, int32_t d, int32_t Di);
int csa2_compress_pack(const uint16_t* hidden, int32_t B, int32_t T, int32_t H,
                       const uint16_t* W, const float* gamma, float eps, float rope_base,
                       const uint16_t* W_idx, const int32_t* first_entry,
                       const csa2_dims* dims, const csa2_cache* cache,
                       void* ws, size_t ws_bytes, void* stream);

/* ---- a1-a4 for several layers from one hidden state --------------------------
 * "DeepSeek-V4.1 架构解析" §01 (causal encoder-decoder): every decoder layer
 * projects its KV from the same hidden state (the last encoder layer's) with
 * its own compression weights.  One GEMM over the layers' stacked weights,
 * then each layer's RMSNorm, RoPE, MXFP4 pack and paged store (R1-R4, R12)
 * into its own cache.
 * hidden bf16 [B][T][H] as for csa2_compress_pack; W_all bf16 [L][d + Di][4H]
 * (layer l: rows 0..d-1 its W, rows d..d+Di-1 its W_idx); Di = 0 (no indexer
 * keys written) or dims->Di; gamma_all fp32 [L][d]; caches: host array of L
 * caches sharing dims (page tables, entry counts and pools may differ).
 * Entries first_entry[b] .. first_entry[b] + T/4 - 1 of every layer's cache
 * are written.  Needs csa2_compress_layers_workspace_size() bytes of workspace.
 * H: multiple of 64; d in {64, 512}; L >= 1. */
size_t csa2_compress_layers_workspace_size(int32_t B, int32_t T, int32_t H, int32_t L, int32_t d, int32_t Di);
int csa2_compress_layers(const uint16_t* hidden, int32_t B, int32_t T, int32_t H, int32_t L,
                         const uint16_t* W_all, int32_t Di, const float* gamma_all, float eps,
                         float rope_base, const int32_t* first_entry, const csa2_dims* dims,
                         const csa2_cache* caches, void* ws, size_t ws_bytes, void* stream);

/* ---- SWA Bounded Replay: a layer's window rebuilt from its last tokens -------
 * "DeepSeek-V4.1 架构解析" §03 (SWA Bounded Replay): the window KV is not kept
 * in the persistent cache; a layer rebuilds it by replaying only the last
 * n_win (128) raw tokens, and tokens early in the replay see a shorter
 * window than the exact state would give them.
 * READING R13: the window row of raw token t is that token's own latent,
 * x_t = RoPE_t(RMSNorm(W_swa h_t)): W_swa bf16 [d][H] without bias, R2's
 * RMSNorm with gain gamma, R3's rotation at t itself (not at an entry
 * position), then R5's FP8 pack.  With the window buffer's first row at the
 * first replayed position, R11 gives a replayed token at p the rows
 * max(first replayed position, p - W + 1) .. p.
 * hidden bf16 [B][n_tok][H]: this layer's hidden states of the replayed
 * tokens, row i of sequence b at raw position tok_pos0[b] + i (tok_pos0 int32
 * [B], device); gamma fp32 [d].  Row i of sequence b is written to window
 * row tok_pos0[b] + i - win->pos0[b]; a row outside [0, dims->swa_cap), or at
 * a negative raw position, is not written and raises CSA2_STATUS_BAD_COUNT.
 * Uses dims->B, d, r and swa_cap (the struct is validated as for every entry
 * point).  Needs csa2_swa_replay_workspace_size() bytes of workspace.
 * H: multiple of 64; d in {64, 512}. */
size_t csa2_swa_replay_workspace_size(int32_t B, int32_t n_tok, int32_t H, int32_t d);
int csa2_swa_replay(const uint16_t* hidden, int32_t B, int32_t n_tok, int32_t H, const uint16_t* W_swa,
                    const float* gamma, float eps, float rope_base, const int32_t* tok_pos0,
                    const csa2_dims* dims, const csa2_window* win, void* ws, size_t ws_bytes,
                    void* stream);

/* ---- a5: index scores of every visible entry (R6, R7) ----------------------
 * idx_q [B][Tq][Hi][Di] (idx_dtype), w fp32 [B][Tq][Hi], q_pos int32 [B][Tq].
 * scores fp32 [B*Tq][score_stride]: column j < n_vis(row) receives s_j;
 * other columns are not written.  blockmax (NULL or fp32
 * [B*Tq][bm_stride]): column b < ceil(n_vis/pool_block) receives the block
 * maximum (R9).  score_stride >= max visible entries of any row. */
int csa2_index_scores(const csa2_dims* dims, const csa2_cache* cache, const void* idx_q,
                      const float* w, const int32_t* q_pos, float* scores,
                      int64_t score_stride, float* blockmax, int64_t bm_stride, void* stream);

/* ---- a6: Top-K of a given fp32 array (bit-exact contract, R8) -------------
 * scores fp32 [rows][stride]; n_valid int32 [rows] (device) or NULL (all
 * `stride` columns valid).  out_idx int32 [rows][k] ascending, -1 padded;
 * out_cnt int32 [rows].  k in 1..4096; stride < 2^31.  With a workspace of
 * csa2_topk_workspace_size() bytes each row is spread over many CTAs (for few,
 * long rows); with ws == NULL one CTA handles each row.  Same result. */
size_t csa2_topk_workspace_size(int64_t rows, int64_t stride, int32_t k);
int csa2_topk_f32(const float* scores, int64_t rows, int64_t stride, const int32_t* n_valid,
                  int32_t k, int32_t* out_idx, int32_t* out_cnt, void* ws, size_t ws_bytes,
                  void* stream);

/* ---- a7: block pool of a given fp32 score array (bit-exact contract, R9) --
 * scores fp32 [rows][stride], n_valid int32 [rows] entries valid per row.
 * out_pool int32 [rows][n_pool_blocks] ascending block ids, -1 padded;
 * out_pool_cnt int32 [rows]; out_blockmax (NULL or fp32 [rows][ceil(stride/block)]). */
int csa2_block_pool_f32(const float* scores, int64_t rows, int64_t stride, const int32_t* n_valid,
                        int32_t block, int32_t n_pool_blocks, int32_t* out_pool,
                        int32_t* out_pool_cnt, float* out_blockmax, void* ws, size_t ws_bytes,
                        void* stream);

/* ---- a5+a6 (+a7) Full, or a8 Reindex: indexer and Top-K in one call -------
 * Full (pool == NULL): scores every visible entry, keeps Top-K into out_idx /
 * out_cnt; if out_pool != NULL also builds the hierarchical pool (R9).
 * Reindex (pool != NULL, pool_cnt int32 [B*Tq]): scores only the pooled
 * positions (R10).  Scratch: csa2_index_topk_workspace_size() bytes. */
size_t csa2_index_topk_workspace_size(const csa2_dims* dims, int32_t max_entries);
int csa2_index_topk(const csa2_dims* dims, const csa2_cache* cache, const void* idx_q,
                    const float* w, const int32_t* q_pos, const int32_t* pool,
                    const int32_t* pool_cnt, int32_t* out_idx, int32_t* out_cnt,
                    int32_t* out_pool, int32_t* out_pool_cnt, int32_t max_entries,
                    void* ws, size_t ws_bytes, void* stream);

/* ---- csa2_index_topk without a caller workspace ---------------------------
 * No counterpart in the paper: a convenience for callers that cannot
 * allocate device memory (for example code that runs while a CUDA graph is
 * being captured, or a serving thread that must never wait on the
 * allocator).  Same arguments and results as csa2_index_topk, but the scratch
 * lives in one fixed 8 MiB array inside the library
 * (csa2_index_topk_noalloc_capacity() bytes), held by every GPU that loads
 * the library until the process exits.  Shapes whose
 * csa2_index_topk_workspace_size() exceeds it are rejected with
 * CSA2_ERR_WORKSPACE.  The first call in a CUDA context looks the array's
 * device address up (cudaGetSymbolAddress) with that context current and
 * caches it for that context; a context re-created by cudaDeviceReset is
 * looked up again.  Make the first call in a context before any stream
 * capture.  The call clears the part of the array that
 * must start at zero.  All calls share the one array: calls that can overlap
 * on the GPU (different streams without ordering between them) race and give
 * wrong results; order them on one stream.  Allocates nothing. */
size_t csa2_index_topk_noalloc_capacity(void);
int csa2_index_topk_noalloc(const csa2_dims* dims, const csa2_cache* cache, const void* idx_q,
                            const float* w, const int32_t* q_pos, const int32_t* pool,
                            const int32_t* pool_cnt, int32_t* out_idx, int32_t* out_cnt,
                            int32_t* out_pool, int32_t* out_pool_cnt, int32_t max_entries,
                            void* stream);

/* ---- a11: gathered sparse MQA attention + FP8 window (R11) ----------------
 * Q bf16 [B][Tq][Hq][d] (already rotated at its own position); idx int32
 * [B][Tq][K] (-1 padded) with cnt int32 [B][Tq]; O fp32 [B][Tq][Hq][d];
 * lse fp32 [B][Tq][Hq] or NULL.  d must be 512 or 64. */
int csa2_sparse_attn(const csa2_dims* dims, const csa2_cache* cache, const csa2_window* win,
                     const uint16_t* Q, const int32_t* q_pos, const int32_t* idx,
                     const int32_t* cnt, float softmax_scale, float* O, float* lse,
                     void* stream);

/* ---- one layer step in any mode -------------------------------------------
 * FULL    : [compress new tokens if hidden != NULL] [pack window rows of the
 *           new tokens if swa_new != NULL] -> index + Top-K (+ pool if
 *           hierarchical) -> attention.
 * REINDEX : [pack window rows] -> pooled rescoring (pool/pool_cnt read) ->
 *           attention.
 * REUSE   : [pack window rows] -> idx_out/cnt_out = idx_in/cnt_in (copied
 *           unless the same buffers) -> attention.
 * swa_new fp32 [B][Tq][d]: window latent of the query tokens, written to
 * window row q_pos - pos0.  Scratch: csa2_layer_workspace_size() bytes. */
typedef struct csa2_layer_args {
  int32_t mode;              /* CSA2_MODE_*                                  */
  int32_t hierarchical;      /* FULL: also build the pool                    */
  csa2_dims dims;
  csa2_cache cache;
  csa2_window window;
  const int32_t* q_pos;      /* [B][Tq]                                      */
  int32_t max_entries;       /* upper bound of any n_entries[b]              */
  /* FULL only, optional compression of the new tokens (hidden == NULL: none) */
  const uint16_t* hidden;    /* bf16 [B][T][H]                               */
  int32_t T, H;
  const uint16_t* W_c;       /* bf16 [d][4H]                                 */
  const uint16_t* W_idx;     /* bf16 [Di][4H] or NULL                        */
  const float* gamma;        /* fp32 [d]                                     */
  float eps, rope_base;
  const int32_t* first_entry;/* [B]                                          */
  /* optional window rows of the query tokens (NULL: none) */
  const float* swa_new;      /* fp32 [B][Tq][d]                              */
  /* indexer query (FULL, REINDEX) */
  const void* idx_q;         /* [B][Tq][Hi][Di]                              */
  const float* idx_w;        /* [B][Tq][Hi]                                  */
  /* attention */
  const uint16_t* Q;         /* bf16 [B][Tq][Hq][d]                          */
  float softmax_scale;
  /* indices */
  const int32_t* idx_in;     /* REUSE: [B][Tq][K]                            */
  const int32_t* cnt_in;     /* REUSE: [B][Tq]                               */
  int32_t* idx_out;          /* [B][Tq][K]                                   */
  int32_t* cnt_out;          /* [B][Tq]                                      */
  int32_t* pool;             /* [B][Tq][n_pool_blocks]: FULL+hier writes, REINDEX reads */
  int32_t* pool_cnt;         /* [B][Tq]                                      */
  /* outputs */
  float* O;                  /* [B][Tq][Hq][d]                               */
  float* lse;                /* [B][Tq][Hq] or NULL                          */
} csa2_layer_args;

size_t csa2_layer_workspace_size(const csa2_layer_args* a);
int csa2_layer(const csa2_layer_args* a, void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
