// Indexer + Top-K for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside a CUDA
// graph being captured, a host thread of a serving loop that must never
// block on the allocator, or an embedding that owns every byte of the device
// heap and hands out only fixed buffers.  For them this file keeps the
// scratch that csa2_index_topk needs (score rows, block maxima, valid counts,
// key histograms) in one file-scope device array of fixed size.  The array
// exists once per GPU that loads the library and lives until the process
// exits; every call shares it.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace csa2 {

// 8 MiB: enough for, e.g., 32 decode rows over 32,768 entries each.
constexpr size_t kNoAllocScratchBytes = 8u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

}  // namespace csa2

using namespace csa2;

extern "C" size_t csa2_index_topk_noalloc_capacity(void) { return kNoAllocScratchBytes; }

extern "C" int csa2_index_topk_noalloc(const csa2_dims* dims, const csa2_cache* cache, const void* idx_q,
                                       const float* w, const int32_t* q_pos, const int32_t* pool,
                                       const int32_t* pool_cnt, int32_t* out_idx, int32_t* out_cnt,
                                       int32_t* out_pool, int32_t* out_pool_cnt, int32_t max_entries,
                                       void* stream) {
  if (!dims) return report_error(CSA2_ERR_INVALID_ARG, "dims must not be NULL");
  const size_t need = csa2_index_topk_workspace_size(dims, max_entries);
  if (need > kNoAllocScratchBytes)
    return report_error(CSA2_ERR_WORKSPACE,
                        "csa2_index_topk_noalloc: this shape needs more scratch than the fixed 8 MiB "
                        "device array (check csa2_index_topk_workspace_size); use csa2_index_topk with "
                        "a caller-allocated workspace instead");
  // device address of the array in the current context (looked up once per context,
  // with that context current, then cached; see symbol_address_cached)
  cudaError_t e = cudaSuccess;
  void* scratch = symbol_address_cached(reinterpret_cast<const void*>(&g_noalloc_scratch), &e);
  if (!scratch)
    return report_error(CSA2_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e)
                                                        : "csa2_index_topk_noalloc: no device address for the scratch");
  // the histogram part of the scratch is cleared by the call itself; the rest
  // is written before it is read
  return index_topk_into(dims, cache, idx_q, w, q_pos, pool, pool_cnt, out_idx, out_cnt, out_pool,
                         out_pool_cnt, max_entries, scratch, kNoAllocScratchBytes,
                         static_cast<cudaStream_t>(stream));
}
