// Column resolution of the selected-token (sparse) paged GQA decode.
//
// The sparse split-K GQA kernel of the sigit.si vLLM "qsa.py" page
// (_qsa_sparse_paged_gqa_splitk_kernel) looks up, for every selected column of
// a query row, the row's request, the logical page of the selected position
// in that request's block table, and the physical page. It drops the column
// when any of them is out of range. This kernel does that lookup once for
// the whole batch and writes the physical slot (page * page_size + offset) of
// every column, or -1 for a dropped one. The decode kernel then gathers
// through the slots as it gathers through kv_indices, with the -1 columns
// masked out of the softmax.
//
// Traffic: 4 B of index, 4 B of token_to_req (cached), 4 B of block table
// and 4 B written per column, against 2 KB of K/V rows per column in the
// decode that follows.
#include <cuda_runtime.h>

#include <cstdint>

#include "gqa_kernels.h"
#include "gqa_ptx.cuh"

namespace gqa {

constexpr int kResolveThreads = 256;

__global__ void __launch_bounds__(kResolveThreads)
    gqa_sparse_resolve_kernel(const int* __restrict__ logical_indices, const int* __restrict__ block_table,
                              const int* __restrict__ token_to_req, int* __restrict__ slots, int64_t n, int topk,
                              int page_size, int page_table_width, int num_requests, int num_cache_blocks) {
  // The decode grid may become resident now; it waits for this grid's slots
  // before its first gather.
  pdl_launch_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int row = static_cast<int>(i / topk);
    const int req = __ldg(token_to_req + row);
    const int t = __ldg(logical_indices + i);
    int slot = -1;
    if (req >= 0 && req < num_requests && t >= 0) {
      const int lp = t / page_size;
      if (lp < page_table_width) {
        const int page = __ldg(block_table + static_cast<int64_t>(req) * page_table_width + lp);
        // page * page_size + offset < num_cache_blocks * page_size, which the host keeps within int32
        if (page >= 0 && page < num_cache_blocks) slot = page * page_size + (t - lp * page_size);
      }
    }
    slots[i] = slot;
  }
}

cudaError_t launch_sparse_resolve(const int* logical_indices, const int* block_table, const int* token_to_req,
                                  int* slots, int rows, int topk, int page_size, int page_table_width,
                                  int num_requests, int num_cache_blocks, int sm_count, cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(rows) * topk;
  int64_t grid = (n + kResolveThreads - 1) / kResolveThreads;
  const int64_t cap = static_cast<int64_t>(sm_count) * (2048 / kResolveThreads);
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  gqa_sparse_resolve_kernel<<<static_cast<int>(grid), kResolveThreads, 0, stream>>>(
      logical_indices, block_table, token_to_req, slots, n, topk, page_size, page_table_width, num_requests,
      num_cache_blocks);
  return cudaGetLastError();
}

}  // namespace gqa
