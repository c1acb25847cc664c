// KV-cache append for the paged GQA decode path: scatter the K and V rows of
// new tokens into their pages.
//
// The row store of the split-K GQA path on the sigit.si vLLM "qsa.py" page
// (_store_qsa_rows_kernel): a row's slot is valid when it lies in
// [0, num_pages * page_size) and then cache[slot] = row; other slots (-1 for
// padding tokens) store nothing. Page size is 1 here, so a slot is a page id
// and a token's rows for all 4 KV heads (1 KB of K, 1 KB of V) move together.
//
// Pure data movement, bounded by HBM: 2 KB read and 2 KB written per token.
// One warp per token, each lane moving four 16-byte vectors (two of K, two of
// V); the source rows are streamed (read once), the pages are written with
// ordinary stores so the next decode finds them in L2 when it runs soon after.
#include <cuda_runtime.h>

#include <cstdint>

#include "gqa_kernels.h"
#include "gqa_plan.h"

namespace gqa {

constexpr int kAppendThreads = 256;
constexpr int kVec16PerPage = kPageBytes / 16;  // 64 x 16 B per 1 KB page

__global__ void __launch_bounds__(kAppendThreads) gqa_kv_append_kernel(const uint4* __restrict__ k_new,
                                                                       const uint4* __restrict__ v_new,
                                                                       const int* __restrict__ slots,
                                                                       uint4* __restrict__ k_cache,
                                                                       uint4* __restrict__ v_cache, int n,
                                                                       int num_pages) {
  const int lane = threadIdx.x & 31;
  const int warps = kAppendThreads / 32;
  const int stride = gridDim.x * warps;
  for (int r = blockIdx.x * warps + (threadIdx.x >> 5); r < n; r += stride) {
    const int slot = __ldg(slots + r);
    if (slot < 0 || slot >= num_pages) continue;  // warp-uniform: padding or out-of-pool slot
    const uint4* ks = k_new + static_cast<int64_t>(r) * kVec16PerPage;
    const uint4* vs = v_new + static_cast<int64_t>(r) * kVec16PerPage;
    const uint4 k0 = __ldcs(ks + lane), k1 = __ldcs(ks + 32 + lane);
    const uint4 v0 = __ldcs(vs + lane), v1 = __ldcs(vs + 32 + lane);
    uint4* kd = k_cache + static_cast<int64_t>(slot) * kVec16PerPage;
    uint4* vd = v_cache + static_cast<int64_t>(slot) * kVec16PerPage;
    kd[lane] = k0;
    kd[32 + lane] = k1;
    vd[lane] = v0;
    vd[32 + lane] = v1;
  }
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int* slots, void* k_cache, void* v_cache,
                             int n, int num_pages, int sm_count, cudaStream_t stream) {
  const int warps = kAppendThreads / 32;
  int grid = (n + warps - 1) / warps;
  const int cap = sm_count * (2048 / kAppendThreads);  // one full wave of resident CTAs
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  gqa_kv_append_kernel<<<grid, kAppendThreads, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slots, static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), n, num_pages);
  return cudaGetLastError();
}

}  // namespace gqa
