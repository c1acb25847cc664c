// gqa_paged_decode_noalloc: the decode entry point for callers that must not
// allocate device memory.
//
// gqa_paged_decode grows a library-owned workspace with cudaMalloc on first
// use (and whenever the tuning asks for a larger one). Some callers cannot let
// that happen: a serving runtime that reserves all free HBM up front for its
// KV-cache pool and owns every later allocation, a caller inside CUDA stream
// capture (where cudaMalloc is not a capturable operation), or a latency-
// critical loop that cannot afford cudaMalloc's implicit device-wide
// synchronisation. This entry point instead keeps the split partials in a
// fixed file-scope device array that the CUDA module loader places in every
// GPU that loads the library (and that stays resident until the process
// exits), so a call allocates nothing.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "gqa_kernels.h"
#include "gqa_paged_decode.h"

namespace {

// Scratch for the fp32 split partials (two slots per decode CTA). Its size is
// GQA_NOALLOC_SCRATCH_BYTES; a plan that would need more runs with fewer
// tier-2 CTAs.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GQA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device. In host code the
// array's name only denotes a host-side shadow, so the address must come from
// cudaGetSymbolAddress, once per device, with that device current.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // clear the sticky launch-independent error
      return GQA_ERR_LAUNCH;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return GQA_OK;
}

}  // namespace

extern "C" int gqa_paged_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* kv_indptr, const int32_t* kv_indices, float sm_scale,
                                        void* out, float* lse, int batch, struct CUstream_st* stream) {
  if (batch == 0) return GQA_OK;
  if (batch < 0) return GQA_ERR_INVALID_ARGUMENT;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != GQA_OK) return rc;
  // the plan is shrunk to the scratch (fewer tier-2 CTAs) rather than overrunning it
  return gqa::decode_in_scratch(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream,
                                scratch, static_cast<size_t>(GQA_NOALLOC_SCRATCH_BYTES));
}
