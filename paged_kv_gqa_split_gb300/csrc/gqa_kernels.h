// Internal interface between the C ABI (gqa_api.cu) and the kernels
// (gqa_decode.cu). Not part of the public header.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace gqa {

// Bits of the sticky device error word.
constexpr int kErrTimeoutFull = 1;   // a consumer waited too long for a stage's data
constexpr int kErrTimeoutEmpty = 2;  // the producer waited too long for a free stage
constexpr int kErrBadPage = 4;       // a kv_indices entry outside [0, num_pages)
constexpr int kErrBadIndptr = 8;     // kv_indptr not starting at 0 / decreasing

struct DecodeParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int* kv_indptr;
  const int* kv_indices;
  void* out;
  float* lse;
  float* part_o;    // [2 * num_ctas][NG][128 dims][8 heads] fp32
  float* part_lse;  // [2 * num_ctas][NG][8 heads] fp32
  const int* skip_if_set;  // optional: return without work if *skip_if_set != 0
  int batch;
  int min_units;
  float scale_log2;        // sm_scale * log2(e)
  int num_pages_check;     // > 0: page ids are range-checked against it
};

struct MergeParams {
  const int* kv_indptr;
  const float* part_o;
  const float* part_lse;
  void* out;
  float* lse;
  const int* skip_if_set;
  int batch;
  int num_decode_ctas;
  int min_units;
  int merge_ctas_per_boundary;
  int use_pdl;
};

// Compile-time variant of the decode kernel.
struct KernelChoice {
  int heads_per_cta;  // NG: KV heads per CTA (4, 2 or 1)
  int tile;           // tokens per pipeline stage (16 or 32)
  int stages;         // pipeline depth
};

int decode_smem_bytes(const KernelChoice& k);
cudaError_t launch_decode(const KernelChoice& k, const DecodeParams& p, int num_ctas, cudaStream_t stream);
cudaError_t launch_merge(int heads_per_cta, const MergeParams& p, cudaStream_t stream);
cudaError_t launch_validate(const int* indptr, const int* indices, int batch, int num_pages, int* err,
                            cudaStream_t stream);
cudaError_t read_and_clear_device_error(int* out);

}  // namespace gqa
