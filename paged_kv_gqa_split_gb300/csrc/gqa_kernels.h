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
constexpr int kErrTicket = 16;       // a split sequence's arrival ticket did not settle

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
  int* err;                // device error word (bit flags below)
  unsigned long long* tickets;  // [num_ctas][NG] arrival tickets of split sequences
  unsigned long long epoch;     // this call's ticket epoch (never 0, < 2^40)
  int batch;
  int min_units;
  float scale_log2;        // sm_scale * log2(e)
  int num_pages_check;     // > 0: page ids are range-checked against it
  int fuse_max_splits;     // split sequences of at most this many pieces are merged by the decode kernel
};

// Default: sequences cut into at most this many pieces are merged inside the
// decode kernel; longer splits go to the merge kernel.
constexpr int kDefaultFuseMaxSplits = 16;

// Merge CTAs per boundary between consecutive decode CTAs.
constexpr int kMergeCtasPerBoundary = 1;

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
  int use_pdl;
  int fuse_max_splits;  // sequences of at most this many pieces were merged by the decode kernel
};

// Compile-time variant of the decode kernel.
enum : int { kGatherLsu = 0, kGatherTma = 1 };

struct KernelChoice {
  int gather;         // kGatherLsu: self-loading warps with cp.async; kGatherTma: producer warp + bulk copies
  int heads_per_cta;  // NG: KV heads per CTA (4, 2 or 1)
  int tile;           // tokens per pipeline stage (16; 32 for the TMA variant)
  int stages;         // pipeline depth
};

int lsu_smem_bytes(int ng, int stages);
cudaError_t launch_decode_lsu(int ng, int stages, const DecodeParams& p, int num_ctas, cudaStream_t stream);
int tma_smem_bytes(int ng, int tile, int stages);
cudaError_t launch_decode_tma(int ng, int tile, int stages, const DecodeParams& p, int num_ctas, cudaStream_t stream);

// Shared memory of a variant, or -1 if it is not compiled in.
inline int decode_smem_bytes(const KernelChoice& k) {
  if (k.gather == kGatherLsu) return k.tile == 16 ? lsu_smem_bytes(k.heads_per_cta, k.stages) : -1;
  if (k.gather == kGatherTma) return tma_smem_bytes(k.heads_per_cta, k.tile, k.stages);
  return -1;
}

// Warps a variant runs per CTA and the most CTAs per SM worth launching.
inline int decode_max_ctas_per_sm(const KernelChoice& k) {
  // LSU: up to 16 gathering warps per SM; TMA: up to 4 consumer warps per SM.
  return k.gather == kGatherLsu ? 16 / k.heads_per_cta : 4 / k.heads_per_cta;
}

inline cudaError_t launch_decode(const KernelChoice& k, const DecodeParams& p, int num_ctas, cudaStream_t stream) {
  if (k.gather == kGatherLsu) return launch_decode_lsu(k.heads_per_cta, k.stages, p, num_ctas, stream);
  if (k.gather == kGatherTma) return launch_decode_tma(k.heads_per_cta, k.tile, k.stages, p, num_ctas, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_merge(int heads_per_cta, const MergeParams& p, cudaStream_t stream);
cudaError_t launch_validate(const int* indptr, const int* indices, int batch, int num_pages, int* err,
                            cudaStream_t stream);
cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int* slots, void* k_cache, void* v_cache,
                             int n, int num_pages, int sm_count, cudaStream_t stream);
cudaError_t read_and_clear_device_error(int* out);
cudaError_t device_error_word(int** ptr);  // device address of the error word (current device)

}  // namespace gqa
