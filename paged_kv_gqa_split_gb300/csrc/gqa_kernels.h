// Internal interface between the C ABI (gqa_api.cu) and the kernels
// (gqa_decode_lsu.cu, gqa_decode_tma.cu, gqa_merge.cu). Not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "gqa_plan.h"

namespace gqa {

// Bits of the sticky device error word.
constexpr int kErrTimeoutFull = 1;   // a consumer waited too long for a stage's data
constexpr int kErrTimeoutEmpty = 2;  // the producer waited too long for a free stage
constexpr int kErrBadPage = 4;       // a kv_indices entry outside [0, num_pages)
constexpr int kErrBadIndptr = 8;     // kv_indptr not starting at 0 / decreasing
constexpr int kErrTicket = 16;       // a split sequence's arrival ticket did not settle
constexpr int kErrMergeWait = 32;    // an in-kernel merge waited too long for a sequence's pieces

struct DecodeParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int* kv_indptr;
  const int* kv_indices;
  void* out;
  float* lse;
  float* part_o;    // [2 * (P1 + P2)][NG][128 dims][8 heads] fp32
  float* part_lse;  // [2 * (P1 + P2)][NG][8 heads] fp32
  const int* skip_if_set;  // optional: return without work if *skip_if_set != 0
  int* err;                // device error word (bit flags below)
  unsigned long long* tickets;  // [P1 + P2][NG] arrival tickets of split sequences
  unsigned long long epoch;     // this call's ticket epoch (never 0, < 2^40)
  int4* split_rec;              // [P1 + P2] per-CTA split records for the merge kernel
  PlanConfig plan;              // the grid is plan.tier1_ctas + plan.tier2_ctas CTAs
  int batch;                    // sequences (sparse mode: query rows)
  int sparse_topk;              // 0: paged mode (kv_indptr / kv_indices); > 0: every row has this many
                                // columns and kv_indices holds their resolved slots (-1: masked out)
  int sparse_total;             // sparse mode: rows * sparse_topk (kv_indptr is not read)
  float scale_log2;        // sm_scale * log2(e)
  int num_pages_check;     // > 0: page ids are range-checked against it
  int fuse_max_splits;     // split sequences of at most this many pieces are merged by the decode kernel
  unsigned long long wait_limit_ns;  // give-up limit of a bounded wait (TMA variant; in-kernel merge)
  int inline_merge;             // one-wave mode: grid = tier-1 CTAs, tier 2 taken from `grab`, merge in-kernel
  unsigned long long* grab;     // [NG] one-wave mode: tier-2 range counters (epoch-tagged)
};

// One-wave mode: a warp walks at most this many ranges (its tier-1 range and
// tier-2 ranges); the host uses the mode only when P2 <= (this - 1) * P1.
constexpr int kMaxWarpRanges = 16;

// How a decode kernel is launched.
enum : int { kLaunchPlain = 0, kLaunchPdl = 1, kLaunchCooperative = 2 };

// Default give-up limit of a bounded mbarrier wait (the drain before exit keeps it).
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;

// Default: every split sequence goes to the merge kernel, whose CTAs share the
// work of one sequence; merging inside the decode kernel (the warp that brings
// a sequence's last piece combines its partials) is a tuning option for
// sequences cut into at most fuse_max_splits pieces.
constexpr int kDefaultFuseMaxSplits = 1;

// Merge CTAs per boundary between consecutive decode CTAs.
constexpr int kMergeCtasPerBoundary = 1;

struct MergeParams {
  const int* kv_indptr;
  const float* part_o;
  const float* part_lse;
  void* out;
  float* lse;
  const int* skip_if_set;
  const int4* split_rec;          // the decode CTAs' split records
  unsigned long long epoch;       // the call's epoch (tags the records)
  PlanConfig plan;  // the decode kernel's plan
  int batch;
  int sparse_topk;   // as in DecodeParams
  int sparse_total;
  int use_pdl;
  int fuse_max_splits;  // sequences of at most this many pieces were merged by the decode kernel
};

// Decode with the split partials in a fixed caller scratch (gqa_api.cu): a plan
// whose partials do not fit uses fewer tier-2 CTAs, down to none. Returns a
// GQA_* code (GQA_ERR_WORKSPACE if even the tier-1 partials do not fit).
int decode_in_scratch(const void* q, const void* k_cache, const void* v_cache, const int* kv_indptr,
                      const int* kv_indices, float sm_scale, void* out, float* lse, int batch, cudaStream_t stream,
                      void* scratch, size_t scratch_bytes);

// Dense MLA decode (gqa_mla.cu): one latent KV head of 576 values per token,
// 512 of them also V; `rows` = s_q * h_q query rows per sequence, a multiple
// of 16. The prep kernels fill kv_indptr_mut / slots_mut (workspace) from
// cache_seqlens and the block table; the decode and merge read them.
struct MlaParams {
  const void* q;             // [B][rows][576] bf16
  const void* kv;            // [num_blocks * page_size][576] bf16 (the cache, slot-major)
  const int* kv_indptr;      // [B + 1]
  int* kv_indptr_mut;        // the same buffer, written by the scan
  const int* slots;          // [T] slot of every cached token, -1 outside the pool
  int* slots_mut;
  void* out;                 // [B][rows][512] bf16
  float* lse;                // [B][h_q][s_q] fp32 natural log, or NULL
  float* part_o;             // [2 * CTAs][16][512] fp32
  float* part_lse;           // [2 * CTAs][16] fp32 (base 2)
  int4* split_rec;           // [2 * CTAs]
  int* err;
  PlanConfig plan;
  unsigned long long epoch;
  int batch, rows, h_q, s_q;
  float scale_log2;
  const int* block_table;  // [batch][width]
  int width, page_size, num_blocks;
  int piece_rows;  // query rows per piece (row group): 16, or 32 / 64 for the tensor-memory kernel's wide tiles
  // tensor-memory kernel, one tier: the first unit of each of the P1 CTAs (and the unit count at
  // [P1]), placed by the scan so that every CTA carries the same tokens plus piece_cost per sequence
  // start; NULL: the plan's equal ranges
  int64_t* bounds;
  int* cost_ptr;   // [B + 1] scratch of the scan: prefix of (length + piece_cost) over non-empty sequences
  int piece_cost;  // tokens one extra piece costs a CTA of the tensor-memory kernel
};

// MLA decode kernels: the tensor-memory kernel (block sizes that are a
// multiple of 32) and the mma.sync kernel with a 3-stage (3 CTAs per SM) or
// 4-stage (2 CTAs per SM) ring.
enum : int { kMlaKernelDefault = 0, kMlaKernelTensorMemory = 1, kMlaKernelMma3 = 3, kMlaKernelMma4 = 4 };
int mla_smem_bytes(int stages);
int mla_ctas_per_sm(int kind);
struct MlaTcMaps {  // 2D tensor maps of the latent cache (boxes of 64 x 32) and of Q (64 x 16)
  CUtensorMap kv;
  CUtensorMap q;
};
bool mla_tc_supported(int page_size);
int mla_tc_piece_rows(int rows);  // 64 / 32 when the rows of a sequence come in multiples of 64 / 32, else 16
bool mla_tc_encode(const MlaParams& p, MlaTcMaps* maps);
cudaError_t launch_mla_tc_decode(const MlaParams& p, const MlaTcMaps& maps, int ctas, cudaStream_t stream);
cudaError_t launch_mla(const MlaParams& p, const int* cache_seqlens, int kind, const MlaTcMaps* maps,
                       cudaStream_t stream);

// Compile-time variant of the decode kernel.
// kGatherLsuF8: FP8 caches only; kGatherLsuCc: the default's gather with the
// contractions on the CUDA cores (a comparison variant)
enum : int { kGatherLsu = 0, kGatherTma = 1, kGatherLsuF8 = 2, kGatherLsuCc = 3 };

struct KernelChoice {
  int gather;         // kGatherLsu: self-loading warps with cp.async; kGatherTma: producer warp + bulk copies
  int heads_per_cta;  // NG: KV heads per CTA (4, 2 or 1)
  int tile;           // tokens per pipeline stage (16; 32 for the TMA variant)
  int stages;         // pipeline depth
};

int lsu_smem_bytes(int ng, int stages);
int lsu_f8_smem_bytes(int stages, int tile);
int lsu_cc_smem_bytes();
cudaError_t launch_decode_lsu_cc(const DecodeParams& p, int num_ctas, cudaStream_t stream);
cudaError_t launch_decode_lsu_f8(int stages, int tile, const DecodeParams& p, int num_ctas, cudaStream_t stream,
                                 int launch);
cudaError_t launch_decode_lsu(int ng, int stages, const DecodeParams& p, int num_ctas, cudaStream_t stream,
                              int launch);
// The selected-token variant (p.sparse_topk > 0): 4 KV heads per CTA, 2 stages.
cudaError_t launch_decode_lsu_sparse(const DecodeParams& p, int num_ctas, cudaStream_t stream, int launch);
// CTAs of a cp.async variant (sparse: the selected-token one) that the current
// device holds at once; 0 for the TMA variant or if unknown.
int decode_coresident_ctas(const KernelChoice& k, bool sparse);
// Resolve the selected columns of a sparse batch to slots (-1: invalid column).
cudaError_t launch_sparse_resolve(const int* logical_indices, const int* block_table, const int* token_to_req,
                                  int* slots, int rows, int topk, int page_size, int page_table_width,
                                  int num_requests, int num_cache_blocks, int sm_count, cudaStream_t stream);
int tma_smem_bytes(int ng, int tile, int stages);
cudaError_t launch_decode_tma(int ng, int tile, int stages, const DecodeParams& p, int num_ctas, cudaStream_t stream);

// Shared memory of a variant, or -1 if it is not compiled in.
inline int decode_smem_bytes(const KernelChoice& k) {
  if (k.gather == kGatherLsu) return k.tile == 16 ? lsu_smem_bytes(k.heads_per_cta, k.stages) : -1;
  if (k.gather == kGatherTma) return tma_smem_bytes(k.heads_per_cta, k.tile, k.stages);
  if (k.gather == kGatherLsuF8) return k.heads_per_cta == 4 ? lsu_f8_smem_bytes(k.stages, k.tile) : -1;
  if (k.gather == kGatherLsuCc) return k.heads_per_cta == 4 && k.tile == 16 && k.stages == 2 ? lsu_cc_smem_bytes() : -1;
  return -1;
}

// Warps a variant runs per CTA and the most CTAs per SM worth launching.
inline int decode_max_ctas_per_sm(const KernelChoice& k) {
  // LSU: up to 16 gathering warps per SM; TMA: up to 4 consumer warps per SM; FP8 and the
  // CUDA-core variant: 3 CTAs (their launch bounds leave 170 registers per thread); FP8 with
  // 32-token stages: 2 (shared memory).
  if (k.gather == kGatherLsuF8) return k.tile == 32 ? 2 : 3;
  if (k.gather == kGatherLsuCc) return 3;
  return k.gather == kGatherLsu ? 16 / k.heads_per_cta : 4 / k.heads_per_cta;
}

inline cudaError_t launch_decode(const KernelChoice& k, const DecodeParams& p, int num_ctas, cudaStream_t stream,
                                 int launch) {
  if (k.gather == kGatherLsu) return launch_decode_lsu(k.heads_per_cta, k.stages, p, num_ctas, stream, launch);
  if (k.gather == kGatherTma) return launch_decode_tma(k.heads_per_cta, k.tile, k.stages, p, num_ctas, stream);
  if (k.gather == kGatherLsuF8) return launch_decode_lsu_f8(k.stages, k.tile, p, num_ctas, stream, launch);
  if (k.gather == kGatherLsuCc) return launch_decode_lsu_cc(p, num_ctas, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_merge(int heads_per_cta, const MergeParams& p, cudaStream_t stream);
cudaError_t launch_validate(const int* indptr, const int* indices, int batch, int num_pages, int* err,
                            cudaStream_t stream);
cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int* slots, void* k_cache, void* v_cache,
                             int n, int num_pages, int sm_count, cudaStream_t stream);
cudaError_t read_and_clear_device_error(int* out);
cudaError_t device_error_word(int** ptr);  // device address of the error word (current device)

// Raises a kernel's dynamic shared-memory limit to `bytes` once per device
// (`done` is the kernel's own flag table, zero-initialised static storage).
// Safe to call from several host threads at once: the attribute call is
// idempotent and the flags are atomic. Devices past the table set it on
// every call.
constexpr int kMaxDevices = 64;
inline cudaError_t set_smem_limit_once(std::atomic<int> (&done)[kMaxDevices], const void* fn, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < kMaxDevices;
  if (tracked && done[dev].load(std::memory_order_acquire) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && tracked) done[dev].store(1, std::memory_order_release);
  return e;
}

}  // namespace gqa
