// LSE merge of split partials, page-table validation and the device error
// word of the paged GQA decode library.
//
// Merge: for a sequence cut into S pieces at decode-CTA boundaries, combine the
// fp32 partials (O_i, LSE_i) with weights w_i = 2^(LSE_i - max LSE) into
// O = sum w_i O_i / sum w_i (bf16) and LSE = max + log2 sum w_i, the merge of
// the split-K GQA path on the sigit.si vLLM "qsa.py" page
// (_qsa_merge_splitk_kernel) plus the merged LSE. It also writes the empty
// sequences (O = 0, LSE = -inf, the early-exit rule of the kernelindex.com page
// "gqa_paged_decode_h32_kv4_d128_ps1").
#include <cuda_runtime.h>

#include "gqa_common.cuh"
#include "gqa_kernels.h"

namespace gqa {

// Sticky device-side error word (bit flags, see gqa_kernels.h). Only set on
// conditions that should never occur with valid inputs; read by the host API.
__device__ int g_device_error;

// -------------------------------------------------------------------- merge
// One CTA per boundary between decode CTAs j and j + 1; it merges the sequence
// cut there only if that sequence has more pieces than the decode kernel
// merges itself (fuse_max_splits). Decode CTA j leaves a 16-byte record of how
// the sequence holding its last unit is cut, so after the decode grid
// completes a merge CTA needs one load to find its work, then one round of
// loads of the partials: each split's LSE and O are folded in with a running
// maximum, so the weights need no second pass. With 6 KB of shared memory, one
// merge CTA fits beside three decode CTAs on an SM (programmatic dependent
// launch) and starts before the decode grid has drained.
constexpr int kMergeThreads = 128;
constexpr int kMergeWarps = kMergeThreads / 32;
// Split counts up to this: one warp per (head, 32-dim chunk) item, all splits;
// above it, the block path spreads each sequence over its boundary CTAs.
constexpr int kMergeSmallSplits = 16;

template <int NG>
__device__ __forceinline__ const float* partial_lse_row(const MergeParams& p, const SeqSplit& sp, int s, int g) {
  const int64_t sid = slot_id(sp.first_cta + s, s == 0 ? sp.first_slot : 0);
  return p.part_lse + (sid * NG + g) * kGroup;
}

template <int NG>
__device__ __forceinline__ const float* partial_o_row(const MergeParams& p, const SeqSplit& sp, int s, int g, int d) {
  const int64_t sid = slot_id(sp.first_cta + s, s == 0 ? sp.first_slot : 0);
  return p.part_o + ((sid * NG + g) * kHeadDim + d) * kGroup;
}

// Running LSE-weighted sum over splits for 8 heads of one dim:
// m = max lse seen, den = sum 2^(lse_i - m), acc = sum 2^(lse_i - m) O_i.
struct MergeAcc {
  float m[8], den[8], acc[8];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      m[h] = -INFINITY;
      den[h] = 0.f;
      acc[h] = 0.f;
    }
  }
  __device__ __forceinline__ void add(const float4& la, const float4& lb, const float4& oa, const float4& ob) {
    const float l8[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
    const float o8[8] = {oa.x, oa.y, oa.z, oa.w, ob.x, ob.y, ob.z, ob.w};
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const float mn = fmaxf(m[h], l8[h]);
      const float sh = mn == -INFINITY ? 0.f : mn;  // all -inf so far (pieces with no valid token)
      const float sc = ex2(m[h] - sh);  // 0 while nothing has been added (m = -inf)
      const float wt = ex2(l8[h] - sh);
      den[h] = den[h] * sc + wt;
      acc[h] = acc[h] * sc + wt * o8[h];
      m[h] = mn;
    }
  }
};

template <int NG>
__global__ void __launch_bounds__(kMergeThreads) gqa_merge_kernel(const MergeParams p) {
  constexpr int kHG = kKvHeads / NG;
  constexpr int kH8 = NG * kGroup;  // query heads per head group
  // row-group states of the block path: [group * cols + col] -> (m[4], den[4], acc[4]); 6 KB,
  // small enough for one merge CTA to sit beside three decode CTAs on an SM
  __shared__ float xw[128][12];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (p.skip_if_set != nullptr && *p.skip_if_set != 0) return;
  const int B = p.batch;
  const int j = blockIdx.x;  // boundary between decode CTAs j and j + 1
  const bool boundary = j + 1 < p.plan.tier1_ctas + p.plan.tier2_ctas;
  // Loads that do not depend on the decode grid go out before the wait, so
  // their round trip overlaps it; nothing waits on them until after it.
  // sparse rows (sparse_topk > 0) are never empty and have no kv_indptr
  const bool sparse = p.sparse_topk > 0;
  const int T = sparse ? p.sparse_total : __ldg(p.kv_indptr + B);
  const bool check_empty = !sparse && j < B;
  const int e_lo = check_empty ? __ldg(p.kv_indptr + j) : 0;
  const int e_hi = check_empty ? __ldg(p.kv_indptr + j + 1) : 0;

  // Everything below reads what the decode grid wrote.
  pdl_wait();
  // The sequence holding decode CTA j's last unit, as that CTA recorded it
  // (read before checking that CTA j had work, to save a round trip).
  const int4 rec = boundary ? __ldcg(p.split_rec + j) : make_int4(0, 0, 0, 0);

  // Empty sequences: O = 0, LSE = -inf (no decode CTA touches them).
  for (int b = j; !sparse && b < B; b += gridDim.x) {
    if (b == j ? e_lo == e_hi : __ldg(p.kv_indptr + b) == __ldg(p.kv_indptr + b + 1)) {
      uint4* ob = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(b) * kQoHeads * kHeadDim);
      for (int i = tid; i < kQoHeads * kHeadDim * 2 / 16; i += kMergeThreads) ob[i] = make_uint4(0, 0, 0, 0);
      if (tid < kQoHeads && p.lse != nullptr) p.lse[static_cast<int64_t>(b) * kQoHeads + tid] = -INFINITY;
    }
  }

  const Plan pl = make_plan(static_cast<int64_t>(T) * kHG, p.plan);
  if (!boundary || pl.begin(j + 1) >= pl.W) return;  // CTA j + 1 has no work: neither has this boundary
  if (static_cast<unsigned>(rec.x) != static_cast<unsigned>(p.epoch)) return;  // CTA j stopped on an error
  const int b = rec.y;
  const int S = rec.w >> 3;
  const int hg = (rec.w >> 1) & 3;
  SeqSplit sp;
  sp.first_cta = rec.z;
  sp.first_slot = rec.w & 1;
  sp.last_cta = sp.first_cta + S - 1;
  if (b < 0 || b >= B || hg >= kHG || S < 1 || sp.first_cta > j) return;
  if (sp.last_cta <= j) return;         // the sequence ends at this boundary: nothing is split here
  if (S <= p.fuse_max_splits) return;  // the decode kernel merged it
  const int rank = j - static_cast<int>(sp.first_cta);  // which of this sequence's S - 1 boundaries
  const int nranks = S - 1;
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.out) + (static_cast<int64_t>(b) * kQoHeads + hg * kH8) * kHeadDim;
  float* lo = p.lse != nullptr ? p.lse + static_cast<int64_t>(b) * kQoHeads + hg * kH8 : nullptr;

  if (S <= kMergeSmallSplits) {
    // (reached when the decode kernel's own merge is turned down by tuning)
    // warp item = (KV head g, 32-dim chunk): lane = one dim of all 8 heads, all splits
    for (int it = warp * nranks + rank; it < NG * 4; it += kMergeWarps * nranks) {
      const int g = it >> 2;
      const int d = (it & 3) * 32 + lane;
      MergeAcc ma;
      ma.init();
#pragma unroll 4
      for (int s = 0; s < S; ++s) {
        const float4* lr = reinterpret_cast<const float4*>(partial_lse_row<NG>(p, sp, s, g));
        const float4* orow = reinterpret_cast<const float4*>(partial_o_row<NG>(p, sp, s, g, d));
        ma.add(lr[0], lr[1], __ldcg(orow), __ldcg(orow + 1));
      }
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float o = ma.den[h] > 0.f ? ma.acc[h] / ma.den[h] : 0.f;  // no valid token anywhere: O = 0
        ob[(g * kGroup + h) * kHeadDim + d] = __float2bfloat16_rn(o);
      }
      if ((it & 3) == 0 && lane == 0 && lo != nullptr) {
#pragma unroll
        for (int h = 0; h < 8; ++h) lo[g * kGroup + h] = ma.den[h] > 0.f ? ma.m[h] + log2f(ma.den[h]) : -INFINITY;
      }
    }
  } else {
    // Block item = (KV head g, dims [d0, d0 + dc)) over all S splits. Threads
    // form rows x cols: a column is one dim and 4 of the 8 heads (16 bytes of
    // a partial O row), a row walks every rows-th split. dc is the smallest
    // power of two whose items fit the sequence's S - 1 boundary CTAs, so a
    // CTA holds about one split's worth of partials (16 KB at NG = 4) and each
    // thread issues its loads in one batch of up to 8 splits.
    const int need = (NG * kHeadDim + nranks - 1) / nranks;
    int dc = 1;
    while (dc < need && dc < 32) dc <<= 1;
    const int cols = 2 * dc;
    const int rows = kMergeThreads / cols;
    const int col = tid % cols, row = tid / cols;
    const int span = cols < 32 ? 32 : cols;        // lanes (or threads) that one row group spans
    const int group = tid / span;                  // row group left after the in-warp combine
    const int ngroups = kMergeThreads / span;
    const bool leader = (tid % span) < cols;
    const int hq = col & 1;                        // heads 4 hq .. 4 hq + 3
    // a row's LSE rows are loaded by its columns 0 and 1 and shuffled to the rest
    const int wcols = cols < 32 ? cols : 32;       // columns of a row within one warp
    const bool lse_loader = (lane & (wcols - 1)) < 2;
    const int lse_src = (lane & ~(wcols - 1)) | hq;
    const int items = NG * (kHeadDim / dc);
    for (int it = rank; it < items; it += nranks) {
      const int g = it / (kHeadDim / dc);
      const int d = (it % (kHeadDim / dc)) * dc + (col >> 1);
      float m[4], den[4], acc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        den[i] = 0.f;
        acc[i] = 0.f;
      }
      for (int s0 = 0; s0 < S; s0 += 8 * rows) {  // same trip count in every lane (the shuffles need it)
        float4 lv[8], ov[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // the whole batch is in flight before the first fold
          const int s = s0 + k * rows + row;
          lv[k] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
          ov[k] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (s < S) {
            if (lse_loader) lv[k] = __ldcg(reinterpret_cast<const float4*>(partial_lse_row<NG>(p, sp, s, g)) + hq);
            ov[k] = __ldcg(reinterpret_cast<const float4*>(partial_o_row<NG>(p, sp, s, g, d)) + hq);
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          lv[k].x = __shfl_sync(0xffffffffu, lv[k].x, lse_src);
          lv[k].y = __shfl_sync(0xffffffffu, lv[k].y, lse_src);
          lv[k].z = __shfl_sync(0xffffffffu, lv[k].z, lse_src);
          lv[k].w = __shfl_sync(0xffffffffu, lv[k].w, lse_src);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float l4[4] = {lv[k].x, lv[k].y, lv[k].z, lv[k].w};
          const float o4[4] = {ov[k].x, ov[k].y, ov[k].z, ov[k].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float mn = fmaxf(m[i], l4[i]);
            if (mn == -INFINITY) continue;  // nothing added yet and a padding split
            const float sc = ex2(m[i] - mn), wt = ex2(l4[i] - mn);
            den[i] = den[i] * sc + wt;
            acc[i] = acc[i] * sc + wt * o4[i];
            m[i] = mn;
          }
        }
      }
      // fold the rows that share a warp (lanes col, col + cols, ...)
      for (int o = cols; o < 32; o <<= 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float m2 = __shfl_xor_sync(0xffffffffu, m[i], o);
          const float d2 = __shfl_xor_sync(0xffffffffu, den[i], o);
          const float a2 = __shfl_xor_sync(0xffffffffu, acc[i], o);
          const float mn = fmaxf(m[i], m2);
          if (mn == -INFINITY) continue;
          const float s1 = ex2(m[i] - mn), s2 = ex2(m2 - mn);
          den[i] = den[i] * s1 + d2 * s2;
          acc[i] = acc[i] * s1 + a2 * s2;
          m[i] = mn;
        }
      }
      // then the row groups, through shared memory
      __syncthreads();  // the previous item's readers are done with xw
      if (leader) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          xw[group * cols + col][i] = m[i];
          xw[group * cols + col][4 + i] = den[i];
          xw[group * cols + col][8 + i] = acc[i];
        }
      }
      __syncthreads();
      if (tid < cols) {
        for (int gi = 1; gi < ngroups; ++gi) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float m2 = xw[gi * cols + col][i];
            const float mn = fmaxf(m[i], m2);
            if (mn == -INFINITY) continue;
            const float s1 = ex2(m[i] - mn), s2 = ex2(m2 - mn);
            den[i] = den[i] * s1 + xw[gi * cols + col][4 + i] * s2;
            acc[i] = acc[i] * s1 + xw[gi * cols + col][8 + i] * s2;
            m[i] = mn;
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int h = g * kGroup + hq * 4 + i;
          ob[h * kHeadDim + d] = __float2bfloat16_rn(den[i] > 0.f ? acc[i] / den[i] : 0.f);
          if (d == 0 && lo != nullptr) lo[h] = den[i] > 0.f ? m[i] + log2f(den[i]) : -INFINITY;
        }
      }
    }
  }
}

// ------------------------------------------------------------ validation
// Checked entry point only: verifies kv_indptr (starts at 0, non-decreasing)
// and that every kv_indices entry is a valid page, before any gather runs.
__global__ void gqa_validate_kernel(const int* __restrict__ indptr, const int* __restrict__ indices, int batch,
                                    int num_pages, int* __restrict__ err) {
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  const int stride = gridDim.x * blockDim.x;
  int bad = 0;
  if (tid == 0 && __ldg(indptr) != 0) bad |= kErrBadIndptr;
  for (int b = tid; b < batch; b += stride) {
    if (__ldg(indptr + b + 1) < __ldg(indptr + b)) bad |= kErrBadIndptr;
  }
  const int total = __ldg(indptr + batch);
  for (int i = tid; i < total; i += stride) {
    const int pg = __ldg(indices + i);
    if (pg < 0 || pg >= num_pages) bad |= kErrBadPage;
  }
  if (bad) atomicOr(err, bad);
}

// ------------------------------------------------------------------- launch
template <int NG>
static cudaError_t launch_merge_impl(const MergeParams& p, cudaStream_t stream) {
  const int ctas = p.plan.tier1_ctas + p.plan.tier2_ctas;
  const int boundaries = ctas > 1 ? ctas - 1 : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(boundaries * kMergeCtasPerBoundary);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = p.use_pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gqa_merge_kernel<NG>, p);
}

cudaError_t launch_merge(int heads_per_cta, const MergeParams& p, cudaStream_t stream) {
  if (heads_per_cta == 4) return launch_merge_impl<4>(p, stream);
  if (heads_per_cta == 2) return launch_merge_impl<2>(p, stream);
  if (heads_per_cta == 1) return launch_merge_impl<1>(p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_validate(const int* indptr, const int* indices, int batch, int num_pages, int* err,
                            cudaStream_t stream) {
  gqa_validate_kernel<<<64, 256, 0, stream>>>(indptr, indices, batch, num_pages, err);
  return cudaGetLastError();
}

cudaError_t read_and_clear_device_error(int* out) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
  *out = v;
  return e;
}

cudaError_t device_error_word(int** ptr) {
  static std::atomic<int*> cached[kMaxDevices];  // one address per device; racing threads store the same one
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int* word = cached[dev].load(std::memory_order_acquire);
  if (word == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return e;
    word = static_cast<int*>(p);
    cached[dev].store(word, std::memory_order_release);
  }
  *ptr = word;
  return cudaSuccess;
}

}  // namespace gqa
