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
// merges itself (fuse_max_splits).
// They hold no shared memory and few registers, so they sit beside the decode
// CTAs (programmatic dependent launch) and run their prologue - locating the
// sequence cut at their boundary - while the decode grid is still running.
// After the decode grid completes, one round of loads remains: each split's
// partial LSE and O are folded in with a running maximum, so the weights need
// no second pass.
constexpr int kMergeThreads = 128;
constexpr int kMergeWarps = kMergeThreads / 32;
// Split counts up to this use the CTA-per-item path (warps share the splits);
// above it, lanes share the splits of one (head, dim) item.
constexpr int kMergeMediumSplits = 64;
// Split counts up to this: one warp per (head, 32-dim chunk) item, all splits.
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
      const float sc = ex2(m[h] - mn);  // 0 while nothing has been added (m = -inf)
      const float wt = ex2(l8[h] - mn);
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
  // cross-warp combine buffer of the medium-split path: one lane's state at a time
  __shared__ float xw[32][3 * kGroup];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (p.skip_if_set != nullptr && *p.skip_if_set != 0) return;
  const int B = p.batch;

  // Empty sequences: O = 0, LSE = -inf (no decode CTA touches them).
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    if (__ldg(p.kv_indptr + b) == __ldg(p.kv_indptr + b + 1)) {
      uint4* ob = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(b) * kQoHeads * kHeadDim);
      for (int i = tid; i < kQoHeads * kHeadDim * 2 / 16; i += kMergeThreads) ob[i] = make_uint4(0, 0, 0, 0);
      if (tid < kQoHeads) p.lse[static_cast<int64_t>(b) * kQoHeads + tid] = -INFINITY;
    }
  }

  const int T = __ldg(p.kv_indptr + B);
  const int64_t W = static_cast<int64_t>(T) * kHG;
  const int64_t q = units_per_cta(W, p.num_decode_ctas, p.min_units);
  const int j = blockIdx.x;  // boundary between decode CTAs j and j + 1
  const int64_t u = static_cast<int64_t>(j + 1) * q;
  if (u >= W) return;
  const int hg = static_cast<int>(u / T);
  const int t = static_cast<int>(u - static_cast<int64_t>(hg) * T);
  const int b = warp_find_seq(p.kv_indptr, B, t, lane);  // every warp searches (L1-resident)
  if (b < 0) return;
  const int seq_lo = __ldg(p.kv_indptr + b);
  if (t == seq_lo) return;  // the boundary falls between two sequences: nothing is split here
  const int seq_hi = __ldg(p.kv_indptr + b + 1);
  const int64_t base_u = static_cast<int64_t>(hg) * T;
  const SeqSplit sp = seq_split(base_u + seq_lo, base_u + seq_hi, q);
  const int S = static_cast<int>(sp.last_cta - sp.first_cta + 1);
  if (S <= p.fuse_max_splits) return;  // the decode kernel merged it
  const int rank = j - static_cast<int>(sp.first_cta);  // which of this sequence's S - 1 boundaries
  const int nranks = S - 1;
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.out) + (static_cast<int64_t>(b) * kQoHeads + hg * kH8) * kHeadDim;
  float* lo = p.lse + static_cast<int64_t>(b) * kQoHeads + hg * kH8;

  // Everything below reads the decode kernel's partials.
  pdl_wait();

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
      for (int h = 0; h < 8; ++h) ob[(g * kGroup + h) * kHeadDim + d] = __float2bfloat16_rn(ma.acc[h] / ma.den[h]);
      if ((it & 3) == 0 && lane == 0) {
#pragma unroll
        for (int h = 0; h < 8; ++h) lo[g * kGroup + h] = ma.m[h] + log2f(ma.den[h]);
      }
    }
  } else if (S <= kMergeMediumSplits) {
    // CTA item = (KV head g, 32-dim chunk): lane = one dim of all 8 heads; the
    // four warps take every fourth split, then fold their states together
    for (int it = rank; it < NG * 4; it += nranks) {
      const int g = it >> 2;
      const int d = (it & 3) * 32 + lane;
      MergeAcc ma;
      ma.init();
#pragma unroll 4
      for (int s = warp; s < S; s += kMergeWarps) {
        const float4* lr = reinterpret_cast<const float4*>(partial_lse_row<NG>(p, sp, s, g));
        const float4* orow = reinterpret_cast<const float4*>(partial_o_row<NG>(p, sp, s, g, d));
        ma.add(lr[0], lr[1], __ldcg(orow), __ldcg(orow + 1));
      }
      for (int src = 1; src < kMergeWarps; ++src) {
        __syncthreads();
        if (warp == src) {
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            xw[lane][h] = ma.m[h];
            xw[lane][8 + h] = ma.den[h];
            xw[lane][16 + h] = ma.acc[h];
          }
        }
        __syncthreads();
        if (warp == 0) {
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            const float m2 = xw[lane][h];
            const float mn = fmaxf(ma.m[h], m2);
            const float s1 = ex2(ma.m[h] - mn), s2 = ex2(m2 - mn);  // a warp that saw no split has m = -inf
            ma.den[h] = ma.den[h] * s1 + xw[lane][8 + h] * s2;
            ma.acc[h] = ma.acc[h] * s1 + xw[lane][16 + h] * s2;
            ma.m[h] = mn;
          }
        }
      }
      if (warp == 0) {
#pragma unroll
        for (int h = 0; h < 8; ++h) ob[(g * kGroup + h) * kHeadDim + d] = __float2bfloat16_rn(ma.acc[h] / ma.den[h]);
        if ((it & 3) == 0 && lane == 0) {
#pragma unroll
          for (int h = 0; h < 8; ++h) lo[g * kGroup + h] = ma.m[h] + log2f(ma.den[h]);
        }
      }
    }
  } else {
    // warp item = (KV head g, dim d): lanes stride over the splits, then one warp
    // reduction; items are dealt boundary-fastest over all of this sequence's CTAs
    const int first_item = warp * nranks + rank;
    const int item_step = kMergeWarps * nranks;
    for (int it = first_item; it < NG * kHeadDim; it += item_step) {
      const int g = it / kHeadDim;
      const int d = it - g * kHeadDim;
      MergeAcc ma;
      ma.init();
#pragma unroll 4
      for (int s = lane; s < S; s += 32) {
        const float4* lr = reinterpret_cast<const float4*>(partial_lse_row<NG>(p, sp, s, g));
        const float4* orow = reinterpret_cast<const float4*>(partial_o_row<NG>(p, sp, s, g, d));
        ma.add(lr[0], lr[1], __ldcg(orow), __ldcg(orow + 1));
      }
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        float mx = ma.m[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float sc = ex2(ma.m[h] - mx);  // lanes that saw no split contribute 0
        float dn = ma.den[h] * sc, ac = ma.acc[h] * sc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          dn += __shfl_xor_sync(0xffffffffu, dn, o);
          ac += __shfl_xor_sync(0xffffffffu, ac, o);
        }
        if (lane == h) {
          ob[(g * kGroup + h) * kHeadDim + d] = __float2bfloat16_rn(ac / dn);
          if (d == 0) lo[g * kGroup + h] = mx + log2f(dn);
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
  const int boundaries = p.num_decode_ctas > 1 ? p.num_decode_ctas - 1 : 1;
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
  static int* cached[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (cached[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return e;
    cached[dev] = static_cast<int*>(p);
  }
  *ptr = cached[dev];
  return cudaSuccess;
}

}  // namespace gqa
