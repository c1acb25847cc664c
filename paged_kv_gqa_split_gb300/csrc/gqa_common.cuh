// Device code shared by the decode kernels: tile flags, the kv_indptr search,
// and the per-warp attention math on one 16-token sub-tile of one KV head:
//   S^T (16 tokens x 8 heads) = K (16 x 128) . Q^T (128 x 8)      8 x mma.sync m16n8k16
//   online base-2 softmax over the 16 tokens (running max m, sum l)
//   O^T (128 dims x 8 heads) += V^T (128 x 16) . P^T (16 x 8)     8 x mma.sync m16n8k16
// The 8 query heads of a KV head are the N = 8 columns of the mma, so no MAC
// is spent on padding; P^T is formed in registers with movmatrix.
//
// Fragment ownership (lane = 4 r + c): S^T rows r and r + 8 (tokens), columns
// 2c and 2c + 1 (heads); O^T rows 16 mt + r and 16 mt + r + 8 (dims), the same
// two heads. Each lane keeps m and l for its two heads over its own tokens;
// the max is made warp-uniform per head every sub-tile, l is reduced at the end.
#pragma once

#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "gqa_plan.h"
#include "gqa_ptx.cuh"

namespace gqa {

enum : int {
  F_QLOAD = 1,   // first tile of a piece: (re)load Q, reset the softmax state
  F_END = 2,     // last tile of a piece: write the result
  F_FINAL = 4,   // the piece is the whole sequence: write bf16 O and LSE directly
  F_SLOT1 = 8,   // partial goes to slot 1 of the CTA (else slot 0)
  F_DONE = 16,   // end of the CTA's work
  F_QREG = 32,   // Q fragments were prefetched into registers when the tile was issued
};

// Largest b in [0, batch) with indptr[b] <= t (needs indptr[0] <= t < indptr[batch]).
// Warp-cooperative 32-ary search: each round samples 32 evenly spaced entries.
// Returns -1 if indptr[0] > t (malformed table).
__device__ __forceinline__ int warp_find_seq(const int* __restrict__ indptr, int batch, int t, int lane) {
  int lo = 0, hi = batch;
  while (hi - lo > 32) {
    const int step = (hi - lo + 31) / 32;
    const int pos = lo + lane * step;
    const int val = pos < hi ? __ldg(indptr + pos) : INT32_MAX;
    const unsigned m = __ballot_sync(0xffffffffu, val <= t);
    if (m == 0) return -1;
    const int k = 31 - __clz(m);
    const int nlo = lo + k * step;
    hi = min(nlo + step, hi);
    lo = nlo;
  }
  const int pos = lo + lane;
  const int val = pos < hi ? __ldg(indptr + pos) : INT32_MAX;
  const unsigned m = __ballot_sync(0xffffffffu, val <= t);
  if (m == 0) return -1;
  return lo + 31 - __clz(m);
}

// kv_indptr[base + lane], or INT32_MAX past the end.
__device__ __forceinline__ int load_indptr_window(const int* __restrict__ indptr, int batch, int base, int lane) {
  const int pos = base + lane;
  return pos <= batch ? __ldg(indptr + pos) : INT32_MAX;
}

// Online-softmax state of one warp (one KV head, 8 query heads) over a piece.
struct HeadState {
  uint32_t qf[16];   // Q^T B-fragments: dims 16 kk + {0..7} (qf[2kk]) and {8..15} (qf[2kk+1])
  float acc[8][4];   // O^T accumulators
  float m0, m1;      // running max (base-2 logits) of heads 2c, 2c + 1
  float l0, l1;      // running sum of 2^(s - m) over this lane's tokens

  __device__ __forceinline__ void reset() {
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
  }
};

// Q^T B-fragments straight from global memory: query rows q[b, h0 .. h0+7, :].
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[16], const __nv_bfloat16* q, int64_t b, int h0, int lane) {
  const int r = lane >> 2, c = lane & 3;
  const uint32_t* row = reinterpret_cast<const uint32_t*>(q + (b * kQoHeads + h0 + r) * kHeadDim) + c;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    qf[2 * kk] = __ldg(row + 8 * kk);
    qf[2 * kk + 1] = __ldg(row + 8 * kk + 4);
  }
}

// One 16-token sub-tile. k_addr / v_addr: this lane's ldmatrix row address for
// dims 0..15 of the sub-tile's K and V rows (row pitch `pitch`, dims contiguous).
// Tokens at index >= valid are masked out (their rows must hold finite values).
__device__ __forceinline__ void attend_subtile(HeadState& st, uint32_t k_addr, uint32_t v_addr, int valid,
                                               float scale_log2, int lane) {
  const int r = lane >> 2;
  float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(k_addr + kk * 32, a0, a1, a2, a3);
    mma_bf16_16816(s, a0, a1, a2, a3, st.qf[2 * kk], st.qf[2 * kk + 1]);
  }
  s[0] = r < valid ? s[0] * scale_log2 : -INFINITY;
  s[1] = r < valid ? s[1] * scale_log2 : -INFINITY;
  s[2] = r + 8 < valid ? s[2] * scale_log2 : -INFINITY;
  s[3] = r + 8 < valid ? s[3] * scale_log2 : -INFINITY;
  float mx0 = fmaxf(s[0], s[2]);
  float mx1 = fmaxf(s[1], s[3]);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  const float mn0 = fmaxf(st.m0, mx0);
  const float mn1 = fmaxf(st.m1, mx1);
  const float a0 = ex2(st.m0 - mn0);
  const float a1 = ex2(st.m1 - mn1);
  st.m0 = mn0;
  st.m1 = mn1;
  const float p0 = ex2(s[0] - mn0), p1 = ex2(s[1] - mn1);  // token r
  const float p2 = ex2(s[2] - mn0), p3 = ex2(s[3] - mn1);  // token r + 8
  // the running sum keeps fp32 probabilities; only the P.V operand is bf16
  st.l0 = st.l0 * a0 + (p0 + p2);
  st.l1 = st.l1 * a1 + (p1 + p3);
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    st.acc[mt][0] *= a0;
    st.acc[mt][1] *= a1;
    st.acc[mt][2] *= a0;
    st.acc[mt][3] *= a1;
  }
  // P^T as the B operand (16 tokens x 8 heads): transpose the two 8x8 blocks
  const uint32_t b0 = movmatrix_trans(pack_bf16(p0, p1));
  const uint32_t b1 = movmatrix_trans(pack_bf16(p2, p3));
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t v0, v1, v2, v3;
    ldsm_x4_trans(v_addr + mt * 32, v0, v1, v2, v3);
    mma_bf16_16816(st.acc[mt], v0, v1, v2, v3, b0, b1);
  }
}

// Normalise and write a finished piece: bf16 O rows q-heads h0 .. h0+7 of
// sequence b plus their LSE (final), or an fp32 partial (O_i, LSE_i) into
// slot `sid` (layout [sid][NG][128 dims][8 heads], LSE [sid][NG][8]).
template <int NG>
__device__ __forceinline__ void finish_piece(const HeadState& st, bool final_piece, int64_t b, int h0, int64_t sid,
                                             int w, __nv_bfloat16* out, float* lse, float* part_o, float* part_lse,
                                             int lane) {
  const int r = lane >> 2, c = lane & 3;
  float lt0 = st.l0, lt1 = st.l1;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    lt0 += __shfl_xor_sync(0xffffffffu, lt0, o);
    lt1 += __shfl_xor_sync(0xffffffffu, lt1, o);
  }
  const float i0 = 1.f / lt0;
  const float i1 = 1.f / lt1;
  const float lse0 = st.m0 + log2f(lt0);
  const float lse1 = st.m1 + log2f(lt1);
  if (final_piece) {
    __nv_bfloat16* ob = out + (b * kQoHeads + h0) * kHeadDim;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      // rows = dims, cols = heads  ->  transpose to rows = heads, cols = dims
      const uint32_t x = movmatrix_trans(pack_bf16(st.acc[mt][0] * i0, st.acc[mt][1] * i1));
      const uint32_t y = movmatrix_trans(pack_bf16(st.acc[mt][2] * i0, st.acc[mt][3] * i1));
      *reinterpret_cast<uint32_t*>(ob + r * kHeadDim + mt * 16 + 2 * c) = x;
      *reinterpret_cast<uint32_t*>(ob + r * kHeadDim + mt * 16 + 8 + 2 * c) = y;
    }
    if (r == 0) *reinterpret_cast<float2*>(lse + b * kQoHeads + h0 + 2 * c) = make_float2(lse0, lse1);
  } else {
    float* po = part_o + (sid * NG + w) * (kHeadDim * kGroup);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      *reinterpret_cast<float2*>(po + (mt * 16 + r) * kGroup + 2 * c) =
          make_float2(st.acc[mt][0] * i0, st.acc[mt][1] * i1);
      *reinterpret_cast<float2*>(po + (mt * 16 + 8 + r) * kGroup + 2 * c) =
          make_float2(st.acc[mt][2] * i0, st.acc[mt][3] * i1);
    }
    if (r == 0) *reinterpret_cast<float2*>(part_lse + (sid * NG + w) * kGroup + 2 * c) = make_float2(lse0, lse1);
  }
}

}  // namespace gqa
