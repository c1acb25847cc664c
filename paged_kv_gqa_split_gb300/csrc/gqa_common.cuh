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

#include "gqa_kernels.h"
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

// First round of warp_find_window for the whole table, which needs no token
// position: the 32 entries it samples (batch > 32) or the window at 0 (batch
// <= 32). Loading it together with kv_indptr[batch] puts both in one round trip.
__device__ __forceinline__ int first_search_round(const int* __restrict__ indptr, int batch, int lane) {
  if (batch > 32) {
    const int step = (batch + 31) / 32;
    const int pos = lane * step;
    return pos < batch ? __ldg(indptr + pos) : INT32_MAX;
  }
  return lane <= batch ? __ldg(indptr + lane) : INT32_MAX;
}

// A 32-entry kv_indptr window win = kv_indptr[base + lane] (INT32_MAX past the
// end) with kv_indptr[base] <= t, found with the 32-ary search of
// warp_find_seq; its last round is the window itself, so no separate window
// load follows. The sequence holding t is at window index 31 - clz(ballot(win
// <= t)), unless every entry is <= t (then the window must move on). `pre`,
// when has_pre, is first_search_round's value for this table. Returns base, or
// -1 if kv_indptr[0] > t (a malformed table).
__device__ __forceinline__ int warp_find_window(const int* __restrict__ indptr, int batch, int t, int lane,
                                                bool has_pre, int pre, int& win) {
  int lo = 0, hi = batch;
  bool use_pre = has_pre;
  while (hi - lo > 32) {
    const int step = (hi - lo + 31) / 32;
    const int pos = lo + lane * step;
    const int val = use_pre ? pre : (pos < hi ? __ldg(indptr + pos) : INT32_MAX);
    use_pre = false;
    const unsigned m = __ballot_sync(0xffffffffu, val <= t);
    if (m == 0) return -1;
    const int k = 31 - __clz(m);
    const int nlo = lo + k * step;
    hi = min(nlo + step, hi);
    lo = nlo;
  }
  win = use_pre ? pre : load_indptr_window(indptr, batch, lo, lane);
  if (__ballot_sync(0xffffffffu, win <= t) == 0) return -1;
  return lo;
}

// Online-softmax state of one warp (one KV head, 8 query heads) over a piece.
struct HeadState {
  uint32_t qf[16];   // Q^T B-fragments: dims 16 kk + {0..7} (qf[2kk]) and {8..15} (qf[2kk+1])
  float acc[8][4];   // O^T accumulators
  float m0, m1;      // running max (base-2 logits) of heads 2c, 2c + 1
  float l0, l1;      // running sum of 2^(s - m) over this lane's tokens
  float qsc;         // FP8 path: 1 / the power of two Q was scaled by for f16
  float cv;          // FP8 path: running power of two >= every V scale of the piece (0: none yet)

  __device__ __forceinline__ void reset() {
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
    cv = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
  }
};

// Q^T B-fragments straight from global memory: query rows q[b, h0 .. h0+7, :].
// PERM (the FP8-cache path): k-block t = 4 kb + j takes, in lane (r, c), the
// dims 64 kb + 16 c + 4 j .. + 3 instead of 16 t + 2 c, +1 and 16 t + 8 + 2 c,
// +1: the same permutation of the contraction dims as the e4m3 K fragments,
// which a lane reads as 16 consecutive bytes of a K row (attend_subtile_f8).
template <bool PERM = false>
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[16], const __nv_bfloat16* q, int64_t b, int h0, int lane) {
  const int r = lane >> 2, c = lane & 3;
  if constexpr (PERM) {
    const __nv_bfloat16* row = q + (b * kQoHeads + h0 + r) * kHeadDim;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(row + 64 * (t >> 2) + 16 * c + 4 * (t & 3)));
      qf[2 * t] = v.x;
      qf[2 * t + 1] = v.y;
    }
  } else {
    const uint32_t* row = reinterpret_cast<const uint32_t*>(q + (b * kQoHeads + h0 + r) * kHeadDim) + c;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qf[2 * kk] = __ldg(row + 8 * kk);
      qf[2 * kk + 1] = __ldg(row + 8 * kk + 4);
    }
  }
}

// One 16-token sub-tile. k_addr / v_addr: this lane's ldmatrix row address for
// dims 0..15 of the sub-tile's K and V rows (row pitch `pitch`, dims contiguous).
// Tokens whose bit in `valid` is clear are masked out (their rows must hold
// finite values); a sub-tile may have none valid.
__device__ __forceinline__ void attend_subtile(HeadState& st, uint32_t k_addr, uint32_t v_addr, unsigned valid,
                                               float scale_log2, int lane) {
  const int r = lane >> 2;
  float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(k_addr + kk * 32, a0, a1, a2, a3);
    mma_bf16_16816(s, a0, a1, a2, a3, st.qf[2 * kk], st.qf[2 * kk + 1]);
  }
  const bool v_lo = (valid >> r) & 1u, v_hi = (valid >> (r + 8)) & 1u;
  s[0] = v_lo ? s[0] * scale_log2 : -INFINITY;
  s[1] = v_lo ? s[1] * scale_log2 : -INFINITY;
  s[2] = v_hi ? s[2] * scale_log2 : -INFINITY;
  s[3] = v_hi ? s[3] * scale_log2 : -INFINITY;
  float mx0 = fmaxf(s[0], s[2]);
  float mx1 = fmaxf(s[1], s[3]);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  const float mn0 = fmaxf(st.m0, mx0);
  const float mn1 = fmaxf(st.m1, mx1);
  // while no valid token has been seen the max is -inf: shift by 0 instead,
  // so that the factors are 2^-inf = 0 rather than 2^(-inf - -inf) = NaN
  const float sh0 = mn0 == -INFINITY ? 0.f : mn0;
  const float sh1 = mn1 == -INFINITY ? 0.f : mn1;
  const float a0 = ex2(st.m0 - sh0);
  const float a1 = ex2(st.m1 - sh1);
  st.m0 = mn0;
  st.m1 = mn1;
  const float p0 = ex2(s[0] - sh0), p1 = ex2(s[1] - sh1);  // token r
  const float p2 = ex2(s[2] - sh0), p3 = ex2(s[3] - sh1);  // token r + 8
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

// 1 / x for x = 2^k with a normal reciprocal (exact: the exponent is negated).
__device__ __forceinline__ float pow2_recip(float x) { return __uint_as_float((254u << 23) - __float_as_uint(x)); }

// FP8-cache form of attend_subtile, straight from the staged e4m3 rows (no
// conversion pass through shared memory; e4m3 -> f16 is exact):
// - K (rows = tokens at a 192-byte pitch): lane (r, c) reads 16 bytes of rows
//   r and r + 8 per 64-dim block with one 128-bit load each and converts them
//   into the A fragments of 4 k-blocks; the contraction dims are thereby
//   permuted within each 64-dim block, and Q's fragments follow the same
//   permutation (load_q_frags<true>).
// - V (rows = tokens at a 144-byte pitch): ldmatrix.trans gives each lane the
//   bytes of tokens 2c, 2c + 1 for dims 2g, 2g + 1; a byte permute pairs the
//   tokens of one dim before the conversion, so A-fragment row g of m-tile mt
//   holds dim 16 mt + 2 g and row g + 8 holds dim 16 mt + 2 g + 1
//   (finish_piece<.., true> writes O accordingly).
// sk_lo / sk_hi and sv_lo / sv_hi are the scales of this lane's tokens r and
// r + 8 for this KV head. A score takes its token's K scale (and Q's
// power-of-two f16 scale, through st.qsc). A probability enters P.V times its
// token's V scale over st.cv, a running power of two no smaller than any V
// scale seen in the piece, so the f16 P operand stays in [0, 1]; acc then
// holds O * l / cv, and l sums the plain probabilities.
__device__ __forceinline__ void attend_subtile_f8(HeadState& st, uint32_t k_addr, uint32_t v_addr, unsigned valid,
                                                  float scale_log2, float sk_lo, float sk_hi, float sv_lo,
                                                  float sv_hi, int lane, int k_pitch) {
  const int r = lane >> 2;
  float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kb = 0; kb < 2; ++kb) {
    uint32_t x[4], y[4];
    ld_shared_u4(k_addr + kb * 64, x[0], x[1], x[2], x[3]);                // row r
    ld_shared_u4(k_addr + 8 * k_pitch + kb * 64, y[0], y[1], y[2], y[3]);  // row r + 8
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = 4 * kb + j;
      mma_f16_16816(s, cvt_e4m3x2_f16x2(x[j]), cvt_e4m3x2_f16x2(y[j]), cvt_e4m3x2_f16x2(x[j] >> 16),
                    cvt_e4m3x2_f16x2(y[j] >> 16), st.qf[2 * t], st.qf[2 * t + 1]);
    }
  }
  const bool v_lo = (valid >> r) & 1u, v_hi = (valid >> (r + 8)) & 1u;
  const float c_lo = scale_log2 * st.qsc * sk_lo, c_hi = scale_log2 * st.qsc * sk_hi;
  s[0] = v_lo ? s[0] * c_lo : -INFINITY;
  s[1] = v_lo ? s[1] * c_lo : -INFINITY;
  s[2] = v_hi ? s[2] * c_hi : -INFINITY;
  s[3] = v_hi ? s[3] * c_hi : -INFINITY;
  float mx0 = fmaxf(s[0], s[2]);
  float mx1 = fmaxf(s[1], s[3]);
  float vm = fmaxf(v_lo ? fabsf(sv_lo) : 0.f, v_hi ? fabsf(sv_hi) : 0.f);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
  }
  const float mn0 = fmaxf(st.m0, mx0);
  const float mn1 = fmaxf(st.m1, mx1);
  const float sh0 = mn0 == -INFINITY ? 0.f : mn0;
  const float sh1 = mn1 == -INFINITY ? 0.f : mn1;
  const float a0 = ex2(st.m0 - sh0);
  const float a1 = ex2(st.m1 - sh1);
  st.m0 = mn0;
  st.m1 = mn1;
  const float cv_new = fmaxf(st.cv, vm > 0.f ? pow2_ceil(vm) : 0.f);
  const float iv = cv_new > 0.f ? pow2_recip(cv_new) : 0.f;
  const float cr = cv_new > 0.f ? st.cv * iv : 1.f;  // exact: powers of two (or st.cv = 0)
  st.cv = cv_new;
  const float p0 = ex2(s[0] - sh0), p1 = ex2(s[1] - sh1);  // token r
  const float p2 = ex2(s[2] - sh0), p3 = ex2(s[3] - sh1);  // token r + 8
  st.l0 = st.l0 * a0 + (p0 + p2);
  st.l1 = st.l1 * a1 + (p1 + p3);
  const float b_a0 = a0 * cr, b_a1 = a1 * cr;
  if (__any_sync(0xffffffffu, b_a0 != 1.f || b_a1 != 1.f)) {  // skipped while no max and no V bound moved
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      st.acc[mt][0] *= b_a0;
      st.acc[mt][1] *= b_a1;
      st.acc[mt][2] *= b_a0;
      st.acc[mt][3] *= b_a1;
    }
  }
  const float w_lo = sv_lo * iv, w_hi = sv_hi * iv;
  const uint32_t b0 = movmatrix_trans(pack_f16(p0 * w_lo, p1 * w_lo));
  const uint32_t b1 = movmatrix_trans(pack_f16(p2 * w_hi, p3 * w_hi));
#pragma unroll
  for (int mp = 0; mp < 4; ++mp) {  // m-tiles 2 mp and 2 mp + 1
    uint32_t t0, t1, t2, t3;        // tokens 0-7 / 8-15 of m-tile 2 mp, then of 2 mp + 1
    ldsm_x4_trans(v_addr + mp * 32, t0, t1, t2, t3);
    mma_f16_16816(st.acc[2 * mp], cvt_e4m3x2_f16x2(__byte_perm(t0, 0, 0x0020)),
                  cvt_e4m3x2_f16x2(__byte_perm(t0, 0, 0x0031)), cvt_e4m3x2_f16x2(__byte_perm(t1, 0, 0x0020)),
                  cvt_e4m3x2_f16x2(__byte_perm(t1, 0, 0x0031)), b0, b1);
    mma_f16_16816(st.acc[2 * mp + 1], cvt_e4m3x2_f16x2(__byte_perm(t2, 0, 0x0020)),
                  cvt_e4m3x2_f16x2(__byte_perm(t2, 0, 0x0031)), cvt_e4m3x2_f16x2(__byte_perm(t3, 0, 0x0020)),
                  cvt_e4m3x2_f16x2(__byte_perm(t3, 0, 0x0031)), b0, b1);
  }
}

// attend_subtile_f8 over a 32-token stage: two 16-token halves (rows 0-15 and
// 16-31 of the staged K and V) share one softmax step, so the max reduction,
// the V-scale bound and the rescale of acc happen once per 32 tokens, and the
// two halves' score contractions run as independent mma chains. sk[i] / sv[i]
// are the scales of this lane's tokens r + 8 i (i = 0..3) for this KV head;
// valid holds one bit per token. The fragment layouts are those of
// attend_subtile_f8, half by half.
__device__ __forceinline__ void attend_tile32_f8(HeadState& st, uint32_t k_addr, uint32_t v_addr, unsigned valid,
                                                 float scale_log2, const float (&sk)[4], const float (&sv)[4], int lane,
                                                 int k_pitch, int v_pitch) {
  const int r = lane >> 2;
  float s[2][4];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf)
#pragma unroll
    for (int i = 0; i < 4; ++i) s[hf][i] = 0.f;
#pragma unroll
  for (int kb = 0; kb < 2; ++kb) {
    uint32_t x[2][4], y[2][4];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const uint32_t a = k_addr + hf * 16 * k_pitch + kb * 64;
      ld_shared_u4(a, x[hf][0], x[hf][1], x[hf][2], x[hf][3]);                // row 16 hf + r
      ld_shared_u4(a + 8 * k_pitch, y[hf][0], y[hf][1], y[hf][2], y[hf][3]);  // row 16 hf + r + 8
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = 4 * kb + j;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
        mma_f16_16816(s[hf], cvt_e4m3x2_f16x2(x[hf][j]), cvt_e4m3x2_f16x2(y[hf][j]),
                      cvt_e4m3x2_f16x2(x[hf][j] >> 16), cvt_e4m3x2_f16x2(y[hf][j] >> 16), st.qf[2 * t],
                      st.qf[2 * t + 1]);
    }
  }
  float mx0 = -INFINITY, mx1 = -INFINITY, vm = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // token r + 8 i: half i / 2, accumulator pair 2 (i % 2)
    const bool v = (valid >> (r + 8 * i)) & 1u;
    const float c = scale_log2 * st.qsc * sk[i];
    float& e0 = s[i >> 1][2 * (i & 1)];
    float& e1 = s[i >> 1][2 * (i & 1) + 1];
    e0 = v ? e0 * c : -INFINITY;
    e1 = v ? e1 * c : -INFINITY;
    mx0 = fmaxf(mx0, e0);
    mx1 = fmaxf(mx1, e1);
    vm = fmaxf(vm, v ? fabsf(sv[i]) : 0.f);
  }
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
  }
  const float mn0 = fmaxf(st.m0, mx0);
  const float mn1 = fmaxf(st.m1, mx1);
  const float sh0 = mn0 == -INFINITY ? 0.f : mn0;
  const float sh1 = mn1 == -INFINITY ? 0.f : mn1;
  const float a0 = ex2(st.m0 - sh0);
  const float a1 = ex2(st.m1 - sh1);
  st.m0 = mn0;
  st.m1 = mn1;
  const float cv_new = fmaxf(st.cv, vm > 0.f ? pow2_ceil(vm) : 0.f);
  const float iv = cv_new > 0.f ? pow2_recip(cv_new) : 0.f;
  const float cr = cv_new > 0.f ? st.cv * iv : 1.f;  // exact: powers of two (or st.cv = 0)
  st.cv = cv_new;
  float pr[2][4];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    pr[hf][0] = ex2(s[hf][0] - sh0);
    pr[hf][1] = ex2(s[hf][1] - sh1);
    pr[hf][2] = ex2(s[hf][2] - sh0);
    pr[hf][3] = ex2(s[hf][3] - sh1);
  }
  st.l0 = st.l0 * a0 + ((pr[0][0] + pr[0][2]) + (pr[1][0] + pr[1][2]));
  st.l1 = st.l1 * a1 + ((pr[0][1] + pr[0][3]) + (pr[1][1] + pr[1][3]));
  const float b_a0 = a0 * cr, b_a1 = a1 * cr;
  if (__any_sync(0xffffffffu, b_a0 != 1.f || b_a1 != 1.f)) {  // skipped while no max and no V bound moved
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      st.acc[mt][0] *= b_a0;
      st.acc[mt][1] *= b_a1;
      st.acc[mt][2] *= b_a0;
      st.acc[mt][3] *= b_a1;
    }
  }
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const float w_lo = sv[2 * hf] * iv, w_hi = sv[2 * hf + 1] * iv;
    const uint32_t b0 = movmatrix_trans(pack_f16(pr[hf][0] * w_lo, pr[hf][1] * w_lo));
    const uint32_t b1 = movmatrix_trans(pack_f16(pr[hf][2] * w_hi, pr[hf][3] * w_hi));
    const uint32_t va = v_addr + hf * 16 * v_pitch;
#pragma unroll
    for (int mp = 0; mp < 4; ++mp) {  // m-tiles 2 mp and 2 mp + 1
      uint32_t t0, t1, t2, t3;
      ldsm_x4_trans(va + mp * 32, t0, t1, t2, t3);
      mma_f16_16816(st.acc[2 * mp], cvt_e4m3x2_f16x2(__byte_perm(t0, 0, 0x0020)),
                    cvt_e4m3x2_f16x2(__byte_perm(t0, 0, 0x0031)), cvt_e4m3x2_f16x2(__byte_perm(t1, 0, 0x0020)),
                    cvt_e4m3x2_f16x2(__byte_perm(t1, 0, 0x0031)), b0, b1);
      mma_f16_16816(st.acc[2 * mp + 1], cvt_e4m3x2_f16x2(__byte_perm(t2, 0, 0x0020)),
                    cvt_e4m3x2_f16x2(__byte_perm(t2, 0, 0x0031)), cvt_e4m3x2_f16x2(__byte_perm(t3, 0, 0x0020)),
                    cvt_e4m3x2_f16x2(__byte_perm(t3, 0, 0x0031)), b0, b1);
    }
  }
}

// ------------------------------------------------- CUDA-core sub-tile
// The same 16-token sub-tile with the two contractions on the CUDA cores
// (fp32 FMAs) instead of mma.sync, for comparing the two on this part. Lane
// (h = lane & 7, g = lane >> 3) holds query head h0 + h and dims 32 g .. 32 g
// + 31: its Q slice in fp32, its slice of O, and the running max and sum of
// head h (every lane of a head sees all 16 tokens, so m and l need no
// reduction). Scores: 32 FMAs per token on the lane's K slice, then two xor
// shuffles sum the four dim groups; P.V: 32 FMAs per token on its V slice,
// with P in fp32.
struct CcState {
  float q[32];
  float acc[32];
  float m, l;
  __device__ __forceinline__ void reset() {
    m = -INFINITY;
    l = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;
  }
};

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// Q slice of lane (h, g) for query heads h0 .. h0 + 7 of sequence b, as 16 bf16 pairs.
__device__ __forceinline__ void load_q_cc(uint32_t (&qf)[16], const __nv_bfloat16* q, int64_t b, int h0, int lane) {
  const uint4* row =
      reinterpret_cast<const uint4*>(q + (b * kQoHeads + h0 + (lane & 7)) * kHeadDim + 32 * (lane >> 3));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = __ldg(row + i);
    qf[4 * i] = v.x;
    qf[4 * i + 1] = v.y;
    qf[4 * i + 2] = v.z;
    qf[4 * i + 3] = v.w;
  }
}

__device__ __forceinline__ void q_to_cc(CcState& cs, const uint32_t (&qf)[16]) {
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    cs.q[2 * k] = bf16_lo(qf[k]);
    cs.q[2 * k + 1] = bf16_hi(qf[k]);
  }
}

// k_rows / v_rows: shared address of token 0's K / V head row (pitch `pitch`).
__device__ __forceinline__ void attend_subtile_cc(CcState& cs, uint32_t k_rows, uint32_t v_rows, int pitch,
                                                  unsigned valid, float scale_log2, int lane) {
  const int g = lane >> 3;
  float s[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    uint32_t x[16];
    const uint32_t a = k_rows + t * pitch + 64 * g;
#pragma unroll
    for (int i = 0; i < 4; ++i) ld_shared_u4(a + 16 * i, x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
    float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;  // four chains
#pragma unroll
    for (int k = 0; k < 16; k += 2) {
      d0 = fmaf(cs.q[2 * k], bf16_lo(x[k]), d0);
      d1 = fmaf(cs.q[2 * k + 1], bf16_hi(x[k]), d1);
      d2 = fmaf(cs.q[2 * k + 2], bf16_lo(x[k + 1]), d2);
      d3 = fmaf(cs.q[2 * k + 3], bf16_hi(x[k + 1]), d3);
    }
    s[t] = (d0 + d1) + (d2 + d3);
  }
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    s[t] += __shfl_xor_sync(0xffffffffu, s[t], 8);
    s[t] += __shfl_xor_sync(0xffffffffu, s[t], 16);
    s[t] = ((valid >> t) & 1u) ? s[t] * scale_log2 : -INFINITY;
  }
  float mx = s[0];
#pragma unroll
  for (int t = 1; t < 16; ++t) mx = fmaxf(mx, s[t]);
  const float mn = fmaxf(cs.m, mx);
  const float sh = mn == -INFINITY ? 0.f : mn;  // nothing valid yet: 2^-inf = 0, not NaN
  const float alpha = ex2(cs.m - sh);
  cs.m = mn;
  float psum = 0.f;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    s[t] = ex2(s[t] - sh);
    psum += s[t];
  }
  cs.l = cs.l * alpha + psum;
#pragma unroll
  for (int j = 0; j < 32; ++j) cs.acc[j] *= alpha;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    uint32_t x[16];
    const uint32_t a = v_rows + t * pitch + 64 * g;
#pragma unroll
    for (int i = 0; i < 4; ++i) ld_shared_u4(a + 16 * i, x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      cs.acc[2 * k] = fmaf(s[t], bf16_lo(x[k]), cs.acc[2 * k]);
      cs.acc[2 * k + 1] = fmaf(s[t], bf16_hi(x[k]), cs.acc[2 * k + 1]);
    }
  }
}

// FP8-cache path: turn bf16 Q fragments into f16 ones scaled by a power of two
// chosen so that the group's largest |q| lands in [2^13, 2^14) (no f16
// overflow; exact for every component down to 2^-27 of that maximum).
// Returns the inverse of the scale, folded into the score scale.
__device__ __forceinline__ float q_frags_to_f16(uint32_t (&qf)[16]) {
  float mx = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&qf[i]);
    mx = fmaxf(mx, fmaxf(fabsf(__low2float(v)), fabsf(__high2float(v))));
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  int e = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu);  // biased exponent of the maximum
  int se = mx > 0.f ? 127 + 13 - (e - 127) : 127;                   // 2^(13 - (e - 127)), or 1
  se = se < 1 ? 1 : (se > 253 ? 253 : se);  // keeps 1 / qs a normal float
  const float qs = __uint_as_float(static_cast<uint32_t>(se) << 23);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&qf[i]);
    qf[i] = pack_f16(__low2float(v) * qs, __high2float(v) * qs);
  }
  return __uint_as_float(static_cast<uint32_t>(254 - se) << 23);  // 1 / qs, exact
}

// Where a piece's sequence was cut: S pieces held by decode CTAs first_cta ..
// first_cta + S - 1; the first of them in slot first_slot, the others in slot 0.
struct SplitInfo {
  int S;
  int first_cta;
  int first_slot;
};

// Epoch-tagged counter word: (call epoch << 24) | count. A word tagged with
// another epoch (an earlier call's, or never-written memory) counts as zero, so
// these counters need no clearing between calls.
//
// Adds one and returns the count before the addition. The first warp of a call
// to find the word stale installs this call's tag with its own addition counted
// (compare-and-swap); additions that other warps made to the stale word before
// that are discarded and retried, so every count from 0 up is handed out exactly
// once. Returns -1 (and sets kErrTicket) if the word could not be claimed, which
// takes many thousands of competing writers.
__device__ __forceinline__ long long tagged_fetch_add(unsigned long long* word, unsigned long long epoch, int* err) {
  unsigned long long v = atomicAdd(word, 1ull);
  for (int it = 0; (v >> 24) != epoch; ++it) {
    if (it >= 64) {
      atomicOr(err, kErrTicket);
      return -1;
    }
    unsigned long long cur = v + 1;  // the word as this warp left it
    for (int k = 0; k < 4096 && (cur >> 24) != epoch; ++k) {
      const unsigned long long prev = atomicCAS(word, cur, (epoch << 24) | 1ull);
      if (prev == cur) return 0;  // installed: this addition took count 0
      cur = prev;
    }
    v = atomicAdd(word, 1ull);  // another warp installed the tag first
  }
  return static_cast<long long>(v & 0xffffffull);
}

// Polls of a counter word that is not installed yet, at 256 ns or more each:
// the wait gives up after about a second.
constexpr int kInstallWaitRounds = 1 << 22;

// One-wave mode: the counter words (tier-2 range counters, arrival tickets)
// each have one installer, a warp that resets the word to this call's tag
// with count 0 at the start of the kernel (atomic exchange). Adds one and
// returns the count before the addition; an addition that found the word
// still stale (the installer had not run yet; every CTA is resident, so it
// will) was discarded by the install, so the warp waits for the tag and adds
// again. No compare-and-swap races: with hundreds of warps adding to one word
// at once, claiming it by compare-and-swap thrashes. Returns -1 (and sets
// kErrTicket) if the tag did not appear within kInstallWaitRounds polls.
__device__ __forceinline__ void install_counter(unsigned long long* word, unsigned long long epoch) {
  atomicExch(word, epoch << 24);
}

__device__ __forceinline__ long long installed_fetch_add(unsigned long long* word, unsigned long long epoch, int* err) {
  for (int it = 0; it < kInstallWaitRounds; ++it) {
    const unsigned long long v = atomicAdd(word, 1ull);
    if ((v >> 24) == epoch) return static_cast<long long>(v & 0xffffffull);
    // not installed yet: wait for the tag, then add again
    while ((ld_acquire_u64(word) >> 24) != epoch && ++it < kInstallWaitRounds) __nanosleep(256);
  }
  atomicOr(err, kErrTicket);
  return -1;
}

// Arrival ticket of one split sequence (one per KV head): counts the pieces
// that have written their partials. Returns the pieces arrived including this
// one, or 0 if the ticket could not be claimed (an error is set).
__device__ __forceinline__ unsigned ticket_arrive(unsigned long long* ticket, unsigned long long epoch, int* err) {
  const long long before = tagged_fetch_add(ticket, epoch, err);
  return before < 0 ? 0u : static_cast<unsigned>(before + 1);
}

// Bounded wait (lane 0 polls, the warp follows) until an arrival ticket reads
// `pieces` arrivals in this call's epoch. The polls are relaxed loads with a
// back-off (many warps may poll one ticket while the arrivals still land on
// it); once the count shows, a fence orders the warp's later loads of the
// partials after the writers' release (their fence before the arrival), and
// __syncwarp carries that order to the other lanes. Returns false (and sets
// kErrMergeWait) after limit_ns.
__device__ __forceinline__ bool wait_ticket(const unsigned long long* ticket, unsigned long long epoch,
                                            unsigned pieces, uint64_t limit_ns, int* err, int lane) {
  int ok = 0;
  if (lane == 0) {
    const uint64_t t0 = global_timer_ns();
    for (;;) {
      const unsigned long long v = ld_relaxed_u64(ticket);
      if ((v >> 24) == epoch && (v & 0xffffffull) >= pieces) {
        ok = 1;
        break;
      }
      if (global_timer_ns() - t0 > limit_ns) {
        atomicOr(err, kErrMergeWait);
        break;
      }
      __nanosleep(256);
    }
    __threadfence();
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Merge the S fp32 partials of one split sequence for one KV head (8 query
// heads h0 .. h0+7) with one warp: w_i = 2^(LSE_i - M), O = sum w_i O_i / sum
// w_i (bf16), LSE = M + log2 sum w_i. Lane l owns dims l, l+32, l+64, l+96.
template <int NG>
__device__ __forceinline__ void merge_split_warp(const float* part_o, const float* part_lse, const SplitInfo& si,
                                                 int w, int64_t b, int h0, __nv_bfloat16* out, float* lse, int lane) {
  float m[8], den[8], acc[4][8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    m[h] = -INFINITY;
    den[h] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j][h] = 0.f;
  }
#pragma unroll 1
  for (int s = 0; s < si.S; ++s) {
    const int64_t sid = slot_id(si.first_cta + s, s == 0 ? si.first_slot : 0);
    const float4* lr = reinterpret_cast<const float4*>(part_lse + (sid * NG + w) * kGroup);
    const float4 la = __ldcg(lr), lb = __ldcg(lr + 1);
    const float l8[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
    float4 o[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4* orow = reinterpret_cast<const float4*>(part_o + ((sid * NG + w) * kHeadDim + lane + 32 * j) * kGroup);
      o[j][0] = __ldcg(orow);
      o[j][1] = __ldcg(orow + 1);
    }
    float sc[8], wt[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const float mn = fmaxf(m[h], l8[h]);
      const float sh = mn == -INFINITY ? 0.f : mn;  // all -inf so far: no NaN from -inf - -inf
      sc[h] = ex2(m[h] - sh);  // 0 while nothing has been added (m = -inf)
      wt[h] = ex2(l8[h] - sh);
      den[h] = den[h] * sc[h] + wt[h];
      m[h] = mn;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float o8[8] = {o[j][0].x, o[j][0].y, o[j][0].z, o[j][0].w, o[j][1].x, o[j][1].y, o[j][1].z, o[j][1].w};
#pragma unroll
      for (int h = 0; h < 8; ++h) acc[j][h] = acc[j][h] * sc[h] + wt[h] * o8[h];
    }
  }
  __nv_bfloat16* ob = out + (b * kQoHeads + h0) * kHeadDim;
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const float inv = den[h] > 0.f ? 1.f / den[h] : 0.f;  // no valid token in any piece: O = 0
#pragma unroll
    for (int j = 0; j < 4; ++j) ob[h * kHeadDim + lane + 32 * j] = __float2bfloat16_rn(acc[j][h] * inv);
  }
  if (lane < 8 && lse != nullptr) {
    float mm = m[0], dd = den[0];
#pragma unroll
    for (int h = 1; h < 8; ++h) {
      if (lane == h) {
        mm = m[h];
        dd = den[h];
      }
    }
    lse[b * kQoHeads + h0 + lane] = mm + log2f(dd);
  }
}

// Bytes one staged partial takes in shared memory: O [128 dims][8 heads] fp32 + 8 LSEs.
constexpr int kStagedPartialBytes = kHeadDim * kGroup * 4 + kGroup * 4;

// merge_split_warp with the partials staged through this warp's shared memory
// (free once its pipeline has drained): up to `cap` partials are fetched with
// cp.async in one round trip, then folded in with the same running-max update.
template <int NG>
__device__ __forceinline__ void merge_split_warp_staged(const float* part_o, const float* part_lse, const SplitInfo& si,
                                                        int w, int64_t b, int h0, __nv_bfloat16* out, float* lse,
                                                        uint32_t stage_smem, const uint8_t* stage_ptr, int cap,
                                                        int lane) {
  float m[8], den[8], acc[4][8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    m[h] = -INFINITY;
    den[h] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j][h] = 0.f;
  }
  for (int s0 = 0; s0 < si.S; s0 += cap) {
    const int n = min(cap, si.S - s0);
    for (int i = 0; i < n; ++i) {
      const int s = s0 + i;
      const int64_t sid = slot_id(si.first_cta + s, s == 0 ? si.first_slot : 0);
      const float* src_o = part_o + (sid * NG + w) * (kHeadDim * kGroup);
      const uint32_t dst = stage_smem + i * kStagedPartialBytes;
#pragma unroll
      for (int c = 0; c < 8; ++c) cp_async_16(dst + (c * 32 + lane) * 16, src_o + (c * 32 + lane) * 4, 16u);
      if (lane < 2) cp_async_16(dst + kHeadDim * kGroup * 4 + lane * 16, part_lse + (sid * NG + w) * kGroup + lane * 4, 16u);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();
    for (int i = 0; i < n; ++i) {
      const float* sp = reinterpret_cast<const float*>(stage_ptr + i * kStagedPartialBytes);
      const float4 la = *reinterpret_cast<const float4*>(sp + kHeadDim * kGroup);
      const float4 lb = *reinterpret_cast<const float4*>(sp + kHeadDim * kGroup + 4);
      const float l8[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
      float sc[8], wt[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float mn = fmaxf(m[h], l8[h]);
        const float sh = mn == -INFINITY ? 0.f : mn;  // all -inf so far: no NaN from -inf - -inf
        sc[h] = ex2(m[h] - sh);  // 0 while nothing has been added (m = -inf)
        wt[h] = ex2(l8[h] - sh);
        den[h] = den[h] * sc[h] + wt[h];
        m[h] = mn;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 x = *reinterpret_cast<const float4*>(sp + (lane + 32 * j) * kGroup);
        const float4 y = *reinterpret_cast<const float4*>(sp + (lane + 32 * j) * kGroup + 4);
        const float o8[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
        for (int h = 0; h < 8; ++h) acc[j][h] = acc[j][h] * sc[h] + wt[h] * o8[h];
      }
    }
    __syncwarp();  // the staging area is reused by the next batch
  }
  __nv_bfloat16* ob = out + (b * kQoHeads + h0) * kHeadDim;
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const float inv = den[h] > 0.f ? 1.f / den[h] : 0.f;  // no valid token in any piece: O = 0
#pragma unroll
    for (int j = 0; j < 4; ++j) ob[h * kHeadDim + lane + 32 * j] = __float2bfloat16_rn(acc[j][h] * inv);
  }
  if (lane < 8 && lse != nullptr) {
    float mm = m[0], dd = den[0];
#pragma unroll
    for (int h = 1; h < 8; ++h) {
      if (lane == h) {
        mm = m[h];
        dd = den[h];
      }
    }
    lse[b * kQoHeads + h0 + lane] = mm + log2f(dd);
  }
}

// Normalise and write a finished piece: bf16 O rows q-heads h0 .. h0+7 of
// sequence b plus their LSE (final), or an fp32 partial (O_i, LSE_i) into
// slot `sid` (layout [sid][NG][128 dims][8 heads], LSE [sid][NG][8]). Returns
// true for a partial of a sequence cut into at most fuse_max_splits pieces:
// the warp must count its arrival (arrive_pieces) after its main loop, and
// merges the sequence if its arrival was the last.
// DP (the FP8-cache path): accumulator row g of m-tile mt holds dim
// 16 mt + 2 g and row g + 8 dim 16 mt + 2 g + 1 (see attend_subtile_f8).
template <int NG, bool DP = false>
__device__ __forceinline__ bool finish_piece(const HeadState& st, bool final_piece, int64_t b, int h0, int64_t sid,
                                             int w, const SplitInfo& si, const DecodeParams& p, int lane,
                                             float oscale = 1.f) {
  const int r = lane >> 2, c = lane & 3;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  float lt0 = st.l0, lt1 = st.l1;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    lt0 += __shfl_xor_sync(0xffffffffu, lt0, o);
    lt1 += __shfl_xor_sync(0xffffffffu, lt1, o);
  }
  // a piece whose tokens were all masked out has l = 0: O = 0, LSE = -inf
  // oscale: the FP8 path's acc holds O * l / cv, so its oscale is cv
  const float i0 = lt0 > 0.f ? oscale / lt0 : 0.f;
  const float i1 = lt1 > 0.f ? oscale / lt1 : 0.f;
  const float lse0 = lt0 > 0.f ? st.m0 + log2f(lt0) : -INFINITY;
  const float lse1 = lt1 > 0.f ? st.m1 + log2f(lt1) : -INFINITY;
  if (final_piece) {
    __nv_bfloat16* ob = out + (b * kQoHeads + h0) * kHeadDim;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      // rows = dims, cols = heads  ->  transpose to rows = heads, cols = dims
      const uint32_t x = movmatrix_trans(pack_bf16(st.acc[mt][0] * i0, st.acc[mt][1] * i1));
      const uint32_t y = movmatrix_trans(pack_bf16(st.acc[mt][2] * i0, st.acc[mt][3] * i1));
      if constexpr (DP) {  // x: dims 4c, 4c + 2; y: dims 4c + 1, 4c + 3 (of m-tile mt)
        *reinterpret_cast<uint2*>(ob + r * kHeadDim + mt * 16 + 4 * c) =
            make_uint2(__byte_perm(x, y, 0x5410), __byte_perm(x, y, 0x7632));
      } else {
        *reinterpret_cast<uint32_t*>(ob + r * kHeadDim + mt * 16 + 2 * c) = x;
        *reinterpret_cast<uint32_t*>(ob + r * kHeadDim + mt * 16 + 8 + 2 * c) = y;
      }
    }
    if (r == 0 && p.lse != nullptr) *reinterpret_cast<float2*>(p.lse + b * kQoHeads + h0 + 2 * c) = make_float2(lse0, lse1);
    return false;
  }
  float* po = p.part_o + (sid * NG + w) * (kHeadDim * kGroup);
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int d_lo = DP ? mt * 16 + 2 * r : mt * 16 + r;          // dim of accumulator row r
    const int d_hi = DP ? mt * 16 + 2 * r + 1 : mt * 16 + 8 + r;  // dim of accumulator row r + 8
    *reinterpret_cast<float2*>(po + d_lo * kGroup + 2 * c) = make_float2(st.acc[mt][0] * i0, st.acc[mt][1] * i1);
    *reinterpret_cast<float2*>(po + d_hi * kGroup + 2 * c) = make_float2(st.acc[mt][2] * i0, st.acc[mt][3] * i1);
  }
  if (r == 0) *reinterpret_cast<float2*>(p.part_lse + (sid * NG + w) * kGroup + 2 * c) = make_float2(lse0, lse1);
  return si.S <= p.fuse_max_splits;  // else the merge kernel combines this sequence
}

// finish_piece for the CUDA-core sub-tile (same outputs and partial layout).
template <int NG>
__device__ __forceinline__ bool finish_piece_cc(const CcState& cs, bool final_piece, int64_t b, int h0, int64_t sid,
                                                int w, const SplitInfo& si, const DecodeParams& p, int lane) {
  const int h = lane & 7, g = lane >> 3;
  const float inv = cs.l > 0.f ? 1.f / cs.l : 0.f;
  const float lse_v = cs.l > 0.f ? cs.m + log2f(cs.l) : -INFINITY;
  if (final_piece) {
    uint4* ob = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + (b * kQoHeads + h0 + h) * kHeadDim +
                                         32 * g);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      ob[i] = make_uint4(pack_bf16(cs.acc[8 * i] * inv, cs.acc[8 * i + 1] * inv),
                         pack_bf16(cs.acc[8 * i + 2] * inv, cs.acc[8 * i + 3] * inv),
                         pack_bf16(cs.acc[8 * i + 4] * inv, cs.acc[8 * i + 5] * inv),
                         pack_bf16(cs.acc[8 * i + 6] * inv, cs.acc[8 * i + 7] * inv));
    if (g == 0 && p.lse != nullptr) p.lse[b * kQoHeads + h0 + h] = lse_v;
    return false;
  }
  float* po = p.part_o + (sid * NG + w) * (kHeadDim * kGroup);
#pragma unroll
  for (int j = 0; j < 32; ++j) po[(32 * g + j) * kGroup + h] = cs.acc[j] * inv;
  if (g == 0) p.part_lse[(sid * NG + w) * kGroup + h] = lse_v;
  return si.S <= p.fuse_max_splits;
}

// Split record of decode CTA `cta`: how the sequence holding the last unit of
// its range is cut (sequence b of head group hg, pieces first_cta .. first_cta
// + S - 1, slot of the first piece), tagged with the low 32 bits of the call's
// epoch. The merge kernel's CTA for the boundary after `cta` reads it instead
// of searching kv_indptr.
__device__ __forceinline__ void write_split_rec(int4* rec, int cta, unsigned long long epoch, int b, int hg,
                                                const SplitInfo& si) {
  rec[cta] = make_int4(static_cast<int>(static_cast<unsigned>(epoch)), b, si.first_cta,
                       (si.S << 3) | (hg << 1) | si.first_slot);
}

// A split piece whose arrival a warp still has to count (see finish_piece): at
// most two per warp, since only the first and the last piece of a CTA's range
// can be partials.
struct OwedMerge {
  SplitInfo si;
  int b, h0;
};

// After its main loop, a warp counts the arrivals of its (at most two) pending
// pieces: one fence makes all of its partials visible device-wide, then lanes
// 0 and 1 move the two tickets in parallel. Bit i of the result is set when
// pending piece i was the last of its sequence to arrive, so this warp owes
// that sequence's merge. Deferring the arrivals keeps the fence and the atomic
// round trips out of the streaming loop.
template <int NG>
__device__ __forceinline__ unsigned arrive_pieces(const OwedMerge (&pend)[2], int n, int w, const DecodeParams& p,
                                                  int lane) {
  __threadfence();
  __syncwarp();
  bool last = false;
  if (lane < n) {
    const SplitInfo si = lane == 0 ? pend[0].si : pend[1].si;
    const unsigned arrived = ticket_arrive(p.tickets + static_cast<int64_t>(si.first_cta) * NG + w, p.epoch, p.err);
    last = arrived == static_cast<unsigned>(si.S);
  }
  return __ballot_sync(0xffffffffu, last);
}

}  // namespace gqa
