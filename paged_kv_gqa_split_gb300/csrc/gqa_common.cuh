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

// Where a piece's sequence was cut: S pieces held by decode CTAs first_cta ..
// first_cta + S - 1; the first of them in slot first_slot, the others in slot 0.
struct SplitInfo {
  int S;
  int first_cta;
  int first_slot;
};

// Arrival ticket of one split sequence (one per KV head): the word holds
// (call epoch << 24) | pieces arrived. A word from an earlier call (another
// epoch) counts as zero, so the tickets need no clearing between calls.
// Returns the number of pieces arrived including this one, or 0 if the CAS
// loop did not settle (then the merge kernel is not told and an error is set).
__device__ __forceinline__ unsigned ticket_arrive(unsigned long long* ticket, unsigned long long epoch, int* err) {
  unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(ticket);
  for (int it = 0; it < (1 << 16); ++it) {
    const unsigned long long nv = ((cur >> 24) == epoch) ? cur + 1 : ((epoch << 24) | 1ull);
    const unsigned long long prev = atomicCAS(ticket, cur, nv);
    if (prev == cur) return static_cast<unsigned>(nv & 0xffffffull);
    cur = prev;
  }
  atomicOr(err, kErrTicket);
  return 0;
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
template <int NG>
__device__ __forceinline__ bool finish_piece(const HeadState& st, bool final_piece, int64_t b, int h0, int64_t sid,
                                             int w, const SplitInfo& si, const DecodeParams& p, int lane) {
  const int r = lane >> 2, c = lane & 3;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  float lt0 = st.l0, lt1 = st.l1;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    lt0 += __shfl_xor_sync(0xffffffffu, lt0, o);
    lt1 += __shfl_xor_sync(0xffffffffu, lt1, o);
  }
  // a piece whose tokens were all masked out has l = 0: O = 0, LSE = -inf
  const float i0 = lt0 > 0.f ? 1.f / lt0 : 0.f;
  const float i1 = lt1 > 0.f ? 1.f / lt1 : 0.f;
  const float lse0 = lt0 > 0.f ? st.m0 + log2f(lt0) : -INFINITY;
  const float lse1 = lt1 > 0.f ? st.m1 + log2f(lt1) : -INFINITY;
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
    if (r == 0 && p.lse != nullptr) *reinterpret_cast<float2*>(p.lse + b * kQoHeads + h0 + 2 * c) = make_float2(lse0, lse1);
    return false;
  }
  float* po = p.part_o + (sid * NG + w) * (kHeadDim * kGroup);
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    *reinterpret_cast<float2*>(po + (mt * 16 + r) * kGroup + 2 * c) = make_float2(st.acc[mt][0] * i0, st.acc[mt][1] * i1);
    *reinterpret_cast<float2*>(po + (mt * 16 + 8 + r) * kGroup + 2 * c) =
        make_float2(st.acc[mt][2] * i0, st.acc[mt][3] * i1);
  }
  if (r == 0) *reinterpret_cast<float2*>(p.part_lse + (sid * NG + w) * kGroup + 2 * c) = make_float2(lse0, lse1);
  return si.S <= p.fuse_max_splits;  // else the merge kernel combines this sequence
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
