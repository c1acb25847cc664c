// Paged-KV GQA decode for sm_103a: split-KV decode kernel and LSE merge kernel.
//
// Problem (kernelindex.com page "gqa_paged_decode_h32_kv4_d128_ps1", kernel and
// run() docstring): 32 query heads over 4 KV heads, head_dim 128, page size 1,
// bf16 q / k_cache / v_cache, CSR page table (kv_indptr, kv_indices). Output
// O[b, h, :] = softmax(sm_scale * q K^T) V in bf16 and a base-2 log-sum-exp
// per (sequence, head) in fp32; an empty sequence gives zeros and -inf.
//
// Decode kernel (one CTA per SM, persistent over a balanced unit range; the
// plan is described in gqa_plan.h):
//   * one producer warp walks the CTA's unit range sequence by sequence and
//     cuts it into tiles of TILE tokens that never cross a sequence. For each
//     tile it gathers the K and V rows of every token (NG heads x 256 B,
//     contiguous inside the page) with one TMA bulk copy per row into a ring of
//     STAGES shared-memory stages, plus the query rows when the tile starts a
//     piece. Completion is tracked by per-stage mbarrier transaction counts.
//   * NG consumer warps, one per KV head, share each staged tile. Per 16-token
//     sub-tile a warp computes S^T = K Q^T (16 tokens x 8 heads) with eight
//     bf16 m16n8k16 mma.sync, an online base-2 softmax with running max and
//     sum, transposes P in registers (movmatrix) and accumulates
//     O^T += V^T P^T (128 dims x 8 heads) with eight more mma.sync.
//   * at the end of a piece the warp writes either the final bf16 O and LSE
//     (the piece is the whole sequence) or an fp32 partial (O_i, LSE_i).
// Merge kernel (launched with programmatic dependent launch): for every
// sequence cut by a CTA boundary, LSE-weighted combination of its partials
// (the merge of the split-K GQA path on the sigit.si vLLM "qsa.py" page,
// extended with the merged LSE); it also writes the empty sequences.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "gqa_kernels.h"
#include "gqa_plan.h"
#include "gqa_ptx.cuh"

namespace gqa {

// Sticky device-side error word (bit flags, see gqa_kernels.h). Only set on
// conditions that should never occur with valid inputs; read by the host API.
__device__ int g_device_error;

// Source of the rows that pad a partly filled 16-token sub-tile: zero K gives
// a finite (masked) score, zero V contributes nothing. Never written.
__device__ __align__(128) uint8_t g_zero_rows[kPageBytes];

enum : int { F_QLOAD = 1, F_END = 2, F_FINAL = 4, F_SLOT1 = 8, F_DONE = 16 };

// Spin limit for every mbarrier wait: a wait that is still unsatisfied after
// this long records an error and the CTA returns.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

template <int NG, int TILE, int STAGES>
struct DecodeCfg {
  static constexpr int kHG = kKvHeads / NG;            // head groups on the unit line
  static constexpr int kRowBytes = NG * kHeadDim * 2;  // one token's NG head rows (K or V)
  static constexpr int kRowPitch = kRowBytes + 16;     // +16 B staggers ldmatrix rows over all banks
  static constexpr int kKOff = 0;
  static constexpr int kVOff = TILE * kRowPitch;
  static constexpr int kQOff = 2 * TILE * kRowPitch;
  static constexpr int kQBytes = NG * kGroup * kHeadDim * 2;
  static constexpr int kHdrOff = kQOff + kQBytes;
  static constexpr int kStageBytes = (kHdrOff + 16 + 127) / 128 * 128;
  static constexpr int kBarOff = STAGES * kStageBytes;
  static constexpr int kSmemBytes = kBarOff + 2 * STAGES * 8 + 16;
  static constexpr int kThreads = (NG + 1) * 32;
  static_assert(TILE == 16 || TILE == 32, "tile is one or two 16-token sub-tiles");
  static_assert(kKvHeads % NG == 0, "NG divides the KV heads");
  static_assert(kSmemBytes <= 227 * 1024, "stage ring exceeds shared memory");
};

// Bounded mbarrier wait. Returns false (after flagging `err_bit` once) when
// the wait exceeds kWaitLimitNs or another role of the CTA already gave up.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_s, int err_bit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort_s) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicOr(&g_device_error, err_bit);
        *abort_s = 1;
        return false;
      }
    }
  }
}

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

__device__ __forceinline__ int load_indptr_window(const int* __restrict__ indptr, int batch, int base, int lane) {
  const int pos = base + lane;
  return pos <= batch ? __ldg(indptr + pos) : INT32_MAX;
}

__device__ __forceinline__ int load_index(const int* __restrict__ idx, int total, int pos) {
  return pos < total ? __ldg(idx + pos) : 0;
}

// ------------------------------------------------------------------ producer
template <int NG, int TILE, int STAGES>
__device__ __forceinline__ void decode_producer(const DecodeParams& p, uint32_t sbase, volatile int* abort_s) {
  using C = DecodeCfg<NG, TILE, STAGES>;
  const int lane = threadIdx.x & 31;
  const uint32_t full0 = sbase + C::kBarOff;
  const uint32_t empty0 = full0 + STAGES * 8;
  const uint64_t pol = l2_policy_evict_first();
  const uint8_t* __restrict__ kc = static_cast<const uint8_t*>(p.k_cache);
  const uint8_t* __restrict__ vc = static_cast<const uint8_t*>(p.v_cache);
  const uint8_t* __restrict__ qb = static_cast<const uint8_t*>(p.q);

  const int B = p.batch;
  const int T = __ldg(p.kv_indptr + B);
  const int64_t W = static_cast<int64_t>(T) * C::kHG;
  const int64_t q = units_per_cta(W, gridDim.x, p.min_units);
  const int64_t u0 = static_cast<int64_t>(blockIdx.x) * q;
  const int64_t u1 = min(u0 + q, W);

  uint32_t tiles = 0;
  bool ok = true;

  // Issue one tile: tokens [tt, tt + cnt) of sequence b, head group hg.
  auto emit = [&](int b, int hg, int tt, int cnt, int flags, int page) -> bool {
    const int stage = tiles % STAGES;
    const uint32_t par = (tiles / STAGES) & 1u;
    if (!wait_bounded(empty0 + 8 * stage, par ^ 1u, abort_s, kErrTimeoutEmpty)) return false;
    const uint32_t sb = sbase + stage * C::kStageBytes;
    const uint32_t bar = full0 + 8 * stage;
    const int nrows = (cnt + 15) & ~15;
    const uint32_t bytes = 2u * nrows * C::kRowBytes + ((flags & F_QLOAD) ? C::kQBytes : 0u);
    if (lane == 0) {
      asm volatile("st.shared.v4.s32 [%0], {%1, %2, %3, %4};" ::"r"(sb + C::kHdrOff), "r"(b), "r"(cnt), "r"(flags),
                   "r"(hg)
                   : "memory");
      mbar_arrive_expect_tx(bar, bytes);
    }
    __syncwarp();
    const int64_t head_off = static_cast<int64_t>(hg) * C::kRowBytes;
    if constexpr (TILE == 16) {
      // lanes 0-15 copy the K row of token lane, lanes 16-31 the V row of token lane-16
      const int j = lane & 15;
      const int pg = __shfl_sync(0xffffffffu, page, j);
      const bool is_v = lane >= 16;
      const uint8_t* src = g_zero_rows;
      if (j < cnt) {
        if (p.num_pages_check > 0 && static_cast<unsigned>(pg) >= static_cast<unsigned>(p.num_pages_check)) {
          atomicOr(&g_device_error, kErrBadPage);
        } else {
          src = (is_v ? vc : kc) + static_cast<int64_t>(pg) * kPageBytes + head_off;
        }
      }
      bulk_g2s(sb + (is_v ? C::kVOff : C::kKOff) + j * C::kRowPitch, src, C::kRowBytes, bar, pol);
    } else {
      const int j = lane;
      if (j < nrows) {
        const uint8_t* ks = g_zero_rows;
        const uint8_t* vs = g_zero_rows;
        if (j < cnt) {
          if (p.num_pages_check > 0 && static_cast<unsigned>(page) >= static_cast<unsigned>(p.num_pages_check)) {
            atomicOr(&g_device_error, kErrBadPage);
          } else {
            ks = kc + static_cast<int64_t>(page) * kPageBytes + head_off;
            vs = vc + static_cast<int64_t>(page) * kPageBytes + head_off;
          }
        }
        bulk_g2s(sb + C::kKOff + j * C::kRowPitch, ks, C::kRowBytes, bar, pol);
        bulk_g2s(sb + C::kVOff + j * C::kRowPitch, vs, C::kRowBytes, bar, pol);
      }
    }
    if ((flags & F_QLOAD) && lane == 0) {
      const uint8_t* src = qb + (static_cast<int64_t>(b) * kQoHeads + hg * NG * kGroup) * kHeadDim * 2;
      bulk_g2s(sb + C::kQOff, src, C::kQBytes, bar);
    }
    ++tiles;
    return true;
  };

  int64_t u = u0;
  while (ok && u < u1) {
    const int hg = static_cast<int>(u / T);
    int t = static_cast<int>(u - static_cast<int64_t>(hg) * T);
    const int t_stop = static_cast<int>(min(static_cast<int64_t>(T), u1 - static_cast<int64_t>(hg) * T));

    // window of 32 consecutive kv_indptr entries starting at the sequence holding t
    int wb = warp_find_seq(p.kv_indptr, B, t, lane);
    if (wb < 0) {
      if (lane == 0) atomicOr(&g_device_error, kErrBadIndptr);
      ok = false;
      break;
    }
    int win = load_indptr_window(p.kv_indptr, B, wb, lane);

    // ring of four 32-entry windows of kv_indices, starting at the 32-aligned block holding t
    int ib = t & ~31;
    int ix0 = load_index(p.kv_indices, T, ib + lane);
    int ix1 = load_index(p.kv_indices, T, ib + 32 + lane);
    int ix2 = load_index(p.kv_indices, T, ib + 64 + lane);
    int ix3 = load_index(p.kv_indices, T, ib + 96 + lane);

    while (ok && t < t_stop) {
      unsigned m;
      for (;;) {
        m = __ballot_sync(0xffffffffu, win <= t);
        if (m != 0xffffffffu) break;
        wb += 31;
        win = load_indptr_window(p.kv_indptr, B, wb, lane);
      }
      if (m == 0) {  // indptr[wb] > t: decreasing kv_indptr
        if (lane == 0) atomicOr(&g_device_error, kErrBadIndptr);
        ok = false;
        break;
      }
      const int k = 31 - __clz(m);
      const int b = wb + k;
      const int seq_lo = __shfl_sync(0xffffffffu, win, k);
      const int seq_hi = __shfl_sync(0xffffffffu, win, k + 1);
      const int p_hi = min(seq_hi, t_stop);
      int pflags = 0;
      if (t == seq_lo && p_hi == seq_hi) pflags |= F_FINAL;
      if (static_cast<int64_t>(hg) * T + t != u0) pflags |= F_SLOT1;

      for (int tt = t; tt < p_hi; tt += TILE) {
        const int cnt = min(TILE, p_hi - tt);
        const int flags = pflags | (tt == t ? F_QLOAD : 0) | (tt + cnt == p_hi ? F_END : 0);
        while (tt >= ib + 32) {
          ix0 = ix1;
          ix1 = ix2;
          ix2 = ix3;
          ib += 32;
          ix3 = load_index(p.kv_indices, T, ib + 96 + lane);
        }
        // page of token tt + lane (tt - ib < 32, so tt + lane - ib < 64)
        const int off = tt + lane - ib;
        const int pa = __shfl_sync(0xffffffffu, ix0, off & 31);
        const int pb = __shfl_sync(0xffffffffu, ix1, off & 31);
        const int page = off < 32 ? pa : pb;
        if (!emit(b, hg, tt, cnt, flags, page)) {
          ok = false;
          break;
        }
      }
      t = p_hi;
    }
    u = static_cast<int64_t>(hg) * T + t_stop;
  }

  if (ok) {
    // end-of-work marker
    const int stage = tiles % STAGES;
    const uint32_t par = (tiles / STAGES) & 1u;
    if (wait_bounded(empty0 + 8 * stage, par ^ 1u, abort_s, kErrTimeoutEmpty)) {
      if (lane == 0) {
        const uint32_t sb = sbase + stage * C::kStageBytes;
        asm volatile("st.shared.v4.s32 [%0], {%1, %1, %2, %1};" ::"r"(sb + C::kHdrOff), "r"(0), "r"(F_DONE)
                     : "memory");
        mbar_arrive(full0 + 8 * stage);
      }
      return;
    }
  }
  // Gave up: make sure no bulk copy is still writing into this CTA's shared
  // memory before it exits (bounded as well).
  *abort_s = 1;
  if (lane == 0) {
    const uint32_t first = tiles > STAGES ? tiles - STAGES : 0;
    for (uint32_t i = first; i < tiles; ++i) {
      const uint32_t bar = full0 + 8 * (i % STAGES);
      const uint32_t par = (i / STAGES) & 1u;
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar, par)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ consumer
template <int NG, int TILE, int STAGES>
__device__ __forceinline__ void decode_consumer(const DecodeParams& p, uint32_t sbase, volatile int* abort_s) {
  using C = DecodeCfg<NG, TILE, STAGES>;
  const int w = threadIdx.x >> 5;  // KV head within the head group
  const int lane = threadIdx.x & 31;
  const int c = lane & 3;   // column pair of the mma fragments: heads 2c, 2c+1
  const int r = lane >> 2;  // row of the mma fragments
  const uint32_t full0 = sbase + C::kBarOff;
  const uint32_t empty0 = full0 + STAGES * 8;
  const float sl2 = p.scale_log2;

  uint32_t qf[16];
  float acc[8][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) qf[i] = 0;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

  // per-lane ldmatrix row offsets inside a stage
  const uint32_t q_lane = C::kQOff + (w * kGroup + (lane & 7)) * (kHeadDim * 2) + (lane >> 3) * 16;
  const uint32_t k_lane = C::kKOff + ((lane & 7) + ((lane >> 3) & 1) * 8) * C::kRowPitch + w * 256 + (lane >> 4) * 16;
  const uint32_t v_lane = C::kVOff + ((lane & 7) + (lane >> 4) * 8) * C::kRowPitch + w * 256 + ((lane >> 3) & 1) * 16;

  for (uint32_t tiles = 0;; ++tiles) {
    const int stage = tiles % STAGES;
    const uint32_t par = (tiles / STAGES) & 1u;
    if (!wait_bounded(full0 + 8 * stage, par, abort_s, kErrTimeoutFull)) return;
    const uint32_t sb = sbase + stage * C::kStageBytes;
    int hb, cnt, flags, hg;
    asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(hb), "=r"(cnt), "=r"(flags), "=r"(hg)
                 : "r"(sb + C::kHdrOff)
                 : "memory");
    if (flags & F_DONE) return;

    if (flags & F_QLOAD) {
#pragma unroll
      for (int j = 0; j < 4; ++j) ldsm_x4(sb + q_lane + j * 64, qf[4 * j], qf[4 * j + 1], qf[4 * j + 2], qf[4 * j + 3]);
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    }

#pragma unroll
    for (int sub = 0; sub < TILE / 16; ++sub) {
      if (sub * 16 < cnt) {
        // S^T (16 tokens x 8 heads) = K (16 x 128) . Q^T (128 x 8)
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t ka = sb + k_lane + sub * 16 * C::kRowPitch;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(ka + kk * 32, a0, a1, a2, a3);
          mma_bf16_16816(s, a0, a1, a2, a3, qf[2 * kk], qf[2 * kk + 1]);
        }
        // base-2 logits; tokens past the tile's count are masked out
        const int tok0 = sub * 16 + r;
        s[0] = tok0 < cnt ? s[0] * sl2 : -INFINITY;
        s[1] = tok0 < cnt ? s[1] * sl2 : -INFINITY;
        s[2] = tok0 + 8 < cnt ? s[2] * sl2 : -INFINITY;
        s[3] = tok0 + 8 < cnt ? s[3] * sl2 : -INFINITY;
        float mx0 = fmaxf(s[0], s[2]);
        float mx1 = fmaxf(s[1], s[3]);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float mn0 = fmaxf(m0, mx0);
        const float mn1 = fmaxf(m1, mx1);
        const float a0 = ex2(m0 - mn0);
        const float a1 = ex2(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        const float p0 = ex2(s[0] - mn0), p1 = ex2(s[1] - mn1);  // token r
        const float p2 = ex2(s[2] - mn0), p3 = ex2(s[3] - mn1);  // token r + 8
        // the running sum keeps fp32 probabilities; only the P.V operand is bf16
        l0 = l0 * a0 + (p0 + p2);
        l1 = l1 * a1 + (p1 + p3);
        const uint32_t plo = pack_bf16(p0, p1);
        const uint32_t phi = pack_bf16(p2, p3);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          acc[mt][0] *= a0;
          acc[mt][1] *= a1;
          acc[mt][2] *= a0;
          acc[mt][3] *= a1;
        }
        // P^T as the B operand (16 tokens x 8 heads): transpose the two 8x8 blocks
        const uint32_t b0 = movmatrix_trans(plo);
        const uint32_t b1 = movmatrix_trans(phi);
        // O^T (128 dims x 8 heads) += V^T (128 x 16) . P^T (16 x 8)
        const uint32_t va = sb + v_lane + sub * 16 * C::kRowPitch;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t v0, v1, v2, v3;
          ldsm_x4_trans(va + mt * 32, v0, v1, v2, v3);
          mma_bf16_16816(acc[mt], v0, v1, v2, v3, b0, b1);
        }
      }
    }
    // the stage's shared memory is no longer read by this warp
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * stage);

    if (flags & F_END) {
      float lt0 = l0, lt1 = l1;
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        lt0 += __shfl_xor_sync(0xffffffffu, lt0, o);
        lt1 += __shfl_xor_sync(0xffffffffu, lt1, o);
      }
      const float i0 = 1.f / lt0;
      const float i1 = 1.f / lt1;
      const float lse0 = m0 + log2f(lt0);
      const float lse1 = m1 + log2f(lt1);
      const int hbase = (hg * NG + w) * kGroup;  // first query head of this KV head
      if (flags & F_FINAL) {
        __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.out) + (static_cast<int64_t>(hb) * kQoHeads + hbase) * kHeadDim;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          // rows = dims, cols = heads  ->  transpose to rows = heads, cols = dims
          const uint32_t x = movmatrix_trans(pack_bf16(acc[mt][0] * i0, acc[mt][1] * i1));
          const uint32_t y = movmatrix_trans(pack_bf16(acc[mt][2] * i0, acc[mt][3] * i1));
          *reinterpret_cast<uint32_t*>(ob + r * kHeadDim + mt * 16 + 2 * c) = x;
          *reinterpret_cast<uint32_t*>(ob + r * kHeadDim + mt * 16 + 8 + 2 * c) = y;
        }
        if (r == 0) *reinterpret_cast<float2*>(p.lse + static_cast<int64_t>(hb) * kQoHeads + hbase + 2 * c) = make_float2(lse0, lse1);
      } else {
        const int64_t sid = slot_id(blockIdx.x, (flags & F_SLOT1) ? 1 : 0);
        float* po = p.part_o + (sid * NG + w) * (kHeadDim * kGroup);  // [dim][head]
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          *reinterpret_cast<float2*>(po + (mt * 16 + r) * kGroup + 2 * c) = make_float2(acc[mt][0] * i0, acc[mt][1] * i1);
          *reinterpret_cast<float2*>(po + (mt * 16 + 8 + r) * kGroup + 2 * c) = make_float2(acc[mt][2] * i0, acc[mt][3] * i1);
        }
        if (r == 0) *reinterpret_cast<float2*>(p.part_lse + (sid * NG + w) * kGroup + 2 * c) = make_float2(lse0, lse1);
      }
    }
  }
}

template <int NG, int TILE, int STAGES>
__global__ void __launch_bounds__((NG + 1) * 32, 1) gqa_decode_kernel(const DecodeParams p) {
  using C = DecodeCfg<NG, TILE, STAGES>;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  volatile int* abort_s = reinterpret_cast<volatile int*>(smem + C::kBarOff + 2 * STAGES * 8);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(sbase + C::kBarOff + 8 * s, 1);                 // full: producer arrival + tx bytes
      mbar_init(sbase + C::kBarOff + 8 * (STAGES + s), NG);     // empty: one arrival per consumer warp
    }
    *abort_s = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // The merge grid may become resident now; it waits for this grid to finish.
  pdl_launch_dependents();
  if (p.skip_if_set != nullptr && *p.skip_if_set != 0) return;
  if ((threadIdx.x >> 5) == NG) {
    decode_producer<NG, TILE, STAGES>(p, sbase, abort_s);
  } else {
    decode_consumer<NG, TILE, STAGES>(p, sbase, abort_s);
  }
}

// -------------------------------------------------------------------- merge
constexpr int kMergeThreads = 256;

template <int NG>
__global__ void __launch_bounds__(kMergeThreads) gqa_merge_kernel(const MergeParams p) {
  constexpr int kHG = kKvHeads / NG;
  constexpr int kH8 = NG * kGroup;  // query heads per head group
  extern __shared__ float wsm[];    // [splits][kH8] LSE, then normalised weights
  __shared__ float s_max[kH8], s_den[kH8];
  __shared__ int s_b;

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
  const int j = blockIdx.x / p.merge_ctas_per_boundary;    // boundary between decode CTAs j and j + 1
  const int sub = blockIdx.x % p.merge_ctas_per_boundary;
  const int64_t u = static_cast<int64_t>(j + 1) * q;
  if (u >= W) return;
  const int hg = static_cast<int>(u / T);
  const int t = static_cast<int>(u - static_cast<int64_t>(hg) * T);
  if (warp == 0) {
    const int b = warp_find_seq(p.kv_indptr, B, t, lane);
    if (lane == 0) s_b = b;
  }
  __syncthreads();
  const int b = s_b;
  if (b < 0) return;
  const int seq_lo = __ldg(p.kv_indptr + b);
  if (t == seq_lo) return;  // the boundary falls between two sequences: nothing is split here
  const int seq_hi = __ldg(p.kv_indptr + b + 1);
  const int64_t base_u = static_cast<int64_t>(hg) * T;
  const SeqSplit sp = seq_split(base_u + seq_lo, base_u + seq_hi, q);
  const int S = static_cast<int>(sp.last_cta - sp.first_cta + 1);
  const int rank = j - static_cast<int>(sp.first_cta);  // which of this sequence's S-1 boundaries
  const int nworkers = (S - 1) * p.merge_ctas_per_boundary;
  const int worker = rank * p.merge_ctas_per_boundary + sub;

  // Everything below reads the decode kernel's partials.
  pdl_wait();

  for (int i = tid; i < S * kH8; i += kMergeThreads) {
    const int s = i / kH8, hh = i - s * kH8;
    const int64_t sid = slot_id(sp.first_cta + s, s == 0 ? sp.first_slot : 0);
    wsm[i] = p.part_lse[sid * kH8 + hh];
  }
  __syncthreads();
  for (int hh = warp; hh < kH8; hh += kMergeThreads / 32) {
    float mx = -INFINITY;
    for (int s = lane; s < S; s += 32) mx = fmaxf(mx, wsm[s * kH8 + hh]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float den = 0.f;
    for (int s = lane; s < S; s += 32) den += ex2(wsm[s * kH8 + hh] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (lane == 0) {
      s_max[hh] = mx;
      s_den[hh] = den;
    }
  }
  __syncthreads();
  for (int i = tid; i < S * kH8; i += kMergeThreads) {
    const int hh = i % kH8;
    wsm[i] = ex2(wsm[i] - s_max[hh]) / s_den[hh];
  }
  __syncthreads();
  if (worker == 0 && tid < kH8) {
    p.lse[static_cast<int64_t>(b) * kQoHeads + hg * kH8 + tid] = s_max[tid] + log2f(s_den[tid]);
  }
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.out) + (static_cast<int64_t>(b) * kQoHeads + hg * kH8) * kHeadDim;

  if (S <= 16) {
    // item = (KV head g, 32-dim chunk); lane = one dim, all 8 heads, loop over the splits
    for (int it = worker * (kMergeThreads / 32) + warp; it < NG * 4; it += nworkers * (kMergeThreads / 32)) {
      const int g = it >> 2;
      const int d = (it & 3) * 32 + lane;
      float a[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) a[h] = 0.f;
#pragma unroll 4
      for (int s = 0; s < S; ++s) {
        const int64_t sid = slot_id(sp.first_cta + s, s == 0 ? sp.first_slot : 0);
        const float4* src = reinterpret_cast<const float4*>(p.part_o + ((sid * NG + g) * kHeadDim + d) * kGroup);
        const float4 x = src[0], y = src[1];
        const float* wt = wsm + s * kH8 + g * kGroup;
        a[0] += wt[0] * x.x; a[1] += wt[1] * x.y; a[2] += wt[2] * x.z; a[3] += wt[3] * x.w;
        a[4] += wt[4] * y.x; a[5] += wt[5] * y.y; a[6] += wt[6] * y.z; a[7] += wt[7] * y.w;
      }
#pragma unroll
      for (int h = 0; h < 8; ++h) ob[(g * kGroup + h) * kHeadDim + d] = __float2bfloat16_rn(a[h]);
    }
  } else {
    // item = (KV head g, dim d); lanes stride over the splits, then a warp reduction
    for (int it = worker * (kMergeThreads / 32) + warp; it < NG * kHeadDim; it += nworkers * (kMergeThreads / 32)) {
      const int g = it / kHeadDim;
      const int d = it - g * kHeadDim;
      float a[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) a[h] = 0.f;
      for (int s = lane; s < S; s += 32) {
        const int64_t sid = slot_id(sp.first_cta + s, s == 0 ? sp.first_slot : 0);
        const float4* src = reinterpret_cast<const float4*>(p.part_o + ((sid * NG + g) * kHeadDim + d) * kGroup);
        const float4 x = src[0], y = src[1];
        const float* wt = wsm + s * kH8 + g * kGroup;
        a[0] += wt[0] * x.x; a[1] += wt[1] * x.y; a[2] += wt[2] * x.z; a[3] += wt[3] * x.w;
        a[4] += wt[4] * y.x; a[5] += wt[5] * y.y; a[6] += wt[6] * y.z; a[7] += wt[7] * y.w;
      }
#pragma unroll
      for (int h = 0; h < 8; ++h) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a[h] += __shfl_xor_sync(0xffffffffu, a[h], o);
      }
      if (lane < 8) {
        float v = a[0];
#pragma unroll
        for (int h = 1; h < 8; ++h) v = (lane == h) ? a[h] : v;
        ob[(g * kGroup + lane) * kHeadDim + d] = __float2bfloat16_rn(v);
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
template <int NG, int TILE, int STAGES>
static cudaError_t launch_decode_impl(const DecodeParams& p, int num_ctas, cudaStream_t stream) {
  using C = DecodeCfg<NG, TILE, STAGES>;
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gqa_decode_kernel<NG, TILE, STAGES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  gqa_decode_kernel<NG, TILE, STAGES><<<num_ctas, C::kThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <int NG>
static cudaError_t launch_merge_impl(const MergeParams& p, cudaStream_t stream) {
  const int boundaries = p.num_decode_ctas > 1 ? p.num_decode_ctas - 1 : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(boundaries * p.merge_ctas_per_boundary);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(p.num_decode_ctas) * NG * kGroup * sizeof(float);
  if (cfg.dynamicSmemBytes > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(gqa_merge_kernel<NG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(cfg.dynamicSmemBytes));
    if (e != cudaSuccess) return e;
  }
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = p.use_pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gqa_merge_kernel<NG>, p);
}

int decode_smem_bytes(const KernelChoice& k) {
  if (k.heads_per_cta == 4 && k.tile == 16 && k.stages == 5) return DecodeCfg<4, 16, 5>::kSmemBytes;
  if (k.heads_per_cta == 4 && k.tile == 16 && k.stages == 4) return DecodeCfg<4, 16, 4>::kSmemBytes;
  if (k.heads_per_cta == 4 && k.tile == 32 && k.stages == 3) return DecodeCfg<4, 32, 3>::kSmemBytes;
  if (k.heads_per_cta == 2 && k.tile == 16 && k.stages == 4) return DecodeCfg<2, 16, 4>::kSmemBytes;
  if (k.heads_per_cta == 1 && k.tile == 16 && k.stages == 4) return DecodeCfg<1, 16, 4>::kSmemBytes;
  return -1;
}

cudaError_t launch_decode(const KernelChoice& k, const DecodeParams& p, int num_ctas, cudaStream_t stream) {
  if (k.heads_per_cta == 4 && k.tile == 16 && k.stages == 5) return launch_decode_impl<4, 16, 5>(p, num_ctas, stream);
  if (k.heads_per_cta == 4 && k.tile == 16 && k.stages == 4) return launch_decode_impl<4, 16, 4>(p, num_ctas, stream);
  if (k.heads_per_cta == 4 && k.tile == 32 && k.stages == 3) return launch_decode_impl<4, 32, 3>(p, num_ctas, stream);
  if (k.heads_per_cta == 2 && k.tile == 16 && k.stages == 4) return launch_decode_impl<2, 16, 4>(p, num_ctas, stream);
  if (k.heads_per_cta == 1 && k.tile == 16 && k.stages == 4) return launch_decode_impl<1, 16, 4>(p, num_ctas, stream);
  return cudaErrorInvalidValue;
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

}  // namespace gqa
