// Split-KV paged GQA decode, TMA-bulk-copy variant (selectable; not the default).
//
// Same problem, plan and math as gqa_decode_lsu.cu. Here one producer warp
// per CTA gathers the K and V rows of every token of a tile (NG heads x 256 B,
// contiguous inside the page) with one cp.async.bulk copy per row into a ring
// of STAGES shared-memory stages whose completion is tracked by mbarrier
// transaction counts, plus the query rows when a tile starts a piece; NG
// consumer warps (one per KV head) share each staged tile. On GB300 the bulk
// copy engine sustains ~25 GB/s per SM for these 1 KB rows whatever the ring
// depth (about 60% of the HBM copy bandwidth), so this variant stays below the
// LSU one; it is kept for comparison and for page layouts with larger pages.
// Every mbarrier wait is bounded: after ~2 s the waiting warp flags an error,
// the CTA lets in-flight copies land and returns.
#include <cuda_runtime.h>

#include "gqa_common.cuh"
#include "gqa_kernels.h"

namespace gqa {

// Source of the rows that pad a partly filled 16-token sub-tile: zero K gives
// a finite (masked) score, zero V contributes nothing. Never written.
__device__ __align__(128) uint8_t g_zero_rows[kPageBytes];

// Spin limit of the drain before exit: the copies a CTA has in flight when it
// gives up are waited for this long at most. The give-up limit of the other
// waits is DecodeParams::wait_limit_ns (normally the same 2 s).
constexpr uint64_t kWaitLimitNs = kDefaultWaitLimitNs;

template <int NG, int TILE, int STAGES>
struct TmaCfg {
  static constexpr int kHG = kKvHeads / NG;            // head groups on the unit line
  static constexpr int kRowBytes = NG * kHeadDim * 2;  // one token's NG head rows (K or V)
  static constexpr int kRowPitch = kRowBytes + 16;     // +16 B staggers ldmatrix rows over all banks
  static constexpr int kKOff = 0;
  static constexpr int kVOff = TILE * kRowPitch;
  static constexpr int kQOff = 2 * TILE * kRowPitch;
  static constexpr int kQBytes = NG * kGroup * kHeadDim * 2;
  static constexpr int kHdrOff = kQOff + kQBytes;
  static constexpr int kStageBytes = (kHdrOff + 32 + 127) / 128 * 128;  // header: 8 ints
  static constexpr int kBarOff = STAGES * kStageBytes;
  static constexpr int kSmemBytes = kBarOff + 2 * STAGES * 8 + 16;
  static constexpr int kThreads = (NG + 1) * 32;
  static_assert(TILE == 16 || TILE == 32, "tile is one or two 16-token sub-tiles");
  static_assert(kKvHeads % NG == 0, "NG divides the KV heads");
  static_assert(kSmemBytes <= 227 * 1024, "stage ring exceeds shared memory");
};

// Bounded mbarrier wait. Returns false (after flagging `err_bit` once) when
// the wait exceeds `limit_ns` or another role of the CTA already gave up.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_s, int* err,
                                             int err_bit, uint64_t limit_ns) {
  // One try_wait may suspend the thread for a system-dependent time, which can
  // outlast a limit below about a millisecond; such a limit spins on the
  // non-blocking test_wait instead. The limit is checked after every attempt
  // (the clock and the shared flag cost little next to it).
  const bool spin = limit_ns < 1000000ull;
  if (spin ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (spin ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (*abort_s) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(err, err_bit);
      *abort_s = 1;
      return false;
    }
  }
}

__device__ __forceinline__ int load_index(const int* __restrict__ idx, int total, int pos) {
  return pos < total ? __ldg(idx + pos) : 0;
}

// ------------------------------------------------------------------ producer
template <int NG, int TILE, int STAGES>
__device__ __forceinline__ void tma_producer(const DecodeParams& p, uint32_t sbase, volatile int* abort_s) {
  using C = TmaCfg<NG, TILE, STAGES>;
  const int lane = threadIdx.x & 31;
  const uint32_t full0 = sbase + C::kBarOff;
  const uint32_t empty0 = full0 + STAGES * 8;
  const uint64_t pol = l2_policy_evict_first();
  const uint8_t* __restrict__ kc = static_cast<const uint8_t*>(p.k_cache);
  const uint8_t* __restrict__ vc = static_cast<const uint8_t*>(p.v_cache);
  const uint8_t* __restrict__ qb = static_cast<const uint8_t*>(p.q);

  const int B = p.batch;
  const int T = __ldg(p.kv_indptr + B);
  const Plan pl = make_plan(static_cast<int64_t>(T) * C::kHG, p.plan);
  const int64_t u0 = pl.begin(blockIdx.x);
  const int64_t u1 = pl.end(blockIdx.x);

  uint32_t tiles = 0;
  bool ok = true;

  // Issue one tile: tokens [tt, tt + cnt) of sequence b, head group hg.
  auto emit = [&](int b, int hg, int tt, int cnt, int flags, int page, const SplitInfo& si) -> bool {
    const int stage = tiles % STAGES;
    const uint32_t par = (tiles / STAGES) & 1u;
    if (!wait_bounded(empty0 + 8 * stage, par ^ 1u, abort_s, p.err, kErrTimeoutEmpty, p.wait_limit_ns)) return false;
    const uint32_t sb = sbase + stage * C::kStageBytes;
    const uint32_t bar = full0 + 8 * stage;
    const int nrows = (cnt + 15) & ~15;
    const uint32_t bytes = 2u * nrows * C::kRowBytes + ((flags & F_QLOAD) ? C::kQBytes : 0u);
    if (lane == 0) {
      st_shared_v4(sb + C::kHdrOff, b, cnt, flags, hg);
      st_shared_v4(sb + C::kHdrOff + 16, si.S, si.first_cta, si.first_slot, 0);
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
          atomicOr(p.err, kErrBadPage);
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
            atomicOr(p.err, kErrBadPage);
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

  int last_b = 0, last_hg = 0;  // the range's last piece, for the split record
  SplitInfo last_si = {1, 0, 0};
  int64_t u = u0;
  while (ok && u < u1) {
    const int hg = static_cast<int>(u / T);
    int t = static_cast<int>(u - static_cast<int64_t>(hg) * T);
    const int t_stop = static_cast<int>(min(static_cast<int64_t>(T), u1 - static_cast<int64_t>(hg) * T));

    // window of 32 consecutive kv_indptr entries starting at the sequence holding t
    int wb = warp_find_seq(p.kv_indptr, B, t, lane);
    if (wb < 0) {
      if (lane == 0) atomicOr(p.err, kErrBadIndptr);
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
        if (lane == 0) atomicOr(p.err, kErrBadIndptr);
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
      const SeqSplit sp = seq_split(pl, static_cast<int64_t>(hg) * T + seq_lo, static_cast<int64_t>(hg) * T + seq_hi);
      const SplitInfo si = {static_cast<int>(sp.last_cta - sp.first_cta + 1), static_cast<int>(sp.first_cta),
                            sp.first_slot};
      last_b = b;
      last_hg = hg;
      last_si = si;

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
        if (!emit(b, hg, tt, cnt, flags, page, si)) {
          ok = false;
          break;
        }
      }
      t = p_hi;
    }
    u = static_cast<int64_t>(hg) * T + t_stop;
  }
  if (ok && u0 < u1 && lane == 0) write_split_rec(p.split_rec, blockIdx.x, p.epoch, last_b, last_hg, last_si);

  bool placed = false;
  if (ok) {
    // end-of-work marker
    const int stage = tiles % STAGES;
    const uint32_t par = (tiles / STAGES) & 1u;
    if (wait_bounded(empty0 + 8 * stage, par ^ 1u, abort_s, p.err, kErrTimeoutEmpty, p.wait_limit_ns)) {
      if (lane == 0) {
        const uint32_t sb = sbase + stage * C::kStageBytes;
        asm volatile("st.shared.v4.s32 [%0], {%1, %1, %2, %1};" ::"r"(sb + C::kHdrOff), "r"(0), "r"(F_DONE)
                     : "memory");
        mbar_arrive(full0 + 8 * stage);
      }
      placed = true;
    }
  }
  if (!placed) *abort_s = 1;  // gave up: the consumers stop at their next wait
  // No bulk copy may still be writing into this CTA's shared memory when it
  // exits. The consumers normally wait for every tile, but one that gave up
  // (its wait ran out) has stopped, so the producer itself waits for the last
  // tiles it issued (bounded as well). After the marker, its stage's earlier
  // tile was released by the consumers and is not waited for again (the
  // marker's arrival moved that barrier on by one more phase).
  if (lane == 0) {
    const uint32_t keep = placed ? STAGES - 1 : STAGES;
    const uint32_t first = tiles > keep ? tiles - keep : 0;
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
__device__ __forceinline__ void tma_consumer(const DecodeParams& p, uint32_t sbase, volatile int* abort_s) {
  using C = TmaCfg<NG, TILE, STAGES>;
  const int w = threadIdx.x >> 5;  // KV head within the head group
  const int lane = threadIdx.x & 31;
  const uint32_t full0 = sbase + C::kBarOff;
  const uint32_t empty0 = full0 + STAGES * 8;
  HeadState st;
  st.reset();
#pragma unroll
  for (int i = 0; i < 16; ++i) st.qf[i] = 0;
  // per-lane ldmatrix row offsets inside a stage (this warp's head is bytes w*256.. of each row)
  const uint32_t q_lane = C::kQOff + (w * kGroup + (lane & 7)) * (kHeadDim * 2) + (lane >> 3) * 16;
  const uint32_t k_lane = C::kKOff + ((lane & 7) + ((lane >> 3) & 1) * 8) * C::kRowPitch + w * 256 + (lane >> 4) * 16;
  const uint32_t v_lane = C::kVOff + ((lane & 7) + (lane >> 4) * 8) * C::kRowPitch + w * 256 + ((lane >> 3) & 1) * 16;

  OwedMerge pend[2];  // split pieces whose arrival is counted after the loop
  int n_pend = 0;
  for (uint32_t tiles = 0;; ++tiles) {
    const int stage = tiles % STAGES;
    const uint32_t par = (tiles / STAGES) & 1u;
    if (!wait_bounded(full0 + 8 * stage, par, abort_s, p.err, kErrTimeoutFull, p.wait_limit_ns)) return;
    const uint32_t sb = sbase + stage * C::kStageBytes;
    int hb, cnt, flags, hg;
    ld_shared_v4(sb + C::kHdrOff, hb, cnt, flags, hg);
    SplitInfo si;
    int unused;
    ld_shared_v4(sb + C::kHdrOff + 16, si.S, si.first_cta, si.first_slot, unused);
    if (flags & F_DONE) break;
    if (flags & F_QLOAD) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ldsm_x4(sb + q_lane + j * 64, st.qf[4 * j], st.qf[4 * j + 1], st.qf[4 * j + 2], st.qf[4 * j + 3]);
      st.reset();
    }
#pragma unroll
    for (int sub = 0; sub < TILE / 16; ++sub) {
      if (sub * 16 < cnt) {
        const int c = cnt - sub * 16;
        attend_subtile(st, sb + k_lane + sub * 16 * C::kRowPitch, sb + v_lane + sub * 16 * C::kRowPitch,
                       c >= 16 ? 0xffffu : ((1u << c) - 1u), p.scale_log2, lane);
      }
    }
    // the stage's shared memory is no longer read by this warp
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * stage);
    if (flags & F_END) {
      const int h0 = (hg * NG + w) * kGroup;
      if (finish_piece<NG>(st, (flags & F_FINAL) != 0, hb, h0, slot_id(blockIdx.x, (flags & F_SLOT1) ? 1 : 0), w,
                           si, p, lane)) {
        pend[n_pend < 2 ? n_pend : 1] = {si, hb, h0};
        n_pend = min(n_pend + 1, 2);
      }
    }
  }
  if (n_pend == 0) return;
  const unsigned owe = arrive_pieces<NG>(pend, n_pend, w, p, lane);
#pragma unroll 1
  for (int i = 0; i < 2; ++i) {
    if (!((owe >> i) & 1u)) continue;
    __threadfence();
    merge_split_warp<NG>(p.part_o, p.part_lse, pend[i].si, w, pend[i].b, pend[i].h0,
                         static_cast<__nv_bfloat16*>(p.out), p.lse, lane);
  }
}

template <int NG, int TILE, int STAGES>
__global__ void __launch_bounds__((NG + 1) * 32, 1) gqa_decode_tma_kernel(const DecodeParams p) {
  using C = TmaCfg<NG, TILE, STAGES>;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  volatile int* abort_s = reinterpret_cast<volatile int*>(smem + C::kBarOff + 2 * STAGES * 8);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(sbase + C::kBarOff + 8 * s, 1);              // full: producer arrival + tx bytes
      mbar_init(sbase + C::kBarOff + 8 * (STAGES + s), NG);  // empty: one arrival per consumer warp
    }
    *abort_s = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // The merge grid may become resident now; it waits for this grid to finish.
  pdl_launch_dependents();
  if (p.skip_if_set != nullptr && *p.skip_if_set != 0) return;
  if ((threadIdx.x >> 5) == NG) {
    tma_producer<NG, TILE, STAGES>(p, sbase, abort_s);
  } else {
    tma_consumer<NG, TILE, STAGES>(p, sbase, abort_s);
  }
}

template <int NG, int TILE, int STAGES>
static cudaError_t launch_tma(const DecodeParams& p, int num_ctas, cudaStream_t stream) {
  using C = TmaCfg<NG, TILE, STAGES>;
  static std::atomic<int> configured[kMaxDevices];
  const cudaError_t e = set_smem_limit_once(
      configured, reinterpret_cast<const void*>(gqa_decode_tma_kernel<NG, TILE, STAGES>), C::kSmemBytes);
  if (e != cudaSuccess) return e;
  gqa_decode_tma_kernel<NG, TILE, STAGES><<<num_ctas, C::kThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

#define GQA_TMA_VARIANTS(X) X(4, 16, 5) X(4, 32, 3) X(1, 16, 4)

int tma_smem_bytes(int ng, int tile, int stages) {
#define X(NG, TL, ST) \
  if (ng == NG && tile == TL && stages == ST) return TmaCfg<NG, TL, ST>::kSmemBytes;
  GQA_TMA_VARIANTS(X)
#undef X
  return -1;
}

cudaError_t launch_decode_tma(int ng, int tile, int stages, const DecodeParams& p, int num_ctas, cudaStream_t stream) {
#define X(NG, TL, ST) \
  if (ng == NG && tile == TL && stages == ST) return launch_tma<NG, TL, ST>(p, num_ctas, stream);
  GQA_TMA_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace gqa
