// Split-KV paged GQA decode, self-loading warps (the default decode kernel).
//
// Problem: the kernelindex.com page "gqa_paged_decode_h32_kv4_d128_ps1" (32
// query heads over 4 KV heads, head_dim 128, page size 1, bf16, CSR page table,
// bf16 O and base-2 LSE). Work split: gqa_plan.h (each CTA an equal share of
// all (token, head group) units; pieces of a sequence cut at CTA boundaries
// leave fp32 partials for the LSE merge kernel).
//
// Each warp owns one KV head of the CTA's head group and runs its own
// pipeline, with no barrier shared with any other warp:
//   * a walker cuts the CTA's unit range into 16-token tiles that never cross
//     a sequence (the kv_indptr window is kept in registers and searched with
//     warp ballots);
//   * for each tile the warp gathers the 256-byte K and V rows of its head for
//     the 16 tokens with 16-byte cp.async (two 256-byte rows per warp
//     instruction, L2 only), into a D-deep ring of private stages; rows past
//     the tile's end are zero-filled. Page ids come from a 256-entry ring in
//     shared memory that is itself filled by cp.async 224 tokens ahead, so no
//     global load sits on the issue path;
//   * the tile D - 1 ahead is issued before the warp waits for the current
//     one, so all D stages are in flight during the wait and D - 1 during the
//     math;
//   * a new piece's Q fragments are loaded into registers when its first tile
//     is issued (or prefetched to L2 if the register set is still in use).
// Measured on GB300 with random 1 KB pages: 16-byte cp.async gathers from 8
// warps per SM reach ~94% of the copy bandwidth, TMA bulk copies of the same
// rows ~60% at any ring depth; hence the LSU path here (the TMA variant is
// gqa_decode_tma.cu).
#include <cuda_runtime.h>

#include "gqa_common.cuh"
#include "gqa_kernels.h"

namespace gqa {

// Per-warp shared memory. bf16 cache (F8 = false): each stage holds the K and
// V head rows of one tile at a 272-byte pitch, ready for ldmatrix. FP8 cache
// (F8 = true): each stage holds the tile's 128-byte e4m3 head rows of K (at a
// 192-byte pitch: the 128-bit row reads of attend_subtile_f8 then hit 8
// distinct bank groups) and of V (at a 144-byte pitch, for ldmatrix), plus
// their per-token scales.
template <int NG, int D, bool F8 = false>
struct LsuCfg {
  static constexpr int kHG = kKvHeads / NG;           // head groups on the unit line
  static constexpr int kTile = 16;                    // tokens per stage (one mma sub-tile)
  static constexpr int kRowPitch = kHeadDim * 2 + 16; // 256 B head row + 16 B: ldmatrix rows hit all banks
  static constexpr int kRowBytes8 = kHeadDim;         // e4m3 head row
  // global row of one token (all 4 KV heads): 1 KB of bf16, or 512 B of e4m3 + 4 fp32 scales
  static constexpr int kGlobalRowBytes = F8 ? kKvHeads * kHeadDim + 4 * kKvHeads : kPageBytes;
  static constexpr int kK8Pitch = 192;                // F8 K row pitch
  static constexpr int kV8Pitch = 144;                // F8 V row pitch
  static constexpr int kKOff = 0;
  static constexpr int kVOff = F8 ? kTile * kK8Pitch : kTile * kRowPitch;
  static constexpr int kSkOff = kVOff + kTile * kV8Pitch;  // F8: K scales of the tile's tokens
  static constexpr int kSvOff = kSkOff + kTile * 4;         // F8: V scales
  static constexpr int kHdrOff = F8 ? kSvOff + kTile * 4 : 2 * kTile * kRowPitch;
  static constexpr int kStageBytes = kHdrOff + 32;    // tile header: 8 ints
  static constexpr int kIdsRing = 256;                // page ids held per warp (tokens)
  static constexpr int kIdsOff = D * kStageBytes;
  static constexpr int kPlanOff = kIdsOff + kIdsRing * 4;  // the warp's copy of the plan (SmemPlan)
  static constexpr int kWarpBytes = kPlanOff + 32;
  static constexpr int kThreads = NG * 32;
  static constexpr int kSmemBytes = NG * kWarpBytes;
  static_assert(D >= 2, "at least double buffering");
  static_assert(kStageBytes % 16 == 0 && kWarpBytes % 16 == 0, "16-byte aligned stages");
  static_assert(kSmemBytes <= 227 * 1024, "ring exceeds shared memory");
};

// What the walker needs of the plan when a piece starts (where the piece's
// sequence is cut), kept in shared memory so that it holds no registers in
// the streaming loop.
struct SmemPlan {
  int64_t W1, q1, q2;
  int P1, unused;
};

__device__ __forceinline__ SeqSplit seq_split_smem(const SmemPlan* sp, int64_t u_lo, int64_t u_hi) {
  Plan pl;
  pl.W1 = sp->W1;
  pl.q1 = sp->q1;
  pl.q2 = sp->q2;
  pl.P1 = sp->P1;
  return seq_split(pl, u_lo, u_hi);
}

struct Tile {
  int b, cnt, flags, hg, tt;
  SplitInfo si;
};

// SP: selected-token (sparse) mode. Every row of the batch is one "sequence" of
// exactly p.sparse_topk columns; kv_indices holds their resolved slots, and a
// slot of -1 (an invalid column) is masked out of the softmax.
// F8: the K/V caches are FP8 rows (kGlobalRowBytes per token): e4m3 values of
// the 4 KV heads, then their fp32 scales.
template <int NG, int D, bool SP, bool F8 = false>
__global__ void __launch_bounds__(NG * 32, F8 ? 3 : 16 / NG) gqa_decode_lsu_kernel(const DecodeParams p) {
  using C = LsuCfg<NG, D, F8>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int w = threadIdx.x >> 5;  // KV head within the head group
  const int lane = threadIdx.x & 31;
  uint8_t* wsm = smem + w * C::kWarpBytes;
  const uint32_t wbase = smem_addr(wsm);
  const int* ids = reinterpret_cast<const int*>(wsm + C::kIdsOff);
  const uint32_t ids_base = wbase + C::kIdsOff;

  // The merge grid may become resident now; it waits for this grid to finish.
  pdl_launch_dependents();
  // Selected-token mode is launched as a dependent of the slot-resolving
  // kernel: nothing that kernel writes is read before this returns. Without a
  // programmatic dependency (every other launch) it returns at once.
  pdl_wait();
  if (p.skip_if_set != nullptr && *p.skip_if_set != 0) return;

  const uint8_t* __restrict__ kc = static_cast<const uint8_t*>(p.k_cache);
  const uint8_t* __restrict__ vc = static_cast<const uint8_t*>(p.v_cache);
  const __nv_bfloat16* __restrict__ qg = static_cast<const __nv_bfloat16*>(p.q);
  const int B = p.batch;
  const int T = SP ? p.sparse_total : __ldg(p.kv_indptr + B);
  SmemPlan* splan = reinterpret_cast<SmemPlan*>(wsm + C::kPlanOff);
  int64_t u0, u1;
  {
    const Plan pl = make_plan(static_cast<int64_t>(T) * C::kHG, p.plan);
    u0 = pl.begin(blockIdx.x);
    u1 = pl.end(blockIdx.x);
    if (lane == 0) *splan = SmemPlan{pl.W1, pl.q1, pl.q2, pl.P1, 0};
    __syncwarp();
  }

  // ------------------------------------------------------------- walker
  int64_t u_next = u0;      // first unit of the next head-group segment
  bool seg_open = false, walk_ok = true;
  int hg = 0, tt = 0, t_stop = 0;  // segment: tokens [tt, t_stop) of head group hg
  int p_hi = 0, p_flags = 0, pb = 0;  // current piece: sequence pb, tokens up to p_hi
  SplitInfo p_si = {1, 0, 0};         // how the piece's sequence is cut across CTAs
  int wb = 0, win = 0;      // kv_indptr[wb + lane]
  int ib = 0;               // page-id ring holds tokens [ib, ib + 256)

  auto request_ids = [&](int pos) {  // page id of token pos into its ring slot (zero past the end)
    cp_async_4(ids_base + (pos & (C::kIdsRing - 1)) * 4, p.kv_indices + min(pos, T - 1), pos < T ? 4u : 0u);
  };

  auto next_tile = [&](Tile& tl) -> bool {
    while (walk_ok) {
      if (seg_open && tt < t_stop) {
        if (tt >= p_hi) {  // a new piece starts at tt: find its sequence
          int seq_lo, seq_hi;
          if (SP) {  // fixed-width rows
            pb = tt / p.sparse_topk;
            seq_lo = pb * p.sparse_topk;
            seq_hi = seq_lo + p.sparse_topk;
          } else {
            unsigned m;
            for (;;) {
              m = __ballot_sync(0xffffffffu, win <= tt);
              if (m != 0xffffffffu) break;
              wb += 31;
              win = load_indptr_window(p.kv_indptr, B, wb, lane);
            }
            if (m == 0) {  // kv_indptr[wb] > tt: a decreasing table
              if (lane == 0) atomicOr(p.err, kErrBadIndptr);
              walk_ok = false;
              break;
            }
            const int k = 31 - __clz(m);
            pb = wb + k;
            seq_lo = __shfl_sync(0xffffffffu, win, k);
            seq_hi = __shfl_sync(0xffffffffu, win, k + 1);
          }
          p_hi = min(seq_hi, t_stop);
          p_flags = F_QLOAD | ((tt == seq_lo && p_hi == seq_hi) ? F_FINAL : 0) |
                    ((static_cast<int64_t>(hg) * T + tt != u0) ? F_SLOT1 : 0);
          const int64_t base_u = static_cast<int64_t>(hg) * T;
          const SeqSplit sp = seq_split_smem(splan, base_u + seq_lo, base_u + seq_hi);
          p_si.S = static_cast<int>(sp.last_cta - sp.first_cta + 1);
          p_si.first_cta = static_cast<int>(sp.first_cta);
          p_si.first_slot = sp.first_slot;
        }
        tl.cnt = min(C::kTile, p_hi - tt);
        tl.flags = p_flags | ((tt + tl.cnt == p_hi) ? F_END : 0);
        tl.b = pb;
        tl.hg = hg;
        tl.tt = tt;
        tl.si = p_si;
        p_flags &= ~F_QLOAD;
        tt += tl.cnt;
        return true;
      }
      if (u_next >= u1) return false;
      // open the next head-group segment of the CTA's unit range
      hg = static_cast<int>(u_next / T);
      tt = static_cast<int>(u_next - static_cast<int64_t>(hg) * T);
      t_stop = static_cast<int>(min(static_cast<int64_t>(T), u1 - static_cast<int64_t>(hg) * T));
      u_next = static_cast<int64_t>(hg) * T + t_stop;
      seg_open = true;
      p_hi = tt;
      // the page ids depend on tt alone: request them first, so that their
      // round trip overlaps the search of kv_indptr
      ib = tt & ~31;
#pragma unroll
      for (int c = 0; c < C::kIdsRing / 32; ++c) request_ids(ib + 32 * c + lane);
      cp_async_commit();
      if (!SP) {
        wb = warp_find_seq(p.kv_indptr, B, tt, lane);
        if (wb >= 0) win = load_indptr_window(p.kv_indptr, B, wb, lane);
      }
      cp_async_wait<0>();
      __syncwarp();
      if (wb < 0) {
        if (lane == 0) atomicOr(p.err, kErrBadIndptr);
        walk_ok = false;
        break;
      }
    }
    return false;
  };

  // -------------------------------------------------------------- issue
  uint32_t qn[16];        // Q fragments of the next piece, loaded at issue time
  bool qn_busy = false;
  int issued = 0;
  bool more = true;
  auto issue = [&]() {
    const uint32_t sb = wbase + (issued % D) * C::kStageBytes;
    Tile tl;
    if (more && next_tile(tl)) {
      // keep the ring at [ib, ib + 256) with tl.tt < ib + 32: the ids this tile
      // reads were requested >= 12 tiles ago and have completed
      while (tl.tt >= ib + 32) {
        request_ids(ib + C::kIdsRing + lane);
        ib += 32;
      }
      int flags = tl.flags;
      const int64_t hoff = static_cast<int64_t>(tl.hg * NG + w) * (F8 ? kHeadDim : kHeadDim * 2);
      const int pc = lane & 15;  // 16-byte column of the 256-byte head row
      // tokens that enter the softmax: the first cnt, less (sparse mode) masked columns
      unsigned mask = tl.cnt >= 16 ? 0xffffu : ((1u << tl.cnt) - 1u);
      if constexpr (F8) {
        // 16 tokens x 8 16-byte chunks of the 128-byte e4m3 head row, for K and V
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tok = 4 * i + (lane >> 3), ch = lane & 7;
          bool valid = tok < tl.cnt;
          int pg = valid ? ids[(tl.tt + tok) & (C::kIdsRing - 1)] : 0;
          if (valid && p.num_pages_check > 0 &&
              static_cast<unsigned>(pg) >= static_cast<unsigned>(p.num_pages_check)) {
            atomicOr(p.err, kErrBadPage);
            valid = false;
            pg = 0;
          }
          const int64_t off = static_cast<int64_t>(pg) * C::kGlobalRowBytes + hoff + ch * 16;
          const uint32_t nbytes = valid ? 16u : 0u;
          cp_async_16(sb + C::kKOff + tok * C::kK8Pitch + ch * 16, kc + off, nbytes);
          cp_async_16(sb + C::kVOff + tok * C::kV8Pitch + ch * 16, vc + off, nbytes);
        }
        {  // the per-token scales of this KV head: lanes 0-15 K, 16-31 V
          const int tok = lane & 15;
          bool valid = tok < tl.cnt;
          int pg = valid ? ids[(tl.tt + tok) & (C::kIdsRing - 1)] : 0;
          if (valid && p.num_pages_check > 0 &&
              static_cast<unsigned>(pg) >= static_cast<unsigned>(p.num_pages_check)) {
            valid = false;
            pg = 0;
          }
          const int64_t off = static_cast<int64_t>(pg) * C::kGlobalRowBytes + kKvHeads * kHeadDim +
                              (tl.hg * NG + w) * 4;
          cp_async_4(sb + (lane < 16 ? C::kSkOff : C::kSvOff) + tok * 4, (lane < 16 ? kc : vc) + off,
                     valid ? 4u : 0u);
        }
      }
#pragma unroll
      for (int i = 0; i < (F8 ? 0 : 8); ++i) {
        const int tok = 2 * i + (lane >> 4);
        bool valid = tok < tl.cnt;
        int pg = valid ? ids[(tl.tt + tok) & (C::kIdsRing - 1)] : 0;
        if (SP) {
          if (pg < 0) {
            valid = false;
            pg = 0;
          }
          const unsigned bal = __ballot_sync(0xffffffffu, valid);  // lanes 0-15: token 2i, 16-31: 2i + 1
          mask = (mask & ~(3u << (2 * i))) | ((bal & 1u) << (2 * i)) | (((bal >> 16) & 1u) << (2 * i + 1));
        }
        if (valid && p.num_pages_check > 0 && static_cast<unsigned>(pg) >= static_cast<unsigned>(p.num_pages_check)) {
          atomicOr(p.err, kErrBadPage);
          valid = false;
          pg = 0;
        }
        const int64_t off = static_cast<int64_t>(pg) * kPageBytes + hoff + pc * 16;
        const uint32_t nbytes = valid ? 16u : 0u;
        cp_async_16(sb + C::kKOff + tok * C::kRowPitch + pc * 16, kc + off, nbytes);
        cp_async_16(sb + C::kVOff + tok * C::kRowPitch + pc * 16, vc + off, nbytes);
      }
      if (flags & F_QLOAD) {
        const int h0 = (tl.hg * NG + w) * kGroup;
        if (!qn_busy) {
          load_q_frags<F8>(qn, qg, tl.b, h0, lane);
          qn_busy = true;
          flags |= F_QREG;
        } else if (lane < 16) {
          prefetch_l2(qg + (static_cast<int64_t>(tl.b) * kQoHeads + h0) * kHeadDim + lane * 64);
        }
      }
      if (lane == 0) {
        st_shared_v4(sb + C::kHdrOff, tl.b, tl.cnt, flags, tl.hg);
        st_shared_v4(sb + C::kHdrOff + 16, tl.si.S, tl.si.first_cta, tl.si.first_slot, static_cast<int>(mask));
      }
    } else if (more) {
      more = false;
      if (lane == 0) st_shared_v4(sb + C::kHdrOff, 0, 0, F_DONE, 0);
    }
    cp_async_commit();  // one group per issue, even when empty
    ++issued;
  };

  // ------------------------------------------------------------ compute
  HeadState st;
  st.reset();
#pragma unroll
  for (int i = 0; i < 16; ++i) st.qf[i] = 0;
  // per-lane ldmatrix row addresses within a stage. F8: K row (lane >> 2) at
  // column (lane & 3) * 16 for the 128-bit reads; V matrix (lane >> 3) is
  // tokens 0-7 / 8-15 of dims block 0 / 1 for ldmatrix.trans.
  const uint32_t k_lane = F8 ? C::kKOff + (lane >> 2) * C::kK8Pitch + (lane & 3) * 16
                             : C::kKOff + ((lane & 7) + ((lane >> 3) & 1) * 8) * C::kRowPitch + (lane >> 4) * 16;
  const uint32_t v_lane = F8 ? C::kVOff + (((lane >> 3) & 1) * 8 + (lane & 7)) * C::kV8Pitch + (lane >> 4) * 16
                             : C::kVOff + ((lane & 7) + (lane >> 4) * 8) * C::kRowPitch + ((lane >> 3) & 1) * 16;

  OwedMerge pend[2];  // split pieces whose arrival is counted after the loop
  int n_pend = 0;
#pragma unroll 1
  for (int i = 0; i < D - 1; ++i) issue();
#pragma unroll 1
  for (int k = 0;; ++k) {
    issue();                 // tile k + D - 1, into the stage tile k - 1 used
    cp_async_wait<D - 1>();  // tile k has landed (one group per tile)
    __syncwarp();
    const uint32_t sb = wbase + (k % D) * C::kStageBytes;
    int hb, cnt, flags, thg;
    ld_shared_v4(sb + C::kHdrOff, hb, cnt, flags, thg);
    SplitInfo si;
    int tok_mask;
    ld_shared_v4(sb + C::kHdrOff + 16, si.S, si.first_cta, si.first_slot, tok_mask);
    if (flags & F_DONE) break;
    const int h0 = (thg * NG + w) * kGroup;
    if (flags & F_QLOAD) {
      if (flags & F_QREG) {
#pragma unroll
        for (int i = 0; i < 16; ++i) st.qf[i] = qn[i];
        qn_busy = false;
      } else {
        load_q_frags<F8>(st.qf, qg, hb, h0, lane);
      }
      st.reset();
      if constexpr (F8) st.qsc = q_frags_to_f16(st.qf);
    }
    if constexpr (F8) {
      const int r = lane >> 2;
      const float sk_lo = ld_shared_f32(sb + C::kSkOff + r * 4), sk_hi = ld_shared_f32(sb + C::kSkOff + (r + 8) * 4);
      const float sv_lo = ld_shared_f32(sb + C::kSvOff + r * 4), sv_hi = ld_shared_f32(sb + C::kSvOff + (r + 8) * 4);
      attend_subtile_f8(st, sb + k_lane, sb + v_lane, static_cast<unsigned>(tok_mask), p.scale_log2, sk_lo, sk_hi,
                        sv_lo, sv_hi, lane, C::kK8Pitch);
    } else {
      attend_subtile(st, sb + k_lane, sb + v_lane, static_cast<unsigned>(tok_mask), p.scale_log2, lane);
    }
    if (flags & F_END) {
      if (finish_piece<NG, F8>(st, (flags & F_FINAL) != 0, hb, h0, slot_id(blockIdx.x, (flags & F_SLOT1) ? 1 : 0),
                               w, si, p, lane, F8 ? st.cv : 1.f)) {
        pend[n_pend < 2 ? n_pend : 1] = {si, hb, h0};
        n_pend = min(n_pend + 1, 2);
      }
    }
    __syncwarp();  // every lane is done with this stage before it is refilled
  }
  cp_async_wait<0>();
  if (w == 0 && lane == 0 && u0 < u1 && walk_ok) write_split_rec(p.split_rec, blockIdx.x, p.epoch, pb, hg, p_si);
  if (n_pend == 0) return;
  // count the pending arrivals; for each that came last, merge the sequence
  // (every other piece's partial is visible by then), staging the partials
  // through the warp's drained ring
  const unsigned owe = arrive_pieces<NG>(pend, n_pend, w, p, lane);
  constexpr int kStageCap = C::kWarpBytes / kStagedPartialBytes;
  static_assert(kStageCap >= 2, "ring too small to stage partials");
#pragma unroll 1
  for (int i = 0; i < 2; ++i) {
    if (!((owe >> i) & 1u)) continue;
    __threadfence();
    merge_split_warp_staged<NG>(p.part_o, p.part_lse, pend[i].si, w, pend[i].b, pend[i].h0,
                                static_cast<__nv_bfloat16*>(p.out), p.lse, wbase, wsm, kStageCap, lane);
  }
}

template <int NG, int D, bool SP, bool F8 = false>
static cudaError_t launch_lsu(const DecodeParams& p, int num_ctas, cudaStream_t stream, bool pdl = false) {
  using C = LsuCfg<NG, D, F8>;
  static std::atomic<int> configured[kMaxDevices];
  const cudaError_t e = set_smem_limit_once(
      configured, reinterpret_cast<const void*>(gqa_decode_lsu_kernel<NG, D, SP, F8>), C::kSmemBytes);
  if (e != cudaSuccess) return e;
  if (!pdl) {
    gqa_decode_lsu_kernel<NG, D, SP, F8><<<num_ctas, C::kThreads, C::kSmemBytes, stream>>>(p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_ctas);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gqa_decode_lsu_kernel<NG, D, SP, F8>, p);
}

#define GQA_LSU_VARIANTS(X) X(4, 3) X(4, 4) X(4, 2) X(2, 3) X(2, 2) X(2, 5) X(1, 3) X(1, 2) X(1, 4) X(1, 6)

int lsu_smem_bytes(int ng, int stages) {
#define X(NG, D) \
  if (ng == NG && stages == D) return LsuCfg<NG, D>::kSmemBytes;
  GQA_LSU_VARIANTS(X)
#undef X
  return -1;
}

cudaError_t launch_decode_lsu(int ng, int stages, const DecodeParams& p, int num_ctas, cudaStream_t stream) {
#define X(NG, D) \
  if (ng == NG && stages == D) return launch_lsu<NG, D, false>(p, num_ctas, stream);
  GQA_LSU_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

// Selected-token mode: one variant, 4 KV heads per CTA and a 2-deep ring;
// pdl: launched as a programmatic dependent of the kernel before it.
cudaError_t launch_decode_lsu_sparse(const DecodeParams& p, int num_ctas, cudaStream_t stream, bool pdl) {
  return launch_lsu<4, 2, true>(p, num_ctas, stream, pdl);
}

// FP8-cache variants: 4 KV heads per CTA, 2, 3 or 4 stages.
#define GQA_LSU_F8_VARIANTS(X) X(4, 2) X(4, 3) X(4, 4)

int lsu_f8_smem_bytes(int stages) {
#define X(NG, D) \
  if (stages == D) return LsuCfg<NG, D, true>::kSmemBytes;
  GQA_LSU_F8_VARIANTS(X)
#undef X
  return -1;
}

cudaError_t launch_decode_lsu_f8(int stages, const DecodeParams& p, int num_ctas, cudaStream_t stream) {
#define X(NG, D) \
  if (stages == D) return launch_lsu<NG, D, false, true>(p, num_ctas, stream);
  GQA_LSU_F8_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace gqa
