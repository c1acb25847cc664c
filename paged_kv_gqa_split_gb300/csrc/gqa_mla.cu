// Dense MLA paged decode: one latent KV head, d_qk = 576 (512 "NoPE" + 64
// "RoPE" values per token), d_v = 512 (the NoPE part is also V), the dense
// decode of the flash_mla_with_kvcache page (docs.flagos.io, FlagGems;
// _dense_decode_dispatch): for every query row (query token i, head h) of
// sequence b, s_t = scale * q . kv_t over all 576 values, O = softmax(s) .
// kv[:, :512] (bf16) and lse = log sum exp(s) (natural log, stored
// [B][h_q][s_q]); a sequence with no cached token gives O = 0, lse = -inf.
//
// GB300 mapping. Two prep kernels turn cache_seqlens and the block table into
// the dense path's CSR form (kv_indptr, and one flat slot per cached token:
// block * page_size + offset, -1 when the table points outside the pool), so
// the dense path's two-tier split plan, walker, split records and tiers
// apply unchanged; the unit is one cached token for one group of 16 query
// rows. A decode CTA has 4 warps that share 16-token tiles of 1152-byte
// latent rows (gathered with 16-byte cp.async into a 3-deep ring, or 4-deep
// at two CTAs per SM, at a 1168-byte pitch) and compute:
//   S = Q K^T: each warp contracts 144 of the 576 dims (its Q fragments stay
//     in registers), the 4 partial 16 x 16 score tiles are summed through
//     shared memory, so every warp holds the full tile in the mma accumulator
//     layout, which is also P's A-fragment layout;
//   online softmax in base 2, identical in every warp;
//   O += P V: each warp owns 128 of the 512 output dims (V fragments by
//     ldmatrix.trans from the same latent rows).
// With double-buffered partial scores one CTA barrier per tile suffices: the
// softmax and P V of tile k share a straight-line block with the partial
// scores of tile k + 1.
// Pieces of a sequence cut across CTAs leave fp32 partials [16 rows][512]
// that gqa_mla_merge_kernel combines.
#include <cuda_runtime.h>

#include <cstdint>

#include "gqa_common.cuh"
#include "gqa_kernels.h"

namespace gqa {

constexpr int kMlaDqk = 576;
constexpr int kMlaDv = 512;
constexpr int kMlaRows = 16;                       // query rows per row group (one m16 tile)
constexpr int kMlaTile = 16;                       // tokens per stage
constexpr int kMlaWarps = 4;
constexpr int kMlaThreads = kMlaWarps * 32;
constexpr int kMlaRowBytes = kMlaDqk * 2;          // 1152
constexpr int kMlaPitch = kMlaRowBytes + 16;       // 1168: 73 16-byte groups, so 8 rows hit 8 bank groups
constexpr int kMlaChunks = kMlaRowBytes / 16;      // 72 16-byte copies per row
constexpr int kMlaKSteps = kMlaDqk / kMlaWarps / 16;  // 9 k-steps of 16 dims per warp (144 dims)
constexpr int kMlaVDims = kMlaDv / kMlaWarps;      // 128 output dims per warp
constexpr int kMlaIdsRing = 256;

// Shared memory of a CTA with ST ring stages.
template <int ST>
struct MlaLayout {
  static constexpr int kStageBytes = kMlaTile * kMlaPitch;                 // 18,688
  static constexpr int kHdrOff = ST * kStageBytes;                        // tile headers: 32 B per stage
  static constexpr int kValidOff = kHdrOff + ST * 32;                     // per stage: one byte per row (slot >= 0)
  static constexpr int kSpartOff = kValidOff + ST * kMlaTile;             // [2][warp][half][lane] float4 partial scores
  static constexpr int kIdsOff = kSpartOff + 2 * kMlaWarps * 32 * 8 * 4;  // per-warp slot rings
  static constexpr int kPlanOff = kIdsOff + kMlaWarps * kMlaIdsRing * 4;  // per-warp plan copies
  static constexpr int kSmemBytes = kPlanOff + kMlaWarps * 32;
};
// the compiled shapes: (3 stages, 3 CTAs per SM) and (4 stages, 2 CTAs per SM)
static_assert(3 * (MlaLayout<3>::kSmemBytes + 1024) <= 228 * 1024, "three 3-stage MLA CTAs per SM");
static_assert(2 * (MlaLayout<4>::kSmemBytes + 1024) <= 228 * 1024, "two 4-stage MLA CTAs per SM");

struct MlaSmemPlan {
  int64_t W1, q1, q2;
  int P1, unused;
};

// ------------------------------------------------------------------ prep
// kv_indptr = exclusive prefix sum of the lengths, each clamped to [0, cap]
// (cap = the block table's width * page_size: tokens past the table have no
// block, and the slot buffer holds batch * cap entries); one CTA.
// Exclusive prefix over the batch of f(b) into out[0..batch] (one CTA of 1024 threads).
template <typename F>
__device__ __forceinline__ void block_exclusive_scan(int batch, F f, int* __restrict__ out, int* warp_sum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (batch + 1023) / 1024;
  const int lo = tid * per, hi = min(batch, lo + per);
  int mine = 0;
  for (int i = lo; i < hi; ++i) mine += f(i);
  int x = mine;  // inclusive warp scan of the chunk sums
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int v = warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    warp_sum[lane] = v;
  }
  __syncthreads();
  int run = x - mine + (warp > 0 ? warp_sum[warp - 1] : 0);  // exclusive prefix of this chunk
  for (int i = lo; i < hi; ++i) {
    out[i] = run;
    run += f(i);
  }
  if (tid == 1023) out[batch] = warp_sum[31];
  __syncthreads();  // warp_sum is reused by the next scan
}

// kv_indptr = exclusive prefix sum of the lengths, each clamped to [0, cap]
// (cap = the block table's width * page_size: tokens past the table have no
// block, and the slot buffer holds batch * cap entries); one CTA. With bounds,
// also the tensor-memory kernel's cost-balanced tier-1 ranges: a sequence
// costs its tokens plus piece_cost (the work an extra piece adds to a CTA), the
// cost line of each row group is cut into P1 equal parts, and each cut is moved
// to the unit it falls on (the first token of a sequence when it falls in that
// sequence's piece cost).
__global__ void __launch_bounds__(1024) gqa_mla_scan_kernel(const int* __restrict__ seqlens, int batch, int cap,
                                                            int* __restrict__ indptr, int* __restrict__ cost_ptr,
                                                            int64_t* __restrict__ bounds, int P1, int HG,
                                                            int piece_cost) {
  __shared__ int warp_sum[32];
  pdl_launch_dependents();
  auto len = [&](int i) { return min(max(__ldg(seqlens + i), 0), cap); };
  block_exclusive_scan(batch, len, indptr, warp_sum);
  if (bounds == nullptr) return;
  block_exclusive_scan(batch, [&](int i) { const int n = len(i); return n > 0 ? n + piece_cost : 0; }, cost_ptr,
                       warp_sum);
  __threadfence_block();
  __syncthreads();
  const int64_t T = indptr[batch], Z = cost_ptr[batch];
  const int64_t Ztot = Z * HG;
  for (int c = threadIdx.x; c <= P1; c += blockDim.x) {
    int64_t u = T * HG;  // the last cut: every unit
    if (c < P1 && Z > 0) {
      const int64_t target = Ztot * c / P1;
      const int64_t hg = target / Z, tr = target - hg * Z;
      int lo = 0, hi = batch;  // the last b with cost_ptr[b] <= tr
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cost_ptr[mid] <= tr) lo = mid; else hi = mid;
      }
      const int n = indptr[lo + 1] - indptr[lo];
      const int64_t off = tr - cost_ptr[lo] - (n > 0 ? piece_cost : 0);
      u = hg * T + indptr[lo] + (off > 0 ? off : 0);
    } else if (c < P1) {
      u = 0;
    }
    bounds[c] = u;
  }
  __threadfence_block();
  __syncthreads();
  if (threadIdx.x == 0) {  // strictly increasing up to the unit count: no empty range but at the end
    int64_t prev = bounds[0];
    for (int c = 1; c < P1; ++c) {
      const int64_t v = min(max(bounds[c], prev + 1), T * HG);
      bounds[c] = v;
      prev = v;
    }
  }
}

// slots[indptr[b] + t] = block_table[b, t / page_size] * page_size + t % page_size, or -1.
// One CTA per (sequence, chunk of kMlaFillChunk tokens), kMlaFillPer independent
// lookups per thread.
constexpr int kMlaFillThreads = 256;
constexpr int kMlaFillPer = 4;
constexpr int kMlaFillChunk = kMlaFillThreads * kMlaFillPer;
__global__ void __launch_bounds__(kMlaFillThreads) gqa_mla_fill_kernel(const int* __restrict__ indptr,
                                                                      const int* __restrict__ block_table,
                                                                      int chunks, int width, int page_size,
                                                                      int num_blocks, int* __restrict__ slots) {
  pdl_launch_dependents();
  pdl_wait();  // indptr comes from the scan kernel
  const int b = blockIdx.x / chunks;
  const int t0 = (blockIdx.x - b * chunks) * kMlaFillChunk + threadIdx.x;
  const int base = __ldg(indptr + b), n = __ldg(indptr + b + 1) - base;
  if (t0 - static_cast<int>(threadIdx.x) >= n) return;
  const int* row = block_table + static_cast<int64_t>(b) * width;
  int page[kMlaFillPer];
#pragma unroll
  for (int k = 0; k < kMlaFillPer; ++k) {
    const int t = t0 + k * kMlaFillThreads, lp = t / page_size;
    page[k] = (t < n && lp < width) ? __ldg(row + lp) : -1;
  }
#pragma unroll
  for (int k = 0; k < kMlaFillPer; ++k) {
    const int t = t0 + k * kMlaFillThreads;
    if (t < n) slots[base + t] = (page[k] >= 0 && page[k] < num_blocks) ? page[k] * page_size + t % page_size : -1;
  }
}

// --------------------------------------------------------------- decode
__device__ __forceinline__ void mla_store_lse(const MlaParams& p, int b, int r, float lse2) {
  // natural log, [B][h_q][s_q]; r is the query row (i * h_q + h)
  p.lse[static_cast<int64_t>(b) * p.rows + (r % p.h_q) * p.s_q + r / p.h_q] = lse2 * 0.6931471805599453f;
}

__device__ __forceinline__ SeqSplit mla_seq_split(const MlaSmemPlan* sp, int64_t u_lo, int64_t u_hi) {
  Plan pl;
  pl.W1 = sp->W1;
  pl.q1 = sp->q1;
  pl.q2 = sp->q2;
  pl.P1 = sp->P1;
  return seq_split(pl, u_lo, u_hi);
}

__device__ __forceinline__ void mla_write_rec(int4* rec, int cta, unsigned long long epoch, int b, int hg,
                                              const SplitInfo& si) {
  // same record as the dense path, with up to 2^24 row groups
  rec[cta] = make_int4(static_cast<int>(static_cast<unsigned>(epoch)), b, si.first_cta, si.S);
  rec[gridDim.x + cta] = make_int4(hg, si.first_slot, 0, 0);
}

template <int ST, int CPS>
__global__ void __launch_bounds__(kMlaThreads, CPS) gqa_mla_decode_kernel(const MlaParams p) {
  using L = MlaLayout<ST>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const uint32_t sbase = smem_addr(smem);
  const int* ids = reinterpret_cast<const int*>(smem + L::kIdsOff + w * kMlaIdsRing * 4);
  const uint32_t ids_base = sbase + L::kIdsOff + w * kMlaIdsRing * 4;

  pdl_launch_dependents();
  pdl_wait();  // kv_indptr and the slots come from the prep kernels
  const uint8_t* __restrict__ kv = static_cast<const uint8_t*>(p.kv);
  const __nv_bfloat16* __restrict__ qg = static_cast<const __nv_bfloat16*>(p.q);
  const int B = p.batch;
  const int T = __ldg(p.kv_indptr + B);
  const int HG = p.rows / kMlaRows;
  MlaSmemPlan* splan = reinterpret_cast<MlaSmemPlan*>(smem + L::kPlanOff + w * 32);
  int64_t u0, u1;
  {
    const Plan pl = make_plan(static_cast<int64_t>(T) * HG, p.plan);
    u0 = pl.begin(blockIdx.x);
    u1 = pl.end(blockIdx.x);
    if (lane == 0) *splan = MlaSmemPlan{pl.W1, pl.q1, pl.q2, pl.P1, 0};
    __syncwarp();
  }

  // ------------------------------------------ walker (the same in every warp)
  int64_t u_next = u0;
  bool seg_open = false, walk_ok = true;
  int hg = 0, tt = 0, t_stop = 0;
  int p_hi = 0, p_flags = 0, pb = 0;
  SplitInfo p_si = {1, 0, 0};
  int wb = 0, win = 0, ib = 0;
  auto request_ids = [&](int pos) {
    cp_async_4(ids_base + (pos & (kMlaIdsRing - 1)) * 4, p.slots + min(pos, T - 1), pos < T ? 4u : 0u);
  };
  struct MTile {
    int b, cnt, flags, hg, tt;
    SplitInfo si;
  };
  auto next_tile = [&](MTile& tl) -> bool {
    while (walk_ok) {
      if (seg_open && tt < t_stop) {
        if (tt >= p_hi) {
          unsigned m;
          for (;;) {
            m = __ballot_sync(0xffffffffu, win <= tt);
            if (m != 0xffffffffu) break;
            wb += 31;
            win = load_indptr_window(p.kv_indptr, B, wb, lane);
          }
          if (m == 0) {
            if (lane == 0) atomicOr(p.err, kErrBadIndptr);
            walk_ok = false;
            break;
          }
          const int k = 31 - __clz(m);
          pb = wb + k;
          const int seq_lo = __shfl_sync(0xffffffffu, win, k);
          const int seq_hi = __shfl_sync(0xffffffffu, win, k + 1);
          p_hi = min(seq_hi, t_stop);
          p_flags = F_QLOAD | ((tt == seq_lo && p_hi == seq_hi) ? F_FINAL : 0) |
                    ((static_cast<int64_t>(hg) * T + tt != u0) ? F_SLOT1 : 0);
          const int64_t base_u = static_cast<int64_t>(hg) * T;
          const SeqSplit sp = mla_seq_split(splan, base_u + seq_lo, base_u + seq_hi);
          p_si.S = static_cast<int>(sp.last_cta - sp.first_cta + 1);
          p_si.first_cta = static_cast<int>(sp.first_cta);
          p_si.first_slot = sp.first_slot;
        }
        tl.cnt = min(kMlaTile, p_hi - tt);
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
      hg = static_cast<int>(u_next / T);
      tt = static_cast<int>(u_next - static_cast<int64_t>(hg) * T);
      t_stop = static_cast<int>(min(static_cast<int64_t>(T), u1 - static_cast<int64_t>(hg) * T));
      u_next = static_cast<int64_t>(hg) * T + t_stop;
      seg_open = true;
      p_hi = tt;
      ib = tt & ~31;
#pragma unroll
      for (int cc = 0; cc < kMlaIdsRing / 32; ++cc) request_ids(ib + 32 * cc + lane);
      cp_async_commit();
      wb = warp_find_seq(p.kv_indptr, B, tt, lane);
      if (wb >= 0) win = load_indptr_window(p.kv_indptr, B, wb, lane);
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

  // ------------------------------------------------------------- issue
  int issued = 0;
  bool more = true;
  auto issue = [&]() {
    const int stage = issued % ST;
    const uint32_t sb = sbase + stage * L::kStageBytes;
    MTile tl;
    if (more && next_tile(tl)) {
      while (tl.tt >= ib + 32) {
        request_ids(ib + kMlaIdsRing + lane);
        ib += 32;
      }
      // 16 rows x 72 chunks: 8 threads per row, each copying chunks (tid & 7) + 8 k
      {
        const int row = tid >> 3;
        const int slot = row < tl.cnt ? ids[(tl.tt + row) & (kMlaIdsRing - 1)] : -1;
        const bool valid = slot >= 0;
        const uint8_t* src = kv + static_cast<int64_t>(valid ? slot : 0) * kMlaRowBytes + (tid & 7) * 16;
        const uint32_t dst = sb + row * kMlaPitch + (tid & 7) * 16;
        // the latent rows stream through L2 first in line for eviction (measured: 152.6 -> 150.6 us
        // per call at 16 rows; within 1% slower when several row groups reread a row)
#pragma unroll
        for (int k = 0; k < kMlaChunks / 8; ++k)
          cp_async_16_evict_first(dst + k * 128, src + k * 128, valid ? 16u : 0u);
        // the row enters the softmax when it is one of the first cnt and its slot is valid
        if ((tid & 7) == 0)
          asm volatile("st.shared.u8 [%0], %1;" ::"r"(sbase + L::kValidOff + stage * kMlaTile + row),
                       "r"(valid ? 1 : 0) : "memory");
      }
      if (tid == 0) {
        const uint32_t hdr = sbase + L::kHdrOff + stage * 32;
        st_shared_v4(hdr, tl.b, tl.cnt, tl.flags, tl.hg);
        st_shared_v4(hdr + 16, tl.si.S, tl.si.first_cta, tl.si.first_slot, 0);
      }
      if ((tl.flags & F_QLOAD) && lane < 16) {  // the piece's Q rows toward L2 for its first tile
        const __nv_bfloat16* qr = qg + (static_cast<int64_t>(tl.b) * p.rows + tl.hg * kMlaRows) * kMlaDqk;
        for (int x = lane + 16 * w; x < kMlaRows * kMlaRowBytes / 128; x += 64) prefetch_l2(qr + x * 64);
      }
    } else if (more) {
      more = false;
      if (tid == 0) st_shared_v4(sbase + L::kHdrOff + stage * 32, 0, 0, F_DONE, 0);
    }
    cp_async_commit();
    ++issued;
  };

  // ----------------------------------------------------------- compute
  // One barrier per tile. Iteration k sums the partial scores of tile k
  // (written by the four warps in iteration k - 1) and runs its softmax; in
  // the same straight-line block this warp computes its partial scores of
  // tile k + 1, independent MMAs that fill the softmax's latency; then P.V of
  // tile k. The partial scores are double-buffered, so the barrier at the top
  // of iteration k + 1 is the only exchange point.
  uint32_t qa[kMlaKSteps][4];  // Q A-fragments: rows g / g+8, dims 144 w + 16 ks + {2c, 2c+8} (+1)
  float acc[kMlaVDims / 8][4];  // O rows g / g+8, dims 128 w + 8 nt + 2c (+1)
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int nt = 0; nt < kMlaVDims / 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  // per-lane ldmatrix addresses inside a stage
  const int mk = lane >> 3;
  const uint32_t k_lane = ((mk >> 1) * 8 + (lane & 7)) * kMlaPitch + (w * 144 + (mk & 1) * 8) * 2;
  const uint32_t v_lane = ((mk & 1) * 8 + (lane & 7)) * kMlaPitch + (w * kMlaVDims + (mk >> 1) * 8) * 2;
  float4* my = reinterpret_cast<float4*>(smem + L::kSpartOff) + w * 64 + lane;  // [buf][warp][half][lane]
  const float4* spart = reinterpret_cast<const float4*>(smem + L::kSpartOff) + lane;
  constexpr int kSpartBuf = kMlaWarps * 64;  // float4 per buffer
  auto load_q = [&](int qb, int qhg) {
    const __nv_bfloat16* qr = qg + (static_cast<int64_t>(qb) * p.rows + qhg * kMlaRows) * kMlaDqk;
#pragma unroll
    for (int ks = 0; ks < kMlaKSteps; ++ks) {
      const int d = w * 144 + ks * 16 + 2 * c;
      qa[ks][0] = __ldg(reinterpret_cast<const uint32_t*>(qr + g * kMlaDqk + d));
      qa[ks][1] = __ldg(reinterpret_cast<const uint32_t*>(qr + (g + 8) * kMlaDqk + d));
      qa[ks][2] = __ldg(reinterpret_cast<const uint32_t*>(qr + g * kMlaDqk + d + 8));
      qa[ks][3] = __ldg(reinterpret_cast<const uint32_t*>(qr + (g + 8) * kMlaDqk + d + 8));
    }
  };
  // this warp's partial scores (its 144 dims) of the tile in stage sb, into buffer buf:
  // tokens 0-7 (my[0]) and 8-15 (my[32]), two accumulation chains each
  auto partial_scores = [&](uint32_t sb, int buf) {
    float sla[4] = {0.f, 0.f, 0.f, 0.f}, slb[4] = {0.f, 0.f, 0.f, 0.f};
    float sha[4] = {0.f, 0.f, 0.f, 0.f}, shb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < kMlaKSteps; ++ks) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(sb + k_lane + ks * 32, b0, b1, b2, b3);
      mma_bf16_16816((ks & 1) ? slb : sla, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
      mma_bf16_16816((ks & 1) ? shb : sha, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
    }
    my[buf * kSpartBuf] = make_float4(sla[0] + slb[0], sla[1] + slb[1], sla[2] + slb[2], sla[3] + slb[3]);
    my[buf * kSpartBuf + 32] = make_float4(sha[0] + shb[0], sha[1] + shb[1], sha[2] + shb[2], sha[3] + shb[3]);
  };

#pragma unroll 1
  for (int i = 0; i < ST - 1; ++i) issue();
  cp_async_wait<ST - 2>();  // this thread's copies of tile 0 have landed
  __syncthreads();
  int hb, cnt, flags, thg;  // header of tile k (stage k % ST)
  ld_shared_v4(sbase + L::kHdrOff, hb, cnt, flags, thg);
  if (!(flags & F_DONE)) {
    load_q(hb, thg);  // the first tile opens a piece
    partial_scores(sbase, 0);
#pragma unroll 1
    for (int k = 0;; ++k) {
      cp_async_wait<ST - 3>();  // this thread's copies of tile k + 1 have landed (tiles up to k + ST - 2 were issued)
      __syncthreads();     // everyone's have; tile k's partial scores are complete; tile k - 1's stage is free
      issue();             // tile k + 2 into that stage
      const int st0 = k % ST, st1 = (k + 1) % ST;
      const uint32_t sb0 = sbase + st0 * L::kStageBytes, sb1 = sbase + st1 * L::kStageBytes;
      int hb1, cnt1, flags1, thg1;
      ld_shared_v4(sbase + L::kHdrOff + st1 * 32, hb1, cnt1, flags1, thg1);
      const bool done1 = flags1 & F_DONE;
      if (!done1 && (flags1 & F_QLOAD)) load_q(hb1, thg1);  // tile k + 1 opens a piece (tile k no longer needs Q)
      // tile k's scores: sum of the four warps' partials
      float s[8];
      {
        const float4* sp = spart + (k & 1) * kSpartBuf;
        const float4 x0 = sp[0], y0 = sp[32], x1 = sp[64], y1 = sp[96], x2 = sp[128], y2 = sp[160], x3 = sp[192],
                     y3 = sp[224];
        s[0] = (x0.x + x1.x) + (x2.x + x3.x); s[1] = (x0.y + x1.y) + (x2.y + x3.y);
        s[2] = (x0.z + x1.z) + (x2.z + x3.z); s[3] = (x0.w + x1.w) + (x2.w + x3.w);
        s[4] = (y0.x + y1.x) + (y2.x + y3.x); s[5] = (y0.y + y1.y) + (y2.y + y3.y);
        s[6] = (y0.z + y1.z) + (y2.z + y3.z); s[7] = (y0.w + y1.w) + (y2.w + y3.w);
      }
      // tile k + 1's partial scores (from stale stage data when it is the end marker: never used)
      partial_scores(sb1, (k + 1) & 1);
      // validity of this lane's tokens 2c, 2c + 1, 8 + 2c, 9 + 2c of tile k (one byte per row)
      const uint8_t* vrow = smem + L::kValidOff + st0 * kMlaTile;
      const unsigned um = (vrow[2 * c] ? 1u : 0u) << (2 * c) | (vrow[2 * c + 1] ? 1u : 0u) << (2 * c + 1) |
                          (vrow[8 + 2 * c] ? 1u : 0u) << (8 + 2 * c) | (vrow[9 + 2 * c] ? 1u : 0u) << (9 + 2 * c);
      // scale, mask, online softmax in base 2 (rows g: s0,1,4,5; g+8: s2,3,6,7)
      const int tk[4] = {2 * c, 2 * c + 1, 8 + 2 * c, 9 + 2 * c};
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const bool ok = (um >> tk[jj]) & 1u;
        const int ia = jj < 2 ? jj : 2 + jj;  // row g entry of token tk[jj]
        const int ib2 = ia + 2;               // row g + 8 entry
        s[ia] = ok ? s[ia] * p.scale_log2 : -INFINITY;
        s[ib2] = ok ? s[ib2] * p.scale_log2 : -INFINITY;
      }
      float mx0 = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[4], s[5]));
      float mx1 = fmaxf(fmaxf(s[2], s[3]), fmaxf(s[6], s[7]));
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float sh0 = mn0 == -INFINITY ? 0.f : mn0, sh1 = mn1 == -INFINITY ? 0.f : mn1;
      const float a0 = ex2(m0 - sh0), a1 = ex2(m1 - sh1);
      m0 = mn0;
      m1 = mn1;
      float pr[8];
      pr[0] = ex2(s[0] - sh0); pr[1] = ex2(s[1] - sh0); pr[4] = ex2(s[4] - sh0); pr[5] = ex2(s[5] - sh0);
      pr[2] = ex2(s[2] - sh1); pr[3] = ex2(s[3] - sh1); pr[6] = ex2(s[6] - sh1); pr[7] = ex2(s[7] - sh1);
      l0 = l0 * a0 + (pr[0] + pr[1] + pr[4] + pr[5]);
      l1 = l1 * a1 + (pr[2] + pr[3] + pr[6] + pr[7]);
      const uint32_t pa0 = pack_bf16(pr[0], pr[1]), pa1 = pack_bf16(pr[2], pr[3]);
      const uint32_t pa2 = pack_bf16(pr[4], pr[5]), pa3 = pack_bf16(pr[6], pr[7]);
      if (!__all_sync(0xffffffffu, a0 == 1.f && a1 == 1.f)) {  // some row's max moved: rescale O
#pragma unroll
        for (int nt = 0; nt < kMlaVDims / 8; ++nt) {
          acc[nt][0] *= a0; acc[nt][1] *= a0; acc[nt][2] *= a1; acc[nt][3] *= a1;
        }
      }
#pragma unroll
      for (int np = 0; np < kMlaVDims / 16; ++np) {  // O += P V of tile k (this warp's 128 dims)
        uint32_t v0, v1, v2, v3;
        ldsm_x4_trans(sb0 + v_lane + np * 32, v0, v1, v2, v3);
        mma_bf16_16816(acc[2 * np], pa0, pa1, pa2, pa3, v0, v1);
        mma_bf16_16816(acc[2 * np + 1], pa0, pa1, pa2, pa3, v2, v3);
      }
      if (flags & F_END) {  // tile k ends its piece: write O and LSE
        SplitInfo si;
        int dummy;
        ld_shared_v4(sbase + L::kHdrOff + st0 * 32 + 16, si.S, si.first_cta, si.first_slot, dummy);
        float lt0 = l0, lt1 = l1;
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
          lt0 += __shfl_xor_sync(0xffffffffu, lt0, o);
          lt1 += __shfl_xor_sync(0xffffffffu, lt1, o);
        }
        const float i0 = lt0 > 0.f ? 1.f / lt0 : 0.f, i1 = lt1 > 0.f ? 1.f / lt1 : 0.f;
        const float lse0 = lt0 > 0.f ? m0 + log2f(lt0) : -INFINITY;  // base 2
        const float lse1 = lt1 > 0.f ? m1 + log2f(lt1) : -INFINITY;
        const int r0 = thg * kMlaRows + g, r1 = r0 + 8;  // query rows (i * h_q + h) of sequence hb
        if (flags & F_FINAL) {
          __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(hb) * p.rows * kMlaDv;
#pragma unroll
          for (int nt = 0; nt < kMlaVDims / 8; ++nt) {
            const int d = w * kMlaVDims + nt * 8 + 2 * c;
            *reinterpret_cast<uint32_t*>(ob + static_cast<int64_t>(r0) * kMlaDv + d) = pack_bf16(acc[nt][0] * i0, acc[nt][1] * i0);
            *reinterpret_cast<uint32_t*>(ob + static_cast<int64_t>(r1) * kMlaDv + d) = pack_bf16(acc[nt][2] * i1, acc[nt][3] * i1);
          }
          if (w == 0 && c == 0 && p.lse != nullptr) {
            mla_store_lse(p, hb, r0, lse0);
            mla_store_lse(p, hb, r1, lse1);
          }
        } else {
          const int64_t sid = slot_id(blockIdx.x, (flags & F_SLOT1) ? 1 : 0);
          float* po = p.part_o + sid * (kMlaRows * kMlaDv);
#pragma unroll
          for (int nt = 0; nt < kMlaVDims / 8; ++nt) {
            const int d = w * kMlaVDims + nt * 8 + 2 * c;
            *reinterpret_cast<float2*>(po + g * kMlaDv + d) = make_float2(acc[nt][0] * i0, acc[nt][1] * i0);
            *reinterpret_cast<float2*>(po + (g + 8) * kMlaDv + d) = make_float2(acc[nt][2] * i1, acc[nt][3] * i1);
          }
          if (w == 0 && c == 0) {
            p.part_lse[sid * kMlaRows + g] = lse0;
            p.part_lse[sid * kMlaRows + g + 8] = lse1;
          }
        }
      }
      if (done1) break;
      if (flags1 & F_QLOAD) {  // tile k + 1 opens a piece
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < kMlaVDims / 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
      }
      hb = hb1;
      cnt = cnt1;
      flags = flags1;
      thg = thg1;
    }
  }
  (void)cnt;
  cp_async_wait<0>();
  if (tid == 0 && u0 < u1 && walk_ok) mla_write_rec(p.split_rec, blockIdx.x, p.epoch, pb, hg, p_si);
}

// ---------------------------------------------------------------- merge
// One CTA per boundary between decode CTAs j and j + 1, as for the dense
// path: it finds the sequence cut there from CTA j's record and, being rank
// r of its S - 1 boundary CTAs, merges a share of the 512 output dims of the
// piece's rows (p.piece_rows: 16 for the mma.sync kernel, 16 or 64 for the
// tensor-memory kernel; one CTA per 16 rows of a piece) over all S pieces. While S * rows fits the weight
// table, the weight of every (piece, row), 2^(lse_s - max) / sum, is
// computed once into shared memory and each output element is then one
// weighted sum of independent loads; longer chains take a running-max loop.
// It also writes the empty sequences.
constexpr int kMlaMergeThreads = 256;
constexpr int kMlaMergeWeights = 1024;  // (piece, row) weights in the table: 64 pieces of 16 rows, 16 of 64
constexpr int kMlaMergeBatch = 4;  // float4 columns per thread per pass

__global__ void __launch_bounds__(kMlaMergeThreads) gqa_mla_merge_kernel(const MlaParams p) {
  __shared__ float wsh[kMlaMergeWeights];  // [piece][row]
  const int R = p.piece_rows;                // rows per piece: 16 or 64
  const int G = R / kMlaRows;                // CTAs per boundary, each merging 16 rows of the piece
  const int tid = threadIdx.x;
  const int B = p.batch;
  const int j = blockIdx.x / G, row0 = (blockIdx.x - j * G) * kMlaRows;
  const bool boundary = j + 1 < p.plan.tier1_ctas + p.plan.tier2_ctas;
  const int T = __ldg(p.kv_indptr + B);
  pdl_wait();
  const int4 rec0 = boundary ? __ldcg(p.split_rec + j) : make_int4(0, 0, 0, 0);
  const int4 rec1 = boundary ? __ldcg(p.split_rec + (p.plan.tier1_ctas + p.plan.tier2_ctas) + j)
                             : make_int4(0, 0, 0, 0);
  for (int b = blockIdx.x; b < B; b += gridDim.x) {  // empty sequences: O = 0, LSE = -inf
    if (__ldg(p.kv_indptr + b) == __ldg(p.kv_indptr + b + 1)) {
      uint4* ob = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(b) * p.rows * kMlaDv);
      for (int i = tid; i < p.rows * kMlaDv * 2 / 16; i += kMlaMergeThreads) ob[i] = make_uint4(0, 0, 0, 0);
      if (p.lse != nullptr)
        for (int i = tid; i < p.rows; i += kMlaMergeThreads) p.lse[static_cast<int64_t>(b) * p.rows + i] = -INFINITY;
    }
  }
  const int HG = p.rows / R;
  const Plan pl = make_plan(static_cast<int64_t>(T) * HG, p.plan);
  if (!boundary || (p.bounds != nullptr ? p.bounds[j + 1] : pl.begin(j + 1)) >= pl.W) return;
  if (static_cast<unsigned>(rec0.x) != static_cast<unsigned>(p.epoch)) return;
  const int b = rec0.y, S = rec0.w, hg = rec1.x;
  const int first_cta = rec0.z, first_slot = rec1.y;
  if (b < 0 || b >= B || hg < 0 || hg >= HG || S < 2 || first_cta > j || first_cta + S - 1 <= j) return;
  const int rank = j - first_cta, nranks = S - 1;
  const int cols = (kMlaDv / 4 + nranks - 1) / nranks;  // float4 columns per rank
  const int c_lo = rank * cols, c_hi = min(kMlaDv / 4, c_lo + cols);
  if (c_lo >= c_hi) return;
  const int ncol = c_hi - c_lo, items = kMlaRows * ncol;
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.out) + (static_cast<int64_t>(b) * p.rows + hg * R + row0) * kMlaDv;
  auto part = [&](int s) {
    return reinterpret_cast<const float4*>(p.part_o + (slot_id(first_cta + s, s == 0 ? first_slot : 0) * R + row0) *
                                                          static_cast<int64_t>(kMlaDv));
  };
  constexpr int W = kMlaRows;  // rows of this CTA
  if (S * W <= kMlaMergeWeights) {
    for (int i = tid; i < S * W; i += kMlaMergeThreads) {
      const int s = i / W, r = i - s * W;
      wsh[s * W + r] = __ldcg(p.part_lse + slot_id(first_cta + s, s == 0 ? first_slot : 0) * R + row0 + r);
    }
    __syncthreads();
    if (tid < W) {  // weights of row tid; pieces with no token (lse = -inf) weigh 0
      float m = -INFINITY;
      for (int s = 0; s < S; ++s) m = fmaxf(m, wsh[s * W + tid]);
      float den = 0.f;
      if (m != -INFINITY)
        for (int s = 0; s < S; ++s) den += ex2(wsh[s * W + tid] - m);
      const float inv = den > 0.f ? 1.f / den : 0.f;
      for (int s = 0; s < S; ++s) wsh[s * W + tid] = m == -INFINITY ? 0.f : ex2(wsh[s * W + tid] - m) * inv;
      if (rank == 0 && p.lse != nullptr) mla_store_lse(p, b, hg * R + row0 + tid, den > 0.f ? m + log2f(den) : -INFINITY);
    }
    __syncthreads();
    for (int i0 = tid; i0 < items; i0 += kMlaMergeThreads * kMlaMergeBatch) {
      float4 a[kMlaMergeBatch];
      int rr[kMlaMergeBatch], cc[kMlaMergeBatch];
#pragma unroll
      for (int k = 0; k < kMlaMergeBatch; ++k) {
        const int it = min(i0 + k * kMlaMergeThreads, items - 1);  // past the end: repeat the last item, unstored
        rr[k] = it / ncol;
        cc[k] = c_lo + (it - rr[k] * ncol);
        a[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll 2
      for (int s = 0; s < S; ++s) {
        const float4* src = part(s);
        float4 o[kMlaMergeBatch];
#pragma unroll
        for (int k = 0; k < kMlaMergeBatch; ++k) o[k] = __ldcg(src + rr[k] * (kMlaDv / 4) + cc[k]);
#pragma unroll
        for (int k = 0; k < kMlaMergeBatch; ++k) {
          const float w = wsh[s * W + rr[k]];
          a[k].x += w * o[k].x;
          a[k].y += w * o[k].y;
          a[k].z += w * o[k].z;
          a[k].w += w * o[k].w;
        }
      }
#pragma unroll
      for (int k = 0; k < kMlaMergeBatch; ++k)
        if (i0 + k * kMlaMergeThreads < items)
          *reinterpret_cast<uint2*>(ob + rr[k] * kMlaDv + cc[k] * 4) =
              make_uint2(pack_bf16(a[k].x, a[k].y), pack_bf16(a[k].z, a[k].w));
    }
    return;
  }
  for (int it = tid; it < items; it += kMlaMergeThreads) {  // long chains: running max per element
    const int r = it / ncol, col = c_lo + (it - r * ncol);
    float m = -INFINITY, den = 0.f, a[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < S; ++s) {
      const float l = __ldcg(p.part_lse + slot_id(first_cta + s, s == 0 ? first_slot : 0) * R + row0 + r);
      const float4 o = __ldcg(part(s) + r * (kMlaDv / 4) + col);
      const float mn = fmaxf(m, l);
      if (mn == -INFINITY) continue;
      const float sc = ex2(m - mn), wt = ex2(l - mn);
      den = den * sc + wt;
      a[0] = a[0] * sc + wt * o.x;
      a[1] = a[1] * sc + wt * o.y;
      a[2] = a[2] * sc + wt * o.z;
      a[3] = a[3] * sc + wt * o.w;
      m = mn;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    *reinterpret_cast<uint2*>(ob + r * kMlaDv + col * 4) =
        make_uint2(pack_bf16(a[0] * inv, a[1] * inv), pack_bf16(a[2] * inv, a[3] * inv));
    if (col == 0 && p.lse != nullptr) mla_store_lse(p, b, hg * R + row0 + r, den > 0.f ? m + log2f(den) : -INFINITY);
  }
}

// --------------------------------------------------------------- launch
int mla_smem_bytes(int stages) { return stages == 3 ? MlaLayout<3>::kSmemBytes : MlaLayout<4>::kSmemBytes; }
int mla_ctas_per_sm(int kind) { return kind == kMlaKernelTensorMemory ? 1 : (kind == kMlaKernelMma4 ? 2 : 3); }

static cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_mla(const MlaParams& p, const int* cache_seqlens, int kind, const MlaTcMaps* maps,
                       cudaStream_t stream) {
  int width = p.width, page_size = p.page_size, num_blocks = p.num_blocks;
  const int cap = width * page_size;
  gqa_mla_scan_kernel<<<1, 1024, 0, stream>>>(cache_seqlens, p.batch, cap, p.kv_indptr_mut, p.cost_ptr, p.bounds,
                                              p.plan.tier1_ctas, p.rows / p.piece_rows, p.piece_cost);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int ctas = p.plan.tier1_ctas + p.plan.tier2_ctas;
  MlaParams pc = p;
  void* args[] = {&pc};
  if (kind == kMlaKernelTensorMemory) {  // reads the block table itself: no slot list
    e = launch_mla_tc_decode(p, *maps, ctas, stream);
  } else {
    {  // one CTA per (sequence, chunk); batch * cap < 2^31 bounds the grid
      int chunks = (cap + kMlaFillChunk - 1) / kMlaFillChunk;
      if (chunks < 1) chunks = 1;
      const int* ip = p.kv_indptr;
      const int* bt = p.block_table;
      int* sl = p.slots_mut;
      void* fargs[] = {&ip, &bt, &chunks, &width, &page_size, &num_blocks, &sl};
      e = launch_pdl(reinterpret_cast<const void*>(gqa_mla_fill_kernel), dim3(p.batch * chunks),
                     dim3(kMlaFillThreads), 0, stream, fargs);
      if (e != cudaSuccess) return e;
    }
    const int stages = kind == kMlaKernelMma4 ? 4 : 3;
    const void* fn = stages == 3 ? reinterpret_cast<const void*>(gqa_mla_decode_kernel<3, 3>)
                                  : reinterpret_cast<const void*>(gqa_mla_decode_kernel<4, 2>);
    const int smem = mla_smem_bytes(stages);
    static std::atomic<int> configured[2][kMaxDevices];
    e = set_smem_limit_once(configured[stages == 3 ? 0 : 1], fn, smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(fn, dim3(ctas), dim3(kMlaThreads), smem, stream, args);
  }
  if (e != cudaSuccess) return e;
  const int per_boundary = p.piece_rows / kMlaRows;  // one merge CTA per 16 rows of a piece
  return launch_pdl(reinterpret_cast<const void*>(gqa_mla_merge_kernel), dim3((ctas > 1 ? ctas - 1 : 1) * per_boundary),
                    dim3(kMlaMergeThreads), 0, stream, args);
}

}  // namespace gqa
