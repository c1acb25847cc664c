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
//
// Two launch modes share this kernel:
//   * static grid (the default): P1 + P2 CTAs, one per virtual CTA of the
//     plan, followed by the LSE merge kernel (gqa_merge.cu), which reads the
//     split records written here;
//   * one wave (p.inline_merge, opt-in): the grid is the P1 tier-1 CTAs, all
//     resident at once (a cooperative launch guarantees it). When a warp has
//     walked its tier-1 range it takes tier-2 ranges (virtual CTAs P1 .. P1 +
//     P2 - 1 of the same plan) from a per-warp-index counter, so the SMs that
//     stream faster take more of the tail without a second wave of CTAs, and
//     publishes a record of where each range's last sequence is cut. After its
//     stream each warp counts the arrival of its split pieces and merges its
//     share of the sequences cut at boundaries c, c + P1, ... (waiting, bounded,
//     for their pieces), staging the partials in its drained ring. Empty
//     sequences are written here too, so a call is this one kernel. Its stream
//     is as fast as the static grid's, but one warp per merge share makes the
//     merge end later than the merge kernel does.
#include <cuda_runtime.h>

#include "gqa_common.cuh"
#include "gqa_kernels.h"

namespace gqa {

// Per-warp shared memory. bf16 cache (F8 = false): each stage holds the K and
// V head rows of one tile at a 272-byte pitch, ready for ldmatrix. FP8 cache
// (F8 = true): each stage holds the tile's 128-byte e4m3 head rows of K (at a
// 192-byte pitch: the 128-bit row reads of attend_subtile_f8 then hit 8
// distinct bank groups) and of V (at a 144-byte pitch, for ldmatrix), plus
// their per-token scales. TT: tokens per stage (16, one mma sub-tile; the FP8
// cache also has a 32-token form).
template <int NG, int D, bool F8 = false, int TT = 16>
struct LsuCfg {
  static constexpr int kHG = kKvHeads / NG;           // head groups on the unit line
  static constexpr int kTile = TT;                    // tokens per stage
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
  // one-wave mode: the ticket ids of the warp's split pieces (at most two per range)
  static constexpr int kArrOff = kPlanOff + 48;
  static constexpr int kWarpBytes = kArrOff + 2 * kMaxWarpRanges * 4;
  // the stage ring and the page-id ring, free once the stream has drained:
  // the in-kernel merge stages partials there
  static constexpr int kStagingBytes = kPlanOff;
  static constexpr int kThreads = NG * 32;
  static constexpr int kSmemBytes = NG * kWarpBytes;
  static_assert(D >= 2, "at least double buffering");
  static_assert(kStageBytes % 16 == 0 && kWarpBytes % 16 == 0, "16-byte aligned stages");
  static_assert(kSmemBytes <= 227 * 1024, "ring exceeds shared memory");
  static_assert(TT == 16 || (F8 && TT == 32), "32-token stages exist for the FP8 cache only");
};

// What the walker needs of the plan when a piece starts (where the piece's
// sequence is cut), kept in shared memory so that it holds no registers in
// the streaming loop.
struct SmemPlan {
  int64_t W1, q1, q2;
  int P1;
  // one-wave mode (kept here, not in registers, since they change only between
  // ranges): the virtual CTA whose range the warp walks, the ranges walked so
  // far; lane 0's count of split pieces noted
  int vcta, n_ranges, n_arr, unused0, unused1;
};
static_assert(sizeof(SmemPlan) == 48, "plan block layout");

__device__ __forceinline__ SeqSplit seq_split_smem(const SmemPlan* sp, int64_t u_lo, int64_t u_hi) {
  Plan pl;
  pl.W1 = sp->W1;
  pl.q1 = sp->q1;
  pl.q2 = sp->q2;
  pl.P1 = sp->P1;
  return seq_split(pl, u_lo, u_hi);
}

struct Tile {
  int b, cnt, flags, hg, tt, vcta;
  SplitInfo si;
};

// Zeros for O and -inf for the LSE of empty sequence b (the early exit of
// the kernelindex.com page's kernel), written by one warp.
__device__ __forceinline__ void write_empty_seq(const DecodeParams& p, int b, int lane) {
  uint4* ob = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(b) * kQoHeads * kHeadDim);
#pragma unroll
  for (int i = 0; i < kQoHeads * kHeadDim * 2 / 16 / 32; ++i) ob[i * 32 + lane] = make_uint4(0, 0, 0, 0);
  if (p.lse != nullptr) p.lse[static_cast<int64_t>(b) * kQoHeads + lane] = -INFINITY;
}

// Issues the copies of pieces s0 .. s0 + n - 1 of a split sequence for one
// merge share into shared memory at `stage`: per piece its 8 LSEs (32 B),
// then O rows d_lo .. d_lo + nd - 1 (8 heads, 32 B each), `per` bytes in all.
template <int NG>
__device__ __forceinline__ void issue_partials(const DecodeParams& p, int first_cta, int first_slot, int w, int d_lo,
                                               int nd, int s0, int n, int per, uint32_t stage, int lane) {
  const int chunks = 2 + 2 * nd;  // 16-byte chunks per piece
  for (int c = lane; c < n * chunks; c += 32) {
    const int i = c / chunks, k = c - i * chunks;
    const int s = s0 + i;
    const int64_t sid = slot_id(first_cta + s, s == 0 ? first_slot : 0);
    const float* src = k < 2 ? p.part_lse + (sid * NG + w) * kGroup + 4 * k
                             : p.part_o + ((sid * NG + w) * kHeadDim + d_lo) * kGroup + 4 * (k - 2);
    cp_async_16(stage + i * per + 16 * k, src, 16u);
  }
}

__device__ __forceinline__ void staged_wait() {
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();
}

template <int NG>
__device__ __forceinline__ void stage_partials(const DecodeParams& p, int first_cta, int first_slot, int w, int d_lo,
                                               int nd, int s0, int n, int per, uint32_t stage, int lane) {
  issue_partials<NG>(p, first_cta, first_slot, w, d_lo, nd, s0, n, per, stage, lane);
  staged_wait();
}

// Running LSE-weighted fold of one staged piece into (m, den, acc) for head q:
// m = max LSE so far, den = sum 2^(LSE_i - m), acc = sum 2^(LSE_i - m) O_i.
// A piece with LSE -inf (no token) adds nothing.
__device__ __forceinline__ bool fold_weights(float& m, float& den, float lse_i, float& sc, float& wt) {
  const float mn = fmaxf(m, lse_i);
  if (mn == -INFINITY) return false;
  sc = ex2(m - mn);
  wt = ex2(lse_i - mn);
  den = den * sc + wt;
  m = mn;
  return true;
}

// Running LSE-weighted fold of four heads: (m, den, acc) take piece i's LSEs
// `l` and O values `o` (one dim) with the weights 2^(LSE_i - m).
struct Fold4 {
  float m[4], den[4], acc[4];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m[j] = -INFINITY;
      den[j] = 0.f;
      acc[j] = 0.f;
    }
  }
  __device__ __forceinline__ void add(const float4& l, const float4& o) {
    const float lv[4] = {l.x, l.y, l.z, l.w}, ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float mn = fmaxf(m[j], lv[j]);
      if (mn == -INFINITY) continue;  // nothing yet and a piece with no token
      const float sc = ex2(m[j] - mn), wt = ex2(lv[j] - mn);
      den[j] = den[j] * sc + wt;
      acc[j] = acc[j] * sc + wt * ov[j];
      m[j] = mn;
    }
  }
  // fold in the state of the lane `o` apart (xor shuffle)
  __device__ __forceinline__ void merge_lane(int o) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m[j], o);
      const float d2 = __shfl_xor_sync(0xffffffffu, den[j], o);
      const float a2 = __shfl_xor_sync(0xffffffffu, acc[j], o);
      const float mn = fmaxf(m[j], m2);
      if (mn == -INFINITY) continue;
      const float s1 = ex2(m[j] - mn), s2 = ex2(m2 - mn);
      den[j] = den[j] * s1 + d2 * s2;
      acc[j] = acc[j] * s1 + a2 * s2;
      m[j] = mn;
    }
  }
};

// Merge share: the pieces 0 .. S - 1 of a split sequence, for query heads
// h0 .. h0 + 7 and dims [d_lo, d_lo + nd). Lane (r = lane >> 1, hh = lane & 1)
// takes heads h0 + 4 hh .. + 3 with 16-byte reads of the staged rows, four
// independent running folds. With at most two dims (the shares of a sequence
// cut into more pieces than there are dims) row r takes pieces r, r + 16, ...
// of every dim and the 16 rows are folded together by xor shuffles; otherwise
// (then S <= 64 and one batch stages every piece) row r takes dim r (+ 16 per
// pass) over all pieces. Few warps run this at once, so it is written for
// short dependency chains rather than for throughput.
template <int NG>
__device__ __forceinline__ void merge_share(const DecodeParams& p, int b, int h0, int first_cta, int first_slot, int S,
                                            int w, int d_lo, int nd, uint32_t stage, int stage_bytes, bool staged,
                                            int lane) {
  const int per = 32 + 32 * nd;
  const int cap = stage_bytes / per;
  const int r = lane >> 1, hh = lane & 1;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + (static_cast<int64_t>(b) * kQoHeads + h0 + 4 * hh) * kHeadDim;
  if (nd <= 2) {
    Fold4 f0, f1;  // dims d_lo and d_lo + 1
    f0.init();
    f1.init();
#pragma unroll 1
    for (int s0 = 0; s0 < S; s0 += cap) {
      const int n = min(cap, S - s0);
      if (!staged) stage_partials<NG>(p, first_cta, first_slot, w, d_lo, nd, s0, n, per, stage, lane);
#pragma unroll 1
      for (int i = r; i < n; i += 16) {
        const uint32_t row = stage + i * per + 16 * hh;
        float4 l, o;
        ld_shared_u4(row, reinterpret_cast<uint32_t&>(l.x), reinterpret_cast<uint32_t&>(l.y),
                     reinterpret_cast<uint32_t&>(l.z), reinterpret_cast<uint32_t&>(l.w));
        ld_shared_u4(row + 32, reinterpret_cast<uint32_t&>(o.x), reinterpret_cast<uint32_t&>(o.y),
                     reinterpret_cast<uint32_t&>(o.z), reinterpret_cast<uint32_t&>(o.w));
        f0.add(l, o);
        if (nd > 1) {
          ld_shared_u4(row + 64, reinterpret_cast<uint32_t&>(o.x), reinterpret_cast<uint32_t&>(o.y),
                       reinterpret_cast<uint32_t&>(o.z), reinterpret_cast<uint32_t&>(o.w));
          f1.add(l, o);
        }
      }
      __syncwarp();  // the staging area is refilled by the next batch
    }
#pragma unroll 1
    for (int o = 2; o < 32; o <<= 1) {
      f0.merge_lane(o);
      f1.merge_lane(o);
    }
    if (r < nd) {
      const Fold4& f = r == 0 ? f0 : f1;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        out[j * kHeadDim + d_lo + r] = __float2bfloat16_rn(f.den[j] > 0.f ? f.acc[j] / f.den[j] : 0.f);
    }
    if (r == 0 && d_lo == 0 && p.lse != nullptr) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        p.lse[static_cast<int64_t>(b) * kQoHeads + h0 + 4 * hh + j] = f0.den[j] > 0.f ? f0.m[j] + log2f(f0.den[j])
                                                                                    : -INFINITY;
    }
    return;
  }
  if (!staged) stage_partials<NG>(p, first_cta, first_slot, w, d_lo, nd, 0, S, per, stage, lane);  // S <= cap here
#pragma unroll 1
  for (int d = r; d < nd + (nd % 16 ? 16 - nd % 16 : 0); d += 16) {  // every lane runs every pass
    Fold4 f;
    f.init();
    const int dd = min(d, nd - 1);  // lanes past nd fold a real dim and write nothing
#pragma unroll 2
    for (int i = 0; i < S; ++i) {
      const uint32_t row = stage + i * per + 16 * hh;
      float4 l, o;
      ld_shared_u4(row, reinterpret_cast<uint32_t&>(l.x), reinterpret_cast<uint32_t&>(l.y),
                   reinterpret_cast<uint32_t&>(l.z), reinterpret_cast<uint32_t&>(l.w));
      ld_shared_u4(row + 32 + 32 * dd, reinterpret_cast<uint32_t&>(o.x), reinterpret_cast<uint32_t&>(o.y),
                   reinterpret_cast<uint32_t&>(o.z), reinterpret_cast<uint32_t&>(o.w));
      f.add(l, o);
    }
    if (d < nd) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        out[j * kHeadDim + d_lo + d] = __float2bfloat16_rn(f.den[j] > 0.f ? f.acc[j] / f.den[j] : 0.f);
    }
    if (d == 0 && d_lo == 0 && p.lse != nullptr) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        p.lse[static_cast<int64_t>(b) * kQoHeads + h0 + 4 * hh + j] = f.den[j] > 0.f ? f.m[j] + log2f(f.den[j])
                                                                                  : -INFINITY;
    }
  }
}

// The dims of an even split of the 128 over the S - 1 boundaries of a
// sequence cut into S pieces that belong to boundary `rank`: [d_lo, d_lo + nd)
// (none when there are more boundaries than dims).
__device__ __forceinline__ void share_dims(int S, int rank, int& d_lo, int& nd) {
  const int nr = S - 1;
  d_lo = rank * kHeadDim / nr;
  nd = (rank + 1) * kHeadDim / nr - d_lo;
}

// One-wave mode: the record of virtual CTA v, written by the warp of KV head
// 0 that walked v's range when it is done: the sequence holding the range's
// last unit (b, head group hg) and how it is cut (S pieces from virtual CTA
// first_cta, the first in slot first_slot). Two 64-bit words (each read and
// written whole), each tagged with the low 27 bits of the call's epoch, so a
// reader takes a record only when both words are this call's.
constexpr int kRecTagBits = 27;
__device__ __forceinline__ unsigned long long rec_tag(unsigned long long epoch) {
  return (epoch & ((1ull << kRecTagBits) - 1)) << (64 - kRecTagBits);
}

__device__ __forceinline__ void write_range_rec(unsigned long long* rec, int v, unsigned long long epoch, int b, int hg,
                                                const SplitInfo& si) {
  const unsigned long long tag = rec_tag(epoch);
  rec[2 * v] = tag | (static_cast<unsigned long long>(si.first_cta) << 20) |
               (static_cast<unsigned long long>(si.S) << 3) | (static_cast<unsigned long long>(hg) << 1) |
               static_cast<unsigned long long>(si.first_slot);
  rec[2 * v + 1] = tag | static_cast<unsigned long long>(static_cast<unsigned>(b));
}

// One-wave mode, after the warp's stream and arrivals: its merge duties, the
// boundaries j = c, c + P1, ... after virtual CTA j for warp w of CTA c (KV
// head w), so every warp gets about the same number whatever ranges it walked.
// Lane k takes boundary k: it waits (bounded) for range j's record, and, when
// the sequence there goes on past j, for all of that sequence's pieces to
// arrive. Then the shares are staged together, as many at a time as the
// drained rings hold, and merged; a share too large to stage at once (a
// sequence cut into more pieces than there are dims) stages its pieces in
// batches on its own.
template <int NG, int HG>
__device__ __noinline__ void run_duties(const DecodeParams& p, int64_t W1, int64_t q1, int64_t q2, int T, int w,
                                        int lane, uint32_t stage, int stage_bytes) {
  Plan pl;
  pl.W = static_cast<int64_t>(T) * HG;
  pl.W1 = W1;
  pl.q1 = q1;
  pl.q2 = q2;
  pl.P1 = p.plan.tier1_ctas;
  pl.P2 = p.plan.tier2_ctas;
  const int j = blockIdx.x + static_cast<int>(gridDim.x) * lane;  // this lane's boundary
  const bool has = j + 1 < pl.P1 + pl.P2 && pl.begin(j + 1) < pl.W;
  const unsigned long long tag = rec_tag(p.epoch);
  const unsigned long long* rec = reinterpret_cast<const unsigned long long*>(p.split_rec);
  int b = 0, fc = 0, S = 0, hg = 0, fs = 0, d_lo = 0, nd = 0;
  int state = has ? 0 : 2;  // 0: waiting for the record, 1: for the pieces, 2: done
  bool ok = true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (state == 0) {
      const unsigned long long a = ld_relaxed_u64(rec + 2 * j), c = ld_relaxed_u64(rec + 2 * j + 1);
      if ((a & ~0ull << (64 - kRecTagBits)) == tag && (c & ~0ull << (64 - kRecTagBits)) == tag) {
        fc = static_cast<int>((a >> 20) & 0x1ffffu);
        S = static_cast<int>((a >> 3) & 0x1ffffu);
        hg = static_cast<int>((a >> 1) & 3u);
        fs = static_cast<int>(a & 1u);
        b = static_cast<int>(c & 0xffffffffu);
        const bool cut = fc + S - 1 > j;  // the sequence goes on past boundary j
        if (cut) share_dims(S, j - fc, d_lo, nd);
        state = cut && nd > 0 ? 1 : 2;
      }
    }
    if (state == 1) {
      const unsigned long long v = ld_relaxed_u64(p.tickets + static_cast<int64_t>(fc) * NG + w);
      if ((v >> 24) == p.epoch && (v & 0xffffffull) >= static_cast<unsigned>(S)) state = 2;
    }
    if (state != 2 && global_timer_ns() - t0 > p.wait_limit_ns) {
      atomicOr(p.err, kErrMergeWait);
      state = 2;
      ok = false;
    }
    if (__all_sync(0xffffffffu, state == 2)) break;
    __nanosleep(256);
  }
  __threadfence();
  __syncwarp();
  const unsigned todo = __ballot_sync(0xffffffffu, ok && nd > 0);
  const int n = 32 - __clz(__ballot_sync(0xffffffffu, has));  // lanes 0 .. n - 1 hold boundaries
#pragma unroll 1
  for (int k = 0; k < n;) {
    // stage shares k, k + 1, ... while they fit, then merge them from shared memory
    uint32_t off = 0;
    int k2 = k;
    for (; k2 < n; ++k2) {
      const int kd = __shfl_sync(0xffffffffu, nd, k2), ks = __shfl_sync(0xffffffffu, S, k2);
      if (!((todo >> k2) & 1u)) continue;
      const int need = ks * (32 + 32 * kd);
      if (off + need > static_cast<uint32_t>(stage_bytes)) break;
      issue_partials<NG>(p, __shfl_sync(0xffffffffu, fc, k2), __shfl_sync(0xffffffffu, fs, k2), w,
                         __shfl_sync(0xffffffffu, d_lo, k2), kd, 0, ks, 32 + 32 * kd, stage + off, lane);
      off += need;
    }
    const bool alone = k2 == k;  // share k does not fit by itself: it stages in batches
    if (alone) k2 = k + 1;
    if (!alone) staged_wait();
    off = 0;
#pragma unroll 1
    for (int i = k; i < k2; ++i) {
      if (!((todo >> i) & 1u)) continue;
      const int ks = __shfl_sync(0xffffffffu, S, i), kd = __shfl_sync(0xffffffffu, nd, i);
      merge_share<NG>(p, __shfl_sync(0xffffffffu, b, i), (__shfl_sync(0xffffffffu, hg, i) * NG + w) * kGroup,
                      __shfl_sync(0xffffffffu, fc, i), __shfl_sync(0xffffffffu, fs, i), ks, w,
                      __shfl_sync(0xffffffffu, d_lo, i), kd, stage + off, alone ? stage_bytes : ks * (32 + 32 * kd),
                      !alone, lane);
      off += ks * (32 + 32 * kd);
    }
    __syncwarp();  // the staging area is reused by the next group
    k = k2;
  }
}

// One-wave mode: install this call's counters. Warp w of CTA c resets the
// arrival tickets of virtual CTAs c, c + P1, ... for KV head w; CTA 0 also
// the tier-2 range counter of warp index w. (Not inlined: it runs once, and
// inlined it costs the streaming loop registers.)
template <int NG>
__device__ __noinline__ void install_call_counters(const DecodeParams& p, int w, int lane) {
  const int ctas = p.plan.tier1_ctas + p.plan.tier2_ctas;
  for (int v = blockIdx.x + static_cast<int>(gridDim.x) * lane; v < ctas; v += 32 * static_cast<int>(gridDim.x))
    install_counter(p.tickets + static_cast<int64_t>(v) * NG + w, p.epoch);
  if (blockIdx.x == 0 && lane == 0) install_counter(p.grab + w, p.epoch);
}

// SP: selected-token (sparse) mode. Every row of the batch is one "sequence" of
// exactly p.sparse_topk columns; kv_indices holds their resolved slots, and a
// slot of -1 (an invalid column) is masked out of the softmax.
// F8: the K/V caches are FP8 rows (kGlobalRowBytes per token): e4m3 values of
// the 4 KV heads, then their fp32 scales.
// CC: the contractions on the CUDA cores (attend_subtile_cc) instead of
// mma.sync, a variant kept for comparing the two.
template <int NG, int D, bool SP, bool F8 = false, bool CC = false, int TT = 16>
__global__ void __launch_bounds__(NG * 32, (F8 || CC) ? (TT == 32 ? 2 : 3) : 16 / NG)
    gqa_decode_lsu_kernel(const DecodeParams p) {
  using C = LsuCfg<NG, D, F8, TT>;
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
  const bool one_wave = !F8 && p.inline_merge != 0;  // the FP8 variants run the static grid only
  const int B = p.batch;
  // kv_indptr[B], the first round of the kv_indptr search and (one-wave mode)
  // this lane's empty-sequence check go out together: one round trip
  const int pre = (SP || F8) ? 0 : first_search_round(p.kv_indptr, B, lane);
  const int T = SP ? p.sparse_total : __ldg(p.kv_indptr + B);
  if (!SP && one_wave) {
    for (int b0 = (blockIdx.x * NG + w) * 32; b0 < B; b0 += gridDim.x * NG * 32) {
      const int b = b0 + lane;
      const bool empty = b < B && __ldg(p.kv_indptr + b) == __ldg(p.kv_indptr + b + 1);
      for (unsigned m = __ballot_sync(0xffffffffu, empty); m != 0; m &= m - 1) write_empty_seq(p, b0 + __ffs(m) - 1, lane);
    }
  }
  SmemPlan* splan = reinterpret_cast<SmemPlan*>(wsm + C::kPlanOff);
  const int64_t W = static_cast<int64_t>(T) * C::kHG;
  int64_t u0, u1;
  {
    const Plan pl = make_plan(W, p.plan);
    u0 = pl.begin(blockIdx.x);
    u1 = pl.end(blockIdx.x);
    if (lane == 0) *splan = SmemPlan{pl.W1, pl.q1, pl.q2, pl.P1, static_cast<int>(blockIdx.x), 1, 0, 0, 0};
    __syncwarp();
  }
  if (one_wave) install_call_counters<NG>(p, w, lane);

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

  // Opens the head-group segment at u_next of the current range. `first`:
  // the warp's first segment, whose kv_indptr search starts from the round
  // loaded beside kv_indptr[B] (a constant at each call site, so `pre` is dead
  // once the first segment is open).
  auto open_segment = [&](bool first) -> bool {
    const int Ti = T;
    hg = static_cast<int>(u_next / Ti);
    tt = static_cast<int>(u_next - static_cast<int64_t>(hg) * Ti);
    t_stop = static_cast<int>(min(static_cast<int64_t>(Ti), u1 - static_cast<int64_t>(hg) * Ti));
    u_next = static_cast<int64_t>(hg) * Ti + t_stop;
    seg_open = true;
    p_hi = tt;
    // the page ids depend on tt alone: request them first, so that their
    // round trip overlaps the search of kv_indptr
    ib = tt & ~31;
#pragma unroll
    for (int c = 0; c < C::kIdsRing / 32; ++c) request_ids(ib + 32 * c + lane);
    cp_async_commit();
    if (!SP) wb = warp_find_window(p.kv_indptr, B, tt, lane, first, pre, win);
    cp_async_wait<0>();
    __syncwarp();
    if (wb < 0) {
      if (lane == 0) atomicOr(p.err, kErrBadIndptr);
      walk_ok = false;
      return false;
    }
    return true;
  };
  // The bf16 variants open their first segment here, its search starting
  // from the round loaded beside kv_indptr[B]; the FP8 variants open it in
  // their first issue (measured: the early open slows their ALU-bound loop
  // by about 5%).
  if (!F8 && u0 < u1) open_segment(true);

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
        tl.vcta = one_wave ? splan->vcta : static_cast<int>(blockIdx.x);
        tl.si = p_si;
        p_flags &= ~F_QLOAD;
        tt += tl.cnt;
        return true;
      }
      if (u_next >= u1) {
        if (!one_wave) return false;
        // the range is walked: publish its record (the merge duty of the
        // boundary after it reads where its last sequence is cut)
        if (w == 0 && lane == 0 && u0 < u1 && walk_ok) write_range_rec(reinterpret_cast<unsigned long long*>(p.split_rec), splan->vcta, p.epoch, pb, hg, p_si);
        const int nr = splan->n_ranges;
        __syncwarp();  // every lane has read the block before lane 0 updates it
        if (nr >= kMaxWarpRanges) return false;  // the other warps take the rest
        const int64_t Wu = static_cast<int64_t>(T) * C::kHG;
        if (p.plan.tier2_ctas <= 0 || splan->W1 >= Wu) return false;  // no tier 2 in this call
        long long v = -1;
        if (lane == 0) v = installed_fetch_add(p.grab + w, p.epoch, p.err);
        v = __shfl_sync(0xffffffffu, v, 0);
        if (v < 0 || v >= p.plan.tier2_ctas) return false;
        const int64_t r0 = splan->W1 + v * splan->q2;
        if (r0 >= Wu) return false;  // tier 2 is used up (later ranges are empty as well)
        u0 = r0;
        u1 = min(r0 + splan->q2, Wu);
        u_next = u0;
        __syncwarp();
        if (lane == 0) {
          splan->vcta = splan->P1 + static_cast<int>(v);
          splan->n_ranges = nr + 1;
        }
        __syncwarp();
      }
      // open the next head-group segment of the range
      if (!open_segment(false)) break;
    }
    return false;
  };

  // -------------------------------------------------------------- issue
  // bf16 K/V head rows are read once: they leave L2 first, ahead of the page ids, Q and the split
  // partials (measured: about 10 us less per call on the large batch, 6 us on the skewed one). Not
  // for the FP8 rows, whose issue-bound loop measured slower with the hint (280 -> 296 us on large;
  // 356 us with it kept off the sectors that neighbouring heads' chunks share).
  const uint64_t stream_pol = F8 ? 0ull : l2_policy_evict_first();
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
      unsigned mask = tl.cnt >= 32 ? 0xffffffffu : ((1u << tl.cnt) - 1u);
      if constexpr (F8) {
        // kTile tokens x 8 16-byte chunks of the 128-byte e4m3 head row, for K and V
#pragma unroll
        for (int i = 0; i < C::kTile / 4; ++i) {
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
        {  // the per-token scales of this KV head: 16 tokens: lanes 0-15 K, 16-31 V; 32: K and V of token lane
          const int tok = C::kTile == 16 ? (lane & 15) : lane;
          bool valid = tok < tl.cnt;
          int pg = valid ? ids[(tl.tt + tok) & (C::kIdsRing - 1)] : 0;
          if (valid && p.num_pages_check > 0 &&
              static_cast<unsigned>(pg) >= static_cast<unsigned>(p.num_pages_check)) {
            valid = false;
            pg = 0;
          }
          const int64_t off = static_cast<int64_t>(pg) * C::kGlobalRowBytes + kKvHeads * kHeadDim +
                              (tl.hg * NG + w) * 4;
          if constexpr (C::kTile == 16) {
            cp_async_4(sb + (lane < 16 ? C::kSkOff : C::kSvOff) + tok * 4, (lane < 16 ? kc : vc) + off,
                       valid ? 4u : 0u);
          } else {
            cp_async_4(sb + C::kSkOff + tok * 4, kc + off, valid ? 4u : 0u);
            cp_async_4(sb + C::kSvOff + tok * 4, vc + off, valid ? 4u : 0u);
          }
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
        cp_async_16_hint(sb + C::kKOff + tok * C::kRowPitch + pc * 16, kc + off, nbytes, stream_pol);
        cp_async_16_hint(sb + C::kVOff + tok * C::kRowPitch + pc * 16, vc + off, nbytes, stream_pol);
      }
      if (flags & F_QLOAD) {
        const int h0 = (tl.hg * NG + w) * kGroup;
        if (!qn_busy) {
          if constexpr (CC)
            load_q_cc(qn, qg, tl.b, h0, lane);
          else
            load_q_frags<F8>(qn, qg, tl.b, h0, lane);
          qn_busy = true;
          flags |= F_QREG;
        } else if (lane < 16) {
          prefetch_l2(qg + (static_cast<int64_t>(tl.b) * kQoHeads + h0) * kHeadDim + lane * 64);
        }
      }
      if (lane == 0) {
        st_shared_v4(sb + C::kHdrOff, tl.b, tl.cnt, flags, tl.hg);
        if constexpr (F8)  // the FP8 variants run the static grid: the virtual CTA is the CTA
          st_shared_v4(sb + C::kHdrOff + 16, tl.si.S, tl.si.first_cta, tl.si.first_slot, static_cast<int>(mask));
        else
          st_shared_v4(sb + C::kHdrOff + 16, tl.si.S, tl.si.first_cta, tl.vcta,
                       static_cast<int>(mask) | (tl.si.first_slot << 16));
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
  CcState cs;  // the CUDA-core variant's state (unused otherwise)
  cs.reset();
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
    int tile_cta, tok_mask;
    if constexpr (F8) {
      ld_shared_v4(sb + C::kHdrOff + 16, si.S, si.first_cta, si.first_slot, tok_mask);
      tile_cta = blockIdx.x;
    } else {
      ld_shared_v4(sb + C::kHdrOff + 16, si.S, si.first_cta, tile_cta, tok_mask);
      si.first_slot = tok_mask >> 16;
      tok_mask &= 0xffff;
    }
    if (flags & F_DONE) break;
    const int h0 = (thg * NG + w) * kGroup;
    if (flags & F_QLOAD) {
      if (flags & F_QREG) {
#pragma unroll
        for (int i = 0; i < 16; ++i) st.qf[i] = qn[i];
        qn_busy = false;
      } else if constexpr (CC) {
        load_q_cc(st.qf, qg, hb, h0, lane);
      } else {
        load_q_frags<F8>(st.qf, qg, hb, h0, lane);
      }
      if constexpr (CC) {
        q_to_cc(cs, st.qf);
        cs.reset();
      } else {
        st.reset();
      }
      if constexpr (F8) st.qsc = q_frags_to_f16(st.qf);
    }
    if constexpr (CC) {
      attend_subtile_cc(cs, sb + C::kKOff, sb + C::kVOff, C::kRowPitch, static_cast<unsigned>(tok_mask), p.scale_log2,
                        lane);
    } else if constexpr (F8 && C::kTile == 32) {
      const int r = lane >> 2;
      float sk[4], sv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sk[i] = ld_shared_f32(sb + C::kSkOff + (r + 8 * i) * 4);
        sv[i] = ld_shared_f32(sb + C::kSvOff + (r + 8 * i) * 4);
      }
      attend_tile32_f8(st, sb + k_lane, sb + v_lane, static_cast<unsigned>(tok_mask), p.scale_log2, sk, sv, lane,
                       C::kK8Pitch, C::kV8Pitch);
    } else if constexpr (F8) {
      const int r = lane >> 2;
      const float sk_lo = ld_shared_f32(sb + C::kSkOff + r * 4), sk_hi = ld_shared_f32(sb + C::kSkOff + (r + 8) * 4);
      const float sv_lo = ld_shared_f32(sb + C::kSvOff + r * 4), sv_hi = ld_shared_f32(sb + C::kSvOff + (r + 8) * 4);
      attend_subtile_f8(st, sb + k_lane, sb + v_lane, static_cast<unsigned>(tok_mask), p.scale_log2, sk_lo, sk_hi,
                        sv_lo, sv_hi, lane, C::kK8Pitch);
    } else {
      attend_subtile(st, sb + k_lane, sb + v_lane, static_cast<unsigned>(tok_mask), p.scale_log2, lane);
    }
    if (flags & F_END) {
      bool owes;
      if constexpr (CC)
        owes = finish_piece_cc<NG>(cs, (flags & F_FINAL) != 0, hb, h0, slot_id(tile_cta, (flags & F_SLOT1) ? 1 : 0), w,
                                   si, p, lane);
      else
        owes = finish_piece<NG, F8>(st, (flags & F_FINAL) != 0, hb, h0, slot_id(tile_cta, (flags & F_SLOT1) ? 1 : 0),
                                    w, si, p, lane, F8 ? st.cv : 1.f);
      if (owes) {
        pend[n_pend < 2 ? n_pend : 1] = {si, hb, h0};
        n_pend = min(n_pend + 1, 2);
      }
      if (one_wave && !(flags & F_FINAL) && lane == 0) {  // a split piece: its arrival is counted after the stream
        const int na = splan->n_arr;
        reinterpret_cast<int*>(wsm + C::kArrOff)[na] = si.first_cta * NG + w;
        splan->n_arr = na + 1;
      }
    }
    __syncwarp();  // every lane is done with this stage before it is refilled
  }
  cp_async_wait<0>();
  __syncwarp();
  if (one_wave) {
    // count this warp's split pieces (one fence publishes all of their
    // partials), then merge the shares that fell to it; the stage and
    // page-id rings have drained and stage the partials
    const int n_arr = splan->n_arr;
    if (n_arr > 0) {
      __threadfence();
      __syncwarp();
      const int* arr = reinterpret_cast<const int*>(wsm + C::kArrOff);
      for (int i = lane; i < n_arr; i += 32) installed_fetch_add(p.tickets + arr[i], p.epoch, p.err);
    }
    run_duties<NG, C::kHG>(p, splan->W1, splan->q1, splan->q2, T, w, lane, wbase, C::kStagingBytes);
    return;
  }
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

// launch: kLaunchPlain, kLaunchPdl (a programmatic dependent of the kernel
// before it on the stream) or kLaunchCooperative (the one-wave mode: every CTA
// resident at once, which the in-kernel merge's waits rely on).
template <int NG, int D, bool SP, bool F8 = false, bool CC = false, int TT = 16>
static cudaError_t launch_lsu(const DecodeParams& p, int num_ctas, cudaStream_t stream, int launch) {
  using C = LsuCfg<NG, D, F8, TT>;
  static std::atomic<int> configured[kMaxDevices];
  const cudaError_t e = set_smem_limit_once(
      configured, reinterpret_cast<const void*>(gqa_decode_lsu_kernel<NG, D, SP, F8, CC, TT>), C::kSmemBytes);
  if (e != cudaSuccess) return e;
  if (launch == kLaunchPlain) {
    gqa_decode_lsu_kernel<NG, D, SP, F8, CC, TT><<<num_ctas, C::kThreads, C::kSmemBytes, stream>>>(p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_ctas);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (launch == kLaunchPdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gqa_decode_lsu_kernel<NG, D, SP, F8, CC, TT>, p);
}

// CTAs of a variant that the current device holds at once (0 if it cannot be
// queried), cached per device.
template <int NG, int D, bool SP, bool F8 = false, int TT = 16>
static int coresident_lsu() {
  using C = LsuCfg<NG, D, F8, TT>;
  static std::atomic<int> configured[kMaxDevices];
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  const int c = cached[dev].load(std::memory_order_acquire);
  if (c > 0) return c;
  const void* fn = reinterpret_cast<const void*>(gqa_decode_lsu_kernel<NG, D, SP, F8, false, TT>);
  if (set_smem_limit_once(configured, fn, C::kSmemBytes) != cudaSuccess) return 0;
  int per_sm = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, C::kThreads, C::kSmemBytes) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int n = per_sm * sms;
  cached[dev].store(n, std::memory_order_release);
  return n;
}

#define GQA_LSU_VARIANTS(X) X(4, 3) X(4, 4) X(4, 2) X(2, 3) X(2, 2) X(2, 5) X(1, 3) X(1, 2) X(1, 4) X(1, 6)

int lsu_smem_bytes(int ng, int stages) {
#define X(NG, D) \
  if (ng == NG && stages == D) return LsuCfg<NG, D>::kSmemBytes;
  GQA_LSU_VARIANTS(X)
#undef X
  return -1;
}

cudaError_t launch_decode_lsu(int ng, int stages, const DecodeParams& p, int num_ctas, cudaStream_t stream,
                              int launch) {
#define X(NG, D) \
  if (ng == NG && stages == D) return launch_lsu<NG, D, false>(p, num_ctas, stream, launch);
  GQA_LSU_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

// Selected-token mode: one variant, 4 KV heads per CTA and a 2-deep ring.
cudaError_t launch_decode_lsu_sparse(const DecodeParams& p, int num_ctas, cudaStream_t stream, int launch) {
  return launch_lsu<4, 2, true>(p, num_ctas, stream, launch);
}

// FP8-cache variants: 4 KV heads per CTA; 16-token stages in a ring of 2, 3
// or 4, or 32-token stages in a ring of 2.
#define GQA_LSU_F8_VARIANTS(X) X(4, 2, 16) X(4, 3, 16) X(4, 4, 16) X(4, 2, 32)

int lsu_f8_smem_bytes(int stages, int tile) {
#define X(NG, D, TT) \
  if (stages == D && tile == TT) return LsuCfg<NG, D, true, TT>::kSmemBytes;
  GQA_LSU_F8_VARIANTS(X)
#undef X
  return -1;
}

cudaError_t launch_decode_lsu_f8(int stages, int tile, const DecodeParams& p, int num_ctas, cudaStream_t stream,
                                 int launch) {
#define X(NG, D, TT) \
  if (stages == D && tile == TT) return launch_lsu<NG, D, false, true, false, TT>(p, num_ctas, stream, launch);
  GQA_LSU_F8_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

// The CUDA-core comparison variant: 4 KV heads per CTA, 2 stages (the
// default's shape), static grid.
int lsu_cc_smem_bytes() { return LsuCfg<4, 2>::kSmemBytes; }

cudaError_t launch_decode_lsu_cc(const DecodeParams& p, int num_ctas, cudaStream_t stream) {
  return launch_lsu<4, 2, false, false, true>(p, num_ctas, stream, kLaunchPlain);
}

int decode_coresident_ctas(const KernelChoice& k, bool sparse) {
  if (sparse) return coresident_lsu<4, 2, true>();
  if (k.gather == kGatherLsuF8) {
#define X(NG, D, TT) \
  if (k.stages == D && k.tile == TT) return coresident_lsu<NG, D, false, true, TT>();
    GQA_LSU_F8_VARIANTS(X)
#undef X
    return 0;
  }
  if (k.gather != kGatherLsu) return 0;
#define X(NG, D) \
  if (k.heads_per_cta == NG && k.stages == D) return coresident_lsu<NG, D, false>();
  GQA_LSU_VARIANTS(X)
#undef X
  return 0;
}

}  // namespace gqa
