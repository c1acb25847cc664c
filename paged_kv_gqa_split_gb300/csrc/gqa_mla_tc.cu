// Dense MLA paged decode on the tensor-memory MMA (tcgen05) path: the same
// operation, plan, partials and split records as gqa_mla_decode_kernel (the
// dense decode of the flash_mla_with_kvcache page: one latent KV head of 576
// values, V = its first 512, natural-log LSE), for block sizes that are a
// multiple of 32 tokens.
//
// A tcgen05.mma costs about 45-80 cycles at small shapes, so the tiles put 128
// tokens on M and the R query rows of a piece (64 when the rows of a sequence
// come in multiples of 64, else 32 when in multiples of 32, else 16) on N:
// S^T = K Q^T (M = 128 tokens, N = R,
// K = 576: 36 MMAs) and O^T += V^T P^T (M = 128 dims x 4 blocks, N = R,
// K = 128 tokens: 32 MMAs) per 128-token tile. With R = 64 one pass over the
// latent rows serves 64 heads, where 16-row pieces would read them four times.
// A tile's 147 KB of latent rows do not fit beside a ring, so they stream
// through a ring of 32 KB units (two 64-dim regions of the 128 rows, loaded by
// 2D tensor copies with 128-byte swizzle): five units feed S^T, and the four V
// units are loaded again (from L2) for the P.V of the tile once its softmax is
// done. The ring holds 6 units at R = 16, 5 at R = 32 and 4 at R = 64, beside
// Q (R rows x 576) and the P^T buffers.
//
// One CTA per SM, in roles:
//   softmax groups (4 warps each, one per 32-lane quarter of tensor memory):
//              thread t owns token t of the tile and RG = min(R, 32) of its
//              scores; the running max of a row moves only when a score
//              passes it by more than 2^8 (a vote over the group decides), so
//              P = 2^(s - m) < 256 in bf16 and the row sums stay per thread
//              until the end of a piece; R / RG groups. A group also
//              rescales its rows of O^T when a max moved, and writes them
//              out (O, or the fp32 partial) at the end of a piece;
//   1 MMA warp (an elected lane issues), 1 producer warp (tensor copies).
// Every hand-off is an mbarrier (or a named barrier inside a softmax group);
// every wait is bounded: on a timeout the CTA flags kErrTimeoutFull or
// kErrTimeoutEmpty and returns after draining its copies and MMAs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "gqa_common.cuh"
#include "gqa_kernels.h"
#include "gqa_tc.cuh"

namespace gqa {
namespace {

constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kTile = 128;                    // tokens per tile (MMA M)
constexpr int kRegionBytes = kTile * 128;     // 16 KB: 128 rows x 64 dims
constexpr int kUnitBytes = 2 * kRegionBytes;  // 32 KB ring unit: two regions
constexpr int kSUnits = 5;                    // regions (0,1) (2,3) (4,5) (6,7) (8)
constexpr int kVUnits = 4;                    // regions (0,1) .. (6,7): dim blocks of 128
constexpr float kRescaleThreshold = 8.f;      // log2 units
constexpr uint64_t kWaitNs = 2000000000ull;

// Shared memory and roles for R query rows per piece.
template <int R>
struct TcCfg {
  static constexpr int RG = R < 32 ? R : 32;         // rows per softmax group
  static constexpr int kGroups = R / RG;             // 1 or 2
  static constexpr int kSoftWarps = 4 * kGroups;
  static constexpr int kMmaWarp = kSoftWarps;
  static constexpr int kProdWarp = kSoftWarps + 1;
  static constexpr int kThreads = (kSoftWarps + 2) * 32;
  static constexpr int kRing = R == 16 ? 6 : (R == 32 ? 5 : 4);
  static constexpr int kPBufs = R == 64 ? 1 : 2;    // P^T buffers (one at R = 64 leaves room for a 4th unit)
  static constexpr int kQRegion = R * 128;           // R rows x 64 dims
  static constexpr int kPBytes = R * kTile * 2;      // P^T: R rows x 128 tokens
  static constexpr int kQOff = kRing * kUnitBytes;
  static constexpr int kPOff = kQOff + 9 * kQRegion;
  static constexpr int kAlphaOff = kPOff + kPBufs * kPBytes;  // [R] f32: the rescale factor of each row
  static constexpr int kLinvOff = kAlphaOff + R * 4;     // [R] f32: 1 / l of each row at a piece's end
  static constexpr int kRedOff = kLinvOff + R * 4;       // [kGroups][4][RG] f32: per-warp row reductions
  static constexpr int kBarOff = (kRedOff + kGroups * 4 * RG * 4 + 7) / 8 * 8;
  // mbarriers
  static constexpr int B_FULL = 0;                 // [kRing] unit loaded (producer arrival + bytes)
  static constexpr int B_EMPTY = B_FULL + kRing;   // [kRing] unit consumed (MMA commit)
  static constexpr int B_QFULL = B_EMPTY + kRing;  // Q of the piece loaded
  static constexpr int B_QFREE = B_QFULL + 1;      // S^T MMAs of the piece's last tile done
  static constexpr int B_SFULL = B_QFREE + 1;      // [2] S^T buffer written (MMA commit)
  static constexpr int B_SFREE = B_SFULL + 2;      // [2] S^T buffer read (one arrival per softmax group)
  static constexpr int B_PREADY = B_SFREE + 2;     // [2] P^T written and O^T rescaled (one per group)
  static constexpr int B_PVDONE = B_PREADY + 2;    // [2] P.V of the tile done (MMA commit)
  static constexpr int B_OFREE = B_PVDONE + 2;     // O^T read by the epilogue (one per group)
  static constexpr int B_FINAL = B_OFREE + 1;      // every MMA of the CTA done
  static constexpr int kBars = B_FINAL + 1;
  static constexpr int kSlotOff = kBarOff + kBars * 8;
  static constexpr int kAbortOff = kSlotOff + 4;
  static constexpr int kSmemBytes = kAbortOff + 4 + 1024;  // the base is rounded up to 1024 B (swizzle atoms)
  static constexpr uint32_t kCols = R == 16 ? 128 : (R == 32 ? 256 : 512);  // S^T at 0 and R, O^T block mb at 2R + R mb
  static_assert(kSmemBytes <= 227 * 1024, "tensor-memory MLA decode exceeds shared memory");
  static_assert(kQOff % 1024 == 0 && kPOff % 1024 == 0, "swizzle atoms need 1024-byte alignment");
  static_assert(2 * R + 4 * R <= static_cast<int>(kCols), "tensor memory columns");
  __host__ __device__ static constexpr uint32_t bar_count(int i) {
    return (i == B_SFREE || i == B_SFREE + 1 || i == B_PREADY || i == B_PREADY + 1 || i == B_OFREE)
               ? static_cast<uint32_t>(kGroups)
               : 1u;
  }
};

struct TcTile {
  int b, hg, tt, t_loc, cnt, flags;
};

// The CTA's tiles in order (each role warp runs its own copy): unit ranges
// [u0, u1) of (row group, token) units, cut at sequence ends and at 128-token
// boundaries of the sequence.
struct TcWalker {
  const int* indptr;
  const int64_t* bounds;  // cost-balanced CTA ranges (one tier), or NULL for the plan's ranges
  int B, T;
  Plan pl;
  int64_t u0, u1, u_next;
  int hg, tt, t_stop, p_lo, p_hi, p_flags, pb, wb, win;
  bool seg_open, ok;
  SplitInfo p_si;

  __device__ int64_t begin_of(int64_t c) const { return bounds != nullptr ? __ldg(bounds + c) : pl.begin(c); }
  // CTA whose range holds unit u: with bounds, the last c with bounds[c] <= u (ranges may be empty)
  __device__ int64_t cta_of(int64_t u) const {
    if (bounds == nullptr) return pl.cta_of(u);
    int lo = 0, hi = pl.P1;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(bounds + mid) <= u) lo = mid; else hi = mid;
    }
    return lo;
  }

  __device__ void init(const int* ip, const int64_t* cuts, int batch, int total, const Plan& plan, int cta) {
    indptr = ip;
    bounds = cuts;
    B = batch;
    T = total;
    pl = plan;
    u0 = cuts != nullptr ? __ldg(cuts + cta) : plan.begin(cta);
    u1 = cuts != nullptr ? __ldg(cuts + cta + 1) : plan.end(cta);
    u_next = u0;
    hg = tt = t_stop = p_lo = p_hi = p_flags = pb = wb = win = 0;
    seg_open = false;
    ok = true;
    p_si = SplitInfo{1, 0, 0};
  }

  __device__ bool next(TcTile& tl, int lane, int* err) {
    while (ok) {
      if (seg_open && tt < t_stop) {
        if (tt >= p_hi) {  // a new piece: the sequence holding token tt
          unsigned m;
          for (;;) {
            m = __ballot_sync(0xffffffffu, win <= tt);
            if (m != 0xffffffffu) break;
            wb += 31;
            win = load_indptr_window(indptr, B, wb, lane);
          }
          if (m == 0) {
            if (lane == 0) atomicOr(err, kErrBadIndptr);
            ok = false;
            break;
          }
          const int k = 31 - __clz(m);
          pb = wb + k;
          p_lo = __shfl_sync(0xffffffffu, win, k);
          const int seq_hi = __shfl_sync(0xffffffffu, win, k + 1);
          p_hi = min(seq_hi, t_stop);
          const int64_t base_u = static_cast<int64_t>(hg) * T;
          p_flags = F_QLOAD | ((tt == p_lo && p_hi == seq_hi) ? F_FINAL : 0) | ((base_u + tt != u0) ? F_SLOT1 : 0);
          const int64_t c_first = cta_of(base_u + p_lo), c_last = cta_of(base_u + seq_hi - 1);
          p_si.S = static_cast<int>(c_last - c_first + 1);
          p_si.first_cta = static_cast<int>(c_first);
          p_si.first_slot = (base_u + p_lo == begin_of(c_first)) ? 0 : 1;
        }
        const int t_loc = tt - p_lo;
        const int lim = tt + (kTile - (t_loc & (kTile - 1)));
        tl.cnt = min(lim, p_hi) - tt;
        tl.flags = p_flags | ((tt + tl.cnt == p_hi) ? F_END : 0);
        tl.b = pb;
        tl.hg = hg;
        tl.tt = tt;
        tl.t_loc = t_loc;
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
      wb = warp_find_seq(indptr, B, tt, lane);
      if (wb < 0) {
        if (lane == 0) atomicOr(err, kErrBadIndptr);
        ok = false;
        break;
      }
      win = load_indptr_window(indptr, B, wb, lane);
    }
    return false;
  }
};

__device__ __forceinline__ void store_lse_nat(const MlaParams& p, int b, int r, float lse2) {
  // natural log, [B][h_q][s_q]; r is the query row (i * h_q + h)
  p.lse[static_cast<int64_t>(b) * p.rows + (r % p.h_q) * p.s_q + r / p.h_q] = lse2 * 0.6931471805599453f;
}

// Bounded wait that ignores the abort flag (draining before exit).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitNs) break;
  }
}

// Whole warp: lane 0 waits (bounded), every lane gets the same answer.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_s, int* err, int err_bit) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = tc_wait(bar, parity, abort_s, err, err_bit, kWaitNs) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Named barrier 1 + gi over the four warps of softmax group gi, with an AND / OR of a predicate.
__device__ __forceinline__ bool group_and(int gi, bool v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.and.pred q, %2, 128, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1 : 0), "r"(1 + gi)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ bool group_or(int gi, bool v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred q, %2, 128, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1 : 0), "r"(1 + gi)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void group_sync(int gi) { asm volatile("bar.sync %0, 128;" ::"r"(1 + gi) : "memory"); }

// Softmax group gi: its first warp waits, the four warps get the same answer.
__device__ __forceinline__ bool group_wait(int gi, bool first_warp, uint32_t bar, uint32_t parity,
                                           volatile int* abort_s, int* err) {
  bool ok = true;
  if (first_warp) ok = warp_wait(bar, parity, abort_s, err, kErrTimeoutFull);
  return group_and(gi, ok);
}

// Row of the 2D tensor copy that loads chunk c (BR rows) of the tile of
// sequence b whose 128-aligned base is tb, or the row past the pool (the copy
// fills zeros) when the chunk misses [t_lo, t_hi) or its block lies outside
// the pool.
template <int BR>
__device__ __forceinline__ int chunk_row(const MlaParams& p, int b, int tb, int c, int t_lo, int t_hi) {
  const int c_lo = tb + c * BR;
  const int zero_row = p.num_blocks * p.page_size;
  if (c_lo + BR <= t_lo || c_lo >= t_hi) return zero_row;
  const int lp = c_lo / p.page_size;
  const int blk = lp < p.width ? __ldg(p.block_table + static_cast<int64_t>(b) * p.width + lp) : -1;
  return (blk >= 0 && blk < p.num_blocks) ? blk * p.page_size + c_lo % p.page_size : zero_row;
}

// Register-array element i (i uniform or not) without local memory.
template <int N>
__device__ __forceinline__ float pick(const float (&a)[N], int i) {
  float v = a[0];
#pragma unroll
  for (int k = 1; k < N; ++k) v = k == i ? a[k] : v;
  return v;
}

template <int BR, int R>
__global__ void __launch_bounds__(TcCfg<R>::kThreads, 1)
    gqa_mla_tc_decode_kernel(const MlaParams p, const __grid_constant__ MlaTcMaps maps) {
  using C = TcCfg<R>;
  constexpr int RG = C::RG;
  constexpr int kChunks = kTile / BR;
  constexpr int kRing = C::kRing;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_s = reinterpret_cast<volatile int*>(sm + C::kAbortOff);
  float* alpha_s = reinterpret_cast<float*>(sm + C::kAlphaOff);
  float* linv_s = reinterpret_cast<float*>(sm + C::kLinvOff);
  auto bar = [&](int i) { return base + C::kBarOff + 8u * static_cast<uint32_t>(i); };

  if (tid == 0) {
    for (int i = 0; i < C::kBars; ++i) mbar_init(bar(i), C::bar_count(i));
    *abort_s = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0) tc_alloc(base + C::kSlotOff, C::kCols);
  pdl_launch_dependents();
  pdl_wait();  // kv_indptr comes from the scan kernel
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + C::kSlotOff);

  const int T = __ldg(p.kv_indptr + p.batch);
  const int HG = p.rows / R;
  const Plan pl = make_plan(static_cast<int64_t>(T) * HG, p.plan);
  TcWalker wk;
  wk.init(p.kv_indptr, p.bounds, p.batch, T, pl, blockIdx.x);
  TcTile tl;
  int* err = p.err;

  if (warp == C::kProdWarp) {
    // ------------------------------------------------------------ producer
    int n = 0, piece = 0;
    int prev_rows[kChunks];  // the previous tile: its V units follow this tile's S units
    bool have_prev = false, good = true;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) prev_rows[c] = 0;
    // ring unit n: regions r0 (and r0 + 1 when nreg = 2) of the tile's chunks
    auto load_unit = [&](int r0, int nreg, const int (&rows)[kChunks]) -> bool {
      const int s = n % kRing;
      if (n >= kRing && !warp_wait(bar(C::B_EMPTY + s), ((n / kRing) - 1) & 1, abort_s, err, kErrTimeoutEmpty))
        return false;
      if (lane == 0) {
        const uint32_t full = bar(C::B_FULL + s);
        mbar_arrive_expect_tx(full, nreg * kRegionBytes);
        for (int g = 0; g < nreg; ++g)
#pragma unroll
          for (int c = 0; c < kChunks; ++c)
            tma_load_2d(base + s * kUnitBytes + g * kRegionBytes + c * BR * 128, &maps.kv, 64 * (r0 + g), rows[c], full);
      }
      __syncwarp();
      ++n;
      return true;
    };
    while (wk.next(tl, lane, err)) {
      if (tl.flags & F_QLOAD) {
        if (piece >= 1 && !warp_wait(bar(C::B_QFREE), (piece - 1) & 1, abort_s, err, kErrTimeoutEmpty)) {
          good = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::B_QFULL), 9 * C::kQRegion);
          const int y = tl.b * p.rows + tl.hg * R;
          for (int r = 0; r < 9; ++r) tma_load_2d(base + C::kQOff + r * C::kQRegion, &maps.q, 64 * r, y, bar(C::B_QFULL));
        }
        __syncwarp();
        ++piece;
      }
      const int tb = tl.t_loc & ~(kTile - 1);
      const int my_row = lane < kChunks ? chunk_row<BR>(p, tl.b, tb, lane, tl.t_loc, tl.t_loc + tl.cnt) : 0;
      int rows[kChunks];
#pragma unroll
      for (int c = 0; c < kChunks; ++c) rows[c] = __shfl_sync(0xffffffffu, my_row, c);
      for (int u = 0; u < kSUnits && good; ++u) good = load_unit(2 * u, u < 4 ? 2 : 1, rows);
      for (int u = 0; u < kVUnits && good && have_prev; ++u) good = load_unit(2 * u, 2, prev_rows);
      if (!good) break;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) prev_rows[c] = rows[c];
      have_prev = true;
    }
    for (int u = 0; u < kVUnits && good && have_prev; ++u) good = load_unit(2 * u, 2, prev_rows);
    if (lane == 0) {  // no tensor copy may still be writing shared memory when the CTA exits
      for (int i = n > kRing ? n - kRing : 0; i < n; ++i) drain_wait(bar(C::B_FULL + i % kRing), (i / kRing) & 1);
      if (piece >= 1) drain_wait(bar(C::B_QFULL), (piece - 1) & 1);
    }
    __syncwarp();
  } else if (warp == C::kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    constexpr uint32_t idesc_s = tc_idesc_bf16(kTile, R, false, false);
    constexpr uint32_t idesc_o = tc_idesc_bf16(128, R, true, false);
    int n = 0, j = 0, piece = -1;
    int pj = -1, p_first = 0, p_piece = 0;  // the tile whose P.V is pending
    bool good = true;
    auto take_unit = [&](int& s) -> bool {
      s = n % kRing;
      if (!warp_wait(bar(C::B_FULL + s), (n / kRing) & 1, abort_s, err, kErrTimeoutFull)) return false;
      ++n;
      return true;
    };
    auto issue_pv = [&]() -> bool {
      if (!warp_wait(bar(C::B_PREADY + (pj & 1)), (pj >> 1) & 1, abort_s, err, kErrTimeoutFull)) return false;
      if (p_first && p_piece >= 1 && !warp_wait(bar(C::B_OFREE), (p_piece - 1) & 1, abort_s, err, kErrTimeoutFull))
        return false;
      tc_fence_after();  // P^T and any O^T rescale were written by other threads before the barrier
      // P^T: N = R rows in 8-row groups (SBO 2048), K = tokens in 8-token core matrices (LBO 128), no swizzle
      const uint64_t dp = tc_sdesc(base + C::kPOff + (pj % C::kPBufs) * C::kPBytes, 128, 16 * 128, kSwizzleNone);
      for (int u = 0; u < kVUnits; ++u) {
        int s;
        if (!take_unit(s)) return false;
        // V^T block u: M = 128 dims over the unit's two regions (LBO), K = tokens in 8-row groups (SBO);
        // the whole warp forms the (uniform) descriptors, one elected lane issues
        const uint64_t dv = tc_sdesc(base + s * kUnitBytes, kRegionBytes, 1024, kSwizzle128B);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          tc_mma_bf16_warp(tmem + 2 * R + R * u, dv + ((kk * 2048) >> 4), dp + ((kk * 256) >> 4), idesc_o,
                           (p_first && kk == 0) ? 0u : 1u);
        tc_commit_warp(bar(C::B_EMPTY + s));
      }
      tc_commit_warp(bar(C::B_PVDONE + (pj & 1)));
      __syncwarp();
      return true;
    };
    while (wk.next(tl, lane, err)) {
      const int sb = j & 1;
      if (tl.flags & F_QLOAD) {
        ++piece;
        if (!warp_wait(bar(C::B_QFULL), piece & 1, abort_s, err, kErrTimeoutFull)) {
          good = false;
          break;
        }
      }
      if (j >= 2 && !warp_wait(bar(C::B_SFREE + sb), ((j >> 1) - 1) & 1, abort_s, err, kErrTimeoutFull)) {
        good = false;
        break;
      }
      // Q as B: N = R rows (SBO 1024 per 8 rows), K-major, 128-byte swizzle, one region per 64 dims
      const uint64_t dq = tc_sdesc(base + C::kQOff, 16, 1024, kSwizzle128B);
      for (int u = 0; u < kSUnits && good; ++u) {
        int s;
        if (!take_unit(s)) {
          good = false;
          break;
        }
        // K rows as A (tensor-copied data: the full barrier alone orders it before the MMA):
        // M = 128 tokens (SBO 1024), K-major, 128-byte swizzle, 16 KB per region
        const uint64_t dk = tc_sdesc(base + s * kUnitBytes, 16, 1024, kSwizzle128B);
        const int nreg = u < 4 ? 2 : 1;
        for (int g = 0; g < nreg; ++g)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16_warp(tmem + R * sb, dk + ((g * kRegionBytes + kk * 32) >> 4),
                             dq + (((2 * u + g) * C::kQRegion + kk * 32) >> 4), idesc_s, (u | g | kk) ? 1u : 0u);
        tc_commit_warp(bar(C::B_EMPTY + s));
      }
      if (!good) break;
      tc_commit_warp(bar(C::B_SFULL + sb));
      if (tl.flags & F_END) tc_commit_warp(bar(C::B_QFREE));
      __syncwarp();
      if (pj >= 0 && !issue_pv()) {
        good = false;
        break;
      }
      pj = j;
      p_first = (tl.flags & F_QLOAD) ? 1 : 0;
      p_piece = piece;
      ++j;
    }
    if (good && pj >= 0) issue_pv();
    if (lane == 0) {  // every MMA done before tensor memory is freed
      tc_commit(bar(C::B_FINAL));
      drain_wait(bar(C::B_FINAL), 0);
      if (wk.u0 < wk.u1 && wk.ok) {  // the split record of the CTA's last piece, as the merge reads it
        p.split_rec[blockIdx.x] =
            make_int4(static_cast<int>(static_cast<unsigned>(p.epoch)), wk.pb, wk.p_si.first_cta, wk.p_si.S);
        p.split_rec[gridDim.x + blockIdx.x] = make_int4(wk.hg, wk.p_si.first_slot, 0, 0);
      }
    }
    __syncwarp();
  } else if (warp < C::kSoftWarps) {
    // ----------------------------------------------- softmax, rescale, epilogue (group gi: rows gi RG ..)
    const int gi = warp >> 2, wq = warp & 3;  // group, tensor-memory quarter (tokens / dims 32 wq ..)
    const int ti = tid - 128 * gi;            // thread within the group
    const bool first_warp = wq == 0;
    const int tok = 32 * wq + lane;           // token of the tile = tensor-memory lane of S^T
    const bool even = (lane & 1) == 0;
    float* red_s = reinterpret_cast<float*>(sm + C::kRedOff) + gi * 4 * RG;
    const uint32_t orow = tmem + (static_cast<uint32_t>(32 * wq) << 16) + 2 * R + gi * RG;  // this group's O^T columns
    float m_used[RG], l_part[RG];
#pragma unroll
    for (int r = 0; r < RG; ++r) {
      m_used[r] = -INFINITY;
      l_part[r] = 0.f;
    }
    int j = 0;
    while (wk.next(tl, lane, err)) {
      const int sb = j & 1;
      const bool first = (tl.flags & F_QLOAD) != 0;
      if (first) {
#pragma unroll
        for (int r = 0; r < RG; ++r) {
          m_used[r] = -INFINITY;
          l_part[r] = 0.f;
        }
      }
      // this warp's 32 tokens lie in one chunk (BR >= 32): is its block in the pool?
      const int tb = tl.t_loc & ~(kTile - 1);
      int blk_ok = 1;
      if (lane == 0) {
        const int lp = (tb + 32 * wq) / p.page_size;
        const int blk = lp < p.width ? __ldg(p.block_table + static_cast<int64_t>(tl.b) * p.width + lp) : -1;
        blk_ok = blk >= 0 && blk < p.num_blocks;
      }
      blk_ok = __shfl_sync(0xffffffffu, blk_ok, 0);
      const int t_abs = tb + tok;
      const bool valid = blk_ok && t_abs >= tl.t_loc && t_abs < tl.t_loc + tl.cnt;
      if (!group_wait(gi, first_warp, bar(C::B_SFULL + sb), (j >> 1) & 1, abort_s, err)) break;
      tc_fence_after();
      float x[RG];
      bool exceed = false;
#pragma unroll
      for (int h = 0; h < RG / 16; ++h) {
        uint32_t v[16];
        tc_ld16(tmem + (static_cast<uint32_t>(32 * wq) << 16) + R * sb + gi * RG + 16 * h, v);
        tc_wait_ld();
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          x[16 * h + r] = valid ? __uint_as_float(v[r]) * p.scale_log2 : -INFINITY;
          exceed |= x[16 * h + r] > m_used[16 * h + r] + kRescaleThreshold;
        }
      }
      tc_fence_before();
      const bool any_exceed = group_or(gi, exceed);  // also: the group's four warps have read S^T buffer sb
      if (ti == 0) mbar_arrive(bar(C::B_SFREE + sb));
      bool moved = false;
      if (any_exceed) {  // per-row maximum of the tile over the 128 tokens; move the rows it passes by > 2^8
#pragma unroll
        for (int r = 0; r < RG; ++r) {
          float m = x[r];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == r) red_s[wq * RG + r] = m;
        }
        group_sync(gi);
#pragma unroll
        for (int r = 0; r < RG; ++r) {
          const float tmax = fmaxf(fmaxf(red_s[r], red_s[RG + r]), fmaxf(red_s[2 * RG + r], red_s[3 * RG + r]));
          float a = 1.f;
          if (tmax > m_used[r] + kRescaleThreshold) {
            a = m_used[r] == -INFINITY ? 0.f : ex2(m_used[r] - tmax);
            m_used[r] = tmax;
            l_part[r] *= a;
            moved = true;
          }
          if (ti == r) alpha_s[gi * RG + r] = a;
        }
        group_sync(gi);  // red_s is reused; alpha_s is written
      }
      const bool rescale = moved && !first;  // the same in every thread of the group
      // P^T buffer j % kPBufs was last read by the P.V of tile j - kPBufs
      if (j >= C::kPBufs) {
        const int jp = j - C::kPBufs;
        if (!group_wait(gi, first_warp, bar(C::B_PVDONE + (jp & 1)), (jp >> 1) & 1, abort_s, err)) break;
      }
      // P = 2^(s - m), row sums, and P^T as the K-major B operand (N = R rows, K = 128 tokens, no
      // swizzle): element (r, t) at (r / 8) * 2048 + (t / 8) * 128 + (r % 8) * 16 + (t % 8) * 2. Lane
      // pairs swap halves so the even lane writes the group's first RG / 2 rows and the odd lane the
      // others, for tokens (t, t + 1), 4 bytes each.
      {
        const int te = tok & ~1;
        const uint32_t pbase = base + C::kPOff + (j % C::kPBufs) * C::kPBytes + (te >> 3) * 128 + (te & 7) * 2;
#pragma unroll
        for (int i = 0; i < RG / 2; ++i) {
          const int hi = RG / 2 + i;
          const float plo = m_used[i] == -INFINITY ? 0.f : ex2(x[i] - m_used[i]);
          const float phi = m_used[hi] == -INFINITY ? 0.f : ex2(x[hi] - m_used[hi]);
          l_part[i] += plo;
          l_part[hi] += phi;
          const float other = __shfl_xor_sync(0xffffffffu, even ? phi : plo, 1);
          const uint32_t pk = even ? pack_bf16(plo, other) : pack_bf16(other, phi);
          const int r = gi * RG + (even ? 0 : RG / 2) + i;
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(pbase + (r >> 3) * 2048 + (r & 7) * 16), "r"(pk) : "memory");
        }
      }
      fence_proxy_async_smem();
      if (rescale) {  // O^T *= alpha on this group's rows, once the P.V of tile j - 1 is done
        if (!group_wait(gi, first_warp, bar(C::B_PVDONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort_s, err)) break;
        tc_fence_after();
#pragma unroll 1
        for (int mb = 0; mb < kDv / 128; ++mb)
#pragma unroll
          for (int c = 0; c < RG / 16; ++c) {
            uint32_t o[16];
            tc_ld16(orow + R * mb + 16 * c, o);
            tc_wait_ld();
#pragma unroll
            for (int rr = 0; rr < 16; ++rr)
              o[rr] = __float_as_uint(__uint_as_float(o[rr]) * alpha_s[gi * RG + 16 * c + rr]);
            tc_st16(orow + R * mb + 16 * c, o);
          }
        tc_wait_st();
        tc_fence_before();
      }
      group_sync(gi);  // P^T written (and O^T rescaled) by the whole group
      if (ti == 0) mbar_arrive(bar(C::B_PREADY + sb));
      if (tl.flags & F_END) {  // row sums over the 128 threads, 1/l and the LSE; O = O^T / l after P.V of tile j
#pragma unroll
        for (int r = 0; r < RG; ++r) {
          float sum = l_part[r];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
          if (lane == r) red_s[wq * RG + r] = sum;
        }
        group_sync(gi);
        if (ti < RG) {
          const float l = red_s[ti] + red_s[RG + ti] + red_s[2 * RG + ti] + red_s[3 * RG + ti];
          linv_s[gi * RG + ti] = l > 0.f ? 1.f / l : 0.f;
          const float lse2 = l > 0.f ? pick(m_used, ti) + log2f(l) : -INFINITY;  // base 2
          const int row = gi * RG + ti;  // row of the piece
          if (tl.flags & F_FINAL) {
            if (p.lse != nullptr) store_lse_nat(p, tl.b, tl.hg * R + row, lse2);
          } else {
            p.part_lse[slot_id(blockIdx.x, (tl.flags & F_SLOT1) ? 1 : 0) * R + row] = lse2;
          }
        }
        if (!group_wait(gi, first_warp, bar(C::B_PVDONE + sb), (j >> 1) & 1, abort_s, err)) break;  // also syncs linv_s
        tc_fence_after();
        const bool fin = (tl.flags & F_FINAL) != 0;
        const int64_t sid = slot_id(blockIdx.x, (tl.flags & F_SLOT1) ? 1 : 0);
#pragma unroll 1
        for (int mb = 0; mb < kDv / 128; ++mb)
#pragma unroll
          for (int c = 0; c < RG / 16; ++c) {
            uint32_t o[16];
            tc_ld16(orow + R * mb + 16 * c, o);
            tc_wait_ld();
            const int dim = 128 * mb + tok;  // tensor-memory lane of O^T = dim within the 128-dim block
            const int row0 = gi * RG + 16 * c;
            if (fin) {
              __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.out) +
                                  (static_cast<int64_t>(tl.b) * p.rows + tl.hg * R + row0) * kDv + dim;
#pragma unroll
              for (int rr = 0; rr < 16; ++rr) ob[rr * kDv] = __float2bfloat16(__uint_as_float(o[rr]) * linv_s[row0 + rr]);
            } else {
              float* po = p.part_o + (sid * R + row0) * kDv + dim;
#pragma unroll
              for (int rr = 0; rr < 16; ++rr) po[rr * kDv] = __uint_as_float(o[rr]) * linv_s[row0 + rr];
            }
          }
        tc_fence_before();
        group_sync(gi);  // the group's O^T reads are done (and linv_s / red_s may be reused)
        if (ti == 0) mbar_arrive(bar(C::B_OFREE));
      }
      ++j;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tc_dealloc(tmem, C::kCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// Rows of 576 bf16 (1152 B apart), read as boxes of 64 values x box_rows rows, 128-byte swizzle.
bool encode_rows(CUtensorMap* map, const void* base, int64_t rows, int box_rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_tiled();
  if (fn == nullptr || rows < 1) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDqk) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int box_rows_for(int page_size) { return page_size % 64 == 0 ? 64 : 32; }

template <int BR, int R>
cudaError_t launch_tc(const MlaParams& p, const MlaTcMaps& maps, int ctas, cudaStream_t stream) {
  static std::atomic<int> configured[kMaxDevices];
  const cudaError_t e = set_smem_limit_once(
      configured, reinterpret_cast<const void*>(gqa_mla_tc_decode_kernel<BR, R>), TcCfg<R>::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(TcCfg<R>::kThreads);
  cfg.dynamicSmemBytes = TcCfg<R>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gqa_mla_tc_decode_kernel<BR, R>, p, maps);
}

}  // namespace

bool mla_tc_supported(int page_size) { return page_size > 0 && page_size % 32 == 0; }

int mla_tc_piece_rows(int rows) { return rows % 64 == 0 ? 64 : (rows % 32 == 0 ? 32 : 16); }

bool mla_tc_encode(const MlaParams& p, MlaTcMaps* maps) {
  return encode_rows(&maps->kv, p.kv, static_cast<int64_t>(p.num_blocks) * p.page_size, box_rows_for(p.page_size)) &&
         encode_rows(&maps->q, p.q, static_cast<int64_t>(p.batch) * p.rows, p.piece_rows);
}

cudaError_t launch_mla_tc_decode(const MlaParams& p, const MlaTcMaps& maps, int ctas, cudaStream_t stream) {
  const bool br64 = box_rows_for(p.page_size) == 64;
  if (p.piece_rows == 64)
    return br64 ? launch_tc<64, 64>(p, maps, ctas, stream) : launch_tc<32, 64>(p, maps, ctas, stream);
  if (p.piece_rows == 32)
    return br64 ? launch_tc<64, 32>(p, maps, ctas, stream) : launch_tc<32, 32>(p, maps, ctas, stream);
  return br64 ? launch_tc<64, 16>(p, maps, ctas, stream) : launch_tc<32, 16>(p, maps, ctas, stream);
}

}  // namespace gqa
