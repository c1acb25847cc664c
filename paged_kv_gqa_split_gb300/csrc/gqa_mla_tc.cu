// Dense MLA paged decode on the tensor-memory MMA (tcgen05) path: the same
// operation, plan, partials and split records as gqa_mla_decode_kernel (the
// dense decode of the flash_mla_with_kvcache page: one latent KV head of 576
// values, V = its first 512, natural-log LSE), for block sizes that are a
// multiple of 32 tokens.
//
// A tcgen05.mma costs about 45 cycles at small shapes, so the tiles put 128
// tokens on M: S^T = K Q^T (M = 128 tokens, N = 16 query rows, K = 576: 36
// MMAs) and O^T += V^T P^T (M = 128 dims x 4 blocks, N = 16, K = 128 tokens:
// 32 MMAs) per 128-token tile. A tile's 147 KB of latent rows do not fit
// beside a ring, so they stream through a 6-deep ring of 32 KB units (two
// 64-dim regions of the 128 rows, loaded by 2D tensor copies with 128-byte
// swizzle): five units feed S^T, and the four V units are loaded again (from
// L2) for the P.V of the tile once its softmax is done.
//
// One CTA per SM, 320 threads in roles:
//   warps 0-3  softmax: thread t owns token t of the tile (tensor-memory lane
//              t of S^T) and its 16 scores; the running max of a row moves
//              only when a score passes it by more than 2^8 (a vote over the
//              128 threads decides), so P = 2^(s - m) < 256 in bf16 and the
//              row sums stay per thread until the end of a piece;
//   warps 4-7  correction and epilogue: rescale O^T when a max moved, and
//              write O (or the fp32 partial) at the end of a piece;
//   warp 8     MMA issue (one thread);
//   warp 9     producer: the tensor copies of Q and of the ring units.
// Every hand-off is an mbarrier (or a named barrier inside the softmax
// group); every wait is bounded: on a timeout the CTA flags kErrTimeoutFull or
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
constexpr int kRows = 16;                          // query rows per piece (one row group)
constexpr int kTile = 128;                         // tokens per tile (MMA M)
constexpr int kRegionBytes = kTile * 128;          // 16 KB: 128 rows x 64 dims
constexpr int kUnitBytes = 2 * kRegionBytes;       // 32 KB ring unit: two regions
constexpr int kRing = 6;
constexpr int kSUnits = 5;                         // regions (0,1) (2,3) (4,5) (6,7) (8)
constexpr int kVUnits = 4;                         // regions (0,1) .. (6,7): dim blocks of 128
constexpr int kQRegion = kRows * 128;              // 2 KB: 16 rows x 64 dims
constexpr int kPBytes = kRows * kTile * 2;         // 4 KB: P^T, 16 rows x 128 tokens
constexpr int kQOff = kRing * kUnitBytes;          // 196,608
constexpr int kPOff = kQOff + 9 * kQRegion;        // 215,040
constexpr int kAlphaOff = kPOff + 2 * kPBytes;     // [2][16] f32
constexpr int kLinvOff = kAlphaOff + 2 * kRows * 4;
constexpr int kFlagOff = kLinvOff + 2 * kRows * 4;  // [2] int
constexpr int kRedOff = kFlagOff + 16;             // [4][16] f32: per-warp row reductions
constexpr int kBarOff = kRedOff + 4 * kRows * 4;
enum : int {
  B_FULL = 0,                 // [kRing] unit loaded (producer arrival + bytes)
  B_EMPTY = B_FULL + kRing,   // [kRing] unit consumed (MMA commit)
  B_QFULL = B_EMPTY + kRing,  // Q of the piece loaded
  B_QFREE,                    // S^T MMAs of the piece's last tile done
  B_SFULL,                    // [2] S^T buffer written (MMA commit)
  B_SFREE = B_SFULL + 2,      // [2] S^T buffer read by the softmax group
  B_DEC = B_SFREE + 2,        // [2] P^T written, rescale decided
  B_PREADY = B_DEC + 2,       // [2] O^T ready for this tile's P.V
  B_PVDONE = B_PREADY + 2,    // [2] P.V of the tile done (MMA commit)
  B_OFREE = B_PVDONE + 2,     // O^T read by the epilogue
  B_CORR,                     // the four correction warps are done with O^T (4 arrivals)
  B_FINAL,                    // every MMA of the CTA done
  B_DACK,                     // [2] the correction warps copied the tile's flag, alpha and 1/l (4 arrivals)
  kBars = B_DACK + 2
};
constexpr int kSlotOff = kBarOff + kBars * 8;
constexpr int kAbortOff = kSlotOff + 4;
constexpr int kSmemUsed = kAbortOff + 4;
constexpr int kSmemBytes = kSmemUsed + 1024;  // the base is rounded up to 1024 B (swizzle atoms)
constexpr int kThreads = 320;
constexpr int kMmaWarp = 8, kProdWarp = 9;
constexpr uint32_t kCols = 128;               // S^T buffers at columns 0 and 16, O^T blocks at 32 + 16 mb
constexpr float kRescaleThreshold = 8.f;      // log2 units
constexpr uint64_t kWaitNs = 2000000000ull;
static_assert(kSmemBytes <= 227 * 1024, "tensor-memory MLA decode exceeds shared memory");
static_assert(kQOff % 1024 == 0 && kPOff % 1024 == 0, "swizzle atoms need 1024-byte alignment");
static_assert(kBarOff % 8 == 0, "mbarriers need 8-byte alignment");

struct TcTile {
  int b, hg, tt, t_loc, cnt, flags;
};

// The CTA's tiles in order (each role warp runs its own copy): unit ranges
// [u0, u1) of (row group, token) units, cut at sequence ends and at 128-token
// boundaries of the sequence.
struct TcWalker {
  const int* indptr;
  int B, T;
  Plan pl;
  int64_t u0, u1, u_next;
  int hg, tt, t_stop, p_lo, p_hi, p_flags, pb, wb, win;
  bool seg_open, ok;
  SplitInfo p_si;

  __device__ void init(const int* ip, int batch, int total, const Plan& plan, int cta) {
    indptr = ip;
    B = batch;
    T = total;
    pl = plan;
    u0 = plan.begin(cta);
    u1 = plan.end(cta);
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
          const SeqSplit sp = seq_split(pl, base_u + p_lo, base_u + seq_hi);
          p_si.S = static_cast<int>(sp.last_cta - sp.first_cta + 1);
          p_si.first_cta = static_cast<int>(sp.first_cta);
          p_si.first_slot = sp.first_slot;
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

// Named barrier 1 over the four softmax warps (threads 0-127), with an AND / OR of a predicate.
__device__ __forceinline__ bool group_and(bool v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.and.pred q, 1, 128, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1 : 0)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ bool group_or(bool v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred q, 1, 128, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1 : 0)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void group_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Softmax group: warp 0 waits, the four warps get the same answer.
__device__ __forceinline__ bool group_wait(uint32_t bar, uint32_t parity, volatile int* abort_s, int* err) {
  bool ok = true;
  if (threadIdx.x < 32) ok = warp_wait(bar, parity, abort_s, err, kErrTimeoutFull);
  return group_and(ok);
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

template <int BR>
__global__ void __launch_bounds__(kThreads, 1)
    gqa_mla_tc_decode_kernel(const MlaParams p, const __grid_constant__ MlaTcMaps maps) {
  constexpr int kChunks = kTile / BR;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_s = reinterpret_cast<volatile int*>(sm + kAbortOff);
  volatile int* flag_s = reinterpret_cast<volatile int*>(sm + kFlagOff);
  float* alpha_s = reinterpret_cast<float*>(sm + kAlphaOff);
  float* linv_s = reinterpret_cast<float*>(sm + kLinvOff);
  float* red_s = reinterpret_cast<float*>(sm + kRedOff);
  auto bar = [&](int i) { return base + kBarOff + 8u * static_cast<uint32_t>(i); };

  if (tid == 0) {
    for (int i = 0; i < kBars; ++i) mbar_init(bar(i), (i == B_CORR || i == B_DACK || i == B_DACK + 1) ? 4u : 1u);
    *abort_s = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0) tc_alloc(base + kSlotOff, kCols);
  pdl_launch_dependents();
  pdl_wait();  // kv_indptr comes from the scan kernel
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + kSlotOff);

  const int T = __ldg(p.kv_indptr + p.batch);
  const int HG = p.rows / kRows;
  const Plan pl = make_plan(static_cast<int64_t>(T) * HG, p.plan);
  TcWalker wk;
  wk.init(p.kv_indptr, p.batch, T, pl, blockIdx.x);
  TcTile tl;
  int* err = p.err;

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    int n = 0, piece = 0;
    int prev_rows[kChunks];  // the previous tile: its V units follow this tile's S units
    bool have_prev = false, good = true;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) prev_rows[c] = 0;
    // ring unit n: regions r0 (and r0 + 1 when nreg = 2) of the tile's chunks
    auto load_unit = [&](int r0, int nreg, const int (&rows)[kChunks]) -> bool {
      const int s = n % kRing;
      if (n >= kRing && !warp_wait(bar(B_EMPTY + s), ((n / kRing) - 1) & 1, abort_s, err, kErrTimeoutEmpty)) return false;
      if (lane == 0) {
        const uint32_t full = bar(B_FULL + s);
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
        if (piece >= 1 && !warp_wait(bar(B_QFREE), (piece - 1) & 1, abort_s, err, kErrTimeoutEmpty)) {
          good = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(B_QFULL), 9 * kQRegion);
          const int y = tl.b * p.rows + tl.hg * kRows;
          for (int r = 0; r < 9; ++r) tma_load_2d(base + kQOff + r * kQRegion, &maps.q, 64 * r, y, bar(B_QFULL));
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
      for (int i = n > kRing ? n - kRing : 0; i < n; ++i) drain_wait(bar(B_FULL + i % kRing), (i / kRing) & 1);
      if (piece >= 1) drain_wait(bar(B_QFULL), (piece - 1) & 1);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    constexpr uint32_t idesc_s = tc_idesc_bf16(kTile, kRows, false, false);
    constexpr uint32_t idesc_o = tc_idesc_bf16(128, kRows, true, false);
    int n = 0, j = 0, piece = -1;
    int pj = -1, p_first = 0, p_piece = 0;  // the tile whose P.V is pending
    bool good = true;
    auto take_unit = [&](int& s) -> bool {
      s = n % kRing;
      if (!warp_wait(bar(B_FULL + s), (n / kRing) & 1, abort_s, err, kErrTimeoutFull)) return false;
      ++n;
      return true;
    };
    auto issue_pv = [&]() -> bool {
      if (!warp_wait(bar(B_PREADY + (pj & 1)), (pj >> 1) & 1, abort_s, err, kErrTimeoutFull)) return false;
      if (p_first && p_piece >= 1 && !warp_wait(bar(B_OFREE), (p_piece - 1) & 1, abort_s, err, kErrTimeoutFull))
        return false;
      tc_fence_after();  // P^T and any O^T rescale were written by other threads before the barrier
      // P^T: N = 16 rows in 8-row groups (SBO 2048), K = tokens in 8-token core matrices (LBO 128), no swizzle
      const uint64_t dp = tc_sdesc(base + kPOff + (pj & 1) * kPBytes, 128, 16 * 128, kSwizzleNone);
      for (int u = 0; u < kVUnits; ++u) {
        int s;
        if (!take_unit(s)) return false;
        if (lane == 0) {
          // V^T block u: M = 128 dims over the unit's two regions (LBO), K = tokens in 8-row groups (SBO)
          const uint64_t dv = tc_sdesc(base + s * kUnitBytes, kRegionBytes, 1024, kSwizzle128B);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            tc_mma_bf16(tmem + 32 + 16 * u, dv + ((kk * 2048) >> 4), dp + ((kk * 256) >> 4), idesc_o,
                        (p_first && kk == 0) ? 0u : 1u);
          tc_commit(bar(B_EMPTY + s));
        }
        __syncwarp();
      }
      if (lane == 0) tc_commit(bar(B_PVDONE + (pj & 1)));
      __syncwarp();
      return true;
    };
    while (wk.next(tl, lane, err)) {
      const int sb = j & 1;
      if (tl.flags & F_QLOAD) {
        ++piece;
        if (!warp_wait(bar(B_QFULL), piece & 1, abort_s, err, kErrTimeoutFull)) {
          good = false;
          break;
        }
      }
      if (j >= 2 && !warp_wait(bar(B_SFREE + sb), ((j >> 1) - 1) & 1, abort_s, err, kErrTimeoutFull)) {
        good = false;
        break;
      }
      // Q as B: N = 16 rows (SBO 1024), K-major, 128-byte swizzle, one 2 KB region per 64 dims
      const uint64_t dq = tc_sdesc(base + kQOff, 16, 1024, kSwizzle128B);
      for (int u = 0; u < kSUnits && good; ++u) {
        int s;
        if (!take_unit(s)) {
          good = false;
          break;
        }
        if (lane == 0) {
          // K rows as A (tensor-copied data: the full barrier alone orders it before the MMA): M = 128 tokens (SBO 1024), K-major, 128-byte swizzle, 16 KB per region
          const uint64_t dk = tc_sdesc(base + s * kUnitBytes, 16, 1024, kSwizzle128B);
          const int nreg = u < 4 ? 2 : 1;
          for (int g = 0; g < nreg; ++g)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_bf16(tmem + 16 * sb, dk + ((g * kRegionBytes + kk * 32) >> 4),
                          dq + (((2 * u + g) * kQRegion + kk * 32) >> 4), idesc_s, (u | g | kk) ? 1u : 0u);
          tc_commit(bar(B_EMPTY + s));
        }
        __syncwarp();
      }
      if (!good) break;
      if (lane == 0) {
        tc_commit(bar(B_SFULL + sb));
        if (tl.flags & F_END) tc_commit(bar(B_QFREE));
      }
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
      tc_commit(bar(B_FINAL));
      drain_wait(bar(B_FINAL), 0);
      if (wk.u0 < wk.u1 && wk.ok) {  // the split record of the CTA's last piece, as the merge reads it
        p.split_rec[blockIdx.x] =
            make_int4(static_cast<int>(static_cast<unsigned>(p.epoch)), wk.pb, wk.p_si.first_cta, wk.p_si.S);
        p.split_rec[gridDim.x + blockIdx.x] = make_int4(wk.hg, wk.p_si.first_slot, 0, 0);
      }
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------- softmax
    const int tok = 32 * warp + lane;  // token of the tile = tensor-memory lane of S^T
    const bool even = (lane & 1) == 0;
    float m_used[kRows], l_part[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      m_used[r] = -INFINITY;
      l_part[r] = 0.f;
    }
    int j = 0;
    while (wk.next(tl, lane, err)) {
      const int sb = j & 1;
      const bool first = (tl.flags & F_QLOAD) != 0;
      if (first) {
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          m_used[r] = -INFINITY;
          l_part[r] = 0.f;
        }
      }
      // this warp's 32 tokens lie in one chunk (BR >= 32): is its block in the pool?
      const int tb = tl.t_loc & ~(kTile - 1);
      int blk_ok = 1;
      if (lane == 0) {
        const int lp = (tb + 32 * warp) / p.page_size;
        const int blk = lp < p.width ? __ldg(p.block_table + static_cast<int64_t>(tl.b) * p.width + lp) : -1;
        blk_ok = blk >= 0 && blk < p.num_blocks;
      }
      blk_ok = __shfl_sync(0xffffffffu, blk_ok, 0);
      const int t_abs = tb + tok;
      const bool valid = blk_ok && t_abs >= tl.t_loc && t_abs < tl.t_loc + tl.cnt;
      if (!group_wait(bar(B_SFULL + sb), (j >> 1) & 1, abort_s, err)) break;
      tc_fence_after();
      uint32_t v[16];
      tc_ld16(tmem + (static_cast<uint32_t>(32 * warp) << 16) + 16 * sb, v);
      tc_wait_ld();
      float x[kRows];
      bool exceed = false;
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        x[r] = valid ? __uint_as_float(v[r]) * p.scale_log2 : -INFINITY;
        exceed |= x[r] > m_used[r] + kRescaleThreshold;
      }
      tc_fence_before();
      const bool any_exceed = group_or(exceed);  // also: every warp has read S^T buffer sb
      if (threadIdx.x == 0) mbar_arrive(bar(B_SFREE + sb));
      float alpha[kRows];
#pragma unroll
      for (int r = 0; r < kRows; ++r) alpha[r] = 1.f;
      bool moved = false;
      if (any_exceed) {  // per-row maximum of the tile over the 128 tokens; move the rows it passes by > 2^8
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          float m = x[r];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == r) red_s[warp * kRows + r] = m;
        }
        group_sync();
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          const float tmax =
              fmaxf(fmaxf(red_s[r], red_s[kRows + r]), fmaxf(red_s[2 * kRows + r], red_s[3 * kRows + r]));
          if (tmax > m_used[r] + kRescaleThreshold) {
            alpha[r] = m_used[r] == -INFINITY ? 0.f : ex2(m_used[r] - tmax);
            m_used[r] = tmax;
            l_part[r] *= alpha[r];
            moved = true;
          }
        }
        group_sync();  // red_s is reused
      }
      const bool rescale = moved && !first;  // the same in every thread
      float pr[kRows];
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        pr[r] = m_used[r] == -INFINITY ? 0.f : ex2(x[r] - m_used[r]);
        l_part[r] += pr[r];
      }
      // P^T as the K-major B operand (N = 16 rows, K = 128 tokens, no swizzle): element (r, t) at
      // (r / 8) * 2048 + (t / 8) * 128 + (r % 8) * 16 + (t % 8) * 2. Lane pairs swap halves so the even
      // lane writes rows 0-7 and the odd lane rows 8-15 of tokens (t, t + 1), 4 bytes each.
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float other = __shfl_xor_sync(0xffffffffu, even ? pr[8 + i] : pr[i], 1);
        pk[i] = even ? pack_bf16(pr[i], other) : pack_bf16(other, pr[8 + i]);
      }
      // P^T buffer sb was last read by the P.V of tile j - 2
      if (j >= 2 && !group_wait(bar(B_PVDONE + sb), ((j >> 1) - 1) & 1, abort_s, err)) break;
      {
        const int te = tok & ~1;
        const uint32_t pb0 = base + kPOff + sb * kPBytes + (even ? 0 : 2048) + (te >> 3) * 128 + (te & 7) * 2;
#pragma unroll
        for (int i = 0; i < 8; ++i) asm volatile("st.shared.u32 [%0], %1;" ::"r"(pb0 + i * 16), "r"(pk[i]) : "memory");
      }
      fence_proxy_async_smem();
      // the correction warps copied slot sb's flag, alpha and 1/l of tile j - 2
      if (j >= 2 && !group_wait(bar(B_DACK + sb), ((j >> 1) - 1) & 1, abort_s, err)) break;
      if (rescale && threadIdx.x < kRows) {
        float a = alpha[0];
#pragma unroll
        for (int r = 1; r < kRows; ++r) a = r == static_cast<int>(threadIdx.x) ? alpha[r] : a;
        alpha_s[sb * kRows + threadIdx.x] = a;
      }
      if (tl.flags & F_END) {  // row sums over the 128 threads; 1/l and the LSE of each row
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          float s = l_part[r];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
          if (lane == r) red_s[warp * kRows + r] = s;
        }
        group_sync();
        if (threadIdx.x < kRows) {
          const int r = threadIdx.x;
          const float l = red_s[r] + red_s[kRows + r] + red_s[2 * kRows + r] + red_s[3 * kRows + r];
          linv_s[sb * kRows + r] = l > 0.f ? 1.f / l : 0.f;
          float mr = m_used[0];
#pragma unroll
          for (int rr = 1; rr < kRows; ++rr) mr = rr == r ? m_used[rr] : mr;
          const float lse2 = l > 0.f ? mr + log2f(l) : -INFINITY;  // base 2
          if (tl.flags & F_FINAL) {
            if (p.lse != nullptr) store_lse_nat(p, tl.b, tl.hg * kRows + r, lse2);
          } else {
            p.part_lse[slot_id(blockIdx.x, (tl.flags & F_SLOT1) ? 1 : 0) * kRows + r] = lse2;
          }
        }
      }
      group_sync();  // P^T, alpha and 1/l written by the whole group; red_s free again
      if (threadIdx.x == 0) {
        flag_s[sb] = rescale ? 1 : 0;
        mbar_arrive(bar(B_DEC + sb));
        if (!rescale) mbar_arrive(bar(B_PREADY + sb));
      }
      ++j;
    }
  } else if (warp < 8) {
    // ------------------------------------------------ correction, epilogue
    const int q = warp - 4;  // tensor-memory lanes 32 q .. 32 q + 31: dims 128 mb + 32 q + lane
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q) << 16) + 32;
    int j = 0, uses = 0;
    while (wk.next(tl, lane, err)) {
      const int sb = j & 1;
      if (!warp_wait(bar(B_DEC + sb), (j >> 1) & 1, abort_s, err, kErrTimeoutFull)) break;
      const bool fix = flag_s[sb] != 0, end = (tl.flags & F_END) != 0;
      float a[kRows], inv[kRows];
#pragma unroll
      for (int rr = 0; rr < kRows; ++rr) {
        a[rr] = fix ? alpha_s[sb * kRows + rr] : 1.f;
        inv[rr] = end ? linv_s[sb * kRows + rr] : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DACK + sb));  // slot sb may be reused for tile j + 2
      if (fix) {  // O^T *= alpha per row, after the P.V of tile j - 1
        if (!warp_wait(bar(B_PVDONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort_s, err, kErrTimeoutFull)) break;
        tc_fence_after();
#pragma unroll
        for (int mb = 0; mb < kDv / 128; ++mb) {
          uint32_t o[16];
          tc_ld16(trow + 16 * mb, o);
          tc_wait_ld();
#pragma unroll
          for (int rr = 0; rr < kRows; ++rr) o[rr] = __float_as_uint(__uint_as_float(o[rr]) * a[rr]);
          tc_st16(trow + 16 * mb, o);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_CORR));
        if (q == 0) {
          if (!warp_wait(bar(B_CORR), uses & 1, abort_s, err, kErrTimeoutFull)) break;
          if (lane == 0) mbar_arrive(bar(B_PREADY + sb));
        }
        ++uses;
      }
      if (end) {  // O = O^T / l after the piece's last P.V
        if (!warp_wait(bar(B_PVDONE + sb), (j >> 1) & 1, abort_s, err, kErrTimeoutFull)) break;
        tc_fence_after();
        const bool fin = (tl.flags & F_FINAL) != 0;
        const int64_t sid = slot_id(blockIdx.x, (tl.flags & F_SLOT1) ? 1 : 0);
#pragma unroll
        for (int mb = 0; mb < kDv / 128; ++mb) {
          uint32_t o[16];
          tc_ld16(trow + 16 * mb, o);
          tc_wait_ld();
          const int dim = 128 * mb + 32 * q + lane;
          if (fin) {
            __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.out) +
                                (static_cast<int64_t>(tl.b) * p.rows + tl.hg * kRows) * kDv + dim;
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) ob[rr * kDv] = __float2bfloat16(__uint_as_float(o[rr]) * inv[rr]);
          } else {
            float* po = p.part_o + sid * (kRows * kDv) + dim;
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) po[rr * kDv] = __uint_as_float(o[rr]) * inv[rr];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_CORR));
        if (q == 0) {
          if (!warp_wait(bar(B_CORR), uses & 1, abort_s, err, kErrTimeoutFull)) break;
          if (lane == 0) mbar_arrive(bar(B_OFREE));
        }
        ++uses;
      }
      ++j;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tc_dealloc(tmem, kCols);
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

}  // namespace

bool mla_tc_supported(int page_size) { return page_size > 0 && page_size % 32 == 0; }

bool mla_tc_encode(const MlaParams& p, MlaTcMaps* maps) {
  return encode_rows(&maps->kv, p.kv, static_cast<int64_t>(p.num_blocks) * p.page_size, box_rows_for(p.page_size)) &&
         encode_rows(&maps->q, p.q, static_cast<int64_t>(p.batch) * p.rows, kRows);
}

cudaError_t launch_mla_tc_decode(const MlaParams& p, const MlaTcMaps& maps, int ctas, cudaStream_t stream) {
  const bool br64 = box_rows_for(p.page_size) == 64;
  static int configured[64][2] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const int vi = br64 ? 1 : 0;
  if (dev >= 0 && dev < 64 && !configured[dev][vi]) {
    const cudaError_t e = br64 ? cudaFuncSetAttribute(gqa_mla_tc_decode_kernel<64>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)
                               : cudaFuncSetAttribute(gqa_mla_tc_decode_kernel<32>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev][vi] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return br64 ? cudaLaunchKernelEx(&cfg, gqa_mla_tc_decode_kernel<64>, p, maps)
              : cudaLaunchKernelEx(&cfg, gqa_mla_tc_decode_kernel<32>, p, maps);
}

}  // namespace gqa
