// C ABI of the paged GQA decode library: argument checks, device checks,
// workspace ownership and the launch sequence (decode kernel, then the LSE
// merge kernel with programmatic dependent launch). Mirrors the run() wrapper
// of the kernelindex.com page "gqa_paged_decode_h32_kv4_d128_ps1" minus its
// host-side moves and its kv_indptr[-1].item() synchronisation: every call is
// asynchronous on the caller's stream.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <chrono>
#include <mutex>

#include "gqa_kernels.h"
#include "gqa_paged_decode.h"
#include "gqa_plan.h"

namespace {

using gqa::KernelChoice;

constexpr int kMaxDevices = 64;
constexpr int kDefaultMinUnits = 32;
// Upper bound on tier-1 decode CTAs a tuning may ask for.
constexpr int kMaxDecodeCtas = 1536;
// Tier 2 by default: 2 CTAs per tier-1 CTA over the last 10 % of the units,
// at least 64 units each.
constexpr int kDefaultTier2PerTier1 = 2;
constexpr int kDefaultTier2Permille = 100;
constexpr int kDefaultTier2MinUnits = 64;
constexpr int kMaxTier2Ctas = 1 << 16;
// Tokens of work an extra piece adds to a CTA of the MLA tensor-memory kernel (the Q reload, the
// drained pipeline and the O epilogue at a sequence boundary: about 16 us at 64 rows, where a
// 128-token tile takes about 5 us), used to balance its CTA ranges.
constexpr int kMlaTcPieceCost = 400;
// Tokens per pipeline stage of the FP8-cache decode with a 2-deep ring.
constexpr int kDefaultF8Tile = 16;
constexpr int kSmemPerSm = 228 * 1024;
constexpr int kSmemReservedPerCta = 1024;
constexpr float kLog2e = 1.4426950408889634f;

struct DeviceState {
  bool queried = false;
  int sm_count = 0;
  int major = 0;
  int minor = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};

struct Tuning {
  int num_ctas = 0;
  int min_units = 0;
  int tier2_ctas = 0;       // -1: one tier; 0: kDefaultTier2PerTier1 per tier-1 CTA; > 0: this many
  int tier2_permille = kDefaultTier2Permille;
  int tier2_min_units = kDefaultTier2MinUnits;
  int fuse_max_splits = gqa::kDefaultFuseMaxSplits;
  KernelChoice kernel = {gqa::kGatherLsu, 4, 16, 2};
  int mla_kernel = gqa::kMlaKernelDefault;
  int merge_mode = 0;  // 0: decode grid + merge kernel; 1: one-wave decode with the merge inside it when possible
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
Tuning g_tune;
// Test hooks (gqa_paged_decode_test_fail_allocs / _test_wait_limit_ns): library
// workspace allocations still to fail as if cudaMalloc had failed, and the
// give-up limit of the TMA variant's bounded waits (0: the default).
int g_fail_allocs = 0;
unsigned long long g_wait_limit_ns = 0;
// Kernels launched by this host thread's latest decode call (see
// gqa_paged_decode_last_launch_count).
thread_local int t_last_launches = 0;
cudaEvent_t g_ev_start = nullptr;
cudaEvent_t g_ev_stop = nullptr;
// Ticket epoch of each call (never 0; 40 bits), so arrival tickets left by an
// earlier call on the same workspace read as empty. The counter starts at a
// value drawn from the clock, so a caller's workspace that holds small-integer
// or zero data (or tickets of another process) does not look like a live ticket.
std::atomic<unsigned long long> g_epoch{
    static_cast<unsigned long long>(std::chrono::steady_clock::now().time_since_epoch().count()) * 0x9E3779B97F4A7C15ull >>
    24};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Fills *st for the current device (cached). Returns a GQA_* code.
int current_device(int* dev_out, DeviceState** st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_LAUNCH;
  DeviceState& s = g_dev[dev];
  if (!s.queried) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return GQA_ERR_LAUNCH;
    s.sm_count = prop.multiProcessorCount;
    s.major = prop.major;
    s.minor = prop.minor;
    s.queried = true;
  }
  *dev_out = dev;
  *st = &s;
  if (s.major != 10 || s.minor != 3) return GQA_ERR_UNSUPPORTED_DEVICE;
  return GQA_OK;
}

int decode_ctas(const DeviceState& st, const Tuning& t) {
  if (t.num_ctas > 0) return t.num_ctas;
  const int smem = gqa::decode_smem_bytes(t.kernel);
  int per_sm = kSmemPerSm / (smem + kSmemReservedPerCta);
  const int cap = gqa::decode_max_ctas_per_sm(t.kernel);
  if (per_sm > cap) per_sm = cap;
  if (per_sm < 1) per_sm = 1;
  return st.sm_count * per_sm;
}

// The plan of a call; the grid is tier1_ctas + tier2_ctas CTAs.
gqa::PlanConfig plan_config(const DeviceState& st, const Tuning& t) {
  gqa::PlanConfig c;
  c.tier1_ctas = decode_ctas(st, t);
  c.tier2_ctas = t.tier2_ctas > 0 ? t.tier2_ctas : (t.tier2_ctas == 0 ? kDefaultTier2PerTier1 * c.tier1_ctas : 0);
  c.min_units = t.min_units > 0 ? t.min_units : kDefaultMinUnits;
  c.tier2_permille = t.tier2_permille;
  c.tier2_min_units = t.tier2_min_units;
  return c;
}

size_t partial_o_floats(int num_ctas, int ng) {
  return static_cast<size_t>(2) * num_ctas * ng * gqa::kGroup * gqa::kHeadDim;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

size_t partial_lse_bytes(int num_ctas, int ng) {
  return static_cast<size_t>(2) * num_ctas * ng * gqa::kGroup * sizeof(float);
}

size_t tickets_bytes(int num_ctas, int ng) { return static_cast<size_t>(num_ctas) * ng * sizeof(unsigned long long); }

size_t split_rec_bytes(int num_ctas) { return static_cast<size_t>(num_ctas) * 16; }

// Tier-2 range counters of the one-wave mode: one 8-byte word per warp index.
size_t grab_bytes() { return static_cast<size_t>(gqa::kKvHeads) * sizeof(unsigned long long); }

// Layout: partial O | partial LSE | arrival tickets | split records | tier-2
// range counters, each 256-byte aligned.
size_t workspace_bytes(int num_ctas, int ng) {
  const size_t o = partial_o_floats(num_ctas, ng) * sizeof(float);
  return round256(o) + round256(partial_lse_bytes(num_ctas, ng)) + round256(tickets_bytes(num_ctas, ng)) +
         round256(split_rec_bytes(num_ctas)) + round256(grab_bytes());
}

int check_args(const void* q, const void* k, const void* v, const int32_t* indptr, const int32_t* indices,
               float sm_scale, const void* out, const float* lse, int batch) {
  if (batch < 0) return GQA_ERR_INVALID_ARGUMENT;
  if (batch == 0) return GQA_OK;
  if (q == nullptr || indptr == nullptr || out == nullptr || lse == nullptr) return GQA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(sm_scale)) return GQA_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16)) return GQA_ERR_INVALID_ARGUMENT;
  if (!aligned(lse, 8) || !aligned(indptr, 4) || !aligned(indices, 4)) return GQA_ERR_INVALID_ARGUMENT;
  return GQA_OK;
}

// Selected-token batch: `rows` query rows of `topk` columns each, resolved
// through a block table (the decode then runs in sparse mode).
struct SparseJob {
  const int32_t* logical_indices;
  const int32_t* block_table;
  const int32_t* token_to_req;
  int topk, page_size, page_table_width, num_requests, num_cache_blocks;
};

// Grows the library-owned workspace of the current device to `need` bytes
// (caller holds g_mu). Returns a GQA_* code.
int library_workspace(DeviceState* st, size_t need, void** ws) {
  if (st->ws_bytes < need) {
    if (st->ws != nullptr) {
      // calls already queued may still read the old buffer
      if (cudaDeviceSynchronize() != cudaSuccess) return GQA_ERR_LAUNCH;
      cudaFree(st->ws);
      st->ws = nullptr;
      st->ws_bytes = 0;
    }
    const bool injected = g_fail_allocs > 0;  // a test hook stands in for a failing cudaMalloc
    if (injected) --g_fail_allocs;
    if (injected || cudaMalloc(&st->ws, need) != cudaSuccess) {
      if (!injected) cudaGetLastError();
      st->ws = nullptr;
      return GQA_ERR_WORKSPACE;
    }
    st->ws_bytes = need;
  }
  *ws = st->ws;
  return GQA_OK;
}

// fit_ws: a caller workspace too small for the tuned plan makes the plan use
// fewer tier-2 CTAs (down to none) instead of failing. sj: selected-token mode
// (indptr and indices unused; the library-owned workspace also holds the
// resolved slots).
int run(const void* q, const void* k, const void* v, const int32_t* indptr, const int32_t* indices, float sm_scale,
        void* out, float* lse, int batch, cudaStream_t stream, void* user_ws, size_t user_ws_bytes, bool checked,
        int num_pages, int* dev_err, bool fit_ws = false, const SparseJob* sj = nullptr, bool fp8 = false) {
  if (sj == nullptr) {
    const int rc0 = check_args(q, k, v, indptr, indices, sm_scale, out, lse, batch);
    if (rc0 != GQA_OK) return rc0;
  }
  int rc = GQA_OK;
  t_last_launches = 0;
  if (batch == 0) return GQA_OK;
  if (checked && (num_pages <= 0 || dev_err == nullptr || !aligned(dev_err, 4))) return GQA_ERR_INVALID_ARGUMENT;
  const int64_t sparse_total = sj != nullptr ? static_cast<int64_t>(batch) * sj->topk : 0;

  int dev = 0;
  DeviceState* st = nullptr;
  Tuning tune;
  gqa::PlanConfig cfg;
  cudaEvent_t ev0, ev1;
  void* ws = nullptr;
  unsigned long long wait_limit_ns = gqa::kDefaultWaitLimitNs;
  bool one_wave = false;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    rc = current_device(&dev, &st);
    if (rc != GQA_OK) return rc;
    tune = g_tune;
    if (g_wait_limit_ns > 0) wait_limit_ns = g_wait_limit_ns;
    if (sj != nullptr) tune.kernel = KernelChoice{gqa::kGatherLsu, 4, 16, 2};  // the one sparse variant
    if (fp8) {  // FP8 caches: the FP8 variant; a cp.async tuning with 4 heads per CTA picks its depth
      const KernelChoice& k = tune.kernel;
      if (k.gather != gqa::kGatherLsuF8) {
        const bool pick = k.gather == gqa::kGatherLsu && k.heads_per_cta == 4 && k.stages >= 2 && k.stages <= 4;
        const int stages = pick ? k.stages : 2;
        tune.kernel = KernelChoice{gqa::kGatherLsuF8, 4, stages == 2 ? kDefaultF8Tile : 16, stages};
      }
    } else if (tune.kernel.gather == gqa::kGatherLsuF8) {  // an FP8 tuning: bf16 caches take the default
      tune.kernel = KernelChoice{gqa::kGatherLsu, 4, 16, 2};
    }
    ev0 = g_ev_start;
    ev1 = g_ev_stop;
    cfg = plan_config(*st, tune);
    const int ng = tune.kernel.heads_per_cta;
    if (fit_ws && user_ws != nullptr) {
      while (cfg.tier2_ctas > 0 && workspace_bytes(cfg.tier1_ctas + cfg.tier2_ctas, ng) > user_ws_bytes) {
        const size_t per_cta = workspace_bytes(2, ng) - workspace_bytes(1, ng);
        const size_t over = workspace_bytes(cfg.tier1_ctas + cfg.tier2_ctas, ng) - user_ws_bytes;
        const int drop = static_cast<int>(over / (per_cta > 0 ? per_cta : 1)) + 1;
        cfg.tier2_ctas = cfg.tier2_ctas > drop ? cfg.tier2_ctas - drop : 0;
      }
    }
    // one wave (the tier-1 CTAs, all resident; tier 2 taken by their warps;
    // merge in the kernel) for the bf16 cp.async variants when the device holds
    // the whole grid and the warps can take all of tier 2
    if (tune.merge_mode == 1 && tune.kernel.gather == gqa::kGatherLsu &&
        cfg.tier2_ctas <= (gqa::kMaxWarpRanges - 1) * cfg.tier1_ctas &&
        cfg.tier1_ctas <= gqa::decode_coresident_ctas(tune.kernel, sj != nullptr))
      one_wave = true;
    const size_t need = workspace_bytes(cfg.tier1_ctas + cfg.tier2_ctas, ng) +
                        round256(static_cast<size_t>(sparse_total) * sizeof(int32_t));
    if (user_ws != nullptr) {
      if (user_ws_bytes < need || !aligned(user_ws, 256)) return GQA_ERR_WORKSPACE;
      ws = user_ws;
    } else {
      rc = library_workspace(st, need, &ws);
      if (rc != GQA_OK) return rc;
    }
  }

  const int ng = tune.kernel.heads_per_cta;
  const int ctas = cfg.tier1_ctas + cfg.tier2_ctas;
  float* part_o = static_cast<float*>(ws);
  const size_t lse_off = round256(partial_o_floats(ctas, ng) * sizeof(float));
  float* part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) + lse_off);
  const size_t tickets_off = lse_off + round256(partial_lse_bytes(ctas, ng));
  unsigned long long* tickets = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + tickets_off);
  const size_t rec_off = tickets_off + round256(tickets_bytes(ctas, ng));
  int4* split_rec = reinterpret_cast<int4*>(static_cast<char*>(ws) + rec_off);
  unsigned long long* grab =
      reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + rec_off + round256(split_rec_bytes(ctas)));
  const unsigned long long epoch = (g_epoch.fetch_add(1) % ((1ull << 40) - 1)) + 1;

  if (sj != nullptr) {  // resolve every selected column to its slot first
    int32_t* slots = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + workspace_bytes(ctas, ng));
    if (gqa::launch_sparse_resolve(sj->logical_indices, sj->block_table, sj->token_to_req, slots, batch, sj->topk,
                                   sj->page_size, sj->page_table_width, sj->num_requests, sj->num_cache_blocks,
                                   st->sm_count, stream) != cudaSuccess)
      return GQA_ERR_LAUNCH;
    indices = slots;
    indptr = nullptr;
  }

  if (checked) {
    if (cudaMemsetAsync(dev_err, 0, sizeof(int), stream) != cudaSuccess) return GQA_ERR_LAUNCH;
    if (gqa::launch_validate(indptr, indices, batch, num_pages, dev_err, stream) != cudaSuccess) return GQA_ERR_LAUNCH;
  }

  int* err_word = nullptr;
  if (gqa::device_error_word(&err_word) != cudaSuccess) return GQA_ERR_LAUNCH;

  gqa::DecodeParams dp{};
  dp.q = q;
  dp.k_cache = k;
  dp.v_cache = v;
  dp.kv_indptr = indptr;
  dp.kv_indices = indices;
  dp.out = out;
  dp.lse = lse;
  dp.part_o = part_o;
  dp.part_lse = part_lse;
  dp.skip_if_set = checked ? dev_err : nullptr;
  dp.err = err_word;
  dp.tickets = tickets;
  dp.epoch = epoch;
  dp.split_rec = split_rec;
  dp.fuse_max_splits = tune.fuse_max_splits;
  dp.batch = batch;
  dp.sparse_topk = sj != nullptr ? sj->topk : 0;
  dp.sparse_total = static_cast<int>(sparse_total);
  dp.plan = cfg;
  dp.scale_log2 = sm_scale * kLog2e;
  dp.num_pages_check = checked ? num_pages : 0;
  dp.wait_limit_ns = wait_limit_ns;
  dp.inline_merge = one_wave ? 1 : 0;
  dp.grab = grab;
  if (one_wave) dp.fuse_max_splits = 1;  // every split sequence is merged by the in-kernel duties

  const bool profile = ev0 != nullptr && ev1 != nullptr;
  if (profile && cudaEventRecord(ev0, stream) != cudaSuccess) return GQA_ERR_LAUNCH;
  // one wave: the tier-1 CTAs only, launched cooperatively. Otherwise the whole
  // grid; in selected-token mode the decode is then a programmatic dependent of
  // the resolve kernel unless events (or the checked path's validation) sit
  // between them.
  const int grid = one_wave ? cfg.tier1_ctas : ctas;
  const int launch = one_wave ? gqa::kLaunchCooperative
                              : (sj != nullptr && !profile && !checked ? gqa::kLaunchPdl : gqa::kLaunchPlain);
  const cudaError_t le = sj != nullptr ? gqa::launch_decode_lsu_sparse(dp, grid, stream, launch)
                                       : gqa::launch_decode(tune.kernel, dp, grid, stream, launch);
  if (le != cudaSuccess) return GQA_ERR_LAUNCH;
  if (profile && cudaEventRecord(ev1, stream) != cudaSuccess) return GQA_ERR_LAUNCH;
  const int before = (sj != nullptr ? 1 : 0) + (checked ? 1 : 0);  // slot resolution, validation
  if (one_wave) {  // the decode kernel merged the split sequences and wrote the empty ones
    t_last_launches = before + 1;
    return GQA_OK;
  }

  gqa::MergeParams mp{};
  mp.kv_indptr = indptr;
  mp.part_o = part_o;
  mp.part_lse = part_lse;
  mp.out = out;
  mp.lse = lse;
  mp.skip_if_set = checked ? dev_err : nullptr;
  mp.batch = batch;
  mp.sparse_topk = dp.sparse_topk;
  mp.sparse_total = dp.sparse_total;
  mp.plan = cfg;
  mp.split_rec = split_rec;
  mp.epoch = epoch;
  mp.use_pdl = profile ? 0 : 1;
  mp.fuse_max_splits = tune.fuse_max_splits;
  if (gqa::launch_merge(ng, mp, stream) != cudaSuccess) return GQA_ERR_LAUNCH;
  t_last_launches = before + 2;
  return GQA_OK;
}

bool valid_kernel(const KernelChoice& k) { return gqa::decode_smem_bytes(k) > 0; }

}  // namespace

namespace gqa {

int decode_in_scratch(const void* q, const void* k_cache, const void* v_cache, const int* kv_indptr,
                      const int* kv_indices, float sm_scale, void* out, float* lse, int batch, cudaStream_t stream,
                      void* scratch, size_t scratch_bytes) {
  if (scratch == nullptr && batch > 0) return GQA_ERR_WORKSPACE;
  return run(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream, scratch, scratch_bytes,
             false, 0, nullptr, true);
}

}  // namespace gqa

extern "C" {

int gqa_paged_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_indptr,
                     const int32_t* kv_indices, float sm_scale, void* out, float* lse, int batch,
                     struct CUstream_st* stream) {
  return run(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream, nullptr, 0, false, 0,
             nullptr);
}

size_t gqa_paged_decode_ws_size(int batch, int64_t total_tokens_upper_bound) {
  (void)batch;
  (void)total_tokens_upper_bound;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  DeviceState* st = nullptr;
  const int rc = current_device(&dev, &st);
  if (rc != GQA_OK && rc != GQA_ERR_UNSUPPORTED_DEVICE) return 0;
  const gqa::PlanConfig c = plan_config(*st, g_tune);
  return workspace_bytes(c.tier1_ctas + c.tier2_ctas, g_tune.kernel.heads_per_cta);
}

int gqa_paged_decode_ws(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_indptr,
                        const int32_t* kv_indices, float sm_scale, void* out, float* lse, int batch,
                        struct CUstream_st* stream, void* workspace, size_t workspace_bytes_) {
  if (workspace == nullptr && batch > 0) return GQA_ERR_WORKSPACE;
  return run(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream, workspace,
             workspace_bytes_, false, 0, nullptr);
}

int gqa_paged_decode_checked(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_indptr,
                             const int32_t* kv_indices, float sm_scale, void* out, float* lse, int batch,
                             struct CUstream_st* stream, int num_pages, int* dev_err) {
  return run(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream, nullptr, 0, true,
             num_pages, dev_err);
}

void gqa_paged_decode_release(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return;
  for (int d = 0; d < kMaxDevices; ++d) {
    if (g_dev[d].ws == nullptr) continue;
    if (cudaSetDevice(d) == cudaSuccess) {
      cudaDeviceSynchronize();
      cudaFree(g_dev[d].ws);
    }
    g_dev[d].ws = nullptr;
    g_dev[d].ws_bytes = 0;
  }
  cudaSetDevice(cur);
}

const char* gqa_paged_decode_strerror(int code) {
  switch (code) {
    case GQA_OK:
      return "success";
    case GQA_ERR_INVALID_ARGUMENT:
      return "invalid argument (null or misaligned pointer, negative batch, non-finite sm_scale or bad tuning)";
    case GQA_ERR_WORKSPACE:
      return "workspace allocation failed or the caller's workspace is too small";
    case GQA_ERR_LAUNCH:
      return "CUDA call or kernel launch failed";
    case GQA_ERR_UNSUPPORTED_DEVICE:
      return "unsupported device: the kernels are built for compute capability 10.3 (sm_103a)";
    default:
      return "unknown error code";
  }
}

int gqa_paged_decode_set_tuning(int num_ctas, int min_units_per_cta, int heads_per_cta, int tile, int stages,
                                int gather, int fused_merge_max_splits, int tier2_ctas, int tier2_permille,
                                int tier2_min_units) {
  if (num_ctas < 0 || min_units_per_cta < 0 || heads_per_cta < 0 || tile < 0 || stages < 0 || gather < 0)
    return GQA_ERR_INVALID_ARGUMENT;
  if (num_ctas > kMaxDecodeCtas || fused_merge_max_splits < -1) return GQA_ERR_INVALID_ARGUMENT;
  if (tier2_ctas < -1 || tier2_ctas > kMaxTier2Ctas || tier2_permille < 0 || tier2_permille > 900 ||
      tier2_min_units < 0)
    return GQA_ERR_INVALID_ARGUMENT;
  Tuning t;
  t.num_ctas = num_ctas;
  t.min_units = min_units_per_cta;
  t.tier2_ctas = tier2_ctas;
  t.tier2_permille = tier2_permille > 0 ? tier2_permille : kDefaultTier2Permille;
  t.tier2_min_units = tier2_min_units > 0 ? tier2_min_units : kDefaultTier2MinUnits;
  t.fuse_max_splits = fused_merge_max_splits == 0 ? gqa::kDefaultFuseMaxSplits
                                                  : (fused_merge_max_splits < 0 ? 1 : fused_merge_max_splits);
  t.kernel.gather = gather;
  t.kernel.heads_per_cta = heads_per_cta > 0 ? heads_per_cta : 4;
  if (gather == gqa::kGatherLsu) {
    t.kernel.tile = tile > 0 ? tile : 16;
    t.kernel.stages = stages > 0 ? stages : 2;
  } else if (gather == gqa::kGatherTma) {
    t.kernel.tile = tile > 0 ? tile : 16;
    t.kernel.stages = stages > 0 ? stages : (t.kernel.tile == 32 ? 3 : (t.kernel.heads_per_cta == 4 ? 5 : 4));
  } else if (gather == gqa::kGatherLsuCc) {
    t.kernel.tile = tile > 0 ? tile : 16;
    t.kernel.stages = stages > 0 ? stages : 2;
  } else if (gather == gqa::kGatherLsuF8) {
    t.kernel.tile = tile > 0 ? tile : kDefaultF8Tile;
    t.kernel.stages = stages > 0 ? stages : 2;
  } else {
    return GQA_ERR_INVALID_ARGUMENT;
  }
  if (!valid_kernel(t.kernel)) return GQA_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> lock(g_mu);
  t.mla_kernel = g_tune.mla_kernel;  // set by gqa_mla_set_tuning
  t.merge_mode = g_tune.merge_mode;  // set by gqa_paged_decode_set_merge_mode
  g_tune = t;
  return GQA_OK;
}

int gqa_paged_decode_last_launch_count(void) { return t_last_launches; }

int gqa_paged_decode_set_merge_mode(int mode) {
  if (mode != 0 && mode != 1) return GQA_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> lock(g_mu);
  g_tune.merge_mode = mode;
  return GQA_OK;
}

int gqa_mla_set_tuning(int kernel) {
  if (kernel != gqa::kMlaKernelDefault && kernel != gqa::kMlaKernelTensorMemory && kernel != gqa::kMlaKernelMma3 &&
      kernel != gqa::kMlaKernelMma4)
    return GQA_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> lock(g_mu);
  g_tune.mla_kernel = kernel;
  return GQA_OK;
}

int gqa_paged_decode_set_profile_events(void* decode_start, void* decode_stop) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_ev_start = static_cast<cudaEvent_t>(decode_start);
  g_ev_stop = static_cast<cudaEvent_t>(decode_stop);
  return GQA_OK;
}

int gqa_paged_kv_append(const void* k_new, const void* v_new, const int32_t* slots, void* k_cache, void* v_cache,
                        int num_tokens, int num_pages, struct CUstream_st* stream) {
  if (num_tokens < 0) return GQA_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return GQA_OK;
  if (k_new == nullptr || v_new == nullptr || slots == nullptr || k_cache == nullptr || v_cache == nullptr)
    return GQA_ERR_INVALID_ARGUMENT;
  if (num_pages <= 0) return GQA_ERR_INVALID_ARGUMENT;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slots, 4))
    return GQA_ERR_INVALID_ARGUMENT;
  int dev = 0;
  DeviceState* st = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    const int rc = current_device(&dev, &st);
    if (rc != GQA_OK) return rc;
  }
  return gqa::launch_kv_append(k_new, v_new, slots, k_cache, v_cache, num_tokens, num_pages, st->sm_count, stream) ==
                 cudaSuccess
             ? GQA_OK
             : GQA_ERR_LAUNCH;
}

int64_t gqa_paged_decode_plan(const int32_t* kv_indptr, int batch, int num_ctas, int min_units_per_cta,
                              int heads_per_cta, int tier2_ctas, int tier2_permille, int tier2_min_units,
                              int64_t* pieces, int64_t capacity) {
  if (kv_indptr == nullptr || batch < 0 || num_ctas <= 0 || min_units_per_cta < 0) return GQA_ERR_INVALID_ARGUMENT;
  if (tier2_ctas < 0 || tier2_ctas > kMaxTier2Ctas || tier2_permille < 0 || tier2_permille > 900 ||
      tier2_min_units < 0)
    return GQA_ERR_INVALID_ARGUMENT;
  if (heads_per_cta != 1 && heads_per_cta != 2 && heads_per_cta != 4) return GQA_ERR_INVALID_ARGUMENT;
  if (batch == 0) return 0;
  if (kv_indptr[0] != 0) return GQA_ERR_INVALID_ARGUMENT;
  for (int b = 0; b < batch; ++b) {
    if (kv_indptr[b + 1] < kv_indptr[b]) return GQA_ERR_INVALID_ARGUMENT;
  }
  const int64_t T = kv_indptr[batch];
  const int hg_count = gqa::kKvHeads / heads_per_cta;
  const int64_t W = T * hg_count;
  gqa::PlanConfig cfg;
  cfg.tier1_ctas = num_ctas;
  cfg.tier2_ctas = tier2_ctas;
  cfg.min_units = min_units_per_cta > 0 ? min_units_per_cta : kDefaultMinUnits;
  cfg.tier2_permille = tier2_permille > 0 ? tier2_permille : kDefaultTier2Permille;
  cfg.tier2_min_units = tier2_min_units > 0 ? tier2_min_units : kDefaultTier2MinUnits;
  const gqa::Plan pl = gqa::make_plan(W, cfg);
  int64_t n = 0;
  for (int64_t cta = 0; cta < static_cast<int64_t>(num_ctas) + tier2_ctas; ++cta) {
    const int64_t u0 = pl.begin(cta);
    const int64_t u1 = pl.end(cta);
    int64_t u = u0;
    while (u < u1) {
      const int64_t hg = u / T;
      const int64_t t = u - hg * T;
      const int64_t t_stop = (u1 - hg * T) < T ? (u1 - hg * T) : T;
      // largest b with kv_indptr[b] <= t (binary search; the table is non-decreasing)
      int lo = 0, hi = batch - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (kv_indptr[mid] <= t) lo = mid; else hi = mid - 1;
      }
      const int b = lo;
      const int64_t seq_lo = kv_indptr[b], seq_hi = kv_indptr[b + 1];
      const int64_t t_hi = seq_hi < t_stop ? seq_hi : t_stop;
      if (t_hi <= t) return GQA_ERR_INVALID_ARGUMENT;  // malformed table
      const bool whole = (t == seq_lo && t_hi == seq_hi);
      const int slot = whole ? -1 : (hg * T + t == u0 ? 0 : 1);
      const gqa::SeqSplit sp = gqa::seq_split(pl, hg * T + seq_lo, hg * T + seq_hi);
      if (n < capacity && pieces != nullptr) {
        int64_t* row = pieces + 9 * n;
        row[0] = cta;
        row[1] = b;
        row[2] = hg;
        row[3] = t;
        row[4] = t_hi;
        row[5] = slot;
        row[6] = sp.first_cta;
        row[7] = sp.last_cta;
        row[8] = sp.first_slot;
      }
      ++n;
      u = hg * T + t_hi;
    }
  }
  return n;
}

int gqa_sparse_paged_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* logical_indices,
                            const int32_t* block_table, const int32_t* token_to_req, float sm_scale, void* out,
                            float* lse, int rows, int topk, int page_size, int num_cache_blocks, int num_requests,
                            int page_table_width, struct CUstream_st* stream) {
  if (rows < 0) return GQA_ERR_INVALID_ARGUMENT;
  if (rows == 0) return GQA_OK;
  if (topk <= 0 || page_size <= 0 || num_cache_blocks <= 0 || num_requests <= 0 || page_table_width <= 0)
    return GQA_ERR_INVALID_ARGUMENT;
  if (static_cast<int64_t>(num_cache_blocks) * page_size > INT32_MAX) return GQA_ERR_INVALID_ARGUMENT;
  if (static_cast<int64_t>(rows) * topk > INT32_MAX) return GQA_ERR_INVALID_ARGUMENT;
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || out == nullptr || logical_indices == nullptr ||
      block_table == nullptr || token_to_req == nullptr)
    return GQA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(sm_scale)) return GQA_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return GQA_ERR_INVALID_ARGUMENT;
  if ((lse != nullptr && !aligned(lse, 8)) || !aligned(logical_indices, 4) || !aligned(block_table, 4) ||
      !aligned(token_to_req, 4))
    return GQA_ERR_INVALID_ARGUMENT;
  const SparseJob sj{logical_indices, block_table, token_to_req, topk, page_size, page_table_width, num_requests,
                     num_cache_blocks};
  return run(q, k_cache, v_cache, nullptr, nullptr, sm_scale, out, lse, rows, stream, nullptr, 0, false, 0, nullptr,
             false, &sj);
}

int gqa_paged_decode_fp8(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_indptr,
                         const int32_t* kv_indices, float sm_scale, void* out, float* lse, int batch,
                         struct CUstream_st* stream) {
  return run(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream, nullptr, 0, false, 0,
             nullptr, false, nullptr, true);
}

int gqa_mla_decode(const void* q, const void* kv_cache, const int32_t* block_table, const int32_t* cache_seqlens,
                   float softmax_scale, void* out, float* lse, int batch, int s_q, int h_q, int page_size,
                   int num_blocks, int page_table_width, struct CUstream_st* stream) {
  if (batch < 0) return GQA_ERR_INVALID_ARGUMENT;
  if (batch == 0) return GQA_OK;
  if (s_q <= 0 || h_q <= 0 || page_size <= 0 || num_blocks <= 0 || page_table_width <= 0)
    return GQA_ERR_INVALID_ARGUMENT;
  const int64_t rows = static_cast<int64_t>(s_q) * h_q;
  if (rows % 16 != 0 || rows > (1 << 20)) return GQA_ERR_INVALID_ARGUMENT;
  if (static_cast<int64_t>(num_blocks) * page_size > INT32_MAX) return GQA_ERR_INVALID_ARGUMENT;
  const int64_t max_tokens = static_cast<int64_t>(batch) * page_table_width * page_size;  // bound on sum(seqlens)
  if (max_tokens > INT32_MAX || max_tokens * (rows / 16) > (int64_t{1} << 40)) return GQA_ERR_INVALID_ARGUMENT;
  if (q == nullptr || kv_cache == nullptr || block_table == nullptr || cache_seqlens == nullptr || out == nullptr)
    return GQA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(softmax_scale)) return GQA_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(block_table, 4) ||
      !aligned(cache_seqlens, 4) || (lse != nullptr && !aligned(lse, 4)))
    return GQA_ERR_INVALID_ARGUMENT;

  DeviceState* st = nullptr;
  int dev = 0;
  gqa::PlanConfig cfg;
  void* ws = nullptr;
  size_t off_indptr = 0, off_slots = 0, off_po = 0, off_pl = 0, off_rec = 0, off_cost = 0, off_bounds = 0;
  bool balanced = false;
  gqa::MlaParams mp{};
  mp.q = q;
  mp.kv = kv_cache;
  mp.batch = batch;
  mp.rows = static_cast<int>(rows);
  mp.block_table = block_table;
  mp.width = page_table_width;
  mp.page_size = page_size;
  mp.num_blocks = num_blocks;
  int mla_kind = gqa::kMlaKernelDefault;
  gqa::MlaTcMaps maps;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    int rc = current_device(&dev, &st);
    if (rc != GQA_OK) return rc;
    const Tuning& t = g_tune;
    mla_kind = t.mla_kernel;
    // default: the tensor-memory kernel when a sequence's rows come in multiples of 32 (one pass over the
    // latent rows serves 32 or 64 rows, where the mma.sync kernel reads them once per 16; measured faster
    // from 32 rows up), mma.sync otherwise (faster at 16 rows)
    mp.piece_rows = 16;
    if (mla_kind == gqa::kMlaKernelDefault)
      mla_kind = rows % 32 == 0 ? gqa::kMlaKernelTensorMemory : gqa::kMlaKernelMma3;
    if (mla_kind == gqa::kMlaKernelTensorMemory) {
      // where the block size allows it (and Q rows fit the 32-bit box coordinates); else the mma.sync kernel
      mp.piece_rows = gqa::mla_tc_piece_rows(static_cast<int>(rows));
      const bool tc = gqa::mla_tc_supported(page_size) && static_cast<int64_t>(batch) * rows < INT32_MAX &&
                      gqa::mla_tc_encode(mp, &maps);
      if (!tc) mp.piece_rows = 16;
      mla_kind = tc ? gqa::kMlaKernelTensorMemory : gqa::kMlaKernelMma3;
    }
    cfg.tier1_ctas = t.num_ctas > 0 ? t.num_ctas : st->sm_count * gqa::mla_ctas_per_sm(mla_kind);  // one wave
    // one tier unless the tuning asks for tier 2: the MLA merge walks a sequence's pieces in turn
    cfg.tier2_ctas = t.tier2_ctas > 0 ? t.tier2_ctas : 0;
    cfg.min_units = t.min_units > 0 ? t.min_units : kDefaultMinUnits;
    cfg.tier2_permille = t.tier2_permille;
    cfg.tier2_min_units = t.tier2_min_units;
    const size_t ctas = static_cast<size_t>(cfg.tier1_ctas) + cfg.tier2_ctas;
    off_indptr = 0;
    off_slots = round256(static_cast<size_t>(batch + 1) * 4);
    off_po = off_slots + round256(static_cast<size_t>(max_tokens) * 4);
    const size_t pr = static_cast<size_t>(mp.piece_rows);
    off_pl = off_po + round256(2 * ctas * pr * 512 * sizeof(float));
    off_rec = off_pl + round256(2 * ctas * pr * sizeof(float));
    // the tensor-memory kernel with one tier: CTA ranges balanced by the scan for the cost of pieces
    // (the scan's 32-bit cost prefix must hold every token plus the piece cost of every sequence)
    balanced = mla_kind == gqa::kMlaKernelTensorMemory && cfg.tier2_ctas == 0 &&
               max_tokens + static_cast<int64_t>(batch) * kMlaTcPieceCost <= INT32_MAX;
    off_cost = off_rec + round256(2 * ctas * 16);
    off_bounds = off_cost + round256(static_cast<size_t>(batch + 1) * 4);
    const size_t need = off_bounds + round256((ctas + 1) * sizeof(int64_t));
    rc = library_workspace(st, need, &ws);
    if (rc != GQA_OK) return rc;
  }
  char* wsb = static_cast<char*>(ws);
  int* err_word = nullptr;
  if (gqa::device_error_word(&err_word) != cudaSuccess) return GQA_ERR_LAUNCH;
  mp.kv_indptr_mut = reinterpret_cast<int*>(wsb + off_indptr);
  mp.kv_indptr = mp.kv_indptr_mut;
  mp.slots_mut = reinterpret_cast<int*>(wsb + off_slots);
  mp.slots = mp.slots_mut;
  mp.out = out;
  mp.lse = lse;
  mp.part_o = reinterpret_cast<float*>(wsb + off_po);
  mp.part_lse = reinterpret_cast<float*>(wsb + off_pl);
  mp.split_rec = reinterpret_cast<int4*>(wsb + off_rec);
  mp.cost_ptr = reinterpret_cast<int*>(wsb + off_cost);
  mp.bounds = balanced ? reinterpret_cast<int64_t*>(wsb + off_bounds) : nullptr;
  mp.piece_cost = kMlaTcPieceCost;
  mp.err = err_word;
  mp.plan = cfg;
  mp.epoch = (g_epoch.fetch_add(1) % ((1ull << 40) - 1)) + 1;
  mp.h_q = h_q;
  mp.s_q = s_q;
  mp.scale_log2 = softmax_scale * kLog2e;
  return gqa::launch_mla(mp, cache_seqlens, mla_kind, &maps, stream) == cudaSuccess
             ? GQA_OK
             : GQA_ERR_LAUNCH;
}

int gqa_paged_decode_test_fail_allocs(int count) {
  if (count < 0) return GQA_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> lock(g_mu);
  g_fail_allocs = count;
  return GQA_OK;
}

int gqa_paged_decode_test_wait_limit_ns(uint64_t ns) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_wait_limit_ns = ns;
  return GQA_OK;
}

int gqa_paged_decode_device_error(int* flags) {
  if (flags == nullptr) return GQA_ERR_INVALID_ARGUMENT;
  if (cudaDeviceSynchronize() != cudaSuccess) return GQA_ERR_LAUNCH;
  return gqa::read_and_clear_device_error(flags) == cudaSuccess ? GQA_OK : GQA_ERR_LAUNCH;
}

}  // extern "C"
