/*
 * gqa_paged_decode.h -- C ABI of the GB300 (sm_103a) paged-KV GQA decode library.
 *
 * The operation is the one stated by the FlashInfer-style problem on the
 * kernelindex.com page "gqa_paged_decode_h32_kv4_d128_ps1" (its kernel and the
 * run() docstring): batched decode attention with grouped-query attention,
 * 32 query heads over 4 KV heads (query head h reads KV head h / 8), head
 * dimension 128, page size 1, bf16 inputs, KV pages addressed through a CSR
 * page table. For every sequence b with n_b = kv_indptr[b+1] - kv_indptr[b]
 * tokens, page p_j = kv_indices[kv_indptr[b] + j] and query head h:
 *
 *   s_j       = sm_scale * dot(q[b,h,:], k_cache[p_j,0,h/8,:])
 *   out[b,h,:] = sum_j softmax(s)_j * v_cache[p_j,0,h/8,:]        (bf16, RNE)
 *   lse[b,h]  = log2(sum_j exp(s_j))                              (fp32)
 *
 * An empty sequence (n_b == 0) gives out[b,:,:] = 0 and lse[b,:] = -inf (the
 * early-exit step of that page's kernel). The log-sum-exp is base 2 of a
 * natural-exponent sum, as that kernel stores it.
 *
 * Layouts (all row-major, contiguous, device memory owned by the caller):
 *   q          [batch][32][128]          bf16, 16-byte aligned
 *   k_cache    [num_pages][1][4][128]    bf16, 16-byte aligned
 *   v_cache    [num_pages][1][4][128]    bf16, 16-byte aligned
 *   kv_indptr  [batch + 1]               int32, kv_indptr[0] == 0, non-decreasing
 *   kv_indices [kv_indptr[batch]]        int32, each in [0, num_pages)
 *   out        [batch][32][128]          bf16, 16-byte aligned (written)
 *   lse        [batch][32]               fp32, 8-byte aligned (written)
 *
 * k_cache, v_cache and kv_indices may be NULL only when kv_indptr[batch] == 0.
 *
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 * stream) and never synchronise the host: the kv_indptr / kv_indices
 * preconditions are not checked by gqa_paged_decode (see
 * gqa_paged_decode_checked). The library owns only its workspace (fp32 split
 * partials); calls that share the library-owned workspace must be ordered on
 * one stream. Calls on different streams at the same time must each pass
 * their own workspace through gqa_paged_decode_ws.
 *
 * Return codes: 0 success; negative values below. No exception crosses the ABI.
 */
#ifndef GQA_PAGED_DECODE_H_
#define GQA_PAGED_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is struct CUstream_st* */

#define GQA_OK 0
#define GQA_ERR_INVALID_ARGUMENT (-1)   /* null/misaligned pointer, batch < 0, non-finite sm_scale, bad tuning */
#define GQA_ERR_WORKSPACE (-2)          /* workspace allocation failed or caller workspace too small */
#define GQA_ERR_LAUNCH (-3)             /* a CUDA call or kernel launch failed */
#define GQA_ERR_UNSUPPORTED_DEVICE (-4) /* not a compute capability 10.3 (GB300) device */

/*
 * Paged GQA decode (the problem's run(q, k_cache, v_cache, kv_indptr,
 * kv_indices, sm_scale) with caller-allocated out / lse). Launches, in order
 * on `stream`: the split-KV decode kernel (each CTA streams an equal share of
 * all cached tokens, split points chosen on the device from kv_indptr) and the
 * LSE merge kernel (combines the pieces of sequences cut at a CTA boundary and
 * writes empty sequences). batch == 0 returns 0 without launching anything.
 * sm_scale is used as given (the problem's default is 1/sqrt(128)).
 */
int gqa_paged_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_indptr,
                     const int32_t* kv_indices, float sm_scale, void* out, float* lse, int batch,
                     struct CUstream_st* stream);

/*
 * Workspace bytes gqa_paged_decode_ws needs on the current device with the
 * current tuning. The split plan bounds the partials by the number of decode
 * CTAs (two slots each), so the size does not grow with batch or
 * total_tokens_upper_bound; both are accepted so callers can size for a
 * workload. Returns 0 if the device cannot be queried.
 */
size_t gqa_paged_decode_ws_size(int batch, int64_t total_tokens_upper_bound);

/*
 * As gqa_paged_decode, with a caller-owned device workspace of at least
 * gqa_paged_decode_ws_size() bytes (256-byte aligned). Returns
 * GQA_ERR_WORKSPACE if it is too small. Use one workspace per concurrent stream.
 */
int gqa_paged_decode_ws(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_indptr,
                        const int32_t* kv_indices, float sm_scale, void* out, float* lse, int batch,
                        struct CUstream_st* stream, void* workspace, size_t workspace_bytes);

/*
 * Debug variant: first checks on the device that kv_indptr starts at 0 and
 * never decreases and that every kv_indices entry lies in [0, num_pages).
 * The result is written to the caller's device int `dev_err` (0 = valid,
 * otherwise bit 4 = bad page id, bit 8 = bad kv_indptr); if it is nonzero the
 * decode and merge kernels return without reading K/V or writing out/lse.
 * Read dev_err after synchronising `stream`. num_pages must be > 0.
 */
int gqa_paged_decode_checked(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_indptr,
                             const int32_t* kv_indices, float sm_scale, void* out, float* lse, int batch,
                             struct CUstream_st* stream, int num_pages, int* dev_err);

/* Free the library-owned workspace on every device (synchronises those devices). */
void gqa_paged_decode_release(void);

/* Static description of a return code. */
const char* gqa_paged_decode_strerror(int code);

/*
 * Tuning for tests and benchmarks (process-wide; 0 keeps the default):
 * num_ctas - tier-1 decode CTAs per call, at most 1536 (default: SMs x CTAs
 *   per SM, one resident wave);
 * min_units_per_cta - smallest share of (token, head group) units a tier-1
 *   CTA takes (default 32); smaller values cut sequences into more pieces;
 * heads_per_cta - KV heads per CTA: 4, 2 or 1 (one warp per KV head);
 * tile, stages - tokens per pipeline stage and ring depth;
 * gather - 0: every warp gathers its own 256-byte K/V head rows with 16-byte
 *   cp.async (default: heads 4, tile 16, stages 2, 3 CTAs per SM);
 *   1: one producer warp per CTA gathers whole page rows with TMA bulk copies
 *   (tile 16 or 32);
 *   3: gather 0's pipeline (heads 4, tile 16, stages 2) with both contractions
 *   on the CUDA cores (fp32 FMAs) instead of mma.sync, a variant kept for
 *   comparing the two on this part;
 * fused_merge_max_splits - a sequence cut into at most this many pieces is
 *   merged by the decode kernel itself (the warp that finishes its last piece
 *   combines them); longer splits go to the merge kernel; default and -1: every
 *   split sequence goes to the merge kernel;
 * tier2_ctas - CTAs of the second tier, which takes the last tier2_permille
 *   thousandths of the units in small ranges that SMs finishing their tier-1
 *   range early pick up (default 2 per tier-1 CTA; -1: one tier only, at most
 *   65536);
 * tier2_permille - share of the units set aside for tier 2 (default 100,
 *   at most 900);
 * tier2_min_units - smallest share a tier-2 CTA takes (default 64).
 * Returns GQA_ERR_INVALID_ARGUMENT for a combination that is not compiled in
 * or a value out of range.
 */
int gqa_paged_decode_set_tuning(int num_ctas, int min_units_per_cta, int heads_per_cta, int tile, int stages,
                                int gather, int fused_merge_max_splits, int tier2_ctas, int tier2_permille,
                                int tier2_min_units);

/*
 * How a call combines the split pieces of its sequences (process-wide, for
 * tests and benchmarks):
 * 0 - default: a grid of every tier-1 and tier-2 decode CTA, followed by the
 *     LSE merge kernel (a programmatic dependent of the decode grid).
 * 1 - one wave: the decode kernel is launched cooperatively with only its
 *     tier-1 CTAs (one per resident slot); their warps take the tier-2 ranges
 *     from counters in the workspace, publish a record of where each range's
 *     last sequence is cut, and after their stream merge the sequences cut at
 *     their share of the boundaries and write the empty sequences, so a call is
 *     a single kernel. Used for the bf16 cp.async variants (dense and
 *     selected-token) when the device holds every tier-1 CTA at once and
 *     tier2_ctas is at most 15 per tier-1 CTA; otherwise (and for the
 *     TMA-gather variant and FP8 caches) a call runs as in 0. Its
 *     stream is as fast as mode 0's decode kernel, but its in-kernel merge
 *     (one warp per share, a chain of dependent round trips) ends later than
 *     the merge kernel, so it is not the default.
 * Returns GQA_ERR_INVALID_ARGUMENT for another value.
 */
int gqa_paged_decode_set_merge_mode(int mode);

/*
 * Kernels launched by the calling host thread's most recent call of
 * gqa_paged_decode, _ws, _checked, _noalloc, _fp8 or gqa_sparse_paged_decode
 * (0 if it launched none, for example batch == 0 or an error before launch):
 * 2 with the merge kernel (the default), 1 in the one-wave mode, plus one for the slot
 * resolution of a selected-token call and one for the checked call's
 * validation. For tests and benchmarks.
 */
int gqa_paged_decode_last_launch_count(void);

/*
 * Profiling hook: when both are non-NULL (cudaEvent_t handles), every later
 * call records `decode_start` just before and `decode_stop` just after the
 * decode kernel on its stream (the merge launch then waits for the decode
 * grid to finish instead of overlapping its launch). Pass NULLs to clear.
 */
int gqa_paged_decode_set_profile_events(void* decode_start, void* decode_stop);

/*
 * KV-cache append: the step that runs before each decode to store the new
 * tokens' K and V. The row store of the split-K GQA path on the sigit.si vLLM
 * "qsa.py" page (_store_qsa_rows_kernel / qsa_store_cache_rows) with page size
 * 1: for r < num_tokens, if 0 <= slots[r] < num_pages then
 *   k_cache[slots[r], 0, :, :] = k_new[r, :, :] and v_cache[slots[r], 0, :, :] = v_new[r, :, :];
 * other slots (for example -1 for padding tokens) store nothing.
 * k_new, v_new: [num_tokens][4][128] bf16, 16-byte aligned; slots: [num_tokens]
 * int32; k_cache, v_cache: [num_pages][1][4][128] bf16, 16-byte aligned, updated
 * in place. Valid slots should be distinct: when two rows name the same page,
 * which one it keeps is unspecified. Asynchronous on `stream`; num_tokens == 0
 * returns 0 without launching.
 */
int gqa_paged_kv_append(const void* k_new, const void* v_new, const int32_t* slots, void* k_cache, void* v_cache,
                        int num_tokens, int num_pages, struct CUstream_st* stream);

/*
 * Host-side view of the split plan (no GPU needed): for a host copy of
 * kv_indptr, the pieces that num_ctas tier-1 plus tier2_ctas tier-2 decode
 * CTAs cut the batch into, with the same arithmetic the decode and merge
 * kernels use (tier2_ctas = 0: one tier; tier2_permille and tier2_min_units
 * as in gqa_paged_decode_set_tuning, 0 = default). Writes up to `capacity`
 * rows of 9 int64 to `pieces`: decode CTA, sequence, head group, first and
 * one-past-last token (sequence-relative to kv_indices), partial slot (-1 for
 * a whole sequence written directly, else 0 / 1), and the merge kernel's view
 * of that sequence: first CTA, last CTA, slot of the first CTA's piece.
 * min_units_per_cta = 0 means the default (32). Returns the number of pieces
 * (which may exceed capacity) or GQA_ERR_INVALID_ARGUMENT.
 */
int64_t gqa_paged_decode_plan(const int32_t* kv_indptr, int batch, int num_ctas, int min_units_per_cta,
                              int heads_per_cta, int tier2_ctas, int tier2_permille, int tier2_min_units,
                              int64_t* pieces, int64_t capacity);

/*
 * gqa_paged_decode over an FP8 KV cache. The cache format follows the FP8
 * cache of the flash_mla_with_kvcache page (docs.flagos.io, FlagGems):
 * float8_e4m3 values followed by one float32 scale per 128 values, a value
 * being e4m3 * scale. For this shape one token row of k_cache (and of
 * v_cache) is 528 bytes: the e4m3 codes of KV heads 0..3 (128 each,
 * head-major, bytes 0..511), then the 4 heads' little-endian float32 scales
 * (bytes 512..527). k_cache, v_cache: [num_pages][528] bytes, 16-byte
 * aligned; every other argument, the result (bf16 O, fp32 base-2 LSE) and
 * the error behaviour are those of gqa_paged_decode.
 *
 * The kernel converts e4m3 to f16 exactly, takes each token's K scale on its
 * score and its V scale on its probability, and computes Q.K and P.V with f16
 * tensor-core operands (Q rescaled by a power of two per KV head so that it
 * cannot overflow f16). It uses 4 KV heads per CTA; a tuning with 4 heads per
 * CTA and 2-4 stages sets its ring depth (default 2).
 */
int gqa_paged_decode_fp8(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_indptr,
                         const int32_t* kv_indices, float sm_scale, void* out, float* lse, int batch,
                         struct CUstream_st* stream);

/*
 * Dense MLA paged decode: the dense decode of the flash_mla_with_kvcache page
 * (docs.flagos.io, FlagGems; flash_mla_with_kvcache without sparse indices),
 * for one latent KV head of d_qk = 576 values per token (512 "NoPE" values,
 * which are also V, then 64 "RoPE" values) and d_v = 512.
 *
 * For sequence b, query token i < s_q and head h < h_q, over the cached
 * tokens t < cache_seqlens[b] at kv_cache[block_table[b * page_table_width
 * + t / page_size]][t % page_size][0][:]:
 * s_t = softmax_scale * q[b][i][h][:] . kv_t[:] (all 576 values),
 * out[b][i][h][:] = sum_t softmax(s)_t kv_t[0:512] (bf16) and, when lse is
 * not NULL, lse[b][h][i] = log sum_t exp(s_t) (natural log, fp32; the page's
 * layout). Not causal within the s_q query tokens (the page's dense kernel
 * supports causal masking only for s_q = 1, where it changes nothing). A
 * sequence with no cached token gives out = 0 and lse = -inf; a token whose
 * block-table entry lies outside [0, num_blocks) is left out.
 *
 * Layouts (caller-owned device memory, contiguous): q [batch][s_q][h_q][576]
 * bf16 and out [batch][s_q][h_q][512] bf16, 16-byte aligned; kv_cache
 * [num_blocks][page_size][1][576] bf16, 16-byte aligned; block_table
 * [batch][page_table_width] int32; cache_seqlens [batch] int32; lse
 * [batch][h_q][s_q] fp32 or NULL. s_q * h_q must be a multiple of 16; a
 * length above page_table_width * page_size counts as that (the tokens past
 * the table have no block); negative lengths count as 0;
 * num_blocks * page_size and batch * page_table_width * page_size must be
 * below 2^31. Asynchronous on `stream`; batch == 0 returns 0 without
 * launching. Uses the library-owned workspace (CSR offsets, one slot per
 * cached token, fp32 partials). Returns GQA_OK, GQA_ERR_INVALID_ARGUMENT,
 * GQA_ERR_WORKSPACE, GQA_ERR_LAUNCH or GQA_ERR_UNSUPPORTED_DEVICE.
 */
int gqa_mla_decode(const void* q, const void* kv_cache, const int32_t* block_table, const int32_t* cache_seqlens,
                   float softmax_scale, void* out, float* lse, int batch, int s_q, int h_q, int page_size,
                   int num_blocks, int page_table_width, struct CUstream_st* stream);

/*
 * Kernel choice of gqa_mla_decode for tests and benchmarks (process-wide):
 * 0 - default: the tensor-memory kernel when s_q * h_q is a multiple of 32 and
 *     page_size a multiple of 32 (one pass over the latent rows serves 32 or
 *     64 query rows); otherwise the mma.sync kernel with a 3-stage ring;
 * 1 - the tensor-memory kernel (tcgen05 MMAs into tensor memory with 128
 *     tokens on M, 2D tensor copies of the latent rows, one CTA per SM; pieces
 *     of 64 query rows when s_q * h_q is a multiple of 64, else 32 when it is a
 *     multiple of 32, else 16) when page_size is a multiple of 32, else the
 *     mma.sync kernel;
 * 3, 4 - the mma.sync kernel (16-row pieces) with a 3-stage ring (three CTAs
 *     per SM) or a 4-stage ring (two CTAs per SM).
 * The tier settings of gqa_paged_decode_set_tuning (tier-1 CTAs, smallest
 * share, tier 2) apply to gqa_mla_decode as well; with num_ctas 0 it takes one
 * CTA per resident slot. Returns GQA_ERR_INVALID_ARGUMENT for another value.
 */
int gqa_mla_set_tuning(int kernel);

/*
 * Selected-token (sparse) paged GQA decode: the sparse split-K GQA path of
 * the sigit.si vLLM "qsa.py" page (qsa_sparse_paged_attention and its
 * _qsa_sparse_paged_gqa_splitk_kernel), for 32 query heads over 4 KV heads
 * of dimension 128.
 *
 * Query row r (of `rows`) belongs to request req = token_to_req[r] and
 * selects `topk` logical token positions t = logical_indices[r * topk + c] of
 * that request. Column c is used when 0 <= req < num_requests, t >= 0,
 * t / page_size < page_table_width, and the physical page
 * p = block_table[req * page_table_width + t / page_size] satisfies
 * 0 <= p < num_cache_blocks; its key and value rows for KV head g are then
 * k_cache[p][t % page_size][g][:] and v_cache[...]. Other columns (for
 * example -1 padding) are left out. Per query head h (KV head h / 8):
 * out[r][h] = softmax over the used columns of sm_scale * q[r][h] . k, times
 * v, in bf16 (a column listed twice counts twice), and, when lse is not NULL,
 * lse[r][h] = log2 sum exp(s) in fp32. A row with no used column gives
 * out = 0 and lse = -inf.
 *
 * Layouts (all device memory owned by the caller, contiguous): q, out
 * [rows][32][128] bf16, 16-byte aligned; k_cache, v_cache
 * [num_cache_blocks][page_size][4][128] bf16, 16-byte aligned;
 * logical_indices [rows][topk] int32; block_table
 * [num_requests][page_table_width] int32; token_to_req [rows] int32; lse
 * [rows][32] fp32 (8-byte aligned) or NULL. The page fixes sm_scale at
 * 1/sqrt(128); here it is an argument.
 *
 * Asynchronous on `stream`. Needs topk, page_size, num_cache_blocks,
 * num_requests, page_table_width > 0, num_cache_blocks * page_size and
 * rows * topk below 2^31; rows == 0 returns 0 without launching. Runs the
 * 4-KV-heads-per-CTA, 2-stage decode variant whatever the tuning's kernel
 * choice (the tuning's CTA counts and tiers apply). Uses the library-owned
 * workspace, which also holds rows * topk resolved slots (4 bytes each).
 * Returns GQA_OK, GQA_ERR_INVALID_ARGUMENT, GQA_ERR_WORKSPACE,
 * GQA_ERR_LAUNCH or GQA_ERR_UNSUPPORTED_DEVICE.
 */
int gqa_sparse_paged_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* logical_indices,
                            const int32_t* block_table, const int32_t* token_to_req, float sm_scale, void* out,
                            float* lse, int rows, int topk, int page_size, int num_cache_blocks, int num_requests,
                            int page_table_width, struct CUstream_st* stream);

/*
 * Synchronise the current device, then read and clear the sticky device error
 * word: bit 1 / 2 = a pipeline wait of the TMA-gather decode variant or the
 * tensor-memory MLA kernel gave up (after ~2 s by default; the kernel drained
 * its copies in flight and returned early, so that call's outputs are not
 * valid), bit 4 = bad page id, bit 8 = bad kv_indptr, bit 16 = an arrival or
 * range counter could not be claimed, bit 32 = an in-kernel merge gave up
 * waiting for a sequence's pieces (that sequence's outputs are not valid).
 * 0 means no error.
 */
int gqa_paged_decode_device_error(int* flags);

/*
 * Test hooks for the library's failure paths; production code has no reason
 * to call them. Both are process-wide.
 *
 * gqa_paged_decode_test_fail_allocs(count): the next `count` allocations of
 * the library-owned workspace fail exactly as a failing cudaMalloc would (the
 * call returns GQA_ERR_WORKSPACE without launching and without writing out /
 * lse; the device workspace is left unallocated). 0 turns it off. Returns
 * GQA_ERR_INVALID_ARGUMENT for count < 0.
 *
 * gqa_paged_decode_test_wait_limit_ns(ns): the give-up limit, in
 * nanoseconds, of the bounded waits of the decode kernels: the mbarrier waits
 * of the TMA-gather variant (gather = 1 in gqa_paged_decode_set_tuning) and,
 * in the one-wave mode, a warp's wait for the pieces of a sequence it merges.
 * 0 restores the default of 2 s. A wait that runs out sets bit 1, 2 or 32 of
 * the device error word; a TMA-variant CTA returns after its copies in flight
 * have landed (that drain keeps the 2 s limit), a merging warp skips that
 * merge. A call made with a tiny limit therefore completes, with outputs that
 * are not valid.
 */
int gqa_paged_decode_test_fail_allocs(int count);
int gqa_paged_decode_test_wait_limit_ns(uint64_t ns);

/*
 * The pages this library follows have no counterpart to this entry point: it
 * is an addition for callers that must not allocate device memory, such as a
 * serving runtime that reserves all free HBM for its KV-cache pool up front, a
 * caller inside CUDA stream capture (cudaMalloc cannot be captured), or a
 * latency-critical loop that cannot take cudaMalloc's device-wide
 * synchronisation. Same arguments and results as gqa_paged_decode, but the
 * split partials live in a fixed device array of GQA_NOALLOC_SCRATCH_BYTES
 * that every GPU loading the library holds until the process exits; the call
 * allocates nothing (no cudaMalloc / cudaFree, directly or through a library).
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture. When the current device and tuning need more scratch than
 * GQA_NOALLOC_SCRATCH_BYTES (gqa_paged_decode_ws_size() tells how much), the
 * call uses fewer tier-2 CTAs so that its partials fit (results agree with
 * gqa_paged_decode's to rounding); it returns GQA_ERR_WORKSPACE, without
 * launching, only if even the tier-1 partials do not fit. All calls on a device
 * share the one array and it keeps the last call's contents (nothing in it
 * needs to start at zero: every partial a call reads, that call wrote first,
 * and the arrival counters carry a per-call tag), so calls whose kernels
 * overlap on the GPU - different streams, or several host threads - race on
 * it and give wrong results: order them on one stream. 32 MiB holds the
 * tier-1 partials of every occupancy-limited launch (16 decode warps per SM,
 * two 4 KB partials each) on a GPU of up to 240 SMs.
 *
 * The array's device address is looked up once per device and kept for the
 * life of the process, so resetting a device (cudaDeviceReset, or destroying
 * its primary context) between calls is not supported: after a reset the
 * kept address no longer belongs to the device's new context.
 */
#define GQA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

int gqa_paged_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_indptr,
                             const int32_t* kv_indices, float sm_scale, void* out, float* lse, int batch,
                             struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_PAGED_DECODE_H_ */
