// Split-KV work plan for paged GQA decode: plain integer arithmetic shared by
// the decode kernel, the merge kernel and the host-side plan enumerator.
//
// The work of one call is a flat line of "units". A unit is one cached token
// for one head group, where a head group is the NG KV heads (and their 8*NG
// query heads) that one CTA handles together. With HG = 4 / NG head groups the
// line holds W = HG * T units, ordered head-group-major and, inside a head
// group, in kv_indices order (sequence by sequence, token by token).
//
// Decode CTA i of P owns the contiguous unit range [i*q, min((i+1)*q, W)) with
//     q = max(min_units, ceil(W / P)),
// so every CTA streams the same number of KV bytes whatever the mix of
// sequence lengths. This is the split-K idea of the split-K GQA kernel on the
// sigit.si vLLM "qsa.py" page (each program covers an even share of the KV
// tiles, partial outputs are merged by LSE weighting), with the share taken
// over the whole ragged batch instead of per sequence.
//
// A sequence (b, hg) covering units [U_lo, U_hi) is cut into one piece per CTA
// range it meets: CTAs i0 = U_lo / q through i1 = (U_hi - 1) / q. If i0 == i1
// the piece is the whole sequence and the decode kernel writes O and LSE
// directly. Otherwise each piece leaves a partial (O_i, LSE_i) in one of two
// slots of its CTA: slot 0 when the piece starts at the CTA's first unit,
// slot 1 otherwise (only a CTA's last piece can be a partial that does not
// start its range, so two slots suffice). The merge kernel recomputes the same
// i0, i1 and slots from kv_indptr alone.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define GQA_HD __host__ __device__ __forceinline__
#else
#define GQA_HD inline
#endif

namespace gqa {

constexpr int kQoHeads = 32;
constexpr int kKvHeads = 4;
constexpr int kGroup = kQoHeads / kKvHeads;  // query heads per KV head
constexpr int kHeadDim = 128;
constexpr int kPageBytes = kKvHeads * kHeadDim * 2;  // one page (page size 1) of K or V, bf16

// Units each decode CTA owns.
GQA_HD int64_t units_per_cta(int64_t total_units, int num_ctas, int min_units) {
  int64_t q = (total_units + num_ctas - 1) / num_ctas;
  if (q < min_units) q = min_units;
  if (q < 1) q = 1;
  return q;
}

// CTAs that meet sequence units [u_lo, u_hi) (u_hi > u_lo) and the partial
// slot used by the first of them.
struct SeqSplit {
  int64_t first_cta;
  int64_t last_cta;
  int first_slot;
};

GQA_HD SeqSplit seq_split(int64_t u_lo, int64_t u_hi, int64_t q) {
  SeqSplit s;
  s.first_cta = u_lo / q;
  s.last_cta = (u_hi - 1) / q;
  s.first_slot = (u_lo == s.first_cta * q) ? 0 : 1;
  return s;
}

// Partial-slot id (index into the workspace's partial arrays).
GQA_HD int64_t slot_id(int64_t cta, int slot) { return 2 * cta + slot; }

}  // namespace gqa
