// Split-KV work plan for paged GQA decode: plain integer arithmetic shared by
// the decode kernel, the merge kernel and the host-side plan enumerator.
//
// The work of one call is a flat line of "units". A unit is one cached token
// for one head group, where a head group is the NG KV heads (and their 8*NG
// query heads) that one CTA handles together. With HG = 4 / NG head groups the
// line holds W = HG * T units, ordered head-group-major and, inside a head
// group, in kv_indices order (sequence by sequence, token by token).
//
// The line is cut into CTA ranges in two tiers. P1 tier-1 CTAs (one resident
// wave) own equal ranges of
//     q1 = max(min_units, ceil((W - W2t) / P1))
// units, where W2t = W * tier2_permille / 1000 is the share set aside for
// tier 2; they cover W1 = min(W, P1 * q1) units. P2 tier-2 CTAs own the rest
// in equal ranges of q2 = max(tier2_min_units, ceil((W - W1) / P2)). Every
// CTA streams the same number of KV bytes within its tier whatever the mix of
// sequence lengths. The tier-1 ranges keep most of the line in long runs; the
// small tier-2 ranges at the end are taken up by whichever SMs finish their
// tier-1 range first (the block scheduler starts a tier-2 CTA as soon as a
// tier-1 CTA leaves), which evens out SMs whose share of memory bandwidth
// differs. This is the split-K idea of the split-K GQA kernel on the sigit.si
// vLLM "qsa.py" page (each program covers a share of the KV tiles, partial
// outputs are merged by LSE weighting), with the shares taken over the whole
// ragged batch instead of per sequence.
//
// A sequence (b, hg) covering units [U_lo, U_hi) is cut into one piece per CTA
// range it meets: CTAs i0 = cta_of(U_lo) through i1 = cta_of(U_hi - 1). If
// i0 == i1 the piece is the whole sequence and the decode kernel writes O and
// LSE directly. Otherwise each piece leaves a partial (O_i, LSE_i) in one of
// two slots of its CTA: slot 0 when the piece starts at the CTA's first unit,
// slot 1 otherwise (only a CTA's last piece can be a partial that does not
// start its range, so two slots suffice). The merge recomputes the same i0,
// i1 and slots from kv_indptr alone.
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

// Host-chosen shape of the plan; the unit count comes from kv_indptr on the device.
struct PlanConfig {
  int tier1_ctas;       // P1 >= 1
  int tier2_ctas;       // P2 >= 0 (0: one tier)
  int min_units;        // floor of q1 (>= 1)
  int tier2_permille;   // share of the units set aside for tier 2, in 1/1000
  int tier2_min_units;  // floor of q2 (>= 1)
};

struct Plan {
  int64_t W;   // units
  int64_t W1;  // units of tier 1
  int64_t q1;  // units per tier-1 CTA
  int64_t q2;  // units per tier-2 CTA
  int P1, P2;

  // First unit of CTA c (may be >= W: the CTA has no work).
  GQA_HD int64_t begin(int64_t c) const { return c < P1 ? c * q1 : W1 + (c - P1) * q2; }
  // One past the last unit of CTA c.
  GQA_HD int64_t end(int64_t c) const {
    const int64_t e = c < P1 ? ((c + 1) * q1 < W1 ? (c + 1) * q1 : W1) : W1 + (c - P1 + 1) * q2;
    return e < W ? e : W;
  }
  // CTA whose range holds unit u (0 <= u < W).
  GQA_HD int64_t cta_of(int64_t u) const { return u < W1 ? u / q1 : P1 + (u - W1) / q2; }
};

GQA_HD Plan make_plan(int64_t total_units, const PlanConfig& c) {
  Plan pl;
  pl.W = total_units;
  pl.P1 = c.tier1_ctas > 0 ? c.tier1_ctas : 1;
  pl.P2 = c.tier2_ctas > 0 ? c.tier2_ctas : 0;
  const int64_t w2_target = pl.P2 > 0 ? total_units * c.tier2_permille / 1000 : 0;
  int64_t q1 = (total_units - w2_target + pl.P1 - 1) / pl.P1;
  if (q1 < c.min_units) q1 = c.min_units;
  if (q1 < 1) q1 = 1;
  pl.q1 = q1;
  pl.W1 = q1 * pl.P1 < total_units ? q1 * pl.P1 : total_units;
  const int64_t w2 = total_units - pl.W1;  // > 0 only when P2 > 0 (then w2 <= w2_target)
  int64_t q2 = pl.P2 > 0 ? (w2 + pl.P2 - 1) / pl.P2 : 1;
  if (q2 < c.tier2_min_units) q2 = c.tier2_min_units;
  if (q2 < 1) q2 = 1;
  pl.q2 = q2;
  return pl;
}

// CTAs that meet sequence units [u_lo, u_hi) (u_hi > u_lo) and the partial
// slot used by the first of them.
struct SeqSplit {
  int64_t first_cta;
  int64_t last_cta;
  int first_slot;
};

GQA_HD SeqSplit seq_split(const Plan& pl, int64_t u_lo, int64_t u_hi) {
  SeqSplit s;
  s.first_cta = pl.cta_of(u_lo);
  s.last_cta = pl.cta_of(u_hi - 1);
  s.first_slot = (u_lo == pl.begin(s.first_cta)) ? 0 : 1;
  return s;
}

// Partial-slot id (index into the workspace's partial arrays).
GQA_HD int64_t slot_id(int64_t cta, int slot) { return 2 * cta + slot; }

}  // namespace gqa
