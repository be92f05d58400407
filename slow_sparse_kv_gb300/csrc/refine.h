// Host side of the selector refinements (refine.cu), shared by the C-ABI
// call sfi_select_refined and the decode driver.  Not part of the public ABI.
#pragma once

#include "sfi_internal.h"

namespace sfi {

// Soft-NMS / exclusivity refinement of a candidate selection: one cluster of
// kRefineCluster CTAs per (sequence, KV head), each holding a contiguous
// slice of the candidates in shared memory.
constexpr int kMaxNmsRadius = 8;   // largest rho (boxes reach 2 rho positions)
constexpr int kRefineCluster = 8;  // CTAs per unit
constexpr int kRefineCT = 512;     // threads per CTA
constexpr int kRefinePer = 24;     // candidates per thread
constexpr int kRefineSlice = kRefineCT * kRefinePer;        // candidates per CTA
constexpr int kRefineCap = kRefineCluster * kRefineSlice;   // candidates per unit (98304)

struct RefineArgs {
  const int32_t* cand;        // [B*H_kv][cstride] candidate positions, ascending
  const int32_t* cand_count;  // [B*H_kv]
  int32_t cstride;
  int32_t slice_cap;          // candidates one CTA's shared memory holds in this launch
  const float* s;             // [B*H_kv][max_len] fused scores
  uint8_t* excl;              // [B][max_len] picks of earlier KV heads (or null)
  float excl_beta;
  int32_t radius;             // rho (0: no suppression)
  float wd[2 * kMaxNmsRadius + 1];  // decay exponent IoU(d)^2 / sigma at distance d
  int32_t* idx;               // [B*H_kv][k]
  int32_t* count;             // [B*H_kv]
  int32_t k;
  int32_t B, H_kv, max_len;
  int32_t g_only;             // >= 0: only the units of this KV head
  SeqMask active;
  uint32_t* status;
};
cudaError_t launch_refine(const RefineArgs& a, cudaStream_t st);

// Candidates the selector keeps per (sequence, KV head): k without Soft-NMS,
// else (k - 1)(4 rho + 1) + 1, at most max_len.
long long refine_candidates(const sfi_layout* L, const sfi_params* P, const sfi_refine* R);

// Host validation of the refinement parameters (mode, rho, sigma, beta and
// the candidate capacity).
sfi_status check_refine(const sfi_layout* L, const sfi_params* P, const sfi_refine* R);

// True when R asks for any refinement.
inline bool refine_active(const sfi_refine& R) { return R.nms_radius > 0 || R.excl_beta > 0.f; }

// Enqueue the refined selection on `st`.  `sa` is a fused-mode selector
// argument block already holding the evidence (f, or logits and statistics),
// key norms, len, s rows (required: the refinement reads them), geometry,
// selection parameters, active mask and status word; this call points its
// output at the candidate buffers (cand [B*H_kv][M], ccount [B*H_kv]) and
// writes the final sets to idx ([B*H_kv][k]) and count.  excl ([B][max_len]
// bytes) is cleared here when R.excl_beta > 0 (else unused, may be null).
sfi_status run_refined_select(SelectArgs sa, const sfi_refine& R, int k, long long M, int32_t* idx,
                              int32_t* count, int32_t* cand, int32_t* ccount, uint8_t* excl,
                              cudaStream_t st);

}  // namespace sfi
