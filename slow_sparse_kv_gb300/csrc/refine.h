// Host side of the selector refinements (refine.cu), shared by the C-ABI
// call sfi_select_refined and the decode driver.  Not part of the public ABI.
#pragma once

#include "sfi_internal.h"

namespace sfi {

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
