// Soft-NMS and cross-head exclusivity refinement of the selection.
//
// SFI (gist.science 2603.12038), section "Selector", names two refinements
// beside the fusion and Top-K: a Soft-NMS that keeps one head from spending
// its budget on neighbouring, correlated tokens, and a cross-head exclusivity
// that penalises a token chosen again by another head.  The pages give no
// formula; the reading built here is
//  * Soft-NMS: greedy Gaussian Soft-NMS (Bodla et al., ICCV 2017) with
//    position i as the box [i - rho, i + rho]: take the largest current score
//    (ties to the lower position), multiply the score of every remaining
//    position j with |i - j| <= 2 rho by exp(-IoU(i, j)^2 / sigma), repeat;
//    the first k positions taken are the selection (in ascending order);
//  * exclusivity: the KV heads of a sequence select in index order, head g
//    ranking s_i * exp(-beta * c_i), c_i = earlier heads whose set holds i.
//
// GPU design.  The greedy is sequential, but a remaining position that beats
// every remaining position within 2 rho of itself (a "local winner") is taken
// by the greedy with its current score whatever is taken before it: nothing
// that can be taken earlier is near enough to lower it, and two local winners
// never lower each other.  So each round takes every local winner at once,
// then applies their decays; the picks and their scores are the greedy's.
// Scores at the pick never increase, so once k taken scores exceed every
// remaining score the greedy's first k picks are known.
// Candidates: if x is the greedy's t-th pick, every position ranked above x
// by its starting score was taken before x or lowered by one of the t - 1
// earlier picks (each lowers at most 4 rho positions), so the first k picks
// lie in the top M = (k - 1)(4 rho + 1) + 1 of E by starting score.  The
// cluster selector (with the exclusivity penalty) writes that top M in
// ascending position order.  A cluster of 8 CTAs per (sequence, KV head)
// holds it in shared memory, each CTA a contiguous slice at 8 bytes a
// candidate (position with two flag bits, current score); the few
// neighbours beyond a slice's ends are read from the next CTA's shared
// memory.  On the decode workloads (k = 4096, rho = 1: M = 20476) two to
// four rounds settle the selection.  A radix select over 64-bit (score,
// position) keys of the taken candidates finds the k-th pick, and an
// ordered compaction writes the picks in ascending position order and
// counts them for the next KV head.
#include <cooperative_groups.h>
#include <math.h>

#include <cmath>
#include <cstring>

#include "common.cuh"
#include "refine.h"

namespace sfi {

static_assert(kRefineSlice % kRefineCT == 0, "candidates split evenly over the threads");
static_assert(kRefinePer <= 32, "per-thread winner masks are 32-bit");
static_assert(kRefineCap <= 0x3fffffff, "positions keep two flag bits");
static_assert(kRefineCT % 32 == 0 && kRefineCT / 32 <= 32, "block reductions");

constexpr uint32_t kTaken = 0x80000000u;  // taken (in an earlier or this round)
constexpr uint32_t kNew = 0x40000000u;    // taken in the current round
constexpr uint32_t kPosMask = 0x3fffffffu;
constexpr int kRefineWarps = kRefineCT / 32;

// (score, position) key: larger score first, then the lower position.
// Never 0 (the low word is 2^32 - 1 - position > 0).
__device__ __forceinline__ uint64_t refine_key(float v, uint32_t pos) {
  return (uint64_t(order_key(v)) << 32) | uint64_t(0xffffffffu - pos);
}

__device__ __forceinline__ uint64_t refine_block_max(uint64_t x, uint64_t* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const uint64_t y = __shfl_xor_sync(kFull, x, o);
    x = y > x ? y : x;
  }
  if (lane == 0) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    x = lane < kRefineWarps ? sh[lane] : 0ull;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const uint64_t y = __shfl_xor_sync(kFull, x, o);
      x = y > x ? y : x;
    }
    if (lane == 0) sh[32] = x;
  }
  __syncthreads();
  x = sh[32];
  __syncthreads();
  return x;
}

__device__ __forceinline__ uint32_t refine_block_sum(uint32_t x, uint32_t* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  if (lane == 0) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    x = lane < kRefineWarps ? sh[lane] : 0u;
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    if (lane == 0) sh[32] = x;
  }
  __syncthreads();
  x = sh[32];
  __syncthreads();
  return x;
}

__device__ __forceinline__ void excl_bump(uint8_t* ex, int p) {
  const uint8_t c = ex[p];
  ex[p] = c < 255 ? uint8_t(c + 1) : c;
}

// One cluster of kRefineCluster CTAs per (sequence, KV head).  CTA `rank`
// holds candidates [rank * slice, (rank + 1) * slice) (ascending positions)
// in shared memory; the 2 rho neighbours of its first and last candidates
// are read from the neighbouring CTAs' shared memory.  Per-round cluster
// values (best remaining key, picks, picks above it) are published by each
// CTA in its own shared memory and read by all after a cluster barrier;
// histogram bins are added into rank 0.  Both come in two sets used by
// alternate rounds or passes, so a set is written while the other may still
// be read.
__global__ void __cluster_dims__(kRefineCluster, 1, 1) __launch_bounds__(kRefineCT, 1)
    refine_kernel(const __grid_constant__ RefineArgs a) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char rsm[];
  __shared__ uint64_t red64[33];
  __shared__ uint32_t red32[33];
  __shared__ uint32_t hist[256];
  __shared__ unsigned long long my_best[2];  // this CTA's per-round values,
  __shared__ uint32_t my_new[2], my_above[2];  // read by every CTA of the cluster
  __shared__ uint32_t c_hist[2][256];          // rank 0: cluster histogram
  __shared__ uint32_t sh_digit, sh_above, sh_whole;  // rank 0: radix decision
  __shared__ uint32_t cta_picks;                      // this CTA's picks
  __shared__ float wd[2 * kMaxNmsRadius + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = int(cl.block_rank());
  const bool one_head = a.g_only >= 0;
  const int ups = one_head ? 1 : a.H_kv;
  const int c = int(blockIdx.x) / kRefineCluster;
  const int b = active_seq(a.active, c / ups);
  if (b < 0 || b >= a.B) return;  // uniform over the cluster (cannot happen for a valid grid)
  const int u = b * a.H_kv + (one_head ? a.g_only : c % ups);
  const int m = a.cand_count[u];
  int32_t* out = a.idx + size_t(u) * a.k;
  const int32_t* cp = a.cand + size_t(u) * a.cstride;
  uint8_t* ex = a.excl ? a.excl + size_t(b) * a.max_len : nullptr;
  const bool lead = rank == 0 && tid == 0;
  if (m < 0 || m > a.cstride) {
    if (lead) {
      set_status(a.status, SFI_DEV_REFINE);
      a.count[u] = 0;
    }
    return;
  }
  if (m <= a.k) {
    // no more candidates than picks (|E| <= k, or no suppression): all of them
    for (int i = rank * kRefineCT + tid; i < m; i += kRefineCluster * kRefineCT) {
      int p = cp[i];
      if (p < 0 || p >= a.max_len) {
        set_status(a.status, SFI_DEV_REFINE);
        p = 0;
      }
      out[i] = p;
      if (ex) excl_bump(ex, p);
    }
    if (lead) a.count[u] = m;
    return;
  }
  const int slice = (m + kRefineCluster - 1) / kRefineCluster;
  if (slice > a.slice_cap) {
    if (lead) {
      set_status(a.status, SFI_DEV_REFINE);
      a.count[u] = 0;
    }
    return;
  }
  uint32_t* ps = reinterpret_cast<uint32_t*>(rsm);
  float* vs = reinterpret_cast<float*>(rsm + size_t(a.slice_cap) * 4);
  const int base = rank * slice;                   // first candidate of this CTA
  const int mine = max(0, min(slice, m - base));  // candidates of this CTA
  const int reach = 2 * a.radius;
  if (tid <= reach) wd[tid] = a.wd[tid];
  if (rank == 0)
    for (int i = tid; i < 2 * 256; i += kRefineCT) (&c_hist[0][0])[i] = 0u;
  // candidate j of the unit, wherever it lives in the cluster
  auto at_ps = [&](int j) -> uint32_t {
    const int l = j - base;
    if (l >= 0 && l < slice) return ps[l];
    const int r = j / slice;
    return *cl.map_shared_rank(ps + (j - r * slice), r);
  };
  auto at_vs = [&](int j) -> float {
    const int l = j - base;
    if (l >= 0 && l < slice) return vs[l];
    const int r = j / slice;
    return *cl.map_shared_rank(vs + (j - r * slice), r);
  };

  // ---- this CTA's candidates and their starting scores s_i * exp(-beta c_i)
  const float* srow = a.s + size_t(u) * a.max_len;
#pragma unroll 4
  for (int j = 0; j < kRefinePer; ++j) {
    const int li = tid + j * kRefineCT;
    if (li < mine) {
      int p = cp[base + li];
      if (p < 0 || p >= a.max_len) {
        set_status(a.status, SFI_DEV_REFINE);
        p = 0;
      }
      float v = srow[p];
      if (ex) v *= excl_factor(ex[p], a.excl_beta);
      ps[li] = uint32_t(p);
      vs[li] = v;
    }
  }
  cl.sync();  // every slice and the cleared totals are visible

  // ---- rounds: take every local winner, then apply the decays
  uint32_t prev = 0;  // this thread's winners of the previous round (bit j)
  uint32_t taken = 0;
  bool settled = false;
  for (int round = 0; round < m; ++round) {
    const int par = round & 1;
    uint32_t win = 0;
    for (int j = 0; j < kRefinePer; ++j) {
      const int li = tid + j * kRefineCT;
      if (li >= mine) break;
      const uint32_t xi = ps[li];
      if (xi & kTaken) continue;
      const int gi = base + li;
      const int pi = int(xi & kPosMask);
      const uint64_t ki = refine_key(vs[li], uint32_t(pi));
      bool ok = true;
      for (int t = 1; t <= reach && ok && gi - t >= 0; ++t) {
        const uint32_t y = at_ps(gi - t);
        if (pi - int(y & kPosMask) > reach) break;
        if (!(y & kTaken) && refine_key(at_vs(gi - t), y & kPosMask) > ki) ok = false;
      }
      for (int t = 1; t <= reach && ok && gi + t < m; ++t) {
        const uint32_t y = at_ps(gi + t);
        if (int(y & kPosMask) - pi > reach) break;
        if (!(y & kTaken) && refine_key(at_vs(gi + t), y & kPosMask) > ki) ok = false;
      }
      if (ok) win |= 1u << j;
    }
    cl.sync();  // every CTA has judged its candidates on the same state
    for (int j = 0; j < kRefinePer; ++j) {
      const int li = tid + j * kRefineCT;
      if ((win >> j) & 1u) {
        ps[li] |= kTaken | kNew;
      } else if ((prev >> j) & 1u) {
        ps[li] &= ~kNew;
      }
    }
    cl.sync();  // this round's picks are marked everywhere
    uint64_t best = 0;  // best remaining key after this round's decays
    for (int j = 0; j < kRefinePer; ++j) {
      const int li = tid + j * kRefineCT;
      if (li >= mine) break;
      const uint32_t xi = ps[li];
      if (xi & kTaken) continue;
      const int gi = base + li;
      const int pi = int(xi & kPosMask);
      float e = 0.f;
      for (int t = 1; t <= reach && gi - t >= 0; ++t) {
        const uint32_t y = at_ps(gi - t);
        const int d = pi - int(y & kPosMask);
        if (d > reach) break;
        if ((y & kNew) && d > 0) e += wd[d];
      }
      for (int t = 1; t <= reach && gi + t < m; ++t) {
        const uint32_t y = at_ps(gi + t);
        const int d = int(y & kPosMask) - pi;
        if (d > reach) break;
        if ((y & kNew) && d > 0) e += wd[d];
      }
      float v = vs[li];
      if (e > 0.f) {
        v *= expf(-e);
        vs[li] = v;
      }
      const uint64_t key = refine_key(v, uint32_t(pi));
      best = key > best ? key : best;
    }
    // cluster totals: each CTA publishes its values in its own shared memory
    // (slot `par`; the other slot is still being read for the previous
    // round) and every CTA reads all of them after the barrier
    const uint64_t best_cta = refine_block_max(best, red64);
    const uint32_t new_cta = refine_block_sum(uint32_t(__popc(win)), red32);
    if (tid == 0) {
      my_best[par] = best_cta;
      my_new[par] = new_cta;
    }
    cl.sync();
    uint64_t best_all = 0;
    for (int r = 0; r < kRefineCluster; ++r) {
      const uint64_t x = *cl.map_shared_rank(&my_best[par], r);
      best_all = x > best_all ? x : best_all;
      taken += *cl.map_shared_rank(&my_new[par], r);
    }
    prev = win;
    if (best_all == 0) {  // every candidate is taken (m > k of them)
      settled = true;
    } else if (taken >= uint32_t(a.k)) {
      uint32_t above = 0;
      for (int j = 0; j < kRefinePer; ++j) {
        const int li = tid + j * kRefineCT;
        if (li >= mine) break;
        const uint32_t xi = ps[li];
        if ((xi & kTaken) && refine_key(vs[li], xi & kPosMask) > best_all) ++above;
      }
      above = refine_block_sum(above, red32);
      if (tid == 0) my_above[par] = above;
      cl.sync();
      uint32_t above_all = 0;
      for (int r = 0; r < kRefineCluster; ++r) above_all += *cl.map_shared_rank(&my_above[par], r);
      if (above_all >= uint32_t(a.k)) settled = true;
    }
    if (settled) break;
  }
  if (!settled) {  // cannot happen: every round takes the best remaining candidate
    if (lead) {
      set_status(a.status, SFI_DEV_REFINE);
      a.count[u] = 0;
    }
    cl.sync();  // no CTA leaves while another may read its shared memory
    return;
  }

  // ---- the k-th largest key among the taken candidates, 8 bits at a time;
  // the picks are the taken keys whose top bits are >= `prefix` (shifted by
  // `cut`), and the search stops once the chosen bin is needed whole
  uint64_t prefix = 0;
  uint32_t krem = uint32_t(a.k);
  int cut = 0;
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    const int par = pass & 1;
    for (int i = tid; i < 256; i += kRefineCT) hist[i] = 0;
    __syncthreads();
    for (int j = 0; j < kRefinePer; ++j) {
      const int li = tid + j * kRefineCT;
      if (li >= mine) break;
      const uint32_t xi = ps[li];
      if (!(xi & kTaken)) continue;
      const uint64_t key = refine_key(vs[li], xi & kPosMask);
      if (pass == 0 || (key >> (shift + 8)) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    for (int i = tid; i < 256; i += kRefineCT)
      if (hist[i]) atomicAdd(cl.map_shared_rank(&c_hist[par][i], 0), hist[i]);
    cl.sync();  // the cluster histogram of this pass is complete in rank 0
    if (rank == 0) {
      if (warp == 0) {
        // lane l holds bins 255 - 8 l down to 248 - 8 l
        uint32_t cnt[8], tot = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          cnt[q] = c_hist[par][255 - 8 * lane - q];
          tot += cnt[q];
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t above = incl - tot;
        if (above < krem && krem <= incl) {
          uint32_t acc = above;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (acc < krem && acc + cnt[q] >= krem) {
              sh_digit = uint32_t(255 - 8 * lane - q);
              sh_above = acc;
              sh_whole = cnt[q] == krem - acc;
            }
            acc += cnt[q];
          }
        }
      }
      // the other set was read in the previous pass: clear it for the next
      for (int i = tid; i < 256; i += kRefineCT) c_hist[par ^ 1][i] = 0u;
    }
    cl.sync();  // rank 0's decision is visible
    const uint32_t digit = *cl.map_shared_rank(&sh_digit, 0);
    const uint32_t whole = *cl.map_shared_rank(&sh_whole, 0);
    krem -= *cl.map_shared_rank(&sh_above, 0);
    prefix = (prefix << 8) | digit;
    cut = shift;
    if (whole) break;  // every key of the chosen bin is a pick
  }

  // ---- the picks in ascending position order: thread t owns this CTA's
  // candidates [t * per, (t + 1) * per); block and cluster offsets follow
  const int per = (mine + kRefineCT - 1) / kRefineCT;
  const int c0 = min(mine, tid * per), c1 = min(mine, c0 + per);
  uint32_t own = 0;
  for (int i = c0; i < c1; ++i) {
    const uint32_t xi = ps[i];
    if ((xi & kTaken) && (refine_key(vs[i], xi & kPosMask) >> cut) >= prefix) ++own;
  }
  uint32_t incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) red32[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t v = lane < kRefineWarps ? red32[lane] : 0u;
    uint32_t w_incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, w_incl, o);
      if (lane >= o) w_incl += y;
    }
    if (lane < kRefineWarps) red32[lane] = w_incl - v;
    if (lane == 31) cta_picks = w_incl;
  }
  cl.sync();  // every CTA's pick count is visible
  uint32_t before = 0, total = 0;
  for (int r = 0; r < kRefineCluster; ++r) {
    const uint32_t n = *cl.map_shared_rank(&cta_picks, r);
    if (r < rank) before += n;
    total += n;
  }
  uint32_t at = before + red32[warp] + incl - own;
  for (int i = c0; i < c1; ++i) {
    const uint32_t xi = ps[i];
    if ((xi & kTaken) && (refine_key(vs[i], xi & kPosMask) >> cut) >= prefix) {
      if (at < uint32_t(a.k)) {
        out[at] = int32_t(xi & kPosMask);
        if (ex) excl_bump(ex, int(xi & kPosMask));
      }
      ++at;
    }
  }
  if (lead) {
    if (total != uint32_t(a.k)) set_status(a.status, SFI_DEV_REFINE);
    a.count[u] = min(int(total), a.k);
  }
  cl.sync();  // no CTA leaves while another may read its shared memory
}

cudaError_t launch_refine(const RefineArgs& a, cudaStream_t st) {
  const size_t smem = size_t(a.slice_cap) * 8;
  cudaError_t e = cudaFuncSetAttribute(refine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(smem));
  if (e != cudaSuccess) return e;
  int n_active = 0;
  for (int b = 0; b < a.B; ++b) n_active += int((a.active.bits[b >> 5] >> (b & 31)) & 1u);
  const int units = n_active * (a.g_only >= 0 ? 1 : a.H_kv);
  if (units == 0) return cudaSuccess;
  refine_kernel<<<units * kRefineCluster, kRefineCT, smem, st>>>(a);
  return cudaGetLastError();
}

long long refine_candidates(const sfi_layout* L, const sfi_params* P, const sfi_refine* R) {
  if (R->nms_radius <= 0) return P->k;
  const long long m = (long long)(P->k - 1) * (4LL * R->nms_radius + 1) + 1;
  return m < L->max_len ? m : L->max_len;
}

struct RefinePlan {
  WsPlan base;
  size_t excl_off, cand_off, ccount_off, total;
  long long M;
};

RefinePlan plan_refine(const sfi_layout* L, const sfi_params* P, const sfi_refine* R) {
  RefinePlan rp{};
  rp.base = plan_workspace(L->batch, L->n_q_heads, L->n_kv_heads, L->head_dim, L->max_len);
  rp.M = refine_candidates(L, P, R);
  const size_t units = size_t(L->batch) * L->n_kv_heads;
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t off = rp.base.total;
  rp.excl_off = off;
  off += a256(size_t(L->batch) * L->max_len);
  rp.cand_off = off;
  off += a256(units * size_t(rp.M) * 4);
  rp.ccount_off = off;
  off += a256(units * 4);
  rp.total = off;
  return rp;
}

sfi_status check_refine(const sfi_layout* L, const sfi_params* P, const sfi_refine* R) {
  if (!R) return fail(SFI_ERR_INVALID_ARG, "refine is NULL");
  if (P->mode != SFI_SELECT_FUSED)
    return fail(SFI_ERR_INVALID_ARG, "Soft-NMS and exclusivity refine the fused SFI selection only");
  if (R->nms_radius < 0) return fail(SFI_ERR_INVALID_ARG, "nms_radius must be >= 0 (got %d)", R->nms_radius);
  if (R->nms_radius > kMaxNmsRadius)
    return fail(SFI_ERR_CAPACITY, "nms_radius %d exceeds the limit %d", R->nms_radius, kMaxNmsRadius);
  if (R->nms_radius > 0 && !(R->nms_sigma > 0.f && std::isfinite(R->nms_sigma)))
    return fail(SFI_ERR_INVALID_ARG, "nms_sigma must be finite and > 0 (got %g)", double(R->nms_sigma));
  if (!(R->excl_beta >= 0.f && std::isfinite(R->excl_beta)))
    return fail(SFI_ERR_INVALID_ARG, "excl_beta must be finite and >= 0 (got %g)", double(R->excl_beta));
  const long long M = refine_candidates(L, P, R);
  if (R->nms_radius > 0 && M > kRefineCap)
    return fail(SFI_ERR_CAPACITY,
                "Soft-NMS keeps (k - 1)(4 rho + 1) + 1 = %lld candidates per (sequence, KV head); "
                "the limit is %d",
                M, kRefineCap);
  return SFI_OK;
}

sfi_status run_refined_select(SelectArgs sa, const sfi_refine& R, int k, long long M, int32_t* idx,
                              int32_t* count, int32_t* cand, int32_t* ccount, uint8_t* excl,
                              cudaStream_t st) {
  const bool excl_on = R.excl_beta > 0.f;
  cudaError_t e = cudaSuccess;
  if (excl_on) {
    e = cudaMemsetAsync(excl, 0, size_t(sa.B) * sa.max_len, st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the exclusivity counts");
  }
  sa.mode = SFI_SELECT_FUSED;
  sa.idx = cand;
  sa.count = ccount;
  sa.k = int(M);
  sa.excl = excl_on ? excl : nullptr;
  sa.excl_beta = R.excl_beta;

  RefineArgs ra;
  std::memset(&ra, 0, sizeof(ra));
  ra.cand = cand;
  ra.cand_count = ccount;
  ra.cstride = int(M);
  ra.slice_cap = R.nms_radius > 0 ? int((M + kRefineCluster - 1) / kRefineCluster) : 0;
  ra.s = sa.s;
  ra.excl = excl_on ? excl : nullptr;
  ra.excl_beta = R.excl_beta;
  ra.radius = R.nms_radius;
  for (int d = 1; d <= 2 * R.nms_radius; ++d) {
    const double box = 2.0 * R.nms_radius + 1.0;
    const double iou = (box - d) / (box + d);
    ra.wd[d] = float(iou * iou / double(R.nms_sigma));
  }
  ra.idx = idx;
  ra.count = count;
  ra.k = k;
  ra.B = sa.B;
  ra.H_kv = sa.H_kv;
  ra.max_len = sa.max_len;
  ra.active = sa.active;
  ra.status = sa.status;

  // With exclusivity the KV heads go one after another (each reads the
  // earlier heads' picks); without it every unit runs in one pair of launches.
  const int passes = excl_on ? sa.H_kv : 1;
  for (int g = 0; g < passes; ++g) {
    sa.g_only = excl_on ? g : -1;
    ra.g_only = sa.g_only;
    e = launch_select(sa, st);
    if (e != cudaSuccess) return cuda_fail(e, "selector launch");
    e = launch_refine(ra, st);
    if (e != cudaSuccess) return cuda_fail(e, "refinement launch");
  }
  return SFI_OK;
}

}  // namespace sfi

using namespace sfi;

extern "C" size_t sfi_select_refined_workspace_size(const sfi_layout* L, const sfi_params* P,
                                                    const sfi_refine* R) {
  if (check_layout(L) != SFI_OK || check_params(P, true) != SFI_OK || check_refine(L, P, R) != SFI_OK)
    return 0;
  return plan_refine(L, P, R).total;
}

extern "C" sfi_status sfi_select_refined(const sfi_layout* L, const sfi_params* P,
                                         const sfi_refine* R, const float* f, const float* knorm,
                                         int32_t* idx_out, int32_t* count_out, float* s_out,
                                         void* ws, size_t ws_bytes, sfi_stream stream) {
  sfi_status s = check_layout(L);
  if (s != SFI_OK) return s;
  if ((s = check_params(P, true)) != SFI_OK) return s;
  if ((s = check_refine(L, P, R)) != SFI_OK) return s;
  if (!f || !knorm || !idx_out || !count_out)
    return fail(SFI_ERR_INVALID_ARG, "f, knorm, idx_out and count_out must be set");
  if (L->max_len > kSelectMaxLen)
    return fail(SFI_ERR_CAPACITY, "the selector holds at most %d positions per row (max_len %d)",
                kSelectMaxLen, L->max_len);
  const RefinePlan rp = plan_refine(L, P, R);
  if (!ws) return fail(SFI_ERR_WORKSPACE, "workspace is NULL");
  if (ws_bytes < rp.total)
    return fail(SFI_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu required",
                ws_bytes, rp.total);
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0)
    return fail(SFI_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  SelectArgs sa{};
  sa.evidence = f;
  sa.knorm = knorm;
  sa.H_q = L->n_q_heads;
  sa.len = L->len;
  sa.s = s_out ? s_out : reinterpret_cast<float*>(w + rp.base.s_off);
  sa.B = L->batch;
  sa.H_kv = L->n_kv_heads;
  sa.max_len = L->max_len;
  sa.n_sink = P->n_sink;
  sa.window = P->window;
  sa.lambda = P->lambda;
  sa.status = reinterpret_cast<uint32_t*>(w + rp.base.status_off);
  attach_select_scratch(sa, w, rp.base);
  for (int b = 0; b < L->batch; ++b) sa.active.bits[b >> 5] |= 1u << (b & 31);
  return run_refined_select(sa, *R, P->k, rp.M, idx_out, count_out,
                            reinterpret_cast<int32_t*>(w + rp.cand_off),
                            reinterpret_cast<int32_t*>(w + rp.ccount_off),
                            reinterpret_cast<uint8_t*>(w + rp.excl_off), st);
}
