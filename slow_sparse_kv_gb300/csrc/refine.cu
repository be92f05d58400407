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
// ascending position order; one 1024-thread CTA per (sequence, KV head)
// holds it in shared memory, 8 bytes a candidate (position with two flag
// bits, current score).  On the decode workloads (k = 4096, rho = 1:
// M = 20476) two to four rounds settle the selection.  A radix select over
// 64-bit (score, position) keys of the taken candidates finds the k-th pick,
// and an ordered compaction writes the picks in ascending position order and
// counts them for the next KV head.
#include <math.h>

#include <cmath>
#include <cstring>

#include "common.cuh"
#include "refine.h"

namespace sfi {

constexpr int kRefineCT = 1024;
constexpr int kRefinePer = kRefineCap / kRefineCT;  // candidates per thread (interleaved)
static_assert(kRefineCap % kRefineCT == 0, "candidates split evenly over the threads");
static_assert(kRefinePer <= 32, "per-thread winner masks are 32-bit");
static_assert(kRefineCap <= 0x3fffffff, "positions keep two flag bits");

constexpr uint32_t kTaken = 0x80000000u;  // taken (in an earlier or this round)
constexpr uint32_t kNew = 0x40000000u;    // taken in the current round
constexpr uint32_t kPosMask = 0x3fffffffu;

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
    x = sh[lane];
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
    x = sh[lane];
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

__global__ void __launch_bounds__(kRefineCT, 1) refine_kernel(const __grid_constant__ RefineArgs a) {
  static_assert(kRefineCT == 1024, "block reductions assume 32 warps");
  extern __shared__ __align__(16) unsigned char rsm[];
  __shared__ uint64_t red64[33];
  __shared__ uint32_t red32[33];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t sh_digit, sh_above, sh_whole;
  __shared__ float wd[2 * kMaxNmsRadius + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool one_head = a.g_only >= 0;
  const int ups = one_head ? 1 : a.H_kv;
  const int b = active_seq(a.active, int(blockIdx.x) / ups);
  if (b < 0 || b >= a.B) return;  // cannot happen for a valid grid
  const int u = b * a.H_kv + (one_head ? a.g_only : int(blockIdx.x) % ups);
  const int m = a.cand_count[u];
  int32_t* out = a.idx + size_t(u) * a.k;
  const int32_t* cp = a.cand + size_t(u) * a.cstride;
  uint8_t* ex = a.excl ? a.excl + size_t(b) * a.max_len : nullptr;
  if (m < 0 || m > a.cstride) {
    if (tid == 0) {
      set_status(a.status, SFI_DEV_REFINE);
      a.count[u] = 0;
    }
    return;
  }
  if (m <= a.k) {
    // no more candidates than picks (|E| <= k, or no suppression): all of them
    for (int i = tid; i < m; i += kRefineCT) {
      int p = cp[i];
      if (p < 0 || p >= a.max_len) {
        set_status(a.status, SFI_DEV_REFINE);
        p = 0;
      }
      out[i] = p;
      if (ex) excl_bump(ex, p);
    }
    if (tid == 0) a.count[u] = m;
    return;
  }
  if (m > a.cap) {
    if (tid == 0) {
      set_status(a.status, SFI_DEV_REFINE);
      a.count[u] = 0;
    }
    return;
  }
  uint32_t* ps = reinterpret_cast<uint32_t*>(rsm);
  float* vs = reinterpret_cast<float*>(rsm + size_t(a.cap) * 4);
  const int reach = 2 * a.radius;
  if (tid <= reach) wd[tid] = a.wd[tid];

  // ---- candidates and their starting scores s_i * exp(-beta c_i)
  const float* srow = a.s + size_t(u) * a.max_len;
#pragma unroll 4
  for (int j = 0; j < kRefinePer; ++j) {
    const int i = tid + j * kRefineCT;
    if (i < m) {
      int p = cp[i];
      if (p < 0 || p >= a.max_len) {
        set_status(a.status, SFI_DEV_REFINE);
        p = 0;
      }
      float v = srow[p];
      if (ex) v *= excl_factor(ex[p], a.excl_beta);
      ps[i] = uint32_t(p);
      vs[i] = v;
    }
  }
  __syncthreads();

  // ---- rounds: take every local winner, then apply the decays
  uint32_t prev = 0;  // this thread's winners of the previous round (bit j)
  uint32_t taken = 0;
  bool settled = false;
  for (int round = 0; round < m; ++round) {
    uint32_t win = 0;
    for (int j = 0; j < kRefinePer; ++j) {
      const int i = tid + j * kRefineCT;
      if (i >= m) break;
      const uint32_t xi = ps[i];
      if (xi & kTaken) continue;
      const int pi = int(xi & kPosMask);
      const uint64_t ki = refine_key(vs[i], uint32_t(pi));
      bool ok = true;
      for (int t = 1; t <= reach && ok && i - t >= 0; ++t) {
        const uint32_t y = ps[i - t];
        if (pi - int(y & kPosMask) > reach) break;
        if (!(y & kTaken) && refine_key(vs[i - t], y & kPosMask) > ki) ok = false;
      }
      for (int t = 1; t <= reach && ok && i + t < m; ++t) {
        const uint32_t y = ps[i + t];
        if (int(y & kPosMask) - pi > reach) break;
        if (!(y & kTaken) && refine_key(vs[i + t], y & kPosMask) > ki) ok = false;
      }
      if (ok) win |= 1u << j;
    }
    __syncthreads();
    for (int j = 0; j < kRefinePer; ++j) {
      const int i = tid + j * kRefineCT;
      if ((win >> j) & 1u) {
        ps[i] |= kTaken | kNew;
      } else if ((prev >> j) & 1u) {
        ps[i] &= ~kNew;
      }
    }
    __syncthreads();
    uint64_t best = 0;  // best remaining key after this round's decays
    for (int j = 0; j < kRefinePer; ++j) {
      const int i = tid + j * kRefineCT;
      if (i >= m) break;
      const uint32_t xi = ps[i];
      if (xi & kTaken) continue;
      const int pi = int(xi & kPosMask);
      float e = 0.f;
      for (int t = 1; t <= reach && i - t >= 0; ++t) {
        const uint32_t y = ps[i - t];
        const int d = pi - int(y & kPosMask);
        if (d > reach) break;
        if ((y & kNew) && d > 0) e += wd[d];
      }
      for (int t = 1; t <= reach && i + t < m; ++t) {
        const uint32_t y = ps[i + t];
        const int d = int(y & kPosMask) - pi;
        if (d > reach) break;
        if ((y & kNew) && d > 0) e += wd[d];
      }
      float v = vs[i];
      if (e > 0.f) {
        v *= expf(-e);
        vs[i] = v;
      }
      const uint64_t key = refine_key(v, uint32_t(pi));
      best = key > best ? key : best;
    }
    const uint64_t best_all = refine_block_max(best, red64);
    taken += refine_block_sum(uint32_t(__popc(win)), red32);
    prev = win;
    if (best_all == 0) {  // every candidate is taken (m > k of them)
      settled = true;
      break;
    }
    if (taken >= uint32_t(a.k)) {
      uint32_t above = 0;
      for (int j = 0; j < kRefinePer; ++j) {
        const int i = tid + j * kRefineCT;
        if (i >= m) break;
        const uint32_t xi = ps[i];
        if ((xi & kTaken) && refine_key(vs[i], xi & kPosMask) > best_all) ++above;
      }
      if (refine_block_sum(above, red32) >= uint32_t(a.k)) {
        settled = true;
        break;
      }
    }
  }
  if (!settled) {  // cannot happen: every round takes the best remaining candidate
    if (tid == 0) {
      set_status(a.status, SFI_DEV_REFINE);
      a.count[u] = 0;
    }
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
    for (int i = tid; i < 256; i += kRefineCT) hist[i] = 0;
    __syncthreads();
    for (int j = 0; j < kRefinePer; ++j) {
      const int i = tid + j * kRefineCT;
      if (i >= m) break;
      const uint32_t xi = ps[i];
      if (!(xi & kTaken)) continue;
      const uint64_t key = refine_key(vs[i], xi & kPosMask);
      if (pass == 0 || (key >> (shift + 8)) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 255 - 8 l down to 248 - 8 l
      uint32_t cnt[8], tot = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        cnt[q] = hist[255 - 8 * lane - q];
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
    __syncthreads();
    prefix = (prefix << 8) | sh_digit;
    krem -= sh_above;
    cut = shift;
    if (sh_whole) break;  // every key of the chosen bin is a pick
  }

  // ---- the picks in ascending position order: thread t owns the candidates
  // [t * per, (t + 1) * per); one block scan of the counts gives its offset
  const int per = (m + kRefineCT - 1) / kRefineCT;
  const int c0 = min(m, tid * per), c1 = min(m, c0 + per);
  uint32_t mine = 0;
  for (int i = c0; i < c1; ++i) {
    const uint32_t xi = ps[i];
    if ((xi & kTaken) && (refine_key(vs[i], xi & kPosMask) >> cut) >= prefix) ++mine;
  }
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) red32[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t v = red32[lane];
    uint32_t w_incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, w_incl, o);
      if (lane >= o) w_incl += y;
    }
    red32[lane] = w_incl - v;
    if (lane == 31) red32[32] = w_incl;
  }
  __syncthreads();
  uint32_t at = red32[warp] + incl - mine;
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
  if (tid == 0) {
    const uint32_t total = red32[32];
    if (total != uint32_t(a.k)) set_status(a.status, SFI_DEV_REFINE);
    a.count[u] = min(int(total), a.k);
  }
}

cudaError_t launch_refine(const RefineArgs& a, cudaStream_t st) {
  const size_t smem = size_t(a.cap) * 8;
  cudaError_t e = cudaFuncSetAttribute(refine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(smem));
  if (e != cudaSuccess) return e;
  int n_active = 0;
  for (int b = 0; b < a.B; ++b) n_active += int((a.active.bits[b >> 5] >> (b & 31)) & 1u);
  const int units = n_active * (a.g_only >= 0 ? 1 : a.H_kv);
  if (units == 0) return cudaSuccess;
  refine_kernel<<<units, kRefineCT, smem, st>>>(a);
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
  ra.cap = R.nms_radius > 0 ? int(M) : 0;
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
  for (int b = 0; b < L->batch; ++b) sa.active.bits[b >> 5] |= 1u << (b & 31);
  return run_refined_select(sa, *R, P->k, rp.M, idx_out, count_out,
                            reinterpret_cast<int32_t*>(w + rp.cand_off),
                            reinterpret_cast<int32_t*>(w + rp.ccount_off),
                            reinterpret_cast<uint8_t*>(w + rp.excl_off), st);
}
