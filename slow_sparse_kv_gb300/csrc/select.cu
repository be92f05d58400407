// Evidence pass and selector kernels.
//
// SFI (gist.science 2603.12038), section "Selector": the slow step's dense
// attention logits give the evidence distribution f; cache statistics (key
// norms) give the prior r; the reverse-KL fusion has the closed form
// s = (1 - lambda) f + lambda r (ko page, section 2.B); Top-K of s is the
// selected memory of the following fast steps.
// Vegas (gist.science 2602.07223), sections 2.A-2.B: the selected prefix set
// is the top-k of the attention logits summed over the collected query rows
// and all query heads.
//
// Evidence pass: f[b][g][i] = (1/G) sum_h 2^(l_{h,i} - M_h) / Z_h from the
// log2-scaled logits and per-head (M, Z) the attention kernel stored.
//
// Selector.  Each selecting unit -- a (sequence, KV head), or a sequence in
// the per-sequence logit-sum mode -- is cut into C chunks of consecutive
// positions, and C is chosen so that all units together give about two CTAs
// per SM: every SM works on the few units of a decode step.  No CTA ever
// waits for another; three launches, each a programmatic dependent of the
// one before it, pass their results through the workspace:
//  1. (fused mode) each chunk sums its key norms over E;
//  2. each chunk forms the scores (f from the logits on the decode path),
//     writes s when asked, the order key of every position of E and adds
//     its histogram of the keys' top 11 bits to the unit's (integer atomics);
//  3. each chunk reads the unit's histogram, which fixes the top digit d0 of
//     the k-th largest key, and writes its keys at or above d0 -- as
//     (key, position), in position order -- to its own region of a list.  The
//     last chunk CTA of the unit to finish (an atomic counter) finds the two
//     lower digits among the keys of bin d0 (few: about 2% of E at the decode
//     workloads) and writes the keys above the k-th, then the lowest-
//     positioned keys equal to it, in ascending position order, so ties go to
//     the lower position exactly as the definition says.  It leaves the
//     histogram and the counter at zero for the next launch.
// All sums run in a fixed order, so the selection does not depend on the
// schedule.
#include <math.h>

#include "common.cuh"
#include "warp_hist.cuh"

namespace sfi {

constexpr int kFpassThreads = 256;
constexpr int kSelT = 512;      // threads of a score or list CTA
constexpr int kSelNuT = 256;    // threads of a key-norm sum CTA
constexpr int kSelU = 8;        // positions in flight per thread
constexpr int kRadixBins = 2048;
constexpr int kRadixShift0 = 21;  // digits: bits 31..21, 20..10, 9..0 of the order key
constexpr int kRadixShift1 = 10;
constexpr int kSelMinChunk = 2048;  // positions per chunk, at least
constexpr int kRun = 8;             // consecutive list positions or entries per thread and tile
constexpr int kListCap = 12288;     // list entries the finisher stages in shared memory (96 KB)

// The G logits of one position ([pos][G] rows are 4*G-byte aligned).
template <int G>
__device__ __forceinline__ void load_row(const float* p, float (&l)[G]) {
  if constexpr (G % 4 == 0) {
#pragma unroll
    for (int j = 0; j < G; j += 4) {
      const float4 x = *reinterpret_cast<const float4*>(p + j);
      l[j] = x.x;
      l[j + 1] = x.y;
      l[j + 2] = x.z;
      l[j + 3] = x.w;
    }
  } else if constexpr (G == 2) {
    const float2 x = *reinterpret_cast<const float2*>(p);
    l[0] = x.x;
    l[1] = x.y;
  } else {
#pragma unroll
    for (int j = 0; j < G; ++j) l[j] = p[j];
  }
}

// f_i = (1/G) sum_h 2^(l_{h,i} - M_h) / Z_h, from log2-scaled logits.
template <int G>
__device__ __forceinline__ float evidence_from_logits(const float (&l)[G], const float (&M)[G],
                                                      const float (&iz)[G]) {
  float acc = 0.f;
#pragma unroll
  for (int hh = 0; hh < G; ++hh) acc = fmaf(exp2f(l[hh] - M[hh]), iz[hh], acc);
  return acc * (1.0f / float(G));
}

template <int G>
__global__ void __launch_bounds__(kFpassThreads) fpass_kernel(const FpassArgs a) {
  const int u = blockIdx.y;
  const int b = u / a.H_kv, g = u % a.H_kv;
  if (!seq_is_slow(a.slow, b)) return;
  const int n = a.len[b];
  if (n < 1 || n > a.max_len) return;
  float M[G], iz[G];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    const size_t qh = size_t(b) * a.H_q + size_t(g) * G + hh;
    M[hh] = a.stats[qh * 2];
    iz[hh] = 1.0f / a.stats[qh * 2 + 1];
  }
  const float* lrow = a.logits + size_t(u) * a.max_len * G;
  float* frow = a.f + size_t(u) * a.max_len;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    float l[G];
    load_row<G>(lrow + size_t(i) * G, l);
    frow[i] = evidence_from_logits<G>(l, M, iz);
  }
}

// Deterministic block sum (fixed reduction tree for a fixed block size).
__device__ float sel_block_sum(float v, float* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(kFull, v, o);
  if (lane == 0) sh[w] = v;
  __syncthreads();
  if (w == 0) {
    v = lane < int(blockDim.x >> 5) ? sh[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(kFull, v, o);
    if (lane == 0) sh[32] = v;
  }
  __syncthreads();
  const float r = sh[32];
  __syncthreads();
  return r;
}

// Exclusive block scan of one packed (gt << 16 | eq) count per thread; also
// returns the block total.  Two barriers.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* sh, uint32_t& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    uint32_t x = lane < nw ? sh[lane] : 0u;
    uint32_t xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, xi, o);
      if (lane >= o) xi += y;
    }
    if (lane < nw) sh[lane] = xi - x;
    if (lane == nw - 1) sh[32] = xi;
  }
  __syncthreads();
  total = sh[32];
  const uint32_t r = sh[w] + incl - v;
  __syncthreads();
  return r;
}

// Pick the digit d with above(d) < krem <= above(d) + hist[d] (above(d)
// counts the keys in higher bins), with the whole block: thread t sums
// NB / kSelT consecutive bins from the top, a block scan gives the count
// above its range, and the one thread whose range holds the krem-th key
// walks its bins.  0 < krem <= the histogram's total.  Ends with a barrier.
template <int NB>
__device__ void block_pick_digit(const uint32_t* hist, uint32_t krem, uint32_t* out_digit,
                                 uint32_t* out_above, uint32_t* scan_sh) {
  constexpr int PER = NB / kSelT;
  static_assert(PER * kSelT == NB, "bins split evenly over the block");
  const int top = NB - 1 - PER * int(threadIdx.x);  // bins top, top - 1, ..., top - PER + 1
  uint32_t c[PER];
  uint32_t sum = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    c[j] = hist[top - j];
    sum += c[j];
  }
  uint32_t tot;
  const uint32_t excl = block_excl_scan(sum, scan_sh, tot);
  if (excl < krem && krem <= excl + sum) {
    uint32_t acc = excl;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      if (acc + c[j] >= krem) {
        *out_digit = uint32_t(top - j);
        *out_above = acc;
        break;
      }
      acc += c[j];
    }
  }
  __syncthreads();
}

// One selecting unit and this CTA's chunk of it.
struct SelUnit {
  int b, unit, u;       // sequence; unit; row of the per-position arrays (b * H_kv in the
                        // per-sequence mode)
  int n, lo, hi, keff;  // length; E = [lo, hi); selection size
  int n_sc, ch;         // positions that get a score; chunk length
  int p0, p1, e0, e1;   // this chunk's positions and its part of E
  bool per_seq, prior, need_radix;
};

// First position of E in chunk c (where chunk c's list region starts).
__device__ __forceinline__ int sel_chunk_e0(const SelUnit& s, int c) {
  return max(s.lo, min(s.n_sc, c * s.ch));
}

// 0: ok; 1: no such unit (cannot happen for a valid grid); 2: length outside
// [1, max_len].  The result is the same in every CTA of the unit.
__device__ __forceinline__ int sel_unit(const SelectArgs& a, int j, int c, int C, SelUnit& s) {
  s.per_seq = a.mode == SFI_SELECT_LOGIT_SUM_SEQ;
  s.prior = a.mode == SFI_SELECT_FUSED;            // key-norm prior and (1 - lambda) weight
  const bool one_head = s.prior && a.g_only >= 0;  // only KV head g_only of each sequence
  const int ups = s.per_seq || one_head ? 1 : a.H_kv;  // units per sequence
  s.b = active_seq(a.active, j / ups);
  if (s.b < 0 || s.b >= a.B) return 1;
  s.unit = s.per_seq ? s.b : s.b * a.H_kv + (one_head ? a.g_only : j % ups);
  s.u = s.per_seq ? s.b * a.H_kv : s.unit;
  s.n = a.len[s.b];
  if (s.n < 1 || s.n > a.max_len) return 2;
  s.lo = s.per_seq ? 0 : a.n_sink;
  s.hi = max(s.lo, s.n - a.window);
  const int ne = s.hi - s.lo;
  s.keff = min(a.k, ne);
  s.n_sc = s.per_seq ? s.hi : s.n;
  s.ch = ((s.n_sc + C - 1) / C + 3) & ~3;
  s.p0 = min(s.n_sc, c * s.ch);
  s.p1 = min(s.n_sc, s.p0 + s.ch);
  s.e0 = max(s.p0, s.lo);
  s.e1 = max(s.e0, min(s.p1, s.hi));
  s.need_radix = s.keff > 0 && s.keff < ne;
  return 0;
}

// The three launches are programmatic dependents of the launch before them:
// each may be scheduled while its predecessor drains, and waits for it before
// any global access.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch 1 (fused mode): this chunk's sum of key norms over E.
__global__ void __launch_bounds__(kSelNuT) sel_nu_kernel(const SelectArgs a) {
  __shared__ float sh[33];
  pdl_wait();
  pdl_trigger();
  SelUnit s;
  if (sel_unit(a, blockIdx.y, blockIdx.x, gridDim.x, s) != 0) return;
  const float* kn = a.knorm + size_t(s.u) * a.max_len;
  float part = 0.f;
  constexpr int V = 16;  // loads in flight per thread
  for (int base = s.e0; base < s.e1; base += kSelNuT * V) {
    float x[V];
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const int i = base + j * kSelNuT + int(threadIdx.x);
      x[j] = i < s.e1 ? kn[i] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < V; ++j) part += x[j];
  }
  const float t = sel_block_sum(part, sh);
  if (threadIdx.x == 0) a.sel_nu[size_t(s.u) * kSelMaxChunks + blockIdx.x] = t;
}

// Launch 2: scores, order keys and the top-digit histogram.  EV_G > 0: the
// evidence comes from the attention kernel's log2-scaled logits [pos][EV_G]
// and per-head (M, Z) (decode path); EV_G == 0: `evidence` holds f (or the
// per-KV-head logit sums).
template <int EV_G>
__global__ void __launch_bounds__(kSelT, 2) sel_score_kernel(const SelectArgs a) {
  __shared__ uint32_t hist[kRadixBins];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, c = blockIdx.x;
  SelUnit s;
  const int r = sel_unit(a, blockIdx.y, c, gridDim.x, s);
  if (r != 0) {
    if (r == 2 && c == 0 && tid == 0) set_status(a.status, SFI_DEV_LEN_OVER_CAP);
    return;  // uniform over the unit
  }
  float coef = 0.f;
  if (s.prior) {
    // the chunks' key-norm sums in one fixed order: every thread of every CTA
    // of the unit forms the same value
    const float* pn = a.sel_nu + size_t(s.u) * kSelMaxChunks;
    const int lane = tid & 31, C = gridDim.x;
    float x = (lane < C ? pn[lane] : 0.f) + (lane + 32 < C ? pn[lane + 32] : 0.f);
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_down_sync(kFull, x, o);
    x = __shfl_sync(kFull, x, 0);
    coef = x > 0.f ? a.lambda / x : 0.f;
  }
  if (s.need_radix)
    for (int i = tid; i < kRadixBins; i += kSelT) hist[i] = 0;
  __syncthreads();
  float M[EV_G > 0 ? EV_G : 1], iz[EV_G > 0 ? EV_G : 1];
  if constexpr (EV_G > 0) {
#pragma unroll
    for (int hh = 0; hh < EV_G; ++hh) {
      const size_t qh = size_t(s.b) * a.H_q + size_t(s.unit % a.H_kv) * EV_G + hh;
      M[hh] = a.stats[qh * 2];
      iz[hh] = 1.0f / a.stats[qh * 2 + 1];
    }
  }
  const float* kn = s.prior ? a.knorm + size_t(s.u) * a.max_len : nullptr;
  float* srow = a.s ? a.s + size_t(s.u) * a.max_len : nullptr;
  // exclusivity: the fused score is written to s as it is; the selection
  // ranks it times exp(-beta * picks of the earlier KV heads)
  const uint8_t* exrow = s.prior && a.excl ? a.excl + size_t(s.b) * a.max_len : nullptr;
  uint32_t* krow = a.sel_keys + size_t(s.u) * a.max_len;
  int32_t* out_idx = a.idx + size_t(s.per_seq ? s.b * a.H_kv : s.unit) * a.k;
  const int n_rows = s.per_seq ? a.H_kv : 1;  // idx rows that receive the set
  const float w_f = s.prior ? 1.0f - a.lambda : 1.0f;
  // U positions per thread at a time, every load issued before any is used
  // (fewer when each position brings G logits, so two CTAs fit an SM)
  constexpr int U = EV_G >= 8 ? 2 : (EV_G >= 4 ? 4 : kSelU);
  for (int base = s.p0; base < s.p1; base += kSelT * U) {
    float lg[U][EV_G > 0 ? EV_G : 1];
    float ev[U], kv[U];
    uint32_t cx[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int i = base + j * kSelT + tid;
      const bool e = i >= s.lo && i < s.hi;
      ev[j] = 0.f;
      kv[j] = 0.f;
      cx[j] = 0u;
      if (i < s.p1) {
        if constexpr (EV_G > 0) {
          load_row<EV_G>(a.logits + (size_t(s.u) * a.max_len + i) * EV_G, lg[j]);
        } else if (s.per_seq) {
          for (int g = 0; g < a.H_kv; ++g)
            ev[j] += a.evidence[(size_t(s.b) * a.H_kv + g) * a.max_len + i];
        } else {
          ev[j] = a.evidence[size_t(s.u) * a.max_len + i];
        }
        if (s.prior && e) kv[j] = kn[i];
        if (exrow && e) cx[j] = exrow[i];
      }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int i = base + j * kSelT + tid;
      const bool in = i < s.p1;
      const bool e = in && i >= s.lo && i < s.hi;
      uint32_t key = 0u;
      if (in) {
        if constexpr (EV_G > 0) ev[j] = evidence_from_logits<EV_G>(lg[j], M, iz);
        float v = w_f * ev[j];
        if (s.prior && e) v = fmaf(coef, kv[j], v);
        if (srow) srow[i] = v;
        v *= excl_factor(cx[j], a.excl_beta);
        key = order_key(v);
        if (e) {
          if (s.need_radix) {
            krow[i] = key;
          } else {  // keep all of E: position lo + t goes to slot t
            for (int g = 0; g < n_rows; ++g) out_idx[size_t(g) * a.k + (i - s.lo)] = i;
          }
        }
      }
      if (s.need_radix) hist_add(hist, key >> kRadixShift0, e);
    }
  }
  if (c == 0 && tid == 0) {
    if (s.per_seq) {
      for (int g = 0; g < a.H_kv; ++g) a.count[s.b * a.H_kv + g] = s.keff;
    } else {
      a.count[s.u] = s.keff;
    }
  }
  if (s.need_radix) {
    __syncthreads();
    uint32_t* gh = a.sel_hist + size_t(s.u) * kRadixBins;
    for (int i = tid; i < kRadixBins; i += kSelT)
      if (hist[i]) atomicAdd(gh + i, hist[i]);
  }
}

// Launch 3: per chunk, the ordered list of keys at or above the k-th key's
// top digit, and the histogram of the next 11 bits of its keys in that
// digit's bin; the unit's last chunk CTA to finish completes the selection.
__global__ void __launch_bounds__(kSelT) sel_list_kernel(const SelectArgs a) {
  __shared__ uint32_t hist[kRadixBins];
  extern __shared__ unsigned long long lst[];     // finisher: the unit's list (kListCap entries)
  __shared__ uint32_t cnt_c[kSelMaxChunks + 1];  // finisher: entries per chunk
  __shared__ uint32_t offs_c[kSelMaxChunks + 1]; // finisher: their exclusive offsets
  __shared__ uint32_t gt_c[kSelMaxChunks + 1];   // finisher: keys above tau per chunk, then offsets
  __shared__ uint32_t eq_c[kSelMaxChunks + 1];   // finisher: keys equal to tau per chunk, then offsets
  __shared__ uint32_t scan_sh[33];
  __shared__ uint32_t sh_digit, sh_above, sh_last;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, c = blockIdx.x, C = gridDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kSelT / 32;
  const unsigned lt = (1u << lane) - 1u;
  SelUnit s;
  if (sel_unit(a, blockIdx.y, c, C, s) != 0 || !s.need_radix) return;  // uniform over the unit
  const uint32_t* krow = a.sel_keys + size_t(s.u) * a.max_len;
  const size_t row0 = size_t(s.u) * a.max_len;
  uint32_t* gh = a.sel_hist + size_t(s.u) * kRadixBins;
  uint32_t* gh2 = a.sel_hist2 + size_t(s.u) * kRadixBins;
  // this chunk's keys (thread t: kRun consecutive positions of each tile of
  // kSelT * kRun) are loaded together with the unit's histogram
  const int ntile = (s.e1 - s.e0 + kSelT * kRun - 1) / (kSelT * kRun);
  const bool one_tile = ntile <= 1;
  uint32_t key[kRun];
  const int i0 = s.e0 + tid * kRun;
  if (one_tile) {
#pragma unroll
    for (int j = 0; j < kRun; ++j) key[j] = i0 + j < s.e1 ? krow[i0 + j] : 0u;
  }
  for (int i = tid; i < kRadixBins; i += kSelT) hist[i] = __ldcg(gh + i);
  __syncthreads();
  block_pick_digit<kRadixBins>(hist, uint32_t(s.keff), &sh_digit, &sh_above, scan_sh);
  const uint32_t d0 = sh_digit;
  const uint32_t krem0 = uint32_t(s.keff) - sh_above;
  for (int i = tid; i < kRadixBins; i += kSelT) hist[i] = 0;  // now: next-digit histogram
  __syncthreads();
  // ---- keys at or above d0, in position order, into this chunk's region of
  // the unit's list (starting at its first position of E); one block scan per
  // tile; the keys of bin d0 also go into the next-digit histogram
  unsigned long long* lrow = a.sel_list + row0 + s.e0;
  uint32_t tot = 0;
  for (int t = 0; t < ntile; ++t) {
    const int ib = s.e0 + t * kSelT * kRun + tid * kRun;
    if (!one_tile) {
#pragma unroll
      for (int j = 0; j < kRun; ++j) key[j] = ib + j < s.e1 ? krow[ib + j] : 0u;
    }
    uint32_t nm = 0;
#pragma unroll
    for (int j = 0; j < kRun; ++j) nm += (ib + j < s.e1 && (key[j] >> kRadixShift0) >= d0) ? 1u : 0u;
    uint32_t ttot;
    uint32_t at = tot + block_excl_scan(nm, scan_sh, ttot);
#pragma unroll
    for (int j = 0; j < kRun; ++j) {
      const bool in = ib + j < s.e1;
      const uint32_t dg = key[j] >> kRadixShift0;
      if (in && dg >= d0)
        lrow[at++] = (static_cast<unsigned long long>(key[j]) << 32) | uint32_t(ib + j);
      hist_add(hist, (key[j] >> kRadixShift1) & (kRadixBins - 1), in && dg == d0);
    }
    tot += ttot;
  }
  __syncthreads();
  for (int i = tid; i < kRadixBins; i += kSelT)
    if (hist[i]) atomicAdd(gh2 + i, hist[i]);
  if (tid == 0) a.sel_cnt[size_t(s.u) * kSelMaxChunks + c] = tot;
  __threadfence();
  __syncthreads();
  if (tid == 0) sh_last = atomicAdd(a.sel_done + s.u, 1u) == uint32_t(C - 1);
  __syncthreads();
  if (!sh_last) return;
  __threadfence();

  // ---------------------------------------------------------------- finisher
  // The second digit d1 comes from the chunks' next-digit histograms; the
  // last 10 bits from the few keys with prefix (d0, d1).  Every walk over the
  // lists gives each warp whole chunks (entries of chunk c: kRun per lane in
  // flight, in position order) -- no search for an entry's chunk.
  for (int i = tid; i < kRadixBins; i += kSelT) hist[i] = __ldcg(gh2 + i);
  for (int i = tid; i < C; i += kSelT) {
    cnt_c[i] = __ldcg(a.sel_cnt + size_t(s.u) * kSelMaxChunks + i);
    gt_c[i] = 0u;
    eq_c[i] = 0u;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive entry offsets of the chunks (two per lane)
    const uint32_t x0 = lane < C ? cnt_c[lane] : 0u, x1 = lane + 32 < C ? cnt_c[lane + 32] : 0u;
    uint32_t i0 = x0, i1 = x1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y0 = __shfl_up_sync(kFull, i0, o), y1 = __shfl_up_sync(kFull, i1, o);
      if (lane >= o) i0 += y0, i1 += y1;
    }
    const uint32_t t0 = __shfl_sync(kFull, i0, 31);
    offs_c[lane] = i0 - x0;
    offs_c[lane + 32] = t0 + i1 - x1;
    if (lane == 31) offs_c[kSelMaxChunks] = t0 + i1;
  }
  block_pick_digit<kRadixBins>(hist, krem0, &sh_digit, &sh_above, scan_sh);  // (barriers)
  const uint32_t p1 = (d0 << (kRadixShift0 - kRadixShift1)) | sh_digit;  // top 22 bits
  const uint32_t krem1 = krem0 - sh_above;
  const uint32_t NE = offs_c[C];  // chunks past C count 0
  // The unit's list, staged in shared memory when it fits: every thread
  // loads kRun * 2 entries at once (the entry's chunk from the offsets), so
  // the walks below read shared memory only.
  const bool staged = NE <= uint32_t(kListCap);
  if (staged) {
    constexpr int V = 2 * kRun;
    for (uint32_t tb = 0; tb < NE; tb += kSelT * V) {
      unsigned long long ent[V];
#pragma unroll
      for (int r = 0; r < V; ++r) {
        const uint32_t e = tb + uint32_t(r) * kSelT + tid;
        ent[r] = 0ull;
        if (e < NE) {
          int lo = 0, hi = C - 1;  // chunk holding e: the largest c with offs_c[c] <= e
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (offs_c[mid] <= e) lo = mid;
            else hi = mid - 1;
          }
          ent[r] = __ldcg(a.sel_list + row0 + sel_chunk_e0(s, lo) + (e - offs_c[lo]));
        }
      }
#pragma unroll
      for (int r = 0; r < V; ++r) {
        const uint32_t e = tb + uint32_t(r) * kSelT + tid;
        if (e < NE) lst[e] = ent[r];
      }
    }
  }
  for (int i = tid; i < kRadixBins; i += kSelT) hist[i] = 0;
  __syncthreads();
  // each warp takes whole chunks, their entries in position order
  auto walk = [&](auto&& body) {
    for (int cc = warp; cc < C; cc += NW) {
      const uint32_t nc = cnt_c[cc];
      if (staged) {
        const unsigned long long* lc = lst + offs_c[cc];
        for (uint32_t jb = 0; jb < nc; jb += 32) {
          const uint32_t jj = jb + lane;
          body(cc, jj < nc, jj < nc ? lc[jj] : 0ull);
        }
      } else {
        const unsigned long long* lc = a.sel_list + row0 + sel_chunk_e0(s, cc);
        for (uint32_t jb = 0; jb < nc; jb += 32 * kRun) {
          unsigned long long ent[kRun];
#pragma unroll
          for (int r = 0; r < kRun; ++r) {
            const uint32_t jj = jb + uint32_t(r) * 32 + lane;
            ent[r] = jj < nc ? __ldcg(lc + jj) : 0ull;
          }
#pragma unroll
          for (int r = 0; r < kRun; ++r) body(cc, jb + uint32_t(r) * 32 + lane < nc, ent[r]);
        }
      }
    }
  };
  // last 10 bits among the keys with prefix p1
  walk([&](int, bool v, unsigned long long e) {
    const uint32_t k = uint32_t(e >> 32);
    hist_add(hist, k & ((1u << kRadixShift1) - 1u), v && (k >> kRadixShift1) == p1);
  });
  __syncthreads();
  block_pick_digit<1 << kRadixShift1>(hist, krem1, &sh_digit, &sh_above, scan_sh);
  const uint32_t tau = (p1 << kRadixShift1) | sh_digit;
  const uint32_t take_eq = krem1 - sh_above;
  // keys above tau and equal to it, per chunk
  walk([&](int cc, bool v, unsigned long long e) {
    const uint32_t k = uint32_t(e >> 32);
    const uint32_t ng = __popc(__ballot_sync(kFull, v && k > tau));
    const uint32_t nq = __popc(__ballot_sync(kFull, v && k == tau));
    if (lane == 0) {  // chunks are walked by one warp each: plain adds
      gt_c[cc] += ng;
      eq_c[cc] += nq;
    }
  });
  __syncthreads();
  if (warp == 0) {  // exclusive offsets over the chunks (two per lane)
    const uint32_t g0 = lane < C ? gt_c[lane] : 0u, g1 = lane + 32 < C ? gt_c[lane + 32] : 0u;
    const uint32_t q0 = lane < C ? eq_c[lane] : 0u, q1 = lane + 32 < C ? eq_c[lane + 32] : 0u;
    uint32_t ig0 = g0, ig1 = g1, iq0 = q0, iq1 = q1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t a0 = __shfl_up_sync(kFull, ig0, o), a1 = __shfl_up_sync(kFull, ig1, o);
      const uint32_t b0 = __shfl_up_sync(kFull, iq0, o), b1 = __shfl_up_sync(kFull, iq1, o);
      if (lane >= o) ig0 += a0, ig1 += a1, iq0 += b0, iq1 += b1;
    }
    const uint32_t tg = __shfl_sync(kFull, ig0, 31), tq = __shfl_sync(kFull, iq0, 31);
    __syncwarp();
    if (lane < C) gt_c[lane] = ig0 - g0, eq_c[lane] = iq0 - q0;
    if (lane + 32 < C) gt_c[lane + 32] = tg + ig1 - g1, eq_c[lane + 32] = tq + iq1 - q1;
  }
  __syncthreads();
  // ordered output: entry goes to slot (keys above tau before it) +
  // min(keys equal to tau before it, take_eq) -- the keys above tau, then the
  // lowest-positioned take_eq keys equal to it, all in position order
  int32_t* out_idx = a.idx + size_t(s.per_seq ? s.b * a.H_kv : s.unit) * a.k;
  const int n_rows = s.per_seq ? a.H_kv : 1;
  int cur = -1;
  uint32_t gb = 0, qb = 0;
  walk([&](int cc, bool v, unsigned long long e) {
    if (cc != cur) {
      cur = cc;
      gb = gt_c[cc];
      qb = eq_c[cc];
    }
    const uint32_t k = uint32_t(e >> 32);
    const int pos = int(uint32_t(e));
    const unsigned bg = __ballot_sync(kFull, v && k > tau);
    const unsigned bq = __ballot_sync(kFull, v && k == tau);
    const uint32_t g_at = gb + __popc(bg & lt), q_at = qb + __popc(bq & lt);
    // slots stay below keff for consistent counts; the bound only guards the
    // output row against an inconsistent list
    if ((bg >> lane) & 1u) {
      const uint32_t slot = g_at + min(q_at, take_eq);
      if (slot < uint32_t(s.keff))
        for (int g = 0; g < n_rows; ++g) out_idx[size_t(g) * a.k + slot] = pos;
    } else if (((bq >> lane) & 1u) && q_at < take_eq && g_at + q_at < uint32_t(s.keff)) {
      for (int g = 0; g < n_rows; ++g) out_idx[size_t(g) * a.k + g_at + q_at] = pos;
    }
    gb += __popc(bg);
    qb += __popc(bq);
  });
  __syncthreads();
  // leave the histograms and the counter at zero for the next launch
  for (int i = tid; i < kRadixBins; i += kSelT) {
    gh[i] = 0u;
    gh2[i] = 0u;
  }
  if (tid == 0) a.sel_done[s.u] = 0u;
}

cudaError_t launch_fpass(const FpassArgs& a, cudaStream_t st) {
  const int G = a.H_q / a.H_kv;
  const int sms = device_sm_count();
  const int units = a.B * a.H_kv;
  int gx = (a.max_len + kFpassThreads * 4 - 1) / (kFpassThreads * 4);
  const int want = (sms * 8 + units - 1) / units;  // enough CTAs to fill the GPU
  gx = max(1, min(gx, max(want, 1)));
  const dim3 grid(gx, units);
  switch (G) {
    case 1: fpass_kernel<1><<<grid, kFpassThreads, 0, st>>>(a); break;
    case 2: fpass_kernel<2><<<grid, kFpassThreads, 0, st>>>(a); break;
    case 4: fpass_kernel<4><<<grid, kFpassThreads, 0, st>>>(a); break;
    case 8: fpass_kernel<8><<<grid, kFpassThreads, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// Chunks per unit: about two CTAs per SM over all selecting units, chunks of
// at least kSelMinChunk positions, at most kSelMaxChunks.
int select_chunks(int units, int max_len) {
  const int sms = device_sm_count();
  int C = (2 * sms + units - 1) / units;
  C = min(C, kSelMaxChunks);
  C = min(C, max(1, (max_len + kSelMinChunk - 1) / kSelMinChunk));
  return max(C, 1);
}

template <typename K>
cudaError_t launch_dependent(K kernel, dim3 grid, int threads, cudaStream_t st,
                             const SelectArgs& a, size_t smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int EV_G>
cudaError_t launch_select_t(const SelectArgs& a, cudaStream_t st) {
  int n_active = 0;
  for (int b = 0; b < a.B; ++b) n_active += int((a.active.bits[b >> 5] >> (b & 31)) & 1u);
  const bool one_unit =
      a.mode == SFI_SELECT_LOGIT_SUM_SEQ || (a.mode == SFI_SELECT_FUSED && a.g_only >= 0);
  const int units = n_active * (one_unit ? 1 : a.H_kv);
  if (units == 0) return cudaSuccess;
  const dim3 grid(select_chunks(units, a.max_len), units);
  cudaError_t e = cudaSuccess;
  if (a.mode == SFI_SELECT_FUSED) e = launch_dependent(sel_nu_kernel, grid, kSelNuT, st, a);
  if (e == cudaSuccess) e = launch_dependent(sel_score_kernel<EV_G>, grid, kSelT, st, a);
  if (e == cudaSuccess) {
    const size_t smem = size_t(kListCap) * sizeof(unsigned long long);
    e = cudaFuncSetAttribute(sel_list_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e == cudaSuccess) e = launch_dependent(sel_list_kernel, grid, kSelT, st, a, smem);
  }
  return e;
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t st) {
  if (!a.logits) return launch_select_t<0>(a, st);
  switch (a.H_q / a.H_kv) {
    case 1: return launch_select_t<1>(a, st);
    case 2: return launch_select_t<2>(a, st);
    case 4: return launch_select_t<4>(a, st);
    case 8: return launch_select_t<8>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sfi
