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
// Selector: one thread-block cluster of 8 CTAs (512 threads each) per
// (sequence, KV head) -- or per sequence in the per-sequence logit-sum mode
// -- launched for the refreshing sequences only.  Each CTA holds the scores
// of one eighth of the positions in shared memory.  The evidence pass forms
// f (from the logits on the decode path) and the CTA's part of the key-norm
// sum over E; after a cluster barrier every CTA writes s and the histogram of
// the top 11 bits of the order key of s over E.  The cluster total of that
// histogram fixes the top digit of the k-th largest key; the keys in that
// bin (few, at the decode workloads) are gathered in rank 0, which finds the
// two lower digits (11 and 10 bits) alone -- or, when the bin holds more than
// kCandCap keys, every CTA runs the two passes over all its keys.  A final
// ordered compaction writes the keys above tau, then the lowest-positioned
// keys equal to tau, in ascending position order, so ties go to the lower
// position exactly as the definition says.  Histograms use warp-aggregated
// shared-memory atomics (the score distribution is very skewed, so many
// lanes hit the same bin).
#include <cooperative_groups.h>
#include <math.h>

#include "common.cuh"
#include "warp_hist.cuh"

namespace sfi {

constexpr int kFpassThreads = 256;
constexpr int kSelCluster = 8;   // CTAs per unit
constexpr int kSelCT = 512;      // threads per selector CTA

constexpr int kSelU = 8;         // positions in flight per selector thread
constexpr int kRadixPasses = 3;  // digits of 11, 11 and 10 bits
constexpr int kRadixBins = 2048;
constexpr int kRadixShift0 = 21;
constexpr int kRadixShift1 = 10;
// Largest cluster-wide count of keys in the k-th key's top bin for which the
// two lower digits are found on a gathered list (it must fit two rows of the
// total histograms).
constexpr int kCandCap = 4096;
static_assert(kCandCap <= (kRadixPasses - 1) * kRadixBins, "gathered list fits hist_g rows 1..2");

// Dynamic shared memory of a selector CTA: its scores (ceil(max_len / 8)
// floats), the candidate list, and, when it fits, a copy of its key norms.
__host__ __device__ constexpr size_t select_cand_offset(int max_len) {
  return (size_t((max_len + kSelCluster - 1) / kSelCluster) * sizeof(float) + 15) / 16 * 16;
}
__host__ __device__ constexpr size_t select_kn_offset(int max_len) {
  return select_cand_offset(max_len) + size_t(kCandCap) * sizeof(uint32_t);
}

// Eight consecutive scores sc[o .. o+7] (o a multiple of 8, scores past `lim`
// read as 0); two 16-byte shared-memory loads when the block is in range.
__device__ __forceinline__ void load8(const float* sc, int o, int lim, float (&v)[8]) {
  if (o + 8 <= lim) {
    const float4 a = *reinterpret_cast<const float4*>(sc + o);
    const float4 b = *reinterpret_cast<const float4*>(sc + o + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = o + j < lim ? sc[o + j] : 0.f;
  }
}

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
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if (lane == 0) sh[w] = v;
  __syncthreads();
  if (w == 0) {
    v = lane < int(blockDim.x >> 5) ? sh[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
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
// NB / kSelCT consecutive bins from the top, a block scan gives the count
// above its range, and the one thread whose range holds the krem-th key
// walks its bins.  0 < krem <= the histogram's total.  Ends with a barrier.
template <int NB>
__device__ void block_pick_digit(const uint32_t* hist, uint32_t krem, uint32_t* out_digit,
                                 uint32_t* out_above, uint32_t* scan_sh) {
  constexpr int PER = NB / kSelCT;
  static_assert(PER * kSelCT == NB, "bins split evenly over the block");
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

// One cluster of kSelCluster CTAs per unit; CTA `rank` owns the positions
// [rank * ch, (rank + 1) * ch) of [0, n) and keeps their scores in shared
// memory.  Cluster-wide quantities (the key-norm sum over E, the radix
// histograms, the compaction offsets) are exchanged through distributed
// shared memory; every CTA takes the same decisions from the same data.
// EV_G > 0: the evidence is computed here from the attention kernel's
// log2-scaled logits [pos][EV_G] and per-head (M, Z) (decode path); EV_G == 0:
// `evidence` holds f (or, per sequence, the per-KV-head logit sums).
template <int EV_G>
__global__ void __cluster_dims__(kSelCluster, 1, 1) __launch_bounds__(kSelCT)
    select_cluster_kernel(const SelectArgs a) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char sel_smem[];
  float* sc = reinterpret_cast<float*>(sel_smem);
  __shared__ uint32_t hist[kRadixBins];
  __shared__ uint32_t hist_loc[kRadixBins];  // this CTA's pass-0 histogram
  // cluster totals, used in rank 0; on the candidate path rows 1-2 hold the
  // gathered candidate keys
  __shared__ uint32_t hist_g[kRadixPasses][kRadixBins];
  // this CTA's keys in the k-th key's top bin (dynamic memory, after the scores)
  uint32_t* cand = reinterpret_cast<uint32_t*>(sel_smem + select_cand_offset(a.max_len));
  __shared__ uint32_t cand_n, sh_tau, sh_take, sh_off;
  __shared__ float shf[33];
  __shared__ float part_nu;
  __shared__ uint32_t cnt_gt, cnt_eq;
  __shared__ uint32_t sh_digit, sh_above;
  __shared__ uint32_t scan_sh[33];

  const int tid = threadIdx.x;
  const int rank = int(cl.block_rank());
  // clusters are launched for the active units only: cluster c serves the
  // (c / units-per-sequence)-th active sequence
  const bool per_seq = a.mode == SFI_SELECT_LOGIT_SUM_SEQ;
  const bool prior = a.mode == SFI_SELECT_FUSED;  // key-norm prior and (1 - lambda) weight
  const bool one_head = prior && a.g_only >= 0;  // only KV head g_only of each sequence
  const int ups = per_seq || one_head ? 1 : a.H_kv;  // units per sequence
  const int c = blockIdx.x / kSelCluster;
  const int b = active_seq(a.active, c / ups);
  if (b < 0 || b >= a.B) return;  // uniform over the cluster (cannot happen for a valid grid)
  const int unit = per_seq ? b : b * a.H_kv + (one_head ? a.g_only : c % ups);
  const int u = per_seq ? b * a.H_kv : unit;
  const int n = a.len[b];
  if (n < 1 || n > a.max_len) {
    if (tid == 0 && rank == 0) set_status(a.status, SFI_DEV_LEN_OVER_CAP);
    return;  // uniform over the cluster
  }
  const int lo = per_seq ? 0 : a.n_sink;
  const int hi = max(lo, n - a.window);
  const int ne = hi - lo;
  const int keff = min(a.k, ne);
  const int n_sc = per_seq ? hi : n;  // positions that receive a score
  const int ch = (n_sc + kSelCluster - 1) / kSelCluster;
  const int p0 = min(n_sc, rank * ch), p1 = min(n_sc, p0 + ch);
  const bool need_radix = keff > 0 && keff < ne;
  const float* kn = prior ? a.knorm + size_t(u) * a.max_len : nullptr;

  // ---------------------------------------------------------------- evidence
  float M[EV_G > 0 ? EV_G : 1], iz[EV_G > 0 ? EV_G : 1];
  if constexpr (EV_G > 0) {
#pragma unroll
    for (int hh = 0; hh < EV_G; ++hh) {
      const size_t qh = size_t(b) * a.H_q + size_t(unit % a.H_kv) * EV_G + hh;
      M[hh] = a.stats[qh * 2];
      iz[hh] = 1.0f / a.stats[qh * 2 + 1];
    }
  }
  // Positions are processed kSelU at a time per thread with every load
  // issued before any is used, so the loop is bound by bandwidth, not by the
  // latency of one load after another.
  float* kns = a.kn_smem ? reinterpret_cast<float*>(sel_smem + select_kn_offset(a.max_len)) : nullptr;
  float part = 0.f;
  for (int base = p0; base < p1; base += kSelCT * kSelU) {
    float lg[kSelU][EV_G > 0 ? EV_G : 1];
    float ev[kSelU], kv[kSelU];
#pragma unroll
    for (int j = 0; j < kSelU; ++j) {
      const int i = base + j * kSelCT + tid;
      ev[j] = 0.f;
      kv[j] = 0.f;
      if (i < p1) {
        if constexpr (EV_G > 0) {
          load_row<EV_G>(a.logits + (size_t(u) * a.max_len + i) * EV_G, lg[j]);
        } else if (per_seq) {
          for (int g = 0; g < a.H_kv; ++g) ev[j] += a.evidence[(size_t(b) * a.H_kv + g) * a.max_len + i];
        } else {
          ev[j] = a.evidence[size_t(u) * a.max_len + i];
        }
        if (prior && i >= lo && i < hi) kv[j] = kn[i];
      }
    }
#pragma unroll
    for (int j = 0; j < kSelU; ++j) {
      const int i = base + j * kSelCT + tid;
      if (i < p1) {
        if constexpr (EV_G > 0) ev[j] = evidence_from_logits<EV_G>(lg[j], M, iz);
        sc[i - p0] = ev[j];
        if (kns) kns[i - p0] = kv[j];
        part += kv[j];
      }
    }
  }
  for (int i = tid; i < kRadixBins; i += kSelCT) {
    hist[i] = 0;
    if (rank == 0) {
      for (int j = 0; j < kRadixPasses; ++j) hist_g[j][i] = 0;
    }
  }
  if (prior) {
    const float t = sel_block_sum(part, shf);
    if (tid == 0) part_nu = t;
  }
  cl.sync();  // partial norm sums and the zeroed cluster histograms are visible
  float coef = 0.f;
  if (prior) {
    float tot = 0.f;
    for (int r = 0; r < kSelCluster; ++r) tot += *cl.map_shared_rank(&part_nu, r);
    coef = tot > 0.f ? a.lambda / tot : 0.f;
  }
  // ---------------------------------------------------------------- scores
  float* srow = a.s ? a.s + size_t(u) * a.max_len : nullptr;
  const float w_f = prior ? 1.0f - a.lambda : 1.0f;
  // exclusivity: the fused score is written to s as it is; the selection
  // ranks it times exp(-beta * picks of the earlier KV heads)
  const uint8_t* exrow = prior && a.excl ? a.excl + size_t(b) * a.max_len : nullptr;
  for (int base = p0; base < p1; base += kSelCT * kSelU) {
    float kv[kSelU];
    uint32_t cx[kSelU];
#pragma unroll
    for (int j = 0; j < kSelU; ++j) {
      const int i = base + j * kSelCT + tid;
      const bool e = i < p1 && i >= lo && i < hi;
      kv[j] = (prior && e) ? (kns ? kns[i - p0] : kn[i]) : 0.f;
      cx[j] = exrow && e ? exrow[i] : 0u;
    }
#pragma unroll
    for (int j = 0; j < kSelU; ++j) {
      const int i = base + j * kSelCT + tid;
      const bool in = i < p1;
      float v = 0.f;
      if (in) {
        v = w_f * sc[i - p0];
        if (prior && i >= lo && i < hi) v = fmaf(coef, kv[j], v);
        if (srow) srow[i] = v;
        v *= excl_factor(cx[j], a.excl_beta);
        sc[i - p0] = v;
      }
      if (need_radix) hist_add(hist, order_key(v) >> kRadixShift0, in && i >= lo && i < hi);
    }
  }
  __syncthreads();

  int32_t* out_idx = a.idx + size_t(per_seq ? b * a.H_kv : unit) * a.k;
  if (need_radix) {
    // ------------------------------------------------------------ radix select
    // Digits of 11, 11 and 10 bits of the order keys of E.  Pass 0's
    // histogram was built with the scores; its cluster total gives the top
    // digit d0 of the k-th key.  Few keys share that digit (at the decode
    // workloads about 2% of E), so when at most kCandCap do, each CTA lists
    // its keys of bin d0 and rank 0 finishes the two lower digits on the
    // gathered list alone; otherwise every CTA runs the two passes over all
    // its keys.  Shared-memory reads go 8 positions per thread (two 16-byte
    // loads) in tiles aligned to the CTA's first position.
    uint32_t prefix = 0, krem = uint32_t(keff);
    const int e0 = max(p0, lo), e1 = min(p1, hi);
    for (int i = tid; i < kRadixBins; i += kSelCT) {
      hist_loc[i] = hist[i];
      if (hist[i]) atomicAdd(cl.map_shared_rank(&hist_g[0][i], 0), hist[i]);
    }
    if (tid == 0) cand_n = 0;
    cl.sync();
    for (int i = tid; i < kRadixBins; i += kSelCT) hist[i] = *cl.map_shared_rank(&hist_g[0][i], 0);
    __syncthreads();
    block_pick_digit<2048>(hist, krem, &sh_digit, &sh_above, scan_sh);
    const uint32_t d0 = sh_digit;
    prefix = d0;
    krem -= sh_above;
    const uint32_t n_cand = hist[d0];  // keys of E with top digit d0, cluster-wide
    uint32_t tau, take_eq;
    if (n_cand <= uint32_t(kCandCap)) {
      // ---- this CTA's keys of bin d0: into its own list and, at offset
      // (keys of bin d0 in lower ranks), into rank 0's gathered list (the
      // rows 1-2 of its total histograms, unused on this path)
      const int lane = tid & 31;
      if (tid < 32) {
        uint32_t v = tid < rank ? *cl.map_shared_rank(&hist_loc[d0], tid) : 0u;
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
        if (tid == 0) sh_off = v;
      }
      __syncthreads();
      const uint32_t my_off = sh_off;
      uint32_t* all_r0 = cl.map_shared_rank(&hist_g[1][0], 0);
      for (int tb = p0; tb < e1; tb += kSelCT * 8) {
        const int i0 = tb + tid * 8;
        float v8[8];
        load8(sc, i0 - p0, p1 - p0, v8);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = i0 + j;
          const uint32_t key = order_key(v8[j]);
          const bool m = i >= e0 && i < e1 && (key >> kRadixShift0) == d0;
          const unsigned bal = __ballot_sync(kFull, m);
          if (bal) {
            uint32_t base = 0;
            if (lane == 0) base = atomicAdd(&cand_n, uint32_t(__popc(bal)));
            base = __shfl_sync(kFull, base, 0);
            if (m) {
              const uint32_t at = base + __popc(bal & ((1u << lane) - 1u));
              cand[at] = key;
              all_r0[my_off + at] = key;
            }
          }
        }
      }
      cl.sync();  // every CTA's list is complete
      if (rank == 0) {
        const uint32_t* all = &hist_g[1][0];  // the n_cand gathered keys
        for (int pass = 1; pass < kRadixPasses; ++pass) {
          const int shift = pass == 1 ? kRadixShift1 : 0;
          const int width = pass == 1 ? kRadixShift0 - kRadixShift1 : kRadixShift1;
          const uint32_t dmask = (1u << width) - 1u;
          const int hs = shift + width;
          for (int i = tid; i < kRadixBins; i += kSelCT) hist[i] = 0;
          __syncthreads();
          for (uint32_t j0 = 0; j0 < n_cand; j0 += kSelCT) {
            const uint32_t j = j0 + tid;
            const uint32_t key = j < n_cand ? all[j] : 0u;
            hist_add(hist, (key >> shift) & dmask, j < n_cand && (key >> hs) == prefix);
          }
          __syncthreads();
          if (width == 11) block_pick_digit<2048>(hist, krem, &sh_digit, &sh_above, scan_sh);
          else block_pick_digit<1024>(hist, krem, &sh_digit, &sh_above, scan_sh);
          prefix = (prefix << width) | sh_digit;
          krem -= sh_above;
        }
        if (tid == 0) {
          sh_tau = prefix;
          sh_take = krem;
        }
      }
      cl.sync();  // tau is known in rank 0; no list is read any more
      tau = *cl.map_shared_rank(&sh_tau, 0);
      take_eq = *cl.map_shared_rank(&sh_take, 0);
    } else {
      for (int pass = 1; pass < kRadixPasses; ++pass) {
        const int shift = pass == 1 ? kRadixShift1 : 0;
        const int width = pass == 1 ? kRadixShift0 - kRadixShift1 : kRadixShift1;
        const uint32_t dmask = (1u << width) - 1u;
        const int hs = shift + width;
        for (int i = tid; i < kRadixBins; i += kSelCT) hist[i] = 0;
        __syncthreads();
        for (int tb = p0; tb < e1; tb += kSelCT * 8) {
          const int i0 = tb + tid * 8;
          float v8[8];
          load8(sc, i0 - p0, p1 - p0, v8);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int i = i0 + j;
            const uint32_t key = order_key(v8[j]);
            const bool m = i >= e0 && i < e1 && (key >> hs) == prefix;
            hist_add(hist, (key >> shift) & dmask, m);
          }
        }
        __syncthreads();
        for (int i = tid; i < kRadixBins; i += kSelCT)
          if (hist[i]) atomicAdd(cl.map_shared_rank(&hist_g[pass][i], 0), hist[i]);
        cl.sync();
        for (int i = tid; i < kRadixBins; i += kSelCT) hist[i] = *cl.map_shared_rank(&hist_g[pass][i], 0);
        __syncthreads();
        if (width == 11) block_pick_digit<2048>(hist, krem, &sh_digit, &sh_above, scan_sh);
        else block_pick_digit<1024>(hist, krem, &sh_digit, &sh_above, scan_sh);
        prefix = (prefix << width) | sh_digit;
        krem -= sh_above;
      }
      tau = prefix;
      take_eq = krem;
    }
    // ------------------------------------------------------------ compaction
    // Ascending positions: warp w walks the contiguous segment
    // [e0 + w * seg, ...) 32 positions per step (lane l takes base + l), so
    // the order is (rank, warp, step, lane).  A counting walk, one block scan
    // of the warps' counts and an exchange of the CTAs' totals give every
    // warp its first output slot.
    constexpr int NW = kSelCT / 32;
    const int lane = tid & 31, warp = tid >> 5;
    const int ne_cta = max(e1 - e0, 0);
    const int seg = ((ne_cta + NW - 1) / NW + 31) / 32 * 32;
    const int s0 = min(e1, e0 + warp * seg), s1 = min(e1, s0 + seg);
    uint32_t wg = 0, wq = 0;
    for (int base = s0; base < s1; base += 32) {
      const int i = base + lane;
      const uint32_t key = i < s1 ? order_key(sc[i - p0]) : 0u;
      wg += __popc(__ballot_sync(kFull, i < s1 && key > tau));
      wq += __popc(__ballot_sync(kFull, i < s1 && key == tau));
    }
    uint32_t tot;
    const uint32_t ex = block_excl_scan(lane == 0 ? (wg << 16) | wq : 0u, scan_sh, tot);  // < 2^16 per CTA
    const uint32_t w_ex = __shfl_sync(kFull, ex, 0);
    if (tid == 0) {
      cnt_gt = tot >> 16;
      cnt_eq = tot & 0xffffu;
    }
    cl.sync();
    uint32_t gb = w_ex >> 16, qb = w_ex & 0xffffu;
    for (int r = 0; r < rank; ++r) {
      gb += *cl.map_shared_rank(&cnt_gt, r);
      qb += *cl.map_shared_rank(&cnt_eq, r);
    }
    const unsigned lt = (1u << lane) - 1u;
    for (int base = s0; base < s1; base += 32) {
      const int i = base + lane;
      const uint32_t key = i < s1 ? order_key(sc[i - p0]) : 0u;
      const unsigned bg = __ballot_sync(kFull, i < s1 && key > tau);
      const unsigned bq = __ballot_sync(kFull, i < s1 && key == tau);
      const uint32_t g_at = gb + __popc(bg & lt), q_at = qb + __popc(bq & lt);
      if ((bg >> lane) & 1u) {
        out_idx[g_at + min(q_at, take_eq)] = i;
      } else if (((bq >> lane) & 1u) && q_at < take_eq) {
        out_idx[g_at + q_at] = i;
      }
      gb += __popc(bg);
      qb += __popc(bq);
    }
  } else {
    // keep all of E (or nothing): position lo + j goes to slot j
    const int e0 = max(p0, lo), e1 = min(min(p1, hi), lo + keff);
    for (int i = e0 + tid; i < e1; i += kSelCT) out_idx[i - lo] = i;
  }
  if (tid == 0 && rank == 0) {
    if (per_seq) {
      for (int g = 0; g < a.H_kv; ++g) a.count[b * a.H_kv + g] = keff;
    } else {
      a.count[u] = keff;
    }
  }
  cl.sync();  // every CTA's set is written, and no CTA leaves while others read its memory
  if (per_seq && a.H_kv > 1) {
    // every KV head of the sequence reads the same set; CTA `rank` copies its share
    const int cs = (keff + kSelCluster - 1) / kSelCluster;
    const int j0 = rank * cs, j1 = min(keff, j0 + cs);
    for (int g = 1; g < a.H_kv; ++g)
      for (int j = j0 + tid; j < j1; j += kSelCT) out_idx[size_t(g) * a.k + j] = out_idx[j];
  }
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

// Dynamic shared memory of a launch; the key-norm copy is kept when the CTA's
// total stays within 227 KB (the static part is about 41 KB).
size_t select_smem_bytes(int max_len, bool kn_smem) {
  const size_t base = select_kn_offset(max_len);
  return kn_smem ? base + size_t((max_len + kSelCluster - 1) / kSelCluster) * sizeof(float) : base;
}

bool select_kn_fits(int max_len) { return select_smem_bytes(max_len, true) <= size_t(180) * 1024; }

template <int EV_G>
cudaError_t launch_select_t(const SelectArgs& args, cudaStream_t st) {
  SelectArgs a = args;
  a.kn_smem = a.mode == SFI_SELECT_FUSED && select_kn_fits(a.max_len) ? 1 : 0;
  const size_t smem = select_smem_bytes(a.max_len, a.kn_smem != 0);
  cudaError_t e = cudaFuncSetAttribute(select_cluster_kernel<EV_G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  int n_active = 0;
  for (int b = 0; b < a.B; ++b) n_active += int((a.active.bits[b >> 5] >> (b & 31)) & 1u);
  const bool one_unit = a.mode == SFI_SELECT_LOGIT_SUM_SEQ || (a.mode == SFI_SELECT_FUSED && a.g_only >= 0);
  const int units = n_active * (one_unit ? 1 : a.H_kv);
  if (units == 0) return cudaSuccess;
  select_cluster_kernel<EV_G><<<units * kSelCluster, kSelCT, smem, st>>>(a);
  return cudaGetLastError();
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
