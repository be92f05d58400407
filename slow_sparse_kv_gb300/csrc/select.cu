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
// Selector: one CTA of 1024 threads per (sequence, KV head) -- or per
// sequence in logit-sum mode.  Pass 1 sums the key norms over the eligible
// set E; pass 2 writes s for every position and builds the histogram of the
// top 8 bits of the order key of s over E; three more 8-bit radix passes
// find the exact k-th largest key tau and how many keys equal to tau to
// keep; a final pass compacts the chosen positions in ascending order (keys
// above tau, then the lowest-positioned keys equal to tau), so ties go to
// the lower position exactly as the definition says.  Histograms use
// warp-aggregated shared-memory atomics (the score distribution is very
// skewed, so many lanes hit the same bin).
#include <math.h>

#include "common.cuh"

namespace sfi {

constexpr int kSelThreads = 1024;
constexpr int kFpassThreads = 256;

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
  const float inv_g = 1.0f / float(G);
  const float* lrow = a.logits + size_t(u) * a.max_len * G;
  float* frow = a.f + size_t(u) * a.max_len;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const float* l = lrow + size_t(i) * G;
    float acc = 0.f;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) acc = fmaf(exp2f(l[hh] - M[hh]), iz[hh], acc);
    frow[i] = acc * inv_g;
  }
}

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
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

__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active) {
  const unsigned m = __ballot_sync(kFull, active);
  if (active) {
    const unsigned peers = __match_any_sync(m, bin);
    const int leader = __ffs(peers) - 1;
    if ((threadIdx.x & 31) == leader) atomicAdd(hist + bin, uint32_t(__popc(peers)));
  }
}

// Pick the digit d with above(d) < krem <= above(d) + hist[d], where
// above(d) counts keys in higher bins.  Warp 0 only.
__device__ void pick_digit(const uint32_t* hist, uint32_t krem, uint32_t* out_digit,
                           uint32_t* out_above) {
  const int lane = threadIdx.x & 31;
  uint32_t c[8];
  uint32_t sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = hist[255 - 8 * lane - j];
    sum += c[j];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t excl = incl - sum;
  if (excl < krem && krem <= incl) {
    uint32_t accum = excl;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (accum + c[j] >= krem) {
        *out_digit = uint32_t(255 - 8 * lane - j);
        *out_above = accum;
        break;
      }
      accum += c[j];
    }
  }
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelectArgs a) {
  __shared__ uint32_t hist[256];
  __shared__ float shf[33];
  __shared__ unsigned long long scan_w[33];
  __shared__ uint32_t sh_digit, sh_above;

  const int tid = threadIdx.x;
  const bool per_seq = a.mode == SFI_SELECT_LOGIT_SUM_SEQ;
  const int b = per_seq ? blockIdx.x : blockIdx.x / a.H_kv;
  if (!seq_is_slow(a.active, b)) return;
  const int u = per_seq ? b * a.H_kv : blockIdx.x;  // row of s / evidence used for scores
  const int n = a.len[b];
  if (n < 1 || n > a.max_len) {
    if (tid == 0) set_status(a.status, SFI_DEV_LEN_OVER_CAP);
    return;
  }
  const int lo = per_seq ? 0 : a.n_sink;
  const int hi = max(lo, n - a.window);
  const int ne = hi - lo;
  const int keff = min(a.k, ne);
  float* srow = a.s + size_t(u) * a.max_len;

  // ---------------------------------------------------------------- scores
  for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
  float coef = 0.f;
  if (!per_seq) {
    const float* kn = a.knorm + size_t(u) * a.max_len;
    float part = 0.f;
    for (int i = lo + tid; i < hi; i += kSelThreads) part += kn[i];
    const float tot = sel_block_sum(part, shf);
    coef = tot > 0.f ? a.lambda / tot : 0.f;
  }
  __syncthreads();
  const bool need_radix = keff > 0 && keff < ne;
  {
    const float* ev = a.evidence + size_t(u) * a.max_len;
    const float* kn = per_seq ? nullptr : a.knorm + size_t(u) * a.max_len;
    const int n_s = per_seq ? hi : n;  // positions that get a score
    const float w_f = 1.0f - a.lambda;
    for (int base = 0; base < n_s; base += kSelThreads) {
      const int i = base + tid;
      const bool in = i < n_s;
      float sc = 0.f;
      if (in) {
        if (per_seq) {
          for (int g = 0; g < a.H_kv; ++g) sc += a.evidence[(size_t(b) * a.H_kv + g) * a.max_len + i];
        } else {
          sc = w_f * ev[i];
          if (i >= lo && i < hi) sc = fmaf(coef, kn[i], sc);
        }
        srow[i] = sc;
      }
      if (need_radix) hist_add(hist, order_key(sc) >> 24, in && i >= lo && i < hi);
    }
  }
  __syncthreads();

  int32_t* out_idx = a.idx + size_t(blockIdx.x * (per_seq ? a.H_kv : 1)) * a.k;
  if (!need_radix) {
    // keep all of E (or nothing)
    for (int j = tid; j < keff; j += kSelThreads) out_idx[j] = lo + j;
  } else {
    // ------------------------------------------------------------ radix select
    uint32_t prefix = 0, krem = uint32_t(keff);
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      if (pass > 0) {
        for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
        __syncthreads();
        for (int base = lo; base < hi; base += kSelThreads) {
          const int i = base + tid;
          const bool in = i < hi;
          const uint32_t key = in ? order_key(srow[i]) : 0u;
          const bool match = in && (key >> (shift + 8)) == prefix;
          hist_add(hist, (key >> shift) & 255u, match);
        }
        __syncthreads();
      }
      if (tid < 32) pick_digit(hist, krem, &sh_digit, &sh_above);
      __syncthreads();
      prefix = (prefix << 8) | sh_digit;
      krem -= sh_above;
      __syncthreads();
    }
    const uint32_t tau = prefix;
    const uint32_t take_eq = krem;
    // ------------------------------------------------------------ compaction
    const int ch = (ne + kSelThreads - 1) / kSelThreads;
    const int c0 = lo + tid * ch, c1 = min(hi, c0 + ch);
    uint32_t cg = 0, ceq = 0;
    for (int i = c0; i < c1; ++i) {
      const uint32_t key = order_key(srow[i]);
      cg += key > tau;
      ceq += key == tau;
    }
    unsigned long long v = (static_cast<unsigned long long>(cg) << 32) | ceq;
    const int lane = tid & 31, w = tid >> 5;
    unsigned long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) scan_w[w] = incl;
    __syncthreads();
    if (tid == 0) {
      unsigned long long s = 0;
      for (int i = 0; i < kSelThreads / 32; ++i) {
        const unsigned long long x = scan_w[i];
        scan_w[i] = s;
        s += x;
      }
    }
    __syncthreads();
    const unsigned long long ex = scan_w[w] + incl - v;
    uint32_t gt_before = uint32_t(ex >> 32), eq_before = uint32_t(ex & 0xffffffffu);
    for (int i = c0; i < c1; ++i) {
      const uint32_t key = order_key(srow[i]);
      if (key > tau) {
        out_idx[gt_before + min(eq_before, take_eq)] = i;
        ++gt_before;
      } else if (key == tau) {
        if (eq_before < take_eq) out_idx[gt_before + eq_before] = i;
        ++eq_before;
      }
    }
  }
  if (tid == 0) {
    if (per_seq) {
      for (int g = 0; g < a.H_kv; ++g) a.count[b * a.H_kv + g] = keff;
    } else {
      a.count[u] = keff;
    }
  }
  if (per_seq && a.H_kv > 1) {
    // every KV head of the sequence reads the same selected set
    __syncthreads();
    for (int g = 1; g < a.H_kv; ++g)
      for (int j = tid; j < keff; j += kSelThreads) out_idx[size_t(g) * a.k + j] = out_idx[j];
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

cudaError_t launch_select(const SelectArgs& a, cudaStream_t st) {
  const int grid = a.mode == SFI_SELECT_LOGIT_SUM_SEQ ? a.B : a.B * a.H_kv;
  select_kernel<<<grid, kSelThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sfi
