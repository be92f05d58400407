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
// positions, one CTA each, in one launch.  C is as large as keeps every CTA
// of the launch resident at once, so that all SMs work on the few units of a
// decode step; the C CTAs of a unit exchange, through the workspace, the
// key-norm sum, the histogram of the order keys' top 11 bits (integer
// atomics) and the keys of the k-th key's top bin, from which every CTA
// finds the lower 21 bits of the k-th key -- or, when that bin is crowded,
// two more digit histograms (11 + 10 bits) and their output counts -- and
// meet at three (up to five) barriers on a counter of the unit.  The keys
// stay in the CTA (shared memory) when they fit.  Ties at the k-th key go to the lower positions exactly as the
// definition says, and every sum runs in a fixed order, so the selection
// does not depend on the schedule.
#include <math.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "common.cuh"

namespace sfi {

constexpr int kFpassThreads = 256;
constexpr int kSelT = 512;      // threads of a selector CTA
constexpr int kSelU = 8;        // positions in flight per thread
constexpr int kRadixBins = 2048;
constexpr int kRadixShift0 = 21;  // digits: bits 31..21, 20..10, 9..0 of the order key
constexpr int kRadixShift1 = 10;
constexpr int kSelMinChunk = 2048;     // positions per chunk, at least
constexpr int kWalk = 8;               // keys per lane in flight in the walks over global keys
constexpr int kSelSmemMax = 100 << 10;  // dynamic shared memory of a selector CTA, at most

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

// Exclusive block scan of one value per thread (a packed pair of counts);
// also returns the block total.  Two barriers.
template <typename T>
__device__ __forceinline__ T block_excl_scan(T v, T* sh, T& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  T incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    T x = lane < nw ? sh[lane] : T(0);
    T xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(kFull, xi, o);
      if (lane >= o) xi += y;
    }
    if (lane < nw) sh[lane] = xi - x;
    if (lane == nw - 1) sh[32] = xi;
  }
  __syncthreads();
  total = sh[32];
  const T r = sh[w] + incl - v;
  __syncthreads();
  return r;
}

// Pick the digit d with above(d) < krem <= above(d) + hist[d] (above(d)
// counts the keys in higher bins), with the whole block: thread t sums
// NB / kSelT consecutive bins from the top, a block scan gives the count
// above its range, and the one thread whose range holds the krem-th key
// walks its bins.  0 < krem <= the histogram's total (else digit 0).  Ends
// with a barrier.
template <int NB>
__device__ __noinline__ void block_pick_digit(const uint32_t* hist, uint32_t krem, uint32_t* out_digit,
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
  // digit 0 unless a thread finds the krem-th key (a histogram left
  // inconsistent by a barrier wait that gave up): the digit stays in range
  if (threadIdx.x == 0) {
    *out_digit = 0u;
    *out_above = 0u;
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

// The launch is a programmatic dependent of the launch before it: it may be
// scheduled while its predecessor drains, and waits for it before any global
// access.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Barrier of the C chunk CTAs of one unit on the unit's counter, in two
// halves so that independent work can run between them.  The counter rests
// with its low 31 bits at zero: chunk 0 adds 2^31 - (C - 1) and every other
// chunk 1, so bit 31 flips exactly when the last CTA arrives and the low bits
// are back at zero -- no reset, whatever C the next launch has.  Arrive:
// after the block's writes, one release add; thread 0 keeps the value it
// replaced.  Wait: until bit 31 differs from that value's.  Every CTA
// arrives at every barrier once, also after one of its waits gave up; a
// wait gives up after `limit` SM clocks and sets SFI_DEV_WAIT_TIMEOUT, and
// returns false from then on (the CTA finishes without waiting).
__device__ __forceinline__ uint32_t unit_arrive(uint32_t* ctr, int c, int C) {
  __syncthreads();
  uint32_t old = 0;
  if (threadIdx.x == 0) {
    const uint32_t add = c == 0 ? 0x80000000u - uint32_t(C - 1) : 1u;
    asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;"
                 : "=r"(old) : "l"(ctr), "r"(add) : "memory");
  }
  return old;
}
__device__ __forceinline__ bool unit_wait(const uint32_t* ctr, uint32_t old, bool ok, long long limit,
                                          uint32_t* status, int* sh_ok) {
  if (threadIdx.x == 0) {
    if (ok && ((ld_acquire_u32(ctr) ^ old) & 0x80000000u) == 0) {
      const long long t0 = clock64();
      while (((ld_acquire_u32(ctr) ^ old) & 0x80000000u) == 0) {
        if (clock64() - t0 > limit) {
          ok = false;
          set_status(status, SFI_DEV_WAIT_TIMEOUT);
          break;
        }
      }
    }
    *sh_ok = ok ? 1 : 0;
  }
  __syncthreads();
  return *sh_ok != 0;
}

// Shared-memory histogram count (native shared atomics resolve equal bins
// within a warp faster than any software aggregation).
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active) {
  if (active) atomicAdd(hist + bin, 1u);
}

// Sum of one count per thread over the block.  Two barriers.
__device__ __forceinline__ uint32_t block_count(uint32_t v, uint32_t* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_down_sync(kFull, v, o);
  if (lane == 0) sh[w] = v;
  __syncthreads();
  uint32_t t = 0;
  for (int i = 0; i < int(blockDim.x >> 5); ++i) t += sh[i];
  __syncthreads();
  return t;
}

// The selector, one launch.  Block (c, j): chunk c of selecting unit j.
//  pass 1  (fused mode) the chunk's key norms over E and their sum, published
//          at barrier 1, whose wait comes after the evidence loads; the
//          chunk's evidence (f from the logits and (M, Z) on the decode path);
//  pass 2  the ranked scores, s when asked, the order keys (in shared memory
//          when the chunk fits, else in the workspace) and their top-11-bit
//          histogram; barrier 2 completes the unit's histogram, which fixes
//          the top digit d0 of the k-th largest key;
//  digits  each chunk writes its keys of bin d0 -- few -- as (key, position)
//          to its own region of the unit's candidate list and publishes its
//          count of keys above bin d0 (barrier 3); every CTA then gathers the
//          candidates and finds the two lower digits among them -- tau, the
//          k-th key, and take_eq, the keys equal to tau that are kept -- and
//          the lower chunks' counts of kept keys.  When bin d0 holds more
//          than kSelCandCap keys, two histogram rounds over all keys
//          (barriers 3 and 4) and a count exchange (barrier 5) do the same;
//  output  every kept position goes to slot (keys above tau before it) +
//          min(keys equal to tau before it, take_eq): the keys above tau,
//          then the lowest-positioned take_eq keys equal to it, ascending.
// With C == 1 a CTA holds its whole unit and waits for no other.  Each
// global histogram is zeroed, a slice per chunk, after the barrier that
// follows its last read.
template <int EV_G>
__global__ void __launch_bounds__(kSelT, 2) sel_kernel(const SelectArgs a) {
  extern __shared__ __align__(16) uint32_t sel_smem[];
  __shared__ uint32_t hist[kRadixBins];
  __shared__ uint32_t scan_sh[33];
  __shared__ unsigned long long scan64[33];
  __shared__ float shf[33];
  __shared__ uint32_t c_off[kSelMaxChunks + 1];  // candidate offsets of the chunks
  __shared__ uint32_t sh_digit, sh_above, sh_gb, sh_qb, sh_nc;
  __shared__ int sh_ok;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, c = blockIdx.x, C = gridDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kSelT / 32;
  const unsigned lt = (1u << lane) - 1u;
  SelUnit s;
  const int rs = sel_unit(a, blockIdx.y, c, C, s);
  if (rs != 0) {
    if (rs == 2 && c == 0 && tid == 0) set_status(a.status, SFI_DEV_LEN_OVER_CAP);
    return;  // uniform over the unit: no barrier of it is reached
  }
  const bool multi = C > 1;
  uint32_t* ctr = a.sel_ctr + size_t(s.u) * 4;
  uint32_t* gh = a.sel_hist + size_t(s.u) * kSelHistWords;
  uint32_t* cnt = a.sel_cnt + size_t(s.u) * kSelMaxChunks * 2;
  // shared memory: [keys | key norms, later the candidates] when the chunk
  // fits, else [candidates] with the keys in the workspace
  uint32_t* keys = a.keys_smem ? sel_smem : a.sel_keys + size_t(s.u) * a.max_len + s.p0;
  float* nu_s = a.keys_smem ? reinterpret_cast<float*>(sel_smem + a.smem_split) : nullptr;
  unsigned long long* cands = reinterpret_cast<unsigned long long*>(sel_smem + a.smem_split);
  bool ok = true;
  auto barrier = [&]() {
    const uint32_t old = unit_arrive(ctr, c, C);
    ok = unit_wait(ctr, old, ok, a.wait_cycles, a.status, &sh_ok);
  };
  // this chunk's slice of global histogram r back to zero (no CTA reads it
  // any more)
  auto zero_slice = [&](int r) {
    const int b0 = c * kRadixBins / C, b1 = (c + 1) * kRadixBins / C;
    for (int i = b0 + tid; i < b1; i += kSelT) gh[r * kRadixBins + i] = 0u;
  };
  if (s.need_radix)
    for (int i = tid; i < kRadixBins; i += kSelT) hist[i] = 0;
  __syncthreads();

  const int lo = s.lo, hi = s.hi;
  const float* kn = s.prior ? a.knorm + size_t(s.u) * a.max_len : nullptr;
  float* srow = a.s ? a.s + size_t(s.u) * a.max_len : nullptr;
  // exclusivity: the fused score is written to s as it is; the selection
  // ranks it times exp(-beta * picks of the earlier KV heads)
  const uint8_t* exrow = s.prior && a.excl ? a.excl + size_t(s.b) * a.max_len : nullptr;
  int32_t* out_idx = a.idx + size_t(s.per_seq ? s.b * a.H_kv : s.unit) * a.k;
  const int n_rows = s.per_seq ? a.H_kv : 1;  // idx rows that receive the set
  const float w_f = s.prior ? 1.0f - a.lambda : 1.0f;
  // score of position i from its evidence; key, s, histogram, and the whole
  // of E when it is all kept (position lo + t goes to slot t)
  auto emit = [&](int i, bool in, float ev, float kv, uint32_t cx, float coef) {
    const bool e = in && i >= lo && i < hi;
    if (!in) return;
    float v = w_f * ev;
    if (s.prior && e) v = fmaf(coef, kv, v);
    if (srow) srow[i] = v;
    v *= excl_factor(cx, a.excl_beta);
    const uint32_t key = order_key(v);
    keys[i - s.p0] = key;
    if (e) {
      if (s.need_radix) hist_add(hist, key >> kRadixShift0, true);
      else
        for (int g = 0; g < n_rows; ++g) out_idx[size_t(g) * a.k + (i - lo)] = i;
    }
  };

  // ---- pass 1
  float coef = 0.f;
  uint32_t bar1_old = 0;
  if (s.prior) {
    float part = 0.f;
    for (int base = s.e0; base < s.e1; base += kSelT * kSelU) {
      float x[kSelU];
#pragma unroll
      for (int j = 0; j < kSelU; ++j) {
        const int i = base + j * kSelT + tid;
        x[j] = i < s.e1 ? kn[i] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kSelU; ++j) {
        const int i = base + j * kSelT + tid;
        part += x[j];
        if (nu_s && i < s.e1) nu_s[i - s.p0] = x[j];
      }
    }
    const float t = sel_block_sum(part, shf);
    if (multi) {
      if (tid == 0) a.sel_nu[size_t(s.u) * kSelMaxChunks + c] = t;
      bar1_old = unit_arrive(ctr, c, C);  // barrier 1: waited for after the evidence loads
    } else {
      coef = t > 0.f ? a.lambda / t : 0.f;
    }
  }
  float M[EV_G > 0 ? EV_G : 1], iz[EV_G > 0 ? EV_G : 1];
  if constexpr (EV_G > 0) {
#pragma unroll
    for (int hh = 0; hh < EV_G; ++hh) {
      const size_t qh = size_t(s.b) * a.H_q + size_t(s.unit % a.H_kv) * EV_G + hh;
      M[hh] = a.stats[qh * 2];
      iz[hh] = 1.0f / a.stats[qh * 2 + 1];
    }
  }
  // U positions per thread at a time, every load issued before any is used
  // (fewer when each position brings G logits, so two CTAs fit an SM)
  constexpr int U = EV_G >= 8 ? 2 : (EV_G >= 4 ? 4 : kSelU);
  for (int base = s.p0; base < s.p1; base += kSelT * U) {
    float lg[U][EV_G > 0 ? EV_G : 1];
    float ev[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int i = base + j * kSelT + tid;
      ev[j] = 0.f;
      if (i < s.p1) {
        if constexpr (EV_G > 0) {
          load_row<EV_G>(a.logits + (size_t(s.u) * a.max_len + i) * EV_G, lg[j]);
        } else if (s.per_seq) {
          for (int g = 0; g < a.H_kv; ++g)
            ev[j] += a.evidence[(size_t(s.b) * a.H_kv + g) * a.max_len + i];
        } else {
          ev[j] = a.evidence[size_t(s.u) * a.max_len + i];
        }
      }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int i = base + j * kSelT + tid;
      const bool in = i < s.p1;
      if (in) {
        if constexpr (EV_G > 0) ev[j] = evidence_from_logits<EV_G>(lg[j], M, iz);
      }
      if (s.prior) {
        if (in) keys[i - s.p0] = __float_as_uint(ev[j]);  // the key once the prior is known
      } else {
        emit(i, in, ev[j], 0.f, 0u, 0.f);
      }
    }
  }

  // ---- pass 2 (fused mode): the prior needs the unit's key-norm sum
  if (s.prior) {
    if (multi) {
      ok = unit_wait(ctr, bar1_old, ok, a.wait_cycles, a.status, &sh_ok);
      // the chunks' sums in one fixed order: every CTA of the unit forms the
      // same value
      const float* pn = a.sel_nu + size_t(s.u) * kSelMaxChunks;
      float x = (lane < C ? __ldcg(pn + lane) : 0.f) + (lane + 32 < C ? __ldcg(pn + lane + 32) : 0.f);
#pragma unroll
      for (int o = 16; o; o >>= 1) x += __shfl_down_sync(kFull, x, o);
      x = __shfl_sync(kFull, x, 0);
      coef = x > 0.f ? a.lambda / x : 0.f;
    } else {
      __syncthreads();  // the key norms kept in shared memory
    }
    // (fewer positions at a time than the global passes: the norms come from
    // shared memory or L2, and a shorter loop body keeps the code small)
    constexpr int U2 = 4;
    for (int base = s.p0; base < s.p1; base += kSelT * U2) {
      float kv[U2];
      uint32_t cx[U2];
#pragma unroll
      for (int j = 0; j < U2; ++j) {
        const int i = base + j * kSelT + tid;
        const bool e = i < s.p1 && i >= lo && i < hi;
        kv[j] = e ? (nu_s ? nu_s[i - s.p0] : kn[i]) : 0.f;
        cx[j] = exrow && e ? exrow[i] : 0u;
      }
#pragma unroll
      for (int j = 0; j < U2; ++j) {
        const int i = base + j * kSelT + tid;
        const bool in = i < s.p1;
        emit(i, in, in ? __uint_as_float(keys[i - s.p0]) : 0.f, kv[j], cx[j], coef);
      }
    }
  }
  if (c == 0 && tid == 0) {
    if (s.per_seq) {
      for (int g = 0; g < a.H_kv; ++g) a.count[s.b * a.H_kv + g] = s.keff;
    } else {
      a.count[s.u] = s.keff;
    }
  }
  if (!s.need_radix) return;

  const int e0 = s.e0 - s.p0, e1 = s.e1 - s.p0;  // this chunk's part of E, in keys[]
  // ---- top digit
  if (multi) {
    __syncthreads();
    for (int i = tid; i < kRadixBins; i += kSelT)
      if (hist[i]) atomicAdd(gh + i, hist[i]);
    barrier();  // 2
    for (int i = tid; i < kRadixBins; i += kSelT) hist[i] = __ldcg(gh + i);
  }
  __syncthreads();
  block_pick_digit<kRadixBins>(hist, uint32_t(s.keff), &sh_digit, &sh_above, scan_sh);
  const uint32_t d0 = sh_digit;
  uint32_t krem = uint32_t(s.keff) - sh_above;
  const bool by_cands = multi && hist[d0] <= uint32_t(kSelCandCap);  // uniform over the unit
  uint32_t tau, take_eq;
  if (by_cands) {
    // ---- this chunk's keys of bin d0 to its region of the candidate list
    // (starting at its first position of E), and its count of keys above
    unsigned long long* row = a.sel_cand + size_t(blockIdx.y) * a.max_len;
    if (tid == 0) sh_nc = 0;
    __syncthreads();
    uint32_t above = 0;
    auto append_walk = [&](auto kw) {
      constexpr int KW = decltype(kw)::value;
      for (int b0 = e0; b0 < e1; b0 += kSelT * KW) {
        uint32_t kk[KW];
#pragma unroll
        for (int r = 0; r < KW; ++r) {
          const int i = b0 + kSelT * r + tid;
          kk[r] = i < e1 ? keys[i] : 0u;
        }
#pragma unroll
        for (int r = 0; r < KW; ++r) {
          const int i = b0 + kSelT * r + tid;
          const uint32_t dg = kk[r] >> kRadixShift0;
          above += (i < e1 && dg > d0) ? 1u : 0u;
          const unsigned m = __ballot_sync(kFull, i < e1 && dg == d0);
          // slots in the chunk's region in any order: only counts and
          // histograms are taken over the candidates
          uint32_t at = 0;
          if (lane == 0 && m) at = atomicAdd(&sh_nc, uint32_t(__popc(m)));
          at = __shfl_sync(kFull, at, 0) + __popc(m & lt);
          if ((m >> lane) & 1u)
            row[s.e0 + at] = (static_cast<unsigned long long>(kk[r]) << 32) | uint32_t(s.p0 + i);
        }
      }
    };
    if (a.keys_smem) append_walk(std::integral_constant<int, 1>{});
    else append_walk(std::integral_constant<int, kWalk>{});
    above = block_count(above, scan_sh);
    if (tid == 0) {
      cnt[2 * c] = above;
      cnt[2 * c + 1] = sh_nc;
    }
    barrier();  // 3
    zero_slice(0);
    // ---- every CTA: the chunks' counts, then the candidates in chunk order
    if (warp == 0) {
      const uint32_t n0 = lane < C ? __ldcg(cnt + 2 * lane + 1) : 0u;
      const uint32_t n1 = lane + 32 < C ? __ldcg(cnt + 2 * (lane + 32) + 1) : 0u;
      const uint32_t a0 = lane < c ? __ldcg(cnt + 2 * lane) : 0u;
      const uint32_t a1 = lane + 32 < c ? __ldcg(cnt + 2 * (lane + 32)) : 0u;
      uint32_t i0 = n0, i1 = n1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y0 = __shfl_up_sync(kFull, i0, o), y1 = __shfl_up_sync(kFull, i1, o);
        if (lane >= o) i0 += y0, i1 += y1;
      }
      const uint32_t t0 = __shfl_sync(kFull, i0, 31);
      c_off[lane] = i0 - n0;
      c_off[lane + 32] = t0 + i1 - n1;
      if (lane == 31) c_off[kSelMaxChunks] = t0 + i1;
      uint32_t g = a0 + a1;
#pragma unroll
      for (int o = 16; o; o >>= 1) g += __shfl_down_sync(kFull, g, o);
      if (lane == 0) sh_gb = g;  // keys above bin d0 in the lower chunks
    }
    for (int i = tid; i < kRadixBins; i += kSelT) hist[i] = 0;
    __syncthreads();
    const uint32_t nc = min(c_off[kSelMaxChunks], uint32_t(kSelCandCap));
    // every entry of every chunk copied straight into shared memory at once
    // (asynchronous 8-byte copies; each warp walks whole chunks); the bounds
    // hold the copy inside the staging area and the row even when a barrier
    // wait gave up and the counts are inconsistent
    for (int cc = warp; cc < C; cc += NW) {
      const int e0c = sel_chunk_e0(s, cc);
      const uint32_t o0 = min(c_off[cc], nc), o1 = max(o0, min(c_off[cc + 1], nc));
      const uint32_t n = min(o1 - o0, uint32_t(max(a.max_len - e0c, 0)));
      const unsigned long long* src = row + e0c;
      const uint32_t dst = smem_addr(cands + o0);
      for (uint32_t jj = lane; jj < n; jj += 32)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst + 8u * jj), "l"(src + jj)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    // ---- the two lower digits among the candidates
    for (uint32_t e = tid; e < nc; e += kSelT)
      hist_add(hist, (uint32_t(cands[e] >> 32) >> kRadixShift1) & (kRadixBins - 1), true);
    __syncthreads();
    block_pick_digit<kRadixBins>(hist, krem, &sh_digit, &sh_above, scan_sh);
    const uint32_t p1 = (d0 << (kRadixShift0 - kRadixShift1)) | sh_digit;  // top 22 bits
    krem -= sh_above;
    for (int i = tid; i < (1 << kRadixShift1); i += kSelT) hist[i] = 0;
    __syncthreads();
    for (uint32_t e = tid; e < nc; e += kSelT) {
      const uint32_t key = uint32_t(cands[e] >> 32);
      hist_add(hist, key & ((1u << kRadixShift1) - 1u), (key >> kRadixShift1) == p1);
    }
    __syncthreads();
    block_pick_digit<1 << kRadixShift1>(hist, krem, &sh_digit, &sh_above, scan_sh);
    tau = (p1 << kRadixShift1) | sh_digit;
    take_eq = krem - sh_above;
    // candidates of the lower chunks above / equal to tau (both counts are
    // below 2^16: one packed block sum)
    uint32_t gq = 0;
    const uint32_t nlow = min(c_off[c], nc);
    for (uint32_t e = tid; e < nlow; e += kSelT) {
      const uint32_t key = uint32_t(cands[e] >> 32);
      gq += key > tau ? 0x10000u : (key == tau ? 1u : 0u);
    }
    gq = block_count(gq, scan_sh);
    if (tid == 0) {
      sh_gb += gq >> 16;
      sh_qb = gq & 0xffffu;
    }
  } else {
    // ---- the two lower digits by histogram rounds over all keys: each
    // round histograms the next digit of the keys that share the prefix so
    // far, takes the unit's total and picks the digit holding the krem-th key
    uint32_t prefix = d0;
    for (int round = 1; round < 3; ++round) {
      const int width = round == 2 ? kRadixShift1 : kRadixShift0 - kRadixShift1;  // 11, 10
      const int shift = round == 1 ? kRadixShift1 : 0;
      const int hs = shift + width;
      __syncthreads();  // the last histogram has been read
      for (int i = tid; i < kRadixBins; i += kSelT) hist[i] = 0;
      __syncthreads();
      for (int b0 = e0; b0 < e1; b0 += kSelT * kSelU) {
        uint32_t kk[kSelU];
#pragma unroll
        for (int j = 0; j < kSelU; ++j) {
          const int i = b0 + j * kSelT + tid;
          kk[j] = i < e1 ? keys[i] : 0u;
        }
#pragma unroll
        for (int j = 0; j < kSelU; ++j) {
          const int i = b0 + j * kSelT + tid;
          hist_add(hist, (kk[j] >> shift) & ((1u << width) - 1u), i < e1 && (kk[j] >> hs) == prefix);
        }
      }
      if (multi) {
        __syncthreads();
        uint32_t* gr = gh + round * kRadixBins;
        for (int i = tid; i < (1 << width); i += kSelT)
          if (hist[i]) atomicAdd(gr + i, hist[i]);
        barrier();  // 3, 4
        zero_slice(round - 1);
        for (int i = tid; i < (1 << width); i += kSelT) hist[i] = __ldcg(gr + i);
      }
      __syncthreads();
      if (round == 1) block_pick_digit<kRadixBins>(hist, krem, &sh_digit, &sh_above, scan_sh);
      else block_pick_digit<1 << kRadixShift1>(hist, krem, &sh_digit, &sh_above, scan_sh);
      prefix = (prefix << width) | sh_digit;
      krem -= sh_above;
    }
    tau = prefix;
    take_eq = krem;
  }

  // ---- ordered output: each warp walks one contiguous segment of the
  // chunk's part of E (lane l at base + l); a counting walk, one block scan
  // and the lower chunks' totals give every warp its first slot
  const int len = max(e1 - e0, 0);
  const int seg = ((len + NW - 1) / NW + 31) / 32 * 32;
  const int s0 = min(e1, e0 + warp * seg), s1 = min(e1, s0 + seg);
  uint32_t wg = 0, wq = 0;
  // (in the walks, KW keys per lane are loaded before any is used: 8 when
  // the keys are in global memory, 1 from shared memory)
  auto count_walk = [&](auto kw) {
    constexpr int KW = decltype(kw)::value;
    for (int base = s0; base < s1; base += 32 * KW) {
      uint32_t kk[KW];
#pragma unroll
      for (int r = 0; r < KW; ++r) {
        const int i = base + 32 * r + lane;
        kk[r] = i < s1 ? keys[i] : 0u;
      }
#pragma unroll
      for (int r = 0; r < KW; ++r) {
        const bool in = base + 32 * r + lane < s1;
        wg += __popc(__ballot_sync(kFull, in && kk[r] > tau));
        wq += __popc(__ballot_sync(kFull, in && kk[r] == tau));
      }
    }
  };
  if (a.keys_smem) count_walk(std::integral_constant<int, 1>{});
  else count_walk(std::integral_constant<int, kWalk>{});
  unsigned long long tot;
  const unsigned long long ex = block_excl_scan<unsigned long long>(
      lane == 0 ? (static_cast<unsigned long long>(wg) << 32) | wq : 0ull, scan64, tot);
  const unsigned long long w_ex = __shfl_sync(kFull, ex, 0);
  if (multi && !by_cands) {
    if (tid == 0) {
      cnt[2 * c] = uint32_t(tot >> 32);
      cnt[2 * c + 1] = uint32_t(tot);
    }
    barrier();  // 5
    zero_slice(2);
    if (warp == 0) {  // totals of the lower chunks
      uint32_t g = 0, q = 0;
      for (int cc = lane; cc < c; cc += 32) {
        g += __ldcg(cnt + 2 * cc);
        q += __ldcg(cnt + 2 * cc + 1);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        g += __shfl_down_sync(kFull, g, o);
        q += __shfl_down_sync(kFull, q, o);
      }
      if (lane == 0) {
        sh_gb = g;
        sh_qb = q;
      }
    }
  } else if (!multi && tid == 0) {
    sh_gb = 0;
    sh_qb = 0;
  }
  __syncthreads();
  uint32_t gb = sh_gb + uint32_t(w_ex >> 32), qb = sh_qb + uint32_t(w_ex);
  auto out_walk = [&](auto kw) {
    constexpr int KW = decltype(kw)::value;
    for (int base = s0; base < s1; base += 32 * KW) {
      uint32_t kk[KW];
#pragma unroll
      for (int r = 0; r < KW; ++r) {
        const int i = base + 32 * r + lane;
        kk[r] = i < s1 ? keys[i] : 0u;
      }
#pragma unroll
      for (int r = 0; r < KW; ++r) {
        const int i = base + 32 * r + lane;
        const unsigned bg = __ballot_sync(kFull, i < s1 && kk[r] > tau);
        const unsigned bq = __ballot_sync(kFull, i < s1 && kk[r] == tau);
        const uint32_t g_at = gb + __popc(bg & lt), q_at = qb + __popc(bq & lt);
        const int pos = s.p0 + i;
        // slots stay below keff for consistent counts; the bound only guards
        // the output row against inconsistent counts (a wait that gave up)
        if ((bg >> lane) & 1u) {
          const uint32_t slot = g_at + min(q_at, take_eq);
          if (slot < uint32_t(s.keff))
            for (int g = 0; g < n_rows; ++g) out_idx[size_t(g) * a.k + slot] = pos;
        } else if (((bq >> lane) & 1u) && q_at < take_eq && g_at + q_at < uint32_t(s.keff)) {
          for (int g = 0; g < n_rows; ++g) out_idx[size_t(g) * a.k + g_at + q_at] = pos;
        }
        gb += __popc(bg);
        qb += __popc(bq);
      }
    }
  };
  if (a.keys_smem) out_walk(std::integral_constant<int, 1>{});
  else out_walk(std::integral_constant<int, kWalk>{});
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

template <typename K>
cudaError_t launch_dependent(K kernel, dim3 grid, int threads, cudaStream_t st,
                             const SelectArgs& a, size_t smem) {
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

// Selector CTAs resident per SM with the largest key buffer (per device).
template <int EV_G>
int sel_blocks_per_sm() {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int n = cached[dev].load();
  if (n == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sel_kernel<EV_G>, kSelT, kSelSmemMax) !=
            cudaSuccess || n < 1)
      n = 1;
    cached[dev].store(n);
  }
  return n;
}

// Chunks per unit: as many as keep every CTA of the launch resident at once
// (the chunks of a unit wait for one another), chunks of at least
// kSelMinChunk positions, at most kSelMaxChunks; one chunk per unit when the
// units alone fill the GPU.  Shared memory: the chunk's keys and key norms
// (the norms' space then holds the unit's candidates) when they fit, else
// the candidates alone.
template <int EV_G>
cudaError_t launch_select_t(const SelectArgs& a0, cudaStream_t st) {
  int n_active = 0;
  for (int b = 0; b < a0.B; ++b) n_active += int((a0.active.bits[b >> 5] >> (b & 31)) & 1u);
  const bool one_unit =
      a0.mode == SFI_SELECT_LOGIT_SUM_SEQ || (a0.mode == SFI_SELECT_FUSED && a0.g_only >= 0);
  const int units = n_active * (one_unit ? 1 : a0.H_kv);
  if (units == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(sel_kernel<EV_G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSelSmemMax);
  if (e != cudaSuccess) return e;
  const int resident = sel_blocks_per_sm<EV_G>() * device_sm_count();
  int C = units <= kSelCandRows ? min(kSelMaxChunks, resident / units) : 1;
  C = min(C, (a0.max_len + kSelMinChunk - 1) / kSelMinChunk);
  C = max(C, 1);
  const int ch = ((a0.max_len + C - 1) / C + 3) & ~3;
  const size_t key_b = size_t(ch) * sizeof(uint32_t);
  const size_t cand_b = C > 1 ? size_t(kSelCandCap) * sizeof(unsigned long long) : 0;
  const size_t both = key_b + std::max(key_b, cand_b);
  SelectArgs a = a0;
  a.keys_smem = both <= size_t(kSelSmemMax) ? 1 : 0;
  a.smem_split = a.keys_smem ? ch : 0;
  a.wait_cycles = wait_limit_cycles();
  return launch_dependent(sel_kernel<EV_G>, dim3(C, units), kSelT, st, a, a.keys_smem ? both : cand_b);
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
