// Split-K decode attention over the KV cache for slow and fast steps.
//
// SFI (gist.science 2603.12038, "Slow-Fast paradigm"): a slow step attends
// densely to the whole history and its logits become the evidence; a fast
// step attends only to the managed sparse state (sink tokens, the selected
// memory, the recent window).  Both are the same computation over a list of
// cache rows per (sequence, KV head) unit -- the list is [0, n) for a slow
// unit and [sinks | selected | window] for a fast one -- so one persistent
// kernel serves a mixed batch.
//
// Design (GB300; the step is HBM-bound: G = H_q / H_kv query heads per KV
// head read every K and V row once):
//  * each unit's 64-row stages are dealt cyclically to a few work items
//    (separate item sizes for slow and fast units); the persistent CTAs (one
//    per SM) take items from a global counter, slow units' items first;
//  * four producer warps stream K and V rows into a ring of up to 6 shared-
//    memory stages with completion on mbarriers: full dense bf16 stages as
//    64 x 64 2-D TMA boxes (128-byte swizzle), gathered rows and partial
//    stages as 16-byte cp.async pieces into the same swizzled layout, fp32
//    dense stages as one bulk copy (cp.async.bulk) per operand;
//  * bf16 caches: eight consumer warps, four per stage, 16 rows each.  The
//    G query vectors sit in registers as the A operand of mma.sync m16n8k16
//    (rows G..15 zero); S = Q K^T comes from ldmatrix'ed K rows (the stages
//    are stored with a 16-byte-chunk XOR swizzle so ldmatrix is conflict-
//    free), the online softmax runs on the accumulator fragments (one head
//    per lane quad, log2 domain), and P is fed back as the A operand of
//    O += P V with ldmatrix.trans'ed V rows (fp32 accumulation throughout;
//    P is rounded to bf16 for the product).  ncu showed the CUDA-core
//    version spending ~79 warp instructions per 256-byte row, which capped
//    it at ~60% of HBM bandwidth; the tensor-core path needs ~6;
//  * fp32 caches (kept exact to 2e-5): eight consumer warps share every
//    stage on CUDA cores, 16-byte row slices per lane, per-row dots finished
//    with a transpose-reduce across the lanes of a row;
//  * slow units also write their logits ([pos][G], log2-scaled) and the key
//    norms, which the evidence pass and the selector read back;
//  * the consumer warps merge their states per item; a unit cut into several
//    items writes per-item partials and the last CTA to finish a unit (an
//    atomic counter per unit, reset after use) merges them into the output.
#pragma once

#include <math.h>

#include <type_traits>

#include "common.cuh"

namespace sfi {

// Dynamic work distribution.  A CTA's first producer warp takes item ids
// from a global counter (a.work_ctr[0]) as it starts each item and publishes
// them through a small ring in shared memory (slot mbarriers: `full` with one
// arrival, `empty` with one arrival from each of the other producer warps and
// from consumer warp 0).  CTAs that start late -- for example on SMs that a
// concurrently running kernel held -- simply take fewer items.  The last CTA
// to finish fetching resets the counters for the next launch.
constexpr int kItemRing = 4;
// words of the sequence-rank table that follows the unit table in shared memory
constexpr int kRankWords = kMaxBatch / 32 + 1;
// misc[] words of the CTA's shared scratch
constexpr int kMiscAbort = 14, kMiscLast = 15, kMiscRing = 16, kMiscCurItem = 24;

template <typename T, int D, int G>
struct AttnCfg {
  static constexpr bool MMA = std::is_same<T, bf16_t>::value;
  static constexpr int DIM = D;
  static constexpr int ES = sizeof(T);
  static constexpr int ROWB = D * ES;       // bytes per cache row
  static constexpr int LPR = ROWB / 16;     // 16-byte chunks (lanes) per row
  static constexpr int EPL = 16 / ES;       // elements per chunk
  static constexpr int RPI = 32 / LPR;      // rows per warp-wide 16-byte access
  static constexpr int R = 4;               // SIMT: rows per lane group per stage
  static constexpr int RB = RPI * R;        // SIMT: rows per warp per stage
  static constexpr int NCW = 8;             // consumer warps
  static constexpr int MW = 16;             // MMA: rows per consumer warp per stage
  static constexpr int CPS = MMA ? 4 : NCW;  // consumer warps per stage
  static constexpr int SR = MMA ? MW * CPS : RB * NCW;  // rows per stage
  // pipeline depth: as many stages as shared memory allows (bytes in flight
  // per SM are what keeps HBM busy), at most 6
  static constexpr size_t FIXED_B = (2 * 6 + 2 * kItemRing) * 8 +                   // mbarriers
                                    (MMA ? 0 : size_t(NCW) * RB * (G + 1) * 4) +  // SIMT scratch
                                    size_t(NCW) * G * (D + 2) * 4 + 128 +          // reduce + misc
                                    (size_t(kMaxUnits) + 1 + kRankWords) * 4;      // unit table
  static constexpr int NS_FIT = int((227 * 1024 - FIXED_B) / (2 * size_t(SR) * ROWB));
  static constexpr int NS = NS_FIT > 6 ? 6 : (NS_FIT < 2 ? 2 : NS_FIT);
  static constexpr int PW = 4;              // producer warps (each copies SR / PW rows)
  static_assert(SR % (PW * RPI) == 0, "stage rows split evenly over the producer warps");
  static constexpr int NT = (NCW + 4) * 32;  // consumers + producer warps
  static constexpr int STAGE_B = SR * ROWB;  // bytes of K (or V) per stage
  static constexpr int NE = (RB * G + 31) / 32;
  static constexpr int V = G * R;
  static constexpr int NV = V >= LPR ? V / LPR : 1;
  static_assert(LPR >= 8 && LPR <= 32, "row must be 128..512 bytes");
  static_assert(R < LPR, "norm reduction assumes one value per lane");
  static_assert(!MMA || G <= 8, "MMA path keeps the heads in rows 0..7 of the tile");
  static constexpr size_t OFF_K = 0;
  static constexpr size_t OFF_V = OFF_K + size_t(NS) * STAGE_B;
  static constexpr size_t OFF_BAR = OFF_V + size_t(NS) * STAGE_B;
  static constexpr size_t OFF_SL = OFF_BAR + (2 * NS + 2 * kItemRing) * 8;  // SIMT scratch
  static constexpr size_t OFF_SN = OFF_SL + (MMA ? 0 : size_t(NCW) * RB * G * 4);
  static constexpr size_t OFF_RED = OFF_SN + (MMA ? 0 : size_t(NCW) * RB * 4);
  static constexpr size_t OFF_MISC = OFF_RED + size_t(NCW) * G * (D + 2) * 4;
  static constexpr size_t OFF_UNITS = OFF_MISC + 128;
  static size_t smem_bytes(int n_units) { return OFF_UNITS + size_t(n_units + 1 + kRankWords) * 4; }
  static constexpr bool OFF_UNITS_MAX_CHECK() {
    return OFF_UNITS + (size_t(kMaxUnits) + 1 + kRankWords) * 4 <= size_t(227) * 1024;
  }
  static_assert(OFF_UNITS_MAX_CHECK(), "shared memory plan exceeds 227 KB");
  // Byte offset of 16-byte chunk c of stage row r.  Tensor-core path: the
  // stage is stored as 64-element column halves [c / 8][row][128 bytes] with
  // the 128-byte swizzle (chunk c % 8 stored at (c % 8) ^ (row % 8)), the
  // layout a 64 x 64 TMA box with CU_TENSOR_MAP_SWIZZLE_128B produces; rows
  // copied with cp.async use the same addresses.  SIMT path: plain rows.
  static __device__ __forceinline__ uint32_t chunk_off(int r, int c) {
    if constexpr (MMA)
      return uint32_t((c >> 3) * (SR * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    else
      return uint32_t(r * ROWB + (c << 4));
  }
};

struct ItemRing {
  uint32_t full, empty;  // mbarrier addresses of slot 0
  volatile int* slot;    // kItemRing item ids
};

// Fetch the next item id for this CTA and publish it (first producer warp).
// A CTA's first item is its own index (no round trip before its first rows
// are requested); later ones come from the work counter, past the grid.
__device__ __forceinline__ int ring_fetch_publish(const AttnArgs& a, int total, const ItemRing& r,
                                                  uint32_t seq, volatile int* abort_flag,
                                                  int lane, unsigned first_id) {
  int it = -1;
  bool fetched_end = false;
  // after an abort the CTA takes no further items (the work counters are
  // then left mid-count: the caller zero-fills the workspace again)
  if (lane == 0 && !(seq > 0 && *abort_flag)) {
    const unsigned x = seq == 0 ? first_id : gridDim.x + atomicAdd(a.work_ctr, 1u);
    if (x < unsigned(total)) {
      it = int(x);
    } else {
      fetched_end = true;
    }
  }
  it = __shfl_sync(kFull, it, 0);
  // no more items for this CTA: the next launch on the stream may start
  // (programmatic dependent launch; it waits for this grid before it reads)
  if (it < 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (lane == 0 && fetched_end) {
    // every CTA fetches past the end exactly once; the last one resets
    if (atomicAdd(a.work_ctr + 1, 1u) == gridDim.x - 1) {
      atomicExch(a.work_ctr, 0u);
      atomicExch(a.work_ctr + 1, 0u);
    }
  }
  const int slot = seq % kItemRing;
  const uint32_t ph = (seq / kItemRing) & 1u;
  if (!warp_ctrl_wait(r.empty + 8 * slot, ph ^ 1u, abort_flag, a.status)) it = -1;
  if (lane == 0) {
    r.slot[slot] = it;
    mbar_arrive(r.full + 8 * slot);
  }
  return it;
}

// Read the next published item id (other producer warps, consumer warp 0).
__device__ __forceinline__ int ring_read(const AttnArgs& a, const ItemRing& r, uint32_t seq,
                                         volatile int* abort_flag, int lane) {
  const int slot = seq % kItemRing;
  const uint32_t ph = (seq / kItemRing) & 1u;
  int it = -1;
  if (warp_ctrl_wait(r.full + 8 * slot, ph, abort_flag, a.status)) it = r.slot[slot];
  __syncwarp();
  if (lane == 0) mbar_arrive(r.empty + 8 * slot);
  return it;
}

// Work item: item i of the n_items items of unit u takes the unit's stages
// i, i + n_items, i + 2 n_items, ... (n_st of them; stage s covers rows
// [s * SR, min((s + 1) * SR, rows))).  The items of a unit thus have equal
// shares (within one stage) and the CTAs that share a unit read
// neighbouring addresses.
struct ItemInfo {
  int u, b, g, n, first, n_items;
  int rows, c_first, c_step, n_st;
  bool slow;
};

// Rows of unit u in this launch (0 for an invalid length).
__device__ __forceinline__ int attn_unit_rows(const AttnArgs& a, int u, bool report) {
  const int b = u / a.H_kv;
  // all three loads go out before any of them is used
  const int n = a.len[b];
  const int cap = a.kv_cap[b];
  const int craw = a.count != nullptr ? a.count[u] : 0;
  if (n < 1 || n > cap || n > a.max_len) {
    if (report) set_status(a.status, SFI_DEV_LEN_OVER_CAP);
    return 0;
  }
  if (seq_is_slow(a.slow, b)) return n;
  const int ns = min(a.n_sink, n);
  const int cnt = min(max(craw, 0), a.idx_stride);
  const int wlo = max(a.n_sink, n - a.window);
  return ns + cnt + max(n - wlo, 0);
}

// Items are numbered largest first: the units of slow sequences (whole
// histories) come before those of fast ones (managed state only), each group
// in sequence order, so the small fast items are the last ones taken and fill
// the end of the launch.  The unit table lives in shared memory as
// [n_units + 1] first-item offsets (in that order) followed by kRankWords
// counts: rank[w] = slow sequences in mask words below w.
__device__ __forceinline__ int nth_set_bit(uint32_t m, int k) {
  for (int i = 0; i < k; ++i) m &= m - 1;
  return __ffs(m) - 1;
}

// Sequence of rank j: the j-th slow sequence if j < n_slow, else the
// (j - n_slow)-th fast one (both in increasing order).
__device__ __forceinline__ int seq_of_rank(const AttnArgs& a, const int* rank, int j) {
  const int nw = (a.B + 31) >> 5;
  const int n_slow = rank[nw];
  int w = 0;
  if (j < n_slow) {
    while (rank[w + 1] <= j) ++w;
    return 32 * w + nth_set_bit(a.slow.bits[w], j - rank[w]);
  }
  const int jf = j - n_slow;  // < B - n_slow, so the scan stops below nw
  while (32 * (w + 1) - rank[w + 1] <= jf) ++w;
  return 32 * w + nth_set_bit(~a.slow.bits[w], jf - (32 * w - rank[w]));
}

// Unit (b * H_kv + g) at position v of the item order.
__device__ __forceinline__ int unit_at(const AttnArgs& a, const int* rank, int v) {
  return seq_of_rank(a, rank, v / a.H_kv) * a.H_kv + v % a.H_kv;
}

// Returns false (in every thread) when some unit needs more than
// kItemSlotsPerUnit items: the merge of a split unit holds that many partial
// results, so such a launch must not run.
template <int NT>
__device__ bool attn_build_units(const AttnArgs& a, int* units, int n_units, int* scratch) {
  // units[v] = first item of the unit at position v, units[n_units] = total items.
  const int t = threadIdx.x;
  int* rank = units + n_units + 1;
  if (t == 0) {
    const int nw = (a.B + 31) >> 5;
    int c = 0;
    for (int w = 0; w < nw; ++w) {
      rank[w] = c;
      c += __popc(a.slow.bits[w]);
    }
    rank[nw] = c;
  }
  __syncthreads();
  const int per = (n_units + NT - 1) / NT;
  const int u0 = min(t * per, n_units), u1 = min(u0 + per, n_units);
  int local = 0;
  int over = 0;
  for (int u = u0; u < u1; ++u) {
    const int uu = unit_at(a, rank, u);
    const int rows = attn_unit_rows(a, uu, blockIdx.x == 0);
    const int rpi = seq_is_slow(a.slow, uu / a.H_kv) ? a.rpi_slow : a.rpi_fast;
    const int it = (rows + rpi - 1) / rpi;
    over |= it > kItemSlotsPerUnit;
    units[u] = it;
    local += it;
  }
  // block exclusive scan of `local`
  const int lane = t & 31, w = t >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scratch[w] = incl;
  over = __syncthreads_or(over);
  if (t == 0) {
    int s = 0;
    for (int i = 0; i < NT / 32; ++i) {
      const int x = scratch[i];
      scratch[i] = s;
      s += x;
    }
    scratch[NT / 32] = s;
  }
  __syncthreads();
  int run = scratch[w] + incl - local;
  for (int u = u0; u < u1; ++u) {
    const int it = units[u];
    units[u] = run;
    run += it;
  }
  if (t == 0) units[n_units] = scratch[NT / 32];
  __syncthreads();
  return over == 0;
}

// report: flag an invalid length (launches without a unit table report it
// from the producer of each unit's first item).
__device__ __forceinline__ ItemInfo attn_resolve(const AttnArgs& a, const int* units, int n_units,
                                                 int it, int sr, bool report = false) {
  ItemInfo I;
  if (a.fast_items > 0) {
    // every unit is fast and has exactly fast_items items: item it belongs to
    // unit it / fast_items (the fast units of a launch without slow ones are
    // in unit order)
    I.u = it / a.fast_items;
    I.first = I.u * a.fast_items;
    I.n_items = a.fast_items;
  } else {
    // largest u with units[u] <= it
    int lo = 0, hi = n_units - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (units[mid] <= it) lo = mid;
      else hi = mid - 1;
    }
    I.u = unit_at(a, units + n_units + 1, lo);
    I.first = units[lo];
    I.n_items = units[lo + 1] - units[lo];
  }
  I.b = I.u / a.H_kv;
  I.g = I.u % a.H_kv;
  I.rows = attn_unit_rows(a, I.u, report && it == I.first);
  const int i = it - I.first, k = I.n_items;
  const int n_stages = (I.rows + sr - 1) / sr;
  I.c_first = i * sr;
  I.c_step = k * sr;
  I.n_st = (n_stages - i + k - 1) / k;
  I.n = a.len[I.b];
  I.slow = seq_is_slow(a.slow, I.b);
  return I;
}

// Producer warp: takes this CTA's items as they are fetched (warp 0 fetches
// and publishes the ids) and fills the stage ring with its share of every
// stage's rows.  Full dense bf16 stages arrive as 2-D TMA boxes; gathered
// rows and partial stages as 16-byte cp.async chunks (XOR-swizzled on the
// tensor-core path), each lane arriving on the stage's mbarrier when its
// copies land; fp32 dense stages use one bulk copy per operand.
template <class C>
__device__ __forceinline__ void attn_produce(const AttnArgs& a, const int* units, int n_units,
                                             int total, unsigned char* smem, uint32_t bar_full,
                                             uint32_t bar_empty, const ItemRing& ring,
                                             volatile int* abort_flag, int pw, int lane,
                                             unsigned first_id) {
  constexpr int D = C::DIM;
  constexpr int RPW = C::SR / C::PW;        // rows of a stage per producer warp
  constexpr int PJ = (RPW + 31) / 32;       // positions per lane
  const int rbase = pw * RPW;               // this warp's first row of every stage
  // the swizzle pattern assumes 1024-byte aligned stage buffers
  const bool tma_ok = (smem_addr(smem) & 1023u) == 0;
  const uint64_t pol = l2_evict_first_policy();
  const uint32_t kbase = smem_addr(smem + C::OFF_K), vbase = smem_addr(smem + C::OFF_V);
  uint32_t stage = 0;
  bool ok = true;
  for (uint32_t iseq = 0; ok; ++iseq) {
    const int it = pw == 0 ? ring_fetch_publish(a, total, ring, iseq, abort_flag, lane, first_id)
                           : ring_read(a, ring, iseq, abort_flag, lane);
    if (it < 0) break;
    // Without a unit table the item's unit is known from its id, so the
    // index entries of its first stage (item i starts at stage i) and the
    // sequence's cache offset are loaded together with the unit's length and
    // count: one round trip to global memory instead of three before the
    // first rows are requested.  An entry is used only if the row turns out
    // to be a selected one (sinks = n_sink, which holds unless n < n_sink).
    int spec[PJ];
    long long kvo_spec = 0;
    const bool spec_ok = a.fast_items > 0;
    if (spec_ok) {
      const int su = it / a.fast_items, si = it - su * a.fast_items;
      const int32_t* ixs = a.idx + size_t(su) * a.idx_stride;
      kvo_spec = a.kv_offset[su / a.H_kv];
#pragma unroll
      for (int j = 0; j < PJ; ++j) {
        const int e = si * C::SR + rbase + lane + 32 * j - a.n_sink;
        spec[j] = (lane + 32 * j < RPW && e >= 0 && e < a.idx_stride) ? __ldg(ixs + e) : 0;
      }
    }
    const ItemInfo I = attn_resolve(a, units, n_units, it, C::SR, spec_ok && pw == 0);
    const long long kvo = spec_ok ? kvo_spec : (long long)a.kv_offset[I.b];
    const size_t head0 = size_t(kvo) + size_t(I.g) * size_t(a.kv_cap[I.b]) * D;
    const char* kb = reinterpret_cast<const char*>(a.k) + head0 * C::ES;
    const char* vb = reinterpret_cast<const char*>(a.v) + head0 * C::ES;
    const int n = I.n;
    const int ns = min(a.n_sink, n);
    const int cnt = I.slow ? 0 : min(max(a.count[I.u], 0), a.idx_stride);
    const int wlo = max(a.n_sink, n - a.window);
    const int32_t* ix = I.slow ? nullptr : a.idx + size_t(I.u) * a.idx_stride;
    // TMA rows of this unit: K viewed as [rows][D]; usable when the slab
    // starts on a whole row and its rows fit the descriptor
    long long row0 = 0;
    bool tma_unit = false;
    if constexpr (C::MMA) {
      const long long off = kvo;
      row0 = off / D + (long long)I.g * a.kv_cap[I.b];
      tma_unit = a.use_tma && tma_ok && I.slow && off % D == 0 && row0 + I.rows < (1LL << 31);
    }
    // Row positions of stage c0 (lane l: rows l, l + 32, ...).  Gathered
    // positions come from the index list in global memory, so the loads
    // for the next stage are issued one stage ahead of their use.
    auto resolve_pos = [&](int c0s, int (&out)[PJ], bool use_spec) {
      const int nrs = min(C::SR, I.rows - c0s);
#pragma unroll
      for (int j = 0; j < PJ; ++j) {
        const int r = rbase + lane + 32 * j;
        const int lp = c0s + r;
        int p = I.slow ? lp : 0;  // rows past the stage are never copied
        if (!I.slow && r < nrs && lane + 32 * j < RPW) {
          if (lp < ns) {
            p = lp;
          } else if (lp < ns + cnt) {
            p = use_spec ? spec[j] : __ldg(ix + (lp - ns));
          } else {
            p = wlo + (lp - ns - cnt);
          }
        }
        out[j] = p;
      }
    };
    int pos_next[PJ];
    // the speculative entries hold ix[lp - n_sink] for the first stage's rows
    resolve_pos(I.c_first, pos_next, spec_ok && ns == a.n_sink);
    for (int si = 0; si < I.n_st; ++si) {
      const int c0 = I.c_first + si * I.c_step;
      const int nr = min(C::SR, I.rows - c0);
      const int slot = stage % C::NS;
      const uint32_t ph = (stage / C::NS) & 1u;
      int pos[PJ];
#pragma unroll
      for (int j = 0; j < PJ; ++j) {
        int p = pos_next[j];
        if (!I.slow && (p < 0 || p >= n)) {
          set_status(a.status, SFI_DEV_BAD_INDEX);
          p = 0;
        }
        pos[j] = p;
      }
      if (si + 1 < I.n_st) resolve_pos(c0 + I.c_step, pos_next, false);
      if (!warp_ctrl_wait(bar_empty + 8 * slot, ph ^ 1u, abort_flag, a.status)) {
        ok = false;
        break;
      }
      const uint32_t kd = kbase + slot * C::STAGE_B, vd = vbase + slot * C::STAGE_B;
      if (tma_unit && nr == C::SR) {
        // full dense stage: 64-row TMA boxes, one per 64-column half
        if (pw == 0 && lane == 0) {
          mbar_arrive_expect_tx(bar_full + 8 * slot, uint32_t(C::SR) * C::ROWB * 2u);
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            tma_load_2d(kd + h * (C::SR * 128), &a.tmk, h * 64, int(row0 + c0), bar_full + 8 * slot, pol);
            tma_load_2d(vd + h * (C::SR * 128), &a.tmv, h * 64, int(row0 + c0), bar_full + 8 * slot, pol);
          }
        } else {
          mbar_arrive(bar_full + 8 * slot);
        }
      } else if (!C::MMA && I.slow) {
        // dense rows: one bulk copy of K and one of V for the whole stage
        if (pw == 0 && lane == 0) {
          mbar_arrive_expect_tx(bar_full + 8 * slot, uint32_t(nr) * C::ROWB * 2u);
          bulk_g2s(kd, kb + size_t(c0) * C::ROWB, uint32_t(nr) * C::ROWB, bar_full + 8 * slot, pol);
          bulk_g2s(vd, vb + size_t(c0) * C::ROWB, uint32_t(nr) * C::ROWB, bar_full + 8 * slot, pol);
        } else {
          mbar_arrive(bar_full + 8 * slot);
        }
      } else {
        // row by row: every lane copies one 16-byte chunk of a row; the
        // row positions were resolved before the wait (pos[]), lane l
        // holding this warp's rows l, l + 32, ...
#pragma unroll
        for (int i = 0; i < RPW / C::RPI; ++i) {
          const int rl = i * C::RPI + lane / C::LPR;
          const int r = rbase + rl;
          const int c = lane % C::LPR;
          const int p = __shfl_sync(kFull, pos[(i * C::RPI) / 32], rl & 31);
          if (r < nr) {
            const size_t so = size_t(p) * C::ROWB + c * 16;
            cp_async16(kd + C::chunk_off(r, c), kb + so, pol);
            cp_async16(vd + C::chunk_off(r, c), vb + so, pol);
          }
        }
        cp_async_arrive_noinc(bar_full + 8 * slot);
      }
      ++stage;
    }
  }
  // Let every copy that was issued land before the CTA can exit.
  const uint32_t first = stage > uint32_t(C::NS) ? stage - C::NS : 0u;
  for (uint32_t s = first; s < stage; ++s) mbar_wait(bar_full + 8 * (s % C::NS), (s / C::NS) & 1u);
}

// Consumer warp, CUDA-core path: process this CTA's stages of one item and
// leave the warp's (max, sum, p.v) state in red.
template <typename T, int D, int G>
__device__ __forceinline__ void attn_item_simt(const AttnArgs& a, const ItemInfo& I,
                                               unsigned char* smem, uint32_t bar_full,
                                               uint32_t bar_empty, volatile int* abort_flag,
                                               uint32_t& stage, int warp, int lane, float* red) {
  using C = AttnCfg<T, D, G>;
  const int li = lane % C::LPR, lg = lane / C::LPR;
  const int hl = lane % G;  // head of this lane's softmax entries
  float* sl = reinterpret_cast<float*>(smem + C::OFF_SL) + warp * C::RB * G;
  float* sn = reinterpret_cast<float*>(smem + C::OFF_SN) + warp * C::RB;
  const uint32_t kbase = smem_addr(smem + C::OFF_K), vbase = smem_addr(smem + C::OFF_V);
  const bool emit = a.emit && I.slow;
  const bool emit_norm = emit && a.knorm != nullptr;
  // key norms of rows below nv are already stored (they never change)
  const int nv = emit_norm && a.knorm_valid ? a.knorm_valid[I.u] : 0;
    float qf[G][C::EPL];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const char* qp = reinterpret_cast<const char*>(a.q) +
                       (size_t(I.b) * a.H_q + size_t(I.g) * G + hh) * C::ROWB + li * 16;
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qp));
      float t[C::EPL];
      Unpack<T>::run(raw, t);
#pragma unroll
      for (int e = 0; e < C::EPL; ++e) qf[hh][e] = t[e] * a.qscale;
    }
    float m[G], acc[G][C::EPL];
    float zl = 0.f;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      m[hh] = -INFINITY;
#pragma unroll
      for (int e = 0; e < C::EPL; ++e) acc[hh][e] = 0.f;
    }

    for (int si = 0; si < I.n_st; ++si) {
      const int c0 = I.c_first + si * I.c_step;
      const int nr = min(C::SR, I.rows - c0);
      const int slot = stage % C::NS;
      const uint32_t ph = (stage / C::NS) & 1u;
      // On a failed wait the warp skips the stage but keeps walking the
      // schedule, so every consumer warp reaches every named barrier.
      const bool have = warp_pipe_wait(bar_full + 8 * slot, ph, abort_flag, a.status, a.wait_cycles);
      const int wr0 = warp * C::RB;
      const bool norm_stage = emit_norm && c0 + nr > nv;
      if (have && wr0 < nr) {
        const int nw = min(C::RB, nr - wr0);
        const uint32_t krow = kbase + slot * C::STAGE_B + (wr0 + lg * C::R) * C::ROWB + li * 16;
        float x[C::V];
        float nn[C::R];
#pragma unroll
        for (int r = 0; r < C::R; ++r) {
          const bool valid = lg * C::R + r < nw;
          uint4 raw = make_uint4(0u, 0u, 0u, 0u);
          if (valid) raw = lds128(krow + r * C::ROWB);
          float kf[C::EPL];
          Unpack<T>::run(raw, kf);
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < C::EPL; ++e) s = fmaf(qf[hh][e], kf[e], s);
            x[hh * C::R + r] = s;
          }
          float s2 = 0.f;
#pragma unroll
          for (int e = 0; e < C::EPL; ++e) s2 = fmaf(kf[e], kf[e], s2);
          nn[r] = s2;
        }
        const int jb = transpose_reduce<C::LPR>(x, li);
#pragma unroll
        for (int i = 0; i < C::NV; ++i) {
          const int j = jb + i;
          const int hh = j / C::R, row = lg * C::R + (j % C::R);
          sl[row * G + hh] = row < nw ? x[i] : -INFINITY;
        }
        if (norm_stage) {
          const int jn = transpose_reduce<C::LPR>(nn, li);
          const int row = lg * C::R + jn;
          if (row < nw) sn[row] = sqrtf(nn[0]);
        }
        __syncwarp();
        // ---- online softmax over this warp's rows
        float lv[C::NE];
        float tmax = -INFINITY;
#pragma unroll
        for (int t = 0; t < C::NE; ++t) {
          const int e = lane + 32 * t;
          lv[t] = e < C::RB * G ? sl[e] : -INFINITY;
          tmax = fmaxf(tmax, lv[t]);
        }
        if (emit) {
          float* lg_out = a.logits + (size_t(I.u) * a.max_len + c0 + wr0) * G;
#pragma unroll
          for (int t = 0; t < C::NE; ++t) {
            const int e = lane + 32 * t;
            if (e < nw * G) lg_out[e] = lv[t];
          }
          if (norm_stage && lane < nw) a.knorm[size_t(I.u) * a.max_len + c0 + wr0 + lane] = sn[lane];
        }
#pragma unroll
        for (int o = G; o < 32; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, o));
        bool changed = false;
        float mn[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float t = __shfl_sync(kFull, tmax, hh);
          mn[hh] = fmaxf(m[hh], t);
          changed |= mn[hh] > m[hh];
        }
        if (changed) {
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            const float al = exp2f(m[hh] - mn[hh]);
#pragma unroll
            for (int e = 0; e < C::EPL; ++e) acc[hh][e] *= al;
            if (hl == hh) zl *= al;
            m[hh] = mn[hh];
          }
        }
        float mine = m[0];
#pragma unroll
        for (int hh = 1; hh < G; ++hh)
          if (hl == hh) mine = m[hh];
#pragma unroll
        for (int t = 0; t < C::NE; ++t) {
          const int e = lane + 32 * t;
          const float p = exp2f(lv[t] - mine);
          zl += p;
          if (e < C::RB * G) sl[e] = p;
        }
        __syncwarp();
        // ---- p . v
        const uint32_t vrow = vbase + slot * C::STAGE_B + (wr0 + lg * C::R) * C::ROWB + li * 16;
#pragma unroll
        for (int r = 0; r < C::R; ++r) {
          const int row = lg * C::R + r;
          if (row < nw) {
            float pp[G];
#pragma unroll
            for (int hh = 0; hh < G; ++hh) pp[hh] = sl[row * G + hh];
            const uint4 raw = lds128(vrow + r * C::ROWB);
            float vf[C::EPL];
            Unpack<T>::run(raw, vf);
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
#pragma unroll
              for (int e = 0; e < C::EPL; ++e) acc[hh][e] = fmaf(pp[hh], vf[e], acc[hh][e]);
          }
        }
      }
      // a stage given up on is released only once its rows have landed, so
      // no copy into the slot is still in flight when it is refilled
      if (!have) mbar_wait(bar_full + 8 * slot, ph);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
      ++stage;
    }

    // ---- merge the lane groups of this warp
#pragma unroll
    for (int o = C::LPR; o < 32; o <<= 1)
#pragma unroll
      for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int e = 0; e < C::EPL; ++e) acc[hh][e] += __shfl_xor_sync(kFull, acc[hh][e], o);
#pragma unroll
    for (int o = G; o < 32; o <<= 1) zl += __shfl_xor_sync(kFull, zl, o);
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      if (lane == hh) {
        red[hh * (D + 2)] = m[hh];
        red[hh * (D + 2) + 1] = zl;
      }
    }
    if (lg == 0) {
#pragma unroll
      for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int e = 0; e < C::EPL; ++e) red[hh * (D + 2) + 2 + li * C::EPL + e] = acc[hh][e];
    }
}

// Consumer warp, tensor-core path (bf16): warp `warp` takes rows
// [16 * (warp % 4), +16) of every stage whose index has parity warp / 4.
// S^T = K Q^T with the warp's 16 K rows as the A operand and the query heads
// as the N dimension (heads G..7 are zero), then O^T += V^T P^T with 16
// dimensions of V^T per A tile and P^T as the B operand, moved from the
// accumulator layout by movmatrix.trans.  fp32 accumulation throughout; P is
// rounded to bf16 for the product.  Lane (g, t) = (lane / 4, lane % 4) holds
// S^T and O^T at rows (or dimensions) g and g + 8 and heads 2t and 2t + 1.
template <int D, int G>
__device__ __forceinline__ void attn_item_mma(const AttnArgs& a, const ItemInfo& I,
                                              unsigned char* smem, uint32_t bar_full,
                                              uint32_t bar_empty, volatile int* abort_flag,
                                              uint32_t& stage, int warp, int lane, float* red) {
  using C = AttnCfg<bf16_t, D, G>;
  constexpr int KS = D / 16;  // 16-dimension k-steps of S^T
  constexpr int DT = D / 16;  // 16-dimension tiles of O^T
  const int g = lane >> 2, t = lane & 3;
  const int wslot = warp & 3, wpar = warp >> 2;
  const uint32_t kbase = smem_addr(smem + C::OFF_K), vbase = smem_addr(smem + C::OFF_V);
  const bool emit = a.emit && I.slow;
  const bool emit_norm = emit && a.knorm != nullptr;
  // key norms of rows below nv are already stored (they never change)
  const int nv = emit_norm && a.knorm_valid ? a.knorm_valid[I.u] : 0;
  const float qs = a.qscale;

  // B operand of S^T: q of head g (zero for heads >= G), bf16 pairs at
  // dimensions 16 ks + 2t and 16 ks + 8 + 2t.
  uint32_t qb[KS][2];
  {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(a.q) +
                           ((size_t(I.b) * a.H_q + size_t(I.g) * G + (g < G ? g : 0)) * D) / 2;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qb[ks][0] = g < G ? __ldg(qrow + ks * 8 + t) : 0u;
      qb[ks][1] = g < G ? __ldg(qrow + ks * 8 + 4 + t) : 0u;
    }
  }
  float acc[DT][4];
#pragma unroll
  for (int c = 0; c < DT; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, zl[2] = {0.f, 0.f};  // heads 2t, 2t + 1
  // ldmatrix row addresses: K rows for the A tiles of S^T, V rows for V^T
  const int krow = (lane & 7) + ((lane >> 3) & 1) * 8, kch = lane >> 4;
  const int vrow = (lane & 7) + ((lane >> 4) & 1) * 8, vch = (lane >> 3) & 1;

  for (int si = 0; si < I.n_st; ++si, ++stage) {
    if (int(stage & 1u) != wpar) continue;
    const int c0 = I.c_first + si * I.c_step;
    const int nr = min(C::SR, I.rows - c0);
    const int slot = stage % C::NS;
    const uint32_t ph = (stage / C::NS) & 1u;
    const bool have = warp_pipe_wait(bar_full + 8 * slot, ph, abort_flag, a.status, a.wait_cycles);
    const int r0 = wslot * C::MW;
    const int nw = min(C::MW, nr - r0);  // valid rows of this warp (may be <= 0)
    if (have && nw > 0) {
      const uint32_t kst = kbase + slot * C::STAGE_B;
      const uint32_t vst = vbase + slot * C::STAGE_B;
      // ---- S^T = K Q^T over the warp's 16 rows (two accumulator chains);
      // with key norms, the squares of the same K fragments.  The two
      // variants are separate loops, so neither carries a branch that would
      // keep the compiler from issuing the next k-step's loads early.
      float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      // Key norms on the tensor cores: the A fragments of the K tile are also
      // the B fragments of K^T, so K K^T (16 x 16, in two 8-column halves)
      // accumulates next to S^T; its diagonal holds the squared row norms.
      float gram[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      auto qk = [&](auto with_norm) {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(kst + C::chunk_off(r0 + krow, 2 * ks + kch), a0, a1, a2, a3);
          mma_bf16_16816(sa[ks & 1], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
          if constexpr (decltype(with_norm)::value) {
            mma_bf16_16816(gram[0], a0, a1, a2, a3, a0, a2);  // columns: rows 0-7
            mma_bf16_16816(gram[1], a0, a1, a2, a3, a1, a3);  // columns: rows 8-15
          }
        }
      };
      const bool norm_stage = emit_norm && c0 + nr > nv;
      if (norm_stage) {
        qk(std::true_type{});
      } else {
        qk(std::false_type{});
      }
      // this lane's logits (log2 domain): [row g / g + 8][head 2t / 2t + 1]
      float l[2][2];
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          l[r][h] = g + 8 * r < nw ? (sa[0][2 * r + h] + sa[1][2 * r + h]) * qs : -INFINITY;
      if (emit) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int rr = g + 8 * r;
          if (rr < nw) {
            float* lo = a.logits + (size_t(I.u) * a.max_len + c0 + r0 + rr) * G;
#pragma unroll
            for (int h = 0; h < 2; ++h)
              if (2 * t + h < G) lo[2 * t + h] = l[r][h];
          }
        }
        if (norm_stage && t == (g >> 1)) {
          // lane (g, g / 2) holds the diagonal entries (g, g) and (g + 8, g + 8)
          const float n0 = (g & 1) ? gram[0][1] : gram[0][0];
          const float n1 = (g & 1) ? gram[1][3] : gram[1][2];
          float* kn = a.knorm + size_t(I.u) * a.max_len + c0 + r0;
          if (g < nw) kn[g] = sqrtf(n0);
          if (g + 8 < nw) kn[g + 8] = sqrtf(n1);
        }
      }
      // ---- online softmax per head over the warp's 16 rows (lanes with the
      // same t share a head; the max runs over g)
      float p[2][2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float tmax = fmaxf(l[0][h], l[1][h]);
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 4));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 8));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 16));
        if (tmax > m[h]) {
          const float al = exp2f(m[h] - tmax);
#pragma unroll
          for (int c = 0; c < DT; ++c) {
            acc[c][h] *= al;
            acc[c][2 + h] *= al;
          }
          zl[h] *= al;
          m[h] = tmax;
        }
        p[0][h] = exp2f(l[0][h] - m[h]);
        p[1][h] = exp2f(l[1][h] - m[h]);
        zl[h] += p[0][h] + p[1][h];
      }
      // P^T as the B operand: rows 0-7 and 8-15, transposed from the
      // accumulator layout (row g, heads 2t..) to (rows 2t.., head g)
      const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p[0][0], p[0][1]));
      const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p[1][0], p[1][1]));
      // rows past the valid ones hold stale or unset data: zero their V
      uint32_t m_lo = 0xffffffffu, m_hi = 0xffffffffu;
      if (nw < C::MW) {
        m_lo = (2 * t < nw ? 0x0000ffffu : 0u) | (2 * t + 1 < nw ? 0xffff0000u : 0u);
        m_hi = (8 + 2 * t < nw ? 0x0000ffffu : 0u) | (9 + 2 * t < nw ? 0xffff0000u : 0u);
      }
      // ---- O^T += V^T P^T, 16 dimensions per tile
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_trans(vst + C::chunk_off(r0 + vrow, 2 * dt + vch), v0, v1, v2, v3);
        mma_bf16_16816(acc[dt], v0 & m_lo, v1 & m_lo, v2 & m_hi, v3 & m_hi, pb0, pb1);
      }
    }
    // a stage given up on is released only once its rows have landed, so
    // no copy into the slot is still in flight when it is refilled
    if (!have) mbar_wait(bar_full + 8 * slot, ph);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
  }
  // ---- warp state of heads 2t, 2t + 1 (sums over the rows g)
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    zl[h] += __shfl_xor_sync(kFull, zl[h], 4);
    zl[h] += __shfl_xor_sync(kFull, zl[h], 8);
    zl[h] += __shfl_xor_sync(kFull, zl[h], 16);
    const int hh = 2 * t + h;
    if (hh < G) {
      float* rw = red + hh * (D + 2);
      if (g == 0) {
        rw[0] = m[h];
        rw[1] = zl[h];
      }
#pragma unroll
      for (int c = 0; c < DT; ++c) {
        rw[2 + 16 * c + g] = acc[c][h];
        rw[2 + 16 * c + g + 8] = acc[c][2 + h];
      }
    }
  }
}

// Merge the n_items partial results of unit I.u (run by the CTA that
// finished its last item; `scr` is free shared scratch of at least
// G * (kItemSlotsPerUnit + 2) floats).  Warp hh < G takes head hh's maxima
// and sums (one item per lane), forms the global max M and the item scale
// factors 2^(m_i - M), and reduces Z; then every thread forms output
// elements as sum_i scale_i a_i[dim] with many loads in flight.  The order
// of every sum is fixed, so the result does not depend on the schedule.
template <int D, int G>
__device__ __forceinline__ void attn_merge_items(const AttnArgs& a, const ItemInfo& I, bool emit,
                                                 float* scr, int tid, int nct) {
  static_assert(G <= 8, "one warp per head");
  static_assert(kItemSlotsPerUnit <= 64, "two items per lane");
  constexpr int P = D + 2;
  const int n = I.n_items;  // <= kItemSlotsPerUnit = 64
  const float* part = a.partials + size_t(I.first) * G * P;
  float* sc = scr;                                 // [n][G]
  float* mz = scr + kItemSlotsPerUnit * G;         // [G][2]: M, Z
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < G) {
    const int hh = warp;
    float m[2], z[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int i = lane + 32 * r;
      m[r] = i < n ? __ldcg(part + (size_t(i) * G + hh) * P) : -INFINITY;
      z[r] = i < n ? __ldcg(part + (size_t(i) * G + hh) * P + 1) : 0.f;
    }
    float M = fmaxf(m[0], m[1]);
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    float Z = 0.f;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int i = lane + 32 * r;
      const float f = i < n && m[r] != -INFINITY ? exp2f(m[r] - M) : 0.f;  // empty items: 0
      if (i < n) sc[i * G + hh] = f;
      Z = fmaf(z[r], f, Z);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) Z += __shfl_xor_sync(kFull, Z, o);
    if (lane == 0) {
      mz[2 * hh] = M;
      mz[2 * hh + 1] = Z;
    }
  }
  named_bar_sync(1, nct);
  for (int j = tid; j < G * D; j += nct) {
    const int hh = j / D, dim = j % D;
    const float* pa = part + size_t(hh) * P + 2 + dim;
    const size_t stride = size_t(G) * P;
    float A = 0.f;
    int i = 0;
    for (; i + 16 <= n; i += 16) {
      float v[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) v[t] = __ldcg(pa + (i + t) * stride);
#pragma unroll
      for (int t = 0; t < 16; ++t) A = fmaf(v[t], sc[(i + t) * G + hh], A);
    }
    for (; i < n; ++i) A = fmaf(__ldcg(pa + i * stride), sc[i * G + hh], A);
    const float M = mz[2 * hh], Z = mz[2 * hh + 1];
    const size_t qh = size_t(I.b) * a.H_q + size_t(I.g) * G + hh;
    a.out[qh * D + dim] = A / Z;
    if (emit && dim == 0) {
      a.stats[qh * 2] = M;
      a.stats[qh * 2 + 1] = Z;
    }
  }
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(AttnCfg<T, D, G>::NT, 1)
    attn_kernel(const __grid_constant__ AttnArgs a) {
  using C = AttnCfg<T, D, G>;
  extern __shared__ __align__(1024) unsigned char smem[];
  // launched as a programmatic dependent: wait until the previous grid on the
  // stream has completed and its writes are visible before any global access
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_units = a.B * a.H_kv;
  int* units = reinterpret_cast<int*>(smem + C::OFF_UNITS);
  int* misc = reinterpret_cast<int*>(smem + C::OFF_MISC);
  const uint32_t bar_full = smem_addr(smem + C::OFF_BAR);
  const uint32_t bar_empty = bar_full + C::NS * 8;

  // the CTA's first item is its own index (later ones from the work counter)
  const unsigned first_id = blockIdx.x;
  const bool fetcher = warp == C::NCW && lane == 0;
  if (a.len_copy && blockIdx.x == 0)
    for (int b = tid; b < a.B; b += C::NT) a.len_copy[b] = a.len[b];
  // A launch of fast units only, each cut into exactly fast_items items (the
  // host checked both item limits), needs no unit table: an item's unit
  // follows from its id, and the first item starts without waiting for the
  // table's loads.
  bool units_fit = true;
  int total;
  if (a.fast_items > 0) {
    total = n_units * a.fast_items;
  } else {
    units_fit = attn_build_units<C::NT>(a, units, n_units, misc);
    total = units[n_units];
  }
  if (total > a.max_items || !units_fit) {
    if (tid == 0 && blockIdx.x == 0) set_status(a.status, SFI_DEV_ITEMS_OVERFLOW);
    // leave the work counters at zero for the next launch
    if (fetcher && atomicAdd(a.work_ctr + 1, 1u) == gridDim.x - 1) {
      atomicExch(a.work_ctr, 0u);
      atomicExch(a.work_ctr + 1, 0u);
    }
    return;
  }
  volatile int* abort_flag = misc + kMiscAbort;  // misc[0..12]: unit-table scan scratch
  ItemRing ring;
  ring.full = bar_empty + C::NS * 8;
  ring.empty = ring.full + kItemRing * 8;
  ring.slot = misc + kMiscRing;
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(bar_full + 8 * s, 32 * C::PW);  // one arrival per producer lane
      mbar_init(bar_empty + 8 * s, C::CPS);  // one arrival per consuming warp
    }
    for (int s = 0; s < kItemRing; ++s) {
      mbar_init(ring.full + 8 * s, 1);
      mbar_init(ring.empty + 8 * s, C::PW);  // other producer warps + consumer warp 0
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp >= C::NCW) {
    attn_produce<C>(a, units, n_units, total, smem, bar_full, bar_empty, ring, abort_flag,
                    warp - C::NCW, lane, first_id);
    return;
  }

  // -------------------------------------------------------------- consumers
  float* red_all = reinterpret_cast<float*>(smem + C::OFF_RED);
  const int nct = C::NCW * 32;
  uint32_t stage = 0;

  volatile int* cur_item = misc + kMiscCurItem;
  for (uint32_t iseq = 0;; ++iseq) {
    // consumer warp 0 takes the item id from the ring and shares it
    if (warp == 0) {
      const int x = ring_read(a, ring, iseq, abort_flag, lane);
      if (lane == 0) *cur_item = x;
    }
    named_bar_sync(1, nct);
    const int it = *cur_item;
    named_bar_sync(1, nct);
    if (it < 0) break;
    const ItemInfo I = attn_resolve(a, units, n_units, it, C::SR);
    const bool emit = a.emit && I.slow;
    float* red = red_all + warp * G * (D + 2);
    // Tensor-core warps split stages by the parity of the CTA's running stage
    // count, so which group holds the item's even stages depends on the
    // CTA's earlier items; merging the groups in item order keeps the result
    // independent of which CTA ran the item.
    const int wflip = C::MMA ? int(stage & 1u) * 4 : 0;
    if constexpr (C::MMA) {
      attn_item_mma<D, G>(a, I, smem, bar_full, bar_empty, abort_flag, stage, warp, lane, red);
    } else {
      attn_item_simt<T, D, G>(a, I, smem, bar_full, bar_empty, abort_flag, stage, warp, lane, red);
    }
    named_bar_sync(1, nct);

    // ---- merge the consumer warps: item result
    float* part = a.partials + size_t(it) * G * (D + 2);
    const bool single = I.n_items == 1;
    for (int j = tid; j < G * D; j += nct) {
      const int hh = j / D, dim = j % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::NCW; ++w) M = fmaxf(M, red_all[(w * G + hh) * (D + 2)]);
      float A = 0.f, Z = 0.f;
#pragma unroll
      for (int w = 0; w < C::NCW; ++w) {
        const float* rw = red_all + ((w ^ wflip) * G + hh) * (D + 2);
        // a warp (or a whole item) without rows holds m = -inf: weight 0
        const float sc = rw[0] == -INFINITY ? 0.f : exp2f(rw[0] - M);
        Z = fmaf(rw[1], sc, Z);
        A = fmaf(rw[2 + dim], sc, A);
      }
      const size_t qh = size_t(I.b) * a.H_q + size_t(I.g) * G + hh;
      if (single) {
        a.out[qh * D + dim] = A / Z;
        if (emit && dim == 0) {
          a.stats[qh * 2] = M;
          a.stats[qh * 2 + 1] = Z;
        }
      } else {
        __stcg(part + hh * (D + 2) + 2 + dim, A);
        if (dim == 0) {
          __stcg(part + hh * (D + 2), M);
          __stcg(part + hh * (D + 2) + 1, Z);
        }
      }
    }
    // a refreshing unit whose rows all have their key norms stored now
    const bool norms_done = emit && a.knorm != nullptr && a.knorm_valid != nullptr;
    if (single && norms_done && tid == 0) a.knorm_valid[I.u] = I.n;
    if (!single) {
      __threadfence();
      named_bar_sync(1, nct);
      if (tid == 0) misc[kMiscLast] = atomicAdd(a.counters + I.u, 1) == I.n_items - 1;
      named_bar_sync(1, nct);
      if (misc[kMiscLast]) {
        __threadfence();
        attn_merge_items<D, G>(a, I, emit, red_all, tid, nct);
        if (tid == 0) {
          a.counters[I.u] = 0;
          if (norms_done) a.knorm_valid[I.u] = I.n;
        }
      }
    }
    named_bar_sync(1, nct);
  }
}

template <typename T, int D, int G>
cudaError_t launch_attn_t(const AttnArgs& a, cudaStream_t st, bool pdl) {
  using C = AttnCfg<T, D, G>;
  const int n_units = a.B * a.H_kv;
  const size_t smem = C::smem_bytes(n_units);
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<T, D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(device_sm_count());
  cfg.blockDim = dim3(C::NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_kernel<T, D, G>, a);
}

}  // namespace sfi
