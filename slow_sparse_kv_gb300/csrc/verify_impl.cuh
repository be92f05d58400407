// Verification attention with Collect-2 logit sums (Vegas).
//
// Vegas (gist.science 2602.07223, section 2 "Verification phase" and 2.A-2.B):
// the verification pass attends densely with the gamma + 1 rows of the draft
// chain, and the attention logits it computes anyway pick the KV entries of
// the next drafting phase: T = argmax over k-subsets of the prefix of the
// logits summed over the collected query rows and all query heads; the
// "Collect-2-Query" variant collects only the first draft row and the bonus
// row.
//
// For each (sequence, KV head) unit the kernel streams the cache once (the
// decode kernel's producer: 64 x 64 TMA boxes) and serves all R = n_rows
// chain rows of the unit's G query heads at once.  The QR = R * G query rows
// are the N dimension of S^T = K Q^T (NTT tiles of 8 columns; tile slot c is
// chain row t_of_slot[c / G], head c % G, collected rows first), so one warp
// holds the logits of every query row for its 16 cache rows: the
// collected-row sum of a position is a reduction over a lane quad, and
// O^T += V^T P^T reuses each V^T tile for all NTT column tiles.  The eight
// consumer warps form two groups by stage parity (each stage is taken by
// four warps, 16 rows each), so two stages are in flight per CTA.  Row t of
// the chain sits at position n - R + t and attends to [0, n - R + t]
// (causal tail).  Every consumer warp ends an item with the full O^T, m and
// z of its rows (the same register layout in every warp); the eight states
// are merged in three fixed rounds through shared memory.
#pragma once

#include <math.h>

#include "attn_kernel.cuh"

namespace sfi {

constexpr int kVerifyMaxTiles = 4;  // QR <= 32

template <int D>
struct VerifyCfg {
  static constexpr bool MMA = true;
  static constexpr int DIM = D;
  static constexpr int ES = 2;
  static constexpr int ROWB = D * ES;
  static constexpr int LPR = ROWB / 16;
  static constexpr int RPI = 32 / LPR;
  static constexpr int NCW = 8;
  static constexpr int MW = 16;
  static constexpr int CPS = 4;  // consumer warps per stage: the two parity groups alternate
  static constexpr int SR = MW * 4;
  static constexpr int PW = 1;  // one producer warp: full stages are TMA boxes
  static constexpr int NT = (NCW + PW) * 32;
  static constexpr int STAGE_B = SR * ROWB;
  // per-lane state of one warp: O^T tiles, then m and z of its 2 columns per tile
  static constexpr int STATE = (D / 16) * kVerifyMaxTiles * 4 + kVerifyMaxTiles * 4;
  static constexpr size_t RED_B = size_t(4) * 32 * STATE * 4;  // four warps' states
  static_assert(size_t(32) * (D + 2) * 4 <= RED_B, "the final [column][D + 2] rows fit the merge buffer");
  static_assert((size_t(kItemSlotsPerUnit) * 32 + 64) * 4 <= RED_B, "item scales fit the merge buffer");
  static constexpr int NS_FIT =
      int((227 * 1024 - 2048 - RED_B - size_t(8 * kVerifyMaxTiles) * (D * 2 + 16) -
           (size_t(kMaxUnits) + 1 + kRankWords) * 4) / (2 * size_t(SR) * ROWB));
  static constexpr int NS = NS_FIT > 6 ? 6 : NS_FIT;
  static_assert(NS >= 2, "verify pipeline does not fit");
  static_assert(SR % (PW * RPI) == 0, "stage rows split evenly over the producer warps");
  static constexpr size_t OFF_K = 0;
  static constexpr size_t OFF_V = OFF_K + size_t(NS) * STAGE_B;
  static constexpr size_t OFF_BAR = OFF_V + size_t(NS) * STAGE_B;
  static constexpr size_t OFF_RED = OFF_BAR + (2 * NS + 2 * kItemRing) * 8;
  // the unit's query rows, [column][D] bf16, rows padded by 16 bytes so the
  // eight rows of an ldmatrix fall in different banks
  static constexpr int QROWB = D * 2 + 16;
  static constexpr size_t OFF_Q = OFF_RED + RED_B;
  static constexpr size_t OFF_MISC = OFF_Q + size_t(8 * kVerifyMaxTiles) * QROWB;
  static constexpr size_t OFF_UNITS = OFF_MISC + 128;
  static size_t smem_bytes(int n_units) { return OFF_UNITS + size_t(n_units + 1 + kRankWords) * 4; }
  static_assert(OFF_UNITS + (size_t(kMaxUnits) + 1 + kRankWords) * 4 <= size_t(227) * 1024,
                "shared memory plan exceeds 227 KB");
  static __device__ __forceinline__ uint32_t chunk_off(int r, int c) {
    return uint32_t((c >> 3) * (SR * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
  }
};

// One warp's running state over an item: O^T[dim][column] (lane (g, t) holds
// dims 16 dt + g (+ 8) of columns 8 j + 2 t (+ 1)), and m, z of its columns.
template <int D, int NTT>
struct VState {
  float acc[D / 16][NTT][4];
  float m[NTT][2], z[NTT][2];
};

// A warp's state in shared memory: element i of lane l at o[i * 32 + l]
// (consecutive lanes in consecutive banks).  `o` points at the warp's block
// plus the lane.
// Combine `o` (the part of the item later in the fixed order) into `s`.
template <int D, int NTT>
__device__ __forceinline__ void vstate_merge(VState<D, NTT>& s, const float* o) {
  constexpr int DT = D / 16;
#pragma unroll
  for (int j = 0; j < NTT; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float mo = o[(DT * NTT * 4 + (j * 2 + h)) * 32];
      const float zo = o[(DT * NTT * 4 + 2 * NTT + (j * 2 + h)) * 32];
      const float M = fmaxf(s.m[j][h], mo);
      const float sa = s.m[j][h] == -INFINITY ? 0.f : exp2f(s.m[j][h] - M);
      const float sb = mo == -INFINITY ? 0.f : exp2f(mo - M);
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
        s.acc[dt][j][h] = fmaf(o[((dt * NTT + j) * 4 + h) * 32], sb, s.acc[dt][j][h] * sa);
        s.acc[dt][j][2 + h] = fmaf(o[((dt * NTT + j) * 4 + 2 + h) * 32], sb, s.acc[dt][j][2 + h] * sa);
      }
      s.z[j][h] = fmaf(zo, sb, s.z[j][h] * sa);
      s.m[j][h] = M;
    }
}

template <int D, int NTT>
__device__ __forceinline__ void vstate_store(const VState<D, NTT>& s, float* o) {
  constexpr int DT = D / 16;
#pragma unroll
  for (int dt = 0; dt < DT; ++dt)
#pragma unroll
    for (int j = 0; j < NTT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[((dt * NTT + j) * 4 + e) * 32] = s.acc[dt][j][e];
#pragma unroll
  for (int j = 0; j < NTT; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      o[(DT * NTT * 4 + (j * 2 + h)) * 32] = s.m[j][h];
      o[(DT * NTT * 4 + 2 * NTT + (j * 2 + h)) * 32] = s.z[j][h];
    }
}

// Consumer warp: this item's stages of the warp's parity, rows
// [16 (warp % 4), +16) of each.
template <int D, int G, int NTT>
__device__ __forceinline__ void verify_item(const VerifyArgs& va, const ItemInfo& I,
                                            unsigned char* smem, uint32_t bar_full,
                                            uint32_t bar_empty, volatile int* abort_flag,
                                            uint32_t& stage, int warp, int lane,
                                            VState<D, NTT>& st) {
  using C = VerifyCfg<D>;
  const AttnArgs& a = va.base;
  constexpr int KS = D / 16;  // k-steps of S^T
  constexpr int DT = D / 16;  // 16-dimension tiles of O^T
  const int g = lane >> 2, t = lane & 3;
  const int wslot = warp & 3, wpar = warp >> 2;
  const int QR = va.R * G;
  const uint32_t kbase = smem_addr(smem + C::OFF_K), vbase = smem_addr(smem + C::OFF_V);
  const float qs = a.qscale;
  const int n_pre = I.n - va.R;

  // B fragments of Q^T come from the query rows staged in shared memory
  // (verify_stage_q, before the item): ldmatrix of 8 columns x 8 dimensions,
  // two column tiles per x4 load; lane l addresses column 8 (2 jj + l / 16) +
  // l % 8 at dimension offset 8 ((l / 8) % 2)
  const uint32_t qbase = smem_addr(smem + C::OFF_Q) + uint32_t(((lane >> 4) * 8 + (lane & 7)) * C::QROWB +
                                                                ((lane >> 3) & 1) * 16);
  // the lane's columns 8 j + 2 t + h: causal limit (-1: padding, never
  // attends) and whether the column is collected
  int lim[NTT][2];
  bool coll[NTT][2];
#pragma unroll
  for (int j = 0; j < NTT; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = 8 * j + 2 * t + h;
      lim[j][h] = c < QR ? I.n - va.R + va.t_of_slot[c / G] : -1;
      coll[j][h] = c < va.ncg;
    }
#pragma unroll
  for (int dt = 0; dt < DT; ++dt)
#pragma unroll
    for (int j = 0; j < NTT; ++j) st.acc[dt][j][0] = st.acc[dt][j][1] = st.acc[dt][j][2] = st.acc[dt][j][3] = 0.f;
#pragma unroll
  for (int j = 0; j < NTT; ++j) st.m[j][0] = st.m[j][1] = -INFINITY, st.z[j][0] = st.z[j][1] = 0.f;
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
      // ---- S^T = K Q^T: two accumulator chains per column tile when the
      // tiles are few (three or more tiles interleave enough chains already)
      constexpr int NCH = NTT >= 3 ? 1 : 2;
      float sa[NTT][2][4];
#pragma unroll
      for (int j = 0; j < NTT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[j][0][e] = sa[j][1][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kst + C::chunk_off(r0 + krow, 2 * ks + kch), a0, a1, a2, a3);
#pragma unroll
        for (int jj = 0; jj < (NTT + 1) / 2; ++jj) {
          uint32_t b0, b1, b2, b3;  // (tile 2 jj: b0, b1), (tile 2 jj + 1: b2, b3)
          ldsm_x4(qbase + uint32_t(16 * jj * C::QROWB + ks * 32), b0, b1, b2, b3);
          mma_bf16_16816(sa[2 * jj][ks % NCH], a0, a1, a2, a3, b0, b1);
          if (2 * jj + 1 < NTT) mma_bf16_16816(sa[2 * jj + 1][ks % NCH], a0, a1, a2, a3, b2, b3);
        }
      }
      // ---- logits (log2 domain, masked) and the collected rows' sums
      float l[NTT][2][2];  // [tile][row g / g + 8][column 2t / 2t + 1]
      float ls[2] = {0.f, 0.f};
#pragma unroll
      for (int j = 0; j < NTT; ++j)
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float raw = sa[j][0][2 * r + h] + sa[j][1][2 * r + h];
            if (coll[j][h]) ls[r] += raw;
            const int pos = c0 + r0 + g + 8 * r;
            l[j][r][h] = (g + 8 * r < nw && pos <= lim[j][h]) ? raw * qs : -INFINITY;
          }
      if (va.lsum) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          ls[r] += __shfl_xor_sync(kFull, ls[r], 1);
          ls[r] += __shfl_xor_sync(kFull, ls[r], 2);
        }
        if (t == 0) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int pos = c0 + r0 + g + 8 * r;
            if (g + 8 * r < nw && pos < n_pre) va.lsum[size_t(I.u) * a.max_len + pos] = ls[r] * va.lscale;
          }
        }
      }
      // ---- online softmax per column (lanes with the same t share columns;
      // the max runs over g)
      uint32_t pb[NTT][2];
#pragma unroll
      for (int j = 0; j < NTT; ++j) {
        float p[2][2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float tmax = fmaxf(l[j][0][h], l[j][1][h]);
          tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 4));
          tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 8));
          tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 16));
          if (tmax > st.m[j][h]) {
            const float al = st.m[j][h] == -INFINITY ? 0.f : exp2f(st.m[j][h] - tmax);
#pragma unroll
            for (int dt = 0; dt < DT; ++dt) {
              st.acc[dt][j][h] *= al;
              st.acc[dt][j][2 + h] *= al;
            }
            st.z[j][h] *= al;
            st.m[j][h] = tmax;
          }
          // a column with every logit masked so far keeps m = -inf: its p is 0
          p[0][h] = l[j][0][h] == -INFINITY ? 0.f : exp2f(l[j][0][h] - st.m[j][h]);
          p[1][h] = l[j][1][h] == -INFINITY ? 0.f : exp2f(l[j][1][h] - st.m[j][h]);
          st.z[j][h] += p[0][h] + p[1][h];
        }
        // P^T of this tile as the B operand: rows 0-7 and 8-15
        pb[j][0] = movmatrix_trans(pack_bf16x2(p[0][0], p[0][1]));
        pb[j][1] = movmatrix_trans(pack_bf16x2(p[1][0], p[1][1]));
      }
      // rows past the valid ones hold stale or unset data: zero their V
      uint32_t m_lo = 0xffffffffu, m_hi = 0xffffffffu;
      if (nw < C::MW) {
        m_lo = (2 * t < nw ? 0x0000ffffu : 0u) | (2 * t + 1 < nw ? 0xffff0000u : 0u);
        m_hi = (8 + 2 * t < nw ? 0x0000ffffu : 0u) | (9 + 2 * t < nw ? 0xffff0000u : 0u);
      }
      // ---- O^T += V^T P^T, one V^T tile for every column tile
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_trans(vst + C::chunk_off(r0 + vrow, 2 * dt + vch), v0, v1, v2, v3);
        v0 &= m_lo;
        v1 &= m_lo;
        v2 &= m_hi;
        v3 &= m_hi;
#pragma unroll
        for (int j = 0; j < NTT; ++j) mma_bf16_16816(st.acc[dt][j], v0, v1, v2, v3, pb[j][0], pb[j][1]);
      }
    }
    // a stage given up on is released only once its rows have landed, so
    // no copy into the slot is still in flight when it is refilled
    if (!have) mbar_wait(bar_full + 8 * slot, ph);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
  }
  // z of each column over the rows g
#pragma unroll
  for (int j = 0; j < NTT; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      st.z[j][h] += __shfl_xor_sync(kFull, st.z[j][h], 4);
      st.z[j][h] += __shfl_xor_sync(kFull, st.z[j][h], 8);
      st.z[j][h] += __shfl_xor_sync(kFull, st.z[j][h], 16);
    }
}

// Stage unit I's query rows in shared memory as [column c][D] bf16 (column
// c = chain row t_of_slot[c / G], head c % G; zero rows past QR up to the 8
// columns of the last tile pair), by all consumer threads.
template <int D, int G>
__device__ __forceinline__ void verify_stage_q(const VerifyArgs& va, const ItemInfo& I,
                                               unsigned char* smem, int tid, int nct) {
  using C = VerifyCfg<D>;
  const AttnArgs& a = va.base;
  const int QR = va.R * G;
  constexpr int CH = D / 8;  // 16-byte chunks per row
  for (int i = tid; i < 8 * kVerifyMaxTiles * CH; i += nct) {
    const int c = i / CH, ch = i % CH;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (c < QR) {
      const int tr = va.t_of_slot[c / G];
      const size_t qh = (size_t(I.b) * va.R + tr) * a.H_q + size_t(I.g) * G + c % G;
      v = __ldg(reinterpret_cast<const uint4*>(a.q) + qh * CH + ch);
    }
    *reinterpret_cast<uint4*>(smem + C::OFF_Q + size_t(c) * C::QROWB + ch * 16) = v;
  }
}

template <int D, int G, int NTT>
__global__ void __launch_bounds__(VerifyCfg<D>::NT, 1)
    verify_kernel(const __grid_constant__ VerifyArgs va) {
  using C = VerifyCfg<D>;
  const AttnArgs& a = va.base;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_units = a.B * a.H_kv;
  int* units = reinterpret_cast<int*>(smem + C::OFF_UNITS);
  int* misc = reinterpret_cast<int*>(smem + C::OFF_MISC);
  const uint32_t bar_full = smem_addr(smem + C::OFF_BAR);
  const uint32_t bar_empty = bar_full + C::NS * 8;
  // the CTA's first item is its own index (later ones from the work counter)
  const unsigned first_id = blockIdx.x;
  const bool fetcher = warp == C::NCW && lane == 0;
  const bool units_fit = attn_build_units<C::NT>(a, units, n_units, misc);  // fast_items is 0
  const int total = units[n_units];
  if (total > a.max_items || !units_fit) {
    if (tid == 0 && blockIdx.x == 0) set_status(a.status, SFI_DEV_ITEMS_OVERFLOW);
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
      mbar_init(bar_full + 8 * s, 32 * C::PW);
      mbar_init(bar_empty + 8 * s, C::CPS);
    }
    for (int s = 0; s < kItemRing; ++s) {
      mbar_init(ring.full + 8 * s, 1);
      mbar_init(ring.empty + 8 * s, C::PW);  // the other producer warps (none) + consumer warp 0
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp >= C::NCW) {
    attn_produce<C>(a, units, n_units, total, smem, bar_full, bar_empty, ring, abort_flag,
                    warp - C::NCW, lane, first_id);
    return;
  }
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  const int nct = C::NCW * 32;
  const int QR = va.R * G;
  constexpr int S = C::STATE;
  uint32_t stage = 0;
  volatile int* cur_item = misc + kMiscCurItem;
  for (uint32_t iseq = 0;; ++iseq) {
    if (warp == 0) {
      const int x = ring_read(a, ring, iseq, abort_flag, lane);
      if (lane == 0) *cur_item = x;
    }
    named_bar_sync(1, nct);
    const int it = *cur_item;
    named_bar_sync(1, nct);
    if (it < 0) break;
    const ItemInfo I = attn_resolve(a, units, n_units, it, C::SR);
    // the group of warps that takes the item's first stage comes first in
    // every merge, so the result does not depend on which CTA ran the item
    const int first = int(stage & 1u);
    verify_stage_q<D, G>(va, I, smem, tid, nct);
    named_bar_sync(1, nct);
    VState<D, NTT> st;
    verify_item<D, G, NTT>(va, I, smem, bar_full, bar_empty, abort_flag, stage, warp, lane, st);
    const int wpar = warp >> 2, wslot = warp & 3;
    // ---- merge the eight warp states: the other group into the first, then
    // slots 2, 3 into 0, 1, then slot 1 into slot 0
    named_bar_sync(1, nct);
    if (wpar != first) vstate_store<D, NTT>(st, red + wslot * 32 * S + lane);
    named_bar_sync(1, nct);
    if (wpar == first) vstate_merge<D, NTT>(st, red + wslot * 32 * S + lane);
    named_bar_sync(1, nct);
    if (wpar == first && wslot >= 2) vstate_store<D, NTT>(st, red + (wslot - 2) * 32 * S + lane);
    named_bar_sync(1, nct);
    if (wpar == first && wslot < 2) vstate_merge<D, NTT>(st, red + wslot * 32 * S + lane);
    named_bar_sync(1, nct);
    if (wpar == first && wslot == 1) vstate_store<D, NTT>(st, red + lane);
    named_bar_sync(1, nct);
    if (wpar == first && wslot == 0) vstate_merge<D, NTT>(st, red + lane);
    named_bar_sync(1, nct);
    // ---- the item's rows [column][M, Z, O] in shared memory, then out
    if (wpar == first && wslot == 0) {
      const int g = lane >> 2, t = lane & 3;
#pragma unroll
      for (int j = 0; j < NTT; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = 8 * j + 2 * t + h;
          if (c < QR) {
            float* rw = red + c * (D + 2);
            if (g == 0) {
              rw[0] = st.m[j][h];
              rw[1] = st.z[j][h];
            }
#pragma unroll
            for (int dt = 0; dt < D / 16; ++dt) {
              rw[2 + 16 * dt + g] = st.acc[dt][j][h];
              rw[2 + 16 * dt + g + 8] = st.acc[dt][j][2 + h];
            }
          }
        }
    }
    named_bar_sync(1, nct);
    float* part = a.partials + size_t(it) * QR * (D + 2);
    const bool single = I.n_items == 1;
    for (int j = tid; j < QR * D; j += nct) {
      const int qr = j / D, dim = j % D;
      const float* rw = red + qr * (D + 2);
      const float M = rw[0], Z = rw[1], A = rw[2 + dim];
      const int tr = va.t_of_slot[qr / G], h = qr % G;
      const size_t oh = (size_t(I.b) * va.R + tr) * a.H_q + size_t(I.g) * G + h;
      if (single) {
        a.out[oh * D + dim] = A / Z;
      } else {
        __stcg(part + qr * (D + 2) + 2 + dim, A);
        if (dim == 0) {
          __stcg(part + qr * (D + 2), M);
          __stcg(part + qr * (D + 2) + 1, Z);
        }
      }
    }
    if (!single) {
      __threadfence();
      named_bar_sync(1, nct);
      if (tid == 0) misc[kMiscLast] = atomicAdd(a.counters + I.u, 1) == I.n_items - 1;
      named_bar_sync(1, nct);
      if (misc[kMiscLast]) {
        __threadfence();
        // the unit's items, merged by this CTA: per column (one warp each)
        // the maximum M over the items and each item's scale 2^(m_i - M)
        // once, in shared memory; then every output element sums its items'
        // partial rows with the loads in flight.  Fixed order throughout.
        const int n = I.n_items;  // <= kItemSlotsPerUnit = 64
        const size_t pstride = size_t(QR) * (D + 2);
        const float* pbase = a.partials + size_t(I.first) * pstride;
        float* sc = red;                              // [n][QR]
        float* mz = red + kItemSlotsPerUnit * 32;     // [QR][2]: M, Z
        for (int c = warp; c < QR; c += C::NCW) {
          float m[2], zz[2];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int i = lane + 32 * r;
            m[r] = i < n ? __ldcg(pbase + i * pstride + c * (D + 2)) : -INFINITY;
            zz[r] = i < n ? __ldcg(pbase + i * pstride + c * (D + 2) + 1) : 0.f;
          }
          float M = fmaxf(m[0], m[1]);
#pragma unroll
          for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
          float Z = 0.f;
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int i = lane + 32 * r;
            const float f = i < n && m[r] != -INFINITY ? exp2f(m[r] - M) : 0.f;
            if (i < n) sc[i * 32 + c] = f;
            Z = fmaf(zz[r], f, Z);
          }
#pragma unroll
          for (int o = 16; o; o >>= 1) Z += __shfl_xor_sync(kFull, Z, o);
          if (lane == 0) {
            mz[2 * c] = M;
            mz[2 * c + 1] = Z;
          }
        }
        named_bar_sync(1, nct);
        for (int j = tid; j < QR * D; j += nct) {
          const int qr = j / D, dim = j % D;
          const float* pa = pbase + qr * (D + 2) + 2 + dim;
          float A = 0.f;
          int i = 0;
          for (; i + 8 <= n; i += 8) {
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = __ldcg(pa + (i + q) * pstride);
#pragma unroll
            for (int q = 0; q < 8; ++q) A = fmaf(v[q], sc[(i + q) * 32 + qr], A);
          }
          for (; i < n; ++i) A = fmaf(__ldcg(pa + i * pstride), sc[i * 32 + qr], A);
          const int tr = va.t_of_slot[qr / G], h = qr % G;
          const size_t oh = (size_t(I.b) * va.R + tr) * a.H_q + size_t(I.g) * G + h;
          a.out[oh * D + dim] = A / mz[2 * qr + 1];
        }
        if (tid == 0) a.counters[I.u] = 0;
      }
    }
    named_bar_sync(1, nct);
  }
}

template <int D, int G, int NTT>
cudaError_t launch_verify_t(const VerifyArgs& va, cudaStream_t st) {
  using C = VerifyCfg<D>;
  const size_t smem = C::smem_bytes(va.base.B * va.base.H_kv);
  cudaError_t e = cudaFuncSetAttribute(verify_kernel<D, G, NTT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  verify_kernel<D, G, NTT><<<device_sm_count(), C::NT, smem, st>>>(va);
  return cudaGetLastError();
}

// Column tiles of 8 for QR = R * G query rows: 1 for G = 1, up to 2 for
// G = 2, up to 4 for G = 4 and G = 8 (QR <= 32).
template <int D>
cudaError_t launch_verify_d(const VerifyArgs& va, int G, cudaStream_t st) {
  const int ntt = (va.R * G + 7) / 8;
#define SFI_VCASE(GG, TT) \
  if (G == GG && ntt == TT) return launch_verify_t<D, GG, TT>(va, st);
  SFI_VCASE(1, 1) SFI_VCASE(2, 1) SFI_VCASE(2, 2)
  SFI_VCASE(4, 1) SFI_VCASE(4, 2) SFI_VCASE(4, 3) SFI_VCASE(4, 4)
  SFI_VCASE(8, 1) SFI_VCASE(8, 2) SFI_VCASE(8, 3) SFI_VCASE(8, 4)
#undef SFI_VCASE
  return cudaErrorInvalidValue;
}

}  // namespace sfi
