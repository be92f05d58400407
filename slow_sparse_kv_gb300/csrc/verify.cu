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
// For each (sequence, KV head) unit the kernel streams the cache once and
// serves all R = n_rows verify rows of the unit's G query heads: the R*G
// query vectors form one or two 16-row tensor-core tiles (QK and PV with
// mma.sync m16n8k16, bf16 operands, fp32 accumulation).  Consumer warps
// 0..3 own tile rows 0..15, warps 4..7 rows 16..31, each warp 16 cache rows of
// every stage.  Row t of the chain sits at position n - R + t and attends to
// [0, n - R + t] (causal tail).  Tile rows are ordered collected rows first,
// so the per-position sum over the collected rows and the group's heads is a
// reduction over the lanes of tile 0 only; it is written per KV head, in
// natural units (q.k / sqrt(d)), for the prefix positions [0, n - R).
#include <math.h>

#include "attn_kernel.cuh"

namespace sfi {

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
  static constexpr int CPS = NCW;  // both tiles read every stage
  static constexpr int SR = MW * 4;
  static constexpr int PW = 4;  // producer warps
  static constexpr int NT = (NCW + PW) * 32;
  static constexpr int STAGE_B = SR * ROWB;
  static constexpr size_t RED_B = size_t(NCW) * 16 * (D + 2) * 4;
  static constexpr int NS_FIT =
      int((227 * 1024 - 2048 - RED_B - (size_t(kMaxUnits) + 1) * 4) / (2 * size_t(SR) * ROWB));
  static constexpr int NS = NS_FIT > 6 ? 6 : NS_FIT;
  static_assert(NS >= 2, "verify pipeline does not fit");
  static constexpr size_t OFF_K = 0;
  static constexpr size_t OFF_V = OFF_K + size_t(NS) * STAGE_B;
  static constexpr size_t OFF_BAR = OFF_V + size_t(NS) * STAGE_B;
  static constexpr size_t OFF_RED = OFF_BAR + (2 * NS + 2 * kItemRing) * 8;
  static constexpr size_t OFF_MISC = OFF_RED + RED_B;
  // collected-row sums passed from tile 1 to tile 0: [stage parity][warp slot][16 rows]
  static constexpr size_t OFF_XCH = OFF_MISC + 128;
  static constexpr size_t OFF_UNITS = OFF_XCH + 2 * 4 * 16 * 4;
  static size_t smem_bytes(int n_units) { return OFF_UNITS + size_t(n_units + 1 + kRankWords) * 4; }
  static_assert(OFF_UNITS + (size_t(kMaxUnits) + 1 + kRankWords) * 4 <= size_t(227) * 1024,
                "shared memory plan exceeds 227 KB");
  static __device__ __forceinline__ uint32_t chunk_off(int r, int c) {
    return uint32_t((c >> 3) * (SR * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
  }
};

template <int D, int G>
__device__ __forceinline__ void verify_item(const VerifyArgs& va, const ItemInfo& I,
                                            unsigned char* smem, uint32_t bar_full,
                                            uint32_t bar_empty, volatile int* abort_flag,
                                            uint32_t& stage, int warp, int lane, float* red) {
  // Collected rows are tile rows [0, ncg): when they reach into tile 1, each
  // tile-1 warp hands its collected sums to the tile-0 warp of the same stage
  // rows through shared memory (a two-warp named barrier per stage, reached
  // by both warps on every stage).
  float* xch = reinterpret_cast<float*>(smem + VerifyCfg<D>::OFF_XCH);
  const bool xtile = va.lsum != nullptr && va.ncg > 16;
  using C = VerifyCfg<D>;
  const AttnArgs& a = va.base;
  constexpr int KS = D / 16;
  constexpr int NTD = D / 8;
  const int QR = va.R * G;
  const int g4 = lane >> 2, t4 = lane & 3;
  const int tile = warp >> 2, wslot = warp & 3;
  const int tile_rows = min(16, max(0, QR - 16 * tile));  // uniform over the warp
  const uint32_t kbase = smem_addr(smem + C::OFF_K), vbase = smem_addr(smem + C::OFF_V);

  // tile rows g4 and g4 + 8 of this warp: chain row t, head h, causal limit
  int lim[2];
  uint32_t qa[KS][4];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int qr = 16 * tile + g4 + 8 * hr;
    const bool real = qr < QR;
    const int t = real ? va.t_of_slot[qr / G] : 0;
    const int h = real ? qr % G : 0;
    lim[hr] = real ? I.n - va.R + t : 0x7fffffff;  // padding rows: unmasked, never written
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(a.q) +
                           (((size_t(I.b) * va.R + t) * a.H_q + size_t(I.g) * G + h) * D) / 2;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][hr] = real ? __ldg(qrow + ks * 8 + t4) : 0u;          // k 2t4..2t4+1
      qa[ks][2 + hr] = real ? __ldg(qrow + ks * 8 + 4 + t4) : 0u;  // k 8+2t4..9+2t4
    }
  }
  float acc[NTD][4];
#pragma unroll
  for (int c = 0; c < NTD; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, z[2] = {0.f, 0.f};
  const float qs = a.qscale;
  const int n_pre = I.n - va.R;

  for (int si = 0; si < I.n_st; ++si, ++stage) {
    const int c0 = I.c_first + si * I.c_step;
    const int nr = min(C::SR, I.rows - c0);
    const int slot = stage % C::NS;
    const uint32_t ph = (stage / C::NS) & 1u;
    const bool have = warp_pipe_wait(bar_full + 8 * slot, ph, abort_flag, a.status, a.wait_cycles);
    const int r0 = wslot * C::MW;
    const int nw = min(C::MW, nr - r0);
    float lsv[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    bool lvalid = false;
    if (have && nw > 0 && tile_rows > 0) {
      const uint32_t kst = kbase + slot * C::STAGE_B;
      const uint32_t vst = vbase + slot * C::STAGE_B;
      float sacc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
        const int row = r0 + nt * 8 + (lane & 7);
#pragma unroll
        for (int kp = 0; kp < KS / 2; ++kp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kst + C::chunk_off(row, kp * 4 + (lane >> 3)), b0, b1, b2, b3);
          const int k0 = 2 * kp, k1 = 2 * kp + 1;
          mma_bf16_16816(sacc[nt], qa[k0][0], qa[k0][1], qa[k0][2], qa[k0][3], b0, b1);
          mma_bf16_16816(sacc[nt], qa[k1][0], qa[k1][1], qa[k1][2], qa[k1][3], b2, b3);
        }
      }
      // collected logit sums of this tile's rows (lanes with g4 == 0 hold them)
      if (va.lsum) {
        const bool c_lo = 16 * tile + g4 < va.ncg, c_hi = 16 * tile + g4 + 8 < va.ncg;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float v = (c_lo ? sacc[nt][j] : 0.f) + (c_hi ? sacc[nt][2 + j] : 0.f);
            v += __shfl_xor_sync(kFull, v, 4);
            v += __shfl_xor_sync(kFull, v, 8);
            v += __shfl_xor_sync(kFull, v, 16);
            lsv[nt][j] = v;
          }
        lvalid = true;
      }
      // logits (log2 domain) of rows g4 (hr 0) and g4 + 8 (hr 1), masked
      float l[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int rr = nt * 8 + 2 * t4 + j;
          const int pos = c0 + r0 + rr;
#pragma unroll
          for (int hr = 0; hr < 2; ++hr)
            l[hr][nt * 2 + j] = (rr < nw && pos <= lim[hr]) ? sacc[nt][2 * hr + j] * qs : -INFINITY;
        }
      uint32_t pa[2][2];  // [hr][nt]
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float tmax = fmaxf(fmaxf(l[hr][0], l[hr][1]), fmaxf(l[hr][2], l[hr][3]));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 2));
        if (tmax > m[hr]) {
          const float al = exp2f(m[hr] - tmax);
#pragma unroll
          for (int c = 0; c < NTD; ++c) {
            acc[c][2 * hr] *= al;
            acc[c][2 * hr + 1] *= al;
          }
          z[hr] *= al;
          m[hr] = tmax;
        }
        float p[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // a row with every logit masked so far keeps m = -inf: its p is 0
          p[j] = l[hr][j] == -INFINITY ? 0.f : exp2f(l[hr][j] - m[hr]);
          z[hr] += p[j];
        }
        pa[hr][0] = pack_bf16x2(p[0], p[1]);
        pa[hr][1] = pack_bf16x2(p[2], p[3]);
      }
      uint32_t m_lo = 0xffffffffu, m_hi = 0xffffffffu;
      if (nw < C::MW) {
        m_lo = (2 * t4 < nw ? 0x0000ffffu : 0u) | (2 * t4 + 1 < nw ? 0xffff0000u : 0u);
        m_hi = (8 + 2 * t4 < nw ? 0x0000ffffu : 0u) | (9 + 2 * t4 < nw ? 0xffff0000u : 0u);
      }
      const int vrow = r0 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(vst + C::chunk_off(vrow, 2 * dp + (lane >> 4)), b0, b1, b2, b3);
        b0 &= m_lo;
        b1 &= m_hi;
        b2 &= m_lo;
        b3 &= m_hi;
        mma_bf16_16816(acc[2 * dp], pa[0][0], pa[1][0], pa[0][1], pa[1][1], b0, b1);
        mma_bf16_16816(acc[2 * dp + 1], pa[0][0], pa[1][0], pa[0][1], pa[1][1], b2, b3);
      }
    }
    if (xtile) {
      float* xb = xch + ((stage & 1u) * 4 + wslot) * 16;
      if (tile == 1 && g4 == 0) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) xb[nt * 8 + 2 * t4 + j] = lsv[nt][j];
      }
      named_bar_sync(2 + wslot, 64);
      if (tile == 0 && g4 == 0) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) lsv[nt][j] += xb[nt * 8 + 2 * t4 + j];
      }
    }
    if (lvalid && tile == 0 && g4 == 0) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int rr = nt * 8 + 2 * t4 + j;
          const int pos = c0 + r0 + rr;
          if (rr < nw && pos < n_pre) va.lsum[size_t(I.u) * a.max_len + pos] = lsv[nt][j] * va.lscale;
        }
    }
    // a stage given up on is released only once its rows have landed, so
    // no copy into the slot is still in flight when it is refilled
    if (!have) mbar_wait(bar_full + 8 * slot, ph);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    z[hr] += __shfl_xor_sync(kFull, z[hr], 1);
    z[hr] += __shfl_xor_sync(kFull, z[hr], 2);
    const int row = g4 + 8 * hr;  // tile row
    float* rw = red + row * (D + 2);
    if (t4 == 0) {
      rw[0] = m[hr];
      rw[1] = z[hr];
    }
#pragma unroll
    for (int c = 0; c < NTD; ++c) {
      rw[2 + 8 * c + 2 * t4] = acc[c][2 * hr];
      rw[2 + 8 * c + 2 * t4 + 1] = acc[c][2 * hr + 1];
    }
  }
}

template <int D, int G>
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
  // the CTA's first item id, fetched while the unit table is built
  unsigned first_id = 0;
  const bool fetcher = warp == C::NCW && lane == 0;
  if (fetcher) first_id = atomicAdd(a.work_ctr, 1u);
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
      mbar_init(ring.empty + 8 * s, C::PW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp >= C::NCW) {
    attn_produce<C>(a, units, n_units, total, smem, bar_full, bar_empty, ring, abort_flag,
                    warp - C::NCW, lane, first_id);
    return;
  }
  float* red_all = reinterpret_cast<float*>(smem + C::OFF_RED);
  const int nct = C::NCW * 32;
  const int QR = va.R * G;
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
    verify_item<D, G>(va, I, smem, bar_full, bar_empty, abort_flag, stage, warp, lane,
                      red_all + warp * 16 * (D + 2));
    named_bar_sync(1, nct);
    float* part = a.partials + size_t(it) * QR * (D + 2);
    const bool single = I.n_items == 1;
    for (int j = tid; j < QR * D; j += nct) {
      const int qr = j / D, dim = j % D;
      const int tile = qr >> 4, row = qr & 15;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) M = fmaxf(M, red_all[((tile * 4 + w) * 16 + row) * (D + 2)]);
      float A = 0.f, Z = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float* rw = red_all + ((tile * 4 + w) * 16 + row) * (D + 2);
        const float sc = rw[0] == -INFINITY ? 0.f : exp2f(rw[0] - M);
        Z = fmaf(rw[1], sc, Z);
        A = fmaf(rw[2 + dim], sc, A);
      }
      const int t = va.t_of_slot[qr / G], h = qr % G;
      const size_t oh = (size_t(I.b) * va.R + t) * a.H_q + size_t(I.g) * G + h;
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
        for (int j = tid; j < QR * D; j += nct) {
          const int qr = j / D, dim = j % D;
          const float* pbase = a.partials + (size_t(I.first) * QR + qr) * (D + 2);
          const size_t pstride = size_t(QR) * (D + 2);
          float M = -INFINITY;
          for (int i = 0; i < I.n_items; ++i) M = fmaxf(M, __ldcg(pbase + i * pstride));
          float A = 0.f, Z = 0.f;
#pragma unroll 4
          for (int i = 0; i < I.n_items; ++i) {
            const float* p = pbase + i * pstride;
            const float pm = __ldcg(p);
            const float sc = pm == -INFINITY ? 0.f : exp2f(pm - M);
            Z = fmaf(__ldcg(p + 1), sc, Z);
            A = fmaf(__ldcg(p + 2 + dim), sc, A);
          }
          const int t = va.t_of_slot[qr / G], h = qr % G;
          const size_t oh = (size_t(I.b) * va.R + t) * a.H_q + size_t(I.g) * G + h;
          a.out[oh * D + dim] = A / Z;
        }
        if (tid == 0) a.counters[I.u] = 0;
      }
    }
    named_bar_sync(1, nct);
  }
}

template <int D, int G>
cudaError_t launch_verify_t(const VerifyArgs& va, cudaStream_t st) {
  using C = VerifyCfg<D>;
  const size_t smem = C::smem_bytes(va.base.B * va.base.H_kv);
  cudaError_t e = cudaFuncSetAttribute(verify_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  verify_kernel<D, G><<<device_sm_count(), C::NT, smem, st>>>(va);
  return cudaGetLastError();
}

cudaError_t launch_verify(const VerifyArgs& va, int D, int G, cudaStream_t st) {
#define SFI_VCASE(DD, GG) \
  if (D == DD && G == GG) return launch_verify_t<DD, GG>(va, st);
  SFI_VCASE(64, 1) SFI_VCASE(64, 2) SFI_VCASE(64, 4) SFI_VCASE(64, 8)
  SFI_VCASE(128, 1) SFI_VCASE(128, 2) SFI_VCASE(128, 4) SFI_VCASE(128, 8)
#undef SFI_VCASE
  return cudaErrorInvalidValue;
}

int verify_stage_rows() { return VerifyCfg<128>::SR; }

}  // namespace sfi
