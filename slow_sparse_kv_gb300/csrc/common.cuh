// Device helpers shared by the libsfi kernels: mbarrier pipeline primitives,
// bulk asynchronous global->shared copies, bounded waits, bf16 unpacking and
// warp reductions.  sm_103a only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sfi_internal.h"

namespace sfi {

constexpr unsigned kFull = 0xffffffffu;
// Default limit of a pipeline wait, in SM clocks (about 2 s); a launch may
// set a shorter one for its consumers' data waits (AttnArgs::wait_cycles).
constexpr long long kWaitCycles = kDefaultWaitCycles;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of the same condition (mbarrier.test_wait never
// suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// Wait for the phase of parity `parity` to complete; false after `limit`
// SM clocks.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          long long limit = kWaitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// Data wait of a whole consumer warp (a stage's rows have landed).  Gives up
// when the CTA's abort flag is set or after `limit` SM clocks (then it sets
// the flag and the status bit).  The result is the same in every lane: true
// only if every lane saw the phase complete, so the warp never diverges
// around the data it guards.  A warp whose wait failed skips the stage's
// arithmetic but still releases the stage and walks the rest of the
// schedule, so the producers and the named barriers never wait for it.
// The first probe does not suspend, and the limit is checked before every
// suspending try, so a wait whose phase is not complete on entry runs out
// after `limit` clocks even when that is shorter than one suspension.
__device__ __forceinline__ bool warp_pipe_wait(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, uint32_t* status,
                                               long long limit) {
  bool ok = mbar_test_wait(bar, parity);
  if (!ok) {
    const long long t0 = clock64();
    while (true) {
      if (*abort_flag) break;
      if (clock64() - t0 > limit) {
        *abort_flag = 1;
        set_status(status, SFI_DEV_WAIT_TIMEOUT);
        break;
      }
      if (mbar_try_wait(bar, parity)) {
        ok = true;
        break;
      }
    }
  }
  return __all_sync(kFull, ok);
}

// Control wait of a whole warp: a free stage slot (producers) or a published
// work-item id.  These phases always complete, because the consumers release
// every stage of every item they walk (even after an abort), so the wait
// ignores the abort flag -- every warp of the CTA then walks the same items
// and stages, and no copy is left in flight when the CTA exits.  It still
// gives up after kWaitCycles (then it sets the abort flag and the status
// bit).
__device__ __forceinline__ bool warp_ctrl_wait(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, uint32_t* status) {
  bool ok = mbar_try_wait(bar, parity);
  if (!ok) {
    const long long t0 = clock64();
    while (true) {
      if (mbar_try_wait(bar, parity)) {
        ok = true;
        break;
      }
      if (clock64() - t0 > kWaitCycles) {
        *abort_flag = 1;
        set_status(status, SFI_DEV_WAIT_TIMEOUT);
        break;
      }
    }
  }
  return __all_sync(kFull, ok);
}

// Bulk asynchronous copy global -> shared of `bytes` (multiple of 16, both
// addresses 16-byte aligned); completion is counted on mbarrier `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// 16-byte asynchronous copy global -> shared through L2 only (cp.async.cg).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "l"(policy)
               : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed;
// the arrival counts toward the barrier's expected count (.noinc).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// 2-D tiled TMA load of one box of `tmap` at element coordinates (x, y) into
// shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policy for data read once per launch (KV rows): evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// ldmatrix: four 8x8 b16 matrices; lanes 8j..8j+7 give the row addresses of
// matrix j, register j receives this lane's two elements of matrix j.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A * B + D for one full m16n8k16 bf16 tile (fp32 accumulation):
// a0 = A[g][2t..], a1 = A[g + 8][2t..], a2 = A[g][2t + 8..], a3 = A[g + 8][2t + 8..];
// b0 = B[2t..][g], b1 = B[2t + 8..][g]; d = {D[g][2t], D[g][2t + 1], D[g + 8][2t], D[g + 8][2t + 1]}.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8 x 8 b16 matrix held one pair per lane (lane 4r + c holds
// row r, columns 2c and 2c + 1): afterwards the lane holds the transposed
// matrix's row r, i.e. the original's column r at rows 2c and 2c + 1.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(x));
  return d;
}

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 16 bytes of storage -> fp32 elements.
template <typename T>
struct Unpack;

template <>
struct Unpack<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void run(const uint4& v, float (&o)[4]) {
    o[0] = __uint_as_float(v.x);
    o[1] = __uint_as_float(v.y);
    o[2] = __uint_as_float(v.z);
    o[3] = __uint_as_float(v.w);
  }
};

struct bf16_t {
  uint16_t bits;
};

template <>
struct Unpack<bf16_t> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void run(const uint4& v, float (&o)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};


__device__ __forceinline__ bool seq_is_slow(const SeqMask& m, int b) {
  return (m.bits[b >> 5] >> (b & 31)) & 1u;
}

// Unsigned key with the order of the float x (larger x, larger key).
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The j-th sequence (in increasing order) whose bit is set in m, or -1.
__device__ __forceinline__ int active_seq(const SeqMask& m, int j) {
  for (int w = 0; w < kMaxBatch / 32; ++w) {
    uint32_t bits = m.bits[w];
    const int c = __popc(bits);
    if (j < c) {
      for (int i = 0; i < j; ++i) bits &= bits - 1;
      return 32 * w + __ffs(bits) - 1;
    }
    j -= c;
  }
  return -1;
}

// Cross-head exclusivity factor exp(-beta * c) of a position that c earlier
// KV heads of the sequence selected (1 when c = 0).
__device__ __forceinline__ float excl_factor(uint32_t c, float beta) {
  return c ? expf(-beta * float(c)) : 1.0f;
}

// Transpose-reduce across LPR lanes (LPR a power of two, lanes grouped by
// lane / LPR): on entry each lane holds V partial values; on exit v[0..NV)
// hold complete sums over the LPR lanes of the entries base .. base+NV-1,
// where NV = max(1, V / LPR).  Each level halves the entries a lane keeps
// and exchanges the other half with its partner, so V values are reduced
// with about V shuffles per lane instead of V * log2(LPR).
template <int C, int O>
struct TransposeReduce {
  template <int V>
  static __device__ __forceinline__ void run(float (&v)[V], int li, int& base) {
    if constexpr (O == 0) {
      return;
    } else if constexpr (C > 1) {
      constexpr int H = C / 2;
      const bool up = (li & O) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float send = up ? v[i] : v[i + H];
        const float keep = up ? v[i + H] : v[i];
        v[i] = keep + __shfl_xor_sync(kFull, send, O);
      }
      if (up) base += H;
      TransposeReduce<H, O / 2>::run(v, li, base);
    } else {
      v[0] += __shfl_xor_sync(kFull, v[0], O);
      TransposeReduce<1, O / 2>::run(v, li, base);
    }
  }
};

template <int LPR, int V>
__device__ __forceinline__ int transpose_reduce(float (&v)[V], int li) {
  int base = 0;
  TransposeReduce<V, LPR / 2>::run(v, li, base);
  return base;
}

}  // namespace sfi
