// Fast step without any allocation: sfi_fast_attn_noalloc.
//
// Some callers cannot hand the library a workspace or call cudaMalloc on
// the path that runs this step: a plug-in interface that passes in only the
// inputs and outputs, or a serving loop that promised to allocate nothing
// after start-up because cudaMalloc can synchronise the whole device.  This
// entry point runs the same fast-step kernel as sfi_fast_attn, but its
// scratch (the status word, one merge counter per (sequence, KV head) and
// the split-K partial results) lives in one file-scope device array of fixed
// size, kNoAllocScratchBytes, that every GPU loading the library keeps until
// the process exits.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "sfi_internal.h"

namespace sfi {

cudaError_t launch_attn_f32(const AttnArgs& a, int D, int G, cudaStream_t st, bool pdl);
cudaError_t launch_attn_bf16(const AttnArgs& a, int D, int G, cudaStream_t st, bool pdl);
int attn_stage_rows_f32(int D);
int attn_stage_rows_bf16(int D);

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr size_t kHeaderBytes = 256;                       // status word
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code `g_noalloc_scratch` is only a stand-in
// for the symbol, never a device address: the address comes from
// cudaGetSymbolAddress, taken once per device.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {nullptr};

sfi_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SFI_ERR_CAPACITY, "device index %d too large", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the no-alloc scratch");
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return SFI_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace sfi

using namespace sfi;

extern "C" sfi_status sfi_fast_attn_noalloc(const sfi_layout* L, const sfi_params* P, const void* q,
                                            const void* k, const void* v, const int32_t* idx,
                                            const int32_t* count, float* out, sfi_stream stream) {
  sfi_status s = check_layout(L);
  if (s != SFI_OK) return s;
  if ((s = check_params(P, false)) != SFI_OK) return s;
  if (!q || !k || !v || !out || !idx || !count)
    return fail(SFI_ERR_INVALID_ARG, "q, k, v, idx, count and out must be set");
  const int G = L->n_q_heads / L->n_kv_heads;
  const long long units = (long long)L->batch * L->n_kv_heads;
  const size_t counters_bytes = round256(size_t(units + 2) * 4);  // + work-distribution counters
  const size_t item_bytes = size_t(G) * (L->head_dim + 2) * 4;
  const size_t avail = kNoAllocScratchBytes - kHeaderBytes - counters_bytes;
  const long long max_items = (long long)(avail / item_bytes);
  if (max_items < units)
    return fail(SFI_ERR_CAPACITY,
                "sfi_fast_attn_noalloc: %lld (sequence, KV head) units need %zu bytes of scratch; "
                "the fixed scratch holds %zu",
                units, size_t(units) * item_bytes + counters_bytes + kHeaderBytes,
                kNoAllocScratchBytes);
  // Work items.  A unit's rows never exceed n_sink + k + window (the
  // selected count is clamped to k and the window to the length), so sizing
  // on that bound -- not on max_len -- keeps every unit within its share.
  // The share is at most kItemSlotsPerUnit items: the merge of a split unit
  // holds that many partial results.  Both limits are checked here, before
  // the launch, so the kernel never meets a unit it cannot merge.
  const long long bound = std::max<long long>(
      1, (long long)P->n_sink + (long long)P->k + (long long)P->window);
  const int sr = L->dtype == SFI_F32 ? attn_stage_rows_f32(L->head_dim)
                                     : attn_stage_rows_bf16(L->head_dim);
  const long long per_unit = std::min<long long>(max_items / units, kItemSlotsPerUnit);
  long long rpi = (bound + per_unit - 1) / per_unit;
  const long long grid = device_sm_count();
  const long long balanced = (units * bound + grid - 1) / grid;
  if (rpi < balanced) rpi = balanced;
  rpi = (rpi + sr - 1) / sr * sr;
  if (rpi > 0x7fffffffLL) rpi = 0x7fffffffLL / sr * sr;
  const long long items_per_unit = (bound + rpi - 1) / rpi;
  if (items_per_unit > kItemSlotsPerUnit || items_per_unit * units > max_items)
    return fail(SFI_ERR_CAPACITY,
                "sfi_fast_attn_noalloc: %lld work items per unit for %lld units exceed the "
                "fixed scratch (%lld items, at most %d per unit)",
                items_per_unit, units, max_items, kItemSlotsPerUnit);
  void* base = nullptr;
  if ((s = scratch_address(&base)) != SFI_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the status word and the
  // merge counters must start at zero.
  cudaError_t e = cudaMemsetAsync(base, 0, kHeaderBytes + counters_bytes, st);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the no-alloc scratch");

  AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  char* w = static_cast<char*>(base);
  a.q = q;
  a.k = k;
  a.v = v;
  a.kv_offset = L->kv_offset;
  a.kv_cap = L->kv_cap;
  a.len = L->len;
  a.out = out;
  a.idx = idx;
  a.count = count;
  a.idx_stride = P->k;
  a.n_sink = P->n_sink;
  a.window = P->window;
  a.B = L->batch;
  a.H_q = L->n_q_heads;
  a.H_kv = L->n_kv_heads;
  a.max_len = L->max_len;
  a.qscale = float(1.4426950408889634 / std::sqrt(double(L->head_dim)));
  a.status = reinterpret_cast<uint32_t*>(w);
  a.wait_cycles = wait_limit_cycles();
  a.counters = reinterpret_cast<int32_t*>(w + kHeaderBytes);
  a.work_ctr = reinterpret_cast<uint32_t*>(a.counters + units);
  a.partials = reinterpret_cast<float*>(w + kHeaderBytes + counters_bytes);
  a.max_items = int(max_items < 0x7fffffff ? max_items : 0x7fffffff);
  a.rpi_slow = a.rpi_fast = int(rpi);
  a.fast_items = int(items_per_unit);
  e = L->dtype == SFI_F32 ? launch_attn_f32(a, L->head_dim, G, st, true)
                          : launch_attn_bf16(a, L->head_dim, G, st, true);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return SFI_OK;
}
