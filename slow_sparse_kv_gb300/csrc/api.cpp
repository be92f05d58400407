// C ABI of libsfi: host-side validation, workspace planning and kernel
// dispatch for the slow step, the selector and the fast step.  Every check
// happens before anything is enqueued; errors carry a thread-local message.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "sfi_internal.h"

namespace sfi {

cudaError_t launch_attn_f32(const AttnArgs& a, int D, int G, cudaStream_t st, bool pdl);
cudaError_t launch_attn_bf16(const AttnArgs& a, int D, int G, cudaStream_t st, bool pdl);
int attn_stage_rows_f32(int D);
int attn_stage_rows_bf16(int D);

namespace {
thread_local std::string g_err;
std::atomic<long long> g_wait_cycles{0};  // 0: kDefaultWaitCycles
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }
}  // namespace

sfi_status fail(sfi_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

sfi_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SFI_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

long long wait_limit_cycles() {
  const long long v = g_wait_cycles.load(std::memory_order_relaxed);
  return v > 0 ? v : kDefaultWaitCycles;
}

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

WsPlan plan_workspace(int B, int H_q, int H_kv, int D, int max_len) {
  (void)D;
  const int G = H_q / H_kv;
  const size_t units = size_t(B) * H_kv;
  WsPlan p{};
  p.max_items = int(units) * kItemSlotsPerUnit;
  size_t off = 0;
  p.status_off = off;
  off += 256;
  p.counters_off = off;
  off += align256((units + 2) * 4);  // merge counters + the two work-distribution counters
  p.partials_off = off;
  off += align256(size_t(p.max_items) * G * (D + 2) * 4);
  p.logits_off = off;
  off += align256(units * size_t(max_len) * G * 4);
  p.stats_off = off;
  off += align256(size_t(B) * H_q * 2 * 4);
  p.s_off = off;
  off += align256(units * size_t(max_len) * 4);
  p.sel_nu_off = off;
  off += align256(units * kSelMaxChunks * 4);
  p.sel_cnt_off = off;
  off += align256(units * kSelMaxChunks * 2 * 4);
  p.sel_hist_off = off;
  off += align256(units * kSelHistWords * 4);
  p.sel_ctr_off = off;
  off += align256(units * 4 * 4);
  p.sel_keys_off = off;
  off += align256(units * size_t(max_len) * 4);
  p.sel_cand_off = off;
  off += align256(std::min(units, size_t(kSelCandRows)) * size_t(max_len) * 8);
  p.total = off;
  return p;
}

void attach_select_scratch(SelectArgs& a, char* ws, const WsPlan& p) {
  a.sel_nu = reinterpret_cast<float*>(ws + p.sel_nu_off);
  a.sel_cnt = reinterpret_cast<uint32_t*>(ws + p.sel_cnt_off);
  a.sel_hist = reinterpret_cast<uint32_t*>(ws + p.sel_hist_off);
  a.sel_ctr = reinterpret_cast<uint32_t*>(ws + p.sel_ctr_off);
  a.sel_keys = reinterpret_cast<uint32_t*>(ws + p.sel_keys_off);
  a.sel_cand = reinterpret_cast<unsigned long long*>(ws + p.sel_cand_off);
}

sfi_status check_layout(const sfi_layout* L) {
  if (!L) return fail(SFI_ERR_INVALID_ARG, "layout is NULL");
  if (L->batch < 1) return fail(SFI_ERR_INVALID_ARG, "batch must be >= 1 (got %d)", L->batch);
  if (L->batch > kMaxBatch)
    return fail(SFI_ERR_CAPACITY, "batch %d exceeds the limit %d", L->batch, kMaxBatch);
  if (L->n_kv_heads < 1 || L->n_q_heads < 1 || L->n_q_heads % L->n_kv_heads != 0)
    return fail(SFI_ERR_INVALID_ARG, "n_q_heads (%d) must be a positive multiple of n_kv_heads (%d)",
                L->n_q_heads, L->n_kv_heads);
  const int G = L->n_q_heads / L->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(SFI_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4 or 8 (got %d)", G);
  if (L->head_dim != 64 && L->head_dim != 128)
    return fail(SFI_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", L->head_dim);
  if (L->dtype != SFI_F32 && L->dtype != SFI_BF16)
    return fail(SFI_ERR_UNSUPPORTED, "dtype must be SFI_F32 or SFI_BF16 (got %d)", L->dtype);
  if (L->max_len < 1) return fail(SFI_ERR_INVALID_ARG, "max_len must be >= 1 (got %d)", L->max_len);
  if (size_t(L->batch) * L->n_kv_heads > size_t(kMaxUnits))
    return fail(SFI_ERR_CAPACITY, "batch * n_kv_heads = %d exceeds the limit %d",
                L->batch * L->n_kv_heads, kMaxUnits);
  if (!L->kv_offset || !L->kv_cap || !L->len)
    return fail(SFI_ERR_INVALID_ARG, "layout kv_offset, kv_cap and len must be device pointers");
  return SFI_OK;
}

sfi_status check_params(const sfi_params* P, bool for_select) {
  if (!P) return fail(SFI_ERR_INVALID_ARG, "params is NULL");
  if (P->k < 1) return fail(SFI_ERR_INVALID_ARG, "k must be >= 1 (got %d)", P->k);
  if (P->n_sink < 0 || P->window < 0)
    return fail(SFI_ERR_INVALID_ARG, "n_sink and window must be >= 0 (got %d, %d)", P->n_sink,
                P->window);
  if (!(P->lambda >= 0.f && P->lambda <= 1.f))
    return fail(SFI_ERR_INVALID_ARG, "lambda must lie in [0, 1] (got %g)", double(P->lambda));
  if (P->mode != SFI_SELECT_FUSED && P->mode != SFI_SELECT_LOGIT_SUM_SEQ &&
      P->mode != SFI_SELECT_LOGIT_SUM_HEAD)
    return fail(SFI_ERR_INVALID_ARG, "unknown selection mode %d", P->mode);
  if (for_select && P->mode != SFI_SELECT_FUSED && (P->lambda != 0.f || P->n_sink != 0))
    return fail(SFI_ERR_INVALID_ARG, "logit-sum selection takes lambda = 0 and n_sink = 0");
  if (!for_select && P->n_sink + (long long)P->window < 1)
    return fail(SFI_ERR_INVALID_ARG,
                "n_sink + window must be >= 1 so every fast step attends to at least one row");
  return SFI_OK;
}

sfi_status check_ws(const sfi_layout* L, void* ws, size_t ws_bytes) {
  const WsPlan p = plan_workspace(L->batch, L->n_q_heads, L->n_kv_heads, L->head_dim, L->max_len);
  if (!ws) return fail(SFI_ERR_WORKSPACE, "workspace is NULL");
  if (ws_bytes < p.total)
    return fail(SFI_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu required",
                ws_bytes, p.total);
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0)
    return fail(SFI_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  return SFI_OK;
}

int stage_rows(int dtype, int D) {
  return dtype == SFI_F32 ? attn_stage_rows_f32(D) : attn_stage_rows_bf16(D);
}

namespace {

// Length of a launch, in stage times of a CTA streaming at its fair share of
// HBM, when `grid` CTAs take items in order: n_a units of rows_a rows split
// into ceil(rows_a / rpi_a) items each, then n_b units of rows_b rows split
// by rpi_b.  List scheduling over the CTAs' free times; each item costs its
// stages (a class-a stage weighted w_a / 10) plus kItemCost (its start,
// epilogue and share of the merge of split units).  Once the last item is taken, the CTAs still busy
// share HBM among fewer streams and speed up to at most `cap` times their
// fair share: their own pipeline bounds them (measured: ~1.5 for plain
// attention, ~1.0 when slow units also write their logits and key norms,
// which holds each stage longer).
double simulate_launch(long long n_a, int rows_a, long long rpi_a, long long n_b, int rows_b,
                       long long rpi_b, int sr, int grid, double cap, int w_a) {
  // times in tenths of a plain stage: a stage of class b costs 10, one of
  // class a w_a, an item's fixed cost 3 stages
  constexpr long long kItemCost = 30;
  const long long w[2] = {w_a, 10};
  // Item costs are integers, so the CTAs' free times are integers: free[t]
  // counts the CTAs free at time t, and the earliest free time only grows as
  // items are handed out.
  long long horizon = 1;
  for (int cls = 0; cls < 2; ++cls) {
    const long long n = cls == 0 ? n_a : n_b;
    const int rows = cls == 0 ? rows_a : rows_b;
    const long long rpi = cls == 0 ? rpi_a : rpi_b;
    if (n > 0 && rows > 0) horizon += n * (ceil_div(rows, sr) * w[cls] + ceil_div(rows, rpi) * kItemCost);
  }
  horizon = horizon / grid + 2 * (ceil_div(std::max(rows_a, rows_b), sr) * std::max(w[0], w[1]) + kItemCost) + 2;
  std::vector<int> free_at(size_t(horizon), 0);
  free_at[0] = grid;
  long long t_min = 0;
  for (int cls = 0; cls < 2; ++cls) {
    const long long n = cls == 0 ? n_a : n_b;
    const int rows = cls == 0 ? rows_a : rows_b;
    const long long rpi = cls == 0 ? rpi_a : rpi_b;
    if (n <= 0 || rows <= 0) continue;
    // k items per unit share the unit's S stages cyclically: S % k items
    // of S / k + 1 stages, then the rest of S / k
    const long long k = ceil_div(rows, rpi), S = ceil_div(rows, sr);
    const long long q = S / k, r = S % k;
    for (long long u = 0; u < n; ++u)
      for (long long i = 0; i < k; ++i) {
        while (free_at[size_t(t_min)] == 0) ++t_min;
        --free_at[size_t(t_min)];
        ++free_at[size_t(t_min + (q + (i < r ? 1 : 0)) * w[cls] + kItemCost)];
      }
  }
  // the tail: remaining work of every CTA after the last item was taken at
  // t_min, shortest first
  double t = double(t_min), done = 0.0;
  int active = grid;
  for (long long x = t_min; x < horizon && active > 0; ++x)
    for (int c = free_at[size_t(x)]; c > 0; --c) {
      const double rem = double(x - t_min);
      if (rem > done) {
        t += (rem - done) / std::min(double(grid) / active, cap);
        done = rem;
      }
      --active;
    }
  return t / 10.0;
}

struct SplitKey {
  long long n_a, n_b;
  int rows_a, rows_b, sr, grid;
  bool emit;
  bool operator==(const SplitKey& o) const {
    return n_a == o.n_a && n_b == o.n_b && rows_a == o.rows_a && rows_b == o.rows_b &&
           sr == o.sr && grid == o.grid && emit == o.emit;
  }
};

// Candidate rows per item splitting `rows` into 1..kmax even items (at least
// min_rpi rows each), distinct.
std::vector<long long> split_candidates(int rows, int kmax, long long min_rpi, int sr) {
  std::vector<long long> c;
  for (int k = 1; k <= kmax; ++k) {
    const long long rpi = std::max(min_rpi, ceil_div(ceil_div(rows, k), sr) * sr);
    if (std::find(c.begin(), c.end(), rpi) == c.end()) c.push_back(rpi);
  }
  return c;
}

}  // namespace

// Item sizes for a launch whose units come in two classes (n_a units of at
// most rows_a rows, taken first, then n_b of at most rows_b): the pair of
// splits -- each class into 1..kItemSlotsPerUnit even items (the workspace
// holds that many partials per unit), the second class into at most 16 --
// with the shortest simulated launch, among those that give every CTA an
// item when any does and the launch is long.  Results are cached per launch shape;
// a decode loop meets only a handful of shapes.
ItemSplit choose_item_split(long long n_a, int rows_a, long long n_b, int rows_b, int sr, int grid,
                            bool emit) {
  if (n_a <= 0 || rows_a <= 0) n_a = 0, rows_a = 0;
  if (n_b <= 0 || rows_b <= 0) n_b = 0, rows_b = 0;
  const SplitKey key{n_a, n_b, rows_a, rows_b, sr, grid, emit};
  const double cap = emit ? 1.0 : 1.5;
  // a stage of a unit that also writes its logits and key norms holds the
  // CTA ~1.5x as long as a plain one (measured per-stage warp times)
  const int w_a = emit ? 15 : 10;
  static std::mutex mu;
  static std::vector<std::pair<SplitKey, ItemSplit>> cache;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const auto& e : cache)
      if (e.first == key) return e.second;
  }
  auto min_rpi = [&](int rows) {
    return std::max<long long>(sr, ceil_div(ceil_div(rows, kItemSlotsPerUnit), sr) * sr);
  };
  const std::vector<long long> ca =
      n_a ? split_candidates(rows_a, kItemSlotsPerUnit, min_rpi(rows_a), sr) : std::vector<long long>{sr};
  const std::vector<long long> cb =
      n_b ? split_candidates(rows_b, 16, min_rpi(rows_b), sr) : std::vector<long long>{sr};
  // In long launches fewer streams than SMs cost more than the tail model
  // shows (measured on dense launches): every CTA gets an item when a split
  // allows it.
  auto items_of = [&](long long ra, long long rb) {
    return (n_a ? n_a * ceil_div(rows_a, ra) : 0) + (n_b ? n_b * ceil_div(rows_b, rb) : 0);
  };
  const double stages = double(n_a) * ceil_div(rows_a, sr) + double(n_b) * ceil_div(rows_b, sr);
  const bool can_fill = stages >= 64.0 * grid && items_of(ca.back(), cb.back()) >= grid;
  ItemSplit best{int(ca.back()), int(cb.back())};
  double best_cost = 1e300;
  for (long long ra : ca)
    for (long long rb : cb) {
      if (can_fill && items_of(ra, rb) < grid) continue;
      const double cost = simulate_launch(n_a, rows_a, ra, n_b, rows_b, rb, sr, grid, cap, w_a);
      if (cost < best_cost) {
        best_cost = cost;
        best = ItemSplit{int(ra), int(rb)};
      }
    }
  std::lock_guard<std::mutex> lk(mu);
  if (cache.size() >= 256) cache.clear();
  cache.emplace_back(key, best);
  return best;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// K (or V) as a 2-D tensor of bf16 rows: dim 0 = D elements, dim 1 = rows.
// The row extent is the largest the descriptor allows; the kernel only ever
// asks for full 64-row boxes that lie inside a (sequence, KV head) slab.
bool encode_rows(CUtensorMap* m, const void* base, int D) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(1) << 31};
  const cuuint64_t strides[1] = {cuuint64_t(D) * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

void attach_tensor_maps(AttnArgs& a, const sfi_layout* L) {
  a.use_tma = 0;
  if (L->dtype != SFI_BF16) return;
  if (reinterpret_cast<uintptr_t>(a.k) % 16 || reinterpret_cast<uintptr_t>(a.v) % 16) return;
  if (encode_rows(&a.tmk, a.k, L->head_dim) && encode_rows(&a.tmv, a.v, L->head_dim)) a.use_tma = 1;
}

void fill_attn_common(AttnArgs& a, const sfi_layout* L, const void* q, const void* k,
                      const void* v, float* out, char* ws, const WsPlan& p) {
  std::memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.kv_offset = L->kv_offset;
  a.kv_cap = L->kv_cap;
  a.len = L->len;
  a.out = out;
  a.B = L->batch;
  a.H_q = L->n_q_heads;
  a.H_kv = L->n_kv_heads;
  a.max_len = L->max_len;
  a.max_items = p.max_items;
  a.qscale = float(1.4426950408889634 / std::sqrt(double(L->head_dim)));
  a.partials = reinterpret_cast<float*>(ws + p.partials_off);
  a.counters = reinterpret_cast<int32_t*>(ws + p.counters_off);
  a.work_ctr = reinterpret_cast<uint32_t*>(a.counters + size_t(L->batch) * L->n_kv_heads);
  a.status = reinterpret_cast<uint32_t*>(ws + p.status_off);
  a.wait_cycles = wait_limit_cycles();
  a.logits = reinterpret_cast<float*>(ws + p.logits_off);
  a.stats = reinterpret_cast<float*>(ws + p.stats_off);
  attach_tensor_maps(a, L);
}

sfi_status run_attn(AttnArgs& a, const sfi_layout* L, long long n_slow_units, int slow_rows,
                    long long n_fast_units, int fast_rows, cudaStream_t st, bool pdl) {
  const int G = L->n_q_heads / L->n_kv_heads;
  const ItemSplit sp = choose_item_split(n_slow_units, slow_rows, n_fast_units, fast_rows,
                                        stage_rows(L->dtype, L->head_dim), device_sm_count(),
                                        a.emit != 0 && n_slow_units > 0);
  a.rpi_slow = sp.rpi_a;
  a.rpi_fast = sp.rpi_b;
  // fast units only: every unit gets the items of the row bound, and the
  // kernel maps item ids to units without a unit table
  a.fast_items = n_slow_units == 0 && n_fast_units > 0 && fast_rows > 0
                     ? int((fast_rows + sp.rpi_b - 1) / sp.rpi_b)
                     : 0;
  const cudaError_t e = L->dtype == SFI_F32 ? launch_attn_f32(a, L->head_dim, G, st, pdl)
                                            : launch_attn_bf16(a, L->head_dim, G, st, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return SFI_OK;
}

int fast_unit_rows_bound(const sfi_layout* L, const sfi_params* P) {
  long long r = (long long)P->n_sink + P->k + P->window;
  return int(r < L->max_len ? r : L->max_len);
}

}  // namespace sfi

using namespace sfi;

extern "C" {

const char* sfi_last_error(void) { return sfi::g_err.c_str(); }

int32_t sfi_device_sm_count(void) { return device_sm_count(); }

sfi_status sfi_set_wait_limit(int64_t cycles) {
  if (cycles < 0) return fail(SFI_ERR_INVALID_ARG, "wait limit must be >= 0 (got %lld)", (long long)cycles);
  g_wait_cycles.store(cycles, std::memory_order_relaxed);
  return SFI_OK;
}

sfi_status sfi_read_status(void* ws, uint32_t* status_host, sfi_stream stream) {
  if (!ws || !status_host) return fail(SFI_ERR_INVALID_ARG, "workspace and status_host must be set");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(status_host, ws, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, 4, st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
  return SFI_OK;
}

size_t sfi_slow_attn_workspace_size(const sfi_layout* L) {
  if (check_layout(L) != SFI_OK) return 0;
  return plan_workspace(L->batch, L->n_q_heads, L->n_kv_heads, L->head_dim, L->max_len).total;
}

size_t sfi_select_workspace_size(const sfi_layout* L, const sfi_params* P) {
  (void)P;
  return sfi_slow_attn_workspace_size(L);
}

size_t sfi_fast_attn_workspace_size(const sfi_layout* L, const sfi_params* P) {
  (void)P;
  return sfi_slow_attn_workspace_size(L);
}

sfi_status sfi_slow_attn(const sfi_layout* L, const void* q, const void* k, const void* v,
                         float* out, float* f_out, float* knorm_out, void* ws, size_t ws_bytes,
                         sfi_stream stream) {
  sfi_status s = check_layout(L);
  if (s != SFI_OK) return s;
  if (!q || !k || !v || !out) return fail(SFI_ERR_INVALID_ARG, "q, k, v and out must be set");
  if ((s = check_ws(L, ws, ws_bytes)) != SFI_OK) return s;
  const WsPlan p = plan_workspace(L->batch, L->n_q_heads, L->n_kv_heads, L->head_dim, L->max_len);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  AttnArgs a;
  fill_attn_common(a, L, q, k, v, out, static_cast<char*>(ws), p);
  for (int b = 0; b < L->batch; ++b) a.slow.bits[b >> 5] |= 1u << (b & 31);
  a.emit = (f_out || knorm_out) ? 1 : 0;
  a.knorm = knorm_out;
  if ((s = run_attn(a, L, (long long)L->batch * L->n_kv_heads, L->max_len, 0, 0, st)) != SFI_OK)
    return s;
  if (f_out) {
    FpassArgs fa{};
    fa.logits = a.logits;
    fa.stats = a.stats;
    fa.len = L->len;
    fa.f = f_out;
    fa.B = L->batch;
    fa.H_q = L->n_q_heads;
    fa.H_kv = L->n_kv_heads;
    fa.max_len = L->max_len;
    fa.slow = a.slow;
    fa.status = a.status;
    const cudaError_t e = launch_fpass(fa, st);
    if (e != cudaSuccess) return cuda_fail(e, "evidence pass launch");
  }
  return SFI_OK;
}

sfi_status sfi_select(const sfi_layout* L, const sfi_params* P, const float* evidence,
                      const float* knorm, int32_t* idx_out, int32_t* count_out, float* s_out,
                      void* ws, size_t ws_bytes, sfi_stream stream) {
  sfi_status s = check_layout(L);
  if (s != SFI_OK) return s;
  if ((s = check_params(P, true)) != SFI_OK) return s;
  if (!evidence || !idx_out || !count_out)
    return fail(SFI_ERR_INVALID_ARG, "evidence, idx_out and count_out must be set");
  if (P->mode == SFI_SELECT_FUSED && !knorm)
    return fail(SFI_ERR_INVALID_ARG, "fused selection needs the key norms");
  if ((s = check_ws(L, ws, ws_bytes)) != SFI_OK) return s;
  if (L->max_len > kSelectMaxLen)
    return fail(SFI_ERR_CAPACITY, "the selector holds at most %d positions per row (max_len %d)",
                kSelectMaxLen, L->max_len);
  const WsPlan p = plan_workspace(L->batch, L->n_q_heads, L->n_kv_heads, L->head_dim, L->max_len);
  char* w = static_cast<char*>(ws);
  SelectArgs a{};
  a.evidence = evidence;
  a.knorm = knorm;
  a.H_q = L->n_q_heads;
  a.len = L->len;
  a.idx = idx_out;
  a.count = count_out;
  a.s = s_out;
  a.B = L->batch;
  a.H_kv = L->n_kv_heads;
  a.max_len = L->max_len;
  a.n_sink = P->n_sink;
  a.window = P->window;
  a.k = P->k;
  a.lambda = P->lambda;
  a.mode = P->mode;
  a.g_only = -1;
  for (int b = 0; b < L->batch; ++b) a.active.bits[b >> 5] |= 1u << (b & 31);
  a.status = reinterpret_cast<uint32_t*>(w + p.status_off);
  attach_select_scratch(a, w, p);
  const cudaError_t e = launch_select(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "selector launch");
  return SFI_OK;
}

sfi_status sfi_fast_attn(const sfi_layout* L, const sfi_params* P, const void* q, const void* k,
                         const void* v, const int32_t* idx, const int32_t* count, float* out,
                         void* ws, size_t ws_bytes, sfi_stream stream) {
  sfi_status s = check_layout(L);
  if (s != SFI_OK) return s;
  if ((s = check_params(P, false)) != SFI_OK) return s;
  if (!q || !k || !v || !out || !idx || !count)
    return fail(SFI_ERR_INVALID_ARG, "q, k, v, idx, count and out must be set");
  if ((s = check_ws(L, ws, ws_bytes)) != SFI_OK) return s;
  const WsPlan p = plan_workspace(L->batch, L->n_q_heads, L->n_kv_heads, L->head_dim, L->max_len);
  AttnArgs a;
  fill_attn_common(a, L, q, k, v, out, static_cast<char*>(ws), p);
  a.idx = idx;
  a.count = count;
  a.idx_stride = P->k;
  a.n_sink = P->n_sink;
  a.window = P->window;
  const int bound = fast_unit_rows_bound(L, P);
  return run_attn(a, L, 0, 0, (long long)L->batch * L->n_kv_heads, bound,
                  static_cast<cudaStream_t>(stream));
}

size_t sfi_verify_attn_workspace_size(const sfi_layout* L, int32_t n_rows) {
  if (check_layout(L) != SFI_OK || n_rows < 1 || n_rows > 8) return 0;
  return plan_workspace(L->batch, L->n_kv_heads * n_rows * (L->n_q_heads / L->n_kv_heads),
                        L->n_kv_heads, L->head_dim, L->max_len)
      .total;
}

sfi_status sfi_verify_attn(const sfi_layout* L, int32_t n_rows, const int32_t* collect_rows,
                           int32_t n_collect, const void* q, const void* k, const void* v,
                           float* out, float* logitsum_out, void* ws, size_t ws_bytes,
                           sfi_stream stream) {
  sfi_status s = check_layout(L);
  if (s != SFI_OK) return s;
  if (!q || !k || !v || !out) return fail(SFI_ERR_INVALID_ARG, "q, k, v and out must be set");
  if (L->dtype != SFI_BF16) return fail(SFI_ERR_UNSUPPORTED, "verify attention takes bf16 caches");
  const int G = L->n_q_heads / L->n_kv_heads;
  if (n_rows < 1 || n_rows > 8 || n_rows * G > 32)
    return fail(SFI_ERR_UNSUPPORTED, "verify rows: need 1 <= n_rows <= 8 and n_rows * G <= 32 (got %d, G %d)",
                n_rows, G);
  int8_t order[8];
  int n_ord = 0;
  bool used[8] = {false, false, false, false, false, false, false, false};
  if (logitsum_out) {
    if (n_collect < 0 || n_collect > n_rows || (n_collect > 0 && !collect_rows))
      return fail(SFI_ERR_INVALID_ARG, "collect_rows must list 0..n_rows distinct rows");
    for (int i = 0; i < n_collect; ++i) {
      const int t = collect_rows[i];
      if (t < 0 || t >= n_rows || used[t])
        return fail(SFI_ERR_INVALID_ARG, "collect row %d invalid or repeated", t);
      used[t] = true;
      order[n_ord++] = int8_t(t);
    }
  } else {
    n_collect = 0;
  }
  for (int t = 0; t < n_rows; ++t)
    if (!used[t]) order[n_ord++] = int8_t(t);
  const int QR = n_rows * G;
  const WsPlan p = plan_workspace(L->batch, L->n_kv_heads * QR, L->n_kv_heads, L->head_dim, L->max_len);
  if (!ws) return fail(SFI_ERR_WORKSPACE, "workspace is NULL");
  if (ws_bytes < p.total)
    return fail(SFI_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu required",
                ws_bytes, p.total);
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0)
    return fail(SFI_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  VerifyArgs va;
  std::memset(&va, 0, sizeof(va));
  fill_attn_common(va.base, L, q, k, v, out, static_cast<char*>(ws), p);
  for (int b = 0; b < L->batch; ++b) va.base.slow.bits[b >> 5] |= 1u << (b & 31);
  va.base.rpi_slow = va.base.rpi_fast =
      // (measured: finer items -- 19 per unit at batch 4 x 65541 rows, 4 per
      // CTA, instead of 8 -- were 25% slower: a split verify item is merged
      // from R * G partial rows, which costs more than the idle tail saved)
      choose_item_split((long long)L->batch * L->n_kv_heads, L->max_len, 0, 0, verify_stage_rows(),
                        device_sm_count(), false).rpi_a;
  va.R = n_rows;
  va.ncg = n_collect * G;
  for (int i = 0; i < n_ord; ++i) va.t_of_slot[i] = order[i];
  va.lsum = logitsum_out;
  va.lscale = float(1.0 / std::sqrt(double(L->head_dim)));
  const cudaError_t e = launch_verify(va, L->head_dim, G, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "verify attention launch");
  return SFI_OK;
}

}  // extern "C"
