// Decode driver of libsfi (sfi_decode_step): the slow/fast schedule of the
// SFI pages ("Slow-Fast paradigm": a slow step near a semantic boundary or
// when the reuse budget is exhausted, fast steps otherwise) on top of the
// attention, evidence and selector kernels.  One context serves every layer
// of a model: each layer keeps its own selection; the decision is taken once
// per token (at layer 0) and shared by all layers.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "refine.h"
#include "sfi_internal.h"

// Overlapped selection (desc.async_select != 0): the selector of layer l runs
// on a high-priority side stream while the caller's stream goes on to layer
// l + 1.  The buffers the selector reads (logits and statistics in the
// workspace, key norms, a copy of len) come in two sets, used by layers of
// even and odd index; a launch that rewrites set p first waits for the last
// selector that read it (event sel_done[p]), which on the in-order side
// stream also orders every earlier selector, including the one that wrote
// the selection the launch reads.  At the last layer the caller's stream
// joins the side stream, so a token's work is complete when the step of its
// last layer is.
struct sfi_ctx {
  sfi_ctx_desc desc;
  sfi::WsPlan plan;
  // device, per buffer set
  char* ws[2] = {nullptr, nullptr};        // attention / selector workspace
  int32_t* len_copy[2] = {nullptr, nullptr};  // [B]
  // Key norms of every layer's cache rows, kept across steps: a cache row
  // never changes, so a refresh computes only the norms of the rows appended
  // since the layer's last refresh (knorm_valid[layer][u] rows are stored).
  float* knorm = nullptr;          // [L][B*H_kv][max_len]
  int32_t* knorm_valid = nullptr;  // [L][B*H_kv]
  // selector refinements (desc.refine): candidate lists, their counts and the
  // exclusivity counts, per buffer set
  bool refine = false;
  long long n_cand = 0;
  int32_t* cand[2] = {nullptr, nullptr};    // [B*H_kv][n_cand]
  int32_t* ccount[2] = {nullptr, nullptr};  // [B*H_kv]
  uint8_t* excl[2] = {nullptr, nullptr};    // [B][max_len]
  int32_t* idx = nullptr;      // [L][B*H_kv][k]
  int32_t* count = nullptr;    // [L][B*H_kv]
  int n_sets = 1;
  bool sel_in_flight = false;  // the last layer step sent its selector to the side stream
  cudaStream_t side = nullptr;
  cudaEvent_t attn_done[2] = {nullptr, nullptr}, sel_done[2] = {nullptr, nullptr};
  // host schedule state
  std::vector<uint8_t> have_sel, slow;
  std::vector<int32_t> since;
  bool decided = false;
  // profiling: rings of event pairs, flushed into the totals when full
  bool profiling = false;
  std::vector<cudaEvent_t> ev_attn, ev_sel;
  size_t n_attn_pending = 0, n_sel_pending = 0;
  double attn_ms = 0.0, sel_ms = 0.0;
  int64_t attn_launches = 0, sel_launches = 0;
};

namespace {

constexpr size_t kProfPairs = 4096;

void free_ctx(sfi_ctx* c) {
  if (!c) return;
  if (c->side) cudaStreamSynchronize(c->side);
  for (cudaEvent_t e : c->ev_attn) cudaEventDestroy(e);
  for (cudaEvent_t e : c->ev_sel) cudaEventDestroy(e);
  for (int p = 0; p < 2; ++p) {
    if (c->attn_done[p]) cudaEventDestroy(c->attn_done[p]);
    if (c->sel_done[p]) cudaEventDestroy(c->sel_done[p]);
    cudaFree(c->ws[p]);
    cudaFree(c->len_copy[p]);
    cudaFree(c->cand[p]);
    cudaFree(c->ccount[p]);
    cudaFree(c->excl[p]);
  }
  if (c->side) cudaStreamDestroy(c->side);
  cudaFree(c->idx);
  cudaFree(c->count);
  cudaFree(c->knorm);
  cudaFree(c->knorm_valid);
  delete c;
}

// Sum the elapsed times of the first n recorded pairs of `ev` (waits for them).
cudaError_t flush_pairs(std::vector<cudaEvent_t>& ev, size_t& n, double& total_ms) {
  if (n == 0) return cudaSuccess;
  cudaError_t e = cudaEventSynchronize(ev[2 * n - 1]);
  for (size_t i = 0; i < n && e == cudaSuccess; ++i) {
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, ev[2 * i], ev[2 * i + 1]);
    total_ms += ms;
  }
  n = 0;
  return e;
}

cudaError_t record_pair(std::vector<cudaEvent_t>& ev, size_t& n, double& total_ms, bool second,
                        cudaStream_t st) {
  if (!second && n == kProfPairs) {
    cudaError_t e = flush_pairs(ev, n, total_ms);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaEventRecord(ev[2 * n + (second ? 1 : 0)], st);
  if (second) ++n;
  return e;
}

}  // namespace

using namespace sfi;

extern "C" {

sfi_status sfi_ctx_create(const sfi_ctx_desc* d, sfi_ctx** out) {
  if (!d || !out) return fail(SFI_ERR_INVALID_ARG, "desc and ctx_out must be set");
  *out = nullptr;
  sfi_layout L{};
  L.batch = d->batch;
  L.n_q_heads = d->n_q_heads;
  L.n_kv_heads = d->n_kv_heads;
  L.head_dim = d->head_dim;
  L.dtype = d->dtype;
  L.max_len = d->max_len;
  static const int64_t dummy64 = 0;
  static const int32_t dummy32 = 0;
  L.kv_offset = &dummy64;  // geometry check only
  L.kv_cap = &dummy32;
  L.len = &dummy32;
  sfi_status s = check_layout(&L);
  if (s != SFI_OK) return s;
  if ((s = check_params(&d->params, false)) != SFI_OK) return s;
  if (d->params.mode != SFI_SELECT_FUSED)
    return fail(SFI_ERR_INVALID_ARG, "the decode driver runs the fused (SFI) selector");
  if (d->n_layers < 1) return fail(SFI_ERR_INVALID_ARG, "n_layers must be >= 1");
  if (d->budget < 0) return fail(SFI_ERR_INVALID_ARG, "budget must be >= 0");
  if (d->max_len > kSelectMaxLen)
    return fail(SFI_ERR_CAPACITY, "the selector holds at most %d positions per row", kSelectMaxLen);
  if ((s = check_refine(&L, &d->params, &d->refine)) != SFI_OK) return s;
  const bool refine = refine_active(d->refine);
  sfi_ctx* c = new (std::nothrow) sfi_ctx();
  if (!c) return fail(SFI_ERR_CAPACITY, "out of host memory");
  c->desc = *d;
  c->plan = plan_workspace(d->batch, d->n_q_heads, d->n_kv_heads, d->head_dim, d->max_len);
  c->n_sets = d->async_select ? 2 : 1;
  const size_t units = size_t(d->batch) * d->n_kv_heads;
  const size_t row = units * size_t(d->max_len) * sizeof(float);
  cudaError_t e = cudaSuccess;
  for (int p = 0; p < c->n_sets && e == cudaSuccess; ++p) {
    e = cudaMalloc(&c->ws[p], c->plan.total);
    if (e == cudaSuccess) e = cudaMemset(c->ws[p], 0, c->plan.total);
    if (e == cudaSuccess) e = cudaMalloc(&c->len_copy[p], size_t(d->batch) * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->attn_done[p], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->sel_done[p], cudaEventDisableTiming);
    if (refine) {
      c->refine = true;
      c->n_cand = refine_candidates(&L, &d->params, &d->refine);
      if (e == cudaSuccess) e = cudaMalloc(&c->cand[p], units * size_t(c->n_cand) * sizeof(int32_t));
      if (e == cudaSuccess) e = cudaMalloc(&c->ccount[p], units * sizeof(int32_t));
      if (e == cudaSuccess) e = cudaMalloc(&c->excl[p], size_t(d->batch) * d->max_len);
    }
  }
  if (e == cudaSuccess && d->async_select) {
    int lo = 0, hi = 0;  // numerically lowest value = highest priority
    e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&c->side, cudaStreamNonBlocking, hi);
  }
  if (e == cudaSuccess)
    e = cudaMalloc(&c->idx, size_t(d->n_layers) * units * d->params.k * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMalloc(&c->count, size_t(d->n_layers) * units * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(c->count, 0, size_t(d->n_layers) * units * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMalloc(&c->knorm, size_t(d->n_layers) * row);
  if (e == cudaSuccess)
    e = cudaMalloc(&c->knorm_valid, size_t(d->n_layers) * units * sizeof(int32_t));
  if (e == cudaSuccess)
    e = cudaMemset(c->knorm_valid, 0, size_t(d->n_layers) * units * sizeof(int32_t));
  if (e != cudaSuccess) {
    free_ctx(c);
    return cuda_fail(e, "allocating the decode context");
  }
  c->have_sel.assign(d->batch, 0);
  c->slow.assign(d->batch, 0);
  c->since.assign(d->batch, 0);
  *out = c;
  return SFI_OK;
}

sfi_status sfi_ctx_destroy(sfi_ctx* c) {
  free_ctx(c);
  return SFI_OK;
}

sfi_status sfi_schedule(int32_t batch, int32_t budget, const uint8_t* is_boundary,
                        uint8_t* have_sel, int32_t* since, uint8_t* slow_out) {
  if (batch < 1 || budget < 0 || !is_boundary || !have_sel || !since || !slow_out)
    return fail(SFI_ERR_INVALID_ARG, "sfi_schedule: bad batch, budget or NULL array");
  for (int b = 0; b < batch; ++b) {
    const bool sl = is_boundary[b] || !have_sel[b] || (budget > 0 && since[b] >= budget);
    slow_out[b] = sl ? 1 : 0;
    if (sl) {
      have_sel[b] = 1;
      since[b] = 0;
    } else {
      since[b] += 1;
    }
  }
  return SFI_OK;
}

sfi_status sfi_ctx_reset(sfi_ctx* c) {
  if (!c) return fail(SFI_ERR_INVALID_ARG, "ctx is NULL");
  std::fill(c->have_sel.begin(), c->have_sel.end(), 0);
  std::fill(c->since.begin(), c->since.end(), 0);
  std::fill(c->slow.begin(), c->slow.end(), 0);
  c->decided = false;
  c->sel_in_flight = false;
  cudaError_t e = c->side ? cudaStreamSynchronize(c->side) : cudaSuccess;
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  for (int p = 0; p < c->n_sets && e == cudaSuccess; ++p) e = cudaMemset(c->ws[p], 0, c->plan.total);
  if (e == cudaSuccess)
    e = cudaMemset(c->knorm_valid, 0,
                   size_t(c->desc.n_layers) * c->desc.batch * c->desc.n_kv_heads * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "zero-filling the context workspace");
  return SFI_OK;
}

sfi_status sfi_ctx_read_status(sfi_ctx* c, uint32_t* status_host, sfi_stream stream) {
  if (!c || !status_host) return fail(SFI_ERR_INVALID_ARG, "ctx and status_host must be set");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  *status_host = 0;
  for (int p = 0; p < c->n_sets; ++p) {
    cudaError_t e = cudaStreamWaitEvent(st, c->sel_done[p], 0);
    if (e != cudaSuccess) return cuda_fail(e, "ordering the status read");
    uint32_t v = 0;
    const sfi_status s = sfi_read_status(c->ws[p], &v, stream);
    if (s != SFI_OK) return s;
    *status_host |= v;
  }
  return SFI_OK;
}

sfi_status sfi_ctx_profile(sfi_ctx* c, int32_t enable) {
  if (!c) return fail(SFI_ERR_INVALID_ARG, "ctx is NULL");
  if (enable && c->ev_attn.empty()) {
    c->ev_attn.resize(2 * kProfPairs, nullptr);
    c->ev_sel.resize(2 * kProfPairs, nullptr);
    for (auto* v : {&c->ev_attn, &c->ev_sel})
      for (auto& e : *v) {
        const cudaError_t r = cudaEventCreate(&e);
        if (r != cudaSuccess) return cuda_fail(r, "creating profiling events");
      }
  }
  c->profiling = enable != 0;
  if (enable) {
    c->n_attn_pending = c->n_sel_pending = 0;
    c->attn_ms = c->sel_ms = 0.0;
    c->attn_launches = c->sel_launches = 0;
  }
  return SFI_OK;
}

sfi_status sfi_ctx_profile_read(sfi_ctx* c, double* attn_ms, int64_t* attn_launches,
                                double* select_ms, int64_t* select_launches) {
  if (!c || !attn_ms || !attn_launches || !select_ms || !select_launches)
    return fail(SFI_ERR_INVALID_ARG, "ctx and every output must be set");
  if (!c->ev_attn.empty()) {
    cudaError_t e = flush_pairs(c->ev_attn, c->n_attn_pending, c->attn_ms);
    if (e == cudaSuccess) e = flush_pairs(c->ev_sel, c->n_sel_pending, c->sel_ms);
    if (e != cudaSuccess) return cuda_fail(e, "reading profiling events");
  }
  *attn_ms = c->attn_ms;
  *attn_launches = c->attn_launches;
  *select_ms = c->sel_ms;
  *select_launches = c->sel_launches;
  return SFI_OK;
}

sfi_status sfi_ctx_slow_mask(const sfi_ctx* c, uint8_t* slow_host) {
  if (!c || !slow_host) return fail(SFI_ERR_INVALID_ARG, "ctx and slow_host must be set");
  std::memcpy(slow_host, c->slow.data(), c->slow.size());
  return SFI_OK;
}

sfi_status sfi_ctx_selection(const sfi_ctx* c, int32_t layer, int32_t* idx_out,
                             int32_t* count_out, sfi_stream stream) {
  if (!c || !idx_out || !count_out)
    return fail(SFI_ERR_INVALID_ARG, "ctx, idx_out and count_out must be set");
  if (layer < 0 || layer >= c->desc.n_layers)
    return fail(SFI_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, c->desc.n_layers);
  const size_t units = size_t(c->desc.batch) * c->desc.n_kv_heads;
  const size_t ni = units * c->desc.params.k;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  for (int p = 0; p < c->n_sets && e == cudaSuccess; ++p)
    e = cudaStreamWaitEvent(st, c->sel_done[p], 0);  // the latest selectors
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(idx_out, c->idx + size_t(layer) * ni, ni * sizeof(int32_t),
                                  cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(count_out, c->count + size_t(layer) * units, units * sizeof(int32_t),
                        cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "copying the selection");
  return SFI_OK;
}

sfi_status sfi_decode_step(sfi_ctx* c, int32_t layer, const uint8_t* is_boundary,
                           const sfi_layout* L, const void* q, const void* k, const void* v,
                           float* out, sfi_stream stream) {
  if (!c) return fail(SFI_ERR_INVALID_ARG, "ctx is NULL");
  sfi_status s = check_layout(L);
  if (s != SFI_OK) return s;
  const sfi_ctx_desc& d = c->desc;
  if (L->batch != d.batch || L->n_q_heads != d.n_q_heads || L->n_kv_heads != d.n_kv_heads ||
      L->head_dim != d.head_dim || L->dtype != d.dtype)
    return fail(SFI_ERR_INVALID_ARG, "layout does not match the context's geometry");
  if (L->max_len > d.max_len)
    return fail(SFI_ERR_CAPACITY, "layout max_len %d exceeds the context's %d", L->max_len,
                d.max_len);
  if (layer < 0 || layer >= d.n_layers)
    return fail(SFI_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, d.n_layers);
  if (!q || !k || !v || !out) return fail(SFI_ERR_INVALID_ARG, "q, k, v and out must be set");
  if (layer == 0) {
    if (!is_boundary) return fail(SFI_ERR_INVALID_ARG, "layer 0 needs the boundary flags");
    s = sfi_schedule(d.batch, d.budget, is_boundary, c->have_sel.data(), c->since.data(),
                     c->slow.data());
    if (s != SFI_OK) return s;
    c->decided = true;
  } else if (!c->decided) {
    return fail(SFI_ERR_INVALID_ARG, "the first decode step must start at layer 0");
  }
  // The context's buffers are laid out for the context's max_len.
  sfi_layout Lc = *L;
  Lc.max_len = d.max_len;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t units = size_t(d.batch) * d.n_kv_heads;
  int32_t* idx = c->idx + size_t(layer) * units * d.params.k;
  int32_t* count = c->count + size_t(layer) * units;

  const int p = c->n_sets == 2 ? (layer & 1) : 0;
  cudaError_t e = cudaSuccess;
  // the last selector that read this buffer set (and every earlier one) is done
  if (c->side) e = cudaStreamWaitEvent(st, c->sel_done[p], 0);
  if (e != cudaSuccess) return cuda_fail(e, "ordering after the selector");
  AttnArgs a;
  fill_attn_common(a, &Lc, q, k, v, out, c->ws[p], c->plan);
  a.len_copy = c->len_copy[p];
  int n_slow = 0;
  for (int b = 0; b < d.batch; ++b)
    if (c->slow[b]) {
      a.slow.bits[b >> 5] |= 1u << (b & 31);
      ++n_slow;
    }
  a.emit = 1;
  a.knorm = c->knorm + size_t(layer) * units * d.max_len;
  a.knorm_valid = c->knorm_valid + size_t(layer) * units;
  a.idx = idx;
  a.count = count;
  a.idx_stride = d.params.k;
  a.n_sink = d.params.n_sink;
  a.window = d.params.window;
  const int fast_bound = fast_unit_rows_bound(&Lc, &d.params);
  if (c->profiling) e = record_pair(c->ev_attn, c->n_attn_pending, c->attn_ms, false, st);
  if (e != cudaSuccess) return cuda_fail(e, "profiling event");
  // Right after a layer whose selector went to the side stream, launch
  // without programmatic dependence: this launch then becomes ready only when
  // the previous one has completed -- together with that selector, which
  // (higher priority) is placed first and runs beside this launch; as a
  // programmatic dependent this launch would take every SM first.
  const bool pdl = !c->sel_in_flight;
  c->sel_in_flight = false;
  if ((s = run_attn(a, &Lc, (long long)n_slow * d.n_kv_heads, d.max_len,
                    (long long)(d.batch - n_slow) * d.n_kv_heads, fast_bound, st, pdl)) != SFI_OK)
    return s;
  if (c->profiling) {
    e = record_pair(c->ev_attn, c->n_attn_pending, c->attn_ms, true, st);
    if (e != cudaSuccess) return cuda_fail(e, "profiling event");
    c->attn_launches += 1;
  }
  if (n_slow == 0) return SFI_OK;
  cudaStream_t ss = st;  // stream of the selector
  if (c->side) {
    ss = c->side;
    e = cudaEventRecord(c->attn_done[p], st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ss, c->attn_done[p], 0);
    if (e != cudaSuccess) return cuda_fail(e, "forking the selector stream");
  }
  if (c->profiling) {
    e = record_pair(c->ev_sel, c->n_sel_pending, c->sel_ms, false, ss);
    if (e != cudaSuccess) return cuda_fail(e, "profiling event");
  }

  // Selector straight from the stored logits (the evidence f is formed on
  // the fly; the decode path has no use for f itself).
  SelectArgs sa{};
  sa.logits = a.logits;
  sa.stats = a.stats;
  sa.H_q = d.n_q_heads;
  sa.knorm = a.knorm;
  sa.len = c->len_copy[p];
  sa.idx = idx;
  sa.count = count;
  sa.s = nullptr;
  sa.B = d.batch;
  sa.H_kv = d.n_kv_heads;
  sa.max_len = d.max_len;
  sa.n_sink = d.params.n_sink;
  sa.window = d.params.window;
  sa.k = d.params.k;
  sa.lambda = d.params.lambda;
  sa.mode = SFI_SELECT_FUSED;
  sa.g_only = -1;
  sa.active = a.slow;
  sa.status = a.status;
  attach_select_scratch(sa, c->ws[p], c->plan);
  if (c->refine) {
    // the refinement reads the fused scores back: they go to the workspace
    sa.s = reinterpret_cast<float*>(c->ws[p] + c->plan.s_off);
    if ((s = run_refined_select(sa, d.refine, d.params.k, c->n_cand, idx, count, c->cand[p],
                                c->ccount[p], c->excl[p], ss)) != SFI_OK)
      return s;
  } else {
    e = launch_select(sa, ss);
    if (e != cudaSuccess) return cuda_fail(e, "selector launch");
  }
  if (c->profiling) {
    e = record_pair(c->ev_sel, c->n_sel_pending, c->sel_ms, true, ss);
    if (e != cudaSuccess) return cuda_fail(e, "profiling event");
    c->sel_launches += 1;
  }
  if (c->side) {
    c->sel_in_flight = true;
    e = cudaEventRecord(c->sel_done[p], ss);
    // join at the last layer: the token's work ends on the caller's stream
    if (e == cudaSuccess && layer == d.n_layers - 1) e = cudaStreamWaitEvent(st, c->sel_done[p], 0);
    if (e != cudaSuccess) return cuda_fail(e, "joining the selector stream");
  }
  return SFI_OK;
}

}  // extern "C"
