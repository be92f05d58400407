// Decode driver of libsfi (sfi_decode_step): the slow/fast schedule of the
// SFI pages ("Slow-Fast paradigm": a slow step near a semantic boundary or
// when the reuse budget is exhausted, fast steps otherwise) on top of the
// attention, evidence and selector kernels.  One context serves every layer
// of a model: each layer keeps its own selection; the decision is taken once
// per token (at layer 0) and shared by all layers.
#include <cuda_runtime.h>

#include <cstring>
#include <new>
#include <vector>

#include "sfi_internal.h"

struct sfi_ctx {
  sfi_ctx_desc desc;
  sfi::WsPlan plan;
  // device
  char* ws = nullptr;          // attention / selector workspace
  float* f = nullptr;          // [B*H_kv][max_len]
  float* knorm = nullptr;      // [B*H_kv][max_len]
  int32_t* idx = nullptr;      // [L][B*H_kv][k]
  int32_t* count = nullptr;    // [L][B*H_kv]
  // host schedule state
  std::vector<uint8_t> have_sel, slow;
  std::vector<int32_t> since;
  bool decided = false;
};

namespace {

void free_ctx(sfi_ctx* c) {
  if (!c) return;
  cudaFree(c->ws);
  cudaFree(c->f);
  cudaFree(c->knorm);
  cudaFree(c->idx);
  cudaFree(c->count);
  delete c;
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
  sfi_ctx* c = new (std::nothrow) sfi_ctx();
  if (!c) return fail(SFI_ERR_CAPACITY, "out of host memory");
  c->desc = *d;
  c->plan = plan_workspace(d->batch, d->n_q_heads, d->n_kv_heads, d->head_dim, d->max_len);
  const size_t units = size_t(d->batch) * d->n_kv_heads;
  const size_t row = units * size_t(d->max_len) * sizeof(float);
  cudaError_t e = cudaMalloc(&c->ws, c->plan.total);
  if (e == cudaSuccess) e = cudaMemset(c->ws, 0, c->plan.total);
  if (e == cudaSuccess) e = cudaMalloc(&c->f, row);
  if (e == cudaSuccess) e = cudaMalloc(&c->knorm, row);
  if (e == cudaSuccess)
    e = cudaMalloc(&c->idx, size_t(d->n_layers) * units * d->params.k * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMalloc(&c->count, size_t(d->n_layers) * units * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(c->count, 0, size_t(d->n_layers) * units * sizeof(int32_t));
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
  cudaError_t e = cudaMemcpyAsync(idx_out, c->idx + size_t(layer) * ni, ni * sizeof(int32_t),
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

  AttnArgs a;
  fill_attn_common(a, &Lc, q, k, v, out, c->ws, c->plan);
  int n_slow = 0;
  for (int b = 0; b < d.batch; ++b)
    if (c->slow[b]) {
      a.slow.bits[b >> 5] |= 1u << (b & 31);
      ++n_slow;
    }
  a.emit = 1;
  a.knorm = c->knorm;
  a.idx = idx;
  a.count = count;
  a.idx_stride = d.params.k;
  a.n_sink = d.params.n_sink;
  a.window = d.params.window;
  const int fast_bound = fast_unit_rows_bound(&Lc, &d.params);
  const long long total = (long long)d.n_kv_heads *
                          ((long long)n_slow * d.max_len + (long long)(d.batch - n_slow) * fast_bound);
  const int max_unit = n_slow ? d.max_len : fast_bound;
  if ((s = run_attn(a, &Lc, total, max_unit, st)) != SFI_OK) return s;
  if (n_slow == 0) return SFI_OK;

  FpassArgs fa{};
  fa.logits = a.logits;
  fa.stats = a.stats;
  fa.len = Lc.len;
  fa.f = c->f;
  fa.B = d.batch;
  fa.H_q = d.n_q_heads;
  fa.H_kv = d.n_kv_heads;
  fa.max_len = d.max_len;
  fa.slow = a.slow;
  fa.status = a.status;
  cudaError_t e = launch_fpass(fa, st);
  if (e != cudaSuccess) return cuda_fail(e, "evidence pass launch");

  SelectArgs sa{};
  sa.evidence = c->f;
  sa.knorm = c->knorm;
  sa.len = Lc.len;
  sa.idx = idx;
  sa.count = count;
  sa.s = reinterpret_cast<float*>(c->ws + c->plan.s_off);
  sa.B = d.batch;
  sa.H_kv = d.n_kv_heads;
  sa.max_len = d.max_len;
  sa.n_sink = d.params.n_sink;
  sa.window = d.params.window;
  sa.k = d.params.k;
  sa.lambda = d.params.lambda;
  sa.mode = SFI_SELECT_FUSED;
  sa.active = a.slow;
  sa.status = a.status;
  e = launch_select(sa, st);
  if (e != cudaSuccess) return cuda_fail(e, "selector launch");
  return SFI_OK;
}

}  // extern "C"
