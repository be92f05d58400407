// Internal declarations of libsfi shared by the C-ABI layer (api.cpp,
// decode.cpp) and the CUDA kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/sfi.h"

namespace sfi {

constexpr int kMaxBatch = 1024;  // sequences per launch (bit mask capacity)
constexpr int kMaxUnits = 4096;  // (sequence, KV head) pairs per launch
constexpr int kItemSlotsPerUnit = 64;  // split-K partial slots per (sequence, KV head)
// Default limit of a pipeline wait, in SM clocks (about 2 s at 2 GHz).
constexpr long long kDefaultWaitCycles = 4000000000LL;

// Bit b set: sequence b runs a slow (dense) step in this launch.
struct SeqMask {
  uint32_t bits[kMaxBatch / 32];
};

// Split-K attention over either the whole cache (slow sequences) or the
// managed sparse state (fast sequences) of every (sequence, KV head) unit.
struct AttnArgs {
  // 2-D TMA descriptors of K and V viewed as [rows][D] bf16 rows with a
  // 128-byte swizzle and 64 x 64 boxes (used when use_tma is set).
  CUtensorMap tmk;
  CUtensorMap tmv;
  int32_t use_tma;
  const void* q;  // [B][H_q][D]
  const void* k;
  const void* v;
  const int64_t* kv_offset;
  const int32_t* kv_cap;
  const int32_t* len;
  float* out;     // [B][H_q][D]
  float* logits;  // [B*H_kv][max_len][G], log2-scaled logits of slow units (emit)
  float* knorm;   // [B*H_kv][max_len] key norms of slow units (nullable)
  // optional [B*H_kv]: rows below knorm_valid[u] already have their key norms
  // in knorm (a cache row never changes); a slow unit computes the rest and
  // sets it to its length
  int32_t* knorm_valid;
  float* stats;   // [B*H_q][2]: (max log2-logit, sum of 2^(l - max)) of slow units
  const int32_t* idx;    // [B*H_kv][idx_stride] selected positions (fast units)
  const int32_t* count;  // [B*H_kv]
  int32_t idx_stride;
  int32_t n_sink;
  int32_t window;
  int32_t B, H_q, H_kv, max_len;
  int32_t rpi_slow, rpi_fast;  // rows per work item of slow and of fast units
  // > 0: no slow unit in the launch and every unit has exactly this many
  // items (its rows dealt over them; items past a short unit's rows are
  // empty); the kernel then builds no unit table
  int32_t fast_items;
  int32_t max_items;
  int32_t emit;    // slow units write logits, stats (and knorm if non-null)
  float qscale;    // log2(e) / sqrt(D)
  SeqMask slow;
  float* partials;     // [max_items][G][D + 2]
  int32_t* counters;   // [B*H_kv], zero between launches
  uint32_t* work_ctr;  // [2]: next item, CTAs done fetching; zero between launches
  int32_t* len_copy;   // optional [B]: the kernel copies len here (for a later selector)
  uint32_t* status;
  // limit of a consumer's wait for a stage's rows, in SM clocks; after it the
  // CTA aborts and sets SFI_DEV_WAIT_TIMEOUT (wait_limit_cycles() by default)
  long long wait_cycles;
};

struct FpassArgs {
  const float* logits;
  const float* stats;
  const int32_t* len;
  float* f;  // [B*H_kv][max_len]
  int32_t B, H_q, H_kv, max_len;
  SeqMask slow;
  uint32_t* status;
};

constexpr int kSelectMaxLen = 327680;  // positions per row a selection takes (documented limit)
constexpr int kSelMaxChunks = 64;      // chunk CTAs per selecting unit, at most
constexpr int kSelHistWords = 3 * 2048;  // a unit's three radix histograms
constexpr int kSelCandCap = 8192;        // candidates (keys of the k-th key's top bin) gathered, at most
constexpr int kSelCandRows = 256;        // units of a launch that split into chunks, at most

struct SelectArgs {
  const float* evidence;  // f (fused mode) or per-KV-head logit sums (logit-sum mode)
  const float* logits;    // if set: compute f from these log2-scaled logits [unit][pos][G]
  const float* stats;     //   and these per-head (M, Z) instead of reading `evidence`
  int32_t H_q;
  const float* knorm;
  const int32_t* len;
  int32_t* idx;    // [B*H_kv][k]
  int32_t* count;  // [B*H_kv]
  float* s;        // [B*H_kv][max_len] fused scores (nullable)
  int32_t B, H_kv, max_len;
  int32_t n_sink, window, k;
  float lambda;
  int32_t mode;
  SeqMask active;
  uint32_t* status;
  // selector scratch (workspace), rows indexed like the per-position arrays
  float* sel_nu;        // [B*H_kv][kSelMaxChunks] chunk sums of key norms over E
  uint32_t* sel_cnt;    // [B*H_kv][kSelMaxChunks][2] keys above / equal to the k-th per chunk
  uint32_t* sel_hist;   // [B*H_kv][kSelHistWords] the three digit histograms, zero between launches
  uint32_t* sel_ctr;    // [B*H_kv][4] barrier counter ([0]; rests with its low 31 bits at zero)
  uint32_t* sel_keys;   // [B*H_kv][max_len] order keys that do not fit in shared memory
  unsigned long long* sel_cand;  // [kSelCandRows][max_len] (key << 32 | position) per selecting unit
  int32_t keys_smem;    // set by the launcher: the keys stay in shared memory
  int32_t smem_split;   // set by the launcher: words of shared memory before the candidates
  long long wait_cycles;  // set by the launcher: limit of each barrier wait, in SM clocks
  // Cross-head exclusivity (fused mode): the ranked score of position i is
  // s_i * exp(-excl_beta * excl[b][i]) when excl is set ([B][max_len] counts).
  const uint8_t* excl;
  float excl_beta;
  int32_t g_only;  // >= 0: only the units of this KV head (fused mode)
};


// Verification attention (Vegas): R chain rows per head, collected logit sums.
struct VerifyArgs {
  AttnArgs base;         // q: [B][R][H_q][D]; out: [B][R][H_q][D]; all units dense
  int32_t R;             // verify rows per sequence
  int32_t ncg;           // collected rows * G (tile rows 0..ncg-1 are collected)
  int8_t t_of_slot[8];   // chain row of each tile slot (slot = tile row / G)
  float* lsum;           // [B*H_kv][max_len] or null
  float lscale;          // 1 / sqrt(D)
};
cudaError_t launch_verify(const VerifyArgs& va, int D, int G, cudaStream_t st);
int verify_stage_rows();

// Workspace plan: one layout serves every call of a given geometry.
struct WsPlan {
  size_t status_off, counters_off, partials_off, logits_off, stats_off, s_off;
  size_t sel_nu_off, sel_cnt_off, sel_hist_off, sel_ctr_off, sel_keys_off, sel_cand_off;
  size_t total;
  int32_t max_items;
};

WsPlan plan_workspace(int B, int H_q, int H_kv, int D, int max_len);

// Point the selector's scratch fields of `a` into workspace `ws` laid out by `p`.
void attach_select_scratch(SelectArgs& a, char* ws, const WsPlan& p);

// Kernel launchers (return the CUDA error of the launch).
cudaError_t launch_fpass(const FpassArgs& a, cudaStream_t st);
cudaError_t launch_select(const SelectArgs& a, cudaStream_t st);

int device_sm_count();
// Pipeline-wait limit given to every attention and verify launch (SM clocks;
// sfi_set_wait_limit changes it for the whole process).
long long wait_limit_cycles();

// Host helpers of the C-ABI layer (api.cpp), shared with the decode driver.
sfi_status check_layout(const sfi_layout* L);
sfi_status check_params(const sfi_params* P, bool for_select);
void fill_attn_common(AttnArgs& a, const sfi_layout* L, const void* q, const void* k,
                      const void* v, float* out, char* ws, const WsPlan& p);
// pdl: launch as a programmatic dependent of the previous launch on `st`
// (it may start while that launch drains; it waits for it before any global
// access).
sfi_status run_attn(AttnArgs& a, const sfi_layout* L, long long n_slow_units, int slow_rows,
                    long long n_fast_units, int fast_rows, cudaStream_t st, bool pdl = true);
int fast_unit_rows_bound(const sfi_layout* L, const sfi_params* P);
// Rows per work item of each unit class: class a (n_a units of at most
// rows_a rows, taken first) and class b (n_b units of at most rows_b).
struct ItemSplit {
  int rpi_a, rpi_b;
};
// emit: class-a units write evidence (their CTAs cannot speed up in a tail).
ItemSplit choose_item_split(long long n_a, int rows_a, long long n_b, int rows_b, int sr, int grid,
                            bool emit);
// Fill a.tmk / a.tmv for bf16 caches (sets a.use_tma; leaves it 0 if the
// driver entry point is unavailable).
void attach_tensor_maps(AttnArgs& a, const sfi_layout* L);
sfi_status fail(sfi_status s, const char* fmt, ...);
sfi_status cuda_fail(cudaError_t e, const char* what);

}  // namespace sfi
