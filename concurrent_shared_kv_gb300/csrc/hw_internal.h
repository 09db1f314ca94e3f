// hw_internal.h - host-side declarations shared by the C ABI (api.cpp) and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hogwild.h"

namespace hw {

// Tokens per scheduling unit (one tile of one block for one kv head).
constexpr int kSimtTile = 64;
constexpr int kTcTile = 128;
// Query heads one tile serves at most (view references to a block x group).
constexpr int kMaxQ = HW_MAX_QHEADS_PER_BLOCK;
// Partial records one (row, kv head) merge can gather: at most one per (view
// entry, CTA) pair whose ranges meet, i.e. <= max_view_blocks + grid - 1.
constexpr int kMaxRecords = 1024;

// Everything a decode kernel needs; passed by value as a kernel parameter.
// A partial record is o[0..D), m, l and padding to whole 128-byte lines: a
// record's stores and loads then touch D / 32 + 1 lines, not one more.
constexpr int kRecPad = 32;

struct DecodeArgs {
  const void *q;
  const void *k;
  const void *v;
  const int32_t *block_start;
  const int32_t *block_len;
  const int32_t *view_block;
  const int32_t *view_offset;
  const int32_t *q_pos;
  const int32_t *q_to_kv;
  void *out;
  float *lse;
  int32_t *err;       // workspace error word (HW_DEV_* bits)
  int32_t *counters;  // [n_rows][Hq] merge arrival counters, zero between calls
  float *partials;    // [slots][kMaxQ][D + kRecPad]: o[0..D), m at D, l at D+1
  // Tensor-core path: nonzero when the caller promises that the work enqueued
  // just before this call on the stream writes neither the K/V pools nor the
  // plan (or metadata) this call reads; the kernel then reads them, and starts
  // its first K/V tiles, before the previous kernel has completed.
  int32_t early;
  // Bound of the merge's wait for an item's records, in SM clock cycles
  // (hw_test_set_merge_wait_limit; ~1 s by default).
  int64_t wait_limit;
#ifdef HW_TRACE
  int32_t trace_call;  // the call's index in the process (layer-timeline build)
#endif
  int32_t n_rows, n_q_heads, n_kv_heads, head_dim, n_blocks, n_view;
  int64_t capacity;
  const uint8_t *plan;  // precomputed plan of the tensor-core kernel (hw_attn_plan), or null
  // hw_attn_decode's plan cache in the workspace (see PlanCache), or null
  uint8_t *cache_base;
  int64_t cache_meta_bytes, cache_plan_bytes;
  // The step's appends: at plan time the caller's arrays (null: none); at
  // decode time the plan's copies.  k_new / v_new: this layer's new tokens,
  // [n_rows][Hkv][D], or null (nothing is written; k and v are then only read).
  const int32_t *append_block, *append_pos;
  const void *k_new, *v_new;
  // Per view entry, the tokens of its block the row attends (negative: all),
  // or null: every entry sees its whole block.  At plan time the caller's
  // array, at decode time the plan's copy.
  const int32_t *view_limit;
  // E4M3 caches: per kv head, the scale of its K and V codes (null: bf16 caches)
  const float *k_scale, *v_scale;
  float scale_log2;   // softmax scale * log2(e): scores live in the log2 domain
  // RoPE phase increments: for pair i, the fraction of a turn per position,
  // frac(w_i / 2pi), as an unsigned 0.64 fixed-point number.  The angle of
  // position p is then (p * phase[i]) mod 2^64 turns, exact in integers.
  uint64_t phase[64];
};

// hw_attn_decode's plan cache: [state: current buffer, arrivals][metadata
// copy 0][metadata copy 1][plan 0][plan 1].  Buffer `cur` holds the plan of
// the metadata in copy `cur`; a plan launch whose metadata differs builds
// into the other buffer and its last CTA makes that one current.  A metadata
// copy is the effective view_block, view_offset ([rows][V] each), q_pos
// [rows], q head -> kv head map [Hq], block_start, block_len [blocks].
struct PlanCacheState {
  int32_t cur;    // 0 or 1
  int32_t count;  // CTAs of the building plan launch that are done (0 between launches)
};
constexpr size_t kPlanCacheStateBytes = 256;
inline __host__ __device__ int64_t plan_cache_meta_words(int64_t n_rows, int64_t n_view, int64_t n_q_heads,
                                                         int64_t n_blocks) {
  return 2 * n_rows * n_view + n_rows + n_q_heads + 2 * n_blocks;
}

// Workspace layout helpers (bytes).  The metadata copies and the plan are
// written by hw_attn_plan and read by hw_attn_decode_planned.
struct WorkspaceLayout {
  size_t err_off, counters_off, partials_off, meta_off, plan_off, cache_off, total;
  size_t cache_meta_bytes, cache_plan_bytes;
  int64_t slots;
};
constexpr size_t kPlanHeaderBytes = 256;
size_t plan_shared_bytes();  // the part of a plan every CTA reads
size_t plan_cta_bytes();     // the part each CTA reads for itself
// From a host copy of a plan region: kPlanExportFields int64 per CTA (unit
// range, number of first tiles, their rows, kv heads, segment flags and
// column groups).  Returns the plan's grid, or -1 when there is no plan (or
// it exceeds max_ctas).
constexpr int kPlanExportFields = 15;
int plan_export_records(const uint8_t *plan_host, int64_t *out, int max_ctas);
WorkspaceLayout workspace_layout(const hw_attn_desc &d, int max_ctas);
// The layout the decode calls use on the current device (their max_ctas).
WorkspaceLayout decode_workspace_layout(const hw_attn_desc &d);

int device_sm_count();  // SMs of the current device, cached; <= 0 on failure

// Launchers (return cudaError_t of the launch).
cudaError_t launch_decode_simt(const DecodeArgs &a, int dtype, int ctas, cudaStream_t s);
cudaError_t launch_decode_tc(const DecodeArgs &a, const CUtensorMap &k_map,
                             const CUtensorMap &v_map, int ctas, cudaStream_t s);
size_t decode_tc_smem_bytes();

// Destinations of hw_attn_plan: metadata copies (int32) and, for the
// tensor-core kernel, the plan (header, shared part, one record per CTA).
struct PlanOut {
  uint8_t *plan;  // null: copy the metadata only
  int32_t records;  // CTAs of the decode launches the plan is for
  int32_t *view_block, *view_offset, *q_pos, *q_to_kv, *block_start, *block_len;
  int32_t *append_block, *append_pos;  // -1 / 0 for every row without an append
  int32_t *view_limit;                 // -1 for every entry without a limit
};
cudaError_t launch_plan(const DecodeArgs &a, const PlanOut &o, cudaStream_t s);
int decode_simt_ctas_per_sm(int dtype, int head_dim);

// One launch commits n_commits ranges (kernel grid row c = commit c).
constexpr int kMaxCommits = 64;  // HW_MAX_COMMITS
struct CommitArgs {
  const void *k_src, *v_src;
  void *k_dst, *v_dst;
  int64_t src_capacity, dst_capacity;
  int32_t n_layers, n_kv_heads, head_dim, n_commits;
  uint64_t phase[64];
  int32_t src_begin[kMaxCommits], dst_offset[kMaxCommits], n_tokens[kMaxCommits];
  int32_t delta[kMaxCommits];  // pos_delta
};
cudaError_t launch_commit(const CommitArgs &a, int dtype, cudaStream_t s);

// Fixed-point phase table for RoPE (host): frac(theta^(-2i/D) / 2pi) * 2^64.
void rope_phase_table(int head_dim, double theta, uint64_t *phase);

}  // namespace hw
