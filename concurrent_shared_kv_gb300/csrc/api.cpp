// api.cpp - the C ABI of libhogwild (declared in include/hogwild.h): argument
// checks on the host, workspace layout, RoPE phase tables, kernel selection.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <atomic>
#include <mutex>

#include "hogwild.h"
#include "hw_internal.h"

namespace hw {

static thread_local int g_last_cuda_error = 0;

// The merge's wait bound for calls made after hw_test_set_merge_wait_limit.
constexpr long long kDefaultMergeWait = 2000000000ll;  // ~1 s at 2 GHz
static std::atomic<long long> g_merge_wait{kDefaultMergeWait};

static int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return HW_ERR_CUDA;
}

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    cache[dev] = n;
  }
  return cache[dev];
}

// frac(w_i / 2pi) * 2^64 with w_i = theta^(-2i/D), in long double so that the
// table is exact to well below one unit of its last place for positions up to
// 2^31.
void rope_phase_table(int head_dim, double theta, uint64_t *phase) {
  const long double two_pi = 6.283185307179586476925286766559005768L;
  for (int i = 0; i < 64; ++i) phase[i] = 0;
  for (int i = 0; i < head_dim / 2 && i < 64; ++i) {
    const long double w = powl(static_cast<long double>(theta),
                               -2.0L * static_cast<long double>(i) / static_cast<long double>(head_dim));
    long double f = w / two_pi;
    f -= floorl(f);
    long double x = ldexpl(f, 64) + 0.5L;
    if (x >= 18446744073709551616.0L) x -= 18446744073709551616.0L;
    phase[i] = static_cast<uint64_t>(x);
  }
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
static PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// TMA map of one bf16 pool [Hkv][capacity][128]: boxes of 128 tokens x 64
// elements (128 bytes, the 128-byte swizzle span), one head at a time.
// Tokens past the capacity read as zeros.
// A [Hkv][capacity][128] pool as 128-token tiles of 128 bytes per row,
// 128-byte swizzled: bf16 in two boxes of 64 elements, E4M3 in one of 128.
static bool make_pool_map(CUtensorMap *m, const void *pool, int64_t capacity, int n_kv_heads,
                          bool e4m3 = false) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t cap = capacity > 0 ? static_cast<cuuint64_t>(capacity) : 1;
  const cuuint64_t esz = e4m3 ? 1 : 2;
  cuuint64_t dims[3] = {128, cap, static_cast<cuuint64_t>(n_kv_heads)};
  cuuint64_t strides[2] = {128 * esz, cap * 128 * esz};
  cuuint32_t box[3] = {e4m3 ? 128u : 64u, static_cast<cuuint32_t>(kTcTile), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Upper bound on the CTAs of any decode launch: slots are sized for it.
static int max_decode_ctas() {
  const int sms = device_sm_count();
  if (sms <= 0) return -1;
  // a merge gathers at most max_view_blocks + grid - 1 records
  const int cap = kMaxRecords - HW_MAX_VIEW_BLOCKS;
  return sms * 4 < cap ? sms * 4 : cap;
}

WorkspaceLayout workspace_layout(const hw_attn_desc &d, int max_ctas) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  WorkspaceLayout L{};
  L.err_off = 0;
  L.counters_off = 256;
  const size_t counters = static_cast<size_t>(d.n_rows) * d.n_q_heads * sizeof(int32_t);
  L.partials_off = L.counters_off + up(counters);
  // segments per kv head: sum over referenced blocks of ceil(refs / rpg)
  // column groups <= n_blocks + floor(entries / rpg) (rpg = references a
  // group holds), then one more slot per CTA
  const int64_t rpg = kMaxQ / (d.n_q_heads / d.n_kv_heads);
  const int64_t n_entries = static_cast<int64_t>(d.n_rows) * d.max_view_blocks;
  L.slots = (d.n_blocks + n_entries / rpg) * d.n_kv_heads + max_ctas;
  const size_t rec = static_cast<size_t>(kMaxQ) * (d.head_dim + kRecPad) * sizeof(float);
  L.meta_off = L.partials_off + up(static_cast<size_t>(L.slots) * rec);
  // metadata copies: view_block, view_offset (rows x V), q_pos, q_to_kv, block_start, block_len,
  // append_block, append_pos, view_limit (rows x V)
  const size_t entries = static_cast<size_t>(d.n_rows) * d.max_view_blocks;
  const size_t meta = (3 * entries + 3 * static_cast<size_t>(d.n_rows) + d.n_q_heads +
                       2 * static_cast<size_t>(d.n_blocks)) *
                      sizeof(int32_t);
  L.plan_off = L.meta_off + up(meta);
  // the tensor-core plan: one record per CTA of its grid (one per SM)
  const int sms = device_sm_count();
  const size_t plan = kPlanHeaderBytes + plan_shared_bytes() +
                      static_cast<size_t>(sms > 0 ? sms : 0) * plan_cta_bytes();
  // hw_attn_decode's plan cache (tensor-core path; see PlanCacheState): it
  // never touches the step's plan of hw_attn_plan
  L.cache_off = L.plan_off + up(plan);
  L.cache_meta_bytes = up(static_cast<size_t>(plan_cache_meta_words(d.n_rows, d.max_view_blocks,
                                                                    d.n_q_heads, d.n_blocks)) *
                          sizeof(int32_t));
  L.cache_plan_bytes = up(plan);
  L.total = L.cache_off + kPlanCacheStateBytes + 2 * L.cache_meta_bytes + 2 * L.cache_plan_bytes;
  return L;
}

WorkspaceLayout decode_workspace_layout(const hw_attn_desc &d) {
  return workspace_layout(d, max_decode_ctas());
}

// The metadata copies of a workspace (written by hw_attn_plan).
struct MetaCopies {
  int32_t *view_block, *view_offset, *q_pos, *q_to_kv, *block_start, *block_len;
  int32_t *append_block, *append_pos, *view_limit;
};
static MetaCopies meta_copies(const hw_attn_desc &d, const WorkspaceLayout &L, void *workspace) {
  int32_t *m = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + L.meta_off);
  const size_t entries = static_cast<size_t>(d.n_rows) * d.max_view_blocks;
  MetaCopies c;
  c.view_block = m;
  c.view_offset = c.view_block + entries;
  c.q_pos = c.view_offset + entries;
  c.q_to_kv = c.q_pos + d.n_rows;
  c.block_start = c.q_to_kv + d.n_q_heads;
  c.block_len = c.block_start + d.n_blocks;
  c.append_block = c.block_len + d.n_blocks;
  c.append_pos = c.append_block + d.n_rows;
  c.view_limit = c.append_pos + d.n_rows;
  return c;
}

static int check_desc(const hw_attn_desc *d) {
  if (!d) return HW_ERR_INVALID;
  if (d->n_rows < 0 || d->n_blocks < 0 || d->max_view_blocks < 0 || d->cache_capacity < 0)
    return HW_ERR_INVALID;
  if (d->n_q_heads <= 0 || d->n_kv_heads <= 0 || d->n_q_heads % d->n_kv_heads != 0)
    return HW_ERR_INVALID;
  if (d->dtype != HW_F32 && d->dtype != HW_BF16 && d->dtype != HW_FP8_E4M3) return HW_ERR_INVALID;
  if (!(d->rope_theta > 1.0) || !std::isfinite(d->rope_theta)) return HW_ERR_INVALID;
  if (!std::isfinite(d->scale)) return HW_ERR_INVALID;
  if (d->head_dim != 64 && d->head_dim != 128) return HW_ERR_UNSUPPORTED;
  if (d->dtype == HW_FP8_E4M3 && d->head_dim != 128) return HW_ERR_UNSUPPORTED;
  if (d->n_blocks > HW_MAX_BLOCKS) return HW_ERR_UNSUPPORTED;
  if (d->n_q_heads > HW_MAX_Q_HEADS) return HW_ERR_UNSUPPORTED;
  if (d->max_view_blocks > HW_MAX_VIEW_BLOCKS) return HW_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->n_rows) * d->max_view_blocks > HW_MAX_VIEW_ENTRIES)
    return HW_ERR_UNSUPPORTED;
  if (d->n_q_heads / d->n_kv_heads > kMaxQ) return HW_ERR_UNSUPPORTED;
  if (d->cache_capacity > INT32_MAX) return HW_ERR_UNSUPPORTED;
  if (d->flags & ~(HW_DESC_VIEW_LIMITS | HW_DESC_EARLY_LOADS)) return HW_ERR_INVALID;
  if ((d->flags & HW_DESC_VIEW_LIMITS) &&
      !((d->dtype == HW_BF16 || d->dtype == HW_FP8_E4M3) && d->head_dim == 128))
    return HW_ERR_UNSUPPORTED;
  return HW_OK;
}

static bool limited(const hw_attn_desc *d) { return (d->flags & HW_DESC_VIEW_LIMITS) != 0; }

}  // namespace hw

using namespace hw;

extern "C" {

int hw_attn_decode_workspace_size(const hw_attn_desc *d, size_t *bytes) {
  const int st = check_desc(d);
  if (st != HW_OK) return st;
  if (!bytes) return HW_ERR_INVALID;
  const int ctas = max_decode_ctas();
  if (ctas <= 0) return cuda_fail(cudaGetLastError());
  *bytes = workspace_layout(*d, ctas).total;
  return HW_OK;
}

int hw_test_set_merge_wait_limit(int64_t cycles) {
  if (cycles < 0) return HW_ERR_INVALID;
  g_merge_wait.store(cycles == 0 ? kDefaultMergeWait : static_cast<long long>(cycles));
  return HW_OK;
}

int hw_workspace_init(void *workspace, size_t bytes, void *stream) {
  if (!workspace || bytes < 256) return HW_ERR_WORKSPACE;
  const cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? HW_OK : cuda_fail(e);
}

}  // extern "C"

namespace hw {

// Workspace checks shared by hw_attn_decode, hw_attn_decode_planned and
// hw_attn_plan (after the description and argument checks); fills the layout.
static int check_workspace(const hw_attn_desc *d, void *workspace, size_t workspace_bytes,
                           WorkspaceLayout *L, int *max_ctas) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return HW_ERR_WORKSPACE;
  *max_ctas = max_decode_ctas();
  if (*max_ctas <= 0) return cuda_fail(cudaGetLastError());
  *L = workspace_layout(*d, *max_ctas);
  if (workspace_bytes < L->total) return HW_ERR_WORKSPACE;
  return HW_OK;
}

static void fill_args(DecodeArgs &a, const hw_attn_desc *d, const WorkspaceLayout &L, void *workspace) {
  std::memset(&a, 0, sizeof a);
  char *ws = static_cast<char *>(workspace);
  a.err = reinterpret_cast<int32_t *>(ws + L.err_off);
  a.counters = reinterpret_cast<int32_t *>(ws + L.counters_off);
  a.partials = reinterpret_cast<float *>(ws + L.partials_off);
  a.early = (d->flags & HW_DESC_EARLY_LOADS) != 0;
#ifdef HW_TRACE
  {
    static std::atomic<int32_t> calls{0};
    a.trace_call = calls++;
  }
#endif
  a.wait_limit = g_merge_wait.load();
  a.n_rows = d->n_rows;
  a.n_q_heads = d->n_q_heads;
  a.n_kv_heads = d->n_kv_heads;
  a.head_dim = d->head_dim;
  a.n_blocks = d->n_blocks;
  a.n_view = d->max_view_blocks;
  a.capacity = d->cache_capacity;
  a.scale_log2 = static_cast<float>(static_cast<double>(d->scale) * 1.4426950408889634074);
  rope_phase_table(d->head_dim, d->rope_theta, a.phase);
  a.cache_meta_bytes = static_cast<int64_t>(L.cache_meta_bytes);  // (the plan cache: use_plan_cache)
  a.cache_plan_bytes = static_cast<int64_t>(L.cache_plan_bytes);
}

static void use_plan_cache(DecodeArgs &a, const WorkspaceLayout &L, void *workspace) {
  a.cache_base = static_cast<uint8_t *>(workspace) + L.cache_off;
}

static bool tensor_core_path(const hw_attn_desc *d) {
  return (d->dtype == HW_BF16 || d->dtype == HW_FP8_E4M3) && d->head_dim == 128;
}
static bool e4m3(const hw_attn_desc *d) { return d->dtype == HW_FP8_E4M3; }

// One decode launch: metadata from the caller (plan null) or from the
// workspace copies with the step's plan.
static int decode_common(const hw_attn_desc *d, const void *q, const void *k_cache,
                         const void *v_cache, const int32_t *block_start, const int32_t *block_len,
                         const int32_t *view_block, const int32_t *view_offset,
                         const int32_t *q_pos, const int32_t *q_to_kv, const uint8_t *plan,
                         void *out, float *lse, void *workspace, const WorkspaceLayout &L,
                         int max_ctas, void *stream, const int32_t *append_block = nullptr,
                         const int32_t *append_pos = nullptr, const void *k_new = nullptr,
                         const void *v_new = nullptr, const int32_t *view_limit = nullptr,
                         const float *k_scale = nullptr, const float *v_scale = nullptr,
                         bool from_cache = false) {
  DecodeArgs a;
  fill_args(a, d, L, workspace);
  if (from_cache) use_plan_cache(a, L, workspace);  // hw_attn_decode: the plan cache
  a.view_limit = view_limit;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.append_block = append_block;
  a.append_pos = append_pos;
  a.k_new = k_new;
  a.v_new = v_new;
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.block_start = block_start;
  a.block_len = block_len;
  a.view_block = view_block;
  a.view_offset = view_offset;
  a.q_pos = q_pos;
  a.q_to_kv = q_to_kv;
  a.out = out;
  a.lse = lse;

  const int sms = device_sm_count();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (tensor_core_path(d)) {
    // tensor-core path: one persistent CTA per SM, K/V tiles by TMA
    a.plan = plan;
    const bool have_pool = d->n_blocks > 0 && d->cache_capacity > 0;
    if (reinterpret_cast<uintptr_t>(q) & 15u) return HW_ERR_INVALID;  // 16-byte query loads
    if (have_pool && ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15u))
      return HW_ERR_INVALID;
    CUtensorMap km, vm;
    std::memset(&km, 0, sizeof km);
    std::memset(&vm, 0, sizeof vm);
    if (have_pool) {
      if (!make_pool_map(&km, k_cache, d->cache_capacity, d->n_kv_heads, e4m3(d)) ||
          !make_pool_map(&vm, v_cache, d->cache_capacity, d->n_kv_heads, e4m3(d)))
        return cuda_fail(cudaErrorInvalidValue);
    }
    e = launch_decode_tc(a, km, vm, sms, s);
  } else {
    const int per_sm = decode_simt_ctas_per_sm(d->dtype, d->head_dim);
    int ctas = sms * (per_sm > 4 ? 4 : per_sm);
    if (ctas > max_ctas) ctas = max_ctas;
    e = launch_decode_simt(a, d->dtype, ctas, s);
  }
  return e == cudaSuccess ? HW_OK : cuda_fail(e);
}

// hw_attn_decode_planned and its E4M3 form, after their own checks.
static int planned_impl(const hw_attn_desc *d, const void *q, const void *k_cache,
                        const void *v_cache, const float *k_scale, const float *v_scale, void *out,
                        float *lse, void *workspace, size_t workspace_bytes, void *stream) {
  if (d->n_rows == 0) return HW_OK;
  if (!q || !out) return HW_ERR_INVALID;
  if (d->n_blocks > 0 && d->cache_capacity > 0 && (!k_cache || !v_cache)) return HW_ERR_INVALID;
  WorkspaceLayout L;
  int max_ctas = 0;
  const int st = check_workspace(d, workspace, workspace_bytes, &L, &max_ctas);
  if (st != HW_OK) return st;
  const MetaCopies m = meta_copies(*d, L, workspace);
  const uint8_t *plan = static_cast<const uint8_t *>(workspace) + L.plan_off;
  return decode_common(d, q, k_cache, v_cache, m.block_start, m.block_len, m.view_block,
                       m.view_offset, m.q_pos, m.q_to_kv, plan, out, lse, workspace, L, max_ctas,
                       stream, nullptr, nullptr, nullptr, nullptr,
                       limited(d) ? m.view_limit : nullptr, k_scale, v_scale);
}

}  // namespace hw

extern "C" {

int hw_attn_decode(const hw_attn_desc *d, const void *q, const void *k_cache, const void *v_cache,
                   const int32_t *block_start, const int32_t *block_len,
                   const int32_t *view_block, const int32_t *view_offset, const int32_t *q_pos,
                   const int32_t *q_to_kv, void *out, float *lse, void *workspace,
                   size_t workspace_bytes, void *stream) {
  int st = check_desc(d);
  if (st != HW_OK) return st;
  if (limited(d)) return HW_ERR_UNSUPPORTED;  // limits come with a plan
  if (e4m3(d)) return HW_ERR_UNSUPPORTED;     // E4M3 caches: planned, with their scales
  if (d->n_rows == 0) return HW_OK;
  if (!q || !out || !q_pos) return HW_ERR_INVALID;
  if (d->max_view_blocks > 0 && (!view_block || !view_offset)) return HW_ERR_INVALID;
  if (d->n_blocks > 0 && (!block_start || !block_len)) return HW_ERR_INVALID;
  // an empty pool (capacity 0) is never read and may be NULL
  if (d->n_blocks > 0 && d->cache_capacity > 0 && (!k_cache || !v_cache)) return HW_ERR_INVALID;
  WorkspaceLayout L;
  int max_ctas = 0;
  st = check_workspace(d, workspace, workspace_bytes, &L, &max_ctas);
  if (st != HW_OK) return st;
  // the tensor-core kernel runs from the workspace's plan cache: the plan of
  // the metadata the last call saw, rebuilt by the launch itself when this
  // call's metadata differs (one launch, no host round trip)
  return decode_common(d, q, k_cache, v_cache, block_start, block_len, view_block, view_offset,
                       q_pos, q_to_kv, nullptr, out, lse, workspace, L, max_ctas, stream, nullptr,
                       nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                       tensor_core_path(d));
}

static int plan_impl(const hw_attn_desc *d, const int32_t *block_start, const int32_t *block_len,
                     const int32_t *view_block, const int32_t *view_offset, const int32_t *q_pos,
                     const int32_t *q_to_kv, const int32_t *append_block,
                     const int32_t *append_pos, void *workspace, size_t workspace_bytes,
                     void *stream, const int32_t *view_limit = nullptr) {
  int st = check_desc(d);
  if (st != HW_OK) return st;
  if (d->n_rows == 0) return HW_OK;
  if (!q_pos) return HW_ERR_INVALID;
  if (d->max_view_blocks > 0 && (!view_block || !view_offset)) return HW_ERR_INVALID;
  if (d->n_blocks > 0 && (!block_start || !block_len)) return HW_ERR_INVALID;
  if ((append_block || view_limit) && !tensor_core_path(d)) return HW_ERR_UNSUPPORTED;
  if (limited(d) != (view_limit != nullptr)) return view_limit ? HW_ERR_INVALID : HW_ERR_UNSUPPORTED;
  WorkspaceLayout L;
  int max_ctas = 0;
  st = check_workspace(d, workspace, workspace_bytes, &L, &max_ctas);
  if (st != HW_OK) return st;
  DecodeArgs a;
  fill_args(a, d, L, workspace);
  a.block_start = block_start;
  a.block_len = block_len;
  a.view_block = view_block;
  a.view_offset = view_offset;
  a.q_pos = q_pos;
  a.q_to_kv = q_to_kv;
  a.append_block = append_block;
  a.append_pos = append_pos;
  a.view_limit = view_limit;
  const MetaCopies m = meta_copies(*d, L, workspace);
  PlanOut o;
  o.plan = tensor_core_path(d) ? static_cast<uint8_t *>(workspace) + L.plan_off : nullptr;
  o.view_block = m.view_block;
  o.view_offset = m.view_offset;
  o.q_pos = m.q_pos;
  o.q_to_kv = m.q_to_kv;
  o.block_start = m.block_start;
  o.block_len = m.block_len;
  o.append_block = m.append_block;
  o.append_pos = m.append_pos;
  o.view_limit = m.view_limit;
  o.records = device_sm_count();
  const cudaError_t e = launch_plan(a, o, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? HW_OK : cuda_fail(e);
}

int hw_attn_plan(const hw_attn_desc *d, const int32_t *block_start, const int32_t *block_len,
                 const int32_t *view_block, const int32_t *view_offset, const int32_t *q_pos,
                 const int32_t *q_to_kv, void *workspace, size_t workspace_bytes, void *stream) {
  return plan_impl(d, block_start, block_len, view_block, view_offset, q_pos, q_to_kv, nullptr,
                   nullptr, workspace, workspace_bytes, stream);
}

int hw_attn_plan_limited(const hw_attn_desc *d, const int32_t *block_start,
                         const int32_t *block_len, const int32_t *view_block,
                         const int32_t *view_offset, const int32_t *view_limit,
                         const int32_t *q_pos, const int32_t *q_to_kv, void *workspace,
                         size_t workspace_bytes, void *stream) {
  if (d && !(d->flags & HW_DESC_VIEW_LIMITS)) return HW_ERR_INVALID;
  if (d && d->n_rows > 0 && d->max_view_blocks > 0 && !view_limit) return HW_ERR_INVALID;
  return plan_impl(d, block_start, block_len, view_block, view_offset, q_pos, q_to_kv, nullptr,
                   nullptr, workspace, workspace_bytes, stream, view_limit);
}

int hw_attn_plan_append(const hw_attn_desc *d, const int32_t *block_start,
                        const int32_t *block_len, const int32_t *view_block,
                        const int32_t *view_offset, const int32_t *q_pos, const int32_t *q_to_kv,
                        const int32_t *append_block, const int32_t *append_pos, void *workspace,
                        size_t workspace_bytes, void *stream) {
  if (d && d->n_rows > 0 && (!append_block || !append_pos)) return HW_ERR_INVALID;
  return plan_impl(d, block_start, block_len, view_block, view_offset, q_pos, q_to_kv,
                   append_block, append_pos, workspace, workspace_bytes, stream);
}

int hw_attn_decode_planned(const hw_attn_desc *d, const void *q, const void *k_cache,
                           const void *v_cache, void *out, float *lse, void *workspace,
                           size_t workspace_bytes, void *stream) {
  int st = check_desc(d);
  if (st != HW_OK) return st;
  if (e4m3(d)) return HW_ERR_UNSUPPORTED;  // hw_attn_decode_planned_fp8 takes the scales
  return planned_impl(d, q, k_cache, v_cache, nullptr, nullptr, out, lse, workspace,
                      workspace_bytes, stream);
}

int hw_attn_decode_planned_fp8(const hw_attn_desc *d, const void *q, const void *k_cache,
                               const void *v_cache, const float *k_scale, const float *v_scale,
                               void *out, float *lse, void *workspace, size_t workspace_bytes,
                               void *stream) {
  int st = check_desc(d);
  if (st != HW_OK) return st;
  if (!e4m3(d)) return HW_ERR_INVALID;
  if (d->n_rows > 0 && (!k_scale || !v_scale)) return HW_ERR_INVALID;
  return planned_impl(d, q, k_cache, v_cache, k_scale, v_scale, out, lse, workspace,
                      workspace_bytes, stream);
}

int hw_plan_export(const hw_attn_desc *d, const void *workspace, size_t workspace_bytes,
                   int64_t *out, int32_t max_ctas, int32_t *n_ctas, void *stream) {
  int st = check_desc(d);
  if (st != HW_OK) return st;
  if (!out || !n_ctas || max_ctas <= 0) return HW_ERR_INVALID;
  if (!tensor_core_path(d)) return HW_ERR_UNSUPPORTED;
  WorkspaceLayout L;
  int max_grid = 0;
  st = check_workspace(d, const_cast<void *>(workspace), workspace_bytes, &L, &max_grid);
  if (st != HW_OK) return st;
  const size_t bytes = kPlanHeaderBytes + plan_shared_bytes() +
                       static_cast<size_t>(device_sm_count()) * plan_cta_bytes();
  std::vector<uint8_t> host(bytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess)
    e = cudaMemcpy(host.data(), static_cast<const uint8_t *>(workspace) + L.plan_off, bytes,
                   cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  const int grid = plan_export_records(host.data(), out, max_ctas);
  if (grid < 0) return HW_ERR_INVALID;
  *n_ctas = grid;
  return HW_OK;
}

// hw_attn_append_decode_planned and its E4M3 form, after their own checks.
static int append_impl(const hw_attn_desc *d, const void *q, const void *k_new, const void *v_new,
                       void *k_cache, void *v_cache, const float *k_scale, const float *v_scale,
                       void *out, float *lse, void *workspace, size_t workspace_bytes,
                       void *stream) {
  if (d->n_rows == 0) return HW_OK;
  if (!tensor_core_path(d)) return HW_ERR_UNSUPPORTED;
  if (!q || !out || !k_new || !v_new) return HW_ERR_INVALID;
  if (d->n_blocks > 0 && d->cache_capacity > 0 && (!k_cache || !v_cache)) return HW_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15u)
    return HW_ERR_INVALID;  // 16-byte loads of the new rows
  WorkspaceLayout L;
  int max_ctas = 0;
  const int st = check_workspace(d, workspace, workspace_bytes, &L, &max_ctas);
  if (st != HW_OK) return st;
  const MetaCopies m = meta_copies(*d, L, workspace);
  const uint8_t *plan = static_cast<const uint8_t *>(workspace) + L.plan_off;
  return decode_common(d, q, k_cache, v_cache, m.block_start, m.block_len, m.view_block,
                       m.view_offset, m.q_pos, m.q_to_kv, plan, out, lse, workspace, L, max_ctas,
                       stream, m.append_block, m.append_pos, k_new, v_new, nullptr, k_scale,
                       v_scale);
}

int hw_attn_append_decode_planned(const hw_attn_desc *d, const void *q, const void *k_new,
                                  const void *v_new, void *k_cache, void *v_cache, void *out,
                                  float *lse, void *workspace, size_t workspace_bytes,
                                  void *stream) {
  int st = check_desc(d);
  if (st != HW_OK) return st;
  if (limited(d) || e4m3(d)) return HW_ERR_UNSUPPORTED;  // E4M3: the _fp8 form takes the scales
  return append_impl(d, q, k_new, v_new, k_cache, v_cache, nullptr, nullptr, out, lse, workspace,
                     workspace_bytes, stream);
}

int hw_attn_append_decode_planned_fp8(const hw_attn_desc *d, const void *q, const void *k_new,
                                      const void *v_new, void *k_cache, void *v_cache,
                                      const float *k_scale, const float *v_scale, void *out,
                                      float *lse, void *workspace, size_t workspace_bytes,
                                      void *stream) {
  int st = check_desc(d);
  if (st != HW_OK) return st;
  if (limited(d)) return HW_ERR_UNSUPPORTED;
  if (!e4m3(d)) return HW_ERR_INVALID;
  if (d->n_rows > 0 && (!k_scale || !v_scale)) return HW_ERR_INVALID;
  return append_impl(d, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, out, lse, workspace,
                     workspace_bytes, stream);
}

static_assert(kMaxCommits == HW_MAX_COMMITS, "commit table size");

// Checks and launch of n commits (hw_block_commit: n = 1).
static int commit_impl(int32_t dtype, int32_t n_layers, int32_t n_kv_heads, int32_t head_dim,
                       double rope_theta, const void *k_src, const void *v_src,
                       int64_t src_capacity, void *k_dst, void *v_dst, int64_t dst_capacity,
                       int32_t n, const int32_t *src_begin, const int32_t *n_tokens,
                       const int32_t *dst_offset, const int32_t *pos_delta, void *stream) {
  if (dtype != HW_F32 && dtype != HW_BF16 && dtype != HW_FP8_E4M3) return HW_ERR_INVALID;
  if (n < 0 || n > HW_MAX_COMMITS) return HW_ERR_INVALID;
  if (n > 0 && (!src_begin || !n_tokens || !dst_offset || !pos_delta)) return HW_ERR_INVALID;
  if (n_layers < 0 || n_kv_heads <= 0 || src_capacity < 0 || dst_capacity < 0) return HW_ERR_INVALID;
  for (int c = 0; c < n; ++c)
    if (n_tokens[c] < 0 || src_begin[c] < 0 || dst_offset[c] < 0) return HW_ERR_INVALID;
  if (!(rope_theta > 1.0) || !std::isfinite(rope_theta)) return HW_ERR_INVALID;
  const int esz = dtype == HW_F32 ? 4 : dtype == HW_FP8_E4M3 ? 1 : 2;
  const int epv = 16 / esz;
  if (head_dim <= 0 || head_dim > 128 || head_dim % (2 * epv) != 0) return HW_ERR_UNSUPPORTED;
  int64_t tokens = 0;
  for (int c = 0; c < n; ++c) tokens += n_tokens[c];
  if (n_layers == 0 || tokens == 0) return HW_OK;
  if (!k_src || !v_src || !k_dst || !v_dst) return HW_ERR_INVALID;
  for (int c = 0; c < n; ++c) {
    if (static_cast<int64_t>(src_begin[c]) + n_tokens[c] > src_capacity) return HW_ERR_CAPACITY;
    if (static_cast<int64_t>(dst_offset[c]) + n_tokens[c] > dst_capacity) return HW_ERR_CAPACITY;
  }
  for (const void *p : {k_src, v_src, static_cast<const void *>(k_dst), static_cast<const void *>(v_dst)})
    if (reinterpret_cast<uintptr_t>(p) & 15u) return HW_ERR_INVALID;

  // Overlap: the address spans of the pools; spans that meet are only allowed
  // when they are the same pool (same base and capacity) and every destination
  // token range is disjoint from every source range.  Destination ranges never
  // meet one another.
  auto disjoint = [](int64_t a0, int64_t na, int64_t b0, int64_t nb) {
    return na == 0 || nb == 0 || a0 + na <= b0 || b0 + nb <= a0;
  };
  for (int c = 0; c < n; ++c)
    for (int e = c + 1; e < n; ++e)
      if (!disjoint(dst_offset[c], n_tokens[c], dst_offset[e], n_tokens[e])) return HW_ERR_OVERLAP;
  bool tokens_disjoint = true;
  for (int c = 0; c < n; ++c)
    for (int e = 0; e < n; ++e)
      if (!disjoint(dst_offset[c], n_tokens[c], src_begin[e], n_tokens[e])) tokens_disjoint = false;
  const int64_t row = static_cast<int64_t>(head_dim) * esz;
  const int64_t src_span = static_cast<int64_t>(n_layers) * n_kv_heads * src_capacity * row;
  const int64_t dst_span = static_cast<int64_t>(n_layers) * n_kv_heads * dst_capacity * row;
  auto meets = [](const void *a, int64_t na, const void *b, int64_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
  };
  for (const void *d : {static_cast<const void *>(k_dst), static_cast<const void *>(v_dst)}) {
    for (const void *sp : {k_src, v_src}) {
      if (!meets(d, dst_span, sp, src_span)) continue;
      if (d == sp && src_capacity == dst_capacity && tokens_disjoint) continue;
      return HW_ERR_OVERLAP;
    }
  }
  if (meets(k_dst, dst_span, v_dst, dst_span)) return HW_ERR_OVERLAP;

  CommitArgs a;
  std::memset(&a, 0, sizeof a);
  a.k_src = k_src;
  a.v_src = v_src;
  a.k_dst = k_dst;
  a.v_dst = v_dst;
  a.src_capacity = src_capacity;
  a.dst_capacity = dst_capacity;
  a.n_layers = n_layers;
  a.n_kv_heads = n_kv_heads;
  a.head_dim = head_dim;
  a.n_commits = n;
  for (int c = 0; c < n; ++c) {
    a.src_begin[c] = src_begin[c];
    a.dst_offset[c] = dst_offset[c];
    a.n_tokens[c] = n_tokens[c];
    a.delta[c] = pos_delta[c];
  }
  rope_phase_table(head_dim, rope_theta, a.phase);
  const cudaError_t e = launch_commit(a, dtype, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? HW_OK : cuda_fail(e);
}

int hw_block_commit(int32_t dtype, int32_t n_layers, int32_t n_kv_heads, int32_t head_dim,
                    double rope_theta, const void *k_src, const void *v_src, int64_t src_capacity,
                    int32_t src_begin, int32_t n_tokens, void *k_dst, void *v_dst,
                    int64_t dst_capacity, int32_t dst_offset, int32_t pos_delta, void *stream) {
  return commit_impl(dtype, n_layers, n_kv_heads, head_dim, rope_theta, k_src, v_src,
                     src_capacity, k_dst, v_dst, dst_capacity, 1, &src_begin, &n_tokens,
                     &dst_offset, &pos_delta, stream);
}

int hw_block_commit_many(int32_t dtype, int32_t n_layers, int32_t n_kv_heads, int32_t head_dim,
                         double rope_theta, const void *k_src, const void *v_src,
                         int64_t src_capacity, void *k_dst, void *v_dst, int64_t dst_capacity,
                         int32_t n_commits, const int32_t *src_begin, const int32_t *n_tokens,
                         const int32_t *dst_offset, const int32_t *pos_delta, void *stream) {
  return commit_impl(dtype, n_layers, n_kv_heads, head_dim, rope_theta, k_src, v_src,
                     src_capacity, k_dst, v_dst, dst_capacity, n_commits, src_begin, n_tokens,
                     dst_offset, pos_delta, stream);
}

int hw_workspace_status(void *workspace, int32_t *flags, void *stream) {
  if (!workspace) return HW_ERR_WORKSPACE;
  if (!flags) return HW_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  int32_t v = 0;
  e = cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (v != 0) {
    e = cudaMemset(workspace, 0, sizeof v);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  *flags = v;
  return HW_OK;
}

int hw_views(int32_t layout, int32_t n_problems, int32_t n_workers, const int32_t *block_len,
             int32_t *view_block, int32_t *view_offset, int32_t *q_pos) {
  if (layout != HW_LAYOUT_COMBINED && layout != HW_LAYOUT_INTERLEAVED &&
      layout != HW_LAYOUT_CONTIGUOUS)
    return HW_ERR_INVALID;
  if (n_problems < 0 || n_workers <= 0) return HW_ERR_INVALID;
  if (n_workers > HW_MAX_REFS_PER_BLOCK) return HW_ERR_UNSUPPORTED;  // W rows name each block
  if (n_problems == 0) return HW_OK;
  if (!block_len || !view_block || !view_offset || !q_pos) return HW_ERR_INVALID;
  const int W = n_workers, V = n_workers + 1;
  const bool others = layout != HW_LAYOUT_INTERLEAVED;
  for (int p = 0; p < n_problems; ++p) {
    const int base = p * (W + 1);
    for (int w = 0; w < W; ++w) {
      const int row = p * W + w;
      int v = 0;
      int64_t pos = 0;
      auto put = [&](int b) {
        view_block[row * V + v] = b;
        view_offset[row * V + v] = static_cast<int32_t>(pos);
        pos += block_len[b];
        ++v;
      };
      put(base);                                    // common cache
      if (others)
        for (int o = 0; o < W; ++o)
          if (o != w) put(base + 1 + o);            // others' unfinished steps, worker order
      put(base + 1 + w);                            // own unfinished step
      for (; v < V; ++v) {                          // unused entries
        view_block[row * V + v] = -1;
        view_offset[row * V + v] = 0;
      }
      if (pos > INT32_MAX) return HW_ERR_INVALID;
      q_pos[row] = static_cast<int32_t>(pos);
    }
  }
  return HW_OK;
}

int hw_views_chunked(int32_t layout, int32_t n_problems, int32_t n_workers, int32_t chunk,
                     const int32_t *block_len, int32_t *view_block, int32_t *view_offset,
                     int32_t *view_limit, int32_t *q_pos) {
  if (chunk <= 0 || n_problems < 0 || n_workers <= 0) return HW_ERR_INVALID;
  // W * chunk rows name each block of a problem
  if (static_cast<int64_t>(n_workers) * chunk > HW_MAX_REFS_PER_BLOCK) return HW_ERR_UNSUPPORTED;
  if (n_problems == 0) return HW_OK;
  if (!block_len || !view_block || !view_offset || !view_limit || !q_pos) return HW_ERR_INVALID;
  const int W = n_workers, V = n_workers + 1, T = chunk;
  for (int p = 0; p < n_problems; ++p)
    for (int w = 0; w < W; ++w)
      if (block_len[p * (W + 1) + 1 + w] < T) return HW_ERR_INVALID;
  // each problem's one-row-per-worker views, then T rows per worker
  std::vector<int32_t> vb(W * V), vo(W * V), qp(W);
  for (int p = 0; p < n_problems; ++p) {
    const int base = p * (W + 1);
    const int st = hw_views(layout, 1, W, block_len + base, vb.data(), vo.data(), qp.data());
    if (st != HW_OK) return st;
    for (int w = 0; w < W; ++w) {
      const int n = block_len[base + 1 + w];
      for (int t = 0; t < T; ++t) {
        const int64_t r = (static_cast<int64_t>(p) * W + w) * T + t;
        for (int v = 0; v < V; ++v) {
          const int b = vb[w * V + v];
          view_block[r * V + v] = b < 0 ? -1 : base + b;
          view_offset[r * V + v] = vo[w * V + v];
          view_limit[r * V + v] = -1;
          if (b == 1 + w) {  // its own block: up to its own token
            view_limit[r * V + v] = n - T + t + 1;
            q_pos[r] = vo[w * V + v] + n - T + t;
          }
        }
      }
    }
  }
  return HW_OK;
}

int hw_views_combined(int32_t n_problems, int32_t n_workers, const int32_t *block_len,
                      int32_t *view_block, int32_t *view_offset, int32_t *q_pos) {
  return hw_views(HW_LAYOUT_COMBINED, n_problems, n_workers, block_len, view_block, view_offset,
                  q_pos);
}

int hw_last_cuda_error(void) { return g_last_cuda_error; }

const char *hw_status_string(int status) {
  switch (status) {
    case HW_OK: return "ok";
    case HW_ERR_INVALID: return "invalid argument";
    case HW_ERR_UNSUPPORTED: return "unsupported configuration";
    case HW_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case HW_ERR_CAPACITY: return "range past the pool capacity";
    case HW_ERR_OVERLAP: return "source and destination overlap";
    case HW_ERR_CUDA: return "CUDA runtime error";
    case HW_ERR_DEVICE: return "device-side metadata error";
    default: return "unknown status";
  }
}

}  // extern "C"
