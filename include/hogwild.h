/*
 * hogwild.h - C ABI of libhogwild: concurrent decode attention over a KV cache
 * that W workers share, and the block commit that moves a finished step into
 * the shared history (Hogwild! Inference), for NVIDIA GB300 (sm_103a).
 *
 * Sources (page title, then section / equation):
 *  - "Hogwild! Inference: Parallel LLM Generation via Concurrent Attention"
 *    (paper-notes page): key design 1 (shared KV cache; the query-rotation
 *    equation rho(q,i_q)[rho(A,i_k^A) (+) rho(B,i_k^B) ...] =
 *    rho(q,i_q-i_k^A)A (+) rho(q,i_q-i_k^B)B ...), key design 2 (combined cache
 *    layout: common cache, other workers' unfinished steps in worker order,
 *    the current worker's own step; a finished step is rotated and moved into
 *    the shared history), implementation notes (a Flash-Decoding style kernel
 *    over many cache blocks; each block stores its KV at block-local positions
 *    and the query rotation supplies the real position).
 *  - omica.com.cn article on Hogwild! Inference: section 2.1 (rotate_query:
 *    frequencies 1/base^(2i/dim), q*cos + rotate_half(q)*sin), section 3.1
 *    (a cache block carries its storage, start and current length), section
 *    3.2 (blockwise scores q_rot.k/sqrt(dim), one softmax across all blocks;
 *    KV work split evenly over the SMs, partial results merged).
 *
 * Conventions shared by every entry point
 *  - The caller owns all memory.  No entry point allocates device memory.
 *  - "dev" marks device pointers, "host" host pointers.  `stream` is a
 *    cudaStream_t passed as void* (NULL = the legacy default stream).  Work is
 *    enqueued on that stream; nothing synchronises unless stated.
 *  - KV pool layout (one K pool and one V pool per layer): [Hkv][capacity][D],
 *    D contiguous, element type `dtype`; a block is the token range
 *    [block_start, block_start + block_len) of every head.  Keys are stored
 *    already rotated by RoPE at block-local positions 0 .. len-1.
 *  - Limits of that layout: every block of a call lives in that one pair of
 *    pools (the kernels address it through one TMA descriptor per pool), so a
 *    cache whose blocks are separate allocations - a per-block pointer, as in
 *    the article's CacheBlock - is laid out in one pool (or copied into one)
 *    before the call; and block_start, block_len and the capacity are 32-bit:
 *    at most 2^31 - 1 tokens per head and pool (larger capacities return
 *    HW_ERR_UNSUPPORTED).
 *  - RoPE pairs element i with element i + D/2 (rotate_half) at frequency
 *    w_i = rope_theta^(-2i/D).
 *  - Every call returns an hw_status.  Argument errors are found on the host
 *    before anything is enqueued.  Errors in device-resident metadata are
 *    recorded in the workspace (see hw_workspace_status) and the affected
 *    blocks are skipped; no kernel traps, faults or waits without a bound.
 */
#ifndef HOGWILD_H
#define HOGWILD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HW_OK = 0,
  HW_ERR_INVALID = -1,     /* bad argument: null pointer, negative size, bad dtype */
  HW_ERR_UNSUPPORTED = -2, /* valid but outside what the kernels handle (see limits) */
  HW_ERR_WORKSPACE = -3,   /* workspace missing, too small or not 256-byte aligned */
  HW_ERR_CAPACITY = -4,    /* commit would write past the destination capacity */
  HW_ERR_OVERLAP = -5,     /* commit source and destination memory overlap */
  HW_ERR_CUDA = -6,        /* a CUDA runtime call failed (hw_last_cuda_error) */
  HW_ERR_DEVICE = -7       /* device-side metadata check failed (hw_workspace_status) */
} hw_status;

/*
 * HW_FP8_E4M3: the K and V pools hold E4M3 codes (1 byte per element; a
 * cached value is the code's value times its kv head's scale, k_scale[h] or
 * v_scale[h]); q and out stay bf16.  head_dim 128; decoded by
 * hw_attn_plan + hw_attn_decode_planned_fp8 and committed by hw_block_commit
 * (the other decode calls return HW_ERR_UNSUPPORTED for it).
 */
typedef enum { HW_F32 = 0, HW_BF16 = 1, HW_FP8_E4M3 = 2 } hw_dtype;

/* Device-side error bits reported by hw_workspace_status. */
enum {
  HW_DEV_BAD_BLOCK = 1,     /* a view names a block id outside [-1, n_blocks) */
  HW_DEV_BAD_RANGE = 2,     /* block_start/len negative or past the pool capacity */
  HW_DEV_BAD_HEADMAP = 4,   /* q_to_kv entry out of range or groups of unequal size */
  HW_DEV_TOO_MANY_REFS = 8, /* more than HW_MAX_REFS_PER_BLOCK view entries name one block
                               (it is skipped), or a (row, q head) gathers more partial
                               results than a merge holds */
  HW_DEV_TIMEOUT = 16,      /* a bounded in-kernel wait expired; results are invalid */
  HW_DEV_BAD_PLAN = 32      /* hw_attn_decode_planned found no plan for this description */
};

/* Limits of this build. */
#define HW_MAX_BLOCKS 256          /* blocks per decode call */
#define HW_MAX_VIEW_BLOCKS 64      /* max_view_blocks */
#define HW_MAX_VIEW_ENTRIES 4096   /* n_rows * max_view_blocks */
/* Query columns one tile serves: a block's columns are (view references to
 * it) x (Hq/Hkv).  A block with more is split into column groups of
 * HW_MAX_QHEADS_PER_BLOCK / (Hq/Hkv) references each, in view-entry order,
 * and each group reads the block's tiles once. */
#define HW_MAX_QHEADS_PER_BLOCK 32
#define HW_MAX_REFS_PER_BLOCK 255  /* view entries naming one block */
#define HW_MAX_Q_HEADS 256         /* n_q_heads */

/* Host-side description of one decode call (all scalars, host memory). */
typedef struct {
  int32_t n_rows;          /* query tokens: one per (problem, worker), >= 0 */
  int32_t n_q_heads;       /* Hq, <= HW_MAX_Q_HEADS */
  int32_t n_kv_heads;      /* Hkv, Hq % Hkv == 0 */
  int32_t head_dim;        /* D: 64 or 128 (bf16 tensor-core path: 128) */
  int32_t n_blocks;        /* entries of block_start / block_len, <= HW_MAX_BLOCKS */
  int32_t max_view_blocks; /* V: width of the per-row view tables */
  int64_t cache_capacity;  /* tokens per head in the K and V pools */
  int32_t dtype;           /* hw_dtype of q, pools and out */
  double rope_theta;       /* RoPE base, > 1 */
  float scale;             /* softmax scale, usually 1/sqrt(D) */
  int32_t flags;           /* HW_DESC_* bits, 0 for none */
} hw_attn_desc;

/*
 * The step's plan carries per-view-entry token limits.  A descriptor with this
 * flag is planned by hw_attn_plan_limited and decoded by
 * hw_attn_decode_planned (bf16) or hw_attn_decode_planned_fp8 (HW_FP8_E4M3)
 * only, head_dim 128: the other decode and plan calls return
 * HW_ERR_UNSUPPORTED for it, and hw_attn_plan_limited returns
 * HW_ERR_INVALID without it.  (The limits run in their own kernel, so that
 * steps without limits pay nothing for them.)
 */
#define HW_DESC_VIEW_LIMITS 1

/*
 * A promise from the caller about the work enqueued just before this call on
 * the same stream (a kernel, a copy, or the previous library call): it writes
 * neither the K/V pools, nor the metadata arrays or plan, that this call
 * reads.  q, out, lse and the workspace's other contents may be anything.
 * With the promise, a bf16 or E4M3 head_dim-128 decode starts while that work
 * finishes: it reads its plan (or builds it from the metadata) and loads its
 * first K/V tiles before the previous kernel has completed, and only its
 * reads of q and its writes wait for it.  In a decode step, set it on every
 * layer after the first one that follows a plan or commit call.  The promise
 * is not checked; breaking it gives results computed from stale K/V data or
 * metadata.  Ignored by the fp32 and head_dim-64 kernels.
 */
#define HW_DESC_EARLY_LOADS 2

/*
 * Bytes of workspace hw_attn_decode needs for `d` on the current device.
 * Writes the size to *bytes.  The workspace holds the error word, the merge
 * arrival counters and the per-split partial results (max, sum of exp,
 * unnormalised output) of the log-sum-exp merge.
 */
int hw_attn_decode_workspace_size(const hw_attn_desc *d, size_t *bytes);

/*
 * Zero a workspace (dev, `bytes` long) on `stream`.  Required once before the
 * first hw_attn_decode that uses it; each decode leaves its counters at zero
 * again for the next call.  A workspace's layout follows its description:
 * zero it again before using it with another one.
 */
int hw_workspace_init(void *workspace, size_t bytes, void *stream);

/*
 * Concurrent decode attention, one layer, one launch.
 *
 * For every row r (a worker's current token) and query head hq with kv head
 * g = q_to_kv ? q_to_kv[hq] : hq / (Hq/Hkv):
 *   for each view entry v (view_block[r][v] = b >= 0, len_b = block_len[b] > 0):
 *     q~ = rho(q[r][hq], q_pos[r] - view_offset[r][v])            (query rotation)
 *     s_j = scale * q~ . K[g][block_start[b] + j],  j < len_b       (block scores)
 *   out[r][hq] = sum_j softmax(s)_j V[g][block_start[b] + j]  over all entries
 *   lse[r][hq] = log sum_j exp(s_j)   (natural log; -inf and out = 0 if empty)
 *
 *  d            host  description (above)
 *  q            dev   [n_rows][Hq][D] dtype, un-rotated queries, 16-byte aligned
 *  k_cache      dev   [Hkv][capacity][D] dtype, keys rotated at block-local positions;
 *                     16-byte aligned; may be NULL when capacity is 0
 *  v_cache      dev   [Hkv][capacity][D] dtype, same rules
 *  block_start  dev   int32 [n_blocks], first pool token of each block
 *  block_len    dev   int32 [n_blocks], tokens in each block
 *  view_block   dev   int32 [n_rows][V], block ids in view order, -1 = unused slot
 *  view_offset  dev   int32 [n_rows][V], i_k^block: tokens before that block in
 *                     that row's view (any int32; the rotation uses i_q - offset)
 *  q_pos        dev   int32 [n_rows], i_q: the query's position in its view
 *  q_to_kv      dev   int32 [Hq] or NULL (grouped heads, hq / (Hq/Hkv))
 *  out          dev   [n_rows][Hq][D] dtype, any element-aligned address (rows
 *                     are written with vector stores when the address allows)
 *  lse          dev   float [n_rows][Hq] or NULL
 *  workspace    dev   >= hw_attn_decode_workspace_size bytes, 256-byte aligned,
 *                     zeroed once with hw_workspace_init; one call at a time
 *  stream       cudaStream_t as void*
 * The same metadata arrays can serve every layer of a step.  Calls that share
 * a workspace must be ordered on one stream.  Pool slots past a block's
 * length are never used in the result, whatever they hold.
 *
 * One launch.  The tensor-core kernel (bf16, head_dim 128) runs from a plan
 * of the work split that the workspace caches: the plan of the metadata the
 * last call on the workspace saw, compared word by word with this call's
 * arrays (contents, not addresses).  A call whose metadata differs - the
 * first layer of a new step - builds the plan in the kernel and caches it
 * for the calls after it.  Which call to use: for a step of many layers,
 * hw_attn_decode on the step's arrays runs within a few percent of
 * hw_attn_plan + hw_attn_decode_planned (which also lets the caller reuse or
 * free its arrays after planning); the planned calls are the ones that take
 * appends, view limits and E4M3 caches.
 */
int hw_attn_decode(const hw_attn_desc *d, const void *q, const void *k_cache, const void *v_cache,
                   const int32_t *block_start, const int32_t *block_len,
                   const int32_t *view_block, const int32_t *view_offset, const int32_t *q_pos,
                   const int32_t *q_to_kv, void *out, float *lse, void *workspace,
                   size_t workspace_bytes, void *stream);

/*
 * The metadata of a decode step, planned once for every layer of the step.
 *
 * In a decode step every layer attends the same views: the block table,
 * the views and positions are per step, only q, K and V change per layer.
 * hw_attn_plan copies the metadata (same arguments and layouts as
 * hw_attn_decode) into `workspace` and, for the tensor-core kernel (bf16 or
 * E4M3 caches, head_dim 128),
 * precomputes the work split, each CTA's first segments and the merge lists
 * there.  hw_attn_decode_planned then runs one layer against that plan, with
 * results identical to hw_attn_decode on the same metadata.  The plan holds a
 * copy of the metadata: the caller may change its own arrays after planning.
 * A plan stays valid until the next hw_attn_plan on the workspace; planned
 * calls must use the same description (checked on the device: a mismatch or
 * a missing plan sets HW_DEV_BAD_PLAN, see hw_workspace_status, and leaves
 * out and lse untouched).  Both enqueue work on `stream` only; the plan is
 * seen by calls enqueued after it on the same stream.
 *
 * A descriptor with HW_DESC_VIEW_LIMITS is planned by hw_attn_plan_limited
 * instead (hw_attn_plan returns HW_ERR_UNSUPPORTED for it); HW_FP8_E4M3
 * caches are planned here (with appends: hw_attn_plan_append) and decoded by
 * hw_attn_decode_planned_fp8 (or hw_attn_append_decode_planned_fp8), while
 * hw_attn_decode_planned returns HW_ERR_UNSUPPORTED for them.
 *
 * Not in the Hogwild! notes, which describe one attention call per layer:
 * this is the usual split of a decode kernel's scheduling from its runs.
 */
int hw_attn_plan(const hw_attn_desc *d, const int32_t *block_start, const int32_t *block_len,
                 const int32_t *view_block, const int32_t *view_offset, const int32_t *q_pos,
                 const int32_t *q_to_kv, void *workspace, size_t workspace_bytes, void *stream);

int hw_attn_decode_planned(const hw_attn_desc *d, const void *q, const void *k_cache,
                           const void *v_cache, void *out, float *lse, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * The step's new tokens written and the layer decoded in one launch.  Every
 * layer of a decode step first appends each worker's new token to its own
 * block - the key stored rotated at its block-local position, like every
 * key of the cache (the Hogwild! notes: keys are kept at positions
 * 0..len-1 of their block) - then attends.
 *
 * hw_attn_plan_append is hw_attn_plan with the step's appends:
 *  append_block  dev  int32 [n_rows], the block row r appends to, -1 = none
 *  append_pos    dev  int32 [n_rows], the block-local position of its token;
 *                     the plan's block_len must already count it:
 *                     0 <= append_pos[r] < block_len[append_block[r]]
 * (copied into the plan like the rest of the metadata; a row whose append
 * falls outside its block sets HW_DEV_BAD_RANGE and is not appended).
 * hw_attn_append_decode_planned then, for every row r with an append and
 * every kv head h,
 *   K[h][block_start[b] + p] = rho(k_new[r][h], p)     (b, p = append_block[r], append_pos[r])
 *   V[h][block_start[b] + p] = v_new[r][h]
 * with k_new, v_new dev [n_rows][Hkv][D] in the cache dtype, the key rotated
 * in fp32 and rounded once to the dtype (nearest, ties to even), and then
 * decodes as hw_attn_decode_planned does, the new tokens included.  Each
 * token is written by the CTA that streams the tile holding it, before that
 * tile is loaded.  A plan from hw_attn_plan has no appends (nothing is
 * written); hw_attn_decode_planned on a plan with appends writes nothing
 * either.  bf16 with head_dim 128 only (HW_ERR_UNSUPPORTED otherwise).
 */
/*
 * Chunked multi-token queries: a worker's chunk of T query tokens is T rows
 * with the same view, row t at position q_pos + t, and within the worker's
 * own block - which holds the chunk's own tokens - each row sees only the
 * tokens up to its own (causal order).  hw_attn_plan_limited is hw_attn_plan
 * with a per-view-entry limit:
 *  view_limit  dev  int32 [n_rows][V]: row r attends only the first
 *                   min(view_limit[r][v], len) tokens of block view_block[r][v];
 *                   a negative value: the whole block
 * (copied into the plan).  hw_attn_decode_planned then applies the limits.
 * bf16 with head_dim 128 only (HW_ERR_UNSUPPORTED otherwise).
 */
/*
 * hw_attn_decode_planned for HW_FP8_E4M3 caches (E4M3 KV storage with
 * per-head scales; the omica.com.cn article on Hogwild! Inference, section 6,
 * names FP8 attention as future work): k_cache and v_cache hold E4M3
 * codes, [Hkv][capacity][128] bytes; k_scale, v_scale (dev, float [Hkv]):
 * a cached key or value is its code's value times its kv head's scale.  q,
 * out and lse as in hw_attn_decode; the plan comes from hw_attn_plan with the
 * same descriptor.  The result is attention over the decoded, scaled cache.
 * HW_ERR_INVALID for another dtype or null scales.
 */
int hw_attn_decode_planned_fp8(const hw_attn_desc *d, const void *q, const void *k_cache,
                               const void *v_cache, const float *k_scale, const float *v_scale,
                               void *out, float *lse, void *workspace, size_t workspace_bytes,
                               void *stream);

int hw_attn_plan_limited(const hw_attn_desc *d, const int32_t *block_start,
                         const int32_t *block_len, const int32_t *view_block,
                         const int32_t *view_offset, const int32_t *view_limit,
                         const int32_t *q_pos, const int32_t *q_to_kv, void *workspace,
                         size_t workspace_bytes, void *stream);

int hw_attn_plan_append(const hw_attn_desc *d, const int32_t *block_start,
                        const int32_t *block_len, const int32_t *view_block,
                        const int32_t *view_offset, const int32_t *q_pos, const int32_t *q_to_kv,
                        const int32_t *append_block, const int32_t *append_pos, void *workspace,
                        size_t workspace_bytes, void *stream);

int hw_attn_append_decode_planned(const hw_attn_desc *d, const void *q, const void *k_new,
                                  const void *v_new, void *k_cache, void *v_cache, void *out,
                                  float *lse, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * hw_attn_append_decode_planned for HW_FP8_E4M3 caches: each new token's key
 * (bf16, rotated at its block-local position in fp32) divided by its kv
 * head's k_scale and its value divided by v_scale, each rounded to the nearest
 * E4M3 code (ties to even, saturating at 448), then the layer decoded as
 * hw_attn_decode_planned_fp8 does.  Planned by hw_attn_plan_append with the
 * same descriptor.  HW_ERR_INVALID for another dtype or null scales.
 */
int hw_attn_append_decode_planned_fp8(const hw_attn_desc *d, const void *q, const void *k_new,
                                      const void *v_new, void *k_cache, void *v_cache,
                                      const float *k_scale, const float *v_scale, void *out,
                                      float *lse, void *workspace, size_t workspace_bytes,
                                      void *stream);

/*
 * For tests: the work split of the plan in `workspace` (bf16 head_dim-128
 * kernel; synchronises `stream`).  Per CTA c < *n_ctas, 15 int64 at
 * out[15 c ..]: its unit range [u0, u1) (units: 128-token tiles of one
 * (block, column group, kv head), kv-head-major, then block, then group,
 * then tile; see HW_MAX_QHEADS_PER_BLOCK), the number of first tiles the
 * plan decodes (min(3, u1 - u0)), their first cache rows, kv heads, segment
 * flags (1: starts its segment within the range, 2: ends it) and column
 * groups, 3 each.  out holds max_ctas records.  HW_ERR_INVALID when the
 * workspace holds no plan.
 */
int hw_plan_export(const hw_attn_desc *d, const void *workspace, size_t workspace_bytes,
                   int64_t *out, int32_t max_ctas, int32_t *n_ctas, void *stream);

/*
 * Size of the fixed scratch array hw_attn_decode_noalloc uses (32 MiB): it
 * covers descriptions whose hw_attn_decode_workspace_size is at most this,
 * e.g. up to about 1450 (block, kv head) pairs with head_dim 128.
 */
#define HW_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * hw_attn_decode for callers that cannot allocate device memory - code that
 * runs inside an allocator or memory pool, plugins whose host runtime owns
 * every device buffer, processes that forbid allocation after start-up.  The
 * pages describe no such variant; it has no counterpart there.
 *
 * Same arguments, meaning and result as hw_attn_decode, without the
 * workspace: the call uses a scratch array of HW_NOALLOC_SCRATCH_BYTES that
 * the library itself holds on every GPU that loads it, until the process
 * exits.  No call allocates or frees memory.
 *  - The first call on a device finds the array's device address and zeroes
 *    it with a synchronous cudaMemset; make that first call before any stream
 *    capture.  Each call then clears the scratch's counters on `stream`.
 *  - Every call shares the one array: calls whose work overlaps on the GPU
 *    (other streams, other host threads) race and give wrong results.
 *    Order them on one stream.
 *  - Returns HW_ERR_WORKSPACE, before enqueuing anything, when `d` needs more
 *    scratch than HW_NOALLOC_SCRATCH_BYTES; use hw_attn_decode then.
 *  - Device-side metadata errors (HW_DEV_*) are recorded in the scratch, in
 *    place of a workspace: hw_noalloc_status reads and clears them.
 *  - The array's device address is looked up once per device ordinal and kept:
 *    calling after cudaDeviceReset (or any reset of the device's primary
 *    context) in the same process is not supported.
 */
int hw_attn_decode_noalloc(const hw_attn_desc *d, const void *q, const void *k_cache,
                           const void *v_cache, const int32_t *block_start,
                           const int32_t *block_len, const int32_t *view_block,
                           const int32_t *view_offset, const int32_t *q_pos,
                           const int32_t *q_to_kv, void *out, float *lse, void *stream);

/*
 * The device error bits (HW_DEV_*, 0 = none) that hw_attn_decode_noalloc calls
 * on the current device recorded since the last read, into *flags, and
 * cleared; like hw_workspace_status, for callers that cannot allocate: it
 * synchronises `stream` and uses plain copies to and from host memory, so it
 * allocates nothing.  0 when no such call ran on the device yet.
 */
int hw_noalloc_status(int32_t *flags, void *stream);

/*
 * Block commit over n_layers layers in one launch (a finished step moves
 * into the shared history; key design 2 of the Hogwild! notes):
 *   K_dst[l][h][dst_offset + j] = rho(K_src[l][h][src_begin + j], pos_delta)
 *   V_dst[l][h][dst_offset + j] = V_src[l][h][src_begin + j]        (bit copy)
 * for l < n_layers, h < Hkv, j < n_tokens.  Pools are [n_layers][Hkv][cap][D]
 * (layer stride Hkv*cap*D elements).  Keys are rotated in fp32 from the stored
 * values and rounded once to dtype (nearest, ties to even); pos_delta may be
 * negative; pos_delta = 0 is a bit copy.  Nothing outside the destination
 * range is written.  Block lengths are the caller's to update.
 *
 *  k_src, v_src   dev  source pools, src_capacity tokens per head
 *  k_dst, v_dst   dev  destination pools, dst_capacity tokens per head
 * Errors: HW_ERR_CAPACITY if a range leaves its pool; HW_ERR_OVERLAP if any
 * destination range shares memory with a source range or with the other
 * destination.  head_dim must be a multiple of 16 bytes / element size * 2.
 */
int hw_block_commit(int32_t dtype, int32_t n_layers, int32_t n_kv_heads, int32_t head_dim,
                    double rope_theta, const void *k_src, const void *v_src, int64_t src_capacity,
                    int32_t src_begin, int32_t n_tokens, void *k_dst, void *v_dst,
                    int64_t dst_capacity, int32_t dst_offset, int32_t pos_delta, void *stream);

/*
 * Several finished steps committed in one launch (workers that finish a step
 * together join the shared history in one go, in the caller's order).
 * Commit c applies the hw_block_commit formula to its own range:
 *   K_dst[l][h][dst_offset[c] + j] = rho(K_src[l][h][src_begin[c] + j], pos_delta[c])
 *   V_dst[l][h][dst_offset[c] + j] = V_src[l][h][src_begin[c] + j]
 * for j < n_tokens[c], with the pools, rounding and layer stride of
 * hw_block_commit.  src_begin, n_tokens, dst_offset, pos_delta: host arrays of
 * n_commits entries, 0 <= n_commits <= HW_MAX_COMMITS.
 * Errors: those of hw_block_commit for each commit, and HW_ERR_OVERLAP when
 * two destination ranges meet.
 */
#define HW_MAX_COMMITS 64
int hw_block_commit_many(int32_t dtype, int32_t n_layers, int32_t n_kv_heads, int32_t head_dim,
                         double rope_theta, const void *k_src, const void *v_src,
                         int64_t src_capacity, void *k_dst, void *v_dst, int64_t dst_capacity,
                         int32_t n_commits, const int32_t *src_begin, const int32_t *n_tokens,
                         const int32_t *dst_offset, const int32_t *pos_delta, void *stream);

/*
 * Synchronises `stream`, reads and clears the device error bits of a
 * workspace (HW_DEV_* flags, 0 = none) into *flags.
 */
int hw_workspace_status(void *workspace, int32_t *flags, void *stream);

/*
 * Host helper: the combined layout of key design 2 for n_problems problems of
 * n_workers workers.  Block ids: problem p owns p*(W+1) (common) and
 * p*(W+1)+1+w (worker w).  Worker w's view: common, the other workers in id
 * order, itself; view_offset = tokens before each block in that view; q_pos =
 * the view's total length.  All arrays host: block_len [n_problems*(W+1)],
 * view_block and view_offset [n_problems*W][W+1], q_pos [n_problems*W].
 */
int hw_views_combined(int32_t n_problems, int32_t n_workers, const int32_t *block_len,
                      int32_t *view_block, int32_t *view_offset, int32_t *q_pos);

/*
 * Host helper: the views of one of the three cache layouts the Hogwild! notes
 * compare in their layout ablation, with the block ids of hw_views_combined.
 *  HW_LAYOUT_COMBINED     common, the other workers in id order, itself
 *                         (token-level visibility and the step history);
 *  HW_LAYOUT_INTERLEAVED  common, itself: only finished steps, committed into
 *                         the common history, are shared (step-level only);
 *                         the other W-1 entries are -1;
 *  HW_LAYOUT_CONTIGUOUS   the combined order over blocks that hold each
 *                         worker's whole generation: nothing is ever
 *                         committed, so the common block stays the prompt
 *                         (token-level only).  The views are the combined
 *                         ones; the difference is the caller's commit policy.
 * view_offset = tokens before each block in the view; q_pos = the view's
 * total length.  Arrays as in hw_views_combined.  HW_ERR_INVALID for an
 * unknown layout; HW_ERR_UNSUPPORTED when a block would be named by more
 * than HW_MAX_REFS_PER_BLOCK rows (n_workers > 255), which the decode calls
 * skip.
 */
typedef enum { HW_LAYOUT_COMBINED = 0, HW_LAYOUT_INTERLEAVED = 1, HW_LAYOUT_CONTIGUOUS = 2 } hw_layout;
int hw_views(int32_t layout, int32_t n_problems, int32_t n_workers, const int32_t *block_len,
             int32_t *view_block, int32_t *view_offset, int32_t *q_pos);

/*
 * Host helper: the views of T-token query chunks (T = chunk > 0), for
 * hw_attn_plan_limited.  Each worker's last T tokens are already in its own
 * block and are queried at once, one row per token: row (p, w, t), index
 * (p*W + w)*T + t, sees the blocks of worker w's view in `layout` (as
 * hw_views), every other block whole and its own block up to its own token -
 * block-local position len - T + t, so view_limit = len - T + t + 1 on that
 * entry and -1 (whole block) on the others; q_pos = that token's position in
 * the view.  All arrays host: view_block, view_offset, view_limit
 * [n_problems*W*T][W+1], q_pos [n_problems*W*T].  HW_ERR_INVALID for an
 * unknown layout or a worker block shorter than T; HW_ERR_UNSUPPORTED when a
 * block would be named by more than HW_MAX_REFS_PER_BLOCK rows (W*T > 255).
 */
int hw_views_chunked(int32_t layout, int32_t n_problems, int32_t n_workers, int32_t chunk,
                     const int32_t *block_len, int32_t *view_block, int32_t *view_offset,
                     int32_t *view_limit, int32_t *q_pos);

/*
 * For tests of the bounded waits (the pages have no counterpart).  The merge
 * step of a decode waits for every partial result of a (row, q head) item
 * with a bound; past it the call gives up on that item (its out and lse rows
 * are left as they were), records HW_DEV_TIMEOUT in the workspace and
 * returns.  This sets that bound, in SM clock cycles, for every decode call
 * made afterwards in the process; 0 restores the default (about one second).
 * HW_ERR_INVALID for a negative value.  A workspace whose call timed out is to
 * be reinitialised (hw_workspace_init) before its next use.
 */
int hw_test_set_merge_wait_limit(int64_t cycles);

/*
 * Layer timeline, for profiling (the pages have no counterpart).  A library
 * built with HW_TRACE (concurrent_shared_kv_gb300/build.py, trace=True)
 * stamps the GPU's global timer (ns) at fixed points of every tensor-core
 * decode launch: for the last 8 decode calls of the process (call index mod
 * 8), 160 CTAs and 24 points each - 0 entry, 1 work before the wait on the
 * previous launch done, 2 that wait returned, 3 first queries ready,
 * 4 first scores, 5 last scores, 6 last records stored, 7 last arrivals,
 * 8 merge phase entered, 10 the first item's records all there, 11 first
 * item merged, 12 exit; and the values 20 items merged, 21 tiles streamed,
 * 22 SM id (0 where a point was not reached).  hw_trace_read copies the
 * table into host memory dst (uint64 [8][160][24]; synchronous);
 * hw_trace_clear zeroes it.  Without HW_TRACE both return
 * HW_ERR_UNSUPPORTED and the kernels carry no stamps.
 */
int hw_trace_read(uint64_t *dst);
int hw_trace_clear(void);

/* Last CUDA error code seen by this thread's library calls (cudaError_t). */
int hw_last_cuda_error(void);

/* Static description of a status code. */
const char *hw_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* HOGWILD_H */
