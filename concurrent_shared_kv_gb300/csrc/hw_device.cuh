// hw_device.cuh - device code shared by the decode kernels: the metadata
// cache, the work plan (KV split over the CTAs), partial records and the
// log-sum-exp merge.
//
// Scheduling (omica.com.cn article, section 3.2: the KV cache is split evenly
// over the SMs and the partial results are merged):
//   column group = up to kMaxQ query columns of one block: the block's
//   columns are its view references x the GQA group G, and its references,
//   in view-entry order, form ng = ceil(refs / (kMaxQ / G)) groups of
//   kMaxQ / G (every worker may attend the common block: a block read by
//   more rows than one tile serves is read once per group);
//   unit      = one tile of `TILE` tokens of one (block, group) for one kv
//   head; units are ordered kv-head-major, then block, then group, then tile
//   (UH units per head); only blocks that some view references take part.
//   Head-major order keeps each head's short worker blocks next to its long
//   common block, instead of stacking every head's short blocks on the last
//   CTAs.
//   segment   = the units of one (block, group, kv head), id seg = h * NS +
//   sord[b] + g (NS segments per head, sord[b] before block b), increasing
//   along the unit order.
//   The split is stream-K over a weighted line: every unit weighs kTileW and
//   every segment start kSegW more (a segment switch costs a record epilogue
//   and a new set of rotated queries), so a CTA that crosses several short
//   worker blocks streams fewer tiles than one inside the long common block.
//   Unit (h, b, g, t) starts at weight h WH + kTileW (ubase[b] + g T + t) +
//   kSegW (sord[b] + g + 1), where T = tiles[b], ubase[b] and sord[b] count
//   the units and segments of a head before block b, and WH = kTileW UH +
//   kSegW NS.  CTA c of C takes the units whose start
//   lies in [floor(c W / C), floor((c+1) W / C)).  C = min(grid,
//   W / (kSegW + kTileW)): unit starts are at most kSegW + kTileW apart, so
//   every working CTA owns at least one unit and the CTAs touching a segment
//   form one contiguous range.
//   A CTA emits one partial record per (segment it touched, query head
//   served) into slot seg + c, unique because seg and c never both stay put
//   as units advance.  Every delivered record bumps the arrival counter of
//   its (row, q head).  After its own units, a merging CTA merges the (row,
//   q head) items given to it - it waits, with a bound, until the item's
//   counter shows every record, then combines them with the whole CTA.  Every
//   CTA a merge waits for is resident: the SIMT kernel's launch is
//   cooperative; the tensor-core kernel's CTAs (one per SM, at most one grid
//   of them waiting) hold their SMs from their start and wait for no one
//   before their records are out.
//
// The view tables, positions and head map are read from global memory once,
// in one round of independent loads, into a shared-memory cache (MetaCache);
// everything later (plan, per-segment metadata, merge lists) reads the cache,
// so no chain of dependent global loads sits on the path once the K/V tiles
// are streaming.  Views with more than kCacheEntries entries fall back to
// global reads.
//
// Group-level helpers take (tid, nt) - the thread's index within the group
// that runs them and the group's size - and a Sync functor that synchronises
// exactly that group.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hw_internal.h"

namespace hw {

// Layer timeline (a build with HW_TRACE only; otherwise the points compile to
// nothing): the globaltimer at point k of CTA c of call n, kept for the last
// kTraceCalls calls, read by hw_trace_read.  Points (tensor-core kernel):
// 0 entry, 1 work before griddepcontrol.wait done, 2 wait returned, 3 first
// queries ready, 4 first scores, 5 last scores, 6 last records stored,
// 7 last arrivals, 8 merge phase entered, 10 first item's records all
// there, 11 first item merged, 12 exit; values: 20 items merged, 21 tiles,
// 22 SM id.
constexpr int kTraceCalls = 8, kTraceCtas = 160, kTracePoints = 24;
#ifdef HW_TRACE
static __device__ unsigned long long g_trace[kTraceCalls][kTraceCtas][kTracePoints];
__device__ __forceinline__ unsigned long long trace_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define HW_TRACE_VAL(a, k, v)                                                          \
  do {                                                                                 \
    if (blockIdx.x < kTraceCtas) g_trace[(a).trace_call % kTraceCalls][blockIdx.x][(k)] = (v); \
  } while (0)
#define HW_TRACE_AT(a, k) HW_TRACE_VAL(a, k, trace_now())
#else
#define HW_TRACE_VAL(a, k, v) \
  do {                        \
  } while (0)
#define HW_TRACE_AT(a, k) HW_TRACE_VAL(a, k, 0)
#endif

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void flag_error(int32_t *err, int bits) {
  atomicOr(reinterpret_cast<int *>(err), bits);
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// cos and sin of the RoPE angle for relative position `rel` and one pair.  The
// angle in turns is (rel * phase) mod 1, computed exactly in 64-bit integers;
// its top bits become a float in [-0.5, 0.5) turns, and sincospif does the
// rest (sin(pi x), cos(pi x) of x = 2 * turns).
__device__ __forceinline__ void rope_cos_sin(int64_t rel, uint64_t phase, float *c, float *s) {
  const uint64_t turns = static_cast<uint64_t>(rel) * phase;  // mod 2^64
  const float t = static_cast<float>(static_cast<int64_t>(turns)) * 0x1p-63f;  // 2 * turns
  sincospif(t, s, c);
}

// The same from the exactly reduced angle through the fast hardware sine and
// cosine: pi * t lies in [-pi, pi), where their absolute error is at most
// 2^-21.41 (CUDA math documentation) - far below the 16 bits that the
// tensor-core path keeps of a rotated query.
__device__ __forceinline__ void rope_cos_sin_fast(int64_t rel, uint64_t phase, float *c, float *s) {
  const uint64_t turns = static_cast<uint64_t>(rel) * phase;  // mod 2^64
  const float t = static_cast<float>(static_cast<int64_t>(turns)) * 0x1p-63f;
  __sincosf(t * 3.14159265358979323846f, s, c);
}

// a / b for a >= 0, b > 0, in 32 bits when both fit.
__device__ __forceinline__ int64_t div_nn(int64_t a, int64_t b) {
  if (((a | b) >> 32) == 0) return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
  return a / b;
}

struct CtaSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// Named barrier over COUNT threads (a multiple of 32).
template <int ID, int COUNT>
struct NamedSync {
  __device__ __forceinline__ void operator()() const {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(COUNT) : "memory");
  }
};

__device__ __forceinline__ unsigned lanemask_lt(int lane) { return (1u << lane) - 1u; }

// ---------------------------------------------------------------------------
// the metadata cache
// ---------------------------------------------------------------------------

constexpr int kCacheEntries = 384;  // view entries (rows x view blocks) held in shared memory
constexpr int kMaxBlockRefs = HW_MAX_REFS_PER_BLOCK;  // view entries naming one block
constexpr int kCacheRows = 384;     // q_pos entries held in shared memory

struct alignas(16) MetaCache {
  uint64_t phase[64];           // RoPE phase increments (the kernel argument's table)
  int32_t vb[kCacheEntries];    // view_block
  int32_t voff[kCacheEntries];  // view_offset
  int32_t qpos[kCacheRows];     // q_pos
  uint8_t kv_of[HW_MAX_Q_HEADS];  // q head -> kv head
  // For the merge only, filled by plan_ranks() while the tiles stream:
  uint8_t rank[kCacheEntries];    // the entry's position among the references to its block
  uint8_t gi_of[HW_MAX_Q_HEADS];  // q head -> its index among the kv head's q heads
  uint8_t rcount[HW_MAX_BLOCKS];  // scratch of plan_ranks
  uint8_t gcount[HW_MAX_Q_HEADS];
  int32_t entries_cached, rows_cached;
};

__device__ __forceinline__ int vb_at(const DecodeArgs &a, const MetaCache &M, int e) {
  return M.entries_cached ? M.vb[e] : __ldg(a.view_block + e);
}
__device__ __forceinline__ int voff_at(const DecodeArgs &a, const MetaCache &M, int e) {
  return M.entries_cached ? M.voff[e] : __ldg(a.view_offset + e);
}
__device__ __forceinline__ int qpos_at(const DecodeArgs &a, const MetaCache &M, int r) {
  return M.rows_cached ? M.qpos[r] : __ldg(a.q_pos + r);
}
// i_q - offset of view entry e (row e / V): the rotation of its queries.
__device__ __forceinline__ int64_t entry_rel(const DecodeArgs &a, const MetaCache &M, int e) {
  return static_cast<int64_t>(qpos_at(a, M, e / a.n_view)) - voff_at(a, M, e);
}

// Rank of entry e among the entries referencing the same block, for views
// too large for the cache: one warp counts the matching earlier entries.
__device__ __forceinline__ int entry_rank_scan(const DecodeArgs &a, int e, int lane) {
  const int b = __ldg(a.view_block + e);
  int cnt = 0;
  for (int base = 0; base < e; base += 32) {
    const int i = base + lane;
    cnt += __popc(__ballot_sync(0xffffffffu, i < e && __ldg(a.view_block + i) == b));
  }
  return cnt;
}

// ---------------------------------------------------------------------------
// the plan: every CTA derives the same unit decomposition from the metadata
// ---------------------------------------------------------------------------

// Weights of a unit (one tile) and of a segment start.  Measured on the 40/8
// head, 16K-token-common workload, a segment start costs about as much as
// three tiles once the records, arrivals and merge wait are counted; the
// ratio can be made finer through kTileW.
constexpr int kTileW = 1;
constexpr int kSegW = 2;

struct PlanCore {
  int32_t tiles[HW_MAX_BLOCKS];      // tiles of one group for one kv head (0: block skipped)
  int32_t start[HW_MAX_BLOCKS];      // first pool token
  int32_t len[HW_MAX_BLOCKS];        // tokens
  int64_t ubase[HW_MAX_BLOCKS + 1];  // first unit of each block within a head; [n] = UH
  uint16_t sord[HW_MAX_BLOCKS + 1];  // segments of a head before block b; [n] = NS
  int64_t UH, U, WH, W;              // units per head and in all; weights likewise
  int32_t NS, C;                     // segments per head; working CTAs
};

// Column groups of block b (0 when it takes no part).
__device__ __forceinline__ int block_groups(const PlanCore &P, int b) { return P.sord[b + 1] - P.sord[b]; }
// View references a column group holds at most, for GQA group size G.
__device__ __forceinline__ int refs_per_group(int G) { return kMaxQ / G; }

// Everything the plan derives that every CTA shares (copied as one block).
struct alignas(16) PlanShared {
  PlanCore plan;
  MetaCache cache;
};

struct PlanScratch {  // only while the plan is built
  int32_t refs[HW_MAX_BLOCKS];
  int32_t kv_cnt[HW_MAX_Q_HEADS];
  int32_t headmap_ok;
};

// Per-segment metadata: the view entries that reference the block and the
// query heads of the kv head.  Query column qi of the tile is (reference
// qi / G, q head qi % G).
struct SegMeta {
  int32_t n_ref;
  int32_t ref_entry[kMaxQ];  // view entries r * V + v, in entry order
  int32_t qhead[kMaxQ];      // q heads of the kv head, in increasing order
};

// First unit of CTA c: the first unit whose weight is >= floor(c W / C).
__device__ __forceinline__ int64_t cta_unit_begin(const PlanCore &P, int n_blocks, int c) {
  if (c >= P.C) return P.U;
  const int64_t w = div_nn(P.W * c, P.C);
  const int h = static_cast<int>(div_nn(w, P.WH));
  const int64_t l = w - static_cast<int64_t>(h) * P.WH;
  // the last block whose weight region [kTileW ubase + kSegW sord, ...) starts
  // at or before l (a block with tiles: an empty one shares its start with
  // the next, and the last start is WH > l), its group whose region (a start
  // weight kSegW, then T tiles) holds l, then that group's first unit
  // starting at or after l (one past its last unit is the next group's
  // first, the next block's or the next head's)
  int lo = 0, hi = n_blocks - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (kTileW * P.ubase[mid] + static_cast<int64_t>(kSegW) * P.sord[mid] <= l) lo = mid; else hi = mid - 1;
  }
  const int64_t T = P.tiles[lo];
  const int64_t off = l - (kTileW * P.ubase[lo] + static_cast<int64_t>(kSegW) * P.sord[lo]);
  const int64_t span = kSegW + kTileW * T;
  const int64_t g = div_nn(off, span);
  const int64_t rem = off - g * span - kSegW;
  return static_cast<int64_t>(h) * P.UH + P.ubase[lo] + g * T +
         (rem > 0 ? (rem + kTileW - 1) / kTileW : 0);
}

// Loads the metadata into the cache (one round of independent loads), checks
// it and builds the unit prefix of a split over `grid` CTAs and this CTA's
// unit range [u_range[0], u_range[1]) in it.  Every thread of the CTA takes
// part (blockDim.x == 256, three __syncthreads inside); one warp does the
// serial part in a single pass.  Errors are recorded by CTA 0.
template <int TILE>
__device__ void build_plan(const DecodeArgs &a, PlanCore &P, MetaCache &M, PlanScratch &S,
                           int64_t (&u_range)[2], int grid) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int Hq = a.n_q_heads, G = Hq / a.n_kv_heads;
  const int E = a.n_rows * a.n_view;
  const bool ecached = E <= kCacheEntries, rcached = a.n_rows <= kCacheRows;

  // 1. every metadata word this CTA needs, as one batch of loads
  int r_vb[2], r_vo[2], r_qp[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int e = tid + k * nt;
    const bool le = ecached && e < E, lr = rcached && e < a.n_rows;
    r_vb[k] = le ? __ldg(a.view_block + e) : 0;
    r_vo[k] = le ? __ldg(a.view_offset + e) : 0;
    r_qp[k] = lr ? __ldg(a.q_pos + e) : 0;
  }
  const bool lb = tid < a.n_blocks, lh = tid < Hq;
  const int r_bs = lb ? __ldg(a.block_start + tid) : 0;
  const int r_bl = lb ? __ldg(a.block_len + tid) : 0;
  const int r_kv = lh ? (a.q_to_kv ? __ldg(a.q_to_kv + tid) : tid / G) : 0;
  if (tid < 64) M.phase[tid] = a.phase[tid];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int e = tid + k * nt;
    if (ecached && e < E) {
      M.vb[e] = r_vb[k];
      M.voff[e] = r_vo[k];
    }
    if (rcached && e < a.n_rows) M.qpos[e] = r_qp[k];
  }
  if (tid == 0) {
    M.entries_cached = ecached;
    M.rows_cached = rcached;
    S.headmap_ok = 1;
  }
  if (lb) {
    P.start[tid] = r_bs;
    P.len[tid] = r_bl;
    S.refs[tid] = 0;
  }
  const bool kv_ok = r_kv >= 0 && r_kv < a.n_kv_heads;
  if (lh) {
    S.kv_cnt[tid] = 0;
    M.kv_of[tid] = static_cast<uint8_t>(kv_ok ? r_kv : 0);
  }
  __syncthreads();

  // 2. references per block and q heads per kv head
  for (int e = tid; e < E; e += nt) {
    const int b = ecached ? M.vb[e] : __ldg(a.view_block + e);
    if (b >= a.n_blocks || b < -1) {
      if (blockIdx.x == 0) flag_error(a.err, HW_DEV_BAD_BLOCK);
    } else if (b >= 0) {
      atomicAdd(&S.refs[b], 1);
    }
  }
  if (lh) {
    if (kv_ok) atomicAdd(&S.kv_cnt[r_kv], 1);
    else S.headmap_ok = 0;
  }
  __syncthreads();

  // 3. one warp: tiles per block, the prefixes, the totals, this CTA's range
  if (warp == 0) {
    for (int h = lane; h < a.n_kv_heads; h += 32)
      if (S.kv_cnt[h] != G) S.headmap_ok = 0;
    __syncwarp();
    const bool hm_ok = S.headmap_ok != 0;
    const int rpg = refs_per_group(G);
    int64_t carry = 0;
    int ncarry = 0;
    for (int base = 0; base < a.n_blocks; base += 32) {
      const int b = base + lane;
      int t = 0, ng = 0;
      if (b < a.n_blocks) {
        const int32_t st = P.start[b], n = P.len[b], refs = S.refs[b];
        if (st < 0 || n < 0 || static_cast<int64_t>(st) + n > a.capacity) {
          if (blockIdx.x == 0) flag_error(a.err, HW_DEV_BAD_RANGE);
        } else if (refs > 0 && n > 0) {
          if (refs > kMaxBlockRefs) {  // (entry ranks are kept in 8 bits)
            if (blockIdx.x == 0) flag_error(a.err, HW_DEV_TOO_MANY_REFS);
          } else {
            t = (n + TILE - 1) / TILE;
            ng = (refs + rpg - 1) / rpg;
          }
        }
        if (!hm_ok) t = ng = 0;
        P.tiles[b] = t;
      }
      const int64_t ub = static_cast<int64_t>(t) * ng;  // the block's units per head
      int64_t incl = ub;
      int sincl = ng;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        const int z = __shfl_up_sync(0xffffffffu, sincl, o);
        if (lane >= o) {
          incl += y;
          sincl += z;
        }
      }
      if (b < a.n_blocks) {
        P.ubase[b] = carry + incl - ub;
        P.sord[b] = static_cast<uint16_t>(ncarry + sincl - ng);
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
      ncarry += __shfl_sync(0xffffffffu, sincl, 31);
    }
    if (lane == 0) {
      if (!hm_ok && blockIdx.x == 0) flag_error(a.err, HW_DEV_BAD_HEADMAP);
      P.ubase[a.n_blocks] = carry;
      P.sord[a.n_blocks] = static_cast<uint16_t>(ncarry);
      P.UH = carry;
      P.U = carry * a.n_kv_heads;
      P.NS = ncarry;
      P.WH = kTileW * carry + static_cast<int64_t>(kSegW) * ncarry;
      P.W = P.WH * a.n_kv_heads;
      const int64_t cmax = P.W / (kSegW + kTileW);
      P.C = static_cast<int>(cmax < static_cast<int64_t>(grid) ? cmax : grid);
    }
    __syncwarp();
    // lanes 0 and 1: the two ends of this CTA's unit range, side by side
    if (lane < 2) {
      const int64_t u = cta_unit_begin(P, a.n_blocks, blockIdx.x + lane);
      u_range[lane] = u;
    }
  }
  __syncthreads();
}

// Entry ranks and q-head group indices for the merge (cached views only):
// warp `wr` ranks the view entries, warp `wg` the q heads.  Called by two
// warps that are idle while the tiles stream; the results are read after a
// later CTA-wide barrier.
__device__ __forceinline__ void plan_ranks(const DecodeArgs &a, MetaCache &M, int warp, int lane,
                                           int wr, int wg) {
  const int E = a.n_rows * a.n_view;
  if (warp == wr && M.entries_cached) {
    for (int b = lane; b < a.n_blocks; b += 32) M.rcount[b] = 0;
    __syncwarp();
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int b = e < E ? M.vb[e] : -1;
      const bool valid = b >= 0 && b < a.n_blocks;
      const unsigned m = __match_any_sync(0xffffffffu, valid ? b : -2 - lane);
      const int before = valid ? M.rcount[b] : 0;
      const int rk = before + __popc(m & lanemask_lt(lane));
      if (e < E) M.rank[e] = static_cast<uint8_t>(rk < 255 ? rk : 255);
      __syncwarp();
      if (valid && lane == 31 - __clz(m)) {
        const int n = before + __popc(m);
        M.rcount[b] = static_cast<uint8_t>(n < 255 ? n : 255);
      }
      __syncwarp();
    }
  } else if (warp == wg) {
    const int Hq = a.n_q_heads;
    for (int h = lane; h < a.n_kv_heads; h += 32) M.gcount[h] = 0;
    __syncwarp();
    for (int base = 0; base < Hq; base += 32) {
      const int hq = base + lane;
      const int g = hq < Hq ? M.kv_of[hq] : 0;
      const unsigned m = __match_any_sync(0xffffffffu, hq < Hq ? g : -2 - lane);
      const int before = hq < Hq ? M.gcount[g] : 0;
      if (hq < Hq) {
        const int gi = before + __popc(m & lanemask_lt(lane));
        M.gi_of[hq] = static_cast<uint8_t>(gi < 255 ? gi : 255);
      }
      __syncwarp();
      if (hq < Hq && lane == 31 - __clz(m)) {
        const int n = before + __popc(m);
        M.gcount[g] = static_cast<uint8_t>(n < 255 ? n : 255);
      }
      __syncwarp();
    }
  }
}

// Block that holds in-head unit u (ubase[b] <= u < ubase[b+1]), by binary search.
__device__ __forceinline__ int block_of_unit(const PlanCore &P, int n_blocks, int64_t u) {
  int lo = 0, hi = n_blocks - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.ubase[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The unit u decoded: block, column group, kv head, tile, the tiles of the
// segment and its first unit.
struct UnitPos {
  int b, g, h, t, tiles;
  int64_t seg_first;
};
__device__ __forceinline__ UnitPos unit_pos(const PlanCore &P, int n_blocks, int64_t u) {
  UnitPos x;
  x.h = static_cast<int>(div_nn(u, P.UH));
  const int64_t local = u - static_cast<int64_t>(x.h) * P.UH;
  x.b = block_of_unit(P, n_blocks, local);
  x.tiles = P.tiles[x.b];
  const int64_t in_block = local - P.ubase[x.b];
  x.g = x.tiles > 0 ? static_cast<int>(div_nn(in_block, x.tiles)) : 0;  // (0: u past the units)
  x.t = static_cast<int>(in_block - static_cast<int64_t>(x.g) * x.tiles);
  x.seg_first = static_cast<int64_t>(x.h) * P.UH + P.ubase[x.b] + static_cast<int64_t>(x.g) * x.tiles;
  return x;
}

// unit_pos of u + 1 from that of u (units run group after group, block after
// block, skipping blocks without tiles, then head after head): O(1) where
// unit_pos costs a division and a binary search over the blocks.
__device__ __forceinline__ void unit_pos_next(const PlanCore &P, int n_blocks, UnitPos &x) {
  if (++x.t < x.tiles) return;
  x.t = 0;
  if (++x.g < block_groups(P, x.b)) {
    x.seg_first += x.tiles;
    return;
  }
  x.g = 0;
  int b = x.b + 1;
  while (b < n_blocks && P.tiles[b] == 0) ++b;
  if (b == n_blocks) {  // the next head, from its first block with tiles
    ++x.h;
    b = 0;
    while (b < n_blocks && P.tiles[b] == 0) ++b;
    if (b == n_blocks) b = 0;  // (no units at all: never reached)
  }
  x.b = b;
  x.tiles = P.tiles[b];
  x.seg_first = static_cast<int64_t>(x.h) * P.UH + P.ubase[b];
}

// Start weight of unit u (strictly increasing in u).
__device__ __forceinline__ int64_t unit_weight(const PlanCore &P, int n_blocks, int64_t u) {
  const int h = static_cast<int>(div_nn(u, P.UH));
  const int64_t local = u - static_cast<int64_t>(h) * P.UH;
  const int b = block_of_unit(P, n_blocks, local);
  const int64_t g = P.tiles[b] > 0 ? div_nn(local - P.ubase[b], P.tiles[b]) : 0;
  return static_cast<int64_t>(h) * P.WH + kTileW * local + static_cast<int64_t>(kSegW) * (P.sord[b] + g + 1);
}

// The CTA that owns unit u: the largest c with floor(c W / C) <= weight(u).
__device__ __forceinline__ int cta_of_unit(const PlanCore &P, int n_blocks, int64_t u) {
  return static_cast<int>(div_nn((unit_weight(P, n_blocks, u) + 1) * P.C - 1, P.W));
}

// The first of the units that read tile t of block b for kv head h (one per
// column group) at or after u0, or -1 when none of them lies before u1.
__device__ __forceinline__ int64_t tile_unit_in(const PlanCore &P, int b, int h, int t, int64_t u0,
                                                int64_t u1) {
  const int64_t T = P.tiles[b];
  const int64_t u_g0 = static_cast<int64_t>(h) * P.UH + P.ubase[b] + t;  // column group 0
  const int64_t g = u0 > u_g0 ? (u0 - u_g0 + T - 1) / T : 0;
  if (g >= block_groups(P, b)) return -1;
  const int64_t u = u_g0 + g * T;
  return u < u1 ? u : -1;
}

// Segment (block b, group g, kv head h): its index along the unit order.
__device__ __forceinline__ int64_t seg_id(const PlanCore &P, int b, int g, int h) {
  return static_cast<int64_t>(h) * P.NS + P.sord[b] + g;
}

// The view entries of column group g of block b (ranks g * rpg .. among the
// entries referencing b, rpg = refs_per_group(G)), in entry order (one warp);
// an entry's position here is its rank within the group.
__device__ __forceinline__ void gather_refs(const DecodeArgs &a, const MetaCache &C, SegMeta &M,
                                            int b, int g, int lane) {
  const int E = a.n_rows * a.n_view;
  const int rpg = refs_per_group(a.n_q_heads / a.n_kv_heads);
  const int first = g * rpg;
  int cnt = 0;
  for (int base = 0; base < E; base += 32) {
    const int e = base + lane;
    const bool m = e < E && vb_at(a, C, e) == b;
    const unsigned mask = __ballot_sync(0xffffffffu, m);
    const int pos = cnt + __popc(mask & lanemask_lt(lane)) - first;
    if (m && pos >= 0 && pos < rpg) M.ref_entry[pos] = e;
    cnt += __popc(mask);
  }
  if (lane == 0) M.n_ref = min(max(cnt - first, 0), rpg);
}

// The q heads of kv head h, in increasing order (one warp); a q head's
// position here is its group index gi.
__device__ __forceinline__ void gather_qheads(const DecodeArgs &a, const MetaCache &C, SegMeta &M,
                                              int h, int lane) {
  int cnt = 0;
  for (int base = 0; base < a.n_q_heads; base += 32) {
    const int hq = base + lane;
    const bool m = hq < a.n_q_heads && C.kv_of[hq] == h;
    const unsigned mask = __ballot_sync(0xffffffffu, m);
    const int pos = cnt + __popc(mask & lanemask_lt(lane));
    if (m && pos < kMaxQ) M.qhead[pos] = hq;
    cnt += __popc(mask);
  }
}

__device__ __forceinline__ float *record_ptr(const DecodeArgs &a, int64_t slot, int qi) {
  return a.partials + (slot * kMaxQ + qi) * static_cast<int64_t>(a.head_dim + kRecPad);
}

// ---------------------------------------------------------------------------
// arrivals and the merge phase
// ---------------------------------------------------------------------------

__device__ __forceinline__ int ld_acquire_gpu(const int32_t *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One arrival on (row, q head) for every view entry referencing the
// segment's column group and every q head of its kv head (M.qhead), one per
// lane: the whole warp calls it, after the group's record stores were
// ordered before it (a barrier the writers took part in, or an mbarrier they
// arrived on).  A column group holds at most kMaxQ columns, so one warp
// covers every arrival; issued together, they cost one trip to L2 instead
// of one each.
__device__ __forceinline__ void arrive_segment(const DecodeArgs &a, const SegMeta &M, int lane) {
  const int G = a.n_q_heads / a.n_kv_heads;
  __threadfence();
  if (lane < M.n_ref * G && lane < kMaxQ) {
    const int r = M.ref_entry[lane / G] / a.n_view;
    atomicAdd(&a.counters[r * a.n_q_heads + M.qhead[lane % G]], 1);
  }
}

// EPL consecutive output elements of a lane: one vector store where the row
// is aligned for it (the output rows start at multiples of D elements, so
// this depends only on the caller's base pointer), else one store each.
template <typename T, int EPL>
__device__ __forceinline__ void store_row_part(T *dst, const T (&v)[EPL]) {
  constexpr int kBytes = EPL * static_cast<int>(sizeof(T));
  static_assert(kBytes == 4 || kBytes == 8 || kBytes == 16, "vector width");
  if ((reinterpret_cast<uintptr_t>(dst) & (kBytes - 1)) == 0) {
    if constexpr (kBytes == 16) {
      uint4 w;
      memcpy(&w, v, 16);
      *reinterpret_cast<uint4 *>(dst) = w;
    } else if constexpr (kBytes == 8) {
      uint2 w;
      memcpy(&w, v, 8);
      *reinterpret_cast<uint2 *>(dst) = w;
    } else {
      uint32_t w;
      memcpy(&w, v, 4);
      *reinterpret_cast<uint32_t *>(dst) = w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < EPL; ++e) dst[e] = v[e];
  }
}

// (m, l) of two partial softmaxes in the log2 domain, combined.
__device__ __forceinline__ void lse_combine(float &M, float &L, float m, float l) {
  if (m == -INFINITY) return;  // nothing to add (and -inf - -inf would be NaN)
  if (m > M) {
    L = L * ex2(M - m) + l;  // ex2(-inf) = 0 when M is still -inf
    M = m;
  } else {
    L += l * ex2(m - M);
  }
}

// Shared scratch of the merge phase, for NL items merged side by side (the
// tensor-core kernel places it in its tile buffers, idle by then).
template <int NL>
struct MergeSmem {
  int32_t list[NL][kMaxRecords];  // record index of each partial: slot * 32 + rank * G + gi
  float acc[8][128];              // per warp partial sums of the output row
  float wm[8], wl[8];             // per warp running max and normaliser
  int32_t rank_tmp[NL][HW_MAX_VIEW_BLOCKS];  // entry ranks of one row (views beyond the cache)
  int32_t n_rec[NL], ok[NL];
};

// Position of CTA c in the order items are dealt: CTAs without units first.
__device__ __forceinline__ int merge_rank(const PlanCore &P, int c, int grid) {
  return c >= P.C ? c - P.C : c + (grid - P.C);
}

// Merge CTAs of the tensor-core kernel: the items go to the nm = ceil(items /
// 2) CTAs with the most units (ties: the lower index first) - the ones that
// finish their units last, so their wait for the other CTAs' records is
// short - while every other CTA retires as soon as its records are out.
__device__ __forceinline__ int merge_ctas(const DecodeArgs &a, int grid) {
  const int items = a.n_rows * a.n_q_heads;
  const int nm = (items + 1) / 2;
  return nm < grid ? nm : grid;
}
// The record list of merge item (row r, q head hq) in view order, built by
// one warp: for every view entry (rank k among the references to its block:
// column group k / rpg, rank k % rpg within it), the records that the CTAs
// c0..c1 touching segment (block, group, kv head) wrote at column
// (k % rpg) * G + gi.  Returns the number
// of records (in every lane); entries at or past `cap` are not written.
// rank_tmp (HW_MAX_VIEW_BLOCKS ints) is scratch for views beyond the cache.
__device__ __forceinline__ int merge_list(const DecodeArgs &a, const PlanCore &P,
                                          const MetaCache &MC, int r, int hq, int32_t *list,
                                          int cap, int32_t *rank_tmp, int lane) {
  const int V = a.n_view, G = a.n_q_heads / a.n_kv_heads;
  const int h = MC.kv_of[hq], gi = MC.gi_of[hq];
  if (!MC.entries_cached) {
    for (int v = 0; v < V; ++v) {
      const int rk = entry_rank_scan(a, r * V + v, lane);
      if (lane == 0) rank_tmp[v] = rk;
    }
    __syncwarp();
  }
  int off = 0;
  for (int v0 = 0; v0 < V; v0 += 32) {
    const int v = v0 + lane;
    int cnt = 0, col = 0;
    int64_t slot0 = 0;
    if (v < V) {
      const int e = r * V + v;
      const int b = vb_at(a, MC, e);
      if (b >= 0 && b < a.n_blocks && P.tiles[b] > 0) {
        const int rpg = refs_per_group(G);
        const int k = MC.entries_cached ? MC.rank[e] : rank_tmp[v];
        const int g = k / rpg;
        const int64_t s0 = static_cast<int64_t>(h) * P.UH + P.ubase[b] + static_cast<int64_t>(g) * P.tiles[b];
        const int c0 = cta_of_unit(P, a.n_blocks, s0);
        cnt = cta_of_unit(P, a.n_blocks, s0 + P.tiles[b] - 1) - c0 + 1;
        slot0 = seg_id(P, b, g, h) + c0;
        col = (k - g * rpg) * G + gi;
      }
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int my = off + incl - cnt;
    for (int j = 0; j < cnt; ++j)
      if (my + j < cap) list[my + j] = static_cast<int32_t>((slot0 + j) * kMaxQ + col);
    off += __shfl_sync(0xffffffffu, incl, 31);
  }
  return off;
}

// The merge phase.  Every thread of every CTA of the grid calls
// it once its own units are done.  Work item = (row r, q head hq): all the
// partial records of that output row, each from one (view entry, CTA) pair.
// A CTA of rank `rank` among the `grid` merging CTAs takes items rank, rank +
// grid, ... (the SIMT kernel: every CTA, those without units first; the
// tensor-core kernel: the merge_ctas CTAs with the most units).  A CTA
// merges up to NL of its items side by side, its warps split evenly between
// them.  The first warp of an item's group lists the item's records from the
// plan (the k-th item of the CTA, k < n_pre, may come with its list
// ready-made at pre_list + k * pre_stride, length pre_n[k] >= 0) and waits
// (bounded) until the item's arrival counter shows every record; the group
// then folds the records, each warp a strided share with kMergeBatch loads
// in flight, and its first warp combines the warps' partials:
//   M = max_i m_i,  L = sum_i l_i 2^(m_i - M),  out = sum_i o_i 2^(m_i - M) / L,
//   lse = (M + log2 L) ln 2;
// an item without records gets out = 0, lse = -inf.
constexpr int kMergeBatch = 4;

// rank / grid: this CTA's position among the nm CTAs that merge (items rank,
// rank + nm, ...); a rank at or past nm merges nothing.
template <typename T, int D, int NL, typename Sync>
__device__ void merge_phase(const DecodeArgs &a, const PlanCore &P, const MetaCache &MC,
                            MergeSmem<NL> &Z, const int32_t *pre_list, const int32_t *pre_n,
                            int n_pre, int pre_stride, int tid, int nt, Sync sync,
                            long long wait_limit, int rank, int grid) {
  constexpr int EPL = D / 32;
  constexpr int64_t RS = D + kRecPad;  // record stride in floats
  constexpr int B = kMergeBatch;
  const int warp = tid >> 5, lane = tid & 31, nwarps = nt >> 5;
  const int items = a.n_rows * a.n_q_heads;
  const int mine = rank >= 0 && rank < grid && rank < items ? (items - rank + grid - 1) / grid : 0;
  if (tid == 0) HW_TRACE_VAL(a, 20, static_cast<unsigned long long>(mine));

  for (int k0 = 0; k0 < mine; k0 += NL) {
    const int np = min(mine - k0, NL);  // items merged side by side
    const int g = nwarps / np;          // warps per item (np <= NL <= nwarps)
    const int p = warp / g, wi = warp - p * g;
    const bool active = p < np;
    const int k = k0 + p;
    const int it = rank + k * grid;
    const int r = it / a.n_q_heads, hq = it - r * a.n_q_heads;
    const bool pre = active && k < n_pre && pre_n[k] >= 0;
    if (active && wi == 0) {
      int n;
      if (pre) {
        n = pre_n[k];
      } else {
        n = merge_list(a, P, MC, r, hq, Z.list[p], kMaxRecords, Z.rank_tmp[p], lane);
        if (n > kMaxRecords) {
          if (lane == 0) flag_error(a.err, HW_DEV_TOO_MANY_REFS);
          n = kMaxRecords;
        }
      }
      if (lane == 0) {
        // every record of the item is delivered (bounded wait: co-resident CTAs)
        bool ok = true;
        if (n > 0) {
          const int32_t *ctr = a.counters + it;
          ok = ld_acquire_gpu(ctr) >= n;
          if (!ok) {
            const long long t0 = clock64();
            while (!(ok = ld_acquire_gpu(ctr) >= n)) {
              if (clock64() - t0 > wait_limit) break;
              __nanosleep(32);
            }
          }
          if (!ok) flag_error(a.err, HW_DEV_TIMEOUT);
        }
        Z.n_rec[p] = n;
        if (k == 0) HW_TRACE_AT(a, 10);
        Z.ok[p] = ok ? 1 : 0;
      }
    }
    sync();
    const int n_rec = active ? Z.n_rec[p] : 0;
    const bool ok = active && Z.ok[p] != 0;
    const int32_t *list = pre ? pre_list + k * pre_stride : Z.list[active ? p : 0];
    // fold: lane j owns elements [j * EPL, (j+1) * EPL) of the row
    float Mw = -INFINITY, Lw = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    if (ok) {
      for (int kb = wi; kb < n_rec; kb += B * g) {
        float m[B], l[B], x[B][EPL];
#pragma unroll
        for (int b = 0; b < B; ++b) {
          const int kk = kb + b * g;
          m[b] = -INFINITY;
          l[b] = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) x[b][e] = 0.f;
          if (kk < n_rec) {
            const float *rec = a.partials + static_cast<int64_t>(list[kk]) * RS;
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(rec + D));
            m[b] = ml.x;
            l[b] = ml.y;
            if constexpr (EPL == 4) {
              const float4 v = __ldcg(reinterpret_cast<const float4 *>(rec + lane * EPL));
              x[b][0] = v.x; x[b][1] = v.y; x[b][2] = v.z; x[b][3] = v.w;
            } else {
              const float2 v = __ldcg(reinterpret_cast<const float2 *>(rec + lane * EPL));
              x[b][0] = v.x; x[b][1] = v.y;
            }
          }
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
          if (m[b] == -INFINITY) continue;  // an empty partial (or none) adds nothing
          const float Mn = fmaxf(Mw, m[b]);
          const float sa = ex2(Mw - Mn), sb = ex2(m[b] - Mn);  // sa = 0 while Mw = -inf
          Lw = Lw * sa + l[b] * sb;
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[e] = acc[e] * sa + x[b][e] * sb;
          Mw = Mn;
        }
      }
    }
    if (active) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) Z.acc[warp][lane * EPL + e] = acc[e];
      if (lane == 0) {
        Z.wm[warp] = Mw;
        Z.wl[warp] = Lw;
      }
    }
    sync();
    if (active && wi == 0) {
      const int64_t ob = static_cast<int64_t>(r) * a.n_q_heads + hq;
      T *orow = reinterpret_cast<T *>(a.out) + ob * D + lane * EPL;
      if (n_rec == 0) {
        // no block of the view has tokens
#pragma unroll
        for (int e = 0; e < EPL; ++e) orow[e] = from_f32<T>(0.f);
        if (lane == 0 && a.lse) a.lse[ob] = -INFINITY;
      } else if (ok) {
        // the g <= 8 warps' partials unrolled over all 8 (indexes wrapped
        // into the arrays, the terms past g skipped): the loads and scale
        // factors are independent of one another, and the sums keep the warp
        // order of a plain loop
        constexpr int kW = 8;
        static_assert(sizeof(Z.wm) / sizeof(Z.wm[0]) == kW, "one partial per warp");
        const int w0 = p * g;
        float wm[kW], wl[kW];
#pragma unroll
        for (int w2 = 0; w2 < kW; ++w2) {
          wm[w2] = w2 < g ? Z.wm[(w0 + w2) & (kW - 1)] : -INFINITY;
          wl[w2] = Z.wl[(w0 + w2) & (kW - 1)];
        }
        float Mx = -INFINITY;
#pragma unroll
        for (int w2 = 0; w2 < kW; ++w2) Mx = fmaxf(Mx, wm[w2]);
        float L = 0.f, sum[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) sum[e] = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kW; ++w2) {
          if (wm[w2] == -INFINITY) continue;
          const float f = ex2(wm[w2] - Mx);
          L += wl[w2] * f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) sum[e] += Z.acc[(w0 + w2) & (kW - 1)][lane * EPL + e] * f;
        }
        // L = 0: view limits left the row no token (its partials are empty)
        const bool any = L > 0.f;
        T ov[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) ov[e] = from_f32<T>(any ? sum[e] / L : 0.f);
        store_row_part(orow, ov);
        if (lane == 0 && a.lse)
          a.lse[ob] = any ? (Mx + __log2f(L)) * 0.69314718055994530942f : -INFINITY;
      }
      if (lane == 0) a.counters[it] = 0;  // re-armed for the next call
      if (lane == 0 && k == 0) HW_TRACE_AT(a, 11);
    }
    sync();  // the scratch is rewritten by the next round
  }
}

}  // namespace hw
