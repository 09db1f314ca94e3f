// hw_device.cuh - device code shared by the decode kernels: the work plan
// (KV split evenly over the CTAs), query rotation, partial records and the
// log-sum-exp merge.
//
// Scheduling (omica.com.cn article, section 3.2: the KV cache is split evenly
// over the SMs and the partial results are merged):
//   unit      = one tile of `TILE` tokens of one block for one kv head;
//   units are ordered kv-head-major, then block, then tile (UH units per
//   head); only blocks that some view references take part.  Head-major
//   order keeps each head's short worker blocks next to its long common
//   block, instead of stacking every head's short blocks on the last CTAs.
//   CTA c of C owns units [floor(c U / C), floor((c+1) U / C)), so every CTA
//   streams the same number of tiles whatever the block lengths are.  C is
//   min(grid, U): every working CTA owns at least one unit, so the CTAs that
//   touch a segment form one contiguous range.
//   segment   = the units of one (block, kv head), id seg = h * n_blocks + b,
//   increasing along the unit order; a CTA emits one partial record per
//   (segment it touched, query head served) into slot seg + c, which is
//   unique because seg and c never both stay put as units advance.
//   Every delivered record bumps the arrival counter of its (row, kv head).
//   The launch is cooperative (all CTAs resident at once): after its own
//   units, CTA c merges the (row, kv head) pairs c, c + grid, ... - it waits,
//   with a bound, until the pair's counter shows every record, then combines
//   them with one warp per query head.  Spreading the merges over the grid
//   keeps them off any single CTA's critical path.
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

// ---------------------------------------------------------------------------
// the plan: every CTA derives the same unit decomposition from the metadata
// ---------------------------------------------------------------------------

struct PlanCore {
  int32_t tiles[HW_MAX_BLOCKS];      // tiles per kv head (0: block skipped)
  int32_t start[HW_MAX_BLOCKS];      // first pool token (valid where tiles > 0)
  int32_t len[HW_MAX_BLOCKS];        // tokens (valid where tiles > 0)
  int64_t ubase[HW_MAX_BLOCKS + 1];  // first unit of each block within a head; [n] = UH
};

struct PlanScratch {  // only while the plan is built
  int32_t refs[HW_MAX_BLOCKS];
  int32_t headmap_ok;
};

// Per-segment metadata: the view entries referencing the block and the query
// heads of the kv head.  Query head qi of the tile is (ref qi / G, head qi % G).
struct SegMeta {
  int32_t n_ref;
  int32_t ref_entry[kMaxQ];  // view entries r * V + v, in entry order
  int32_t qhead[kMaxQ];      // q heads of the kv head, in increasing order
};

struct MergeScratch {
  int32_t mv_qi[HW_MAX_VIEW_BLOCKS];   // rank of the entry among its block's references
  int64_t mv_seg[HW_MAX_VIEW_BLOCKS];  // segment id b * Hkv + h, -1 = no records
  int32_t mv_c0[HW_MAX_VIEW_BLOCKS], mv_c1[HW_MAX_VIEW_BLOCKS];
  float red[32];
};

// Unit range of CTA c.
__device__ __forceinline__ int64_t cta_unit_begin(int64_t U, int c, int C) {
  return (U * c) / C;
}
// The CTA that owns unit u: the largest c with floor(c U / C) <= u.
__device__ __forceinline__ int cta_of_unit(int64_t u, int64_t U, int C) {
  return static_cast<int>(((u + 1) * C - 1) / U);
}

// Validates the metadata and builds the unit prefix.  Every thread of the CTA
// takes part (blockDim.x threads, __syncthreads inside).
template <int TILE>
__device__ void build_plan(const DecodeArgs &a, PlanCore &P, PlanScratch &S) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int G = a.n_q_heads / a.n_kv_heads;
  for (int b = tid; b < a.n_blocks; b += nt) S.refs[b] = 0;
  if (tid == 0) S.headmap_ok = 1;
  __syncthreads();
  const int E = a.n_rows * a.n_view;
  for (int e = tid; e < E; e += nt) {
    const int b = a.view_block[e];
    if (b >= a.n_blocks || b < -1) {
      if (blockIdx.x == 0) flag_error(a.err, HW_DEV_BAD_BLOCK);
    } else if (b >= 0) {
      atomicAdd(&S.refs[b], 1);
    }
  }
  if (a.q_to_kv) {
    // every kv head must serve exactly G query heads
    for (int h = tid; h < a.n_kv_heads; h += nt) {
      int cnt = 0;
      for (int hq = 0; hq < a.n_q_heads; ++hq) cnt += (a.q_to_kv[hq] == h);
      if (cnt != G) S.headmap_ok = 0;
    }
    for (int hq = tid; hq < a.n_q_heads; hq += nt) {
      const int g = a.q_to_kv[hq];
      if (g < 0 || g >= a.n_kv_heads) S.headmap_ok = 0;
    }
  }
  __syncthreads();
  if (!S.headmap_ok && tid == 0 && blockIdx.x == 0) flag_error(a.err, HW_DEV_BAD_HEADMAP);
  for (int b = tid; b < a.n_blocks; b += nt) {
    const int32_t s = a.block_start[b], n = a.block_len[b];
    int t = 0;
    if (s < 0 || n < 0 || static_cast<int64_t>(s) + n > a.capacity) {
      if (blockIdx.x == 0) flag_error(a.err, HW_DEV_BAD_RANGE);
    } else if (S.refs[b] > 0 && n > 0) {
      if (S.refs[b] * G > kMaxQ) {
        if (blockIdx.x == 0) flag_error(a.err, HW_DEV_TOO_MANY_REFS);
      } else {
        t = (n + TILE - 1) / TILE;
      }
    }
    P.tiles[b] = S.headmap_ok ? t : 0;
    P.start[b] = s;
    P.len[b] = n;
  }
  __syncthreads();
  if (tid < 32) {
    // exclusive prefix over blocks of tiles (units of one kv head), one warp
    int64_t carry = 0;
    for (int base = 0; base < a.n_blocks; base += 32) {
      const int b = base + tid;
      const int64_t x = (b < a.n_blocks) ? static_cast<int64_t>(P.tiles[b]) : 0;
      int64_t incl = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      if (b < a.n_blocks) P.ubase[b] = carry + incl - x;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (tid == 0) P.ubase[a.n_blocks] = carry;
  }
  __syncthreads();
}

// Total units: UH per kv head.
__device__ __forceinline__ int64_t total_units(const PlanCore &P, const DecodeArgs &a) {
  return P.ubase[a.n_blocks] * a.n_kv_heads;
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

// The unit u decoded: block, kv head, tile, and the segment's first unit.
struct UnitPos {
  int b, h, t, tiles;
  int64_t seg_first;
};
__device__ __forceinline__ UnitPos unit_pos(const PlanCore &P, int n_blocks, int64_t u) {
  UnitPos x;
  const int64_t UH = P.ubase[n_blocks];
  x.h = static_cast<int>(u / UH);
  const int64_t local = u - static_cast<int64_t>(x.h) * UH;
  x.b = block_of_unit(P, n_blocks, local);
  x.tiles = P.tiles[x.b];
  x.t = static_cast<int>(local - P.ubase[x.b]);
  x.seg_first = static_cast<int64_t>(x.h) * UH + P.ubase[x.b];
  return x;
}

// First unit of segment (b, h) and its id.
__device__ __forceinline__ int64_t seg_first_unit_of(const PlanCore &P, int n_blocks, int b, int h) {
  return static_cast<int64_t>(h) * P.ubase[n_blocks] + P.ubase[b];
}
__device__ __forceinline__ int64_t seg_id(int n_blocks, int b, int h) {
  return static_cast<int64_t>(h) * n_blocks + b;
}

// Number of CTAs whose unit ranges touch segment (b, h).
__device__ __forceinline__ int seg_ctas(const PlanCore &P, int n_blocks, int b, int h, int64_t U,
                                        int C) {
  const int tl = P.tiles[b];
  if (tl == 0) return 0;
  const int64_t s0 = seg_first_unit_of(P, n_blocks, b, h);
  return cta_of_unit(s0 + tl - 1, U, C) - cta_of_unit(s0, U, C) + 1;
}

// Records expected for (row r, kv head h): one per (view entry, CTA) pair.
__device__ __forceinline__ int expected_records(const DecodeArgs &a, const PlanCore &P, int r,
                                                int h, int64_t U, int C) {
  int n = 0;
  for (int v = 0; v < a.n_view; ++v) {
    const int b = a.view_block[r * a.n_view + v];
    if (b >= 0 && b < a.n_blocks) n += seg_ctas(P, a.n_blocks, b, h, U, C);
  }
  return n;
}

// The query heads served by kv head h, in increasing order (one warp).
__device__ __forceinline__ void gather_qheads(const DecodeArgs &a, SegMeta &M, int h, int lane) {
  const int G = a.n_q_heads / a.n_kv_heads;
  if (!a.q_to_kv) {
    for (int i = lane; i < G; i += 32) M.qhead[i] = h * G + i;
  } else {
    int cnt = 0;
    for (int base = 0; base < a.n_q_heads; base += 32) {
      const int hq = base + lane;
      const bool m = hq < a.n_q_heads && a.q_to_kv[hq] == h;
      const unsigned mask = __ballot_sync(0xffffffffu, m);
      const int pos = cnt + __popc(mask & ((1u << lane) - 1u));
      if (m && pos < G) M.qhead[pos] = hq;
      cnt += __popc(mask);
    }
  }
}

// View entries referencing block b, in entry order (one warp).
__device__ __forceinline__ void gather_refs(const DecodeArgs &a, SegMeta &M, int b, int lane) {
  const int E = a.n_rows * a.n_view;
  int cnt = 0;
  for (int base = 0; base < E; base += 32) {
    const int e = base + lane;
    const bool m = e < E && a.view_block[e] == b;
    const unsigned mask = __ballot_sync(0xffffffffu, m);
    const int pos = cnt + __popc(mask & ((1u << lane) - 1u));
    if (m && pos < kMaxQ) M.ref_entry[pos] = e;
    cnt += __popc(mask);
  }
  if (lane == 0) M.n_ref = cnt;
}

__device__ __forceinline__ float *record_ptr(const DecodeArgs &a, int64_t slot, int qi) {
  return a.partials + (slot * kMaxQ + qi) * static_cast<int64_t>(a.head_dim + 4);
}

// out = 0, lse = -inf for every query head of kv head h in row r (empty view).
template <typename T>
__device__ void write_empty(const DecodeArgs &a, const int32_t *qhead, int r, int tid, int nt) {
  const int G = a.n_q_heads / a.n_kv_heads;
  for (int i = tid; i < G * a.head_dim; i += nt) {
    const int gi = i / a.head_dim, d = i % a.head_dim;
    const int hq = qhead[gi];
    reinterpret_cast<T *>(a.out)[(static_cast<int64_t>(r) * a.n_q_heads + hq) * a.head_dim + d] =
        from_f32<T>(0.f);
    if (d == 0 && a.lse) a.lse[static_cast<int64_t>(r) * a.n_q_heads + hq] = -INFINITY;
  }
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
// segment's block and every q head of kv head h (M.qhead).  One thread calls
// it, after the group's record stores were ordered before it (a barrier the
// writers took part in, or an mbarrier they arrived on).
__device__ __forceinline__ void arrive_segment(const DecodeArgs &a, const SegMeta &M, int h) {
  (void)h;
  const int G = a.n_q_heads / a.n_kv_heads;
  __threadfence();
  for (int j = 0; j < M.n_ref && j < kMaxQ; ++j) {
    const int r = M.ref_entry[j] / a.n_view;
    for (int gi = 0; gi < G; ++gi) atomicAdd(&a.counters[r * a.n_q_heads + M.qhead[gi]], 1);
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

// Shared scratch of the merge phase (at most ~20 KB; the tensor-core kernel
// places it in its tile buffers, idle by then).
struct MergeSmem {
  MergeScratch X;
  int32_t list[kMaxRecords];  // record index of each partial: slot * 32 + rank * G + gi
  float mlist[kMaxRecords];   // its max m (log2 domain)
  float acc[8][128];          // per warp partial sums of the output row
  int32_t nb_before[HW_MAX_BLOCKS];  // blocks with tiles before b (segment ordinals)
  int32_t rank_part[8];
  int32_t n_rec, ok, rank;
  float M, L;
};

// Ordinal of the segment that holds unit u, in unit order.
__device__ __forceinline__ int seg_ordinal(const PlanCore &P, const MergeSmem &Z, int n_blocks,
                                           int nb_total, int64_t u) {
  const int64_t UH = P.ubase[n_blocks];
  const int h = static_cast<int>(u / UH);
  const int b = block_of_unit(P, n_blocks, u - static_cast<int64_t>(h) * UH);
  return h * nb_total + Z.nb_before[b];
}

// The merge phase.  Every thread of every CTA of the (cooperative) grid calls
// it once its own units are done.  Work item = (row r, q head hq): all the
// partial records of that output row, each from one (view entry, CTA) pair.
// Items go to CTAs in order of how many segments they processed (idle and
// lightly loaded CTAs first), so the merges do not queue behind the slowest
// CTAs.  An item's owner prepares the record list, waits (bounded) until the
// item's arrival counter shows every record, then merges with the whole CTA:
//   M = max_i m_i,  L = sum_i l_i 2^(m_i - M),  out = sum_i o_i 2^(m_i - M) / L,
//   lse = (M + log2 L) ln 2.
template <typename T, int D, typename Sync>
__device__ void merge_phase(const DecodeArgs &a, const PlanCore &P, MergeSmem &Z, int64_t U,
                            int C, int tid, int nt, Sync sync, long long wait_limit) {
  constexpr int EPL = D / 32;
  constexpr int64_t RS = D + 4;  // record stride in floats
  const int V = a.n_view;
  const int warp = tid >> 5, lane = tid & 31, nwarps = nt >> 5;
  const int G = a.n_q_heads / a.n_kv_heads;
  const int items = a.n_rows * a.n_q_heads;
  const int grid = static_cast<int>(gridDim.x);
  MergeScratch &X = Z.X;

  // ---- this CTA's rank among the grid: fewer segments first, then index
  if (tid < 32) {
    int cnt = 0;
    for (int base = 0; base < a.n_blocks; base += 32) {
      const int b = base + lane;
      const bool ne = b < a.n_blocks && P.tiles[b] > 0;
      const unsigned m = __ballot_sync(0xffffffffu, ne);
      if (b < a.n_blocks) Z.nb_before[b] = cnt + __popc(m & ((1u << lane) - 1u));
      cnt += __popc(m);
    }
    if (lane == 0) Z.n_rec = cnt;  // number of non-empty blocks, for the ordinals
  }
  sync();
  const int nb_total = Z.n_rec;
  auto nseg_of = [&](int c) -> int {
    if (U == 0 || c >= C) return 0;
    const int64_t u0 = cta_unit_begin(U, c, C), u1 = cta_unit_begin(U, c + 1, C);
    return seg_ordinal(P, Z, a.n_blocks, nb_total, u1 - 1) - seg_ordinal(P, Z, a.n_blocks, nb_total, u0) + 1;
  };
  const int me = blockIdx.x;
  const int my_n = nseg_of(me);
  int before = 0;
  for (int c = tid; c < grid; c += nt) {
    const int nc = nseg_of(c);
    before += (nc < my_n || (nc == my_n && c < me)) ? 1 : 0;
  }
  for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
  if (lane == 0) Z.rank_part[warp] = before;
  sync();
  if (tid == 0) {
    int rk = 0;
    for (int w2 = 0; w2 < nwarps; ++w2) rk += Z.rank_part[w2];
    Z.rank = rk;
  }
  sync();
  const int rank = Z.rank;

  for (int it = rank; it < items; it += grid) {
    const int r = it / a.n_q_heads, hq = it % a.n_q_heads;
    int h = hq / G, gi = hq % G;
    if (a.q_to_kv) {
      h = a.q_to_kv[hq];
      gi = 0;
      for (int q2 = 0; q2 < hq; ++q2) gi += (a.q_to_kv[q2] == h);
      if (h < 0 || h >= a.n_kv_heads || gi >= G) continue;  // flagged by the plan
    }
    const int expected = expected_records(a, P, r, h, U, C);
    if (expected == 0) continue;  // written as empty at the start
    if (warp == 0) {
      // per view entry: its block's segment, the CTA range that wrote records,
      // and its rank among the entries that reference the same block
      for (int v = lane; v < V; v += 32) {
        const int b = a.view_block[r * V + v];
        X.mv_seg[v] = -1;
        X.mv_qi[v] = 0;
        if (b >= 0 && b < a.n_blocks && P.tiles[b] > 0) {
          const int64_t s0 = seg_first_unit_of(P, a.n_blocks, b, h);
          X.mv_seg[v] = seg_id(a.n_blocks, b, h);
          X.mv_c0[v] = cta_of_unit(s0, U, C);
          X.mv_c1[v] = cta_of_unit(s0 + P.tiles[b] - 1, U, C);
        }
      }
      __syncwarp();
      const int E = r * V + V;
      for (int base = 0; base < E; base += 32) {
        const int i = base + lane;
        const int x = (i < E) ? a.view_block[i] : -2;
        for (int v = 0; v < V; ++v) {
          const int e = r * V + v;
          const int b = __shfl_sync(0xffffffffu, x, (e - base) & 31);
          const int bb = (e >= base && e < base + 32) ? b : a.view_block[e];
          const unsigned m = __ballot_sync(0xffffffffu, i < e && x == bb);
          if (lane == 0) X.mv_qi[v] += __popc(m);
        }
      }
      __syncwarp();
      // the flat record list: (view entry, CTA) pairs in view order
      int off = 0;
      for (int v = 0; v < V; ++v) {
        if (X.mv_seg[v] < 0) continue;
        const int c0 = X.mv_c0[v], cnt = X.mv_c1[v] - c0 + 1;
        const int base_rec = X.mv_qi[v] * G + gi;
        for (int j = lane; j < cnt; j += 32)
          if (off + j < kMaxRecords)
            Z.list[off + j] = static_cast<int32_t>((X.mv_seg[v] + c0 + j) * kMaxQ + base_rec);
        off += cnt;
      }
      if (lane == 0) {
        if (off > kMaxRecords) {
          flag_error(a.err, HW_DEV_TOO_MANY_REFS);
          off = kMaxRecords;
        }
        Z.n_rec = off;
      }
    }
    if (tid == 0) {
      // every record of the item is delivered (bounded wait: co-resident CTAs)
      const int32_t *ctr = a.counters + it;
      bool ok = ld_acquire_gpu(ctr) >= expected;
      if (!ok) {
        const long long t0 = clock64();
        while (!(ok = ld_acquire_gpu(ctr) >= expected)) {
          if (clock64() - t0 > wait_limit) break;
          __nanosleep(32);
        }
      }
      if (!ok) flag_error(a.err, HW_DEV_TIMEOUT);
      Z.ok = ok ? 1 : 0;
    }
    sync();
    const int n_rec = Z.n_rec;
    if (Z.ok) {
      if (warp == 0) {  // pass A: the maxima and the normaliser
        float Mx = -INFINITY, Lx = 0.f;
        for (int k = lane; k < n_rec; k += 32) {
          const float *rec = a.partials + static_cast<int64_t>(Z.list[k]) * RS;
          const float m = __ldcg(rec + D);
          Z.mlist[k] = m;
          lse_combine(Mx, Lx, m, __ldcg(rec + D + 1));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float m2 = __shfl_xor_sync(0xffffffffu, Mx, o);
          const float l2 = __shfl_xor_sync(0xffffffffu, Lx, o);
          lse_combine(Mx, Lx, m2, l2);
        }
        if (lane == 0) {
          Z.M = Mx;
          Z.L = Lx;
        }
      }
      sync();
      // pass B: warp w takes records w, w + nwarps, ...; lane j owns elements
      // [j * EPL, (j+1) * EPL) of the row
      const float Mx = Z.M;
      float acc[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
#pragma unroll 4
      for (int k = warp; k < n_rec; k += nwarps) {
        const float w = ex2(Z.mlist[k] - Mx);
        const float *o = a.partials + static_cast<int64_t>(Z.list[k]) * RS + lane * EPL;
        if constexpr (EPL == 4) {
          const float4 x = __ldcg(reinterpret_cast<const float4 *>(o));
          acc[0] += w * x.x;
          acc[1] += w * x.y;
          acc[2] += w * x.z;
          acc[3] += w * x.w;
        } else {
          const float2 x = __ldcg(reinterpret_cast<const float2 *>(o));
          acc[0] += w * x.x;
          acc[1] += w * x.y;
        }
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) Z.acc[warp][lane * EPL + e] = acc[e];
      sync();
      if (tid < D) {
        float sum = 0.f;
        for (int w2 = 0; w2 < nwarps; ++w2) sum += Z.acc[w2][tid];
        const int64_t ob = static_cast<int64_t>(r) * a.n_q_heads + hq;
        reinterpret_cast<T *>(a.out)[ob * D + tid] = from_f32<T>(sum / Z.L);
        if (tid == 0 && a.lse) a.lse[ob] = (Z.M + __log2f(Z.L)) * 0.69314718055994530942f;
      }
    }
    sync();
    if (tid == 0) a.counters[it] = 0;  // re-armed for the next call
  }
}

}  // namespace hw
