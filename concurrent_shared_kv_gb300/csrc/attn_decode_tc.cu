// attn_decode_tc.cu - concurrent decode attention for bf16 (or E4M3, see
// Ring<true>) caches with head_dim 128 on the sm_100 tensor cores (tcgen05 +
// TMEM), K/V tiles staged by TMA.
//
// The path is HBM-bound: every K/V tile is read once per column group and
// serves every query head of the group that attends it (view references to
// the block times the GQA group, up to 32 a group; hw_device.cuh).  At 16-20 flop per KV byte the CUDA cores would be
// the ceiling, so the two small products run on the tensor cores:
//   S^T [128 tokens x 64]      = K_tile [128 x 128] . [Q~hi; Q~lo]^T   (TMEM, fp32)
//   O^T [128 d x 32 heads]     += V_tile^T [128 x 128 tokens] . P^T
// with Q~ the rotated queries (Hogwild! notes, key design 1: the query is
// rotated once per block by i_q - i_k^block; the keys stay as stored).
//
// One CTA per SM, persistent over its share of the units (hw_device.cuh).
// Warp roles, all synchronised by mbarriers with bounded waits:
//   warp 0     TMA producer: K and V tiles into a 3-stage ring
//   warp 1     MMA issuer (one thread) and TMEM owner
//   warps 2-5  softmax: S from TMEM, running max / sum, P (bf16) into smem;
//              segment epilogue: O from TMEM -> partial records
// then all eight warps of the CTAs that merge (the ones with the most units)
// take part in the merge phase (hw_device.cuh).
//   warps 6-7  rotated queries of the next segment: fp32, scale folded in,
//              split into bf16 hi + lo parts so that S keeps ~16 mantissa bits.
// QK multiplies the K tile with hi and lo stacked as one 64-column operand:
// one pass of 8 MMAs reads each K slice once, S_hi and S_lo land in separate
// TMEM columns and the softmax adds them in fp32.  (Each tcgen05.mma of this
// kernel costs stream time whatever its N - about 85 ns for M = 128, measured,
// and independent accumulators do not shorten it - so fewer, wider products
// pay.)
//
// Variants (template parameters of decode_tc_kernel): the step's new tokens
// written first (appends); per-view-entry token limits (query chunks); E4M3
// caches with per-kv-head scales; hw_attn_decode's plan cache (the plan of the
// metadata the last call saw, rebuilt in the kernel when the metadata
// differs) in place of hw_attn_plan's plan.  Consecutive launches overlap
// (programmatic dependent launch, see the kernel's entry).
#include <cuda.h>

#include <cuda_fp8.h>

#include <cfloat>
#include <climits>

#include "hw_device.cuh"
#include "hw_sm100.cuh"

namespace hw {

using namespace sm100;

namespace {

constexpr int kThreads = 256;
constexpr int kStages = 3;
constexpr int kT = kTcTile;                   // 128 tokens per tile
constexpr int kN = kMaxQ;                     // 32 query heads per tile (MMA N)
constexpr uint32_t kBox = 128 * 64 * 2;       // [128 rows][64 bf16], 128-B swizzled
constexpr uint32_t kStageBytes = 4 * kBox;    // K lo, K hi, V lo, V hi
// Q~ buffer: [d half (0-63, 64-127)][part (hi, lo)][32 columns][64 bf16],
// 128-byte swizzled: per d half, 64 rows (hi columns, then lo columns) at a
// 128-byte stride - the B operand of one N = 64 product.
constexpr uint32_t kQPart = kN * 64 * 2;      // one part of one d half: 4 KB
constexpr uint32_t kQHalf = 2 * kQPart;       // hi + lo of one d half: 8 KB
constexpr uint32_t kQBytes = 2 * kQHalf;
constexpr uint32_t kPBytes = kT * kN * 2;     // [128 tokens][32 heads], 64-B swizzled; it
                                              // lives in the stage's K region, free once
                                              // the tile's QK product has completed
static_assert(kPBytes <= 2 * kBox, "P fits the K region of a stage");
constexpr uint32_t kSCols = 2 * kN;           // S buffer: S_hi [0,32), S_lo [32,64)
constexpr uint32_t kTmemCols = 256;           // S0 [0,64)  S1 [64,128)  O0 [128,160)  O1 [160,192);
                                              // segment k accumulates in O[k & 1]
constexpr float kLazy = 8.f;                  // rescale only when the max grows by > 2^8
// E4M3 caches: P goes to the tensor cores as E4M3 codes of 2^6 p with p <=
// 2^2, so 2^6 p <= 256 stays below E4M3's largest value (448) while weights
// down to 2^-12 of the running max stay normal numbers (>= 2^-6) with their
// full precision; the factor leaves O and l exactly (a power of two).
constexpr float kLazyF8 = 2.f;
constexpr float kPScaleF8 = 64.f, kPUnscaleF8 = 1.f / 64.f;

// E4M3 caches.  A stage holds the tile's K codes ([128 rows][128 codes],
// 128-B swizzled; P takes their place once QK has completed), then its V
// codes in the same layout: 32 KB a stage, four in the ring.  Both products
// run as kind::f8f6f4 on the codes straight from TMA.  QK against the rotated
// queries split into four E4M3 parts (N = 128: S = S0 + S1/16 + S2/256 +
// S3/4096, about 16 significant bits, like the bf16 path's hi + lo).  PV with
// V^T MN-major (one 128-B atom along d) against P split into two E4M3 parts,
// the nearest code and the residual times 16, stacked on N (N = 64: O = O_hi
// + O_lo/16, about 8 significant bits of P, like the bf16 path's bf16 P).
// The sums l of the P columns come from the tensor cores too: the same P
// against a constant tile of E4M3 ones (in the ring's unused fifth 32 KB),
// so each of the 128 result rows holds every column's sum.  TMEM: S 2 x 128
// columns, O 2 x 64, L 2 x 64 (512 allocated).
constexpr uint32_t kF8Box = 128 * 128;
constexpr uint32_t kF8StageBytes = 2 * kF8Box;
constexpr int kMaxStages = 4;
constexpr int kF8Parts = 4;
template <bool kFp8>
struct Ring {
  static constexpr int NS = kFp8 ? kMaxStages : kStages;                 // stages
  static constexpr uint32_t SB = kFp8 ? kF8StageBytes : kStageBytes;     // bytes per stage
  static constexpr uint32_t SC = kFp8 ? kF8Parts * kN : kSCols;          // S columns per buffer
  static constexpr uint32_t CO = 2 * SC;                                 // first O column
  static constexpr uint32_t VOFF = kFp8 ? kF8Box : 2 * kBox;             // V (lo box) in a stage
  static constexpr uint32_t OC = kFp8 ? 2 * kN : kN;                     // O columns per buffer
  static constexpr uint32_t LC = CO + 2 * OC;                            // E4M3: first L column
  static constexpr uint32_t TC = kFp8 ? 512 : kTmemCols;                 // TMEM columns
};
// E4M3: the ones tile's offset in the ring ([128 rows][128 ones], 16 KB)
constexpr uint32_t kOnesOff = Ring<true>::NS * Ring<true>::SB;
static_assert(kOnesOff + kF8Box <= kStages * kStageBytes, "E4M3 ones tile fits the ring");
static_assert(Ring<true>::LC + 2 * Ring<true>::OC <= Ring<true>::TC, "E4M3 L columns");
static_assert(Ring<true>::NS * Ring<true>::SB <= kStages * kStageBytes, "E4M3 ring");
static_assert(Ring<true>::CO + 2 * Ring<true>::OC <= Ring<true>::TC, "E4M3 TMEM columns");
static_assert(Ring<false>::CO + 2 * Ring<false>::OC <= Ring<false>::TC, "bf16 TMEM columns");
static_assert(kF8Parts * kN * 128 <= kQBytes, "E4M3 query parts fit the Q~ buffer");

constexpr int kWarpTma = 0, kWarpMma = 1, kWarpSoft = 2, kWarpQ = 6;
constexpr int kPre = 4;  // slots of query-side segment metadata
constexpr int kPreList = 64;  // records of a merge list built ahead of the merge
constexpr int kPreItems = 2;  // merge items of a CTA whose lists a plan builds
constexpr int kAppList = 8;   // new tokens of a CTA a plan lists (more: found by a scan)
// Named barriers: 1 softmax warps, 2 query warps, 3 prologue warps.

// Query-side metadata of a segment: its view references and q heads, and per
// query column qi = (reference qi / G, q head qi % G) the q row to read and
// the rotation i_q - offset of its reference.
struct SegQ {
  SegMeta m;
  int32_t qrow[kMaxQ];  // row * Hq + q head
  int32_t minlim;       // fewest tokens of the block a column attends (view limits), <= len
  int64_t rel[kMaxQ];
};

// What the plan derives for one CTA (copied as one block).
struct alignas(16) CtaPlan {
  int64_t u0, u1;          // its units
  int64_t us[kPre];        // first unit of its segments 0 .. kPre-1 (u1 where none)
  SegQ pre[kPre];          // query-side metadata of segment j in pre[j % kPre]
  int32_t mpre[kPreItems][kPreList];  // record lists of its first merge items
  int32_t mpre_n[kPreItems];          // their lengths, or -1 (not built)
  int32_t mrank;           // its rank among the CTAs by units (merge_ctas: it merges if < nm)
  int32_t c_log;           // the split's CTA index of this work (see "plans": the order of
                           // the records is by rank, so a launch's CTA b runs rank b)
  int32_t trow[kStages];   // its first tiles (the ring's first fill): first cache row,
  uint8_t th[kStages];     // kv head,
  uint8_t tfl[kStages];    // segment flags (see TileRef)
  uint8_t n_first;         // how many (min(kStages, u1 - u0)); 0 without a plan
  int32_t app_n;           // new tokens this CTA writes (hw_attn_plan_append), 0: none
  int32_t app_tile;        // its first tile (from u0) that holds one of them
  // the first kAppList of them: (row * Hkv + kv head), cache row, block-local position
  int32_t app_pair[kAppList], app_row[kAppList], app_pos[kAppList];
};

struct TcSmem {
  alignas(1024) uint8_t stage[kStages][kStageBytes];
  alignas(1024) uint8_t q[kQBytes];
  PlanShared ps;
  CtaPlan cp;
  int32_t meta_nref;   // references of the current segment, handed to the softmax warps
  alignas(16) float red[2][kN][4];  // per tile: column maxima of the 4 softmax warps (read as float4)
  float lsave[2][4][kN];  // per segment parity: column sums of l of the 4 softmax warps
  float msave[2][kN];     // per segment parity: the reference maxima
  int32_t abort_flag;
  int32_t tiles_done;  // tiles whose P the softmax warps have written (progress only)
  uint8_t tflags[kMaxStages];  // per stage: the tile starts (1) / ends (2) its segment
  int32_t plan_ok;     // the loaded plan is usable
  int32_t cache_cur;   // the plan cache's current buffer (hw_attn_decode)
  uint32_t tmem_base;
  float q_mul;         // E4M3: the current segment's score factor (Q~ part scale x k_scale)
  float v_mul[4];      // E4M3: per segment mod 4, the v_scale of its kv head
  int32_t qmax[8];     // E4M3: per query-warp maxima |Q~| (ordered ints)
  alignas(8) uint64_t k_full[kMaxStages];
  uint64_t v_full[kMaxStages], kv_empty[kMaxStages];
  uint64_t q_full, q_empty;
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[kMaxStages];  // P of the stage's tile written (the softmax may run ahead)
  uint64_t p_empty, mma_done;
  uint64_t o_full[2], o_empty[2];  // per O buffer: segment done / epilogue read it
  uint64_t rec_ready[4];           // per segment mod 4: records written, arrivals due
  uint64_t plan_bar;               // a loaded plan has landed
  uint64_t app_bar;                // this CTA's new tokens are written (and fenced)
};

// ------------------------------------------------------------------- plans
//
// hw_attn_plan runs plan_kernel once per decode step: it copies the metadata
// into the workspace and, for this kernel, writes what every launch of the
// step would otherwise derive again - a header, the shared plan (PlanShared:
// unit prefix and metadata cache with ranks) and one CtaPlan per CTA (unit
// range, first segments' query metadata, first merge list).  A planned
// launch copies the shared part and its own record into shared memory with
// two bulk copies and starts streaming at once.

constexpr uint32_t kPlanMagic = 0x4c505748u;  // "HWPL"

struct PlanHeader {
  uint32_t magic;
  int32_t grid, n_rows, n_q_heads, n_kv_heads, head_dim, n_blocks, n_view;
  int64_t capacity;
  int32_t limited;  // planned with view limits: decoded by the limited kernel only
};
static_assert(sizeof(PlanHeader) <= kPlanHeaderBytes, "plan header");
static_assert(sizeof(PlanShared) % 16 == 0 && sizeof(CtaPlan) % 16 == 0, "bulk copy sizes");

__device__ __forceinline__ const uint8_t *plan_cta_record(const uint8_t *plan, int c) {
  return plan + kPlanHeaderBytes + sizeof(PlanShared) + static_cast<size_t>(c) * sizeof(CtaPlan);
}

// The launch's RoPE table (MetaCache::phase, the first field of the shared
// part's metadata) is written into shared memory at the kernel's entry: the
// plan copies skip those bytes.
constexpr uint32_t kPhaseOff = offsetof(PlanShared, cache) + offsetof(MetaCache, phase);
constexpr uint32_t kPhaseBytes = sizeof(MetaCache::phase);
static_assert(kPhaseOff % 16 == 0 && kPhaseBytes % 16 == 0, "the phase table is a whole number of 16-B chunks");

// Does a plan header describe a launch of `grid` CTAs with these arguments?
__device__ __forceinline__ bool header_matches(const DecodeArgs &a, const PlanHeader &h, int grid) {
  return h.magic == kPlanMagic && h.grid == grid && h.n_rows == a.n_rows &&
         h.n_q_heads == a.n_q_heads && h.n_kv_heads == a.n_kv_heads && h.head_dim == a.head_dim &&
         h.n_blocks == a.n_blocks && h.n_view == a.n_view && h.capacity == a.capacity &&
         (h.limited != 0) == (a.view_limit != nullptr);
}

// hw_attn_plan's plan into shared memory with bulk copies completing on
// plan_bar: the header (into the query buffer, idle until the queries are
// rotated; checked once it lands), the shared part around the RoPE table,
// and this CTA's record.
__device__ __forceinline__ void issue_plan_copies(const DecodeArgs &a, TcSmem &S) {
  constexpr uint32_t kHdr = (sizeof(PlanHeader) + 15) & ~15u;
  constexpr uint32_t kTail = sizeof(PlanShared) - kPhaseOff - kPhaseBytes;
  const uint8_t *src = a.plan + kPlanHeaderBytes;
  uint8_t *dst = reinterpret_cast<uint8_t *>(&S.ps);
  mbar_arrive_expect_tx(&S.plan_bar, kHdr + kPhaseOff + kTail + sizeof(CtaPlan));
  bulk_g2s(S.q, a.plan, kHdr, &S.plan_bar);
  bulk_g2s(dst, src, kPhaseOff, &S.plan_bar);
  bulk_g2s(dst + kPhaseOff + kPhaseBytes, src + kPhaseOff + kPhaseBytes, kTail, &S.plan_bar);
  bulk_g2s(&S.cp, plan_cta_record(a.plan, blockIdx.x), sizeof(CtaPlan), &S.plan_bar);
}

// The header of a plan through L2 (another launch may have written it).
__device__ __forceinline__ PlanHeader load_header_cg(const uint8_t *plan) {
  static_assert(sizeof(PlanHeader) % 4 == 0, "header words");
  uint32_t w[sizeof(PlanHeader) / 4];
  for (size_t i = 0; i < sizeof(PlanHeader) / 4; ++i) w[i] = __ldcg(reinterpret_cast<const uint32_t *>(plan) + i);
  PlanHeader h;
  memcpy(&h, w, sizeof h);
  return h;
}

// ------------------------------------------------------------- plan cache
//
// hw_attn_decode plans every call itself, but the layers of a step share
// their metadata: the workspace keeps the plan of the metadata it last saw,
// double-buffered (PlanCacheState).  A plan launch compares the call's
// metadata with the copy beside the current plan; on a match it writes
// nothing, otherwise it builds the plan and the copy into the other buffer
// and its last CTA makes that buffer current.  The decode launch after it
// takes the current buffer: under the early-loads promise, before its wait,
// when that buffer already matches (the plan launch wrote nothing, or has
// finished); otherwise after the wait, when the plan launch is complete.
__device__ __forceinline__ int32_t *cache_state(const DecodeArgs &a) {
  return reinterpret_cast<int32_t *>(a.cache_base);
}
__device__ __forceinline__ int32_t *cache_meta(const DecodeArgs &a, int k) {
  return reinterpret_cast<int32_t *>(a.cache_base + kPlanCacheStateBytes + k * a.cache_meta_bytes);
}
__device__ __forceinline__ uint8_t *cache_plan(const DecodeArgs &a, int k) {
  return a.cache_base + kPlanCacheStateBytes + 2 * a.cache_meta_bytes + k * a.cache_plan_bytes;
}
// The current buffer; acquired, so that its plan and copy read complete.
__device__ __forceinline__ int cache_current(const DecodeArgs &a) {
  return ld_acquire_gpu(cache_state(a)) & 1;
}

// Word j of the caller's metadata in the copy's layout (cache_write_meta).
__device__ __forceinline__ int32_t caller_meta_word(const DecodeArgs &a, int j) {
  const int E = a.n_rows * a.n_view, R = a.n_rows, Hq = a.n_q_heads, nb = a.n_blocks;
  if (j < E) return __ldg(a.view_block + j);
  if ((j -= E) < E) return __ldg(a.view_offset + j);
  if ((j -= E) < R) return __ldg(a.q_pos + j);
  if ((j -= R) < Hq) return a.q_to_kv ? __ldg(a.q_to_kv + j) : j / (Hq / a.n_kv_heads);
  if ((j -= Hq) < nb) return __ldg(a.block_start + j);
  return __ldg(a.block_len + j - nb);
}

// The decode's fetch from the plan cache, in one round of loads: cached plan
// k (its shared part and this CTA's record, into registers), its header and
// metadata copy, and the caller's metadata; when they describe this launch
// the plan goes to shared memory.  Every thread takes part.  Returns whether
// it matched (the same in every thread).
__device__ bool cache_fetch(const DecodeArgs &a, int k, PlanShared &ps, CtaPlan &cp, int tid, int nt) {
  constexpr int kShared = sizeof(PlanShared) / 16, kRec = sizeof(CtaPlan) / 16, kPer = 4;
  static_assert(kShared <= kPer * 256 && kRec <= 256, "one round of loads of 256 threads");
  const uint8_t *plan = cache_plan(a, k);
  const uint4 *src = reinterpret_cast<const uint4 *>(plan + kPlanHeaderBytes);
  const uint4 *rsrc = reinterpret_cast<const uint4 *>(plan_cta_record(plan, blockIdx.x));
  uint4 v[kPer], rv = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int r = 0; r < kPer; ++r)
    if (tid + r * nt < kShared) v[r] = __ldcg(src + tid + r * nt);
  if (tid < kRec) rv = __ldcg(rsrc + tid);
  bool same = true;
  if (tid == 0) same = header_matches(a, load_header_cg(plan), static_cast<int>(gridDim.x));
  const int words = static_cast<int>(plan_cache_meta_words(a.n_rows, a.n_view, a.n_q_heads, a.n_blocks));
  const int32_t *m = cache_meta(a, k);
#pragma unroll 4
  for (int j = tid; j < words; j += nt) same &= __ldcg(m + j) == caller_meta_word(a, j);
  same = __syncthreads_and(same);
  if (same) {
    uint4 *dst = reinterpret_cast<uint4 *>(&ps);
    constexpr int kP0 = kPhaseOff / 16, kP1 = (kPhaseOff + kPhaseBytes) / 16;  // (the launch's table)
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int i = tid + r * nt;
      if (i < kShared && (i < kP0 || i >= kP1)) dst[i] = v[r];
    }
    if (tid < kRec) reinterpret_cast<uint4 *>(&cp)[tid] = rv;
  }
  return same;
}

// The caller's metadata into copy k (the layout caller_meta_word reads).
__device__ void cache_write_meta(const DecodeArgs &a, int k, int tid, int nt) {
  const int E = a.n_rows * a.n_view, R = a.n_rows, Hq = a.n_q_heads, nb = a.n_blocks;
  const int G = Hq / a.n_kv_heads;
  int32_t *m = cache_meta(a, k);
  for (int i = tid; i < E; i += nt) {
    m[i] = __ldg(a.view_block + i);
    m[E + i] = __ldg(a.view_offset + i);
  }
  m += 2 * E;
  for (int i = tid; i < R; i += nt) m[i] = __ldg(a.q_pos + i);
  m += R;
  for (int i = tid; i < Hq; i += nt) m[i] = a.q_to_kv ? __ldg(a.q_to_kv + i) : i / G;
  m += Hq;
  for (int i = tid; i < nb; i += nt) {
    m[i] = __ldg(a.block_start + i);
    m[nb + i] = __ldg(a.block_len + i);
  }
}

__device__ __forceinline__ void set_abort(TcSmem &S, const DecodeArgs &a) {
  if (atomicExch(&S.abort_flag, 1) == 0) flag_error(a.err, HW_DEV_TIMEOUT);
}
__device__ __forceinline__ bool aborted(TcSmem &S) {
  return *reinterpret_cast<volatile int32_t *>(&S.abort_flag) != 0;
}
// Bounded wait; on timeout the CTA winds down.
__device__ __forceinline__ bool wait_or_abort(TcSmem &S, const DecodeArgs &a, uint64_t *bar,
                                              uint32_t parity) {
  if (aborted(S)) return false;
  if (mbar_wait(bar, parity)) return true;
  set_abort(S, a);
  return false;
}

__device__ __forceinline__ bool seg_first_unit(const UnitPos &x, int64_t u, int64_t u0) {
  return u == u0 || u == x.seg_first;
}
__device__ __forceinline__ bool seg_last_unit(const UnitPos &x, int64_t u, int64_t u1) {
  return u + 1 == u1 || u + 1 == x.seg_first + x.tiles;
}

// Named barrier 1 over the 128 softmax threads, returning the OR of `pred`.
__device__ __forceinline__ bool bar_red_or_128(bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"(pred ? 1u : 0u)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&p);
}

__device__ __forceinline__ float f16_lo(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// Elements j, j + 1 of a register array as one float pair, and back: the
// paired fp32 instructions of sm_100 (__ffma2_rn and the like: two
// correctly rounded operations in one) then halve the softmax's arithmetic
// instructions with results identical to the scalar ones.
__device__ __forceinline__ float2 pair_at(const uint32_t (&r)[32], int j) {
  return make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
}
__device__ __forceinline__ void pair_put(uint32_t (&r)[32], int j, float2 v) {
  r[j] = __float_as_uint(v.x);
  r[j + 1] = __float_as_uint(v.y);
}
__device__ __forceinline__ float2 fpair(float a) { return make_float2(a, a); }

// The E4M3 codes (low byte first) of 16 (s - h) for the pair s, where h is
// the f16x2 value of s's codes: s goes to f16 (11 bits), the residual is
// exact there, and its codes are the nearest (saturating).
__device__ __forceinline__ uint16_t e4m3x2_residual(float2 s, uint32_t h) {
  uint32_t sh, rh;
  uint16_t lo;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(sh) : "f"(s.y), "f"(s.x));  // (s.x in the low half)
  asm("{\n\t.reg .b32 t;\n\tsub.rn.f16x2 t, %1, %2;\n\tmul.rn.f16x2 %0, t, %3;\n\t}"
      : "=r"(rh)
      : "r"(sh), "r"(h), "r"(0x4C004C00u));  // 16.0 in both halves
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(lo) : "r"(rh));
  return lo;
}

// Two E4M3 codes (low byte first) as f16x2, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t codes) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes & 0xffffu), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// ------------------------------------------------------------------ roles

// Spin (bounded) until the phase with this parity completes: the producer
// re-issues a stage the moment it is released, without the wake-up delay of
// a suspended wait.
__device__ __forceinline__ bool spin_or_abort(TcSmem &S, const DecodeArgs &a, uint64_t *bar,
                                              uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_test(bar, parity)) {
    if (aborted(S)) return false;
    if (clock64() - t0 > kWaitLimit) {
      set_abort(S, a);
      return false;
    }
  }
  return true;
}

// The tile of unit u in a CTA's range [u0, u1): its first cache row, its kv
// head, and whether it starts (1) / ends (2) its segment within the range.
struct TileRef {
  int row, h;
  uint8_t flags;
};
__device__ __forceinline__ TileRef tile_ref(const PlanCore &P, int n_blocks, int64_t u, int64_t u0,
                                            int64_t u1) {
  const UnitPos x = unit_pos(P, n_blocks, u);
  TileRef t;
  t.row = P.start[x.b] + x.t * kT;
  t.h = x.h;
  t.flags = (seg_first_unit(x, u, u0) ? 1 : 0) | (seg_last_unit(x, u, u1) ? 2 : 0);
  return t;
}

template <bool kFp8>
__device__ __forceinline__ uint8_t *stage_ptr(TcSmem &S, int s) {
  return &S.stage[0][0] + s * Ring<kFp8>::SB;  // (the ring as one byte array)
}

// Streams the CTA's tiles through the ring.  The first n_first come decoded
// from the plan, so that the ring fills without waiting on the unit
// arithmetic; the others are decoded while their stage is still busy.
// The tiles i_begin .. i_end-1 of the range: at entry the first ones into
// the empty ring (i_begin = 0, i_end at most the ring and before the first
// tile with a new token), then the others (i_begin = the count issued).
// Returns the index after the last tile issued.
template <bool kFp8>
__device__ int producer(const DecodeArgs &a, TcSmem &S, const CUtensorMap *tk,
                        const CUtensorMap *tv, int64_t u0, int64_t u1, bool appending,
                        int i_begin, int64_t i_end) {
  constexpr int NS = Ring<kFp8>::NS;
  const uint64_t pol = policy_evict_first();
  const int n_first = S.cp.n_first;
  // the first tile holding a new token is loaded only once the tokens are
  // written (and fenced for the copy engine)
  const int app_tile = appending ? S.cp.app_tile : -1;
  int i = i_begin;
  const int64_t u_stop = u1 < u0 + i_end ? u1 : u0 + i_end;  // (u1 still decides the flags)
  for (int64_t u = u0 + i_begin; u < u_stop; ++u, ++i) {
    const int s = i % NS;
    // the tile's coordinates first, so that only the copy waits for the stage
    TileRef t;
    if (i < n_first) {
      t.row = S.cp.trow[i];
      t.h = S.cp.th[i];
      t.flags = S.cp.tfl[i];
    } else {
      t = tile_ref(S.ps.plan, a.n_blocks, u, u0, u1);
    }
    uint8_t *st = stage_ptr<kFp8>(S, s);
    if (i >= NS && !spin_or_abort(S, a, &S.kv_empty[s], ((i / NS) & 1) ^ 1)) break;
    if (i == app_tile && !spin_or_abort(S, a, &S.app_bar, 0)) break;
    // read by the MMA thread once the stage's copies are seen complete (the
    // arrive below releases this store)
    S.tflags[s] = t.flags;
    if constexpr (kFp8) {
      // K codes at the stage's start, V codes after them
      mbar_arrive_expect_tx(&S.k_full[s], kF8Box);
      tma_load_3d(st, tk, &S.k_full[s], 0, t.row, t.h, pol);
      mbar_arrive_expect_tx(&S.v_full[s], kF8Box);
      tma_load_3d(st + Ring<kFp8>::VOFF, tv, &S.v_full[s], 0, t.row, t.h, pol);
      continue;
    }
    mbar_arrive_expect_tx(&S.k_full[s], 2 * kBox);
    tma_load_3d(st, tk, &S.k_full[s], 0, t.row, t.h, pol);
    tma_load_3d(st + kBox, tk, &S.k_full[s], 64, t.row, t.h, pol);
    mbar_arrive_expect_tx(&S.v_full[s], 2 * kBox);
    tma_load_3d(st + 2 * kBox, tv, &S.v_full[s], 0, t.row, t.h, pol);
    tma_load_3d(st + 3 * kBox, tv, &S.v_full[s], 64, t.row, t.h, pol);
  }
  return i;
}

// No copy may still be landing in shared memory when the CTA retires: the
// last NS of the n issued tiles are waited for.
template <bool kFp8>
__device__ void producer_drain(TcSmem &S, int n) {
  constexpr int NS = Ring<kFp8>::NS;
  for (int j = (n > NS ? n - NS : 0); j < n; ++j) {
    mbar_wait(&S.k_full[j % NS], (j / NS) & 1);
    mbar_wait(&S.v_full[j % NS], (j / NS) & 1);
  }
}

// Issues the products in a fixed order - QK(0), QK(1), then PV(i), QK(i+2) -
// each after a (bounded) spin on its inputs.  QK(i+2) is not needed before
// the softmax warps are done with tile i+1, so issuing PV(i) first costs
// nothing.  The thread is on the critical path of every stage's release, so
// it does no more than wait and issue: the tile's segment flags come from
// the producer (tflags), and the operand descriptors are a base plus a
// constant offset per k-step (the start address is the descriptor's low
// field, 14 bits of address >> 4: shared addresses stay below 2^18).
template <bool kFp8>
__device__ void mma_issuer(const DecodeArgs &a, TcSmem &S, uint32_t tmem, int64_t u0, int64_t u1) {
  using R = Ring<kFp8>;
  constexpr int NS = R::NS;
  // QK: K tile, [Q~hi; Q~lo] (bf16) or the four E4M3 parts of Q~: K-major.
  // PV: V tile, P (bf16; E4M3: the codes and [P hi, P lo]): both MN-major.
  constexpr uint32_t idesc_qk = kFp8 ? idesc_e4m3(128, R::SC, 0, 0) : idesc_bf16(128, R::SC, 0, 0);
  constexpr uint32_t idesc_pv = kFp8 ? idesc_e4m3(128, R::OC, 1, 1) : idesc_bf16(128, kN, 1, 1);
  const int n = static_cast<int>(u1 - u0);
  const uint32_t stage0 = smem_u32(S.stage[0]), qbase = smem_u32(S.q);
  const uint64_t a_qk = smem_desc(stage0, 16, 1024, kSw128);    // + (stage, k-step) offset >> 4
  const uint64_t b_qk = smem_desc(qbase, 16, 1024, kSw128);
  const uint64_t a_pv = smem_desc(stage0 + R::VOFF, kBox, 1024, kSw128);
  const uint64_t a_ones = smem_desc(stage0 + kOnesOff, kBox, 1024, kSw128);  // (E4M3)
  const uint64_t b_pv = smem_desc(stage0, 512, 512, kSw64);
  int seg_q = -1, seg_p = -1;
  auto qk = [&](int i) {
    const int s = i % NS, sb = i & 1;
    if (!spin_or_abort(S, a, &S.k_full[s], (i / NS) & 1)) return;
    const uint32_t flags = S.tflags[s];
    if (flags & 1) ++seg_q;
    if (!spin_or_abort(S, a, &S.s_empty[sb], ((i >> 1) & 1) ^ 1)) return;
    if ((flags & 1) && !spin_or_abort(S, a, &S.q_full, seg_q & 1)) return;
    tc_fence_after();
    const uint64_t as = a_qk + ((s * R::SB) >> 4);
    if constexpr (kFp8) {
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4)  // 4 k-steps of 32 codes (32 bytes) over d
        mma_f8(tmem + sb * R::SC, as + ((k4 * 32) >> 4), b_qk + ((k4 * 32) >> 4), idesc_qk, k4 > 0);
    } else {
#pragma unroll
      for (int k8 = 0; k8 < 8; ++k8) {  // 8 k-steps of 16 over d
        const uint32_t ao = (k8 >> 2) * kBox + (k8 & 3) * 32, bo = (k8 >> 2) * kQHalf + (k8 & 3) * 32;
        mma_bf16(tmem + sb * R::SC, as + (ao >> 4), b_qk + (bo >> 4), idesc_qk, k8 > 0);
      }
    }
    mma_commit(&S.s_full[sb]);
    if (flags & 2) mma_commit(&S.q_empty);
  };
  auto pv = [&](int i) {
    const int s = i % NS;
    if (!spin_or_abort(S, a, &S.p_full[s], (i / NS) & 1)) return;
    if (!spin_or_abort(S, a, &S.v_full[s], (i / NS) & 1)) return;
    const uint32_t flags = S.tflags[s];
    const bool first = flags & 1;
    if (first) ++seg_p;
    if (first && !spin_or_abort(S, a, &S.o_empty[seg_p & 1], ((seg_p >> 1) & 1) ^ 1)) return;
    tc_fence_after();
    // V^T: MN-major, d 0-63 and 64-127 in two 128-B swizzle atoms kBox apart
    // (E4M3: all 128 d in one atom), 8-token groups 1024 B apart.  P^T:
    // MN-major, 32 heads (E4M3: the 32 hi and 32 lo codes) = one 64-B atom,
    // 8-token groups 512 B apart, in the stage's K region.
    const uint64_t as = a_pv + ((s * R::SB) >> 4), bs = b_pv + ((s * R::SB) >> 4);
    if constexpr (kFp8) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // 4 k-steps of 32 tokens
        mma_f8(tmem + R::CO + (seg_p & 1) * R::OC, as + ((kk * 4096) >> 4), bs + ((kk * 2048) >> 4),
               idesc_pv, !(first && kk == 0));
      // the column sums of P: ones^T . P^T (the ones tile in V's layout)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_f8(tmem + R::LC + (seg_p & 1) * R::OC, a_ones + ((kk * 4096) >> 4),
               bs + ((kk * 2048) >> 4), idesc_pv, !(first && kk == 0));
    } else {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // 8 k-steps of 16 tokens
        mma_bf16(tmem + R::CO + (seg_p & 1) * R::OC, as + ((kk * 2048) >> 4),
                 bs + ((kk * 1024) >> 4), idesc_pv, !(first && kk == 0));
    }
    mma_commit(&S.kv_empty[s]);
    mma_commit(&S.p_empty);
    if (flags & 2) mma_commit(&S.o_full[seg_p & 1]);
  };
  // one call site each: QK(0), QK(1), PV(0), QK(2), PV(1), ...
  for (int j = 0; j < n + 2 && !aborted(S); ++j) {
    if (j >= 2) pv(j - 2);
    if (j < n) qk(j);
  }
  mma_commit(&S.mma_done);
  mbar_wait(&S.mma_done, 0);
}

// The tokens of its block that view entry e attends: all len, or fewer under
// a view limit.
__device__ __forceinline__ int entry_limit(const int32_t *view_limit, int e, int len) {
  if (!view_limit) return len;
  const int v = __ldg(view_limit + e);
  return v >= 0 && v < len ? v : len;
}

// Query-side metadata of segment (block b, column group g, kv head h) into X, by one warp (shared memory
// only, except for views beyond the metadata cache), with the fewest tokens
// any of its columns attends (len when no view limit cuts the block).
template <bool kLimit>
__device__ void seg_pre(const DecodeArgs &a, const PlanCore &P, const MetaCache &C, SegQ &X, int b,
                        int g, int h, int lane) {
  const int len = P.len[b];
  const int G = a.n_q_heads / a.n_kv_heads;
  gather_refs(a, C, X.m, b, g, lane);
  gather_qheads(a, C, X.m, h, lane);
  __syncwarp();
  int lim = len;
  if (lane < X.m.n_ref * G) {
    const int e = X.m.ref_entry[lane / G];
    X.qrow[lane] = (e / a.n_view) * a.n_q_heads + X.m.qhead[lane % G];
    X.rel[lane] = entry_rel(a, C, e);
    if (kLimit) lim = entry_limit(a.view_limit, e, len);
  }
  if (kLimit) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) lim = min(lim, __shfl_xor_sync(0xffffffffu, lim, o));
  }
  if (lane == 0) X.minlim = lim;
  __syncwarp();
}

// One item of the rotated queries: column qi, elements 8c..8c+7 and their
// RoPE partners 64+8c..64+8c+7, and the column's rotation i_q - offset.  Only
// columns below nq are rotated: the rows of Q~ past them feed S columns that
// the softmax neither reads nor lets into P (their P is zero).
struct QItem {
  uint4 lo, hi;
  int64_t rel;
};
__device__ __forceinline__ void load_item(const DecodeArgs &a, const SegQ &X, int qi, int c,
                                          QItem &it) {
  const __nv_bfloat16 *qp = reinterpret_cast<const __nv_bfloat16 *>(a.q) +
                            static_cast<int64_t>(X.qrow[qi]) * 128;
  it.lo = __ldg(reinterpret_cast<const uint4 *>(qp + 8 * c));
  it.hi = __ldg(reinterpret_cast<const uint4 *>(qp + 64 + 8 * c));
  it.rel = X.rel[qi];
}

// The item rotated and scaled by scale * log2(e) (scores leave the MMA in
// log2 units), then split into bf16 hi and lo parts.  out[0..3]: hi of d
// 8c.., hi of d 64+8c.., lo of d 8c.., lo of d 64+8c.. (16 bytes each).
__device__ __forceinline__ void rot_item(const DecodeArgs &a, const TcSmem &S, const QItem &it, int c,
                                        uint4 (&out)[4]) {
  const uint32_t lo32[4] = {it.lo.x, it.lo.y, it.lo.z, it.lo.w};
  const uint32_t hi32[4] = {it.hi.x, it.hi.y, it.hi.z, it.hi.w};
  uint32_t w[4][4];
#pragma unroll
  for (int e2 = 0; e2 < 4; ++e2) {
    float ylo[2], yhi[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const float x0 = __uint_as_float(h2 ? (lo32[e2] & 0xffff0000u) : (lo32[e2] << 16));
      const float x1 = __uint_as_float(h2 ? (hi32[e2] & 0xffff0000u) : (hi32[e2] << 16));
      float cs, sn;
      rope_cos_sin_fast(it.rel, S.ps.cache.phase[8 * c + 2 * e2 + h2], &cs, &sn);
      ylo[h2] = (x0 * cs - x1 * sn) * a.scale_log2;
      yhi[h2] = (x1 * cs + x0 * sn) * a.scale_log2;
    }
    const __nv_bfloat162 hl = __floats2bfloat162_rn(ylo[0], ylo[1]);
    const __nv_bfloat162 hh = __floats2bfloat162_rn(yhi[0], yhi[1]);
    const __nv_bfloat162 ll = __floats2bfloat162_rn(ylo[0] - __low2float(hl), ylo[1] - __high2float(hl));
    const __nv_bfloat162 lh = __floats2bfloat162_rn(yhi[0] - __low2float(hh), yhi[1] - __high2float(hh));
    w[0][e2] = *reinterpret_cast<const uint32_t *>(&hl);
    w[1][e2] = *reinterpret_cast<const uint32_t *>(&hh);
    w[2][e2] = *reinterpret_cast<const uint32_t *>(&ll);
    w[3][e2] = *reinterpret_cast<const uint32_t *>(&lh);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) out[k] = make_uint4(w[k][0], w[k][1], w[k][2], w[k][3]);
}

// Store one item into the Q~ buffer: column qi of the hi and lo parts of both
// d halves (128 B per row), 16-B chunk c swizzled by qi % 8 (the 128-byte
// swizzle the MMA descriptor expects; lo row 32 + qi has the same pattern).
__device__ __forceinline__ void store_item(uint32_t qbase, int qi, int c, const uint4 (&v)[4]) {
  const uint32_t off = qi * 128 + ((static_cast<uint32_t>(c) ^ (qi & 7)) << 4);
  st_shared_v4(qbase + off, v[0].x, v[0].y, v[0].z, v[0].w);                     // hi, d 0-63
  st_shared_v4(qbase + kQHalf + off, v[1].x, v[1].y, v[1].z, v[1].w);            // hi, d 64-127
  st_shared_v4(qbase + kQPart + off, v[2].x, v[2].y, v[2].z, v[2].w);            // lo, d 0-63
  st_shared_v4(qbase + kQHalf + kQPart + off, v[3].x, v[3].y, v[3].z, v[3].w);   // lo, d 64-127
}

// E4M3 caches: the item's 16 rotated values (y[0..7]: d 8c..8c+7, y[8..15]:
// d 64+8c..), scaled by scale * log2(e), before the segment's part scale is
// known; the largest magnitude is returned.
__device__ __forceinline__ float rot_item_f32(const DecodeArgs &a, const TcSmem &S, const QItem &it,
                                              int c, float (&y)[16]) {
  const uint32_t lo32[4] = {it.lo.x, it.lo.y, it.lo.z, it.lo.w};
  const uint32_t hi32[4] = {it.hi.x, it.hi.y, it.hi.z, it.hi.w};
  float mx = 0.f;
#pragma unroll
  for (int e2 = 0; e2 < 4; ++e2) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const float x0 = __uint_as_float(h2 ? (lo32[e2] & 0xffff0000u) : (lo32[e2] << 16));
      const float x1 = __uint_as_float(h2 ? (hi32[e2] & 0xffff0000u) : (hi32[e2] << 16));
      float cs, sn;
      rope_cos_sin_fast(it.rel, S.ps.cache.phase[8 * c + 2 * e2 + h2], &cs, &sn);
      const int j = 2 * e2 + h2;
      y[j] = (x0 * cs - x1 * sn) * a.scale_log2;
      y[8 + j] = (x1 * cs + x0 * sn) * a.scale_log2;
      mx = fmaxf(mx, fmaxf(fabsf(y[j]), fabsf(y[8 + j])));
    }
  }
  return mx;
}

// The power of two c with max / c < 448 (the largest E4M3 value): the
// segment's Q~ parts hold y / c.
__device__ __forceinline__ int part_exponent(float mx) {
  int e = 0;
  if (mx > 0.f) frexpf(mx * (1.f / 448.f), &e);
  return e;
}

// The item as four E4M3 parts, z = y / c ~ a0 + a1/16 + a2/256 + a3/4096 (each
// part the residual of the ones before, times 16), into Q~ rows 32 j + qi of
// part j: 8 codes at byte 8c (d 8c..) and 8 at byte 64 + 8c (d 64 + 8c..),
// 16-B chunks swizzled by qi % 8 like the bf16 buffer.
__device__ __forceinline__ void store_item_e4m3(uint32_t qbase, int qi, int c, const float (&y)[16],
                                                float inv_c) {
  uint32_t w[kF8Parts][4];
#pragma unroll
  for (int j = 0; j < kF8Parts; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) w[j][k] = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {  // value pairs: y[2k], y[2k + 1]
    float2 z = make_float2(y[2 * k] * inv_c, y[2 * k + 1] * inv_c);
#pragma unroll
    for (int j = 0; j < kF8Parts; ++j) {
      const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(z, __NV_SATFINITE, __NV_E4M3);
      w[j][k >> 1] |= static_cast<uint32_t>(q) << (16 * (k & 1));
      if (j + 1 < kF8Parts) {
        const uint32_t h = e4m3x2_to_f16x2(q);
        z = make_float2((z.x - f16_lo(h)) * 16.f, (z.y - f16_hi(h)) * 16.f);
      }
    }
  }
  const uint32_t sub = 8u * (c & 1);
#pragma unroll
  for (int j = 0; j < kF8Parts; ++j) {
    const int row = 32 * j + qi;
    const uint32_t rb = qbase + row * 128;
    st_shared_v2(rb + (((c >> 1) ^ (row & 7)) << 4) + sub, w[j][0], w[j][1]);
    st_shared_v2(rb + (((4 + (c >> 1)) ^ (row & 7)) << 4) + sub, w[j][2], w[j][3]);
  }
}

// Max over a warp of a non-negative float.
__device__ __forceinline__ float warp_max_nonneg(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// First unit after the segment that holds unit u.
__device__ __forceinline__ int64_t next_segment(const PlanCore &P, int n_blocks, int64_t u) {
  const UnitPos x = unit_pos(P, n_blocks, u);
  return x.seg_first + x.tiles;
}

// Prologue of warps 2-7 (nt = 192), or of warps 2-5 alone (nt = 128) while warps 6-7
// write the CTA's new tokens: the metadata of segment 0 (warp 2), then its
// queries rotated into the Q~ buffer.
template <bool kFp8>
__device__ void query_prologue(const DecodeArgs &a, TcSmem &S, int64_t u0, int64_t u1, int nt) {
  const int t = threadIdx.x - kWarpSoft * 32;  // 0 .. nt-1
  const int w = t >> 5, lane = t & 31;
  const int G = a.n_q_heads / a.n_kv_heads;
  auto sync = [nt]() {
    if (nt == 192)
      asm volatile("bar.sync 3, 192;" ::: "memory");
    else
      asm volatile("bar.sync 3, 128;" ::: "memory");
  };
  sync();
  const SegQ &X = S.cp.pre[0];
  const int nq = min(X.m.n_ref * G, kN);
  // items t and t + nt of the nq * 8 <= 256 (column, 16-byte chunk) items
  const int n_items = nq * 8;
  const int t1 = t + nt;
  const uint32_t qbase = smem_u32(S.q);
  QItem q0, q1;
  if (t < n_items) load_item(a, X, t >> 3, t & 7, q0);
  if (t1 < n_items) load_item(a, X, t1 >> 3, t1 & 7, q1);
  if constexpr (kFp8) {
    // the segment's head scales, the largest |Q~| over all items, then parts
    float ks = 1.f, vs = 1.f;
    if (t == 0) {
      const int h = unit_pos(S.ps.plan, a.n_blocks, u0).h;
      ks = __ldg(a.k_scale + h);
      vs = __ldg(a.v_scale + h);
    }
    float y0[16], y1[16], mx = 0.f;
    if (t < n_items) mx = rot_item_f32(a, S, q0, t & 7, y0);
    if (t1 < n_items) mx = fmaxf(mx, rot_item_f32(a, S, q1, t1 & 7, y1));
    mx = warp_max_nonneg(mx);
    if (lane == 0) S.qmax[w] = __float_as_int(mx);
    sync();
    for (int k = 0; k < nt / 32; ++k) mx = fmaxf(mx, __int_as_float(S.qmax[k]));
    const int e = part_exponent(mx);
    const float inv_c = ldexpf(1.f, -e);
    if (t < n_items) store_item_e4m3(qbase, t >> 3, t & 7, y0, inv_c);
    if (t1 < n_items) store_item_e4m3(qbase, t1 >> 3, t1 & 7, y1, inv_c);
    if (t == 0) {
      S.meta_nref = X.m.n_ref;
      S.q_mul = ldexpf(ks, e);
      S.v_mul[0] = vs;
    }
    fence_proxy_async_smem();
    sync();
    if (t == 0) mbar_arrive(&S.q_full);  // phase 0: segment 0
    return;
  }
  if (t < n_items) {
    uint4 v[4];
    rot_item(a, S, q0, t & 7, v);
    store_item(qbase, t >> 3, t & 7, v);
  }
  if (t1 < n_items) {
    uint4 v[4];
    rot_item(a, S, q1, t1 & 7, v);
    store_item(qbase, t1 >> 3, t1 & 7, v);
  }
  if (t == 0) S.meta_nref = X.m.n_ref;
  fence_proxy_async_smem();
  sync();
  if (t == 0) {
    mbar_arrive(&S.q_full);  // phase 0: segment 0
    HW_TRACE_AT(a, 3);
  }
}

// The CTA's new tokens (hw_attn_append_decode_planned), by warps 6-7: for
// every (row, kv head) whose appended token lies in a tile of this CTA, the
// key rotated at its block-local position - in fp32 from the stored values,
// rounded once to bf16, the block commit's arithmetic - and the value copied,
// into the cache rows that tile's copies will read.  The writes are fenced
// for the async proxy before the producer is released.
// (E4M3 caches: the rotated key divided by its head's k_scale, the value by
// v_scale, each rounded to the nearest code, saturating.)
template <bool kFp8>
__device__ void append_tokens(const DecodeArgs &a, TcSmem &S, int64_t u0, int64_t u1) {
  const int tq = threadIdx.x - kWarpQ * 32;  // 0..63
  const int lane = tq & 31, wq = tq >> 5;
  const PlanCore &P = S.ps.plan;
  const int Hkv = a.n_kv_heads, npairs = a.n_rows * Hkv;
  const __nv_bfloat16 *kn = static_cast<const __nv_bfloat16 *>(a.k_new);
  const __nv_bfloat16 *vn = static_cast<const __nv_bfloat16 *>(a.v_new);
  __nv_bfloat16 *kc = static_cast<__nv_bfloat16 *>(const_cast<void *>(a.k));
  __nv_bfloat16 *vc = static_cast<__nv_bfloat16 *>(const_cast<void *>(a.v));
  uint8_t *kc8 = static_cast<uint8_t *>(const_cast<void *>(a.k));
  uint8_t *vc8 = static_cast<uint8_t *>(const_cast<void *>(a.v));
  auto code = [](float x) {  // nearest E4M3 code, ties to even, saturating
    return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
  };
  // one (row, kv head) token by the whole warp: lane l the pairs (l, l + 64)
  // and (l + 32, l + 96)
  auto write_token = [&](int pr, int pos, int row) {
    const int r = pr / Hkv, h = pr - r * Hkv;
    const int64_t s_off = (static_cast<int64_t>(r) * Hkv + h) * 128;
    const int64_t d_off = (static_cast<int64_t>(h) * a.capacity + row) * 128;
    float kinv = 1.f, vinv = 1.f;
    if constexpr (kFp8) {
      kinv = 1.f / __ldg(a.k_scale + h);
      vinv = 1.f / __ldg(a.v_scale + h);
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int i = lane + 32 * half;
      const float x0 = __bfloat162float(kn[s_off + i]), x1 = __bfloat162float(kn[s_off + i + 64]);
      float cs, sn;
      rope_cos_sin(pos, a.phase[i], &cs, &sn);
      const float y0 = __fmaf_rn(x0, cs, -__fmul_rn(x1, sn));
      const float y1 = __fmaf_rn(x1, cs, __fmul_rn(x0, sn));
      if constexpr (kFp8) {
        kc8[d_off + i] = code(y0 * kinv);
        kc8[d_off + i + 64] = code(y1 * kinv);
        vc8[d_off + i] = code(__bfloat162float(vn[s_off + i]) * vinv);
        vc8[d_off + i + 64] = code(__bfloat162float(vn[s_off + i + 64]) * vinv);
      } else {
        kc[d_off + i] = __float2bfloat16_rn(y0);
        kc[d_off + i + 64] = __float2bfloat16_rn(y1);
        vc[d_off + i] = vn[s_off + i];
        vc[d_off + i + 64] = vn[s_off + i + 64];
      }
    }
  };
  if (S.cp.app_n <= kAppList) {
    // the plan lists them
    for (int e = wq; e < S.cp.app_n; e += 2) write_token(S.cp.app_pair[e], S.cp.app_pos[e], S.cp.app_row[e]);
  } else {
    // more than the plan lists: every (row, kv head) pair is checked
    for (int base = wq * 32; base < npairs; base += 64) {
      const int pr = base + lane;
      int pos = 0, row = 0;
      bool mine = false;
      if (pr < npairs) {
        const int r = pr / Hkv, h = pr - r * Hkv;
        const int b = __ldg(a.append_block + r);
        if (b >= 0 && b < a.n_blocks && P.tiles[b] > 0) {
          pos = __ldg(a.append_pos + r);
          if (pos >= 0 && pos < P.len[b]) {
            // (every CTA reading the token's tile, for any column group, writes
            // it - the same bytes - before its own copy of the tile)
            mine = tile_unit_in(P, b, h, pos / kT, u0, u1) >= 0;
            row = P.start[b] + pos;
          }
        }
      }
      unsigned m = __ballot_sync(0xffffffffu, mine);
      while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        write_token(__shfl_sync(0xffffffffu, pr, src), __shfl_sync(0xffffffffu, pos, src),
                    __shfl_sync(0xffffffffu, row, src));
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  NamedSync<2, 64>()();
  if (tq == 0) mbar_arrive(&S.app_bar);
}

// Rotated queries of segments 1, 2, ... (segment 0 came from the prologue),
// and the arrivals of finished segments.  The values of segment j are loaded
// (from L2: prefetched two segments ahead) and computed in registers while
// the tensor cores still work on segment j - 1; they are written once the
// single Q~ buffer is released.  Then the warps count segment j - 2's
// records (fence + one atomic per view reference and q head): two segments
// late, so that neither these global-memory operations nor the softmax
// warps' record stores sit on the path of the next rotated queries.  Last,
// the metadata of segment j + 2 goes into the slot segment j - 2 vacated,
// and its queries are prefetched into L2.
template <bool kLimit, bool kFp8>
__device__ void qprep(const DecodeArgs &a, TcSmem &S, int64_t u0, int64_t u1) {
  const int tq = threadIdx.x - kWarpQ * 32;  // 0..63
  const int lane = threadIdx.x & 31, wq = tq >> 5;
  const int G = a.n_q_heads / a.n_kv_heads;
  NamedSync<2, 64> sync;
  const uint32_t qbase = smem_u32(S.q);
  auto arrivals = [&](int done) {
    // A wait that gives up (HW_DEV_TIMEOUT) does not leave the loop: both
    // warps keep the same control flow so the named barrier stays balanced.
    wait_or_abort(S, a, &S.rec_ready[done & 3], (done >> 2) & 1);
    if (wq == 0) arrive_segment(a, S.cp.pre[done % kPre].m, lane);
    if (tq == 0) HW_TRACE_AT(a, 7);
  };
  int64_t u = S.cp.us[1];  // segment 1
  int64_t u_prep = S.cp.us[kPre - 1] < u1 ? next_segment(S.ps.plan, a.n_blocks, S.cp.us[kPre - 1]) : u1;  // segment kPre
  for (int seg = 1;; ++seg) {
    if (u >= u1) {
      // no segment seg.  Until the last records arrive, prepare the merge
      // (a plan brings it): ranks and group indices, and the list of the
      // CTA's first item - once the softmax warps are past their first
      // tiles, so as not to slow them
      if (seg >= 2) arrivals(seg - 2);
      arrivals(seg - 1);
      break;
    }
    const SegQ &X = S.cp.pre[seg % kPre];
    const int nq = min(X.m.n_ref * G, kN);
    // items tq + 64 k of the nq * 8: column (tq >> 3) + 8 k, chunk tq & 7
    QItem raw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if ((tq >> 3) + 8 * k < nq) load_item(a, X, (tq >> 3) + 8 * k, tq & 7, raw[k]);
    if constexpr (kFp8) {
      float ks = 1.f, vs = 1.f;
      if (tq == 0) {
        const int h = unit_pos(S.ps.plan, a.n_blocks, u).h;
        ks = __ldg(a.k_scale + h);
        vs = __ldg(a.v_scale + h);
      }
      float y[4][16], mx = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if ((tq >> 3) + 8 * k < nq) mx = fmaxf(mx, rot_item_f32(a, S, raw[k], tq & 7, y[k]));
      mx = warp_max_nonneg(mx);
      if (lane == 0) S.qmax[6 + wq] = __float_as_int(mx);
      sync();
      mx = fmaxf(__int_as_float(S.qmax[6]), __int_as_float(S.qmax[7]));
      const int e = part_exponent(mx);
      const float inv_c = ldexpf(1.f, -e);
      wait_or_abort(S, a, &S.q_empty, (seg - 1) & 1);
      if (tq == 0) {
        S.meta_nref = X.m.n_ref;
        S.q_mul = ldexpf(ks, e);
        S.v_mul[seg & 3] = vs;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if ((tq >> 3) + 8 * k < nq) store_item_e4m3(qbase, (tq >> 3) + 8 * k, tq & 7, y[k], inv_c);
    } else {
      uint4 v[4][4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if ((tq >> 3) + 8 * k < nq) rot_item(a, S, raw[k], tq & 7, v[k]);
      // The Q~ buffer and the hand-off metadata are free once segment seg-1's
      // QK products completed and every softmax warp read the hand-off.
      wait_or_abort(S, a, &S.q_empty, (seg - 1) & 1);
      if (tq == 0) S.meta_nref = X.m.n_ref;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if ((tq >> 3) + 8 * k < nq) store_item(qbase, (tq >> 3) + 8 * k, tq & 7, v[k]);
    }
    fence_proxy_async_smem();
    sync();
    if (tq == 0) mbar_arrive(&S.q_full);
    if (seg >= 2) {
      arrivals(seg - 2);
      sync();  // the slot of segment seg - 2 is read; it now takes segment seg + 2
      if (u_prep < u1) {
        const UnitPos x = unit_pos(S.ps.plan, a.n_blocks, u_prep);
        SegQ &N = S.cp.pre[(seg + 2) % kPre];
        if (wq == 0) seg_pre<kLimit>(a, S.ps.plan, S.ps.cache, N, x.b, x.g, x.h, lane);
        u_prep = x.seg_first + x.tiles;
      }
      sync();
    }
    u = next_segment(S.ps.plan, a.n_blocks, u);
  }
}

// Butterfly transpose-reduce over the warp: on entry v[j] is this lane's
// value of column j; on exit lane j holds op over all 32 lanes of column j
// in v[0] (31 shuffles for 32 columns).
template <bool MAX>
__device__ __forceinline__ void transpose_reduce(float (&v)[kN], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
#pragma unroll
    for (int k = 0; k < off; ++k) {
      const bool up = (lane & off) != 0;
      const float mine = up ? v[k + off] : v[k];
      const float other = __shfl_xor_sync(0xffffffffu, up ? v[k] : v[k + off], off);
      v[k] = MAX ? fmaxf(mine, other) : mine + other;
    }
  }
}

// Records of a finished segment: O (TMEM buffer seg & 1) and the handed-over
// (m, l) of each query head -> partial records in the workspace.  Runs one
// tile after the segment's end, when its last P.V product has (nearly always)
// completed; the arrivals are left to the query warps.
// (E4M3 caches: O = O_hi + O_lo / 16, times the v_scale of the segment's kv
// head.)
template <bool kFp8>
__device__ void segment_records(const DecodeArgs &a, TcSmem &S, uint32_t tl, int seg, int64_t sid,
                                int nq, int ws, int lane, int row, NamedSync<1, 128> sync,
                                float vmul, bool fin) {
  using R = Ring<kFp8>;
  wait_or_abort(S, a, &S.o_full[seg & 1], (seg >> 1) & 1);
  tc_fence_after();
  __syncwarp();
  uint32_t o[32];
  tmem_ld32(tl + R::CO + (seg & 1) * R::OC, o);
  tmem_wait_ld();
  if constexpr (kFp8) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // O_lo, 16 columns at a time
      uint32_t t[16];
      tmem_ld16(tl + R::CO + (seg & 1) * R::OC + kN + 16 * h, t);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j)
        o[16 * h + j] = __float_as_uint(__fmaf_rn(__uint_as_float(t[j]), 0.0625f, __uint_as_float(o[16 * h + j])));
    }
  }
  // E4M3: l of column `lane` from the L buffer (every TMEM row holds every
  // column's sum), L_hi + L_lo / 16, without the 2^6 of P
  // (lane 0's row, through lsave, which E4M3 does not use otherwise)
  float l_col = 0.f;
  if (kFp8 && ws == 0) {
    float(*ls)[kN] = S.lsave[seg & 1];
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // L_hi 0-15, 16-31, L_lo 0-15, 16-31
      uint32_t t[16];
      tmem_ld16(tl + R::LC + (seg & 1) * R::OC + (q >> 1) * kN + 16 * (q & 1), t);
      tmem_wait_ld();
      if (lane == 0) {
#pragma unroll
        for (int c = 0; c < 16; ++c) ls[q >> 1][16 * (q & 1) + c] = __uint_as_float(t[c]);
      }
    }
    __syncwarp();
    l_col = __fmaf_rn(ls[1][lane], 0.0625f, ls[0][lane]) * kPUnscaleF8;
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&S.o_empty[seg & 1]);
  sync();  // every warp's lsave of this segment is in place
  const int64_t slot = sid + S.cp.c_log;
  if constexpr (kFp8) {
#pragma unroll
    for (int j = 0; j < kN; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * vmul);
  }
  // 16-byte stores, 8 instructions a thread instead of 32 scalar ones (the
  // tail's cost follows its count of global store instructions: the scalar
  // stores took ~0.86 us, measured with globaltimer stamps).  The CTA's last
  // records (fin: every copy and product is done, the ring is idle) go
  // through stage 0; the others by a 4 x 4 transpose within each group of
  // four lanes, which gives lane 4q + r the elements d = 4q .. 4q+3 (of the
  // warp's 32) of column 4b + r, for each block b of four columns.
  if (fin) {
    float *stg = reinterpret_cast<float *>(S.stage[0]);
    constexpr int kPitch = 132;  // floats a column: 16-B rows, conflict-free
#pragma unroll
    for (int j = 0; j < kN; ++j) stg[j * kPitch + row] = __uint_as_float(o[j]);
    sync();
    const int t = threadIdx.x - kWarpSoft * 32;  // 0..127
#pragma unroll
    for (int k = 0; k < kN * 128 / 4 / 128; ++k) {
      const int f4 = k * 128 + t, j = f4 >> 5, c = f4 & 31;  // column j, chunk c of 32
      if (j < nq)
        *reinterpret_cast<float4 *>(record_ptr(a, slot, j) + 4 * c) =
            *reinterpret_cast<const float4 *>(stg + j * kPitch + 4 * c);
    }
  } else {
    const int r4 = lane & 3;
    const int d0 = row - r4;  // first element of the lane's group
#pragma unroll
    for (int b = 0; b < kN / 4; ++b) {
      float v0 = __uint_as_float(o[4 * b]), v1 = __uint_as_float(o[4 * b + 1]);
      float v2 = __uint_as_float(o[4 * b + 2]), v3 = __uint_as_float(o[4 * b + 3]);
      const bool odd = lane & 1, hi = lane & 2;
      float t = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
      if (odd) v0 = t; else v1 = t;
      t = __shfl_xor_sync(0xffffffffu, odd ? v2 : v3, 1);
      if (odd) v2 = t; else v3 = t;
      t = __shfl_xor_sync(0xffffffffu, hi ? v0 : v2, 2);
      if (hi) v0 = t; else v2 = t;
      t = __shfl_xor_sync(0xffffffffu, hi ? v1 : v3, 2);
      if (hi) v1 = t; else v3 = t;
      const int j = 4 * b + r4;
      if (j < nq) *reinterpret_cast<float4 *>(record_ptr(a, slot, j) + d0) = make_float4(v0, v1, v2, v3);
    }
  }
  if (ws == 0 && lane < nq) {
    const float(*ls)[kN] = S.lsave[seg & 1];
    const float l = kFp8 ? l_col : ls[0][lane] + ls[1][lane] + ls[2][lane] + ls[3][lane];
    *reinterpret_cast<float2 *>(record_ptr(a, slot, lane) + 128) = make_float2(S.msave[seg & 1][lane], l);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&S.rec_ready[seg & 3]);
  if (threadIdx.x == kWarpSoft * 32) HW_TRACE_AT(a, 6);
}

// kLimit: the plan carries view limits, so a column may attend only part of
// a block.  kFp8: E4M3 caches (four S parts; P as two E4M3 parts).
template <bool kLimit, bool kFp8>
__device__ void softmax_role(const DecodeArgs &a, TcSmem &S, uint32_t tmem, int64_t u0,
                             int64_t u1) {
  using R = Ring<kFp8>;
  constexpr float lazy = kFp8 ? kLazyF8 : kLazy;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ws = warp - kWarpSoft;              // 0..3
  const int qd = warp & 3;                      // TMEM lane quadrant of this warp
  const int row = qd * 32 + lane;               // token of the tile (S) / element d (O)
  const uint32_t tl = tmem + (static_cast<uint32_t>(qd * 32) << 16);
  const int G = a.n_q_heads / a.n_kv_heads;
  const int n = static_cast<int>(u1 - u0);
  NamedSync<1, 128> sync;

  // A wait that gives up (HW_DEV_TIMEOUT) does not leave the loop: every
  // thread of the group keeps the same control flow, so the named barriers
  // below are always reached by all 128 threads; after an abort no wait
  // blocks any more and the CTA runs to its end on stale data.
  // m_run[j]: reference max of column j (the same in every lane); m_mine:
  // the one of column `lane`, from which the others are broadcast.  They
  // start at -FLT_MAX, not -inf: a column that a view limit keeps from every
  // token of its segment then gets p = 2^(-inf) = 0 (l = 0, an empty record)
  // where -inf - -inf would give NaN.
  float m_run[kN], l_part[kN], m_mine = -FLT_MAX;
  int seg = -1, nq = 0;
  // view limits of the segment: the fewest tokens a column attends, and the
  // count of column `lane` (broadcast to the others on the tiles that need it)
  int minlim = INT_MAX, lim_mine = INT_MAX;
  float qmul = 1.f, vmul = 1.f, pend_vmul = 1.f;  // E4M3: score and output factors
  int pend = -1, pend_nq = 0;  // segment whose records are due
  int64_t pend_sid = 0;        // (its seg_id)
  UnitPos x = unit_pos(S.ps.plan, a.n_blocks, u0);  // then advanced unit by unit
  for (int i = 0; i < n; ++i) {
    const int64_t u = u0 + i;
    if (i > 0) unit_pos_next(S.ps.plan, a.n_blocks, x);
    const bool first = seg_first_unit(x, u, u0), last = seg_last_unit(x, u, u1);
    if (first) {
      ++seg;
      wait_or_abort(S, a, &S.q_full, seg & 1);
      nq = min(S.meta_nref * G, kN);
      if constexpr (kFp8) {
        qmul = S.q_mul;
        vmul = S.v_mul[seg & 3] * kPUnscaleF8;  // (O is 2^6 times too large)
      }
      if constexpr (kLimit) {
        // the segment's metadata stays in its slot until its records are out
        const SegQ &X = S.cp.pre[seg % kPre];
        const int len = S.ps.plan.len[x.b];
        minlim = X.minlim;
        lim_mine = len;
        if (minlim < len && lane < nq)
          lim_mine = entry_limit(a.view_limit, X.m.ref_entry[lane / G], len);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.q_empty);  // this warp has read the hand-off
#pragma unroll
      for (int j = 0; j < kN; ++j) {
        m_run[j] = -FLT_MAX;
        l_part[j] = 0.f;
      }
      m_mine = -FLT_MAX;
    }
    const int sb = i & 1, s = i % R::NS;
    const int base = x.t * kT;  // the tile's first token in its block
    const int valid = min(kT, S.ps.plan.len[x.b] - base);
    const bool tok_ok = row < valid;
    wait_or_abort(S, a, &S.s_full[sb], (i >> 1) & 1);
    if (threadIdx.x == kWarpSoft * 32 && i == 0) HW_TRACE_AT(a, 4);
    if (threadIdx.x == kWarpSoft * 32 && i == n - 1) {
      HW_TRACE_AT(a, 5);
      HW_TRACE_VAL(a, 21, n);
    }
    tc_fence_after();
    __syncwarp();
    uint32_t r[32], r2[32];
    tmem_ld32(tl + sb * R::SC, r);        // S_hi (E4M3: part 0)
    tmem_ld32(tl + sb * R::SC + kN, r2);  // S_lo (E4M3: part 1)
    tmem_wait_ld();
    if constexpr (kFp8) {
#pragma unroll
      for (int j = 0; j < kN; j += 2)
        pair_put(r, j, __ffma2_rn(pair_at(r2, j), fpair(0.0625f), pair_at(r, j)));
      tmem_ld32(tl + sb * R::SC + 2 * kN, r2);  // part 2
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < kN; j += 2)
        pair_put(r, j, __ffma2_rn(pair_at(r2, j), fpair(0.00390625f), pair_at(r, j)));
      tmem_ld32(tl + sb * R::SC + 3 * kN, r2);  // part 3
      tmem_wait_ld();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.s_empty[sb]);
    if constexpr (kFp8) {
#pragma unroll
      for (int j = 0; j < kN; j += 2)
        pair_put(r, j, __fmul2_rn(__ffma2_rn(pair_at(r2, j), fpair(0.000244140625f), pair_at(r, j)),
                                  fpair(qmul)));
    } else {
#pragma unroll
      for (int j = 0; j < kN; j += 2) pair_put(r, j, __fadd2_rn(pair_at(r, j), pair_at(r2, j)));
    }

    float sc[kN];
    if (!kLimit || base + kT <= minlim) {
#pragma unroll
      for (int j = 0; j < kN; ++j) sc[j] = __uint_as_float(r[j]);
      if (!tok_ok) {  // (a row past the block end: a ragged tile only)
#pragma unroll
        for (int j = 0; j < kN; ++j) sc[j] = -INFINITY;
      }
    } else {
      // some column's view limit ends in this tile (a chunk's own tokens);
      // limits never exceed the block, so they cover valid too
#pragma unroll
      for (int j = 0; j < kN; ++j) {
        const int lim = __shfl_sync(0xffffffffu, lim_mine, j);
        sc[j] = (tok_ok && base + row < lim) ? __uint_as_float(r[j]) : -INFINITY;
      }
    }

    // Lazy rescaling: the reference max m_run moves only when some score
    // exceeds it by more than kLazy (log2 units; E4M3: kLazyF8), so p <= 2^kLazy and O is
    // rarely touched.  The common case needs only this one CTA-group vote;
    // exact column maxima are taken on the rare tiles that need them (the
    // first tile of a segment always does: m_run starts at -inf).
    bool exceed = false;
#pragma unroll
    for (int j = 0; j < kN; ++j) exceed |= (j < nq) && (sc[j] > m_run[j] + lazy);
    if (bar_red_or_128(exceed)) {
      float(*red)[4] = S.red[i & 1];
      float v[kN];
#pragma unroll
      for (int j = 0; j < kN; ++j) v[j] = sc[j];
      transpose_reduce<true>(v, lane);
      red[lane][ws] = v[0];
      sync();
      // lane j: the tile maximum of column j over the four warps, the new
      // reference and its rescale factor (0 when the old one was -inf);
      // then every lane takes all 32 by shuffles
      const float4 t4 = *reinterpret_cast<const float4 *>(red[lane]);
      const float tmax = fmaxf(fmaxf(t4.x, t4.y), fmaxf(t4.z, t4.w));
      const float m_old = m_mine;
      if (lane < nq && tmax > m_old + lazy) m_mine = tmax;
      const float a_mine = (m_mine == m_old) ? 1.f : ex2(m_old - m_mine);
      float alpha[kN];
#pragma unroll
      for (int j = 0; j < kN; ++j) {
        m_run[j] = __shfl_sync(0xffffffffu, m_mine, j);
        alpha[j] = __shfl_sync(0xffffffffu, a_mine, j);
        if (!kFp8) l_part[j] *= alpha[j];
      }
      if (!first) {
        // O must hold every earlier tile before it is rescaled
        wait_or_abort(S, a, &S.p_empty, (i - 1) & 1);
        tc_fence_after();
        __syncwarp();
#pragma unroll
        for (int h = 0; h < (kFp8 ? 4 : 1); ++h) {  // (E4M3: O_hi, O_lo, L_hi, L_lo)
          const uint32_t col = (h < 2 ? R::CO : R::LC) + (seg & 1) * R::OC + (h & 1) * kN;
          uint32_t o[32];
          tmem_ld32(tl + col, o);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < kN; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha[j]);
          tmem_st32(tl + col, o);
          tmem_wait_st();
        }
        tc_fence_before();
      }
    }
    // P row of this token: 64 bytes (bf16: 32 heads; E4M3: the 32 hi codes,
    // then the 32 lo codes) = four 16-B chunks.  The sum uses the same
    // rounded weights the P.V product sees.
    uint32_t pk[16];
    if constexpr (kFp8) {
#pragma unroll
      for (int k = 0; k < 16; ++k) pk[k] = 0;
#pragma unroll
      for (int j = 0; j < kN; j += 2) {
        const float2 d = __fadd2_rn(make_float2(sc[j], sc[j + 1]), make_float2(-m_run[j], -m_run[j + 1]));
        const float p0 = (j < nq) ? ex2(d.x) : 0.f;
        const float p1 = (j + 1 < nq) ? ex2(d.y) : 0.f;
        // 2^6 p (see kPScaleF8, <= 256 < 448) as hi + lo / 16: hi its
        // nearest code, lo that of the residual of its f16 value times 16
        // (E4M3's grid, subnormals included: about 8 significant bits in all,
        // like the bf16 path's P).  l is the tensor cores' sum of these very
        // codes (the ones product).  (The conversion instructions: splitting
        // with fp32 arithmetic instead - Veltkamp's split - took ~40 % more
        // per tile.)
        const float2 sv = __fmul2_rn(make_float2(p0, p1), fpair(kPScaleF8));
        const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(sv, __NV_SATFINITE, __NV_E4M3);
        const uint16_t lo = e4m3x2_residual(sv, e4m3x2_to_f16x2(h));
        pk[j >> 2] |= static_cast<uint32_t>(h) << (16 * ((j >> 1) & 1));
        pk[8 + (j >> 2)] |= static_cast<uint32_t>(lo) << (16 * ((j >> 1) & 1));
      }
    } else {
#pragma unroll
      for (int j = 0; j < kN; j += 2) {
        const float2 d = __fadd2_rn(make_float2(sc[j], sc[j + 1]), make_float2(-m_run[j], -m_run[j + 1]));
        const float p0 = (j < nq) ? ex2(d.x) : 0.f;
        const float p1 = (j + 1 < nq) ? ex2(d.y) : 0.f;
        pk[j / 2] = pack_bf16(p0, p1);
        const float2 lsum = __fadd2_rn(make_float2(l_part[j], l_part[j + 1]),
                                       make_float2(__uint_as_float(pk[j / 2] << 16),
                                                   __uint_as_float(pk[j / 2] & 0xffff0000u)));
        l_part[j] = lsum.x;
        l_part[j + 1] = lsum.y;
      }
    }
    if (valid < kT) {
      // V rows past the block end may hold anything: zero them (p = 0 there,
      // but 0 * NaN would still poison the sum)
      wait_or_abort(S, a, &S.v_full[s], (i / R::NS) & 1);
      if (!tok_ok) {
        const uint32_t v0 = smem_u32(stage_ptr<kFp8>(S, s)) + R::VOFF + row * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          st_shared_v4(v0 + c * 16, 0, 0, 0, 0);
          if (!kFp8) st_shared_v4(v0 + kBox + c * 16, 0, 0, 0, 0);
        }
      }
    }
    // in the K region of the tile's stage (QK of this tile has completed:
    // s_full), 64-B swizzle
    const uint32_t prow = smem_u32(stage_ptr<kFp8>(S, s)) + row * 64;
    const uint32_t swz = (row >> 1) & 3;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      st_shared_v4(prow + ((c ^ swz) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.p_full[s]);
    if (threadIdx.x == kWarpSoft * 32) *reinterpret_cast<volatile int32_t *>(&S.tiles_done) = i + 1;

    if (pend >= 0) {  // records of the previous segment, one tile late
      segment_records<kFp8>(a, S, tl, pend, pend_sid, pend_nq, ws, lane, row, sync, pend_vmul, false);
      pend = -1;
    }
    if (last) {
      // hand over (m, l) of every query head; the records follow one tile later
      if constexpr (!kFp8) {  // (E4M3: l comes from TMEM with the records)
        float v[kN];
#pragma unroll
        for (int j = 0; j < kN; ++j) v[j] = l_part[j];
        transpose_reduce<false>(v, lane);
        S.lsave[seg & 1][ws][lane] = v[0];
      }
      if (ws == 0) S.msave[seg & 1][lane] = m_mine;
      pend = seg;
      pend_sid = seg_id(S.ps.plan, x.b, x.g, x.h);
      pend_nq = nq;
      pend_vmul = vmul;
    }
  }
  if (pend >= 0)
    segment_records<kFp8>(a, S, tl, pend, pend_sid, pend_nq, ws, lane, row, sync, pend_vmul, true);
}

constexpr int kPlanWarps = kThreads / 32;

__device__ __forceinline__ void copy16(uint8_t *dst, const void *src, size_t bytes, int tid, int nt) {
  const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
  uint4 *d4 = reinterpret_cast<uint4 *>(dst);
  for (size_t i = tid; i < bytes / 16; i += nt) d4[i] = s4[i];
}

// Record of decode CTA c of R (into cp, and then, unless `plan` is null, at
// the position of the CTA's rank in `plan`), by a group of nw warps (wi: this
// warp's index in it; sync: the group's barrier): warp 0 derives the unit
// range, first tiles, rank and new tokens, then the warps share the first
// segments' query metadata and the first merge lists.  ubeg: first unit of
// every decode CTA ([R] = U); rank_tmp: per-warp scratch of merge_list.
template <typename Sync>
__device__ void plan_record(const DecodeArgs &a, const PlanShared &ps, const int64_t *ubeg,
                            CtaPlan &cp, int32_t (*rank_tmp)[HW_MAX_VIEW_BLOCKS], int c, int R,
                            uint8_t *plan, int wi, int nw, int lane, Sync sync) {
  const PlanCore &P = ps.plan;
  const int64_t u0 = ubeg[c], u1 = ubeg[c + 1];
  if (wi == 0) {
    if (lane == 0) {
      cp.u0 = u0;
      cp.u1 = u1;
      cp.c_log = c;
      int64_t u = u0;
      for (int k = 0; k < kPre; ++k) {
        cp.us[k] = u;
        if (u < u1) u = next_segment(P, a.n_blocks, u);
      }
    }
    // the first tiles (the ring's first fill)
    const int nf = static_cast<int>(min(static_cast<int64_t>(kStages), u1 - u0));
    if (lane < kStages) {
      TileRef t = {0, 0, 0};
      if (lane < nf) t = tile_ref(P, a.n_blocks, u0 + lane, u0, u1);
      cp.trow[lane] = t.row;
      cp.th[lane] = static_cast<uint8_t>(t.h);
      cp.tfl[lane] = t.flags;
    }
    if (lane == 0) cp.n_first = static_cast<uint8_t>(nf);
    // its rank by units (which CTAs merge: merge_ctas): the CTAs with more
    // units, or as many and a lower index, come first
    const int64_t mine = u1 - u0;
    int before = 0;
    for (int c2 = lane; c2 < R; c2 += 32) {
      const int64_t u2 = ubeg[c2 + 1] - ubeg[c2];
      before += c2 != c && (u2 > mine || (u2 == mine && c2 < c)) ? 1 : 0;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
    if (lane == 0) cp.mrank = before;
    // the step's new tokens that lie in its tiles (a token outside its
    // block is an error and skipped): how many, the first tile that holds
    // one, and the first kAppList of them
    int app_n = 0, app_tile = INT_MAX;
    if (a.append_block) {
      const int Hkv = a.n_kv_heads, npairs = a.n_rows * Hkv;
      for (int base = 0; base < npairs; base += 32) {
        const int pr = base + lane;
        bool in = false;
        int row = 0, pos = 0;
        int64_t u = -1;
        if (pr < npairs) {
          const int r = pr / Hkv, h = pr - r * Hkv;
          const int b = __ldg(a.append_block + r);
          if (b >= 0) {
            pos = __ldg(a.append_pos + r);
            if (b >= a.n_blocks || pos < 0 || pos >= P.len[b]) {
              if (c == 0 && h == 0) flag_error(a.err, HW_DEV_BAD_RANGE);
            } else if (P.tiles[b] > 0) {  // (a block no view reads takes no part)
              // the first of its units that read the token's tile (one per
              // column group): every CTA reading it writes the token - the
              // same bytes - before its own copy of the tile
              u = tile_unit_in(P, b, h, pos / kT, u0, u1);
              in = u >= 0;
              row = P.start[b] + pos;
            }
          }
        }
        const unsigned m = __ballot_sync(0xffffffffu, in);
        const int k = app_n + __popc(m & lanemask_lt(lane));
        if (in && k < kAppList) {
          cp.app_pair[k] = pr;
          cp.app_row[k] = row;
          cp.app_pos[k] = pos;
        }
        app_n += __popc(m);
        if (in) app_tile = min(app_tile, static_cast<int>(u - u0));
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1)
        app_tile = min(app_tile, __shfl_xor_sync(0xffffffffu, app_tile, o));
    }
    if (lane == 0) {
      cp.app_n = app_n;
      cp.app_tile = app_tile;
    }
  }
  sync();
  // the query-side metadata of its first segments, then the record lists of
  // its first merge items (item k: rank + k * nm), shared by the warps
  for (int k = wi; k < kPre; k += nw) {
    if (cp.us[k] < u1) {
      const UnitPos x = unit_pos(P, a.n_blocks, cp.us[k]);
      seg_pre<true>(a, P, ps.cache, cp.pre[k], x.b, x.g, x.h, lane);
    }
  }
  const int nm = merge_ctas(a, R), mrank = cp.mrank;
  for (int k = 0; k < kPreItems; ++k) {
    if ((kPre + k) % nw != wi) continue;
    const int it = mrank + k * nm;
    int n = -1;
    if (mrank < nm && it < a.n_rows * a.n_q_heads) {
      n = merge_list(a, P, ps.cache, it / a.n_q_heads, it % a.n_q_heads, cp.mpre[k], kPreList,
                     rank_tmp[wi], lane);
      if (n > kPreList) n = -1;
    }
    if (lane == 0) cp.mpre_n[k] = n;
  }
  sync();
  // at the position of its rank: a decode launch's CTA b (CTAs are placed in
  // index order, the low ones on the SMs the previous launch frees first) runs
  // the b-th heaviest share, so the heaviest shares - which also merge - get
  // their SMs first and the light ones take the SMs freed last
  if (plan)
    copy16(const_cast<uint8_t *>(plan_cta_record(plan, mrank)), &cp, sizeof(CtaPlan),
           wi * 32 + lane, nw * 32);
  sync();  // (cp may be the group's next record)
}

__device__ __forceinline__ void write_plan_header(const DecodeArgs &a, uint8_t *plan, int grid) {
  PlanHeader h;
  h.magic = kPlanMagic;
  h.grid = grid;
  h.n_rows = a.n_rows;
  h.n_q_heads = a.n_q_heads;
  h.n_kv_heads = a.n_kv_heads;
  h.head_dim = a.head_dim;
  h.n_blocks = a.n_blocks;
  h.n_view = a.n_view;
  h.capacity = a.capacity;
  h.limited = a.view_limit != nullptr;
  *reinterpret_cast<PlanHeader *>(plan) = h;
}

struct WarpSync {
  __device__ __forceinline__ void operator()() const { __syncwarp(); }
};

// hw_attn_decode when the plan cache holds another metadata's plan (current
// buffer `cur`): every CTA builds the plan from the caller's metadata - the
// shared part, and its own record as CTA c of the split - into shared
// memory, and writes it into the other buffer for the calls that follow
// (CTA 0: the shared part, the header and the metadata copy; every CTA: its
// record at its rank).  The last CTA done makes that buffer current, before
// it lets the next launch start.  Every thread takes part.
__device__ __noinline__ void build_cached_plan(const DecodeArgs &a, TcSmem &S, int cur) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = static_cast<int>(gridDim.x);
  struct Scratch {  // in stage 0, which no copy has touched yet
    PlanScratch build;
    int64_t ubeg[kThreads + 1];
    int32_t rank_tmp[kPlanWarps][HW_MAX_VIEW_BLOCKS];
  };
  static_assert(sizeof(Scratch) <= kStageBytes, "plan scratch fits a stage");
  Scratch &Z = *reinterpret_cast<Scratch *>(S.stage[0]);
  int64_t unused[2];
  build_plan<kT>(a, S.ps.plan, S.ps.cache, Z.build, unused, R);
  plan_ranks(a, S.ps.cache, warp, lane, 0, 1);
  for (int c = tid; c <= R; c += kThreads) Z.ubeg[c] = cta_unit_begin(S.ps.plan, a.n_blocks, c);
  __syncthreads();
  const int target = cur ^ 1;
  uint8_t *plan = cache_plan(a, target);
  plan_record(a, S.ps, Z.ubeg, S.cp, Z.rank_tmp, blockIdx.x, R, plan, warp, kPlanWarps, lane,
              CtaSync());
  if (blockIdx.x == 0) {
    copy16(plan + kPlanHeaderBytes, &S.ps, sizeof(PlanShared), tid, kThreads);
    cache_write_meta(a, target, tid, kThreads);
    if (tid == 0) write_plan_header(a, plan, R);
  }
  // every CTA's stores before its arrival, the arrivals before the switch
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int32_t *st = cache_state(a);
    if (atomicAdd(st + 1, 1) == R - 1) {
      __threadfence();
      st[1] = 0;
      asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(st), "r"(target) : "memory");
      __threadfence();
    }
  }
  __syncthreads();
}

// Every launch runs from a plan: hw_attn_plan's, or (kCache) hw_attn_decode's
// plan cache, rebuilt by the launch itself when its metadata differs.
// kAppend: the layer's new tokens are written first; kLimit (no appends): the
// plan carries view limits; kFp8: E4M3 caches with per-kv-head scales.  Each
// combination is its own kernel, so that no path carries another's code (a
// second softmax loop in the same kernel, even one never entered, cost the
// plain path 8 %).
template <bool kAppend, bool kLimit, bool kFp8, bool kCache>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem &S = *reinterpret_cast<TcSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    HW_TRACE_AT(a, 0);
    unsigned sm;
    asm("mov.u32 %0, %%smid;" : "=r"(sm));
    HW_TRACE_VAL(a, 22, sm);
  }
  // Launched as a programmatic dependent of the previous kernel on the
  // stream: this CTA may start while that grid's last CTAs still run (an SM
  // holds one CTA of this kernel, so only SMs they left), and the next
  // launch may be placed likewise.  Before griddepcontrol.wait it writes no
  // global memory and reads only what cannot be in flight: an L2 prefetch of
  // q (which never changes a result) and - when the caller promised that the
  // previous work writes neither (a.early) - its plan or metadata and its
  // first K/V tiles.  The next launch on the stream may start once every CTA
  // holds its plan (below): a plan launch that follows may then rewrite it.
  if (tid == 0) {
    // the plan's barrier first: under the early-loads promise its copies are
    // issued before the other set-up
    mbar_init(&S.plan_bar, 1);
    fence_mbar_init();
    if (!kCache && a.early) issue_plan_copies(a, S);
    tma_prefetch_desc(&tm_k);  // (kernel parameters)
    tma_prefetch_desc(&tm_v);
    for (int s = 0; s < Ring<kFp8>::NS; ++s) {
      mbar_init(&S.p_full[s], 4);  // one per softmax warp
      mbar_init(&S.k_full[s], 1);
      mbar_init(&S.v_full[s], 1);
      mbar_init(&S.kv_empty[s], 1);
    }
    mbar_init(&S.q_full, 1);
    mbar_init(&S.q_empty, 5);  // last QK of the segment + each softmax warp's read
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.s_full[b], 1);
      mbar_init(&S.s_empty[b], 4);  // one per softmax warp
    }
    mbar_init(&S.p_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.o_full[b], 1);
      mbar_init(&S.o_empty[b], 4);    // one per softmax warp
    }
    for (int b = 0; b < 4; ++b) mbar_init(&S.rec_ready[b], 4);  // one per softmax warp
    mbar_init(&S.mma_done, 1);
    mbar_init(&S.app_bar, 1);
    S.abort_flag = 0;
    S.tiles_done = 0;
    S.plan_ok = 1;
    fence_mbar_init();
  }
  // this launch's RoPE table (no plan copy writes these bytes)
  if (tid >= kThreads - 64) S.ps.cache.phase[tid - (kThreads - 64)] = a.phase[tid - (kThreads - 64)];
  if (warp == kWarpMma) {
    tmem_alloc(&S.tmem_base, Ring<kFp8>::TC);
    tmem_relinquish();
  }
  if (tid == 32) {
    // Every CTA warms L2 with its share of q before any K/V tile is asked
    // for: query loads then hit L2 instead of queueing behind the tile
    // stream.  q is [n_rows][Hq][128] bf16, a multiple of 256 bytes.
    const uint64_t total = static_cast<uint64_t>(a.n_rows) * a.n_q_heads * 256;
    const uint64_t per = ((total + gridDim.x - 1) / gridDim.x + 255) & ~static_cast<uint64_t>(255);
    const uint64_t off = per * blockIdx.x;
    if (off < total) {
      const uint32_t n = static_cast<uint32_t>(total - off < per ? total - off : per);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                       reinterpret_cast<const uint8_t *>(a.q) + off), "r"(n)
                   : "memory");
    }
  }
  if (kAppend && tid == 64) {
    // likewise the layer's new tokens (k_new, v_new: [n_rows][Hkv][128] bf16),
    // which the CTAs that write them read early, under the first tiles
    const uint64_t total = static_cast<uint64_t>(a.n_rows) * a.n_kv_heads * 256;
    const uint64_t per = ((total + gridDim.x - 1) / gridDim.x + 255) & ~static_cast<uint64_t>(255);
    const uint64_t off = per * blockIdx.x;
    if (off < total) {
      const uint32_t n = static_cast<uint32_t>(total - off < per ? total - off : per);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                       reinterpret_cast<const uint8_t *>(a.k_new) + off), "r"(n)
                   : "memory");
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                       reinterpret_cast<const uint8_t *>(a.v_new) + off), "r"(n)
                   : "memory");
    }
  }

  if constexpr (kFp8) {
    // the ones tile of the l product (E4M3 1.0 = 0x38 in every byte, so its
    // swizzle is moot), seen by the tensor cores after the barrier below
    uint4 *ones = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(S.stage) + kOnesOff);
    for (int i = tid; i < static_cast<int>(kF8Box / 16); i += kThreads)
      ones[i] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
    fence_proxy_async_smem();
  }
  // The plan: the shared part and this CTA's record, into shared memory -
  // hw_attn_plan's with two bulk copies, or the plan cache's (see "plan
  // cache") with loads through L2, or built here when the cache holds
  // another metadata's plan.  Errors it finds are recorded after
  // griddepcontrol.wait.
  bool plan_timeout = false;
  auto get_plan = [&]() {
    if constexpr (kCache) {
      // (the launch before this one, if it rebuilt the cache, switched
      // buffers before it let this one start)
      if (tid == 0) S.cache_cur = cache_current(a);
      __syncthreads();
      const int k = S.cache_cur;
      if (!cache_fetch(a, k, S.ps, S.cp, tid, kThreads)) build_cached_plan(a, S, k);
    } else {
      if (tid == 0 && !a.early) issue_plan_copies(a, S);
      __syncthreads();  // the barriers are initialised
      if (!mbar_wait(&S.plan_bar, 0)) {
        plan_timeout = true;
        S.plan_ok = 0;
      }
      if (tid == 0 &&
          !header_matches(a, *reinterpret_cast<const PlanHeader *>(S.q), static_cast<int>(gridDim.x)))
        S.plan_ok = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };
  const bool early = a.early != 0;
  int issued = 0;  // tiles the producer issued before griddepcontrol.wait
  if (early) {
    get_plan();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the first tiles into the empty ring (not past the first tile that
    // holds a new token: those are written after the wait)
    if (tid == 0 && S.plan_ok && S.cp.u0 < S.cp.u1) {
      int64_t n0 = Ring<kFp8>::NS;
      if (kAppend && S.cp.app_n > 0 && S.cp.app_tile < n0) n0 = S.cp.app_tile;
      issued = producer<kFp8>(a, S, &tm_k, &tm_v, S.cp.u0, S.cp.u1, false, 0, n0);
    }
  }
  if (tid == 0) HW_TRACE_AT(a, 1);
  // The previous grid is complete (and its writes visible to this grid) once
  // griddepcontrol.wait returns.  Under the early-loads promise one thread
  // of the query warps waits for it; the others meet that thread at the
  // query prologue's first barrier (or, without units, at the CTA barrier
  // below) before they touch q or any global state, so they start together
  // instead of waking one by one (~0.3 us a layer; bf16 caches: the E4M3
  // prologue measured no gain).
  const bool lone = early && !kAppend && !kFp8 && warp >= kWarpSoft && tid != kWarpSoft * 32;
  if (!lone) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) HW_TRACE_AT(a, 2);
  if (!early) {
    get_plan();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  if (plan_timeout) flag_error(a.err, HW_DEV_TIMEOUT);
  const uint32_t tmem = S.tmem_base;
  const bool ok = S.plan_ok != 0;
  if (!ok && tid == 0 && blockIdx.x == 0) flag_error(a.err, HW_DEV_BAD_PLAN);
  const int64_t u0 = ok ? S.cp.u0 : 0, u1 = ok ? S.cp.u1 : 0;
  if (u0 < u1) {
    const bool appending = kAppend && S.cp.app_n > 0;
    if (warp == kWarpTma) {
      if (lane == 0) {
        const int n = producer<kFp8>(a, S, &tm_k, &tm_v, u0, u1, appending, issued, u1 - u0);
        producer_drain<kFp8>(S, n);
      }
    } else if (warp == kWarpMma) {
      if (lane == 0) mma_issuer<kFp8>(a, S, tmem, u0, u1);
    } else {
      if (appending && warp >= kWarpQ)
        append_tokens<kFp8>(a, S, u0, u1);
      else
        query_prologue<kFp8>(a, S, u0, u1, appending ? 128 : 192);
      if (warp < kWarpQ)
        softmax_role<kLimit, kFp8>(a, S, tmem, u0, u1);
      else
        qprep<kLimit, kFp8>(a, S, u0, u1);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, Ring<kFp8>::TC);
  }
  // the merge scratch lives in the tile buffers: every copy and MMA is done
  static_assert(sizeof(MergeSmem<8>) <= kStageBytes, "merge scratch must fit in a stage");
  // Only the merge CTAs (merge_ctas: the ones with the most units) take
  // items; every other CTA retires here, and the next launch's CTA can take
  // its SM.
  if (tid == 0) HW_TRACE_AT(a, 8);
  if (ok)
    merge_phase<__nv_bfloat16, 128, 8>(a, S.ps.plan, S.ps.cache,
                                       *reinterpret_cast<MergeSmem<8> *>(S.stage[0]),
                                       &S.cp.mpre[0][0], S.cp.mpre_n, kPreItems, kPreList, tid,
                                       kThreads, CtaSync(), a.wait_limit, S.cp.mrank,
                                       merge_ctas(a, static_cast<int>(gridDim.x)));
  if (tid == 0) HW_TRACE_AT(a, 12);
}

// The plan of the decode launches of `o.records` CTAs (see "plans" above):
// every CTA derives the shared part, then its warps write CTA records - one
// record per warp at a time: warp w of CTA b writes records b + grid w,
// b + grid (w + 8), ... - each at the position of the CTA's rank.  CTA 0 also writes the
// metadata copies (hw_attn_plan), the shared part and the header.  With
// o.plan null and no plan cache only the metadata is copied.
constexpr int kPlanRecordsPerCta = 2 * kPlanWarps;  // a launch's grid: records / this
struct PlanSmem {
  PlanShared ps;
  PlanScratch scratch;
  int64_t ubeg[kThreads + 1];  // first unit of every decode CTA; [records] = U
  CtaPlan cp[kPlanWarps];      // the record each warp is building
  int32_t rank_tmp[kPlanWarps][HW_MAX_VIEW_BLOCKS];
};

__global__ void __launch_bounds__(kThreads, 1)
    plan_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ PlanOut o) {
  extern __shared__ uint8_t smem_raw[];
  PlanSmem &S = *reinterpret_cast<PlanSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 15) &
                                              ~static_cast<uintptr_t>(15));
  const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.n_rows * a.n_view, G = a.n_q_heads / a.n_kv_heads;
  const int R = o.records;
  // A plain launch, once per decode step.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint8_t *plan = o.plan;
  if (blockIdx.x == 0 && o.view_block) {
    for (int i = tid; i < E; i += nt) {
      o.view_block[i] = a.view_block[i];
      o.view_offset[i] = a.view_offset[i];
    }
    for (int i = tid; i < a.n_rows; i += nt) o.q_pos[i] = a.q_pos[i];
    for (int i = tid; i < a.n_blocks; i += nt) {
      o.block_start[i] = a.block_start[i];
      o.block_len[i] = a.block_len[i];
    }
    for (int i = tid; i < a.n_q_heads; i += nt) o.q_to_kv[i] = a.q_to_kv ? a.q_to_kv[i] : i / G;
    for (int i = tid; i < a.n_rows; i += nt) {
      o.append_block[i] = a.append_block ? a.append_block[i] : -1;
      o.append_pos[i] = a.append_block ? a.append_pos[i] : 0;
    }
    for (int i = tid; i < E; i += nt) o.view_limit[i] = a.view_limit ? a.view_limit[i] : -1;
  }
  if (!plan) return;
  PlanCore &P = S.ps.plan;
  int64_t unused[2];
  build_plan<kT>(a, P, S.ps.cache, S.scratch, unused, R);
  plan_ranks(a, S.ps.cache, warp, lane, 0, 1);
  for (int c = tid; c <= R; c += nt) S.ubeg[c] = cta_unit_begin(P, a.n_blocks, c);
  __syncthreads();
  for (int c = blockIdx.x + gridDim.x * warp; c < R; c += gridDim.x * kPlanWarps)
    plan_record(a, S.ps, S.ubeg, S.cp[warp], &S.rank_tmp[warp], c, R, plan, 0, 1, lane, WarpSync());
  if (blockIdx.x == 0) {
    copy16(plan + kPlanHeaderBytes, &S.ps, sizeof(PlanShared), tid, nt);
    if (tid == 0) write_plan_header(a, plan, R);
  }
}

}  // namespace

static_assert(sizeof(TcSmem) + 1024 <= 232448, "shared memory of one CTA per SM");

}  // namespace hw

extern "C" int hw_trace_read(uint64_t *dst) {
#ifdef HW_TRACE
  if (!dst) return HW_ERR_INVALID;
  return cudaMemcpyFromSymbol(dst, hw::g_trace, sizeof(hw::g_trace)) == cudaSuccess ? HW_OK : HW_ERR_CUDA;
#else
  (void)dst;
  return HW_ERR_UNSUPPORTED;
#endif
}

extern "C" int hw_trace_clear(void) {
#ifdef HW_TRACE
  static unsigned long long zero[hw::kTraceCalls][hw::kTraceCtas][hw::kTracePoints];
  return cudaMemcpyToSymbol(hw::g_trace, zero, sizeof(zero)) == cudaSuccess ? HW_OK : HW_ERR_CUDA;
#else
  return HW_ERR_UNSUPPORTED;
#endif
}

namespace hw {
size_t decode_tc_smem_bytes() { return sizeof(TcSmem) + 1024; }
size_t plan_shared_bytes() { return sizeof(PlanShared); }
size_t plan_cta_bytes() { return sizeof(CtaPlan); }

int plan_export_records(const uint8_t *plan_host, int64_t *out, int max_ctas) {
  const PlanHeader &h = *reinterpret_cast<const PlanHeader *>(plan_host);
  if (h.magic != kPlanMagic || h.grid <= 0 || h.grid > max_ctas) return -1;
  const PlanCore &P = reinterpret_cast<const PlanShared *>(plan_host + kPlanHeaderBytes)->plan;
  for (int b = 0; b < h.grid; ++b) {
    const CtaPlan &cp = *reinterpret_cast<const CtaPlan *>(
        plan_host + kPlanHeaderBytes + sizeof(PlanShared) + static_cast<size_t>(b) * sizeof(CtaPlan));
    if (cp.c_log < 0 || cp.c_log >= h.grid) return -1;
    int64_t *o = out + static_cast<int64_t>(cp.c_log) * kPlanExportFields;  // in split order
    o[0] = cp.u0;
    o[1] = cp.u1;
    o[2] = cp.n_first;
    for (int i = 0; i < kStages; ++i) {
      o[3 + i] = cp.trow[i];
      o[6 + i] = cp.th[i];
      o[9 + i] = cp.tfl[i];
      o[12 + i] = 0;
      if (i < cp.n_first) {
        // the tile's column group, from the plan's unit tables
        const int64_t local = (cp.u0 + i) % P.UH;
        int b = 0;
        while (b + 1 < h.n_blocks && P.ubase[b + 1] <= local) ++b;
        o[12 + i] = P.tiles[b] > 0 ? (local - P.ubase[b]) / P.tiles[b] : -1;
      }
    }
  }
  return h.grid;
}

cudaError_t launch_plan(const DecodeArgs &a, const PlanOut &o, cudaStream_t s) {
  const size_t smem = sizeof(PlanSmem) + 16;
  static bool configured = false;
  if (!configured) {
    const cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  // records are the decode launches' CTAs (ranked by one warp's lanes, at
  // most kThreads of them)
  if (o.records <= 0 || o.records > kThreads) return cudaErrorInvalidConfiguration;
  const int grid = o.plan ? (o.records + kPlanRecordsPerCta - 1) / kPlanRecordsPerCta : 1;
  plan_kernel<<<grid, kThreads, smem, s>>>(a, o);
  return cudaGetLastError();
}

cudaError_t launch_decode_tc(const DecodeArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                             int ctas, cudaStream_t s) {
  // a plan holds at most kThreads records (ranked by one warp's lanes)
  if (ctas > kThreads) return cudaErrorInvalidConfiguration;
  const size_t smem = decode_tc_smem_bytes();
  // planned launches run their own instantiations: without the plan-building
  // (and, without appends, the append) code the kernel is far smaller
  // every decode runs from a plan: hw_attn_plan's, or the plan cache's (only
  // for the plain bf16 call, hw_attn_decode)
  if (a.cache_base ? (a.plan || a.k_new || a.k_scale || a.view_limit) : !a.plan)
    return cudaErrorInvalidValue;
  const int which = a.cache_base ? 0
                    : a.k_new ? (a.k_scale ? 6 : 2)
                    : a.k_scale ? (a.view_limit ? 5 : 4)
                    : a.view_limit ? 3 : 1;
  void (*const kernels[7])(DecodeArgs, CUtensorMap, CUtensorMap) = {
      decode_tc_kernel<false, false, false, true>, decode_tc_kernel<false, false, false, false>,
      decode_tc_kernel<true, false, false, false>, decode_tc_kernel<false, true, false, false>,
      decode_tc_kernel<false, false, true, false>, decode_tc_kernel<false, true, true, false>,
      decode_tc_kernel<true, false, true, false>};
  void (*kernel)(DecodeArgs, CUtensorMap, CUtensorMap) = kernels[which];
  static bool configured[7] = {false, false, false, false, false, false, false};
  if (!configured[which]) {
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured[which] = true;
  }
  // A programmatic dependent of the previous kernel on the stream (see the
  // kernel's entry).  Not a cooperative launch: the merge CTAs wait (with a
  // bound) only for CTAs of this grid, which hold their SMs from their start
  // and wait for no one, so every CTA this grid waits for is placed - an SM
  // frees as soon as a CTA of the previous grid, which never waits for this
  // one, retires.  The CTAs that merge nothing retire early, and the next
  // launch's CTAs take those SMs at once.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a, tk, tv);
}

}  // namespace hw
