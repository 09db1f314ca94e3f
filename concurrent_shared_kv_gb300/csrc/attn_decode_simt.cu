// attn_decode_simt.cu - concurrent decode attention on the CUDA cores (fp32
// FMA, fp32 accumulation).  It serves fp32 caches, where the tolerance rules
// out tensor-core rounding, and bf16 caches with head_dim 64.
//
// Per CTA: the plan of hw_device.cuh, then for every segment (block b, kv
// head h) in its unit range:
//   1. the view entries that reference b and the q heads of h give up to 32
//      query heads; each is rotated once by i_q - offset of that entry
//      (Hogwild! notes, key design 1: rho(q, i_q - i_k^block));
//   2. K and V tiles of 64 tokens are read from HBM once for all of them;
//   3. scores and an online softmax in the log2 domain; P.V accumulates in
//      registers;
//   4. a partial record (m, l, o) per query head goes to the workspace; after
//      its units every CTA takes part in the merge phase (omica.com.cn
//      article, section 3.2: split over SMs, partial results merged).
#include "hw_device.cuh"

namespace hw {

constexpr int kSimtThreads = 256;

template <int D>
struct SimtSmem {
  PlanCore plan;
  MetaCache cache;
  PlanScratch scratch;
  int64_t u_range[2];
  SegMeta meta;
  MergeSmem<1> merge;
  alignas(16) float q[kMaxQ][D + 4];
  alignas(16) float k[kSimtTile][D + 4];
  alignas(16) float v[kSimtTile][D + 4];
  alignas(16) float p[kMaxQ][kSimtTile + 4];
  float m_run[kMaxQ], l_run[kMaxQ], alpha[kMaxQ];
};

template <typename T>
struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
};

template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &u, float *out);
template <>
__device__ __forceinline__ void unpack16<float>(const uint4 &u, float *out) {
  out[0] = __uint_as_float(u.x);
  out[1] = __uint_as_float(u.y);
  out[2] = __uint_as_float(u.z);
  out[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4 &u, float *out) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[2 * i] = __uint_as_float(w[i] << 16);
    out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// K and V rows [row0, row0 + valid) of kv head h into smem as fp32; rows past
// `valid` are zero so that they add nothing to P.V.
template <typename T, int D>
__device__ __forceinline__ void load_tile(const DecodeArgs &a, SimtSmem<D> &S, int h,
                                          int64_t row0, int valid) {
  constexpr int EPV = Vec16<T>::N;
  constexpr int CPR = D / EPV;  // 16-byte chunks per row
  const T *kb = reinterpret_cast<const T *>(a.k) + (static_cast<int64_t>(h) * a.capacity + row0) * D;
  const T *vb = reinterpret_cast<const T *>(a.v) + (static_cast<int64_t>(h) * a.capacity + row0) * D;
  for (int idx = threadIdx.x; idx < kSimtTile * CPR; idx += kSimtThreads) {
    const int row = idx / CPR, col = (idx % CPR) * EPV;
    float kf[EPV], vf[EPV];
    if (row < valid) {
      const uint4 ku = __ldcs(reinterpret_cast<const uint4 *>(kb + static_cast<int64_t>(row) * D + col));
      const uint4 vu = __ldcs(reinterpret_cast<const uint4 *>(vb + static_cast<int64_t>(row) * D + col));
      unpack16<T>(ku, kf);
      unpack16<T>(vu, vf);
    } else {
#pragma unroll
      for (int i = 0; i < EPV; ++i) kf[i] = vf[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < EPV; i += 4) {
      *reinterpret_cast<float4 *>(&S.k[row][col + i]) = make_float4(kf[i], kf[i + 1], kf[i + 2], kf[i + 3]);
      *reinterpret_cast<float4 *>(&S.v[row][col + i]) = make_float4(vf[i], vf[i + 1], vf[i + 2], vf[i + 3]);
    }
  }
}

template <typename T, int D>
__device__ void simt_segment(const DecodeArgs &a, SimtSmem<D> &S, int b, int g, int h, int t0, int t1) {
  PlanCore &P = S.plan;
  SegMeta &M = S.meta;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.n_q_heads / a.n_kv_heads;
  if (warp == 0) {
    gather_refs(a, S.cache, M, b, g, lane);
    gather_qheads(a, S.cache, M, h, lane);
  }
  __syncthreads();
  const int nq = M.n_ref * G;  // <= kMaxQ: a column group holds at most that many

  // 1. rotated queries: q~ = rho(q, i_q - offset), fp32
  for (int idx = tid; idx < nq * (D / 2); idx += kSimtThreads) {
    const int qi = idx / (D / 2), i = idx % (D / 2);
    const int e = M.ref_entry[qi / G];
    const int r = e / a.n_view;
    const int hq = M.qhead[qi % G];
    const int64_t rel = entry_rel(a, S.cache, e);
    const T *qp = reinterpret_cast<const T *>(a.q) + (static_cast<int64_t>(r) * a.n_q_heads + hq) * D;
    const float x0 = to_f32<T>(qp[i]), x1 = to_f32<T>(qp[i + D / 2]);
    float cs, sn;
    rope_cos_sin(rel, a.phase[i], &cs, &sn);
    S.q[qi][i] = x0 * cs - x1 * sn;
    S.q[qi][i + D / 2] = x1 * cs + x0 * sn;
  }
  for (int qi = tid; qi < kMaxQ; qi += kSimtThreads) {
    S.m_run[qi] = -INFINITY;
    S.l_run[qi] = 0.f;
  }
  constexpr int QSTEP = kSimtThreads / D;  // q heads sharing one d column
  constexpr int QPT = kMaxQ / QSTEP;       // q heads per thread in P.V
  const int dcol = tid % D, qbase = tid / D;
  float acc[QPT];
#pragma unroll
  for (int k = 0; k < QPT; ++k) acc[k] = 0.f;
  __syncthreads();

  const int len = P.len[b];
  const int64_t row_base = P.start[b];
  for (int t = t0; t < t1; ++t) {
    const int tok0 = t * kSimtTile;
    const int valid = min(kSimtTile, len - tok0);
    load_tile<T, D>(a, S, h, row_base + tok0, valid);
    __syncthreads();

    // 2-3. scores, tile max, probabilities (warp w owns q heads w, w+8, ...)
    for (int qq = warp; qq < nq; qq += kSimtThreads / 32) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
      for (int d4 = 0; d4 < D; d4 += 4) {
        const float4 qv = *reinterpret_cast<const float4 *>(&S.q[qq][d4]);
        const float4 k0 = *reinterpret_cast<const float4 *>(&S.k[lane][d4]);
        const float4 k1 = *reinterpret_cast<const float4 *>(&S.k[lane + 32][d4]);
        s0 += qv.x * k0.x + qv.y * k0.y + qv.z * k0.z + qv.w * k0.w;
        s1 += qv.x * k1.x + qv.y * k1.y + qv.z * k1.z + qv.w * k1.w;
      }
      s0 = (lane < valid) ? s0 * a.scale_log2 : -INFINITY;
      s1 = (lane + 32 < valid) ? s1 * a.scale_log2 : -INFINITY;
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_old = S.m_run[qq];
      const float m_new = fmaxf(m_old, mx);
      const float p0 = ex2(s0 - m_new), p1 = ex2(s1 - m_new);
      float sum = p0 + p1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      S.p[qq][lane] = p0;
      S.p[qq][lane + 32] = p1;
      if (lane == 0) {
        const float alpha = ex2(m_old - m_new);  // 0 on the first tile
        S.alpha[qq] = alpha;
        S.m_run[qq] = m_new;
        S.l_run[qq] = S.l_run[qq] * alpha + sum;
      }
    }
    __syncthreads();

    // P.V: thread owns column dcol for q heads qbase, qbase + QSTEP, ...
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      const int qi = qbase + k * QSTEP;
      if (qi < nq) acc[k] *= S.alpha[qi];
    }
    for (int tt = 0; tt < valid; tt += 4) {
      const float v0 = S.v[tt][dcol], v1 = S.v[tt + 1][dcol];
      const float v2 = S.v[tt + 2][dcol], v3 = S.v[tt + 3][dcol];
#pragma unroll
      for (int k = 0; k < QPT; ++k) {
        const int qi = qbase + k * QSTEP;
        if (qi < nq) {
          const float4 pp = *reinterpret_cast<const float4 *>(&S.p[qi][tt]);
          acc[k] += pp.x * v0 + pp.y * v1 + pp.z * v2 + pp.w * v3;
        }
      }
    }
    __syncthreads();
  }

  // 4. partial records into slot seg + c, then arrival and merges
  const int64_t slot = seg_id(P, b, g, h) + blockIdx.x;
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int qi = qbase + k * QSTEP;
    if (qi < nq) {
      float *rec = record_ptr(a, slot, qi);
      rec[dcol] = acc[k];
      if (dcol == 0) {
        rec[D] = S.m_run[qi];
        rec[D + 1] = S.l_run[qi];
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (tid < 32) arrive_segment(a, M, tid);
  __syncthreads();  // the segment metadata is rewritten by the next segment
}

template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads) decode_simt_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem<D> &S = *reinterpret_cast<SimtSmem<D> *>(smem_raw);
  PlanCore &P = S.plan;
  build_plan<kSimtTile>(a, P, S.cache, S.scratch, S.u_range, static_cast<int>(gridDim.x));
  plan_ranks(a, S.cache, threadIdx.x >> 5, threadIdx.x & 31, 0, 1);  // read by the merge
  int64_t u = S.u_range[0];
  const int64_t u_end = S.u_range[1];
  while (u < u_end) {
    const UnitPos x = unit_pos(P, a.n_blocks, u);
    const int64_t seg_stop = min(x.seg_first + x.tiles, u_end);
    simt_segment<T, D>(a, S, x.b, x.g, x.h, static_cast<int>(u - x.seg_first),
                       static_cast<int>(seg_stop - x.seg_first));
    u = seg_stop;
  }
  __syncthreads();
  merge_phase<T, D, 1>(a, P, S.cache, S.merge, nullptr, nullptr, 0, 0, threadIdx.x, kSimtThreads,
                    CtaSync(), a.wait_limit,
                       merge_rank(P, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x)),
                       static_cast<int>(gridDim.x));
}

template <typename T, int D>
static cudaError_t launch_simt(const DecodeArgs &a, int ctas, cudaStream_t s) {
  const size_t smem = sizeof(SimtSmem<D>);
  static bool configured = false;  // per instantiation; attribute is per function
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel<T, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  // cooperative: the merge phase waits on other CTAs, so all must be resident
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kSimtThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_simt_kernel<T, D>, a);
}

template <typename T, int D>
static int simt_occupancy() {
  const size_t smem = sizeof(SimtSmem<D>);
  if (cudaFuncSetAttribute(decode_simt_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<T, D>, kSimtThreads,
                                                    smem) != cudaSuccess || n < 1)
    return 1;
  return n;
}

int decode_simt_ctas_per_sm(int dtype, int head_dim) {
  if (dtype == HW_F32) return head_dim == 64 ? simt_occupancy<float, 64>() : simt_occupancy<float, 128>();
  return head_dim == 64 ? simt_occupancy<__nv_bfloat16, 64>() : simt_occupancy<__nv_bfloat16, 128>();
}

cudaError_t launch_decode_simt(const DecodeArgs &a, int dtype, int ctas, cudaStream_t s) {
  if (dtype == HW_F32) {
    return a.head_dim == 64 ? launch_simt<float, 64>(a, ctas, s) : launch_simt<float, 128>(a, ctas, s);
  }
  return a.head_dim == 64 ? launch_simt<__nv_bfloat16, 64>(a, ctas, s)
                          : launch_simt<__nv_bfloat16, 128>(a, ctas, s);
}

}  // namespace hw
