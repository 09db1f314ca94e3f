// block_commit.cu - move finished steps into the shared history (Hogwild!
// notes, key design 2: a finished step's KV is rotated and moved into the
// common cache).  For each commit c of the launch:
//
//   K_dst[l][h][dst_offset_c + j] = rho(K_src[l][h][src_begin_c + j], delta_c)
//   V_dst[l][h][dst_offset_c + j] = V_src[l][h][src_begin_c + j]
//
// HBM-bound: every byte is read once and written once.  A thread owns one
// 16-byte chunk of the first half of a key row and the matching chunk of the
// second half (RoPE pairs i and i + D/2), so the rotation needs no exchange;
// V moves as the same two 16-byte chunks.  cos/sin of delta * w_i are made
// once per CTA in shared memory from the integer phase table.  E4M3 pools are
// rotated on their codes' values (a head's scale carries over unchanged) and
// rounded back to the nearest code, saturating at 448.
#include <cuda_fp8.h>

#include "hw_device.cuh"

namespace hw {

constexpr int kCommitThreads = 256;

template <typename T>
__device__ __forceinline__ uint4 rotate16(const uint4 &lo, const uint4 &hi, const float *cs,
                                          const float *sn, bool upper);

template <>
__device__ __forceinline__ uint4 rotate16<float>(const uint4 &lo, const uint4 &hi, const float *cs,
                                                 const float *sn, bool upper) {
  const float xl[4] = {__uint_as_float(lo.x), __uint_as_float(lo.y), __uint_as_float(lo.z),
                       __uint_as_float(lo.w)};
  const float xh[4] = {__uint_as_float(hi.x), __uint_as_float(hi.y), __uint_as_float(hi.z),
                       __uint_as_float(hi.w)};
  float y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    y[i] = upper ? __fmaf_rn(xh[i], cs[i], __fmul_rn(xl[i], sn[i]))
                 : __fmaf_rn(xl[i], cs[i], -__fmul_rn(xh[i], sn[i]));
  return make_uint4(__float_as_uint(y[0]), __float_as_uint(y[1]), __float_as_uint(y[2]),
                    __float_as_uint(y[3]));
}

template <>
__device__ __forceinline__ uint4 rotate16<__nv_bfloat16>(const uint4 &lo, const uint4 &hi,
                                                         const float *cs, const float *sn,
                                                         bool upper) {
  const uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w};
  const uint32_t wh[4] = {hi.x, hi.y, hi.z, hi.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float y[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float xl = __uint_as_float(e ? (wl[i] & 0xffff0000u) : (wl[i] << 16));
      const float xh = __uint_as_float(e ? (wh[i] & 0xffff0000u) : (wh[i] << 16));
      const int j = 2 * i + e;
      y[e] = upper ? __fmaf_rn(xh, cs[j], __fmul_rn(xl, sn[j]))
                   : __fmaf_rn(xl, cs[j], -__fmul_rn(xh, sn[j]));
    }
    const __nv_bfloat162 p = __floats2bfloat162_rn(y[0], y[1]);  // round to nearest even
    out[i] = *reinterpret_cast<const uint32_t *>(&p);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

struct E4M3 {  // storage tag: one E4M3 code
  uint8_t code;
};

template <>
__device__ __forceinline__ uint4 rotate16<E4M3>(const uint4 &lo, const uint4 &hi, const float *cs,
                                                const float *sn, bool upper) {
  const uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w};
  const uint32_t wh[4] = {hi.x, hi.y, hi.z, hi.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t word = 0;
#pragma unroll
    for (int p = 0; p < 2; ++p) {  // two e4m3 pairs of the word
      const __half2 l2(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(wl[i] >> (16 * p)), __NV_E4M3));
      const __half2 h2(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(wh[i] >> (16 * p)), __NV_E4M3));
      const float2 xl = __half22float2(l2), xh = __half22float2(h2);
      const int j = 4 * i + 2 * p;
      float2 y;
      y.x = upper ? __fmaf_rn(xh.x, cs[j], __fmul_rn(xl.x, sn[j]))
                  : __fmaf_rn(xl.x, cs[j], -__fmul_rn(xh.x, sn[j]));
      y.y = upper ? __fmaf_rn(xh.y, cs[j + 1], __fmul_rn(xl.y, sn[j + 1]))
                  : __fmaf_rn(xl.y, cs[j + 1], -__fmul_rn(xh.y, sn[j + 1]));
      const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
      word |= static_cast<uint32_t>(q) << (16 * p);
    }
    out[i] = word;
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Grid row c (blockIdx.y) commits range c; its CTAs stride over the range's
// (layer, head, token, chunk) items.
template <typename T>
__global__ void __launch_bounds__(kCommitThreads) block_commit_kernel(const __grid_constant__ CommitArgs a) {
  constexpr int EPV = 16 / sizeof(T);
  __shared__ float cs[64], sn[64];
  const int c = blockIdx.y;
  const int D = a.head_dim, n_tokens = a.n_tokens[c];
  const int64_t delta = a.delta[c];
  for (int i = threadIdx.x; i < D / 2; i += blockDim.x) rope_cos_sin(delta, a.phase[i], &cs[i], &sn[i]);
  __syncthreads();
  const int half_chunks = (D / 2) / EPV;
  const int64_t rows = static_cast<int64_t>(a.n_layers) * a.n_kv_heads * n_tokens;
  const int64_t total = rows * half_chunks;
  const bool copy_only = (delta == 0);
  const int64_t src_begin = a.src_begin[c], dst_offset = a.dst_offset[c];
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = idx / half_chunks;
    const int ch = static_cast<int>(idx % half_chunks);
    const int64_t j = row % n_tokens, lh = row / n_tokens;  // lh = layer * Hkv + h
    const int64_t so = (lh * a.src_capacity + src_begin + j) * D + ch * EPV;
    const int64_t dof = (lh * a.dst_capacity + dst_offset + j) * D + ch * EPV;
    const T *ks = reinterpret_cast<const T *>(a.k_src);
    const T *vs = reinterpret_cast<const T *>(a.v_src);
    T *kd = reinterpret_cast<T *>(a.k_dst);
    T *vd = reinterpret_cast<T *>(a.v_dst);
    const uint4 klo = __ldcs(reinterpret_cast<const uint4 *>(ks + so));
    const uint4 khi = __ldcs(reinterpret_cast<const uint4 *>(ks + so + D / 2));
    const uint4 vlo = __ldcs(reinterpret_cast<const uint4 *>(vs + so));
    const uint4 vhi = __ldcs(reinterpret_cast<const uint4 *>(vs + so + D / 2));
    uint4 ylo = klo, yhi = khi;
    if (!copy_only) {
      ylo = rotate16<T>(klo, khi, cs + ch * EPV, sn + ch * EPV, false);
      yhi = rotate16<T>(klo, khi, cs + ch * EPV, sn + ch * EPV, true);
    }
    *reinterpret_cast<uint4 *>(kd + dof) = ylo;
    *reinterpret_cast<uint4 *>(kd + dof + D / 2) = yhi;
    *reinterpret_cast<uint4 *>(vd + dof) = vlo;
    *reinterpret_cast<uint4 *>(vd + dof + D / 2) = vhi;
  }
}

cudaError_t launch_commit(const CommitArgs &a, int dtype, cudaStream_t s) {
  const int epv = dtype == HW_F32 ? 4 : dtype == HW_FP8_E4M3 ? 16 : 8;
  int64_t work = 0;
  for (int c = 0; c < a.n_commits; ++c)
    work += static_cast<int64_t>(a.n_layers) * a.n_kv_heads * a.n_tokens[c] * ((a.head_dim / 2) / epv);
  if (work == 0) return cudaSuccess;
  // about eight CTAs per SM in all, shared evenly by the commits
  const int sms = device_sm_count();
  int64_t ctas = (work + kCommitThreads - 1) / kCommitThreads;
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 152) * 8;
  if (ctas > cap) ctas = cap;
  const int64_t per = (ctas + a.n_commits - 1) / a.n_commits;
  const dim3 grid(static_cast<unsigned>(per > 0 ? per : 1), static_cast<unsigned>(a.n_commits));
  if (dtype == HW_F32)
    block_commit_kernel<float><<<grid, kCommitThreads, 0, s>>>(a);
  else if (dtype == HW_FP8_E4M3)
    block_commit_kernel<E4M3><<<grid, kCommitThreads, 0, s>>>(a);
  else
    block_commit_kernel<__nv_bfloat16><<<grid, kCommitThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace hw
