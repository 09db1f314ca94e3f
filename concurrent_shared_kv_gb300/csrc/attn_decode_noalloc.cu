// attn_decode_noalloc.cu - hw_attn_decode_noalloc: the decode attention call
// for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run attention:
// code inside a custom allocator or memory pool, plugins and runtimes that
// own all device memory and hand out only fixed buffers, or processes that
// must not allocate after start-up.  hw_attn_decode needs a caller-provided
// workspace (merge counters and partial softmax records); this entry point
// instead uses one fixed scratch array that lives in the library itself.
//
// The scratch is a file-scope __device__ array of HW_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  In
// host code the array's name only stands in for the symbol - it is not a
// device address - so the device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, and passed
// to the kernels like any other workspace pointer.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "hogwild.h"
#include "hw_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[HW_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};
// the description of each device's last call (the scratch's layout follows it)
hw_attn_desc g_last_desc[kMaxDevices];
bool g_have_desc[kMaxDevices] = {false};

// Device address of the scratch on the current device; the first call per
// device looks it up and zero-fills the whole array (synchronously).
int scratch_for_current_device(void **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return HW_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return HW_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return HW_ERR_CUDA;
    e = cudaMemset(p, 0, HW_NOALLOC_SCRATCH_BYTES);
    if (e != cudaSuccess) return HW_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return HW_OK;
}

}  // namespace

extern "C" int hw_attn_decode_noalloc(const hw_attn_desc *d, const void *q, const void *k_cache,
                                      const void *v_cache, const int32_t *block_start,
                                      const int32_t *block_len, const int32_t *view_block,
                                      const int32_t *view_offset, const int32_t *q_pos,
                                      const int32_t *q_to_kv, void *out, float *lse,
                                      void *stream) {
  if (!d) return HW_ERR_INVALID;
  // view limits and E4M3 caches come with a plan
  if ((d->flags & HW_DESC_VIEW_LIMITS) || d->dtype == HW_FP8_E4M3) return HW_ERR_UNSUPPORTED;
  size_t need = 0;
  int st = hw_attn_decode_workspace_size(d, &need);
  if (st != HW_OK) return st;
  if (need > HW_NOALLOC_SCRATCH_BYTES) return HW_ERR_WORKSPACE;  // beyond the fixed scratch
  if (d->n_rows == 0) return HW_OK;
  void *scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != HW_OK) return st;
  // The error word and the merge counters must start at zero.  Every call
  // leaves the counters at zero again, but a call that gave up on a wait may
  // not have, so they are cleared on the stream before each call.
  const hw::WorkspaceLayout L = hw::decode_workspace_layout(*d);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(scratch, 0, L.partials_off, s);
  if (e != cudaSuccess) return HW_ERR_CUDA;
  // The decode's plan cache lives in the scratch at offsets that follow the
  // description: after a change of description its state and the header of
  // its first plan buffer are cleared too, so that the next call rebuilds it
  // (a workspace would be zeroed again likewise).
  bool fresh;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HW_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    fresh = !g_have_desc[dev] || std::memcmp(&g_last_desc[dev], d, sizeof *d) != 0;
    g_last_desc[dev] = *d;
    g_have_desc[dev] = true;
  }
  if (fresh) {
    unsigned char *base = static_cast<unsigned char *>(scratch) + L.cache_off;
    e = cudaMemsetAsync(base, 0, hw::kPlanCacheStateBytes, s);
    if (e == cudaSuccess)
      e = cudaMemsetAsync(base + hw::kPlanCacheStateBytes + 2 * L.cache_meta_bytes, 0,
                          hw::kPlanHeaderBytes, s);
    if (e != cudaSuccess) return HW_ERR_CUDA;
  }
  return hw_attn_decode(d, q, k_cache, v_cache, block_start, block_len, view_block, view_offset,
                        q_pos, q_to_kv, out, lse, scratch, HW_NOALLOC_SCRATCH_BYTES, stream);
}

// The scratch's error word (its first 4 bytes, like a workspace's): read into
// host memory and cleared, with plain copies - nothing is allocated.  A device
// whose scratch was never set up has no error.
extern "C" int hw_noalloc_status(int32_t *flags, void *stream) {
  if (!flags) return HW_ERR_INVALID;
  *flags = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return HW_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return HW_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    scratch = g_scratch_ptr[dev];
  }
  if (!scratch) return HW_OK;
  e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaMemcpy(flags, scratch, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(scratch, 0, sizeof(int32_t));
  return e == cudaSuccess ? HW_OK : HW_ERR_CUDA;
}
