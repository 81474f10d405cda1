// kdtv_verify_attn_noalloc: the whole verify-attention path with its scratch in
// a fixed, file-scope device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot call cudaMalloc at the point where they
// run the attention -- for example code executing inside a memory-pool or
// arena allocator that owns all device memory, plugins of an inference server
// that only hand kernels pre-registered buffers, or environments where device
// allocation is forbidden after start-up.  Such callers still own and pass
// every input and output; only the scratch moves into this library.
//
// The scratch array lives in this library's device image, so every GPU that
// loads the library holds KDTV_NOALLOC_SCRATCH_BYTES of device memory until
// the process exits.  All calls share it: calls that overlap on the GPU (two
// streams, or two host threads) race on it and must be serialised by the
// caller.  Each call clears the status word at the start of the scratch; the
// other scratch regions are fully written before they are read.

#include "kdtv_internal.cuh"

#include <string.h>

namespace {

// Fixed scratch: status word, q_lat, split-KV partials and o_lat of one call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDTV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];   // device address of g_noalloc_scratch, per device

// Host-side lookup of the array's device address.  In host code the symbol
// g_noalloc_scratch is only a stand-in, not a device address; the real
// address comes from cudaGetSymbolAddress, once per device, with that device
// current.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDTV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KDTV_ERR_UNSUPPORTED;
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KDTV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KDTV_OK;
}

__global__ void copy_status_kernel(const unsigned int* src, unsigned int* dst) {
  if (threadIdx.x == 0) *dst = *src;
}

}  // namespace

extern "C" int kdtv_verify_attn_noalloc(const kdtv_dims* dims, const void* q_nope,
                                        const void* q_rope, const void* W_UK, const void* W_UV,
                                        const void* c_kv, const void* k_rope,
                                        const int32_t* parent, const int32_t* prefix_len,
                                        const int32_t* page_table, float* out,
                                        unsigned int* status_out, cudaStream_t stream) {
  if (!dims || !status_out) return KDTV_ERR_INVALID_ARG;
  kdtv_dims d;
  memcpy(&d, dims, sizeof(d));
  d.workspace = nullptr;
  d.workspace_bytes = 0;
  const size_t need = kdtv_workspace_size(&d);
  if (need == 0) return KDTV_ERR_INVALID_ARG;
  if (need > (size_t)KDTV_NOALLOC_SCRATCH_BYTES) return KDTV_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  int st = scratch_for_current_device(&scratch);
  if (st != KDTV_OK) return st;
  d.workspace = scratch;
  d.workspace_bytes = KDTV_NOALLOC_SCRATCH_BYTES;
  st = kdtv_verify_attn(&d, q_nope, q_rope, W_UK, W_UV, c_kv, k_rope, parent, prefix_len,
                        page_table, out, stream);
  if (st != KDTV_OK) return st;
  copy_status_kernel<<<1, 32, 0, stream>>>(static_cast<const unsigned int*>(scratch), status_out);
  return cudaGetLastError() == cudaSuccess ? KDTV_OK : KDTV_ERR_CUDA;
}
