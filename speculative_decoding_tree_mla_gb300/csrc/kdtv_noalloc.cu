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

#include <cuda.h>
#include <mutex>
#include <string.h>

namespace {

// Fixed scratch: status word, q_lat, split-KV partials and o_lat of one call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDTV_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch, per device, tagged with the id of the
// CUDA context it was looked up in.  If that context is destroyed and a new
// one created (cudaDeviceReset, or the primary context released and retained
// again), the module is loaded again and the array may move: a different
// context id triggers a fresh lookup.
constexpr int kMaxDevices = 64;
struct ScratchSlot {
  unsigned long long ctx_id;
  void* ptr;
};
ScratchSlot g_slot[kMaxDevices];
std::mutex g_slot_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// The driver's context queries, resolved through the runtime (the library
// does not link libcuda).
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  if (!get_current || !get_id) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      return false;
    get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      return false;
    get_id = reinterpret_cast<CtxGetIdFn>(p);
  }
  CUcontext ctx = nullptr;
  return get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, id) == CUDA_SUCCESS;
}

// Host-side lookup of the array's device address.  In host code the symbol
// g_noalloc_scratch is only a stand-in, not a device address; the real
// address comes from cudaGetSymbolAddress, with the device current, the first
// time a call runs in a given context on that device.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDTV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KDTV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_slot_mu);
  unsigned long long ctx = 0;
  if (!current_context_id(&ctx)) {
    // No context is current on this host thread yet: the runtime binds the
    // device's primary context during the lookup itself.
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p ||
        !current_context_id(&ctx))
      return KDTV_ERR_CUDA;
    g_slot[dev].ptr = p;
    g_slot[dev].ctx_id = ctx;
  }
  ScratchSlot& s = g_slot[dev];
  if (!s.ptr || s.ctx_id != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KDTV_ERR_CUDA;
    s.ptr = p;
    s.ctx_id = ctx;
  }
  *out = s.ptr;
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
  size_t need = 0;
  int st = kdtv::plan_status(&d, &need);   // the same host-side codes as kdtv_verify_attn
  if (st != KDTV_OK) return st;
  if (need > (size_t)KDTV_NOALLOC_SCRATCH_BYTES) return KDTV_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != KDTV_OK) return st;
  d.workspace = scratch;
  d.workspace_bytes = KDTV_NOALLOC_SCRATCH_BYTES;
  st = kdtv_verify_attn(&d, q_nope, q_rope, W_UK, W_UV, c_kv, k_rope, parent, prefix_len,
                        page_table, out, stream);
  if (st != KDTV_OK) return st;
  copy_status_kernel<<<1, 32, 0, stream>>>(static_cast<const unsigned int*>(scratch), status_out);
  return cudaGetLastError() == cudaSuccess ? KDTV_OK : KDTV_ERR_CUDA;
}
