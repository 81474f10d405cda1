// Internal declarations shared by the CUDA translation units of libkdtv.
// Nothing here is part of the public ABI (include/kdtv.h is).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "kdtv.h"

namespace kdtv {

constexpr int kMaxNodes = 128;        // ancestor masks are 4 x u32
constexpr int kMaxLatent = 512;       // d_c bound on the fp32 path
constexpr int kMaxRope = 64;
constexpr int kStatusBytes = 256;

// Status word layout at the start of the workspace.
struct DeviceStatus {
  unsigned int code;      // first kdtv_status recorded by any kernel (0 = OK)
  unsigned int detail;    // kernel-specific detail of that first error
  unsigned int abort;     // set with the code: lets other CTAs stop early
  unsigned int pad[61];
};

__device__ __forceinline__ void record_error(DeviceStatus* st, unsigned int code,
                                             unsigned int detail) {
  if (atomicCAS(&st->code, 0u, code) == 0u) {
    st->detail = detail;
  }
  atomicExch(&st->abort, 1u);
}

// Per-call plan: how the key range of each request is cut into split-KV
// chunks and where each workspace region lives.  Computed identically by
// kdtv_workspace_size and kdtv_verify_attn.
struct Plan {
  bool tensor_core;       // bf16 tcgen05 path
  int rows;               // B * N * H query rows, row = (b * N + i) * H + h
  int t_cap;              // max keys per request the cache layout can hold
  int chunk;              // keys per split
  int splits;             // splits per request (ceil(t_cap / chunk))
  int heads_per_cta;      // SIMT attention: heads sharing one CTA
  int sms;                // streaming multiprocessors of the current device
  // tensor-core path (stream-K): CTA pairs, W bounds, partial slots
  int sk_clusters, sk_wmin, sk_wforce, rt_count, slots;
  int sk_gap;             // virtual units before each non-empty row tile but the first (0 or kSkBoundary)
  bool kv_widen;          // fp8 cache widened to bf16 copies at off_kvc / off_kvr
  size_t off_qlat, off_part_o, off_part_ml, off_olat, off_sk, off_anc, off_kvc, off_kvr, total;
};

// Device-side view of the call (passed by value to kernels).
struct Args {
  int B, N, H, d_nope, d_rope, d_v, d_c;
  int dtype;              // kdtv_dtype
  float kv_scale;         // cache dequantisation scale (1 unless KDTV_BF16_FP8KV)
  float o_scale;          // factor on each o_lat row in the combine (kv_scale when the
                          // tensor-core path reads a widened, unscaled fp8 cache; else 1)
  int page_size, t_stride, max_pages, num_pages;
  float scale;
  unsigned int flags;
  int chunk, splits;
  const void* q_nope;
  const void* q_rope;
  const void* W_UK;
  const void* W_UV;
  const void* c_kv;
  const void* k_rope;
  const void* c_kv8;      // fp8 cache widened into c_kv / k_rope before the attention
  const void* k_rope8;    // (tensor-core path, KDTV_BF16_FP8KV), else nullptr
  const int32_t* parent;
  const int32_t* prefix_len;
  const int32_t* page_table;
  float* out;
  DeviceStatus* status;
  void* q_lat;            // fp32 (SIMT) or bf16 (tensor core) [rows, d_c]
  float* part_o;          // [splits, rows, d_c] fp32 (split layout)
  __nv_bfloat16* part_o16;  // [slots, 128, d_c] bf16 with a stream-K plan (unnormalised o_lat)
  float* part_ml;         // [splits, rows, 2] or [slots, 128, 2]  (running max m, sum l)
  float* o_lat;           // [rows, d_c]
  // Stream-K plan of the tensor-core attention (nullptr: split layout).
  int* sk;                // kSkHeader ints {V, W, clusters, R}, then {vS_r, u_r, base_r} per row
                          // tile (vS_r: the tile's start in the virtual sequence, see
                          // sk_gap), then the row tile of each CTA pair's first piece, then
                          // (16-byte aligned) 8 ints per pair: {r, vS_r, u_r, base_r} of that
                          // tile, L_b, the pair's count of key tiles
  uint32_t* anc_g;        // [B, N, 4] ancestor masks, written by the plan kernel
  int rt_count;           // 128-row tiles per request
  int sk_clusters;        // CTA pairs launched
  int sk_wmin;            // lower bound on W (units per CTA pair)
  int sk_wforce;          // forced W from kv_chunk (0 = none)
  int sk_gap;             // virtual units before each non-empty row tile but the first
};

constexpr int kSkHeader = 4;
// Cost of a piece boundary in the stream-K schedule, in 64-key units (writing
// one piece's partial and loading the next piece's Q cost about six tiles of
// work).  With a gap of this many virtual units before every non-empty row
// tile but the first, a CTA pair whose range crosses into another row tile
// takes that many key tiles fewer.
constexpr int kSkBoundary = 6;

// Where the partials of query row `row` live: `count` partial rows at part
// row index base + k * step (k = 0 .. count-1).  With a stream-K plan the
// row's 128-row tile r was cut into pieces at the multiples of W inside its
// virtual range (vS_r, vS_r + u_r); its pieces hold consecutive slots
// base_r .. base_r + count - 1.
struct PartialRef {
  long long base, step;
  int count;
};
__device__ __forceinline__ PartialRef partials_of_row(const Args& a, long long row) {
  PartialRef p;
  if (!a.sk) {
    p.base = row;
    p.step = (long long)a.B * a.N * a.H;
    p.count = a.splits;
    return p;
  }
  const int nh = a.N * a.H;
  const int b = (int)(row / nh), rr = (int)(row % nh);
  const int r = (rr / 128) * a.B + b, tr = rr % 128;   // lane-major row tiles
  const int W = a.sk[1];
  const int* e = a.sk + kSkHeader + 3 * r;
  const int S = e[0], u = e[1], base = e[2];   // S = vS_r
  p.count = u > 0 ? 1 + ((S + u + W - 1) / W - 1 - S / W) : 0;
  p.base = (long long)base * 128 + tr;
  p.step = 128;
  return p;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__nv_fp8_e4m3 x) { return static_cast<float>(x); }

// Row of logical position t of request b in a cache tensor with `width`
// elements per row; -1 if the page id is out of range.
__device__ __forceinline__ long long cache_row(const Args& a, int b, int t) {
  if (a.page_size == 0) return (long long)b * a.t_stride + t;
  int page = a.page_table[(long long)b * a.max_pages + t / a.page_size];
  if (page < 0 || page >= a.num_pages) return -1;
  return (long long)page * a.page_size + (t % a.page_size);
}

// Walks node i's root path, building its ancestor mask (bit a set for every a
// on the path, i included).  Returns false, after recording BAD_TREE, if
// parent[] is not a topologically ordered tree rooted at node 0.
__device__ __forceinline__ bool ancestor_mask(const Args& a, int b, int i,
                                              uint32_t mask[4]) {
  const int32_t* par = a.parent + (long long)b * a.N;
  mask[0] = mask[1] = mask[2] = mask[3] = 0u;
  if (par[0] != -1) {
    record_error(a.status, KDTV_ERR_BAD_TREE, (unsigned)b);
    return false;
  }
  int j = i;
  for (int step = 0; step <= a.N; ++step) {   // parent[j] < j bounds the walk
    mask[j >> 5] |= 1u << (j & 31);
    if (j == 0) return true;
    int p = par[j];
    if (p < 0 || p >= j) {
      record_error(a.status, KDTV_ERR_BAD_TREE, (unsigned)(b * 65536 + j));
      return false;
    }
    j = p;
  }
  return false;
}

// Same walk over a copy of parent[b][0 .. N) already in shared memory.
__device__ __forceinline__ bool ancestor_mask_smem(const Args& a, int b, const int32_t* par, int i,
                                                   uint32_t mask[4]) {
  mask[0] = mask[1] = mask[2] = mask[3] = 0u;
  if (par[0] != -1) {
    record_error(a.status, KDTV_ERR_BAD_TREE, (unsigned)b);
    return false;
  }
  int j = i;
  for (int step = 0; step <= a.N; ++step) {
    mask[j >> 5] |= 1u << (j & 31);
    if (j == 0) return true;
    int p = par[j];
    if (p < 0 || p >= j) {
      record_error(a.status, KDTV_ERR_BAD_TREE, (unsigned)(b * 65536 + j));
      return false;
    }
    j = p;
  }
  return false;
}

__device__ __forceinline__ bool prefix_ok(const Args& a, int b, int* L) {
  int l = a.prefix_len[b];
  int cap = a.page_size ? a.max_pages * a.page_size : a.t_stride;
  if (l < 0 || (long long)l + a.N > cap) {
    record_error(a.status, KDTV_ERR_BAD_PREFIX, (unsigned)b);
    return false;
  }
  *L = l;
  return true;
}

// Launch with an optional programmatic-dependent-launch attribute: the kernel
// may begin while the previous kernel of the stream drains, and must call
// griddepcontrol.wait before touching that kernel's outputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Launchers (one per translation unit).
cudaError_t launch_simt(const Args& a, const Plan& p, cudaStream_t s,
                        cudaEvent_t* ev);
cudaError_t launch_tc(const Args& a, const Plan& p, cudaStream_t s,
                      cudaEvent_t* ev);
cudaError_t launch_absorb(const Args& a, cudaStream_t s, bool bf16_out);
cudaError_t launch_combine_uproj(const Args& a, const Plan& p, cudaStream_t s,
                                 cudaEvent_t* ev);
// after_plan: may start beside the attention plan kernel (programmatic launch)
cudaError_t launch_absorb_tc(const Args& a, cudaStream_t s, bool after_plan);
cudaError_t launch_combine_uproj_tc(const Args& a, const Plan& p, cudaStream_t s,
                                    cudaEvent_t* ev);
// fp8 cache (a.c_kv8, a.k_rope8) -> bf16 copies in the same layout (a.c_kv,
// a.k_rope) of the rows the call reads
cudaError_t launch_kv_widen(const Args& a, int sms, cudaStream_t s, bool pdl);
bool absorb_tc_ok(const Args& a);
bool combine_uproj_tc_ok(const Args& a);
int tc_supported(const kdtv_dims* d);
// Status kdtv_verify_attn returns on the host for these dims, and the
// workspace bytes they need (0 unless KDTV_OK).
int plan_status(const kdtv_dims* d, size_t* bytes);
// SMs of the current device (0 if it cannot be queried).
int device_sm_count();
int tc_launches(const kdtv_dims* d, int splits);

}  // namespace kdtv
