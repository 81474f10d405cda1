// FP8 E4M3 latent cache on the tensor-core path: the rows of the cache that a
// call reads are widened to bf16 in the workspace, in the layout of the input
// (contiguous [B, t_stride, d] or paged [num_pages, 64, d]), and the bf16
// attention runs on that copy.
//
// The widening is exact: every E4M3 value (3 mantissa bits, exponents 2^-9 ..
// 2^8) is an f16 value and every such f16 value a bf16 value.  The scale is
// not applied here; the caller folds kv_scale into the softmax scale (scores
// are linear in the keys) and into the combine's 1 / l (o_lat is linear in
// the values), so a power-of-two kv_scale gives exactly the bf16 path's
// arithmetic on the dequantised cache.

#include "kdtv_internal.cuh"
#include "kdtv_ptx.cuh"

namespace kdtv {
namespace {

constexpr int kRows = 64;        // rows per work item: one 64-key tile (one page)
constexpr int kThreads = 256;

// 8 E4M3 bytes -> 8 bf16 (16 bytes), element order kept.
__device__ __forceinline__ uint4 widen8(const uint2& v) {
  const uint32_t src[4] = {v.x & 0xffffu, v.x >> 16, v.y & 0xffffu, v.y >> 16};
  uint32_t out[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)src[k], __NV_E4M3);
    const float2 f = __half22float2(__half2(h));
    const __nv_bfloat162 b = __float22bfloat162_rn(f);
    out[k] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// One 64-row item: row `r` of the item is source row `row0 + r`; rows with
// r >= live are written as zeros (contiguous layout: keys past L_b + N that
// the last 64-key tile still loads, masked out of the softmax).  Each lane
// moves 8-byte groups, so a warp reads 256 and writes 512 contiguous bytes
// per instruction; all of a thread's loads are issued before its stores.
__device__ __forceinline__ void widen_item(const uint8_t* __restrict__ ckv8,
                                           const uint8_t* __restrict__ kr8,
                                           __nv_bfloat16* __restrict__ ckv,
                                           __nv_bfloat16* __restrict__ kr, long long row0,
                                           int nrows, int live) {
  // c_kv: 64 rows x 64 groups = 4096 groups, 16 per thread; k_rope: 64 rows x
  // 8 groups = 512 groups, 2 per thread.
  constexpr int kGc = 512 / 8, kGr = 64 / 8;
  constexpr int kPc = kRows * kGc / kThreads, kPr = kRows * kGr / kThreads;
  uint2 vc[kPc], vr[kPr];
#pragma unroll
  for (int k = 0; k < kPc; ++k) {
    const int g = threadIdx.x + k * kThreads, r = g / kGc;
    vc[k] = (r < nrows && r < live)
                ? __ldg(reinterpret_cast<const uint2*>(ckv8 + (row0 + r) * 512) + (g % kGc))
                : make_uint2(0u, 0u);
  }
#pragma unroll
  for (int k = 0; k < kPr; ++k) {
    const int g = threadIdx.x + k * kThreads, r = g / kGr;
    vr[k] = (r < nrows && r < live)
                ? __ldg(reinterpret_cast<const uint2*>(kr8 + (row0 + r) * 64) + (g % kGr))
                : make_uint2(0u, 0u);
  }
#pragma unroll
  for (int k = 0; k < kPc; ++k) {
    const int g = threadIdx.x + k * kThreads, r = g / kGc;
    if (r < nrows) reinterpret_cast<uint4*>(ckv + (row0 + r) * 512)[g % kGc] = widen8(vc[k]);
  }
#pragma unroll
  for (int k = 0; k < kPr; ++k) {
    const int g = threadIdx.x + k * kThreads, r = g / kGr;
    if (r < nrows) reinterpret_cast<uint4*>(kr + (row0 + r) * 64)[g % kGr] = widen8(vr[k]);
  }
}

// Work item u = b * tiles + k: request b's 64-key tile k (contiguous) or
// page-table slot k (paged).  Items past a request's last tile do nothing.
// Reads the fp8 cache at a.c_kv8 / a.k_rope8 and writes the bf16 copies the
// attention kernel reads at a.c_kv / a.k_rope (workspace).  It runs beside the
// plan and absorb kernels and completes after them, so the attention kernel's
// wait on this grid covers all three.
__global__ void __launch_bounds__(kThreads) kv_widen_kernel(const Args a, long long tiles) {
  ptx::grid_dep_launch();   // the attention kernel may start its prologue early
  const uint8_t* ckv8 = static_cast<const uint8_t*>(a.c_kv8);
  const uint8_t* kr8 = static_cast<const uint8_t*>(a.k_rope8);
  __nv_bfloat16* ckv = static_cast<__nv_bfloat16*>(const_cast<void*>(a.c_kv));
  __nv_bfloat16* kr = static_cast<__nv_bfloat16*>(const_cast<void*>(a.k_rope));
  const long long total = (long long)a.B * tiles;
  const int cap = a.page_size ? a.max_pages * a.page_size : a.t_stride;
  for (long long u = blockIdx.x; u < total; u += gridDim.x) {
    const int b = (int)(u / tiles), k = (int)(u % tiles);
    const int L = a.prefix_len[b];
    const bool ok = L >= 0 && (long long)L + a.N <= cap;   // else the attention reports it
    if (a.page_size == 0) {
      // A bad prefix still gets its first tile zeroed: the last tile of
      // request b - 1 may run into it when t_stride is not a multiple of 64.
      const int T = ok ? L + a.N : 0;
      const int ntiles = T > 0 ? (T + kRows - 1) / kRows : 1;
      if (k >= ntiles) continue;
      const int t0 = k * kRows;
      const int nrows = min(kRows, a.t_stride - t0);
      widen_item(ckv8, kr8, ckv, kr, (long long)b * a.t_stride + t0, nrows, T - t0);
    } else {
      if (!ok || k >= (L + a.N + kRows - 1) / kRows) continue;
      const int page = a.page_table[(long long)b * a.max_pages + k];
      if (page < 0 || page >= a.num_pages) continue;       // the attention reports it
      // Whole pages: a page shared by two requests is written with the same
      // bytes by both.
      widen_item(ckv8, kr8, ckv, kr, (long long)page * kRows, kRows, kRows);
    }
  }
  ptx::grid_dep_wait();     // the plan and absorb kernels launched before this one
}

}  // namespace

cudaError_t launch_kv_widen(const Args& a, int sms, cudaStream_t st, bool pdl) {
  if (a.d_c != 512 || a.d_rope != 64 || (a.page_size != 0 && a.page_size != kRows))
    return cudaErrorInvalidValue;
  for (const void* p : {a.c_kv8, a.k_rope8, a.c_kv, a.k_rope})
    if (!p || (reinterpret_cast<uintptr_t>(p) & 15u)) return cudaErrorMisalignedAddress;
  const long long cap = a.page_size ? (long long)a.max_pages * a.page_size : a.t_stride;
  const long long tiles = (cap + kRows - 1) / kRows;
  const long long total = (long long)a.B * tiles;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kv_widen_kernel, kThreads, 0) !=
          cudaSuccess || per_sm < 1)
    per_sm = 1;
  long long grid = (long long)(sms > 0 ? sms : 152) * per_sm;   // all resident at once
  if (grid > total) grid = total;
  if (grid < 1) grid = 1;
  return launch_ex(kv_widen_kernel, dim3((unsigned)grid), dim3(kThreads), 0, st, pdl, a, tiles);
}

}  // namespace kdtv
