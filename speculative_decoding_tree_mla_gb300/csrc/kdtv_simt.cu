// CUDA-core (SIMT) path of kdtv_verify_attn: fp32 arithmetic throughout.
//
// This is the precision path for float32 inputs (the tensor cores have no
// fp32-exact kind) and a second, independent implementation for bf16 inputs
// (KDTV_FLAG_SIMT).  Four kernels, one per step of the path:
//   absorb_kernel   q_lat = W_UK[h]^T q_nope                  (fp32 out)
//   attn_kernel     tree-masked scores, online softmax, P.c_kv per split
//   combine_kernel  log-sum-exp merge of the split partials
//   uproj_kernel    out = W_UV[h] o_lat
// The operation is the tree-verify MLA-absorb attention of "The Moment of
// Proof: Validating a Native CUDA Speculative Decoding Engine", sections
// "The Context: Building a Native DDTree Engine from Scratch" and "Input
// Knowledge Required".

#include "kdtv_internal.cuh"

#include <math.h>

namespace kdtv {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerBlock = 16;   // absorb / up-projection rows per CTA
constexpr int kKeyTile = 32;        // keys per attention tile (one per lane)
constexpr int kMaxHeadsPerCta = 16;
constexpr int kMaxOutPerThread = kMaxHeadsPerCta * kMaxLatent / kThreads;  // 32

template <typename TO> __device__ __forceinline__ TO store_as(float x);
template <> __device__ __forceinline__ float store_as<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 store_as<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

template <typename T, typename TO>
__global__ void __launch_bounds__(kThreads) absorb_kernel(Args a) {
  extern __shared__ float q_s[];                    // [kRowsPerBlock][d_nope]
  const int h = blockIdx.x;
  const int r0 = blockIdx.y * kRowsPerBlock;        // r = b * N + i
  const int BN = a.B * a.N;
  const T* q = static_cast<const T*>(a.q_nope);
  for (int idx = threadIdx.x; idx < kRowsPerBlock * a.d_nope; idx += blockDim.x) {
    int r = idx / a.d_nope, e = idx - r * a.d_nope;
    q_s[idx] = (r0 + r < BN)
                   ? to_f32(q[((long long)(r0 + r) * a.H + h) * a.d_nope + e])
                   : 0.f;
  }
  __syncthreads();
  const T* Wk = static_cast<const T*>(a.W_UK) + (long long)h * a.d_nope * a.d_c;
  TO* ql = static_cast<TO*>(a.q_lat);
  for (int d = threadIdx.x; d < a.d_c; d += blockDim.x) {
    float acc[kRowsPerBlock];
#pragma unroll
    for (int r = 0; r < kRowsPerBlock; ++r) acc[r] = 0.f;
    for (int e = 0; e < a.d_nope; ++e) {
      float w = to_f32(Wk[(long long)e * a.d_c + d]);
#pragma unroll
      for (int r = 0; r < kRowsPerBlock; ++r) acc[r] = fmaf(q_s[r * a.d_nope + e], w, acc[r]);
    }
#pragma unroll
    for (int r = 0; r < kRowsPerBlock; ++r)
      if (r0 + r < BN) ql[((long long)(r0 + r) * a.H + h) * a.d_c + d] = store_as<TO>(acc[r]);
  }
}

// One CTA: request b, node i, heads g0 .. g0+ng-1, keys of split s.
// T: element type of q_rope; TC: element type of the cache (times kv_scale).
template <typename T, typename TC>
__global__ void __launch_bounds__(kThreads) attn_kernel(Args a, int G) {
  extern __shared__ float smem[];
  const int D = a.d_c + a.d_rope;
  const int Dp = D + 1;                             // padded row: no bank conflicts
  float* q_s = smem;                                // [G][D]
  float* k_s = q_s + G * D;                         // [kKeyTile][Dp]
  float* p_s = k_s + kKeyTile * Dp;                 // [G][kKeyTile]
  float* m_s = p_s + G * kKeyTile;                  // [G]
  float* l_s = m_s + G;                             // [G]
  float* al_s = l_s + G;                            // [G]
  __shared__ uint32_t anc[4];
  __shared__ int ok_s, L_s;
  __shared__ int vis_s[kKeyTile];

  const int HG = (a.H + G - 1) / G;
  const int i = blockIdx.x / HG;
  const int g0 = (blockIdx.x - i * HG) * G;
  const int ng = min(G, a.H - g0);
  const int s = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    int L = 0;
    uint32_t m[4];
    ok_s = prefix_ok(a, b, &L) && ancestor_mask(a, b, i, m);
    L_s = L;
    anc[0] = m[0]; anc[1] = m[1]; anc[2] = m[2]; anc[3] = m[3];
  }
  __syncthreads();
  if (!ok_s) return;
  const int L = L_s, Tb = L + a.N;
  const int k0 = s * a.chunk, k1 = min(Tb, k0 + a.chunk);
  const long long row0 = ((long long)b * a.N + i) * a.H + g0;
  const long long rows = (long long)a.B * a.N * a.H;
  float* ml = a.part_ml + ((long long)s * rows + row0) * 2;

  if (k0 >= k1) {                                   // nothing of this request here
    for (int g = tid; g < ng; g += blockDim.x) { ml[2 * g] = -INFINITY; ml[2 * g + 1] = 0.f; }
    return;
  }

  const float* ql = static_cast<const float*>(a.q_lat);
  const T* qr = static_cast<const T*>(a.q_rope);
  for (int idx = tid; idx < ng * D; idx += blockDim.x) {
    int g = idx / D, d = idx - g * D;
    long long row = row0 + g;
    q_s[idx] = d < a.d_c ? ql[row * a.d_c + d] : to_f32(qr[row * a.d_rope + (d - a.d_c)]);
  }
  for (int g = tid; g < G; g += blockDim.x) { m_s[g] = -INFINITY; l_s[g] = 0.f; }

  const int n_out = G * a.d_c;                      // owned (g, d) accumulators
  float o[kMaxOutPerThread];
#pragma unroll
  for (int j = 0; j < kMaxOutPerThread; ++j) o[j] = 0.f;

  const TC* ckv = static_cast<const TC*>(a.c_kv);
  const TC* kr = static_cast<const TC*>(a.k_rope);
  __syncthreads();

  for (int t0 = k0; t0 < k1; t0 += kKeyTile) {
    if (tid < kKeyTile) {
      int t = t0 + tid, v = 0;
      if (t < k1) {
        if (t < L) v = 1;
        else { int j = t - L; v = (anc[j >> 5] >> (j & 31)) & 1; }
        if (v && cache_row(a, b, t) < 0) { record_error(a.status, KDTV_ERR_BAD_PAGE, b); v = 0; }
      }
      vis_s[tid] = v;
    }
    __syncthreads();
    for (int idx = tid; idx < kKeyTile * D; idx += blockDim.x) {
      int kk = idx / D, d = idx - kk * D;
      float x = 0.f;
      if (vis_s[kk]) {
        long long r = cache_row(a, b, t0 + kk);
        x = (d < a.d_c ? to_f32(ckv[r * a.d_c + d]) : to_f32(kr[r * a.d_rope + (d - a.d_c)])) *
            a.kv_scale;
      }
      k_s[kk * Dp + d] = x;
    }
    __syncthreads();
    for (int idx = tid; idx < G * kKeyTile; idx += blockDim.x) {
      int g = idx / kKeyTile, kk = idx - g * kKeyTile;
      float sc = -INFINITY;
      if (g < ng && vis_s[kk]) {
        const float* qg = q_s + g * D;
        const float* kt = k_s + kk * Dp;
        float acc = 0.f;
        for (int d = 0; d < D; ++d) acc = fmaf(qg[d], kt[d], acc);
        sc = acc * a.scale;
      }
      p_s[idx] = sc;
    }
    __syncthreads();
    for (int g = warp; g < ng; g += blockDim.x / 32) {   // online softmax, one warp per head
      float sc = p_s[g * kKeyTile + lane];
      float mt = sc;
#pragma unroll
      for (int off = 16; off; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      float m_old = m_s[g];
      float m_new = fmaxf(m_old, mt);
      float p = (sc == -INFINITY) ? 0.f : expf(sc - m_new);
      float ps = p;
#pragma unroll
      for (int off = 16; off; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      float alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
      p_s[g * kKeyTile + lane] = p;
      __syncwarp();
      if (lane == 0) {
        l_s[g] = l_s[g] * alpha + ps;
        m_s[g] = m_new;
        al_s[g] = alpha;
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kMaxOutPerThread; ++j) {
      int idx = tid + j * kThreads;
      if (idx < n_out) {
        int g = idx / a.d_c, d = idx - g * a.d_c;
        if (g < ng) {
          float acc = o[j] * al_s[g];
          const float* pg = p_s + g * kKeyTile;
#pragma unroll 8
          for (int kk = 0; kk < kKeyTile; ++kk) acc = fmaf(pg[kk], k_s[kk * Dp + d], acc);
          o[j] = acc;
        }
      }
    }
    __syncthreads();
  }

  float* po = a.part_o + ((long long)s * rows + row0) * a.d_c;
#pragma unroll
  for (int j = 0; j < kMaxOutPerThread; ++j) {
    int idx = tid + j * kThreads;
    if (idx < n_out) {
      int g = idx / a.d_c;
      if (g < ng) po[idx] = o[j];
    }
  }
  for (int g = tid; g < ng; g += blockDim.x) { ml[2 * g] = m_s[g]; ml[2 * g + 1] = l_s[g]; }
}

// o_lat[row] = o_scale * sum_s e^{m_s - m*} o_s / sum_s e^{m_s - m*} l_s over
// the row's partials (split-KV ranges, or the pieces of a stream-K plan).
__global__ void __launch_bounds__(128) combine_kernel(Args a) {
  const long long row = blockIdx.x;
  __shared__ float w_s[1024];
  __shared__ float inv_l;
  const PartialRef pr = partials_of_row(a, row);
  const int S = pr.count < 1024 ? pr.count : 1024;
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    for (int s = 0; s < S; ++s) {
      const float* ml = a.part_ml + (pr.base + s * pr.step) * 2;
      if (ml[1] > 0.f) m = fmaxf(m, ml[0]);
    }
    float l = 0.f;
    for (int s = 0; s < S; ++s) {
      const float* ml = a.part_ml + (pr.base + s * pr.step) * 2;
      float w = (ml[1] > 0.f) ? expf(ml[0] - m) : 0.f;
      w_s[s] = w;
      l += w * ml[1];
    }
    inv_l = l > 0.f ? a.o_scale / l : 0.f;
  }
  __syncthreads();
  for (int d = threadIdx.x; d < a.d_c; d += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < S; ++s)
      if (w_s[s] != 0.f) {
        const long long i = (pr.base + s * pr.step) * a.d_c + d;
        acc = fmaf(w_s[s], a.sk ? __bfloat162float(a.part_o16[i]) : a.part_o[i], acc);
      }
    a.o_lat[row * a.d_c + d] = acc * inv_l;
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) uproj_kernel(Args a) {
  extern __shared__ float o_s[];                    // [kRowsPerBlock][d_c]
  const int h = blockIdx.x;
  const int r0 = blockIdx.y * kRowsPerBlock;
  const int BN = a.B * a.N;
  for (int idx = threadIdx.x; idx < kRowsPerBlock * a.d_c; idx += blockDim.x) {
    int r = idx / a.d_c, d = idx - r * a.d_c;
    o_s[idx] = (r0 + r < BN) ? a.o_lat[((long long)(r0 + r) * a.H + h) * a.d_c + d] : 0.f;
  }
  __syncthreads();
  const T* Wv = static_cast<const T*>(a.W_UV) + (long long)h * a.d_v * a.d_c;
  for (int v = threadIdx.x; v < a.d_v; v += blockDim.x) {
    float acc[kRowsPerBlock];
#pragma unroll
    for (int r = 0; r < kRowsPerBlock; ++r) acc[r] = 0.f;
    const T* wrow = Wv + (long long)v * a.d_c;
    for (int d = 0; d < a.d_c; ++d) {
      float w = to_f32(wrow[d]);
#pragma unroll
      for (int r = 0; r < kRowsPerBlock; ++r) acc[r] = fmaf(o_s[r * a.d_c + d], w, acc[r]);
    }
#pragma unroll
    for (int r = 0; r < kRowsPerBlock; ++r)
      if (r0 + r < BN) a.out[((long long)(r0 + r) * a.H + h) * a.d_v + v] = acc[r];
  }
}

template <typename T, typename TO>
void launch_absorb_typed(const Args& a, cudaStream_t st) {
  const int BN = a.B * a.N;
  dim3 grid_rows(a.H, (BN + kRowsPerBlock - 1) / kRowsPerBlock);
  size_t sm_abs = sizeof(float) * kRowsPerBlock * a.d_nope;
  absorb_kernel<T, TO><<<grid_rows, kThreads, sm_abs, st>>>(a);
}

template <typename T>
void launch_uproj_typed(const Args& a, cudaStream_t st) {
  const int BN = a.B * a.N;
  dim3 grid_rows(a.H, (BN + kRowsPerBlock - 1) / kRowsPerBlock);
  size_t sm_up = sizeof(float) * kRowsPerBlock * a.d_c;
  uproj_kernel<T><<<grid_rows, kThreads, sm_up, st>>>(a);
}

template <typename T, typename TC>
cudaError_t launch_typed(const Args& a, const Plan& p, cudaStream_t st, cudaEvent_t* ev) {
  launch_absorb_typed<T, float>(a, st);
  if (ev) cudaEventRecord(ev[1], st);

  const int G = p.heads_per_cta;
  const int D = a.d_c + a.d_rope;
  size_t sm_attn = sizeof(float) * ((size_t)G * D + (size_t)kKeyTile * (D + 1) +
                                    (size_t)G * kKeyTile + 3 * G);
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<T, TC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sm_attn);
  if (e != cudaSuccess) return e;
  dim3 grid_attn(a.N * ((a.H + G - 1) / G), a.splits, a.B);
  attn_kernel<T, TC><<<grid_attn, kThreads, sm_attn, st>>>(a, G);
  if (ev) cudaEventRecord(ev[2], st);
  return launch_combine_uproj(a, p, st, ev);
}

}  // namespace

cudaError_t launch_absorb(const Args& a, cudaStream_t st, bool bf16_out) {
  if (a.dtype == KDTV_BF16 || a.dtype == KDTV_BF16_FP8KV) {
    if (bf16_out) launch_absorb_typed<__nv_bfloat16, __nv_bfloat16>(a, st);
    else launch_absorb_typed<__nv_bfloat16, float>(a, st);
  } else {
    launch_absorb_typed<float, float>(a, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine_uproj(const Args& a, const Plan& p, cudaStream_t st,
                                 cudaEvent_t* ev) {
  if (p.splits > 1024) return cudaErrorInvalidValue;
  combine_kernel<<<(unsigned)p.rows, 128, 0, st>>>(a);
  if (ev) cudaEventRecord(ev[3], st);
  if (a.dtype == KDTV_BF16 || a.dtype == KDTV_BF16_FP8KV) launch_uproj_typed<__nv_bfloat16>(a, st);
  else launch_uproj_typed<float>(a, st);
  if (ev) cudaEventRecord(ev[4], st);
  return cudaGetLastError();
}

cudaError_t launch_simt(const Args& a, const Plan& p, cudaStream_t s, cudaEvent_t* ev) {
  if (p.splits > 1024) return cudaErrorInvalidValue;
  if (p.heads_per_cta * a.d_c > kMaxOutPerThread * kThreads) return cudaErrorInvalidValue;
  if (a.dtype == KDTV_BF16_FP8KV) return launch_typed<__nv_bfloat16, __nv_fp8_e4m3>(a, p, s, ev);
  return a.dtype == KDTV_BF16 ? launch_typed<__nv_bfloat16, __nv_bfloat16>(a, p, s, ev)
                              : launch_typed<float, float>(a, p, s, ev);
}

}  // namespace kdtv
