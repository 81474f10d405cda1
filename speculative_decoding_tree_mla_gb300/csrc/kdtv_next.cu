// The DDTree loop steps around the verify attention ("The Moment of Proof:
// Validating a Native CUDA Speculative Decoding Engine", section "The Context:
// Building a Native DDTree Engine from Scratch": a GPU best-first tree
// builder, a greedy tree-accept kernel, KV cache post-verify compaction):
//
//   tree_build_kernel    best-first draft tree from per-depth top-K proposals
//   tree_accept_kernel   longest root path whose draft tokens match the
//                        target's greedy tokens
//   compact_kernel       move the accepted nodes' latent rows next to the prefix
//
// One CTA per request for each: the trees have at most 128 nodes, so the
// work is latency-bound and stays inside one SM.

#include "kdtv_internal.cuh"

#include <math.h>

namespace kdtv {
namespace {

// ---- greedy tree accept ------------------------------------------------------------------
// One warp per request.  From node u, the next node is the lowest-indexed
// child c (parent[c] == u) with draft_tok[c] == target_argmax[u]; found with
// a ballot over 32 candidate nodes at a time.  parent[] values are only
// compared, never used as addresses, so a malformed tree cannot fault.
__global__ void __launch_bounds__(32) tree_accept_kernel(int N, const int32_t* __restrict__ parent,
                                                         const int32_t* __restrict__ draft_tok,
                                                         const int32_t* __restrict__ target_argmax,
                                                         int32_t* __restrict__ path,
                                                         int32_t* __restrict__ path_len,
                                                         int32_t* __restrict__ bonus) {
  const int b = blockIdx.x, lane = threadIdx.x;
  const int32_t* par = parent + (long long)b * N;
  const int32_t* tok = draft_tok + (long long)b * N;
  const int32_t* am = target_argmax + (long long)b * N;
  int32_t* out = path + (long long)b * N;
  int u = 0, len = 1;
  if (lane == 0) out[0] = 0;
  for (int step = 1; step < N; ++step) {
    const int want = am[u];
    int next = -1;
    for (int base = u + 1; base < N && next < 0; base += 32) {
      const int c = base + lane;
      const bool hit = c < N && par[c] == u && tok[c] == want;
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (m) next = base + __ffs(m) - 1;
    }
    if (next < 0) break;
    u = next;
    if (lane == 0) out[len] = u;
    ++len;
  }
  for (int k = len + lane; k < N; k += 32) out[k] = -1;
  if (lane == 0) { path_len[b] = len; bonus[b] = am[u]; }
}

// ---- KV compaction ----------------------------------------------------------------------
// Rows L + path[k] -> L + k, in chunks of kRowsChunk accepted nodes: a chunk
// is read completely into shared memory before any of its rows is written.
// Race-free because path is strictly increasing with path[k] >= k: the
// sources of later chunks (L + path[k'] >= L + k') are never destinations of
// earlier ones (L + k < L + k').
constexpr int kCompactThreads = 256;
constexpr int kRowsChunk = 16;

template <typename T>
__global__ void __launch_bounds__(kCompactThreads) compact_kernel(
    int N, int d_c, int d_rope, int page_size, int t_stride, int max_pages, int num_pages,
    T* __restrict__ c_kv, T* __restrict__ k_rope, const int32_t* __restrict__ prefix_len,
    const int32_t* __restrict__ path, const int32_t* __restrict__ path_len,
    const int32_t* __restrict__ page_table, unsigned int* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char cbuf[];
  T* rows = reinterpret_cast<T*>(cbuf);            // [kRowsChunk][d_c + d_rope]
  const int b = blockIdx.x;
  const int W = d_c + d_rope;
  const int L = prefix_len[b];
  const int n = path_len[b];
  const int32_t* pth = path + (long long)b * N;
  const int cap = page_size ? max_pages * page_size : t_stride;
  if (L < 0 || n < 1 || n > N || (long long)L + N > cap) {
    if (threadIdx.x == 0) atomicCAS(status, 0u, (unsigned)KDTV_ERR_BAD_PREFIX);
    return;
  }
  __shared__ int bad;
  if (threadIdx.x == 0) {
    bad = 0;
    for (int k = 0; k < n; ++k) {
      const int p = pth[k];
      if (p < k || p >= N || (k > 0 && p <= pth[k - 1])) bad = 1;
    }
    if (page_size)
      for (int p = L / page_size; p <= (L + N - 1) / page_size; ++p) {
        const int pg = page_table[(long long)b * max_pages + p];
        if (pg < 0 || pg >= num_pages) bad = 2;
      }
    if (bad) atomicCAS(status, 0u, bad == 1 ? (unsigned)KDTV_ERR_BAD_TREE : (unsigned)KDTV_ERR_BAD_PAGE);
  }
  __syncthreads();
  if (bad) return;
  auto row_of = [&](int t) -> long long {
    if (!page_size) return (long long)b * t_stride + t;
    return (long long)page_table[(long long)b * max_pages + t / page_size] * page_size +
           t % page_size;
  };
  for (int k0 = 0; k0 < n; k0 += kRowsChunk) {
    const int nk = min(kRowsChunk, n - k0);
    for (int idx = threadIdx.x; idx < nk * W; idx += blockDim.x) {
      const int k = idx / W, d = idx - k * W;
      const long long r = row_of(L + pth[k0 + k]);
      rows[idx] = d < d_c ? c_kv[r * d_c + d] : k_rope[r * d_rope + (d - d_c)];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nk * W; idx += blockDim.x) {
      const int k = idx / W, d = idx - k * W;
      const long long r = row_of(L + k0 + k);
      if (d < d_c) c_kv[r * d_c + d] = rows[idx];
      else k_rope[r * d_rope + (d - d_c)] = rows[idx];
    }
    __syncthreads();
  }
}

// ---- best-first tree build ----------------------------------------------------------------
// One CTA per request.  The frontier holds every candidate child (parent
// node, rank k) with its float32 score; each step takes the best candidate
// (highest score, then lower parent index, then lower k) with a block-wide
// reduction, appends it as the next node and adds its K children.
constexpr int kBuildThreads = 128;

struct Cand {
  float s;
  int key;   // parent * 65536 + k  (lower is preferred on equal scores)
};

__device__ __forceinline__ bool better(const Cand& a, const Cand& b) {
  return a.s > b.s || (a.s == b.s && a.key < b.key);
}

__global__ void __launch_bounds__(kBuildThreads) tree_build_kernel(
    int D, int K, int N, const float* __restrict__ logp, const int32_t* __restrict__ tokens,
    const int32_t* __restrict__ root_token, int32_t* __restrict__ parent_out,
    int32_t* __restrict__ token_out, int32_t* __restrict__ depth_out,
    float* __restrict__ score_out, int32_t* __restrict__ n_out) {
  extern __shared__ __align__(16) unsigned char sbuf[];
  float* cs = reinterpret_cast<float*>(sbuf);               // [N*K] candidate scores
  int* ck = reinterpret_cast<int*>(cs + N * K);             // [N*K] keys (-1 = taken/empty)
  int* ndepth = ck + N * K;                                 // [N]
  float* nscore = reinterpret_cast<float*>(ndepth + N);     // [N]
  __shared__ Cand red[kBuildThreads / 32];
  __shared__ Cand best_s;
  const int b = blockIdx.x, tid = threadIdx.x;
  const float* lp = logp + (long long)b * D * K;
  const int32_t* tk = tokens + (long long)b * D * K;
  int32_t* par = parent_out + (long long)b * N;
  int32_t* tok = token_out + (long long)b * N;
  int32_t* dep = depth_out + (long long)b * N;
  float* sco = score_out + (long long)b * N;

  for (int i = tid; i < N * K; i += blockDim.x) ck[i] = -1;
  if (tid == 0) {
    par[0] = -1; tok[0] = root_token[b]; dep[0] = 0; sco[0] = 0.f;
    ndepth[0] = 0; nscore[0] = 0.f;
  }
  __syncthreads();
  if (D > 0)
    for (int k = tid; k < K; k += blockDim.x) { cs[k] = 0.f + lp[k]; ck[k] = k; }
  __syncthreads();
  int n = 1;
  while (n < N) {
    Cand mine{-INFINITY, 0x7fffffff};
    bool any = false;
    for (int i = tid; i < n * K; i += blockDim.x) {
      if (ck[i] < 0) continue;
      Cand c{cs[i], ck[i]};
      if (!any || better(c, mine)) { mine = c; any = true; }
    }
    for (int off = 16; off; off >>= 1) {
      Cand o{__shfl_xor_sync(0xffffffffu, mine.s, off), __shfl_xor_sync(0xffffffffu, mine.key, off)};
      const bool oany = __shfl_xor_sync(0xffffffffu, (int)any, off);
      if (oany && (!any || better(o, mine))) { mine = o; any = true; }
    }
    if ((tid & 31) == 0) red[tid >> 5] = any ? mine : Cand{-INFINITY, -1};
    __syncthreads();
    if (tid == 0) {
      Cand bb{-INFINITY, -1};
      for (int w = 0; w < kBuildThreads / 32; ++w) {
        const Cand c = red[w];
        if (c.key < 0) continue;
        if (bb.key < 0 || better(c, bb)) bb = c;
      }
      best_s = bb;
    }
    __syncthreads();
    const Cand bb = best_s;
    if (bb.key < 0) break;                       // frontier empty
    const int u = bb.key >> 16, k = bb.key & 0xffff;
    const int d = ndepth[u];
    if (tid == 0) {
      ck[u * K + k] = -1;                        // taken
      par[n] = u; tok[n] = tk[d * K + k]; dep[n] = d + 1; sco[n] = bb.s;
      ndepth[n] = d + 1; nscore[n] = bb.s;
    }
    __syncthreads();
    if (d + 1 < D)
      for (int kk = tid; kk < K; kk += blockDim.x) {
        cs[n * K + kk] = __fadd_rn(bb.s, lp[(d + 1) * K + kk]);
        ck[n * K + kk] = n * 65536 + kk;
      }
    ++n;
    __syncthreads();
  }
  for (int i = n + tid; i < N; i += blockDim.x) { par[i] = -1; tok[i] = -1; dep[i] = -1; sco[i] = -INFINITY; }
  if (tid == 0) n_out[b] = n;
}

}  // namespace
}  // namespace kdtv

using namespace kdtv;

extern "C" int kdtv_tree_accept(int B, int N, const int32_t* parent, const int32_t* draft_tok,
                                const int32_t* target_argmax, int32_t* path, int32_t* path_len,
                                int32_t* bonus, cudaStream_t stream) {
  if (B <= 0 || N <= 0 || N > kMaxNodes) return B <= 0 || N <= 0 ? KDTV_ERR_INVALID_ARG : KDTV_ERR_UNSUPPORTED;
  if (!parent || !draft_tok || !target_argmax || !path || !path_len || !bonus)
    return KDTV_ERR_INVALID_ARG;
  tree_accept_kernel<<<B, 32, 0, stream>>>(N, parent, draft_tok, target_argmax, path, path_len,
                                           bonus);
  return cudaGetLastError() == cudaSuccess ? KDTV_OK : KDTV_ERR_CUDA;
}

extern "C" int kdtv_compact_kv(const kdtv_dims* d, void* c_kv, void* k_rope,
                               const int32_t* prefix_len, const int32_t* path,
                               const int32_t* path_len, const int32_t* page_table,
                               unsigned int* status, cudaStream_t stream) {
  if (!d || !c_kv || !k_rope || !prefix_len || !path || !path_len || !status)
    return KDTV_ERR_INVALID_ARG;
  if (d->B <= 0 || d->N <= 0 || d->d_c <= 0 || d->d_rope <= 0) return KDTV_ERR_INVALID_ARG;
  if (d->N > kMaxNodes) return KDTV_ERR_UNSUPPORTED;
  if ((d->page_size > 0) != (page_table != nullptr)) return KDTV_ERR_INVALID_ARG;
  if (d->page_size == 0 && d->t_stride < d->N) return KDTV_ERR_INVALID_ARG;
  if (d->page_size > 0 && (d->max_pages <= 0 || d->num_pages <= 0)) return KDTV_ERR_INVALID_ARG;
  const int W = d->d_c + d->d_rope;
  if (d->dtype == KDTV_BF16) {
    const size_t sm = sizeof(__nv_bfloat16) * kRowsChunk * W;
    compact_kernel<__nv_bfloat16><<<d->B, kCompactThreads, sm, stream>>>(
        d->N, d->d_c, d->d_rope, d->page_size, d->t_stride, d->max_pages, d->num_pages,
        static_cast<__nv_bfloat16*>(c_kv), static_cast<__nv_bfloat16*>(k_rope), prefix_len, path,
        path_len, page_table, status);
  } else if (d->dtype == KDTV_F32) {
    const size_t sm = sizeof(float) * kRowsChunk * W;
    compact_kernel<float><<<d->B, kCompactThreads, sm, stream>>>(
        d->N, d->d_c, d->d_rope, d->page_size, d->t_stride, d->max_pages, d->num_pages,
        static_cast<float*>(c_kv), static_cast<float*>(k_rope), prefix_len, path, path_len,
        page_table, status);
  } else {
    return KDTV_ERR_INVALID_ARG;
  }
  return cudaGetLastError() == cudaSuccess ? KDTV_OK : KDTV_ERR_CUDA;
}

extern "C" int kdtv_tree_build(int B, int D, int K, int N, const float* logp,
                               const int32_t* tokens, const int32_t* root_token,
                               int32_t* parent, int32_t* token, int32_t* depth, float* score,
                               int32_t* n_nodes, cudaStream_t stream) {
  if (B <= 0 || D < 0 || K <= 0 || N <= 0) return KDTV_ERR_INVALID_ARG;
  if (N > kMaxNodes || K > 64 || D > 4096) return KDTV_ERR_UNSUPPORTED;
  if ((D > 0 && (!logp || !tokens)) || !root_token || !parent || !token || !depth || !score ||
      !n_nodes)
    return KDTV_ERR_INVALID_ARG;
  const size_t sm = (size_t)N * K * (sizeof(float) + sizeof(int)) + (size_t)N * 8;
  if (sm > 48 * 1024 &&
      cudaFuncSetAttribute(tree_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sm) != cudaSuccess)
    return KDTV_ERR_CUDA;
  tree_build_kernel<<<B, kBuildThreads, sm, stream>>>(D, K, N, logp, tokens, root_token, parent,
                                                      token, depth, score, n_nodes);
  return cudaGetLastError() == cudaSuccess ? KDTV_OK : KDTV_ERR_CUDA;
}
