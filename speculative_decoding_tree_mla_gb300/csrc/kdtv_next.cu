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
// One warp per request.  Candidate child k of node u (slot u K + k) is one
// 64-bit word whose unsigned order is the preference order: the score's
// order-preserving bits in the high half (higher score first); in the low
// half, (2^25 - 1 - (64 u + k)) << 7 (a lower parent and then a lower k win
// ties) with the parent's depth in the low 7 bits (N <= 128, K <= 64 and the
// depths used are below 128, so the key is unique and the depth never decides
// the order); 0 is a taken or absent child.  Each node keeps the word of its
// best remaining child in a register of lane (node % 32), so a step is:
//   * a warp-wide maximum over the node words (two 32-bit reductions: the
//     high half, then the low half among the lanes holding the highest);
//   * the winner becomes node n;
//   * the lanes recompute the best remaining child of the winner's parent and
//     the best child of the new node (K children each, one per lane), and the
//     two owning lanes update their registers.
// The proposals of the depths a tree can reach (min(D, N - 1)) are staged in
// shared memory first; the nodes are written out at the end.
constexpr int kBuildThreads = 32;

__device__ __forceinline__ uint32_t order_bits(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_order_bits(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
__device__ __forceinline__ unsigned long long cand_word(float s, int u, int k, int parent_depth) {
  const uint32_t key = 0x1ffffffu - (uint32_t)(u * 64 + k);
  return ((unsigned long long)order_bits(s) << 32) | (key << 7) | (uint32_t)parent_depth;
}
// This lane's node words (nodes lane, lane + 32, lane + 64, lane + 96): set
// the one of node x to w if this lane owns it.
__device__ __forceinline__ void set_node_word(unsigned long long& n0, unsigned long long& n1,
                                              unsigned long long& n2, unsigned long long& n3,
                                              int x, int lane, unsigned long long w) {
  const bool mine = (x & 31) == lane;
  const int j = x >> 5;
  n0 = (mine && j == 0) ? w : n0;
  n1 = (mine && j == 1) ? w : n1;
  n2 = (mine && j == 2) ? w : n2;
  n3 = (mine && j == 3) ? w : n3;
}
// Maximum of a 64-bit word over the warp.
__device__ __forceinline__ unsigned long long warp_max_word(unsigned long long w) {
  const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(w >> 32));
  const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(w >> 32) == hi ? (uint32_t)w : 0u);
  return ((unsigned long long)hi << 32) | lo;
}

__global__ void __launch_bounds__(kBuildThreads) tree_build_kernel(
    int D, int K, int N, const float* __restrict__ logp, const int32_t* __restrict__ tokens,
    const int32_t* __restrict__ root_token, int32_t* __restrict__ parent_out,
    int32_t* __restrict__ token_out, int32_t* __restrict__ depth_out,
    float* __restrict__ score_out, int32_t* __restrict__ n_out) {
  extern __shared__ __align__(16) unsigned char sbuf[];
  const int Ds = D < N - 1 ? D : N - 1;                      // depths whose proposals are used
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(sbuf);   // [N*K]
  int* ndepth = reinterpret_cast<int*>(cand + N * K + N);   // [N]
  float* lps = reinterpret_cast<float*>(ndepth + N);        // [Ds*K] staged log-probabilities
  int* tks = reinterpret_cast<int*>(lps + Ds * K);          // [Ds*K] staged tokens
  int* opar = tks + Ds * K;                                 // [N] outputs, written out at the end
  int* otok = opar + N;
  float* osco = reinterpret_cast<float*>(otok + N);
  const int b = blockIdx.x, lane = threadIdx.x;
  const float* lp = logp + (long long)b * D * K;
  const int32_t* tk = tokens + (long long)b * D * K;

#pragma unroll 4
  for (int i = lane; i < Ds * K; i += 32) { lps[i] = lp[i]; tks[i] = tk[i]; }
  __syncwarp();
  unsigned long long nb0 = 0ull, nb1 = 0ull, nb2 = 0ull, nb3 = 0ull;   // nodes lane, lane + 32, ...
  // the root and its children
  {
    unsigned long long m = 0ull;
    if (Ds > 0)
      for (int k = lane; k < K; k += 32) {
        const unsigned long long w = cand_word(__fadd_rn(0.f, lps[k]), 0, k, 0);
        cand[k] = w;
        m = max(m, w);
      }
    m = warp_max_word(m);
    if (lane == 0) {
      nb0 = m;
      opar[0] = -1; otok[0] = root_token[b]; osco[0] = 0.f;
      ndepth[0] = 0;
    }
  }
  __syncwarp();
  int n = 1;
  while (n < N) {
    const unsigned long long win = warp_max_word(max(max(nb0, nb1), max(nb2, nb3)));
    if (win == 0ull) break;                       // frontier empty
    const float sw = from_order_bits((uint32_t)(win >> 32));
    const uint32_t low = (uint32_t)win;
    const int d = (int)(low & 127u);              // the parent's depth
    const int key = (int)(0x1ffffffu - (low >> 7));
    const int u = key >> 6, k = key & 63;
    const bool grow = d + 1 < Ds;
    // the parent's remaining children, and the new node's children
    unsigned long long mu = 0ull, mn = 0ull;
    for (int kk = lane; kk < K; kk += 32) {
      unsigned long long wu = cand[u * K + kk];
      if (kk == k) { wu = 0ull; cand[u * K + kk] = 0ull; }   // taken
      mu = max(mu, wu);
      if (grow) {
        const unsigned long long wn = cand_word(__fadd_rn(sw, lps[(d + 1) * K + kk]), n, kk, d + 1);
        cand[n * K + kk] = wn;
        mn = max(mn, wn);
      }
    }
    mu = warp_max_word(mu);
    mn = warp_max_word(mn);
    set_node_word(nb0, nb1, nb2, nb3, u, lane, mu);
    set_node_word(nb0, nb1, nb2, nb3, n, lane, mn);
    if (lane == 0) {
      opar[n] = u; otok[n] = tks[d * K + k]; osco[n] = sw;
      ndepth[n] = d + 1;
    }
    __syncwarp();
    ++n;
  }
  __syncwarp();
  int32_t* par = parent_out + (long long)b * N;
  int32_t* tok = token_out + (long long)b * N;
  int32_t* dep = depth_out + (long long)b * N;
  float* sco = score_out + (long long)b * N;
  for (int i = lane; i < N; i += 32) {
    const bool live = i < n;
    par[i] = live ? opar[i] : -1;
    tok[i] = live ? otok[i] : -1;
    dep[i] = live ? ndepth[i] : -1;
    sco[i] = live ? osco[i] : -INFINITY;
  }
  if (lane == 0) n_out[b] = n;
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
  } else if (d->dtype == KDTV_BF16_FP8KV) {   // one-byte cache elements, moved as bytes
    const size_t sm = sizeof(unsigned char) * kRowsChunk * W;
    compact_kernel<unsigned char><<<d->B, kCompactThreads, sm, stream>>>(
        d->N, d->d_c, d->d_rope, d->page_size, d->t_stride, d->max_pages, d->num_pages,
        static_cast<unsigned char*>(c_kv), static_cast<unsigned char*>(k_rope), prefix_len, path,
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
  const int Ds = D < N - 1 ? D : N - 1;
  const size_t sm = (size_t)(N * K + N) * sizeof(unsigned long long) + (size_t)N * 4 * sizeof(int) +
                    (size_t)Ds * K * (sizeof(float) + sizeof(int));
  if (sm > 48 * 1024 &&
      cudaFuncSetAttribute(tree_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sm) != cudaSuccess)
    return KDTV_ERR_CUDA;
  tree_build_kernel<<<B, kBuildThreads, sm, stream>>>(D, K, N, logp, tokens, root_token, parent,
                                                      token, depth, score, n_nodes);
  return cudaGetLastError() == cudaSuccess ? KDTV_OK : KDTV_ERR_CUDA;
}
