/*
 * kdtv.h — tree-verify MLA-absorb attention on GB300 (sm_103a), C ABI.
 *
 * The operation.  In DDTree speculative decoding the target model scores every
 * node of a draft token tree in one forward pass under a custom attention
 * mask: a node sees the committed prefix plus only its own tree ancestors, and
 * MLA's absorbed form folds the key/value up-projections (w_kc / w_vc) into
 * the attention ("The Moment of Proof: Validating a Native CUDA Speculative
 * Decoding Engine", section "Input Knowledge Required"; the kernel is the
 * "tree-verify MLA-absorb attention kernel with visibility masking" of section
 * "The Context: Building a Native DDTree Engine from Scratch").  For request
 * b, node i and head h:
 *
 *   q_lat   = W_UK[h]^T q_nope[b,i,h]                       (absorb)
 *   Vis(i)  = {0 .. L_b-1} U {L_b + a : a on the root path of i, i included}
 *   s_t     = scale * (q_lat . c_kv[b,t] + q_rope[b,i,h] . k_rope[b,t]),  t in Vis(i)
 *   o_lat   = sum_t softmax(s)_t c_kv[b,t]
 *   out     = W_UV[h] o_lat                                  (up-projection)
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller.  The library
 *     allocates no memory; scratch lives in the caller's workspace.  One
 *     exception: kdtv_verify_attn_noalloc (end of this file) takes its scratch
 *     from a fixed array in the library's own device image.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and never
 *     synchronise, except kdtv_get_device_status.
 *   - Layouts are row-major with the last dimension contiguous.
 *   - Return value: KDTV_OK or a KDTV_ERR_* code found on the host before any
 *     launch.  Conditions only the device can see (a malformed parent[], a
 *     prefix that overflows the cache, a bad page id, a wait that ran out) are
 *     recorded in the workspace status word; read it with
 *     kdtv_get_device_status (kdtv_verify_attn_noalloc instead copies it to
 *     its status_out argument; kdtv_get_device_status does not apply to it).
 *     The affected rows are left unwritten; nothing traps, and the CUDA
 *     context stays usable.
 *   - Calls that share a workspace must not overlap on the GPU.  Host threads
 *     may call at the same time with separate workspaces.
 */
#ifndef KDTV_H
#define KDTV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDTV_ABI_VERSION 2

/* Element type of q_nope, q_rope, W_UK, W_UV, c_kv and k_rope.  `out` is
 * always float32. */
enum kdtv_dtype {
  KDTV_F32 = 0,      /* every input float32; computed on CUDA cores in fp32   */
  KDTV_BF16 = 1,     /* every input bf16; tensor cores, fp32 accumulation     */
  KDTV_BF16_FP8KV = 2 /* q_nope, q_rope, W_UK, W_UV bf16; the latent cache c_kv
                        and k_rope one byte per element, OCP FP8 E4M3 (4-bit
                        exponent with bias 7, 3-bit mantissa, no infinities,
                        S.1111.111 = NaN), value = fp8 * kv_scale.  Tensor
                        cores (the default where KDTV_BF16 has them): the
                        rows a call reads are first widened exactly to bf16
                        copies in the workspace (kdtv_workspace_size grows
                        by 2 * (d_c + d_rope) bytes per cache row), rows past
                        L_b + N in a request's last 64-key tile written as
                        zeros; KDTV_FLAG_SIMT: fp32 on CUDA cores            */
};

enum kdtv_status {
  KDTV_OK = 0,
  KDTV_ERR_INVALID_ARG = 1,     /* null pointer, non-positive dim, bad layout field,
                                   workspace too small                           */
  KDTV_ERR_UNSUPPORTED = 2,     /* N > 128, or dims outside what a path supports  */
  KDTV_ERR_CUDA = 3,            /* a CUDA call or launch failed                   */
  KDTV_ERR_BAD_TREE = 4,        /* device: parent[b][0] != -1 or parent[b][i] not
                                   in [0, i)                                      */
  KDTV_ERR_DEVICE_TIMEOUT = 5,  /* device: a bounded wait ran out                 */
  KDTV_ERR_BAD_PREFIX = 6,      /* device: prefix_len[b] < 0 or L_b + N exceeds
                                   t_stride / max_pages * page_size               */
  KDTV_ERR_BAD_PAGE = 7         /* device: a page id outside [0, num_pages)       */
};

/* kdtv_dims.flags */
#define KDTV_FLAG_SIMT 0x1u          /* bf16 / fp8-cache inputs on the CUDA-core
                                        path (the tensor-core path is the
                                        default)                                  */
#define KDTV_FLAG_SIMT_PROJ 0x2u     /* bf16: tensor-core attention, but the absorb,
                                        split combine and up-projection on CUDA
                                        cores                                     */
#define KDTV_FLAG_TEST_STALL 0x100u  /* TEST ONLY: the attention kernel waits on a
                                        barrier that nothing arrives on, with a
                                        ~20 ms limit, so the timeout path can be
                                        checked; the call then reports
                                        KDTV_ERR_DEVICE_TIMEOUT                  */

typedef struct kdtv_dims {
  int32_t B;          /* requests in the batch                                  */
  int32_t N;          /* tree nodes per request, 1..128                         */
  int32_t H;          /* attention heads                                        */
  int32_t d_nope;     /* qk_nope head dim                                       */
  int32_t d_rope;     /* qk_rope head dim                                       */
  int32_t d_v;        /* v head dim                                             */
  int32_t d_c;        /* kv_lora (latent) dim                                   */
  int32_t dtype;      /* enum kdtv_dtype                                        */
  int32_t page_size;  /* 0: contiguous cache; 64: paged cache                   */
  int32_t t_stride;   /* contiguous: rows per request in c_kv / k_rope          */
  int32_t max_pages;  /* paged: length of each page_table row                   */
  int32_t num_pages;  /* paged: physical pages held by c_kv / k_rope            */
  float scale;        /* softmax scale; <= 0 selects 1/sqrt(d_nope + d_rope)    */
  uint32_t flags;     /* KDTV_FLAG_*                                            */
  int32_t kv_chunk;   /* keys per split-KV chunk; 0 = chosen by the library     */
  float kv_scale;     /* KDTV_BF16_FP8KV: dequantisation scale of the cache;
                         <= 0 selects 1.  Ignored for the other dtypes          */
  void* workspace;          /* device scratch, >= kdtv_workspace_size() bytes,
                               256-byte aligned, owned by the caller             */
  size_t workspace_bytes;
  cudaEvent_t* phase_events; /* optional: NULL, or 5 events recorded on `stream`
                               at the start of the call and after the absorb,
                               the attention, the split-KV combine and the
                               up-projection                                     */
} kdtv_dims;

/* Bytes of workspace kdtv_verify_attn needs for these dims on the current
 * device (the split-KV plan depends on the device's SM count).  Returns 0 if
 * the dims are invalid. */
size_t kdtv_workspace_size(const kdtv_dims* dims);

/*
 * kdtv_verify_attn — the whole hot path: absorb, tree-masked attention over
 * the latent cache with online softmax and split-KV, split combine, W_UV
 * up-projection.
 *
 *   q_nope     [B, N, H, d_nope]
 *   q_rope     [B, N, H, d_rope]   already rotated
 *   W_UK       [H, d_nope, d_c]    k_nope[h] = W_UK[h] c
 *   W_UV       [H, d_v, d_c]       v[h]      = W_UV[h] c
 *   c_kv       contiguous: [B, t_stride, d_c];  paged: [num_pages, page_size, d_c]
 *   k_rope     contiguous: [B, t_stride, d_rope]; paged: [num_pages, page_size, d_rope]
 *              (one rope head shared by all heads, already rotated)
 *   parent     [B, N] int32: parent[b][0] = -1, parent[b][i] in [0, i)
 *   prefix_len [B] int32: committed prefix L_b >= 0; the tree nodes' own latent
 *              rows sit at positions L_b .. L_b + N - 1
 *   page_table [B, max_pages] int32: physical page of logical page p of request b
 *              (NULL iff page_size == 0); only entries p < ceil((L_b+N)/page_size)
 *              are read
 *   out        [B, N, H, d_v] float32, written in full on success
 *
 * bf16 needs d_c == 512 and d_rope == 64 (the Kimi-K2 / DeepSeek latent
 * layout) unless KDTV_FLAG_SIMT is set; fp32 takes d_c <= 512, d_rope <= 64,
 * d_nope <= 512, d_v <= 512.
 */
int kdtv_verify_attn(const kdtv_dims* dims, const void* q_nope, const void* q_rope,
                     const void* W_UK, const void* W_UV, const void* c_kv,
                     const void* k_rope, const int32_t* parent,
                     const int32_t* prefix_len, const int32_t* page_table,
                     float* out, cudaStream_t stream);

/* Synchronises `stream`, then returns the first device-side error recorded in
 * the workspace by the last call that used it (KDTV_OK if none). */
int kdtv_get_device_status(const kdtv_dims* dims, cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char* kdtv_strerror(int status);

/* Number of kernels kdtv_verify_attn launches for these dims (for launch
 * accounting), or -1 if the dims are invalid. */
int kdtv_launches_per_call(const kdtv_dims* dims);

/* ---- the loop steps around the verify attention -------------------------------------
 * "The Moment of Proof: Validating a Native CUDA Speculative Decoding Engine",
 * section "The Context: Building a Native DDTree Engine from Scratch", names a
 * GPU best-first tree builder, a greedy tree-accept kernel and post-verify KV
 * cache compaction.  Each runs one CTA per request (trees have <= 128 nodes).
 */

/*
 * kdtv_tree_accept — greedy acceptance ("The Build That Proved It: Compiling
 * the Native DDTree Speculative Decoding Engine", section "The Output Knowledge
 * Created": the accept kernel keeps the longest prefix match).  Node 0 is the
 * root (the last committed token).  From node u the walk moves to the
 * lowest-indexed child c of u with draft_tok[c] == target_argmax[u] and stops
 * when there is none.
 *   parent, draft_tok, target_argmax  [B, N] int32 (device)
 *   path      [B, N] int32 out: accepted node indices (path[0] = 0), then -1
 *   path_len  [B] int32 out: accepted nodes including the root
 *   bonus     [B] int32 out: target_argmax at the last accepted node
 * Commits path_len - 1 draft tokens plus the bonus token.  parent[] is only
 * compared, never dereferenced, so a malformed tree cannot fault.  Returns
 * KDTV_ERR_INVALID_ARG / KDTV_ERR_UNSUPPORTED (N > 128) / KDTV_ERR_CUDA.
 */
int kdtv_tree_accept(int B, int N, const int32_t* parent, const int32_t* draft_tok,
                     const int32_t* target_argmax, int32_t* path, int32_t* path_len,
                     int32_t* bonus, cudaStream_t stream);

/*
 * kdtv_compact_kv — post-verify KV compaction, in place ("The Moment of
 * Truth: Validating a Custom CUDA Inference Engine for Kimi K2.6", section
 * "What the Output Tells Us": kept rows are gathered into a compact cache
 * without an in-place race).  For each request b the latent rows at positions
 * prefix_len[b] + path[b][k] move to prefix_len[b] + k, k < path_len[b]; all
 * other rows are untouched.  Uses dims->B, N, d_c, d_rope, dtype, page_size,
 * t_stride, max_pages, num_pages (same layouts as kdtv_verify_attn); c_kv and
 * k_rope are modified in place.  path must be strictly increasing with
 * path[k] >= k (as kdtv_tree_accept produces).  Device-side problems (bad
 * path, prefix overflow, bad page id) leave that request untouched and set
 * *status (device word, first error wins) to KDTV_ERR_BAD_TREE /
 * KDTV_ERR_BAD_PREFIX / KDTV_ERR_BAD_PAGE.  Requests must not share pages.
 */
int kdtv_compact_kv(const kdtv_dims* dims, void* c_kv, void* k_rope,
                    const int32_t* prefix_len, const int32_t* path, const int32_t* path_len,
                    const int32_t* page_table, unsigned int* status, cudaStream_t stream);

/*
 * kdtv_tree_build — best-first draft tree from per-depth top-K proposals
 * ("The Moment of Proof: Validating a Native CUDA Speculative Decoding
 * Engine", section "The Context: Building a Native DDTree Engine from
 * Scratch": the GPU builder that replaces a per-request CPU heap).
 * Node 0 is the root (root_token[b], depth 0, score 0).  A node at depth d < D
 * offers K candidate children (tokens[b][d][k], score + logp[b][d][k], float32
 * addition); the best candidate (highest score, then lower parent index, then
 * lower k) becomes the next node until N nodes exist or no candidate is left.
 *   logp [B, D, K] float32, tokens [B, D, K] int32, root_token [B] int32
 *   parent, token, depth [B, N] int32 out; score [B, N] float32 out (node
 *   order is topological; unused slots are -1 / -inf); n_nodes [B] int32 out.
 * logp must hold no NaN: the place of a NaN score in the order is unspecified.
 * Returns KDTV_ERR_INVALID_ARG, KDTV_ERR_UNSUPPORTED (N > 128, K > 64) or
 * KDTV_ERR_CUDA.
 */
int kdtv_tree_build(int B, int D, int K, int N, const float* logp, const int32_t* tokens,
                    const int32_t* root_token, int32_t* parent, int32_t* token,
                    int32_t* depth, float* score, int32_t* n_nodes, cudaStream_t stream);

/* ---- allocation-free variant ----------------------------------------------------------
 * The pages have no counterpart to this entry point; it exists for callers of
 * this library that cannot call cudaMalloc where they run the attention (code
 * inside an arena or pool allocator that owns all device memory, server
 * plugins that may only touch pre-registered buffers, or processes that
 * forbid device allocation after start-up).
 *
 * kdtv_verify_attn_noalloc computes exactly what kdtv_verify_attn computes,
 * with the same arguments, but takes its scratch from a fixed array of
 * KDTV_NOALLOC_SCRATCH_BYTES that lives in this library's device image
 * (dims->workspace and dims->workspace_bytes are ignored).  It allocates
 * nothing.  Every GPU that loads the library holds that array until the
 * process exits.
 *   - Returns KDTV_ERR_UNSUPPORTED, before any launch, if the call needs more
 *     scratch than KDTV_NOALLOC_SCRATCH_BYTES (kdtv_workspace_size(dims) larger
 *     than the array); every other host-side error is the code
 *     kdtv_verify_attn returns for the same dims and pointers.
 *   - status_out: device pointer to one unsigned int; when the call's kernels
 *     have finished it holds the call's device status (KDTV_OK or a device-side
 *     KDTV_ERR_* as kdtv_get_device_status would report).  Asynchronous on
 *     `stream` like every other entry point.
 *   - The first call on a device looks up the array's device address with
 *     that device current (cudaGetSymbolAddress), and again only if the
 *     device's CUDA context has since been replaced; make that first call
 *     before any stream capture on that device.  Concurrent first calls from
 *     several host threads are safe.
 *   - All calls share the one array per device: calls that may overlap on the
 *     GPU (different streams or host threads) race and must be serialised by
 *     the caller.
 */
#define KDTV_NOALLOC_SCRATCH_BYTES (64u << 20)

int kdtv_verify_attn_noalloc(const kdtv_dims* dims, const void* q_nope, const void* q_rope,
                             const void* W_UK, const void* W_UV, const void* c_kv,
                             const void* k_rope, const int32_t* parent,
                             const int32_t* prefix_len, const int32_t* page_table,
                             float* out, unsigned int* status_out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* KDTV_H */
