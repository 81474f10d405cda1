// Host side of the C ABI declared in include/kdtv.h: argument validation, the
// split-KV plan, workspace carving and dispatch to the CUDA-core or the
// tensor-core path.  Allocates nothing.

#include "kdtv_internal.cuh"

#include <math.h>
#include <string.h>

#include <atomic>

namespace kdtv {
namespace {

constexpr int kMaxDevices = 64;
// SM count per device, cached on first use; host threads may race to fill an
// entry (with the same value), hence atomics.
std::atomic<int> g_sm_count[kMaxDevices];

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < kMaxDevices) {
    const int c = g_sm_count[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
  return n;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int check_dims(const kdtv_dims* d) {
  if (!d) return KDTV_ERR_INVALID_ARG;
  if (d->B <= 0 || d->N <= 0 || d->H <= 0 || d->d_nope <= 0 || d->d_rope <= 0 ||
      d->d_v <= 0 || d->d_c <= 0)
    return KDTV_ERR_INVALID_ARG;
  if (d->dtype != KDTV_F32 && d->dtype != KDTV_BF16 && d->dtype != KDTV_BF16_FP8KV)
    return KDTV_ERR_INVALID_ARG;
  if (d->page_size < 0 || d->kv_chunk < 0) return KDTV_ERR_INVALID_ARG;
  if (d->page_size == 0) {
    if (d->t_stride < d->N) return KDTV_ERR_INVALID_ARG;
  } else {
    if (d->max_pages <= 0 || d->num_pages <= 0) return KDTV_ERR_INVALID_ARG;
    if ((long long)d->max_pages * d->page_size > (1ll << 30)) return KDTV_ERR_INVALID_ARG;
  }
  if (d->N > kMaxNodes) return KDTV_ERR_UNSUPPORTED;
  if (d->d_c > kMaxLatent || d->d_rope > kMaxRope || d->d_nope > 512 || d->d_v > 512)
    return KDTV_ERR_UNSUPPORTED;
  if ((long long)d->B * d->N * d->H > (1ll << 28)) return KDTV_ERR_UNSUPPORTED;
  return KDTV_OK;
}

// The dims the tensor-core kernels see: an fp8 cache is widened to bf16 first.
kdtv_dims tc_view(const kdtv_dims* d) {
  kdtv_dims v = *d;
  if (v.dtype == KDTV_BF16_FP8KV) v.dtype = KDTV_BF16;
  return v;
}

bool use_tensor_cores(const kdtv_dims* d) {
  if (d->dtype != KDTV_BF16 && d->dtype != KDTV_BF16_FP8KV) return false;
  const kdtv_dims v = tc_view(d);
  return !(d->flags & KDTV_FLAG_SIMT) && tc_supported(&v);
}

int make_plan(const kdtv_dims* d, Plan* p) {
  int st = check_dims(d);
  if (st != KDTV_OK) return st;
  if (d->dtype == KDTV_BF16 && !(d->flags & KDTV_FLAG_SIMT) && !tc_supported(d))
    return KDTV_ERR_UNSUPPORTED;
  memset(p, 0, sizeof(*p));
  p->tensor_core = use_tensor_cores(d);
  p->rows = d->B * d->N * d->H;
  p->t_cap = d->page_size ? d->max_pages * d->page_size : d->t_stride;
  const int sms = sm_count() > 0 ? sm_count() : 152;   // no device: size for a GB300
  p->sms = sms;
  const size_t rows = (size_t)p->rows;
  size_t off = kStatusBytes;
  if (p->tensor_core) {
    // Stream-K: one CTA pair per two SMs, each taking W consecutive 64-key
    // units of the (row tile, key tile) sequence (row tiles lane-major:
    // r = tile index * B + request); W is at least
    // wmin so that a row tile is cut into at most 63 pieces (the combine
    // kernel merges up to 64 partials per row).
    p->rt_count = (d->N * d->H + 127) / 128;
    const long long R = (long long)d->B * p->rt_count;
    const long long u_cap = (p->t_cap + 63) / 64;
    p->sk_wmin = (int)((u_cap + 61) / 62);
    if (p->sk_wmin < 1) p->sk_wmin = 1;
    p->sk_wforce = d->kv_chunk > 0 ? (d->kv_chunk + 63) / 64 : 0;
    long long clusters = sms / 2 > 0 ? sms / 2 : 1;
    // The boundary-aware plan (a gap of kSkBoundary virtual units before each
    // non-empty row tile but the first) where it measured faster: pairs
    // whose ranges are short (the whole cache capacity under 128 key tiles
    // per pair), and paged batches whose row tiles outnumber the pairs.
    // Elsewhere (one long request; contiguous batches of a few thousand keys
    // per request) the plain plan's kernel instance is as fast or faster.
    p->sk_gap = (R * u_cap < 128 * clusters || (d->page_size && R > clusters)) ? kSkBoundary : 0;
    const long long v_cap = R * u_cap + (long long)p->sk_gap * (R - 1);
    if (p->sk_wforce > 0) {
      const long long w = p->sk_wforce > p->sk_wmin ? p->sk_wforce : p->sk_wmin;
      const long long need = (v_cap + w - 1) / w;
      if (need > clusters) clusters = need;
    }
    if (clusters > (1 << 20) || v_cap >= (1ll << 30)) return KDTV_ERR_UNSUPPORTED;
    p->sk_clusters = (int)clusters;
    p->slots = (int)(R + clusters + 1);
    p->chunk = 64;
    p->splits = 1;
    p->off_qlat = off;    off = align256(off + rows * d->d_c * sizeof(float));
    p->off_part_o = off;  off = align256(off + (size_t)p->slots * 128 * d->d_c * sizeof(__nv_bfloat16));
    p->off_part_ml = off; off = align256(off + (size_t)p->slots * 128 * 2 * sizeof(float));
    p->off_olat = off;    off = align256(off + rows * d->d_c * sizeof(float));
    // header, {S, u, base} per row tile, first row tile per pair, then 8-int
    // first-piece records per pair (16-byte aligned)
    p->off_sk = off;      off = align256(off + (size_t)(kSkHeader + 3 * R + clusters + 3 + 8 * clusters) * sizeof(int));
    p->off_anc = off;     off = align256(off + (size_t)d->B * d->N * 4 * sizeof(uint32_t));
    if (d->dtype == KDTV_BF16_FP8KV) {
      // bf16 copies of the fp8 cache, in the input's layout
      const size_t kv_rows = d->page_size ? (size_t)d->num_pages * d->page_size
                                          : (size_t)d->B * d->t_stride;
      p->kv_widen = true;
      p->off_kvc = off;   off = align256(off + kv_rows * d->d_c * sizeof(__nv_bfloat16));
      p->off_kvr = off;   off = align256(off + kv_rows * d->d_rope * sizeof(__nv_bfloat16));
    }
  } else {
    p->heads_per_cta = d->H < 16 ? d->H : 16;
    long long base = (long long)d->B * d->N * ((d->H + p->heads_per_cta - 1) / p->heads_per_cta);
    long long want = (2ll * sms + base - 1) / base;
    long long max_s = (p->t_cap + 63) / 64;
    if (want < 1) want = 1;
    if (want > max_s) want = max_s;
    int chunk = (int)((p->t_cap + want - 1) / want);
    chunk = (chunk + 31) / 32 * 32;
    if (d->kv_chunk > 0) chunk = d->kv_chunk;
    p->chunk = chunk;
    p->splits = (p->t_cap + chunk - 1) / chunk;
    if (p->splits > 1024) return KDTV_ERR_UNSUPPORTED;
    p->off_qlat = off;    off = align256(off + rows * d->d_c * sizeof(float));
    p->off_part_o = off;  off = align256(off + (size_t)p->splits * rows * d->d_c * sizeof(float));
    p->off_part_ml = off; off = align256(off + (size_t)p->splits * rows * 2 * sizeof(float));
    p->off_olat = off;    off = align256(off + rows * d->d_c * sizeof(float));
  }
  p->total = off;
  return KDTV_OK;
}

}  // namespace
}  // namespace kdtv

using namespace kdtv;

namespace kdtv {
// Host-side plan check of a call: the status kdtv_verify_attn returns before
// any launch for these dims (KDTV_OK, INVALID_ARG or UNSUPPORTED) and, when
// OK, the workspace bytes it needs.
int plan_status(const kdtv_dims* d, size_t* bytes) {
  Plan p;
  const int st = make_plan(d, &p);
  if (bytes) *bytes = st == KDTV_OK ? p.total : 0;
  return st;
}
int device_sm_count() { return sm_count(); }
}  // namespace kdtv

extern "C" size_t kdtv_workspace_size(const kdtv_dims* d) {
  Plan p;
  if (make_plan(d, &p) != KDTV_OK) return 0;
  return p.total;
}

extern "C" int kdtv_launches_per_call(const kdtv_dims* d) {
  Plan p;
  if (make_plan(d, &p) != KDTV_OK) return -1;
  if (!p.tensor_core) return 4;
  const kdtv_dims v = tc_view(d);
  return tc_launches(&v, p.splits) + (p.kv_widen ? 1 : 0);
}

extern "C" int kdtv_verify_attn(const kdtv_dims* d, const void* q_nope, const void* q_rope,
                                const void* W_UK, const void* W_UV, const void* c_kv,
                                const void* k_rope, const int32_t* parent,
                                const int32_t* prefix_len, const int32_t* page_table,
                                float* out, cudaStream_t stream) {
  Plan p;
  int st = make_plan(d, &p);
  if (st != KDTV_OK) return st;
  if (!q_nope || !q_rope || !W_UK || !W_UV || !c_kv || !k_rope || !parent || !prefix_len ||
      !out)
    return KDTV_ERR_INVALID_ARG;
  if ((d->page_size > 0) != (page_table != nullptr)) return KDTV_ERR_INVALID_ARG;
  if (!d->workspace || (reinterpret_cast<uintptr_t>(d->workspace) & 255u) ||
      d->workspace_bytes < p.total)
    return KDTV_ERR_INVALID_ARG;

  Args a;
  memset(&a, 0, sizeof(a));
  a.B = d->B; a.N = d->N; a.H = d->H;
  a.d_nope = d->d_nope; a.d_rope = d->d_rope; a.d_v = d->d_v; a.d_c = d->d_c;
  a.dtype = d->dtype;
  a.page_size = d->page_size; a.t_stride = d->t_stride;
  a.max_pages = d->max_pages; a.num_pages = d->num_pages;
  a.scale = d->scale > 0.f ? d->scale : 1.0f / sqrtf((float)(d->d_nope + d->d_rope));
  a.kv_scale = (d->dtype == KDTV_BF16_FP8KV && d->kv_scale > 0.f) ? d->kv_scale : 1.0f;
  a.o_scale = 1.0f;
  a.flags = d->flags;
  a.chunk = p.chunk; a.splits = p.splits;
  a.q_nope = q_nope; a.q_rope = q_rope; a.W_UK = W_UK; a.W_UV = W_UV;
  a.c_kv = c_kv; a.k_rope = k_rope;
  a.parent = parent; a.prefix_len = prefix_len; a.page_table = page_table;
  a.out = out;
  char* ws = static_cast<char*>(d->workspace);
  a.status = reinterpret_cast<DeviceStatus*>(ws);
  a.q_lat = ws + p.off_qlat;
  a.part_o = reinterpret_cast<float*>(ws + p.off_part_o);
  a.part_ml = reinterpret_cast<float*>(ws + p.off_part_ml);
  a.o_lat = reinterpret_cast<float*>(ws + p.off_olat);
  if (p.tensor_core) {
    a.part_o = nullptr;
    a.part_o16 = reinterpret_cast<__nv_bfloat16*>(ws + p.off_part_o);
    a.sk = reinterpret_cast<int*>(ws + p.off_sk);
    a.anc_g = reinterpret_cast<uint32_t*>(ws + p.off_anc);
    a.rt_count = p.rt_count;
    a.sk_clusters = p.sk_clusters;
    a.sk_wmin = p.sk_wmin;
    a.sk_wforce = p.sk_wforce;
    a.sk_gap = p.sk_gap;
  }

  cudaEvent_t* ev = d->phase_events;
  if (ev && cudaEventRecord(ev[0], stream) != cudaSuccess) return KDTV_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, kStatusBytes, stream) != cudaSuccess) return KDTV_ERR_CUDA;
  if (p.kv_widen) {
    // The bf16 kernels read exact bf16 copies of the fp8 values, written by
    // a widening kernel ahead of the attention; kv_scale moves onto the
    // scores and onto o_lat (both linear in the cache).
    a.c_kv8 = a.c_kv;
    a.k_rope8 = a.k_rope;
    a.c_kv = ws + p.off_kvc;
    a.k_rope = ws + p.off_kvr;
    a.dtype = KDTV_BF16;
    a.scale *= a.kv_scale;
    a.o_scale = a.kv_scale;
  }
  cudaError_t e = p.tensor_core ? launch_tc(a, p, stream, ev) : launch_simt(a, p, stream, ev);
  return e == cudaSuccess ? KDTV_OK : KDTV_ERR_CUDA;
}

extern "C" int kdtv_get_device_status(const kdtv_dims* d, cudaStream_t stream) {
  if (!d || !d->workspace) return KDTV_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KDTV_ERR_CUDA;
  unsigned int code = 0;
  if (cudaMemcpy(&code, d->workspace, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KDTV_ERR_CUDA;
  return (int)code;
}

extern "C" const char* kdtv_strerror(int s) {
  switch (s) {
    case KDTV_OK: return "KDTV_OK";
    case KDTV_ERR_INVALID_ARG: return "KDTV_ERR_INVALID_ARG";
    case KDTV_ERR_UNSUPPORTED: return "KDTV_ERR_UNSUPPORTED";
    case KDTV_ERR_CUDA: return "KDTV_ERR_CUDA";
    case KDTV_ERR_BAD_TREE: return "KDTV_ERR_BAD_TREE";
    case KDTV_ERR_DEVICE_TIMEOUT: return "KDTV_ERR_DEVICE_TIMEOUT";
    case KDTV_ERR_BAD_PREFIX: return "KDTV_ERR_BAD_PREFIX";
    case KDTV_ERR_BAD_PAGE: return "KDTV_ERR_BAD_PAGE";
    default: return "KDTV_ERR_UNKNOWN";
  }
}
