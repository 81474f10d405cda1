// Tensor-core (tcgen05) kernels for the two per-head projections around the
// attention, the absorbed form's w_kc / w_vc halves ("The Moment of Proof:
// Validating a Native CUDA Speculative Decoding Engine", section "Input
// Knowledge Required"):
//
//   absorb_tc_kernel            q_lat[r, h, :] = W_UK[h]^T q_nope[r, h, :]   (bf16 out)
//   combine_uproj_small_kernel  o_lat = log-sum-exp merge of the split partials,
//   combine_uproj_pipe_kernel   out[r, h, :] = W_UV[h] o_lat                 (fp32 out);
//                               the first for batches whose grid fits one wave,
//                               the second (K-chunk pipeline) for larger ones
//
// Both run transposed so the weight matrix is the 128-row MMA operand and the
// query rows are the MMA N dimension: D[128 x rows] = W-block . X^T, with the
// weight tile loaded by TMA (W_UK read as an MN-major operand) and the result
// read back lane-per-output-feature, which makes the global writes coalesced.

#include <cuda.h>

#include "kdtv_internal.cuh"
#include "kdtv_ptx.cuh"
#include "kdtv_tmap.cuh"

namespace kdtv {
namespace {

using namespace ptx;

constexpr int kThreads = 128;
constexpr uint64_t kLimitNs = 2000000000ull;

// ---- A1: absorb -----------------------------------------------------------------------
constexpr int AB_M = 128;                  // latent columns per CTA
constexpr int AB_NR = 128;                 // query rows (b, i) per CTA

// Shared memory of absorb_tc_kernel for a given d_nope: A = two MN atoms of
// d_nope e-rows x 128 B, B = d_nope/64 chunks of AB_NR rows x 128 B, barriers.
__host__ __device__ constexpr int ab_off_b(int d_nope) { return 2 * d_nope * 128; }
__host__ __device__ constexpr int ab_off_bar(int d_nope) {
  return ab_off_b(d_nope) + (d_nope / 64) * AB_NR * 128;
}
__host__ __device__ constexpr int ab_smem(int d_nope) { return ab_off_bar(d_nope) + 64 + 1024; }

__global__ void __launch_bounds__(kThreads, 1)
absorb_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_q,
                 const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d0 = blockIdx.x * AB_M;
  const int h = blockIdx.y;
  const int r0 = blockIdx.z * AB_NR;
  const int BNr = a.B * a.N;
  const int nr = min(AB_NR, BNr - r0);
  const int kch = a.d_nope / 64;             // 64-wide K chunks
  const int off_b = ab_off_b(a.d_nope), off_bar = ab_off_bar(a.d_nope);
  const uint32_t bar_full = sbase + off_bar, bar_mma = bar_full + 8;
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(sm + off_bar + 16);
  grid_dep_launch();   // the attention kernel may start its prologue early

  if (tid == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) { tmem_alloc(sbase + off_bar + 16, AB_NR); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  bool ok = true;
  if (tid == 0) {
    const uint32_t w_bytes = 2u * a.d_nope * 128u;
    mbar_expect_tx(bar_full, w_bytes + kch * AB_NR * 128u);
    for (int c = 0; c < 2; ++c)       // W_UK[h][:, d0 + 64c : +64]: e-rows x 64 d
      tma_load_2d(sbase + c * a.d_nope * 128, &tm_w, bar_full, d0 + 64 * c, h * a.d_nope);
    for (int k = 0; k < kch; ++k)     // q_nope rows r0.. of head h, e in [64k, 64k+64)
      tma_load_2d(sbase + off_b + k * AB_NR * 128, &tm_q, bar_full, h * a.d_nope + 64 * k, r0);
    ok = wait(bar_full, 0, a.status, kLimitNs, 101);
    if (ok) {
      tc_fence_after();
      // D[128 rows x 128 d] = q_nope rows (A, K-major) x W_UK block (B, MN-major);
      // rows past the last query row are zero-filled by TMA and never stored.
      const uint32_t idesc = idesc_bf16(AB_NR, AB_M, /*a_mn=*/0, /*b_mn=*/1);
      for (int kk = 0; kk < a.d_nope / 16; ++kk) {
        uint64_t ad = smem_desc(sbase + off_b + (kk >> 2) * AB_NR * 128 + (kk & 3) * 32, 16, 1024);
        // B (MN-major): 64-column atoms a.d_nope*128 B apart, 8 e-rows per 1 KiB.
        uint64_t bd = smem_desc(sbase + kk * 16 * 128, a.d_nope * 128, 1024);
        mma_bf16(tmem, ad, bd, idesc, kk > 0);
      }
    }
    mma_commit(bar_mma);
  }
  __syncwarp();
  ok = wait(bar_mma, 0, a.status, kLimitNs, 102) && ok;
  ok = __all_sync(0xffffffffu, ok);
  tc_fence_after();
  if (ok && warp * 32 < nr) {
    // TMEM lane = query row: each thread writes its row's 128 latent columns
    // as sixteen 16-byte vectors.
    const int r = warp * 32 + lane;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.q_lat) +
                                          ((long long)(r0 + (r < nr ? r : 0)) * a.H + h) * 512 + d0);
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll
    for (int c = 0; c < AB_M / 32; ++c) {
      float v[32];
      tmem_ld32(tmem + lane_addr + 32 * c, v);
      tmem_wait_ld();
      if (r < nr) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[4 * c + q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]),
                                      pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                      pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                                      pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) { tc_fence_after(); tmem_dealloc(tmem, AB_NR); }
  // Launched beside the attention plan: this grid completes only after the
  // plan has, so the attention kernel's wait on it covers both.
  grid_dep_wait();
}

// ---- A5 + A6, small batches: the whole W_UV[h] in shared memory ------------------------
// UP_NR query rows (b, i) per CTA: 16, 32 or 64, the smallest whose grid
// (heads x row blocks) runs in one wave at one CTA per SM.  Shared memory: A = W_UV[h] as 8
// chunks of 128 v-rows x 64 d; B = merged o_lat rows (bf16) as 8 chunks of
// UP_NR rows x 64 d; per-row split weights; barriers.
constexpr int UP_MAX_SPLITS = 64;
constexpr int UP_OFF_B = 8 * 128 * 128;
__host__ __device__ constexpr int up_off_w(int nr) { return UP_OFF_B + 8 * nr * 128; }
__host__ __device__ constexpr int up_off_pr(int nr) { return up_off_w(nr) + nr * UP_MAX_SPLITS * 4; }
__host__ __device__ constexpr int up1_off_bar(int nr) { return up_off_pr(nr) + nr * 16 + 16; }
__host__ __device__ constexpr int up1_smem(int nr) { return up1_off_bar(nr) + 64 + 1024; }
__host__ __device__ constexpr int up_tmem_cols(int nr) { return nr < 32 ? 32 : nr; }

constexpr int UP_THREADS = 256;   // all warps merge partials
constexpr int UP_BATCH = 4;       // row/8-column units merged per thread per pass

template <int UP_NR>
__global__ void __launch_bounds__(UP_THREADS, 1)
combine_uproj_small_kernel(const __grid_constant__ CUtensorMap tm_w, const Args a) {
  constexpr int UP_OFF_W = up_off_w(UP_NR), UP_OFF_PR = up_off_pr(UP_NR), UP_OFF_BAR = up1_off_bar(UP_NR);
  constexpr int kCols = up_tmem_cols(UP_NR);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int r0 = blockIdx.y * UP_NR;
  const int BNr = a.B * a.N;
  const int nr = min(UP_NR, BNr - r0);
  float* wts = reinterpret_cast<float*>(sm + UP_OFF_W);
  // per row: partial row index of its partial s = pr_base[r] + s * pr_step[r]
  long long* pr_base = reinterpret_cast<long long*>(sm + UP_OFF_PR);
  int* pr_step = reinterpret_cast<int*>(sm + UP_OFF_PR + UP_NR * 8);
  int* s_max = reinterpret_cast<int*>(sm + UP_OFF_PR + UP_NR * 12);
  const uint32_t bar_full = sbase + UP_OFF_BAR, bar_mma = bar_full + 8;
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(sm + UP_OFF_BAR + 16);

  if (tid == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) { tmem_alloc(sbase + UP_OFF_BAR + 16, kCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == 0) {   // W_UV[h]: 128 v-rows x 512 d, eight 64-column chunks
    mbar_expect_tx(bar_full, 8 * 128 * 128);
    for (int k = 0; k < 8; ++k)
      tma_load_2d(sbase + k * 128 * 128, &tm_w, bar_full, 64 * k, h * 128);
  }

  grid_dep_wait();   // the split partials are written by the attention kernel

  // Partial weights per row, with 1 / sum_s e^{m_s - m*} l_s folded in.  The
  // UP_THREADS / UP_NR threads of a row (adjacent lanes) take every
  // (UP_THREADS / UP_NR)-th partial and meet by shuffles, so the (m, l) loads
  // of a row are in flight together.
  constexpr int kTpr = UP_THREADS / UP_NR;
  static_assert(kTpr >= 2 && kTpr <= 32 && (kTpr & (kTpr - 1)) == 0, "threads per row");
  if (tid == 0) *s_max = 0;
  for (int i = tid; i < UP_NR * UP_MAX_SPLITS; i += UP_THREADS) wts[i] = 0.f;
  __syncthreads();
  {
    const int r = tid / kTpr, sub = tid % kTpr;
    const bool live = r < nr;
    const PartialRef pr = partials_of_row(a, (long long)(r0 + (live ? r : 0)) * a.H + h);
    const int S = live ? (pr.count < UP_MAX_SPLITS ? pr.count : UP_MAX_SPLITS) : 0;
    if (sub == 0) {
      pr_base[r] = live ? pr.base : 0;
      pr_step[r] = live ? (int)pr.step : 0;
    }
    constexpr int kPer = UP_MAX_SPLITS / kTpr;        // partials per thread at most
    float2 ml[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int s = sub + k * kTpr;
      ml[k] = s < S ? *reinterpret_cast<const float2*>(a.part_ml + (pr.base + (long long)s * pr.step) * 2)
                    : make_float2(-INFINITY, 0.f);
    }
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (ml[k].y > 0.f) m = fmaxf(m, ml[k].x);
#pragma unroll
    for (int o = 1; o < kTpr; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const float e = ml[k].y > 0.f ? expf(ml[k].x - m) : 0.f;
      ml[k].x = e;
      l += e * ml[k].y;
    }
#pragma unroll
    for (int o = 1; o < kTpr; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    const float inv = l > 0.f ? a.o_scale / l : 0.f;
    float* w = wts + r * UP_MAX_SPLITS;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int s = sub + k * kTpr;
      if (s < S) w[s] = ml[k].x * inv;
    }
    if (live && sub == 0) atomicMax(s_max, S);
  }
  __syncthreads();
  const int S = *s_max;

  // o_lat rows -> bf16, 128-byte swizzled K-major operand: row r, 8-column unit u.
  // Each pass merges UP_BATCH units per thread; the bf16 partials of up to four
  // pieces are loaded per step, 4 x UP_BATCH x 16 bytes in flight per thread.
  for (int base = tid; base < UP_NR * 64; base += UP_THREADS * UP_BATCH) {
    float acc[UP_BATCH][8];
#pragma unroll
    for (int uu = 0; uu < UP_BATCH; ++uu)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[uu][e] = 0.f;
    for (int s0 = 0; s0 < S; s0 += 4) {
      uint4 x[4][UP_BATCH];
      float ws[4][UP_BATCH];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int s = s0 + q;
#pragma unroll
        for (int uu = 0; uu < UP_BATCH; ++uu) {
          const int idx = base + uu * UP_THREADS;
          const int r = idx >> 6, u = idx & 63;
          ws[q][uu] = (s < S && idx < UP_NR * 64 && r < nr) ? wts[r * UP_MAX_SPLITS + s] : 0.f;
          x[q][uu] = ws[q][uu] != 0.f
                         ? *reinterpret_cast<const uint4*>(
                               a.part_o16 + (pr_base[r] + (long long)s * pr_step[r]) * 512 + 8 * u)
                         : make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int uu = 0; uu < UP_BATCH; ++uu) {
          const float w = ws[q][uu];
          const uint32_t wv[4] = {x[q][uu].x, x[q][uu].y, x[q][uu].z, x[q][uu].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[uu][2 * j] = fmaf(w, __uint_as_float(wv[j] << 16), acc[uu][2 * j]);
            acc[uu][2 * j + 1] = fmaf(w, __uint_as_float(wv[j] & 0xffff0000u), acc[uu][2 * j + 1]);
          }
        }
    }
#pragma unroll
    for (int uu = 0; uu < UP_BATCH; ++uu) {
      const int idx = base + uu * UP_THREADS;
      if (idx >= UP_NR * 64) continue;
      const int r = idx >> 6, u = idx & 63;
      uint32_t pk[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) pk[j] = pack_bf16x2(acc[uu][2 * j], acc[uu][2 * j + 1]);
      const uint32_t addr = sbase + UP_OFF_B + (u >> 3) * UP_NR * 128 + r * 128 +
                            (((u & 7) ^ (r & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                   :: "r"(addr), "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]) : "memory");
    }
  }
  fence_async_smem();
  __syncthreads();

  bool ok = true;
  if (tid == 0) {
    ok = wait(bar_full, 0, a.status, kLimitNs, 111);
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, UP_NR, 0, 0);
      for (int kk = 0; kk < 32; ++kk) {
        uint64_t ad = smem_desc(sbase + (kk >> 2) * 128 * 128 + (kk & 3) * 32, 16, 1024);
        uint64_t bd = smem_desc(sbase + UP_OFF_B + (kk >> 2) * UP_NR * 128 + (kk & 3) * 32, 16, 1024);
        mma_bf16(tmem, ad, bd, idesc, kk > 0);
      }
    }
    mma_commit(bar_mma);
  }
  __syncwarp();
  ok = wait(bar_mma, 0, a.status, kLimitNs, 112) && ok;
  ok = __all_sync(0xffffffffu, ok);
  tc_fence_after();
  if (ok && warp < 4) {
    const int v = warp * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    for (int c0 = 0; c0 < UP_NR; c0 += 32) {
      float x[32];
      tmem_ld32(tmem + lane_addr + c0, x);   // columns past UP_NR (< kCols) are ignored
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int r = c0 + j;
        if (r < nr) a.out[((long long)(r0 + r) * a.H + h) * 128 + v] = x[j];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) { tc_fence_after(); tmem_dealloc(tmem, kCols); }
}

// ---- A5 + A6, large batches: W_UV[h] and o_lat streamed in K-chunks ---------------------
// CTA (h, row block) computes out[r, h, :] for NR query rows r = (b, i) of
// head h:  D[128 v x NR] (TMEM, fp32) = W_UV[h] (A: 128 v x 512 d, K-major)
// . o_lat^T (B: NR rows x 512 d, K-major, bf16), over eight K-chunks of 64
// latent columns.  Each chunk passes through one of kUpStages shared-memory
// stages: TMA brings the chunk of W_UV[h] (16 KiB), all 256 threads merge
// the rows' partials of those 64 columns (log-sum-exp weights) into the bf16
// B tile, and one thread issues the chunk's four MMAs.  While the tensor core
// runs chunk k the threads merge chunk k+1, and only 3 x (16 KiB + NR x
// 128 B) of shared memory is held, so several CTAs share an SM and NR can
// grow to 256 rows (one wave for large batches).
constexpr int kUpStages = 3;
constexpr int kUpChunks = 8;                  // 512 latent columns / 64
constexpr int kUpABytes = 128 * 128;          // W_UV chunk: 128 v-rows x 64 d bf16
__host__ __device__ constexpr int up_stage_bytes(int nr) { return kUpABytes + nr * 128; }
__host__ __device__ constexpr int up_off_bar(int nr) { return kUpStages * up_stage_bytes(nr); }
__host__ __device__ constexpr int up_smem(int nr) { return up_off_bar(nr) + 128 + 1024; }

template <int NR>
__global__ void __launch_bounds__(UP_THREADS, 2)
combine_uproj_pipe_kernel(const __grid_constant__ CUtensorMap tm_w, const Args a) {
  static_assert(NR >= 32 && NR <= 256 && (NR & (NR - 1)) == 0, "rows per CTA");
  constexpr int kTpr = UP_THREADS / NR;        // threads per row (1 .. 8)
  constexpr int kUnits = 8 / kTpr;             // 16-byte units (8 columns) of a chunk per thread
  constexpr int kPB = kUnits >= 2 ? 16 / kUnits : 8;   // pieces whose loads are in flight together
  constexpr uint32_t kStage = up_stage_bytes(NR);
  constexpr int kCols = up_tmem_cols(NR);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int r0 = blockIdx.y * NR;
  const int BNr = a.B * a.N;
  const int nr = min(NR, BNr - r0);
  auto A_FULL = [&](int s) -> uint32_t { return sbase + up_off_bar(NR) + 8u * s; };
  auto EMPTY = [&](int s) -> uint32_t { return sbase + up_off_bar(NR) + 8u * (kUpStages + s); };
  const uint32_t bar_done = sbase + up_off_bar(NR) + 8u * (2 * kUpStages);
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(sm + up_off_bar(NR) + 64);

  if (tid == 0) {
    for (int s = 0; s < kUpStages; ++s) {
      mbar_init(A_FULL(s), 1);
      mbar_init(EMPTY(s), 1);
    }
    mbar_init(bar_done, 1);
    fence_mbar_init();
  }
  if (warp == 0) { tmem_alloc(sbase + up_off_bar(NR) + 64, kCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == 0)   // the first chunks of W_UV[h] do not depend on the attention kernel
    for (int k = 0; k < kUpStages; ++k) {
      mbar_expect_tx(A_FULL(k), kUpABytes);
      tma_load_2d(sbase + k * kStage, &tm_w, A_FULL(k), 64 * k, h * 128);
    }

  grid_dep_wait();   // the split partials are written by the attention kernel

  // This thread's row and its partials: m* over the pieces that saw a key, and
  // o_scale / l* folded into the weights.
  const int r = tid / kTpr, sub = tid % kTpr;
  const bool live = r < nr;
  const PartialRef pr = partials_of_row(a, (long long)(r0 + (live ? r : 0)) * a.H + h);
  const int S = live ? pr.count : 0;
  float m = -INFINITY, l = 0.f;
  for (int s = 0; s < S; ++s) {
    const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + (pr.base + (long long)s * pr.step) * 2);
    if (ml.y > 0.f) m = fmaxf(m, ml.x);
  }
  for (int s = 0; s < S; ++s) {
    const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + (pr.base + (long long)s * pr.step) * 2);
    if (ml.y > 0.f) l += expf(ml.x - m) * ml.y;
  }
  const float inv = l > 0.f ? a.o_scale / l : 0.f;

  bool ok = true;
  for (int kc = 0; kc < kUpChunks; ++kc) {
    const int stg = kc % kUpStages;
    const uint32_t st_a = sbase + stg * kStage, st_b = st_a + kUpABytes;
    if (kc >= kUpStages) {
      // the MMAs of chunk kc - kUpStages have read this stage
      ok = wait(EMPTY(stg), ((kc / kUpStages) - 1) & 1, a.status, kLimitNs, 113) && ok;
      if (tid == 0) {
        mbar_expect_tx(A_FULL(stg), kUpABytes);
        tma_load_2d(st_a, &tm_w, A_FULL(stg), 64 * kc, h * 128);
      }
    }
    // Merge columns 64 kc + 8 u .. + 7 of row r for this thread's units u.
    float acc[kUnits][8];
#pragma unroll
    for (int uu = 0; uu < kUnits; ++uu)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[uu][e] = 0.f;
    for (int s0 = 0; s0 < S; s0 += kPB) {
      uint4 x[kPB][kUnits];
      float w[kPB];
#pragma unroll
      for (int q = 0; q < kPB; ++q) {
        const int s = s0 + q;
        w[q] = 0.f;
        if (s < S) {
          const long long prow = pr.base + (long long)s * pr.step;
          const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + prow * 2);
          w[q] = ml.y > 0.f ? expf(ml.x - m) * inv : 0.f;
        }
#pragma unroll
        for (int uu = 0; uu < kUnits; ++uu)
          x[q][uu] = w[q] != 0.f
                         ? *reinterpret_cast<const uint4*>(
                               a.part_o16 + (pr.base + (long long)(s0 + q) * pr.step) * 512 + 64 * kc +
                               8 * (sub * kUnits + uu))
                         : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int q = 0; q < kPB; ++q)
#pragma unroll
        for (int uu = 0; uu < kUnits; ++uu) {
          const uint32_t wv[4] = {x[q][uu].x, x[q][uu].y, x[q][uu].z, x[q][uu].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[uu][2 * j] = fmaf(w[q], __uint_as_float(wv[j] << 16), acc[uu][2 * j]);
            acc[uu][2 * j + 1] = fmaf(w[q], __uint_as_float(wv[j] & 0xffff0000u), acc[uu][2 * j + 1]);
          }
        }
    }
    // bf16 B tile, 128-byte swizzled K-major: row r, 16-byte unit u at (u ^ (r & 7))
#pragma unroll
    for (int uu = 0; uu < kUnits; ++uu) {
      const int u = sub * kUnits + uu;
      uint32_t pk[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) pk[j] = pack_bf16x2(acc[uu][2 * j], acc[uu][2 * j + 1]);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                   :: "r"(st_b + r * 128 + (((u & 7) ^ (r & 7)) << 4)), "r"(pk[0]), "r"(pk[1]),
                      "r"(pk[2]), "r"(pk[3]) : "memory");
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      ok = wait(A_FULL(stg), (kc / kUpStages) & 1, a.status, kLimitNs, 111) && ok;
      if (ok) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16(128, NR, 0, 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tmem, smem_desc(st_a + kk * 32, 16, 1024), smem_desc(st_b + kk * 32, 16, 1024),
                   idesc, (kc > 0 || kk > 0));
      }
      mma_commit(EMPTY(stg));
    }
  }
  if (tid == 0) mma_commit(bar_done);
  __syncwarp();
  ok = wait(bar_done, 0, a.status, kLimitNs, 112) && ok;
  ok = __all_sync(0xffffffffu, ok);
  tc_fence_after();
  // TMEM lane = v (quadrant warp & 3), column = row: warps 0-3 take the first
  // half of the rows, warps 4-7 the second (all rows when NR == 32).
  constexpr int kHalfCols = NR >= 64 ? NR / 2 : NR;
  const int c_beg = (warp >> 2) * kHalfCols;
  if (ok && c_beg < NR) {
    const int v = (warp & 3) * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    for (int c0 = c_beg; c0 < c_beg + kHalfCols; c0 += 32) {
      float x[32];
      tmem_ld32(tmem + lane_addr + c0, x);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int rr = c0 + j;
        if (rr < nr) a.out[((long long)(r0 + rr) * a.H + h) * 128 + v] = x[j];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) { tc_fence_after(); tmem_dealloc(tmem, kCols); }
}

}  // namespace

bool absorb_tc_ok(const Args& a) {
  return a.dtype == KDTV_BF16 && a.d_c == 512 && a.d_nope % 64 == 0 && a.d_nope <= 256;
}

bool combine_uproj_tc_ok(const Args& a) {
  // reads the bf16 partials of a stream-K plan
  return a.dtype == KDTV_BF16 && a.d_c == 512 && a.d_v == 128 && a.sk != nullptr;
}

cudaError_t launch_absorb_tc(const Args& a, cudaStream_t st, bool after_plan) {
  if (!absorb_tc_ok(a)) return launch_absorb(a, st, /*bf16_out=*/true);
  CUtensorMap tw, tq;
  const uint64_t BNr = (uint64_t)a.B * a.N;
  if (encode_2d(&tw, a.W_UK, (uint64_t)a.H * a.d_nope, 512, 64, a.d_nope) != CUDA_SUCCESS ||
      encode_2d(&tq, a.q_nope, BNr, (uint64_t)a.H * a.d_nope, 64, AB_NR) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int smem = ab_smem(a.d_nope);
  cudaError_t e = cudaFuncSetAttribute(absorb_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(512 / AB_M, a.H, (unsigned)((BNr + AB_NR - 1) / AB_NR));
  return launch_ex(absorb_tc_kernel, grid, dim3(kThreads), smem, st, after_plan, tw, tq, a);
}

namespace {
template <int NR>
cudaError_t launch_combine_small(const CUtensorMap& tw, const Args& a, cudaStream_t st, bool pdl) {
  cudaError_t e = cudaFuncSetAttribute(combine_uproj_small_kernel<NR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, up1_smem(NR));
  if (e != cudaSuccess) return e;
  const unsigned nblk = (unsigned)(((long long)a.B * a.N + NR - 1) / NR);
  return launch_ex(combine_uproj_small_kernel<NR>, dim3(a.H, nblk), dim3(UP_THREADS), up1_smem(NR),
                   st, pdl, tw, a);
}

template <int NR>
cudaError_t launch_combine_pipe(const CUtensorMap& tw, const Args& a, cudaStream_t st, bool pdl) {
  cudaError_t e = cudaFuncSetAttribute(combine_uproj_pipe_kernel<NR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, up_smem(NR));
  if (e != cudaSuccess) return e;
  const unsigned nblk = (unsigned)(((long long)a.B * a.N + NR - 1) / NR);
  return launch_ex(combine_uproj_pipe_kernel<NR>, dim3(a.H, nblk), dim3(UP_THREADS), up_smem(NR),
                   st, pdl, tw, a);
}
}  // namespace

// Which combine + up-projection kernel, and its rows per CTA.  Small batches
// (the grid fits one wave at one CTA per SM with 16, 32 or 64 rows): the
// kernel that holds all of W_UV[h] and merges every column of its rows in one
// pass, with many loads in flight.  Larger ones: the K-chunk pipeline, two
// CTAs per SM with 64 or 128 rows, or one with 256.  Returns rows per CTA,
// negative for the small-batch kernel.
int combine_uproj_choice(const Args& a, int sms) {
  const long long bn = (long long)a.B * a.N;
  for (int nr = 16; nr <= 64; nr <<= 1)
    if ((long long)a.H * ((bn + nr - 1) / nr) <= sms) return -nr;
  for (int nr = 64; nr <= 128; nr <<= 1)
    if ((long long)a.H * ((bn + nr - 1) / nr) <= 2ll * sms) return nr;
  return 256;
}

cudaError_t launch_combine_uproj_tc(const Args& a, const Plan& p, cudaStream_t st,
                                    cudaEvent_t* ev) {
  if (!combine_uproj_tc_ok(a)) return launch_combine_uproj(a, p, st, ev);
  CUtensorMap tw;
  if (encode_2d(&tw, a.W_UV, (uint64_t)a.H * 128, 512, 64, 128) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (ev) cudaEventRecord(ev[3], st);   // the combine is fused into the up-projection
  // Overlap with the attention kernel's tail unless phase events split the call.
  const bool pdl = ev == nullptr;
  const int c = combine_uproj_choice(a, p.sms);
  cudaError_t e = c == -16 ? launch_combine_small<16>(tw, a, st, pdl)
                : c == -32 ? launch_combine_small<32>(tw, a, st, pdl)
                : c == -64 ? launch_combine_small<64>(tw, a, st, pdl)
                : c == 64  ? launch_combine_pipe<64>(tw, a, st, pdl)
                : c == 128 ? launch_combine_pipe<128>(tw, a, st, pdl)
                           : launch_combine_pipe<256>(tw, a, st, pdl);
  if (ev) cudaEventRecord(ev[4], st);
  return e;
}

}  // namespace kdtv
