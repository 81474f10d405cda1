// Tensor-core (tcgen05) kernels for the two per-head projections around the
// attention, the absorbed form's w_kc / w_vc halves ("The Moment of Proof:
// Validating a Native CUDA Speculative Decoding Engine", section "Input
// Knowledge Required"):
//
//   absorb_tc_kernel         q_lat[r, h, :] = W_UK[h]^T q_nope[r, h, :]   (bf16 out)
//   combine_uproj_tc_kernel  o_lat = log-sum-exp merge of the split partials,
//                            out[r, h, :] = W_UV[h] o_lat                 (fp32 out)
//
// The absorb takes the query rows as the 128-row MMA operand and the W_UK
// block, loaded by TMA, as the MN-major N operand: D[128 rows x 128 d], read
// back lane-per-row, rounded to bf16 in shared memory and stored by TMA.  The
// combine runs transposed, so that W_UV[h] is the 128-row operand and the
// query rows are the MMA N dimension: D[128 v x rows] = W_UV[h] . o_lat^T,
// read back lane-per-output-feature, which makes its fp32 global writes
// coalesced.

#include <cuda.h>

#include "kdtv_internal.cuh"
#include "kdtv_ptx.cuh"
#include "kdtv_tmap.cuh"

namespace kdtv {
namespace {

using namespace ptx;

constexpr uint64_t kLimitNs = 2000000000ull;

// ---- A1: absorb -----------------------------------------------------------------------
// CTA (latent block, head h, row-block group z) computes the 128 x 128 tiles
// q_lat[rows of block rb, h, d0 .. d0+127] for rb = z, z + G, z + 2G, ...: the
// W_UK block is loaded once and the query blocks stream through two stages.
// Per tile, one MMA chain D[128 rows x 128 d] (TMEM, two buffers) = q_nope
// rows (A, K-major) . W_UK block (B, MN-major).  The epilogue warps round D
// to bf16 into the stage the MMAs have just read (128-byte swizzled, the
// output tensor map's layout) and one thread stores it with TMA, which writes
// whole lines; the stage is then refilled with the tile two ahead.
constexpr int AB_M = 128;                  // latent columns per tile
constexpr int AB_NR = 128;                 // query rows (b, i) per tile
constexpr int AB_THREADS = 160;            // warps 0-3: epilogue (TMEM lane quadrants); 4: TMA + MMA
constexpr int AB_STAGE_OUT = 2 * AB_NR * 128;   // a bf16 output tile as two 64-column boxes

// Shared memory of absorb_tc_kernel for a given d_nope: the W_UK block (two
// MN atoms of d_nope e-rows x 128 B), two stages each holding a query block
// (d_nope/64 chunks of AB_NR rows x 128 B) or an output tile, barriers.
__host__ __device__ constexpr int ab_stage(int d_nope) {
  return (d_nope / 64) * AB_NR * 128 > AB_STAGE_OUT ? (d_nope / 64) * AB_NR * 128 : AB_STAGE_OUT;
}
__host__ __device__ constexpr int ab_off_q(int d_nope) { return 2 * d_nope * 128; }
__host__ __device__ constexpr int ab_off_bar(int d_nope) { return ab_off_q(d_nope) + 2 * ab_stage(d_nope); }
__host__ __device__ constexpr int ab_smem(int d_nope) { return ab_off_bar(d_nope) + 64 + 1024; }

__global__ void __launch_bounds__(AB_THREADS, 1)
absorb_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_o, const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d0 = blockIdx.x * AB_M;
  const int h = blockIdx.y;
  const int z = blockIdx.z, G = gridDim.z;
  const int RB = (a.B * a.N + AB_NR - 1) / AB_NR;
  const int nk = (RB - z + G - 1) / G;       // this CTA's tiles (z < RB)
  const int kch = a.d_nope / 64;             // 64-wide K chunks
  const int stage = ab_stage(a.d_nope), off_q = ab_off_q(a.d_nope), off_bar = ab_off_bar(a.d_nope);
  // barriers: W landed; [2] query stage landed; [2] MMA chain done; [2] output tile stored
  const uint32_t bar_w = sbase + off_bar;
  auto BAR_Q = [&](int s) -> uint32_t { return bar_w + 8u * (1 + s); };
  auto BAR_MMA = [&](int s) -> uint32_t { return bar_w + 8u * (3 + s); };
  auto BAR_OUT = [&](int s) -> uint32_t { return bar_w + 8u * (5 + s); };
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(sm + off_bar + 56);
  grid_dep_launch();   // the attention kernel may start its prologue early

  if (tid == 0) {
    for (int b = 0; b < 7; ++b) mbar_init(bar_w + 8u * b, 1);
    fence_mbar_init();
  }
  if (warp == 4) { tmem_alloc(sbase + off_bar + 56, 2 * AB_M); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 4) {
    if (lane == 0) {
      const uint32_t q_bytes = (uint32_t)kch * AB_NR * 128u;
      auto load_q = [&](int k) {   // query block of tile k -> stage k & 1
        const int s = k & 1;
        mbar_expect_tx(BAR_Q(s), q_bytes);
        for (int c = 0; c < kch; ++c)   // q_nope rows of head h, e in [64c, 64c+64)
          tma_load_2d(sbase + off_q + s * stage + c * AB_NR * 128, &tm_q, BAR_Q(s),
                      h * a.d_nope + 64 * c, (z + k * G) * AB_NR);
      };
      mbar_expect_tx(bar_w, 2u * a.d_nope * 128u);
      for (int c = 0; c < 2; ++c)       // W_UK[h][:, d0 + 64c : +64]: e-rows x 64 d
        tma_load_2d(sbase + c * a.d_nope * 128, &tm_w, bar_w, d0 + 64 * c, h * a.d_nope);
      load_q(0);
      if (nk > 1) load_q(1);
      for (int k = 2; k < nk; ++k)      // later query blocks: into L2 now
        for (int c = 0; c < kch; ++c)
          tma_prefetch_2d(&tm_q, h * a.d_nope + 64 * c, (z + k * G) * AB_NR);
      // D[128 rows x 128 d] = q_nope rows (A, K-major) x W_UK block (B, MN-major);
      // rows past the last query row are zero-filled by TMA and never stored.
      const uint32_t idesc = idesc_bf16(AB_NR, AB_M, /*a_mn=*/0, /*b_mn=*/1);
      bool ok = wait(bar_w, 0, a.status, kLimitNs, 101);
      for (int k = 0; ok && k < nk; ++k) {
        const int s = k & 1;
        // stage s was refilled (and TMEM buffer s released) after tile k-2's store
        if (!wait(BAR_Q(s), (k >> 1) & 1, a.status, kLimitNs, 102)) break;
        tc_fence_after();
        const uint32_t qs = sbase + off_q + s * stage;
        for (int kk = 0; kk < a.d_nope / 16; ++kk) {
          uint64_t ad = smem_desc(qs + (kk >> 2) * AB_NR * 128 + (kk & 3) * 32, 16, 1024);
          // B (MN-major): 64-column atoms a.d_nope*128 B apart, 8 e-rows per 1 KiB.
          uint64_t bd = smem_desc(sbase + kk * 16 * 128, a.d_nope * 128, 1024);
          mma_bf16(tmem + AB_M * s, ad, bd, idesc, kk > 0);
        }
        mma_commit(BAR_MMA(s));
        if (k + 2 < nk) {
          ok = wait(BAR_OUT(s), (k >> 1) & 1, a.status, kLimitNs, 103);
          if (ok) load_q(k + 2);
        }
      }
    }
    __syncwarp();
  } else {
    // TMEM lane = the tile's row warp*32 + lane: its 128 latent columns go to
    // row r of the two 64-column boxes, 16-byte chunk j at (j ^ (r & 7)) * 16.
    const int r = warp * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    for (int k = 0; k < nk; ++k) {
      const int s = k & 1;
      // the four warps agree on going on (named barrier 1 with an AND), so none
      // is left waiting at the barrier below after another gave up
      const uint32_t got = wait(BAR_MMA(s), (k >> 1) & 1, a.status, kLimitNs, 104) ? 1u : 0u;
      uint32_t all;
      asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                   "barrier.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                   : "=r"(all) : "r"(got) : "memory");
      if (!all) break;
      tc_fence_after();
      const uint32_t os = sbase + off_q + s * stage;
#pragma unroll
      for (int c = 0; c < AB_M / 32; ++c) {
        float v[32];
        tmem_ld32(tmem + lane_addr + AB_M * s + 32 * c, v);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int J = 4 * c + q;       // 16-byte chunk of the row's 256 bytes
          const uint32_t dst = os + (J >> 3) * AB_NR * 128 + r * 128 + ((J & 7) ^ (r & 7)) * 16;
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                       :: "r"(dst), "r"(pack_bf16x2(v[8 * q], v[8 * q + 1])),
                          "r"(pack_bf16x2(v[8 * q + 2], v[8 * q + 3])),
                          "r"(pack_bf16x2(v[8 * q + 4], v[8 * q + 5])),
                          "r"(pack_bf16x2(v[8 * q + 6], v[8 * q + 7])) : "memory");
        }
      }
      fence_async_smem();   // the tile's generic writes -> the TMA store's reads
      tc_fence_before();
      asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
      if (tid == 0) {
        const int x = h * 512 + d0, y = (z + k * G) * AB_NR;
        tma_store_2d(&tm_o, os, x, y);
        tma_store_2d(&tm_o, os + AB_NR * 128, x + 64, y);
        bulk_commit();
        bulk_wait_read_all();   // stage s and TMEM buffer s may be reused
        mbar_arrive(BAR_OUT(s));
      }
      __syncwarp();
    }
    if (tid == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) { tc_fence_after(); tmem_dealloc(tmem, 2 * AB_M); }
  // Launched beside the attention plan: this grid completes only after the
  // plan has, so the attention kernel's wait on it covers both.
  grid_dep_wait();
}

// ---- A5 + A6: split combine fused with the W_UV up-projection ---------------------------
// CTA (h, row block) computes out[r, h, :] for NR query rows r = (b, i) of
// head h:  D[128 v x NR] (TMEM, fp32) = W_UV[h] (A: 128 v x 512 d, K-major)
// . o_lat^T (B: NR rows x 512 d, K-major, bf16), over eight K-chunks of 64
// latent columns; o_lat is the log-sum-exp merge of the row's piece
// partials.  The merge is latency-bound (the partials come from L2 or DRAM),
// so it runs in as few passes of loads as registers allow: each pass merges
// CG chunks of kPB pieces at once, and the first pass's loads are in flight
// while the rows' (m, l) are read.  W_UV[h] sits in kAS shared-memory
// stages: all eight chunks when the grid fits one CTA per SM, else a ring of
// four, refilled from L2 (prefetched at the start) as the MMAs free them.
constexpr int UP_THREADS = 256;    // all warps merge partials
constexpr int kUpChunks = 8;       // 512 latent columns / 64
constexpr int kUpABytes = 128 * 128;   // W_UV chunk: 128 v-rows x 64 d bf16
__host__ __device__ constexpr int up_tpr(int nr) { return UP_THREADS / nr; }      // threads per row
__host__ __device__ constexpr int up_units(int nr) { return 8 / up_tpr(nr); }     // 16-byte units per chunk
__host__ __device__ constexpr int up_cg(int nr) {                                 // chunks per pass
  return up_units(nr) <= 2 ? 4 : up_units(nr) == 4 ? 2 : 1;
}
__host__ __device__ constexpr int up_pb(int nr) { return up_cg(nr) * up_units(nr) <= 4 ? 4 : 1; }
__host__ __device__ constexpr int up_off_b(int as) { return as * kUpABytes; }
__host__ __device__ constexpr int up_off_bar(int nr, int as) { return up_off_b(as) + up_cg(nr) * nr * 128; }
__host__ __device__ constexpr int up_smem(int nr, int as) { return up_off_bar(nr, as) + 8 * 20 + 16 + 1024; }
__host__ __device__ constexpr int up_tmem_cols(int nr) { return nr < 32 ? 32 : nr; }

template <int NR, int kAS>
__global__ void __launch_bounds__(UP_THREADS, kAS == kUpChunks ? 1 : 2)
combine_uproj_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const Args a) {
  static_assert(NR >= 32 && NR <= 256 && (NR & (NR - 1)) == 0, "rows per CTA");
  static_assert(kAS == kUpChunks || kAS == 4, "W_UV stages");
  constexpr int kTpr = up_tpr(NR), kUnits = up_units(NR), CG = up_cg(NR), kPB = up_pb(NR);
  constexpr int kPasses = kUpChunks / CG;
  static_assert(kAS >= CG, "a pass's W_UV chunks are resident together");
  constexpr int kCols = up_tmem_cols(NR);
  constexpr int kOffB = up_off_b(kAS), kOffBar = up_off_bar(NR, kAS);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int r0 = blockIdx.y * NR;
  const int BNr = a.B * a.N;
  const int nr = min(NR, BNr - r0);
  auto A_FULL = [&](int s) -> uint32_t { return sbase + kOffBar + 8u * s; };
  auto A_EMPTY = [&](int s) -> uint32_t { return sbase + kOffBar + 8u * (kAS + s); };
  const uint32_t bar_b = sbase + kOffBar + 8u * (2 * kAS);      // a pass's MMAs read the B slots
  const uint32_t bar_done = bar_b + 8u;
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(sm + kOffBar + 8 * 20);

  if (tid == 0) {
    for (int s = 0; s < kAS; ++s) {
      mbar_init(A_FULL(s), 1);
      mbar_init(A_EMPTY(s), 1);
    }
    mbar_init(bar_b, 1);
    mbar_init(bar_done, 1);
    fence_mbar_init();
  }
  if (warp == 0) { tmem_alloc(sbase + kOffBar + 8 * 20, kCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == 0) {   // W_UV[h] does not depend on the attention kernel
    for (int k = 0; k < kAS; ++k) {
      mbar_expect_tx(A_FULL(k), kUpABytes);
      tma_load_2d(sbase + k * kUpABytes, &tm_w, A_FULL(k), 64 * k, h * 128);
    }
    for (int k = kAS; k < kUpChunks; ++k) tma_prefetch_2d(&tm_w, 64 * k, h * 128);
  }

  grid_dep_wait();   // the split partials are written by the attention kernel

  const int r = tid / kTpr, sub = tid % kTpr;
  const bool live = r < nr;
  const PartialRef pr = partials_of_row(a, (long long)(r0 + (live ? r : 0)) * a.H + h);
  const int S = live ? pr.count : 0;

  // A pass's loads: kPB pieces from s0, CG chunks from c0, this thread's units.
  uint4 x[kPB][CG][kUnits];
  float2 ml[kPB];
  auto load = [&](int s0, int c0) {
#pragma unroll
    for (int q = 0; q < kPB; ++q) {
      const int s = s0 + q;
      const long long prow = pr.base + (long long)s * pr.step;
      ml[q] = s < S ? *reinterpret_cast<const float2*>(a.part_ml + prow * 2) : make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int c = 0; c < CG; ++c)
#pragma unroll
        for (int uu = 0; uu < kUnits; ++uu)
          x[q][c][uu] = s < S ? *reinterpret_cast<const uint4*>(a.part_o16 + prow * 512 + 64 * (c0 + c) +
                                                                 8 * (sub * kUnits + uu))
                              : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  load(0, 0);   // in flight while the rows' (m, l) are read

  // m* over the pieces that saw a key, and o_scale / l* (one pass, l follows
  // the running max), eight loads in flight at a time
  float m = -INFINITY, l = 0.f;
  for (int t0 = 0; t0 < S; t0 += 8) {
    float2 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      v[q] = t0 + q < S ? *reinterpret_cast<const float2*>(a.part_ml + (pr.base + (long long)(t0 + q) * pr.step) * 2)
                        : make_float2(-INFINITY, 0.f);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (v[q].y > 0.f) {
        if (v[q].x > m) {
          l = m == -INFINITY ? 0.f : l * expf(m - v[q].x);
          m = v[q].x;
        }
        l += expf(v[q].x - m) * v[q].y;
      }
  }
  const float inv = l > 0.f ? a.o_scale / l : 0.f;

  bool ok = true;
  for (int g = 0; g < kPasses; ++g) {
    const int c0 = g * CG;
    float acc[CG][kUnits][8];
#pragma unroll
    for (int c = 0; c < CG; ++c)
#pragma unroll
      for (int uu = 0; uu < kUnits; ++uu)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[c][uu][e] = 0.f;
    for (int s0 = 0; s0 < S || s0 == 0; s0 += kPB) {
      if (g > 0 || s0 > 0) load(s0, c0);
#pragma unroll
      for (int q = 0; q < kPB; ++q) {
        const float w = ml[q].y > 0.f ? expf(ml[q].x - m) * inv : 0.f;   // 0 for a piece that saw no key
#pragma unroll
        for (int c = 0; c < CG; ++c)
#pragma unroll
          for (int uu = 0; uu < kUnits; ++uu) {
            const uint32_t wv[4] = {x[q][c][uu].x, x[q][c][uu].y, x[q][c][uu].z, x[q][c][uu].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              acc[c][uu][2 * j] = fmaf(w, __uint_as_float(wv[j] << 16), acc[c][uu][2 * j]);
              acc[c][uu][2 * j + 1] = fmaf(w, __uint_as_float(wv[j] & 0xffff0000u), acc[c][uu][2 * j + 1]);
            }
          }
      }
    }
    // the B slots are rewritten: the previous pass's MMAs must have read them
    if (g > 0) ok = wait(bar_b, (g - 1) & 1, a.status, kLimitNs, 114) && ok;
    // bf16 B slot c, 128-byte swizzled K-major: row r, 16-byte unit u at (u ^ (r & 7))
#pragma unroll
    for (int c = 0; c < CG; ++c)
#pragma unroll
      for (int uu = 0; uu < kUnits; ++uu) {
        const int u = sub * kUnits + uu;
        uint32_t pk[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) pk[j] = pack_bf16x2(acc[c][uu][2 * j], acc[c][uu][2 * j + 1]);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                     :: "r"(sbase + kOffB + c * NR * 128 + r * 128 + (((u & 7) ^ (r & 7)) << 4)),
                        "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]) : "memory");
      }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, NR, 0, 0);
#pragma unroll
      for (int c = 0; c < CG; ++c) {
        const int kc = c0 + c, stg = kc % kAS;
        ok = wait(A_FULL(stg), (kc / kAS) & 1, a.status, kLimitNs, 111) && ok;
        if (ok) {
          tc_fence_after();
          const uint32_t st_a = sbase + stg * kUpABytes, st_b = sbase + kOffB + c * NR * 128;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem, smem_desc(st_a + kk * 32, 16, 1024), smem_desc(st_b + kk * 32, 16, 1024),
                     idesc, (kc > 0 || kk > 0));
        }
        if (kAS < kUpChunks) mma_commit(A_EMPTY(stg));
      }
      mma_commit(bar_b);
      // refill the ring with the chunks kAS ahead once these MMAs have read it
      if (kAS < kUpChunks)
        for (int c = 0; c < CG; ++c) {
          const int kc = c0 + c, nk = kc + kAS, stg = kc % kAS;
          if (nk >= kUpChunks) continue;
          ok = wait(A_EMPTY(stg), (kc / kAS) & 1, a.status, kLimitNs, 113) && ok;
          mbar_expect_tx(A_FULL(stg), kUpABytes);
          tma_load_2d(sbase + stg * kUpABytes, &tm_w, A_FULL(stg), 64 * nk, h * 128);
        }
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
    for (int cc = c_beg; cc < c_beg + kHalfCols; cc += 32) {
      float y[32];
      tmem_ld32(tmem + lane_addr + cc, y);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int rr = cc + j;
        if (rr < nr) a.out[((long long)(r0 + rr) * a.H + h) * 128 + v] = y[j];
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
  if (reinterpret_cast<uintptr_t>(a.q_lat) & 15u) return cudaErrorMisalignedAddress;
  CUtensorMap tw, tq, to;
  const uint64_t BNr = (uint64_t)a.B * a.N;
  if (encode_2d(&tw, a.W_UK, (uint64_t)a.H * a.d_nope, 512, 64, a.d_nope) != CUDA_SUCCESS ||
      encode_2d(&tq, a.q_nope, BNr, (uint64_t)a.H * a.d_nope, 64, AB_NR) != CUDA_SUCCESS ||
      encode_2d(&to, a.q_lat, BNr, (uint64_t)a.H * 512, 64, AB_NR) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int smem = ab_smem(a.d_nope);
  cudaError_t e = cudaFuncSetAttribute(absorb_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // Row blocks per CTA: the (latent block, head) CTAs take every row block
  // unless they leave most of one wave idle; then the row blocks are split
  // into G groups.
  const int rb = (int)((BNr + AB_NR - 1) / AB_NR);
  const int sms = device_sm_count() > 0 ? device_sm_count() : 152;
  const int per_sm = 228 * 1024 / (smem + 1024);
  const long long ctas = 4ll * a.H;
  int g = (int)((long long)sms * (per_sm > 0 ? per_sm : 1) / ctas);
  g = g < 1 ? 1 : g > rb ? rb : g;
  dim3 grid(512 / AB_M, a.H, (unsigned)g);
  return launch_ex(absorb_tc_kernel, grid, dim3(AB_THREADS), smem, st, after_plan, tw, tq, to, a);
}

namespace {
template <int NR, int kAS>
cudaError_t launch_combine(const CUtensorMap& tw, const Args& a, cudaStream_t st, bool pdl) {
  constexpr int smem = up_smem(NR, kAS);
  static_assert(smem <= 227 * 1024 && (kAS == kUpChunks || 2 * smem <= 226 * 1024), "shared memory");
  cudaError_t e = cudaFuncSetAttribute(combine_uproj_tc_kernel<NR, kAS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned nblk = (unsigned)(((long long)a.B * a.N + NR - 1) / NR);
  return launch_ex(combine_uproj_tc_kernel<NR, kAS>, dim3(a.H, nblk), dim3(UP_THREADS), smem, st, pdl,
                   tw, a);
}
}  // namespace

// Rows per CTA of the combine + up-projection: the smallest of 32, 64, 128,
// 256 whose grid (heads x row blocks) runs in one wave at two CTAs per SM.
// Returns it negated when the grid also fits one CTA per SM: then all of
// W_UV[h] stays in shared memory.
int combine_uproj_choice(const Args& a, int sms) {
  const long long bn = (long long)a.B * a.N;
  int nr = 32;
  while (nr < 256 && (long long)a.H * ((bn + nr - 1) / nr) > 2ll * sms) nr <<= 1;
  return (long long)a.H * ((bn + nr - 1) / nr) <= sms ? -nr : nr;
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
  cudaError_t e = c == -32  ? launch_combine<32, kUpChunks>(tw, a, st, pdl)
                : c == -64  ? launch_combine<64, kUpChunks>(tw, a, st, pdl)
                : c == -128 ? launch_combine<128, kUpChunks>(tw, a, st, pdl)
                : c == -256 ? launch_combine<256, kUpChunks>(tw, a, st, pdl)
                : c == 32   ? launch_combine<32, 4>(tw, a, st, pdl)
                : c == 64   ? launch_combine<64, 4>(tw, a, st, pdl)
                : c == 128  ? launch_combine<128, 4>(tw, a, st, pdl)
                            : launch_combine<256, 4>(tw, a, st, pdl);
  if (ev) cudaEventRecord(ev[4], st);
  return e;
}

}  // namespace kdtv
