// Tensor-core (tcgen05) path of kdtv_verify_attn: bf16 inputs, the MLA
// latent layout d_c = 512, d_rope = 64, fp32 accumulation.
//
// The attention step (tree-masked scores, online softmax, P . c_kv) of the
// "tree-verify MLA-absorb attention kernel with visibility masking" ("The
// Moment of Proof: Validating a Native CUDA Speculative Decoding Engine",
// section "The Context: Building a Native DDTree Engine from Scratch").
//
// Work decomposition.  A work item is (request b, tile of 128 query rows,
// split-KV key range).  Query rows are (node, head) pairs with the head
// fastest, so one tile holds 128/H nodes; every row of a node shares that
// node's ancestor mask.  An item runs on a CLUSTER OF TWO CTAs that split
// the latent dimension:
//   CTA 0 holds q_lat[:, 0:256] and q_rope, and reads c_kv[:, 0:256] + k_rope;
//   CTA 1 holds q_lat[:, 256:512] and reads c_kv[:, 256:512].
// Per 64-key tile each CTA computes the partial score tile S_c = Q_c K_c^T
// (all 128 rows) on tcgen05 into TMEM and accumulates its own half of the
// latent output, O_c += P . c_kv[:, 256c : 256c+256] (all 128 rows).
//
// The softmax rows are split between the pair: CTA c owns the rows in TMEM
// lanes 32q + 16c .. 32q + 16c + 15 of each lane quadrant q.  For every tile
// a CTA sends the peer the peer's rows of its partial scores (fp16, one exact
// power-of-two scale per row), adds the peer's partial for its own rows to its
// exact fp32 partial, runs the online softmax of its own rows, and returns the
// P rows (bf16, one 2 KiB bulk copy per quadrant) so that both CTAs hold the
// full P tile for their P . V.  When a row's reference maximum moves, its
// owner also sends the rescale factor, and each CTA rescales its half of O.
//
// TMEM (512 columns per CTA): O_c [0, 256) fp32; q_lat half [256, 384) as
// bf16 pairs (the A operand of Q.K^T); two score buffers [384, 448) and
// [448, 512).  Shared memory: a 4-stage TMA ring of 64-key cache tiles
// (128-byte swizzled 64-column chunks; the same tile is the K-major B operand
// of Q.K^T and the MN-major B operand of P.V), q_rope (CTA 0), the P tile
// (K-major A operand of P.V), two receive buffers for the peer's scores and
// four for its rescale factors.  Key tiles are also prefetched into L2 a few
// tiles ahead of the ring.
//
// Warp roles (352 threads): warp 0 issues TMA loads; warp 1 owns TMEM and
// issues Q.K^T; warps 2-5 (one per lane quadrant) quantise and send the
// peer's score rows; warps 6-9 (one per quadrant, four threads per row in
// the .16x256b TMEM layout, so row maxima and sums meet by warp shuffles) run
// the softmax of the CTA's own rows; warp 10 issues P.V.  Warps 2-9 also load
// Q into TMEM and write the partial o_lat.  Every wait is bounded (2 s, or
// ~20 ms with KDTV_FLAG_TEST_STALL); on timeout the kernel records
// KDTV_ERR_DEVICE_TIMEOUT, lets in-flight copies land, drains its MMAs, frees
// TMEM and returns.

#include <cuda.h>
#include <cuda_fp16.h>

#include "kdtv_internal.cuh"
#include "kdtv_ptx.cuh"
#include "kdtv_tmap.cuh"

namespace kdtv {
namespace {

using namespace ptx;

constexpr int BM = 128;          // query rows per tile (MMA M)
constexpr int BN = 64;           // keys per tile (MMA N of Q.K^T)
constexpr int CH = 64;           // bf16 columns per 128-byte swizzled chunk
constexpr int kHalf = 256;       // latent columns per CTA
constexpr int kStages = 4;
constexpr int kPrefetch = 3;     // key tiles prefetched into L2 beyond the stages in flight
constexpr int kMaxCh = 5;        // CTA 0: 4 latent chunks + 1 rope chunk per key tile
constexpr int kKVChunk = BN * CH * 2;   // 8 KiB
constexpr int kQRopeBytes = BM * CH * 2;
constexpr int kPBytes = BM * BN * 2;    // the P tile: 128 rows x 64 keys bf16, 128B-swizzled
constexpr int kPQuadBytes = 16 * BN * 2;   // one quadrant's own P rows (contiguous, 2 KiB)
// Score exchange: the peer's 64 rows as fp16 in the receiving softmax
// thread's order: 16-byte chunk m (0..3) of thread t of quadrant q at
// ((q * 4 + m) * 32 + t) * 16, so one warp store is a contiguous 512-byte
// block; then one word per (q, t) holding its two rows' shifts.
constexpr int kRxData = 4 * 4 * 32 * 16;
constexpr int kRxBytes = kRxData + 4 * 32 * 4;
constexpr int kRxStride = (kRxBytes + 127) / 128 * 128;
constexpr int kAfBufs = 4;              // rescale-factor buffers, [BM] floats each
constexpr int kAfBytes = 64 * 4;        // the peer's 64 rows per tile
constexpr int kThreads = 480;
constexpr int kWarpPV = 14;
constexpr int kTmemCols = 512;
constexpr int kColO = 0;
constexpr int kColQ = 256;
constexpr int kColS = 384;       // + 64 * buffer

constexpr int OFF_KV = 0;
constexpr int OFF_QR = OFF_KV + kStages * kMaxCh * kKVChunk;
constexpr int OFF_P = OFF_QR + kQRopeBytes;
constexpr int OFF_RX = OFF_P + kPBytes;                        // two receive buffers
constexpr int OFF_AF = OFF_RX + 2 * kRxStride;                 // [kAfBufs][BM] floats
constexpr int OFF_ANC = OFF_AF + kAfBufs * BM * 4;
constexpr int OFF_PAR = OFF_ANC + kMaxNodes * 16;              // staged parent[]
constexpr int OFF_MREF = OFF_PAR + kMaxNodes * 4;              // [2 parities][BM] reference maxima
constexpr int OFF_LPART = OFF_MREF + 2 * BM * 4;                // [m | l][BM] of the odd-tile warps
constexpr int OFF_BAR = OFF_LPART + 2 * BM * 4;
constexpr int kNumBars = 40;
constexpr int OFF_MISC = OFF_BAR + kNumBars * 8;
constexpr int kSmemBytes = OFF_MISC + 64 + 1024;   // + slack for 1 KiB alignment
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(OFF_QR % 1024 == 0 && OFF_P % 1024 == 0, "128B-swizzled tiles need 1 KiB alignment");
static_assert(OFF_RX % 16 == 0 && kRxStride % 16 == 0 && OFF_AF % 16 == 0, "async store alignment");
static_assert(kThreads == 32 * (kWarpPV + 1), "warp roles");

// Barrier indices (derived from kStages so the groups never overlap).
enum Bar : int {
  B_QR_FULL = 0,
  B_Q_READY = 1,                     // 8 warps stored their part of Q in TMEM
  B_KV_FULL = 2,                     // [kStages]
  B_KV_EMPTY = B_KV_FULL + kStages,  // [kStages]
  B_S_FULL = B_KV_EMPTY + kStages,   // [2] Q.K^T of the tile completed
  B_S_FREE = B_S_FULL + 2,           // [2] senders and softmax read the scores
  B_RX_FULL = B_S_FREE + 2,          // [2] the peer's score rows landed (tx)
  B_TX_OK = B_RX_FULL + 2,           // [2] the peer consumed what we sent (remote)
  B_AF_FULL = B_TX_OK + 2,           // [kAfBufs] the peer's rescale factors landed (tx)
  B_P_FULL = B_AF_FULL + kAfBufs,    // our softmax wrote its P rows
  B_P_RX = B_P_FULL + 1,             // the peer's P rows landed (tx)
  B_P_EMPTY = B_P_RX + 1,            // [2] P.V of an even / odd tile completed in both CTAs
  B_O_FULL = B_P_EMPTY + 2,
  B_MMA_DONE = B_O_FULL + 1,         // both MMA issuers drained
  B_STALL = B_MMA_DONE + 1,
  B_MREF = B_STALL + 1,              // [2 parities][4 quadrants] reference maxima published
  B_LSUM = B_MREF + 8,               // the odd-tile softmax warps published their (m, l)
  B_COUNT = B_LSUM + 1
};
static_assert(B_COUNT <= kNumBars, "barrier slots");

// Wait sites (reported as the timeout detail).
enum Site { W_Q = 1, W_KV_FULL, W_KV_EMPTY, W_P_FULL, W_S_FULL, W_TX_OK, W_RX_FULL,
            W_P_EMPTY, W_O_FULL, W_STALL, W_DRAIN, W_S_FREE, W_AF, W_P_RX, W_MREF, W_LSUM };

struct TcCfg {
  int row_tiles;               // ceil(N * H / 128)
  unsigned long long limit_ns; // bound on every wait
};

// 2^e as a float for e in [-126, 127] (exact).
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// Shift that maps max |v| into [2^14, 2^15): the fp16 range with headroom.
// Capped at 100 so that every nonzero fp16 value times 2^-shift is a normal
// float.
__device__ __forceinline__ int fp16_shift(float amax) {
  if (!(amax > 0.f)) return 0;
  const int e = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127;   // floor(log2(amax))
  const int sh = 14 - e;
  return sh < -126 ? -126 : (sh > 100 ? 100 : sh);
}

// Three-input maximum (one instruction on sm_100-class GPUs).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Scale 16 O rows (a .16x256b warp slice: rows base + t/4 and base + t/4 + 8)
// of this CTA's 256 O columns by alpha_a / alpha_b.
__device__ __forceinline__ void rescale_o_rows(uint32_t taddr, float alpha_a, float alpha_b) {
#pragma unroll 1
  for (int cc = 0; cc < kHalf / 64; ++cc) {
    uint32_t ov[32];
    tmem_ld_16x256b_x8(taddr + 64 * cc, ov);
    tmem_wait_ld();
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      ov[4 * k] = __float_as_uint(__uint_as_float(ov[4 * k]) * alpha_a);
      ov[4 * k + 1] = __float_as_uint(__uint_as_float(ov[4 * k + 1]) * alpha_a);
      ov[4 * k + 2] = __float_as_uint(__uint_as_float(ov[4 * k + 2]) * alpha_b);
      ov[4 * k + 3] = __float_as_uint(__uint_as_float(ov[4 * k + 3]) * alpha_b);
    }
    tmem_st_16x256b_x8(taddr + 64 * cc, ov);
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_qrope,
               const __grid_constant__ CUtensorMap tm_ckv,
               const __grid_constant__ CUtensorMap tm_krope, const Args a, const TcCfg cfg) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int item = blockIdx.x >> 1;
  const int rt = item % cfg.row_tiles;
  const int s = (item / cfg.row_tiles) % a.splits;
  const int b = item / (cfg.row_tiles * a.splits);
  const int nch = rank == 0 ? 5 : 4;
  uint32_t* anc = reinterpret_cast<uint32_t*>(sm + OFF_ANC);
  volatile int* misc = reinterpret_cast<volatile int*>(sm + OFF_MISC);
  auto BAR = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8u * i; };
  DeviceStatus* st = a.status;
  const uint64_t limit = cfg.limit_ns;
  grid_dep_launch();   // the combine kernel may start its weight loads early

  // ---- prologue: barriers, validation, ancestor masks, TMEM ------------------------
  if (tid == 0) {
    mbar_init(BAR(B_QR_FULL), 1);
    mbar_init(BAR(B_Q_READY), 8);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(BAR(B_KV_FULL + i), 1);
      mbar_init(BAR(B_KV_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(B_S_FULL + i), 1);
      mbar_init(BAR(B_S_FREE + i), 8);    // 4 sender + 4 softmax warps read the scores
      mbar_init(BAR(B_RX_FULL + i), 1);   // armed with expect_tx; filled by the peer's st.async
      mbar_init(BAR(B_TX_OK + i), 4);     // one relaxed arrival per peer softmax warp
    }
    for (int i = 0; i < kAfBufs; ++i) mbar_init(BAR(B_AF_FULL + i), 1);
    mbar_init(BAR(B_P_FULL), 4);          // our 4 softmax warps
    mbar_init(BAR(B_P_RX), 1);            // armed with expect_tx; filled by the peer's bulk copies
    // P.V commits of both CTAs (multicast), one barrier per tile parity: each
    // softmax warp waits only for the other parity's tiles, so it sees every
    // phase of the barrier it waits on in order.
    mbar_init(BAR(B_P_EMPTY + 0), 2);
    mbar_init(BAR(B_P_EMPTY + 1), 2);
    mbar_init(BAR(B_O_FULL), 1);
    mbar_init(BAR(B_MMA_DONE), 2);
    mbar_init(BAR(B_STALL), 1);
    for (int i = 0; i < 8; ++i) mbar_init(BAR(B_MREF + i), 1);
    mbar_init(BAR(B_LSUM), 4);
    mbar_expect_tx(BAR(B_RX_FULL + 0), kRxBytes);   // exchanges of tiles 0 and 1
    mbar_expect_tx(BAR(B_RX_FULL + 1), kRxBytes);
    for (int i = 0; i < kAfBufs; ++i) mbar_expect_tx(BAR(B_AF_FULL + i), kAfBytes);
    mbar_expect_tx(BAR(B_P_RX), 4 * kPQuadBytes);
    fence_mbar_init();
    int L = 0;
    int ok = prefix_ok(a, b, &L) ? 1 : 0;
    if (ok && a.page_size) {
      const int T = L + a.N;
      const int k0 = s * a.chunk, k1 = min(T, k0 + a.chunk);
      for (int p = k0 / a.page_size; k0 < k1 && p <= (k1 - 1) / a.page_size; ++p) {
        int page = a.page_table[(long long)b * a.max_pages + p];
        if (page < 0 || page >= a.num_pages) {
          record_error(st, KDTV_ERR_BAD_PAGE, (unsigned)b);
          ok = 0;
          break;
        }
      }
    }
    misc[1] = ok;
    misc[2] = L;
    misc[3] = 1;   // tree ok until a walker says otherwise
  }
  int32_t* par_s = reinterpret_cast<int32_t*>(sm + OFF_PAR);
  if (tid < a.N) par_s[tid] = a.parent[(long long)b * a.N + tid];
  __syncthreads();
  if (tid < a.N) {
    uint32_t m[4];
    bool good = ancestor_mask_smem(a, b, par_s, tid, m);
    anc[4 * tid + 0] = m[0]; anc[4 * tid + 1] = m[1];
    anc[4 * tid + 2] = m[2]; anc[4 * tid + 3] = m[3];
    if (!good) misc[3] = 0;
  }
  if (warp == 1) {
    tmem_alloc(sbase + OFF_MISC, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();   // the peer's barriers are initialised before any remote access

  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const bool ok = misc[1] && misc[3];
  const int L = misc[2];
  const int T = L + a.N;
  const int k0 = s * a.chunk;
  const int k1 = min(T, k0 + a.chunk);
  const int nt = (ok && k1 > k0) ? (k1 - k0 + BN - 1) / BN : 0;
  const long long req_row0 = (long long)b * a.N * a.H;    // first global row of request b
  const int nrows = a.N * a.H;

  if (warp == 0) {
    // ---- TMA producer --------------------------------------------------------------
    if (lane == 0 && nt > 0) {
      prefetch_tmap(&tm_ckv);
      const int qrow = (int)(req_row0 + (long long)rt * BM);
      if (rank == 0) {
        mbar_expect_tx(BAR(B_QR_FULL), kQRopeBytes);
        tma_load_2d(sbase + OFF_QR, &tm_qrope, BAR(B_QR_FULL), 0, qrow);
      }
      // Cache row of key tile j (paged: through the page table).
      auto tile_row = [&](int j) -> int {
        const int t0 = k0 + j * BN;
        return a.page_size ? a.page_table[(long long)b * a.max_pages + t0 / a.page_size] * a.page_size
                           : b * a.t_stride + t0;
      };
      auto prefetch = [&](int j) {
        const int row = tile_row(j);
        for (int c = 0; c < 4; ++c) tma_prefetch_2d(&tm_ckv, (int)rank * kHalf + c * CH, row);
        if (rank == 0) tma_prefetch_2d(&tm_krope, 0, row);
      };
      for (int j = kStages; j < kStages + kPrefetch && j < nt; ++j) prefetch(j);
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int stg = j % kStages;
        if (j >= kStages &&
            !wait(BAR(B_KV_EMPTY + stg), ((j / kStages) - 1) & 1, st, limit, W_KV_EMPTY))
          break;
        const int row = tile_row(j);
        mbar_expect_tx(BAR(B_KV_FULL + stg), nch * kKVChunk);
        const uint32_t dst = sbase + OFF_KV + stg * kMaxCh * kKVChunk;
        for (int c = 0; c < 4; ++c)
          tma_load_2d(dst + c * kKVChunk, &tm_ckv, BAR(B_KV_FULL + stg),
                      (int)rank * kHalf + c * CH, row);
        if (rank == 0) tma_load_2d(dst + 4 * kKVChunk, &tm_krope, BAR(B_KV_FULL + stg), 0, row);
        issued = j + 1;
        if (j + kStages + kPrefetch < nt) prefetch(j + kStages + kPrefetch);
      }
      // Drain: every issued copy has landed before this CTA may exit.
      if (rank == 0) wait(BAR(B_QR_FULL), 0, st, limit, W_DRAIN);
      for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j)
        wait(BAR(B_KV_FULL + j % kStages), (j / kStages) & 1, st, limit, W_DRAIN);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- Q.K^T issuer (also owns TMEM) ------------------------------------------------
    if (lane == 0 && nt > 0) {
      constexpr uint32_t kIdescQK = idesc_bf16(BM, BN, 0, 0);
      bool alive = wait(BAR(B_Q_READY), 0, st, limit, W_Q);
      if (alive && rank == 0) alive = wait(BAR(B_QR_FULL), 0, st, limit, W_Q);
      for (int j = 0; alive && j < nt; ++j) {
        const int stg = j % kStages, buf = j & 1;
        alive = wait(BAR(B_KV_FULL + stg), (j / kStages) & 1, st, limit, W_KV_FULL);
        // the score buffer is rewritten: senders and softmax must have read tile j-2
        if (alive && j >= 2)
          alive = wait(BAR(B_S_FREE + buf), ((j >> 1) - 1) & 1, st, limit, W_S_FREE);
        if (!alive) break;
        tc_fence_after();
        const uint32_t d = tmem + kColS + 64 * buf;
        const uint32_t kv = sbase + OFF_KV + stg * kMaxCh * kKVChunk;
#pragma unroll
        for (int kk = 0; kk < kHalf / 16; ++kk) {       // latent half: A = q_lat in TMEM
          uint64_t bd = smem_desc(kv + (kk >> 2) * kKVChunk + (kk & 3) * 32, 16, 1024);
          mma_bf16_ts(d, tmem + kColQ + 8 * kk, bd, kIdescQK, kk > 0);
        }
        if (rank == 0) {
#pragma unroll
          for (int kk = 0; kk < CH / 16; ++kk) {        // rope: A = q_rope in smem
            uint64_t ad = smem_desc(sbase + OFF_QR + kk * 32, 16, 1024);
            uint64_t bd = smem_desc(kv + 4 * kKVChunk + kk * 32, 16, 1024);
            mma_bf16(d, ad, bd, kIdescQK, 1);
          }
        }
        mma_commit(BAR(B_S_FULL + buf));
      }
      mma_commit(BAR(B_MMA_DONE));                 // drain every issued MMA (both issuers)
      wait(BAR(B_MMA_DONE), 0, st, limit, W_DRAIN);
    }
    __syncwarp();
  } else if (warp == kWarpPV) {
    // ---- P.V issuer: O_c += P . c_kv[:, 256c : 256c+256] ------------------------------
    if (lane == 0 && nt > 0) {
      constexpr uint32_t kIdescPV = idesc_bf16(BM, kHalf, 0, 1);
      bool alive = true;
      int p_armed = 1;                             // phases of B_P_RX armed so far
      for (int j = 0; j < nt; ++j) {
        const int stg = j % kStages;
        alive = wait(BAR(B_P_FULL), j & 1, st, limit, W_P_FULL);
        if (alive) alive = wait(BAR(B_P_RX), j & 1, st, limit, W_P_RX);
        // already complete (Q.K^T of tile j read this stage); orders the TMA data
        if (alive) alive = wait(BAR(B_KV_FULL + stg), (j / kStages) & 1, st, limit, W_KV_FULL);
        if (!alive) break;
        // arm the peer's P rows of tile j+1 before our commit lets the peer send them
        if (j + 1 < nt) { mbar_expect_tx(BAR(B_P_RX), 4 * kPQuadBytes); ++p_armed; }
        tc_fence_after();
        const uint32_t kv = sbase + OFF_KV + stg * kMaxCh * kKVChunk;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // A = P (K-major, 128B rows); B = V = c_kv columns of this CTA,
          // MN-major: 64-column chunks kKVChunk apart (LBO), 8-key groups 1 KiB apart (SBO).
          uint64_t ad = smem_desc(sbase + OFF_P + kk * 32, 16, 1024);
          uint64_t bd = smem_desc(kv + kk * 16 * 128, kKVChunk, 1024);
          mma_bf16(tmem + kColO, ad, bd, kIdescPV, (j > 0 || kk > 0));
        }
        mma_commit(BAR(B_KV_EMPTY + stg));
        mma_commit_multicast(BAR(B_P_EMPTY + (j & 1)), 0x3);   // both CTAs may overwrite P
      }
      if (alive) mma_commit(BAR(B_O_FULL));
      // After an abort: let the peer's P rows of an armed, unconsumed phase land.
      if (!alive && p_armed > 0) drain_wait(BAR(B_P_RX), (p_armed - 1) & 1, 200000ull);
      mma_commit(BAR(B_MMA_DONE));                 // drain every issued MMA (both issuers)
      wait(BAR(B_MMA_DONE), 0, st, limit, W_DRAIN);
    }
    __syncwarp();
  } else {
    // ---- warps 2..13: quadrant q = warp % 4 (its TMEM lanes 32q .. 32q+31) ------------
    const int q = warp & 3;
    const bool is_softmax = warp >= 6;
    const int par = is_softmax ? (warp - 6) >> 2 : 0;   // softmax: even (0) or odd (1) tiles
    const int c = lane & 3;
    // .16x256b slices: own rows (softmax) at 32q + 16 rank, peer rows (sender) at
    // 32q + 16 (1 - rank); thread t holds rows base + t/4 and base + t/4 + 8.
    const int own_base = 32 * q + 16 * (int)rank, peer_base = 32 * q + 16 * (int)peer;
    const uint32_t lane_own = static_cast<uint32_t>(own_base) << 16;
    const uint32_t lane_peer = static_cast<uint32_t>(peer_base) << 16;
    const uint32_t lane32 = static_cast<uint32_t>(32 * q) << 16;
    bool alive = true;

    if (nt > 0 && par == 0) {
      grid_dep_wait();   // q_lat is written by the absorb kernel
      // Q half of tile row 32q + lane -> TMEM [kColQ, +128) as bf16 pairs
      // (.32x32b layout); the sender warp stores words 0..63, the even-tile softmax
      // warp 64..127.
      const int rq = rt * BM + 32 * q + lane;
      const bool vq = rq < nrows;
      const int g = is_softmax ? 1 : 0;
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(a.q_lat) + (req_row0 + (vq ? rq : 0)) * 512 +
          rank * kHalf + 128 * g);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t w[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint4 x = vq ? src[8 * h + v] : make_uint4(0u, 0u, 0u, 0u);
          w[4 * v] = x.x; w[4 * v + 1] = x.y; w[4 * v + 2] = x.z; w[4 * v + 3] = x.w;
        }
        tmem_st32u(tmem + lane32 + kColQ + 64 * g + 32 * h, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_Q_READY));
    }

    if (!is_softmax) {
      // ---- sender: the peer's score rows -> the peer's receive buffer ---------------
      for (int j = 0; alive && j < nt; ++j) {
        const int buf = j & 1;
        alive = __all_sync(0xffffffffu, wait(BAR(B_S_FULL + buf), (j >> 1) & 1, st, limit, W_S_FULL));
        if (!alive) break;
        tc_fence_after();
        uint32_t v[32];
        tmem_ld_16x256b_x8(tmem + lane_peer + kColS + 64 * buf, v);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_S_FREE + buf));
        // one power-of-two scale per row: the row's 64 values are spread over
        // the 4 threads t with the same t / 4
        float ma = 0.f, mb = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          ma = max3f(ma, fabsf(__uint_as_float(v[4 * k])), fabsf(__uint_as_float(v[4 * k + 1])));
          mb = max3f(mb, fabsf(__uint_as_float(v[4 * k + 2])), fabsf(__uint_as_float(v[4 * k + 3])));
        }
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
        const int sha = fp16_shift(ma), shb = fp16_shift(mb);
        const float sca = pow2f(sha), scb = pow2f(shb);
        uint32_t w[16];                            // rows a then b, key pairs 8k + 2c
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          __half2 ha = __floats2half2_rn(__uint_as_float(v[4 * k]) * sca,
                                         __uint_as_float(v[4 * k + 1]) * sca);
          __half2 hb = __floats2half2_rn(__uint_as_float(v[4 * k + 2]) * scb,
                                         __uint_as_float(v[4 * k + 3]) * scb);
          w[k] = *reinterpret_cast<uint32_t*>(&ha);
          w[8 + k] = *reinterpret_cast<uint32_t*>(&hb);
        }
        // the peer has consumed what we sent into this receive buffer two tiles ago
        if (j >= 2) {
          alive = __all_sync(0xffffffffu, wait(BAR(B_TX_OK + buf), ((j >> 1) - 1) & 1, st, limit,
                                               W_TX_OK));
          if (!alive) break;
        }
        const uint32_t rxp = mapa(sbase + OFF_RX + buf * kRxStride, peer);
        const uint32_t rxfull_remote = mapa(BAR(B_RX_FULL + buf), peer);
#pragma unroll
        for (int m = 0; m < 4; ++m)
          st_async_v4u(rxp + ((q * 4 + m) * 32 + lane) * 16, w[4 * m], w[4 * m + 1], w[4 * m + 2],
                       w[4 * m + 3], rxfull_remote);
        st_async_u32(rxp + kRxData + (q * 32 + lane) * 4,
                     ((uint32_t)sha & 0xffffu) | ((uint32_t)shb << 16), rxfull_remote);
      }
    } else {
      // ---- softmax of this CTA's rows ra = own_base + t/4, rb = ra + 8 ---------------
      // Thread t holds keys 8k + 2c, 8k + 2c + 1 (k = 0..7) of each 64-key tile.
      const int ra = own_base + (lane >> 2), rb = ra + 8;
      const bool va = rt * BM + ra < nrows, vb = rt * BM + rb < nrows;
      const float sl2 = a.scale * 1.4426950408889634f;   // scores in log2 units
      const float* af = reinterpret_cast<const float*>(sm + OFF_AF);
      float* mref = reinterpret_cast<float*>(sm + OFF_MREF);
      float* lpart = reinterpret_cast<float*>(sm + OFF_LPART);
      // Reference maxima last used by this warp and its row sums relative to them.
      float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
      const int lead = 6 + 4 * par;               // the warp that re-arms this parity's receive barriers

      if (nt > 0 && (a.flags & KDTV_FLAG_TEST_STALL))
        alive = __all_sync(0xffffffffu, wait(BAR(B_STALL), 0, st, limit, W_STALL));

      // This warp takes the tiles j = par, par + 2, ...; the running reference
      // maxima pass between the two warps of the quadrant through shared memory.
      int next_rx = par;                          // first receive phase not yet consumed
      int next_af = par;
      for (int j = par; alive && j < nt; j += 2) {
        const int buf = j & 1;
        alive = __all_sync(0xffffffffu, wait(BAR(B_S_FULL + buf), (j >> 1) & 1, st, limit, W_S_FULL));
        if (!alive) break;
        tc_fence_after();
        uint32_t v[32];                            // own partial scores (fp32)
        tmem_ld_16x256b_x8(tmem + lane_own + kColS + 64 * buf, v);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_S_FREE + buf));   // QK^T of tile j+2 may overwrite

        // + the peer's partial scores for our rows (its st.async filled rx[buf])
        alive = __all_sync(0xffffffffu,
                           wait<true>(BAR(B_RX_FULL + buf), (j >> 1) & 1, st, limit, W_RX_FULL));
        if (!alive) break;
        next_rx = j + 2;
        if (warp == lead && lane == 0 && j + 2 < nt) mbar_expect_tx(BAR(B_RX_FULL + buf), kRxBytes);
        float sa[16], sb[16];
        {
          const uint32_t rxb = sbase + OFF_RX + buf * kRxStride;
          uint32_t pw[16], shw;
#pragma unroll
          for (int m = 0; m < 4; ++m)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(pw[4 * m]), "=r"(pw[4 * m + 1]), "=r"(pw[4 * m + 2]), "=r"(pw[4 * m + 3])
                         : "r"(rxb + ((q * 4 + m) * 32 + lane) * 16) : "memory");
          asm volatile("ld.shared.b32 %0, [%1];" : "=r"(shw) : "r"(rxb + kRxData + (q * 32 + lane) * 4)
                       : "memory");
          const float pia = pow2f(-(int)(int16_t)(shw & 0xffffu));
          const float pib = pow2f(-(int)(int16_t)(shw >> 16));
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&pw[k]));
            const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&pw[8 + k]));
            sa[2 * k] = fmaf(fa.x, pia, __uint_as_float(v[4 * k]));
            sa[2 * k + 1] = fmaf(fa.y, pia, __uint_as_float(v[4 * k + 1]));
            sb[2 * k] = fmaf(fb.x, pib, __uint_as_float(v[4 * k + 2]));
            sb[2 * k + 1] = fmaf(fb.y, pib, __uint_as_float(v[4 * k + 3]));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_relaxed(mapa(BAR(B_TX_OK + buf), peer));  // consumed

        // visibility mask (only tiles that reach past the prefix, or rows past the end)
        const int tb = k0 + j * BN;
        if (!(va && vb && tb + BN <= L)) {
#pragma unroll
          for (int rsel = 0; rsel < 2; ++rsel) {
            const bool vrow = rsel ? vb : va;
            const int node = vrow ? (rt * BM + (rsel ? rb : ra)) / a.H : 0;
            float* sv = rsel ? sb : sa;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int t = tb + 8 * (i >> 1) + 2 * c + (i & 1);
              bool vis = false;
              if (vrow && t < k1) {
                if (t < L) {
                  vis = true;
                } else {
                  const int jn = t - L;
                  vis = (anc[4 * node + (jn >> 5)] >> (jn & 31)) & 1u;
                }
              }
              if (!vis) sv[i] = -INFINITY;
            }
          }
        }
        // row maxima: 16 keys per thread, then the row's four threads
        float mta = max3f(sa[0], sa[1], sa[2]), mtb = max3f(sb[0], sb[1], sb[2]);
#pragma unroll
        for (int k = 3; k < 15; k += 2) {
          mta = max3f(mta, sa[k], sa[k + 1]);
          mtb = max3f(mtb, sb[k], sb[k + 1]);
        }
        mta = fmaxf(mta, sa[15]);
        mtb = fmaxf(mtb, sb[15]);
        mta = fmaxf(mta, __shfl_xor_sync(0xffffffffu, mta, 1));
        mtb = fmaxf(mtb, __shfl_xor_sync(0xffffffffu, mtb, 1));
        mta = fmaxf(mta, __shfl_xor_sync(0xffffffffu, mta, 2)) * sl2;
        mtb = fmaxf(mtb, __shfl_xor_sync(0xffffffffu, mtb, 2)) * sl2;

        // the reference maxima after tile j-1 (the other warp of this quadrant)
        float mpa = -INFINITY, mpb = -INFINITY;
        if (j >= 1) {
          alive = __all_sync(0xffffffffu, wait(BAR(B_MREF + 4 * (par ^ 1) + q), ((j - 1) >> 1) & 1,
                                               st, limit, W_MREF));
          if (!alive) break;
          mpa = mref[(par ^ 1) * BM + ra];
          mpb = mref[(par ^ 1) * BM + rb];
        }
        // lazy rescale: move the reference max only when it grows by > 8 (log2);
        // alpha rescales O (all tiles so far) to the new reference
        float alpha_a = 1.f, alpha_b = 1.f;
        float mna = mpa, mnb = mpb;
        if (mta > mpa + 8.f) {
          if (mpa != -INFINITY) alpha_a = ex2(mpa - mta);
          mna = mta;
        }
        if (mtb > mpb + 8.f) {
          if (mpb != -INFINITY) alpha_b = ex2(mpb - mtb);
          mnb = mtb;
        }
        if (c == 0) {
          mref[par * BM + ra] = mna;
          mref[par * BM + rb] = mnb;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_MREF + 4 * par + q));
        // this warp's row sums follow the reference
        if (mna != m_a) {
          if (m_a != -INFINITY) l_a *= ex2(m_a - mna);
          m_a = mna;
        }
        if (mnb != m_b) {
          if (m_b != -INFINITY) l_b *= ex2(m_b - mnb);
          m_b = mnb;
        }
        // our rows' rescale factors -> the peer (it rescales its half of O)
        {
          const int afb = j & (kAfBufs - 1);
          const uint32_t afr = mapa(BAR(B_AF_FULL + afb), peer);
          if (c < 2)
            st_async_u32(mapa(sbase + OFF_AF + (afb * BM + (c ? rb : ra)) * 4, peer),
                         __float_as_uint(c ? alpha_b : alpha_a), afr);
        }
        const float nma = m_a == -INFINITY ? 0.f : -m_a, nmb = m_b == -INFINITY ? 0.f : -m_b;
        uint32_t pa[8], pb[8];                     // bf16 pairs of P: keys 8k + 2c, +1
        float psa = 0.f, psb = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          pa[k] = pack_bf16x2(ex2(fmaf(sa[2 * k], sl2, nma)), ex2(fmaf(sa[2 * k + 1], sl2, nma)));
          pb[k] = pack_bf16x2(ex2(fmaf(sb[2 * k], sl2, nmb)), ex2(fmaf(sb[2 * k + 1], sl2, nmb)));
          psa += __uint_as_float(pa[k] << 16) + __uint_as_float(pa[k] & 0xffff0000u);
          psb += __uint_as_float(pb[k] << 16) + __uint_as_float(pb[k] & 0xffff0000u);
        }
        l_a += psa;
        l_b += psb;

        // P (single buffer) is free, and O stable, once P.V of tile j-1 completed in
        // both CTAs (the (j-1)/2-th phase of the other parity's barrier)
        if (j >= 1) {
          alive = __all_sync(0xffffffffu, wait(BAR(B_P_EMPTY + ((j - 1) & 1)), ((j - 1) >> 1) & 1, st,
                                               limit, W_P_EMPTY));
          if (!alive) break;
        }
        // P rows ra, rb: the pair for keys 8k + 2c is 4 bytes at offset 4c of the
        // row's 16-byte chunk k, stored 128B-swizzled (chunk k of row r at k ^ (r & 7)).
        {
          const uint32_t prow_a = sbase + OFF_P + ra * 128 + 4 * c;
          const uint32_t prow_b = sbase + OFF_P + rb * 128 + 4 * c;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            asm volatile("st.shared.b32 [%0], %1;" :: "r"(prow_a + ((k ^ (ra & 7)) << 4)), "r"(pa[k]) : "memory");
            asm volatile("st.shared.b32 [%0], %1;" :: "r"(prow_b + ((k ^ (rb & 7)) << 4)), "r"(pb[k]) : "memory");
          }
        }
        fence_async_smem();                         // visible to the tensor core and the copy engine
        __syncwarp();
        if (lane == 0) {
          // our 16 rows of this quadrant are one contiguous 2 KiB block
          const uint32_t off = OFF_P + own_base * 128;
          bulk_copy_to_peer(mapa(sbase + off, peer), sbase + off, kPQuadBytes,
                            mapa(BAR(B_P_RX), peer));
        }
        // the peer's rescale factors for its rows of this quadrant: both halves of
        // O must carry the same reference maxima before P.V of this tile
        const int afb = j & (kAfBufs - 1);
        alive = __all_sync(0xffffffffu,
                           wait<true>(BAR(B_AF_FULL + afb), (j / kAfBufs) & 1, st, limit, W_AF));
        if (!alive) break;
        next_af = j + 2;
        const float qa = af[afb * BM + (ra ^ 16)], qb = af[afb * BM + (rb ^ 16)];
        if (warp == lead && lane == 0 && j + kAfBufs < nt)
          mbar_expect_tx(BAR(B_AF_FULL + afb), kAfBytes);
        if (__any_sync(0xffffffffu, alpha_a != 1.f || alpha_b != 1.f || qa != 1.f || qb != 1.f)) {
          tc_fence_after();
          rescale_o_rows(tmem + lane_own + kColO, alpha_a, alpha_b);
          rescale_o_rows(tmem + lane_peer + kColO, qa, qb);
          tmem_wait_st();
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_P_FULL));
      }

      // After an abort, let what the peer may still be sending land before exit
      // (receive phases that were armed but not consumed); bounded, errors ignored.
      if (!alive) {
        if (next_rx < nt) drain_wait(BAR(B_RX_FULL + (next_rx & 1)), (next_rx >> 1) & 1, 200000ull);
        for (int t = next_af; t < next_af + kAfBufs && t < nt; t += 2)
          drain_wait(BAR(B_AF_FULL + (t & (kAfBufs - 1))), (t / kAfBufs) & 1, 200000ull);
      }

      // (m, l) of our rows: row sums meet across the row's four threads
      l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
      l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
      l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
      l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
      // the odd-tile warp hands its (m, l) to the even-tile warp, which merges
      // them (the later reference is the larger) and writes the row's (m, l)
      if (par == 1) {
        if (c == 0) {
          lpart[ra] = m_a; lpart[BM + ra] = l_a;
          lpart[rb] = m_b; lpart[BM + rb] = l_b;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_LSUM));
      } else if (ok) {
        alive = __all_sync(0xffffffffu, wait(BAR(B_LSUM), 0, st, limit, W_LSUM)) && alive;
        if (alive) {
          const float m1a = lpart[ra], l1a = lpart[BM + ra], m1b = lpart[rb], l1b = lpart[BM + rb];
          const float ma = fmaxf(m_a, m1a), mb = fmaxf(m_b, m1b);
          l_a = (m_a == -INFINITY ? 0.f : l_a * ex2(m_a - ma)) + (m1a == -INFINITY ? 0.f : l1a * ex2(m1a - ma));
          l_b = (m_b == -INFINITY ? 0.f : l_b * ex2(m_b - mb)) + (m1b == -INFINITY ? 0.f : l1b * ex2(m1b - mb));
          m_a = ma;
          m_b = mb;
        }
      }
      if (ok && alive && c == 0 && par == 0) {
        const long long rows = (long long)a.B * a.N * a.H;
#pragma unroll
        for (int rsel = 0; rsel < 2; ++rsel) {
          const bool vrow = rsel ? vb : va;
          const float l = rsel ? l_b : l_a, m = rsel ? m_b : m_a;
          if (vrow) {
            float* ml = a.part_ml + ((long long)s * rows + req_row0 + rt * BM + (rsel ? rb : ra)) * 2;
            const bool has = nt > 0 && l > 0.f;
            ml[0] = has ? m * 0.6931471805599453f : -INFINITY;
            ml[1] = has ? l : 0.f;
          }
        }
      }
    }

    // ---- epilogue: unnormalised partial o_lat half of rows 32q .. 32q+31 ----------------
    // (.32x32b: thread = row; the sender warp writes O columns 0..127, the softmax 128..255)
    if (alive && nt > 0 && par == 0)
      alive = __all_sync(0xffffffffu, wait(BAR(B_O_FULL), 0, st, limit, W_O_FULL));
    const int r = 32 * q + lane;
    const int rr = rt * BM + r;
    if (ok && alive && nt > 0 && par == 0) {
      const long long rows = (long long)a.B * a.N * a.H;
      const int g = is_softmax ? 1 : 0;
      float* po = a.part_o + ((long long)s * rows + req_row0 + (rr < nrows ? rr : 0)) * a.d_c +
                  rank * kHalf + 128 * g;
      tc_fence_after();
      for (int cc = 0; cc < 4; ++cc) {
        float ov[32];
        tmem_ld32(tmem + lane32 + kColO + 128 * g + 32 * cc, ov);
        tmem_wait_ld();
        if (rr < nrows) {
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4*>(po + 32 * cc + k) =
                make_float4(ov[k], ov[k + 1], ov[k + 2], ov[k + 3]);
        }
      }
    }
  }

  // ---- teardown ------------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();   // the peer may still arrive on our barriers until here
}

int row_tiles_of(const kdtv_dims* d) { return (d->N * d->H + BM - 1) / BM; }

}  // namespace

namespace {
// The driver's tensor-map encoder, resolved through the runtime so that the
// library does not link libcuda (it must load on hosts without a driver).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

// 2-D bf16 tensor map with a 128-byte swizzle: rows x cols (row stride
// cols * 2 bytes), box = box_rows x box_cols.
CUresult encode_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_cols, uint32_t box_rows, uint64_t row_stride_elems) {
  EncodeTiledFn fn = encoder();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {(row_stride_elems ? row_stride_elems : cols) * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int tc_supported(const kdtv_dims* d) {
  if (d->dtype != KDTV_BF16 || d->d_c != 512 || d->d_rope != 64) return 0;
  if (d->page_size != 0 && d->page_size != 64) return 0;
  if (d->kv_chunk % BN) return 0;
  return 1;
}

int tc_launches(const kdtv_dims* d, int splits) {
  if (d->flags & KDTV_FLAG_SIMT_PROJ) return 4;
  Args a;
  a.dtype = d->dtype; a.d_c = d->d_c; a.d_v = d->d_v; a.d_nope = d->d_nope; a.splits = splits;
  return 2 + (combine_uproj_tc_ok(a) ? 1 : 2);
}

// Split-KV chunk: pick the split count s that minimises the modelled
// makespan  ceil(2 * items(s) / SMs) / s  (two CTAs per item, one CTA per
// SM), with a small per-split cost for the partials it writes and merges.
int tc_chunk(const kdtv_dims* d, int sms) {
  const long long base = (long long)d->B * row_tiles_of(d);
  const int t_cap = d->page_size ? d->max_pages * d->page_size : d->t_stride;
  const int max_s = (t_cap + 511) / 512;
  int best_s = 1;
  double best = 1e30;
  for (int s = 1; s <= (max_s < 64 ? max_s : 64); ++s) {
    const double waves = (double)((2 * base * s + sms - 1) / sms);
    const double cost = waves / s + 0.02 * s;
    if (cost < best - 1e-9) { best = cost; best_s = s; }
  }
  int chunk = (t_cap + best_s - 1) / best_s;
  return (chunk + BN - 1) / BN * BN;
}

cudaError_t launch_tc(const Args& a, const Plan& p, cudaStream_t st, cudaEvent_t* ev) {
  for (const void* ptr : {a.q_rope, a.c_kv, a.k_rope, static_cast<const void*>(a.q_lat)})
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return cudaErrorMisalignedAddress;
  const long long rows = (long long)a.B * a.N * a.H;
  const long long kv_rows = a.page_size ? (long long)a.num_pages * a.page_size
                                        : (long long)a.B * a.t_stride;
  CUtensorMap tqr, tck, tkr;
  if (encode_2d(&tqr, a.q_rope, rows, 64, CH, BM) != CUDA_SUCCESS ||
      encode_2d(&tck, a.c_kv, kv_rows, 512, CH, BN) != CUDA_SUCCESS ||
      encode_2d(&tkr, a.k_rope, kv_rows, 64, CH, BN) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  const bool simt_proj = a.flags & KDTV_FLAG_SIMT_PROJ;
  cudaError_t e = simt_proj ? launch_absorb(a, st, /*bf16_out=*/true) : launch_absorb_tc(a, st);
  if (e != cudaSuccess) return e;
  if (ev) cudaEventRecord(ev[1], st);

  TcCfg cfg;
  cfg.row_tiles = (a.N * a.H + BM - 1) / BM;
  cfg.limit_ns = (a.flags & KDTV_FLAG_TEST_STALL) ? 20000000ull : 2000000000ull;
  const long long items = (long long)a.B * cfg.row_tiles * a.splits;
  if (2 * items > 0x7fffffffll) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes);
  if (e != cudaSuccess) return e;
  // Overlap with the absorb kernel's tail unless phase events split the call.
  e = launch_ex(attn_tc_kernel, dim3((unsigned)(2 * items)), dim3(kThreads), kSmemBytes, st,
                /*pdl=*/ev == nullptr && !simt_proj, tqr, tck, tkr, a, cfg);
  if (e != cudaSuccess) return e;
  if (ev) cudaEventRecord(ev[2], st);
  return simt_proj ? launch_combine_uproj(a, p, st, ev) : launch_combine_uproj_tc(a, p, st, ev);
}

}  // namespace kdtv
