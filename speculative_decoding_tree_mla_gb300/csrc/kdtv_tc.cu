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
// Each CTA computes a partial score tile S_c = Q_c K_c^T on tcgen05 into TMEM,
// the two partials are exchanged through distributed shared memory and
// summed, both CTAs run the same online softmax on S = S_0 + S_1 (so they
// agree bit for bit), and each accumulates its own half of the latent output
// O_c += P . c_kv[:, 256c : 256c+256] in TMEM.
//
// TMEM (512 columns per CTA): O_c [0, 256) fp32; q_lat half [256, 384) as
// bf16 pairs (the A operand of Q.K^T); two score buffers [384, 448) and
// [448, 512).  Shared memory: a 3-stage TMA ring of 64-key cache tiles
// (128-byte swizzled 64-column chunks; the same tile is the K-major B operand
// of Q.K^T and the MN-major B operand of P.V), q_rope (CTA 0), two P tiles
// (the K-major A operand of P.V), and two receive buffers of the score
// exchange.  Key tiles are prefetched into L2 a few tiles ahead of the ring.
//
// Warp roles (480 threads): warp 0 issues TMA loads; warp 1 owns TMEM and
// issues Q.K^T; warps 2-5 (one thread per query row) quantise each partial
// score tile to fp16 once, write it back into the score buffer for their own
// softmax and stream it to the peer with st.async; warps 6-13 (16 rows each,
// four threads per row in the .16x256b TMEM layout, so row maxima and sums
// meet by warp shuffles) add the peer's partial, mask, run the online
// softmax, write P to shared memory and finally write the partial o_lat;
// warp 14 issues P.V.  A score buffer is reused once its scores are read, so
// Q.K^T runs up to two tiles ahead of the softmax, and two receive buffers
// let the transfer of tile j+1 overlap the softmax of tile j.  Every wait is
// bounded (2 s, or ~20 ms with KDTV_FLAG_TEST_STALL); on timeout the kernel
// records KDTV_ERR_DEVICE_TIMEOUT, drains its in-flight copies and MMAs,
// frees TMEM and returns.

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
constexpr int kStages = 3;
constexpr int kPrefetch = 3;     // key tiles prefetched into L2 beyond the stages in flight
constexpr int kMaxCh = 5;        // CTA 0: 4 latent chunks + 1 rope chunk per key tile
constexpr int kKVChunk = BN * CH * 2;   // 8 KiB
constexpr int kQRopeBytes = BM * CH * 2;
// Score exchange buffers.  A partial score row travels as 64 fp16 values
// scaled by an exact power of two chosen from the row's largest magnitude (so
// it cannot overflow and keeps 11 significant bits relative to that maximum),
// 128 bytes per row in the order the softmax threads read it, then one 32-bit
// exponent per row.
constexpr int kRxData = BM * BN * 2;
constexpr int kRxBytes = kRxData + BM * 4;
constexpr int kThreads = 480;    // TMA, QK^T issuer, 4 senders, 8 softmax, P.V issuer
constexpr int kWarpPV = 14;      // the P.V issuer warp
constexpr int kPBytes = BM * BN * 2;   // one P tile: 128 rows x 64 keys bf16, 128B-swizzled
constexpr int kTmemCols = 512;
constexpr int kColO = 0;
constexpr int kColQ = 256;
constexpr int kColSP = 384;      // + 64 * buffer

constexpr int OFF_KV = 0;
constexpr int OFF_QR = OFF_KV + kStages * kMaxCh * kKVChunk;
constexpr int kRxStride = (kRxBytes + 1023) / 1024 * 1024;
constexpr int OFF_P = OFF_QR + kQRopeBytes;                  // two P tiles (A of P.V)
constexpr int OFF_RX = OFF_P + 2 * kPBytes;                   // two receive buffers
constexpr int OFF_ANC = OFF_RX + 2 * kRxStride;
constexpr int OFF_PAR = OFF_ANC + kMaxNodes * 16;               // staged parent[]
constexpr int OFF_LSUM = OFF_PAR + kMaxNodes * 4;               // [l | m][BM] floats (epilogue)
constexpr int OFF_OSH = OFF_LSUM + 2 * BM * 4;                   // [2 tiles][BM] own fp16 shifts
constexpr int OFF_BAR = OFF_OSH + 2 * BM * 4;
constexpr int kNumBars = 40;
constexpr int OFF_MISC = OFF_BAR + kNumBars * 8;
constexpr int kSmemBytes = OFF_MISC + 64 + 1024;   // + slack for 1 KiB alignment
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(OFF_P % 1024 == 0 && OFF_RX % 1024 == 0 && OFF_QR % 1024 == 0,
              "128B-swizzled tiles need 1 KiB alignment");
static_assert(kThreads == 32 * (kWarpPV + 1), "warp roles");

// Barrier indices (derived from kStages so the groups never overlap).
enum Bar : int {
  B_QR_FULL = 0, B_Q_READY = 1, B_KV_FULL = 2,
  B_KV_EMPTY = B_KV_FULL + kStages,
  B_S_FULL = B_KV_EMPTY + kStages,   // [2]
  B_S_FREE = B_S_FULL + 2,           // [2] the softmax has read the quantised own scores
  B_OWN = B_S_FREE + 2,              // [2] senders wrote the quantised own scores
  B_P_FULL = B_OWN + 2,              // [2]
  B_P_EMPTY = B_P_FULL + 2,          // [2]
  B_O_FULL = B_P_EMPTY + 2,
  B_RX_FULL = B_O_FULL + 1,          // [2]
  B_TX_OK = B_RX_FULL + 2,           // [2]
  B_STALL = B_TX_OK + 2,
  B_MMA_DONE = B_STALL + 1,
  B_LSUM = B_MMA_DONE + 1,           // softmax warps published the rows' (l, m)
  B_COUNT = B_LSUM + 1
};
static_assert(B_COUNT <= kNumBars, "barrier slots");

// Wait sites (reported as the timeout detail).
enum Site { W_Q = 1, W_KV_FULL, W_KV_EMPTY, W_P_FULL, W_S_FULL, W_TX_OK, W_RX_FULL,
            W_P_EMPTY, W_O_FULL, W_STALL, W_DRAIN, W_S_FREE, W_OWN };

struct TcCfg {
  int row_tiles;               // ceil(N * H / 128)
  unsigned long long limit_ns; // bound on every wait
};

// 2^e as a float for e in [-126, 127] (exact).
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// Shift that maps max |v| into [2^14, 2^15): the fp16 range with headroom.
// Capped at 100 so that every nonzero fp16 value times 2^-shift is a normal
// float: the dequantised products are then exact in both CTAs.
__device__ __forceinline__ int fp16_shift(float amax) {
  if (!(amax > 0.f)) return 0;
  const int e = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127;   // floor(log2(amax))
  const int sh = 14 - e;
  return sh < -126 ? -126 : (sh > 100 ? 100 : sh);
}

__device__ __forceinline__ float max32(const float (&v)[32]) {
  float m[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) m[i] = fmaxf(v[2 * i], v[2 * i + 1]);
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
  return m[0];
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
      mbar_init(BAR(B_S_FREE + i), 8);    // 8 softmax warps have read the own scores
      mbar_init(BAR(B_OWN + i), 4);       // 4 sender warps quantised them
      mbar_init(BAR(B_P_FULL + i), 8);
      mbar_init(BAR(B_P_EMPTY + i), 1);
      mbar_init(BAR(B_RX_FULL + i), 1);   // armed with expect_tx; filled by the peer's st.async
      mbar_init(BAR(B_TX_OK + i), 8);     // one relaxed arrival per peer softmax warp
    }
    mbar_init(BAR(B_O_FULL), 1);
    mbar_init(BAR(B_STALL), 1);
    mbar_init(BAR(B_MMA_DONE), 2);      // both MMA issuers drained
    mbar_init(BAR(B_LSUM), 8);
    mbar_expect_tx(BAR(B_RX_FULL + 0), kRxBytes);   // exchange of tiles 0 and 1
    mbar_expect_tx(BAR(B_RX_FULL + 1), kRxBytes);
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
  cluster_sync();   // the peer's barriers are initialised before any remote arrive

  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const bool ok = misc[1] && misc[3];
  const int L = misc[2];
  const int T = L + a.N;
  const int k0 = s * a.chunk;
  const int k1 = min(T, k0 + a.chunk);
  const int nt = (ok && k1 > k0) ? (k1 - k0 + BN - 1) / BN : 0;
  const long long req_row0 = (long long)b * a.N * a.H;    // first global row of request b

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
      // L2 prefetch kPrefetch tiles ahead of the loads, so that a refilled
      // stage finds its tile in L2 rather than in DRAM.
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
        const uint32_t d = tmem + kColSP + 64 * buf;
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
  } else if (warp < 6) {
    // ---- sender warps 2..5: own partial scores -> the peer's receive buffer ----------
    int* osh = reinterpret_cast<int*>(sm + OFF_OSH);
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    bool alive = true;
    for (int j = 0; alive && j < nt; ++j) {
      const int buf = j & 1;
      alive = __all_sync(0xffffffffu, wait(BAR(B_S_FULL + buf), (j >> 1) & 1, st, limit, W_S_FULL));
      if (!alive) break;
      tc_fence_after();
      float sv[2][32];
      tmem_ld32(tmem + lane_addr + kColSP + 64 * buf, sv[0]);
      tmem_ld32(tmem + lane_addr + kColSP + 64 * buf + 32, sv[1]);
      tmem_wait_ld();
      // Quantise the partial scores once, to fp16 with an exact power-of-two
      // scale per row; the same words go to the peer and, through the first 32
      // columns of this score buffer, to our own softmax warps.
      uint32_t w[32];
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fmaxf(fabsf(sv[0][k]), fabsf(sv[1][k])));
      const int sh = fp16_shift(amax);
      const float sc = pow2f(sh);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          __half2 h2 = __floats2half2_rn(sv[hh][2 * k] * sc, sv[hh][2 * k + 1] * sc);
          w[16 * hh + k] = *reinterpret_cast<uint32_t*>(&h2);
        }
      tmem_st32u(tmem + lane_addr + kColSP + 64 * buf, w);
      osh[buf * BM + r] = sh;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_OWN + buf));
      // the peer has consumed what we sent into this receive buffer two tiles ago
      if (j >= 2) {
        alive = __all_sync(0xffffffffu, wait(BAR(B_TX_OK + buf), ((j >> 1) - 1) & 1, st, limit,
                                             W_TX_OK));
        if (!alive) break;
      }
      // Receive layout, chunk-major: 16-byte chunk m = 2c + h of row r at
      // (m * BM + r) * 16 holds words {2c, 2c+1, 2c+8, 2c+9} (h = 0) or
      // {2c+16, 2c+17, 2c+24, 2c+25} (h = 1), the words one .16x256b softmax
      // thread (c = t % 4) needs; one warp store is a contiguous 512-byte
      // block.  The rows' shifts follow the data.
      const uint32_t rx_row = mapa(sbase + OFF_RX + buf * kRxStride + r * 16, peer);
      const uint32_t rxfull_remote = mapa(BAR(B_RX_FULL + buf), peer);
#pragma unroll
      for (int cq = 0; cq < 4; ++cq)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int w0 = 2 * cq + 16 * h;
          st_async_v4u(rx_row + (2 * cq + h) * BM * 16, w[w0], w[w0 + 1], w[w0 + 8], w[w0 + 9],
                       rxfull_remote);
        }
      st_async_u32(mapa(sbase + OFF_RX + buf * kRxStride + kRxData + r * 4, peer), (uint32_t)sh,
                   rxfull_remote);
    }
  } else if (warp < kWarpPV) {
    // ---- softmax warps 6..13 ------------------------------------------------------------
    // Warp (q, g) owns tile rows 32q + 16g .. +15 (TMEM lane quadrant q).  In the
    // .16x256b layout thread t holds rows ra = base + t/4 and rb = ra + 8, keys
    // 16k + 4c .. 16k + 4c + 3 (c = t % 4, k = 0..3) of each 64-key tile, so the
    // four threads of a row meet through two shuffles.
    const int q = warp & 3;
    const int g = (warp - 6) >> 2;
    const int c = lane & 3;
    const int ra = 32 * q + 16 * g + (lane >> 2), rb = ra + 8;
    const uint32_t lane16 = static_cast<uint32_t>(32 * q + 16 * g) << 16;
    const uint32_t lane32 = static_cast<uint32_t>(32 * q) << 16;
    const int nrows = a.N * a.H;
    const bool va = rt * BM + ra < nrows, vb = rt * BM + rb < nrows;
    const float sl2 = a.scale * 1.4426950408889634f;   // scores in log2 units
    float* lsum = reinterpret_cast<float*>(sm + OFF_LSUM);
    const int* osh = reinterpret_cast<const int*>(sm + OFF_OSH);
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
    bool alive = true;

    if (nt > 0) {
      grid_dep_wait();   // q_lat is written by the absorb kernel
      // Q half of tile row 32q + lane, latent columns 128g .. 128g+127 of this
      // CTA's half -> TMEM [kColQ + 64g, +64) as bf16 pairs (.32x32b layout).
      const int rq = rt * BM + 32 * q + lane;
      const bool vq = rq < nrows;
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

    if (nt > 0 && (a.flags & KDTV_FLAG_TEST_STALL))
      alive = __all_sync(0xffffffffu, wait(BAR(B_STALL), 0, st, limit, W_STALL));

    int consumed = 0;                            // exchange tiles received so far
    for (int j = 0; alive && j < nt; ++j) {
      const int buf = j & 1;
      alive = __all_sync(0xffffffffu, wait(BAR(B_OWN + buf), (j >> 1) & 1, st, limit, W_OWN));
      if (!alive) break;
      tc_fence_after();
      // own quantised partial scores (fp16 pairs, columns 0..31 of the score buffer)
      uint32_t ow[16];
      tmem_ld_16x256b_x4(tmem + lane16 + kColSP + 64 * buf, ow);
      const float oia = pow2f(-osh[buf * BM + ra]), oib = pow2f(-osh[buf * BM + rb]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_S_FREE + buf));   // QK^T of tile j+2 may overwrite

      // + the peer's partial scores (its st.async filled rx[buf]).  Both products
      // are exact (fp16 times a power of two), so own + peer rounds to the same
      // float in both CTAs whichever is added first.
      alive = __all_sync(0xffffffffu,
                         wait<true>(BAR(B_RX_FULL + buf), (j >> 1) & 1, st, limit, W_RX_FULL));
      if (!alive) break;
      consumed = j + 1;
      if (warp == 6 && lane == 0 && j + 2 < nt) mbar_expect_tx(BAR(B_RX_FULL + buf), kRxBytes);
      float sa[16], sb[16];
      {
        const uint32_t rxb = sbase + OFF_RX + buf * kRxStride;
        int psa, psb;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(psa) : "r"(rxb + kRxData + ra * 4) : "memory");
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(psb) : "r"(rxb + kRxData + rb * 4) : "memory");
        const float pia = pow2f(-psa), pib = pow2f(-psb);
#pragma unroll
        for (int rsel = 0; rsel < 2; ++rsel) {
          const int row = rsel ? rb : ra;
          const float pinv = rsel ? pib : pia, oinv = rsel ? oib : oia;
          float* sv = rsel ? sb : sa;
          uint32_t pw[8];
#pragma unroll
          for (int h = 0; h < 2; ++h)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(pw[4 * h]), "=r"(pw[4 * h + 1]), "=r"(pw[4 * h + 2]),
                           "=r"(pw[4 * h + 3])
                         : "r"(rxb + ((2 * c + h) * BM + row) * 16) : "memory");
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              // key 16k + 4c + 2e (+1): own word ow[4k + 2 rsel + e], peer word pw[2k + e]
              const float2 fo = __half22float2(*reinterpret_cast<const __half2*>(&ow[4 * k + 2 * rsel + e]));
              const float2 fp = __half22float2(*reinterpret_cast<const __half2*>(&pw[2 * k + e]));
              sv[4 * k + 2 * e] = fmaf(fp.x, pinv, fo.x * oinv);
              sv[4 * k + 2 * e + 1] = fmaf(fp.y, pinv, fo.y * oinv);
            }
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
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int t = tb + 16 * k + 4 * c + e;
              bool vis = false;
              if (vrow && t < k1) {
                if (t < L) {
                  vis = true;
                } else {
                  const int jn = t - L;
                  vis = (anc[4 * node + (jn >> 5)] >> (jn & 31)) & 1u;
                }
              }
              if (!vis) sv[4 * k + e] = -INFINITY;
            }
        }
      }
      // row maxima: 16 keys per thread, then the row's four threads
      float mta = sa[0], mtb = sb[0];
#pragma unroll
      for (int k = 1; k < 16; ++k) { mta = fmaxf(mta, sa[k]); mtb = fmaxf(mtb, sb[k]); }
      mta = fmaxf(mta, __shfl_xor_sync(0xffffffffu, mta, 1));
      mtb = fmaxf(mtb, __shfl_xor_sync(0xffffffffu, mtb, 1));
      mta = fmaxf(mta, __shfl_xor_sync(0xffffffffu, mta, 2)) * sl2;
      mtb = fmaxf(mtb, __shfl_xor_sync(0xffffffffu, mtb, 2)) * sl2;

      // lazy rescale: move the reference max only when it grows by > 8 (log2);
      // the four threads of a row take the same decision from the same inputs
      float alpha_a = 1.f, alpha_b = 1.f;
      bool rescale = false;
      if (mta > m_a + 8.f) {
        if (m_a != -INFINITY) { alpha_a = ex2(m_a - mta); rescale = true; }
        l_a *= alpha_a;
        m_a = mta;
      }
      if (mtb > m_b + 8.f) {
        if (m_b != -INFINITY) { alpha_b = ex2(m_b - mtb); rescale = true; }
        l_b *= alpha_b;
        m_b = mtb;
      }
      const float nma = m_a == -INFINITY ? 0.f : -m_a, nmb = m_b == -INFINITY ? 0.f : -m_b;
      uint32_t pk[16];                            // [row][k][pair]: bf16 pairs of P
      float psa = 0.f, psb = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t ha = pack_bf16x2(ex2(fmaf(sa[2 * k], sl2, nma)), ex2(fmaf(sa[2 * k + 1], sl2, nma)));
        const uint32_t hb = pack_bf16x2(ex2(fmaf(sb[2 * k], sl2, nmb)), ex2(fmaf(sb[2 * k + 1], sl2, nmb)));
        pk[k] = ha;
        pk[8 + k] = hb;
        psa += __uint_as_float(ha << 16) + __uint_as_float(ha & 0xffff0000u);
        psb += __uint_as_float(hb << 16) + __uint_as_float(hb & 0xffff0000u);
      }
      l_a += psa;
      l_b += psb;

      // the P buffer is free once P.V of tile j-2 (same buffer) has completed;
      // O is stable once P.V of tile j-1 has completed
      if (j >= 2) {
        alive = __all_sync(0xffffffffu,
                           wait(BAR(B_P_EMPTY + buf), ((j >> 1) - 1) & 1, st, limit, W_P_EMPTY));
        if (!alive) break;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        if (j >= 1) {
          alive = __all_sync(0xffffffffu, wait(BAR(B_P_EMPTY + (buf ^ 1)), ((j - 1) >> 1) & 1, st,
                                               limit, W_P_EMPTY));
          if (!alive) break;
        }
        tc_fence_after();
        for (int cc = 0; cc < kHalf / 64; ++cc) {     // this warp's 16 rows x 256 O columns
          uint32_t ov[32];
          const uint32_t oa = tmem + lane16 + kColO + 64 * cc;
          tmem_ld_16x256b_x8(oa, ov);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            ov[4 * k] = __float_as_uint(__uint_as_float(ov[4 * k]) * alpha_a);
            ov[4 * k + 1] = __float_as_uint(__uint_as_float(ov[4 * k + 1]) * alpha_a);
            ov[4 * k + 2] = __float_as_uint(__uint_as_float(ov[4 * k + 2]) * alpha_b);
            ov[4 * k + 3] = __float_as_uint(__uint_as_float(ov[4 * k + 3]) * alpha_b);
          }
          tmem_st_16x256b_x8(oa, ov);
        }
        tmem_wait_st();
        tc_fence_before();
      }
      // P rows ra, rb: keys 16k + 4c .. +3 are 8 bytes at offset 8(c & 1) of the
      // row's 16-byte chunk 2k + c/2, stored 128B-swizzled (chunk m of row r at
      // m ^ (r & 7)): the K-major A operand layout of P.V.
      {
        const uint32_t pb = sbase + OFF_P + buf * kPBytes;
#pragma unroll
        for (int rsel = 0; rsel < 2; ++rsel) {
          const int row = rsel ? rb : ra;
          const uint32_t prow = pb + (row >> 3) * 1024 + (row & 7) * 128 + 8 * (c & 1);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            asm volatile("st.shared.v2.b32 [%0], {%1, %2};"
                         :: "r"(prow + (((2 * k + (c >> 1)) ^ (row & 7)) << 4)),
                            "r"(pk[8 * rsel + 2 * k]), "r"(pk[8 * rsel + 2 * k + 1]) : "memory");
        }
      }
      fence_async_smem();                         // visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_P_FULL + buf));
    }

    // After an abort, let score rows the peer may still be sending land before exit
    // (receive phases that were armed but not consumed); bounded, errors ignored.
    for (int t = consumed; t < consumed + 2 && t < nt; ++t)
      drain_wait(BAR(B_RX_FULL + (t & 1)), (t >> 1) & 1, 200000ull);

    // ---- epilogue: unnormalised partial o_lat half, (m, l) -----------------------------
    // Row sums meet across the row's four threads; the (m, l) of every row go
    // through shared memory to the .32x32b read-out below (thread = row
    // 32q + lane, O columns 128g .. 128g+127).
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    if (alive && nt > 0)
      alive = __all_sync(0xffffffffu, wait(BAR(B_O_FULL), 0, st, limit, W_O_FULL));
    float l_sum = 0.f, m_row = -INFINITY;
    const int r = 32 * q + lane;                 // read-out row
    const int rr = rt * BM + r;
    const bool row_valid = rr < nrows;
    if (alive && nt > 0) {
      if (c == 0) {
        lsum[ra] = l_a; lsum[BM + ra] = m_a;
        lsum[rb] = l_b; lsum[BM + rb] = m_b;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_LSUM));
      alive = __all_sync(0xffffffffu, wait(BAR(B_LSUM), 0, st, limit, W_O_FULL));
      if (alive) { l_sum = lsum[r]; m_row = lsum[BM + r]; }
    }
    // tcgen05.ld is warp-collective: every lane loads, only valid rows store.
    const bool has_data = ok && alive && nt > 0 && row_valid && l_sum > 0.f;
    if (ok && alive && row_valid && g == 0) {
      const long long rows = (long long)a.B * a.N * a.H;
      float* ml = a.part_ml + ((long long)s * rows + req_row0 + rr) * 2;
      if (rank == 0) {
        ml[0] = has_data ? m_row * 0.6931471805599453f : -INFINITY;
        ml[1] = has_data ? l_sum : 0.f;
      }
    }
    if (ok && alive && nt > 0 && __any_sync(0xffffffffu, has_data)) {
      const long long rows = (long long)a.B * a.N * a.H;
      float* po = a.part_o + ((long long)s * rows + req_row0 + (has_data ? rr : 0)) * a.d_c +
                  rank * kHalf + 128 * g;
      tc_fence_after();
      for (int cc = 0; cc < 4; ++cc) {
        float ov[32];
        tmem_ld32(tmem + lane32 + kColO + 128 * g + 32 * cc, ov);
        tmem_wait_ld();
        if (has_data) {
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4*>(po + 32 * cc + k) =
                make_float4(ov[k], ov[k + 1], ov[k + 2], ov[k + 3]);
        }
      }
    }
  } else {
    // ---- P.V issuer (warp 14): O_c += P . c_kv[:, 256c : 256c+256] -------------------
    if (lane == 0 && nt > 0) {
      constexpr uint32_t kIdescPV = idesc_bf16(BM, kHalf, 0, 1);
      bool alive = true;
      for (int j = 0; j < nt; ++j) {
        const int stg = j % kStages, buf = j & 1;
        alive = wait(BAR(B_P_FULL + buf), (j >> 1) & 1, st, limit, W_P_FULL);
        // already complete (Q.K^T of tile j read this stage); orders the TMA data
        if (alive) alive = wait(BAR(B_KV_FULL + stg), (j / kStages) & 1, st, limit, W_KV_FULL);
        if (!alive) break;
        tc_fence_after();
        const uint32_t kv = sbase + OFF_KV + stg * kMaxCh * kKVChunk;
        const uint32_t pb = sbase + OFF_P + buf * kPBytes;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // A = P (K-major, 128B rows); B = V = c_kv columns of this CTA,
          // MN-major: 64-column chunks kKVChunk apart (LBO), 8-key groups 1 KiB apart (SBO).
          uint64_t ad = smem_desc(pb + kk * 32, 16, 1024);
          uint64_t bd = smem_desc(kv + kk * 16 * 128, kKVChunk, 1024);
          mma_bf16(tmem + kColO, ad, bd, kIdescPV, (j > 0 || kk > 0));
        }
        mma_commit(BAR(B_KV_EMPTY + stg));
        mma_commit(BAR(B_P_EMPTY + buf));
      }
      if (alive) mma_commit(BAR(B_O_FULL));
      mma_commit(BAR(B_MMA_DONE));                 // drain every issued MMA (both issuers)
      wait(BAR(B_MMA_DONE), 0, st, limit, W_DRAIN);
    }
    __syncwarp();
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
