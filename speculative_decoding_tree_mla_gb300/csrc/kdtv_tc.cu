// Tensor-core (tcgen05) path of kdtv_verify_attn: bf16 inputs, the MLA
// latent layout d_c = 512, d_rope = 64, fp32 accumulation.
//
// The attention step (tree-masked scores, online softmax, P . c_kv) of the
// "tree-verify MLA-absorb attention kernel with visibility masking" ("The
// Moment of Proof: Validating a Native CUDA Speculative Decoding Engine",
// section "The Context: Building a Native DDTree Engine from Scratch").
//
// Work decomposition (stream-K).  Query rows are (node, head) pairs with the
// head fastest, cut into 128-row tiles per request; the work of a row tile is
// its sequence of 64-key tiles.  Row tiles are ordered lane-major, r = rt * B
// + b (tile index within the request first), so that the pairs that run side
// by side hold the same tile index of neighbouring requests, or different
// tiles of one request at nearby keys; a request's cache is then shared in
// L2 by its row tiles instead of being swept once per tile.  All (row tile,
// key tile) units form one sequence and CTA pair c takes the W consecutive
// units [cW, (c+1)W),
// split into pieces at row-tile boundaries; each piece writes one partial
// (m, l, o_lat) that the combine kernel merges.  A small plan kernel computes
// the unit offsets, W and the partial slots (and each request's ancestor
// masks) on the device, so ragged batches are spread evenly.  A pair is a
// CLUSTER OF TWO CTAs that split the latent dimension:
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
// [448, 512).  Shared memory (all of the 227 KiB a CTA may have; the dynamic
// base must be 1 KiB aligned, which the kernel checks):
//   - a 5-slot TMA ring of the latent half of 64-key cache tiles (128-byte
//     swizzled 64-column chunks; the same slot is the K-major B operand of
//     Q.K^T and the MN-major B operand of P.V), freed by P.V;
//   - a 2-slot ring of the tiles' rope halves, freed as soon as Q.K^T read
//     them (the rope only enters Q.K^T);
//   - q_rope (this CTA's 32 rope dimensions of the piece's rows);
//   - TWO P tiles (K-major A operand of P.V), for even and odd key tiles, so
//     that the softmax of tile g writes P while P.V of tile g-1 still reads the
//     other one: only a rescale of O (rare with the lazy reference maxima)
//     waits for P.V of tile g-1;
//   - two receive buffers for the peer's scores, four for its rescale factors
//     and the reference maxima and row sums of the 64 rows each CTA owns.
// Key tiles are also prefetched into L2 a few tiles ahead of the ring.
//
// Warp roles (480 threads): warp 0 issues TMA loads; warp 1 owns TMEM and
// issues Q.K^T; warps 2-5 (one per lane quadrant) load each piece's Q into
// TMEM and quantise and send the peer's score rows; warps 6-13 (two per
// quadrant, taking even and odd tiles, four threads per row in the .16x256b
// TMEM layout, so row maxima and sums meet by warp shuffles; the running
// reference maxima pass between the two through shared memory) run the
// softmax of the CTA's own rows and write each piece's partial o_lat; warp 14
// issues P.V.  Every wait is bounded (2 s, or ~20 ms with
// KDTV_FLAG_TEST_STALL); on timeout the kernel records
// KDTV_ERR_DEVICE_TIMEOUT, lets in-flight copies land, drains its MMAs, frees
// TMEM and returns.

#include <cuda.h>
#include <cuda_fp16.h>

#include <atomic>

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
constexpr int kStages = 5;       // latent ring slots (freed by P.V)
constexpr int kRopeSlots = 2;    // rope ring slots (freed by Q.K^T)
constexpr int kPrefetch = 3;     // key tiles prefetched into L2 beyond the stages in flight
// The paged producer prefetches fewer: its page-table rows are loaded ahead
// as well, and a shorter distance measured faster (paged batch of 64 requests:
// 557.2, 549.6, 561.6, 563.5 and 574.8 us per call for 0, 2, 3, 6 and 10).
constexpr int kPagedPrefetch = 2;
constexpr int kRopeHalf = 32;    // rope dimensions per CTA (64-byte rows, 64-byte swizzle)
constexpr int kKVChunk = BN * CH * 2;   // 8 KiB
constexpr int kRopeChunk = BN * kRopeHalf * 2;            // 4 KiB of k_rope per key tile
constexpr int kStageBytes = 4 * kKVChunk;                 // 4 latent chunks of 64 columns
constexpr int kQRopeBytes = BM * kRopeHalf * 2;
constexpr int kPBytes = BM * BN * 2;    // the P tile: 128 rows x 64 keys bf16, 128B-swizzled
constexpr int kPQuadBytes = 16 * BN * 2;   // one quadrant's own P rows (contiguous, 2 KiB)
// Score exchange: the peer's 64 rows as fp16 in the receiving softmax
// thread's order: 16-byte chunk m (0..3) of thread t of quadrant q at
// ((q * 4 + m) * 32 + t) * 16, so one warp store is a contiguous 512-byte
// block; then one word per (q, t) holding its two rows' shifts.
constexpr int kRxData = 4 * 4 * 32 * 16;
constexpr int kRxBytes = kRxData + 4 * 8 * 4;   // + one shift word per row pair
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
constexpr int OFF_ROPE = OFF_KV + kStages * kStageBytes;       // [kRopeSlots] rope halves
constexpr int OFF_QR = OFF_ROPE + kRopeSlots * kRopeChunk;
constexpr int OFF_P = OFF_QR + kQRopeBytes;                    // two P tiles (even / odd key tiles)
constexpr int OFF_RX = OFF_P + 2 * kPBytes;                    // two receive buffers
constexpr int OFF_AF = OFF_RX + 2 * kRxStride;                 // [kAfBufs][64] floats (peer rows)
constexpr int OFF_MREF = OFF_AF + kAfBufs * 64 * 4;             // [2 parities][64] reference maxima
constexpr int OFF_LPART = OFF_MREF + 2 * 64 * 4;                // [m | l][64] of the odd-tile warps
constexpr int OFF_BAR = OFF_LPART + 2 * 64 * 4;
constexpr int kNumBars = 50;
constexpr int OFF_MISC = OFF_BAR + kNumBars * 8;
constexpr int kSmemBytes = OFF_MISC + 64;   // the base must be 1 KiB aligned (checked)
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(kStageBytes % 1024 == 0 && OFF_ROPE % 1024 == 0 && kRopeChunk % 1024 == 0 &&
              OFF_QR % 1024 == 0 && OFF_P % 1024 == 0 && kPBytes % 1024 == 0,
              "swizzled tiles need 1 KiB alignment");
static_assert(OFF_RX % 16 == 0 && kRxStride % 16 == 0 && OFF_AF % 16 == 0, "async store alignment");
static_assert(kThreads == 32 * (kWarpPV + 1), "warp roles");

// Barrier indices (derived from kStages so the groups never overlap).
enum Bar : int {
  B_QR_FULL = 0,
  B_Q_READY = 1,                     // 8 warps stored their part of Q in TMEM
  B_KV_FULL = 2,                     // [kStages] latent slot and its tile's rope slot landed
  B_KV_EMPTY = B_KV_FULL + kStages,  // [kStages] P.V read the latent slot
  B_R_EMPTY = B_KV_EMPTY + kStages,  // [kRopeSlots] Q.K^T read the rope slot
  B_S_FULL = B_R_EMPTY + kRopeSlots, // [2] Q.K^T of the tile completed
  B_S_FREE = B_S_FULL + 2,           // [2] senders and softmax read the scores
  B_RX_FULL = B_S_FREE + 2,          // [2] the peer's score rows landed in receive buffer g & 1 (tx)
  B_TX_OK = B_RX_FULL + 2,           // [2] the peer consumed what we sent into buffer g & 1 (remote)
  B_AF_FULL = B_TX_OK + 2,           // [kAfBufs] the peer's rescale factors landed (tx)
  B_P_FULL = B_AF_FULL + kAfBufs,    // [2] our softmax wrote its P rows of an even / odd tile
  B_P_RX = B_P_FULL + 2,             // [2] the peer's P rows of an even / odd tile landed (tx)
  B_P_EMPTY = B_P_RX + 2,            // [2] P.V of an even / odd tile completed in both CTAs
  B_O_FULL = B_P_EMPTY + 2,          // [2] a piece's O is complete, for the even / odd-tile warps
  B_MMA_DONE = B_O_FULL + 2,         // both MMA issuers drained
  B_STALL = B_MMA_DONE + 1,
  B_MREF = B_STALL + 1,              // [2 parities][4 quadrants] reference maxima published
  B_LSUM = B_MREF + 8,               // the odd-tile softmax warps published their (m, l)
  B_Q_EMPTY = B_LSUM + 1,            // Q.K^T of a piece completed: TMEM Q may be reloaded
  B_QR_EMPTY = B_Q_EMPTY + 1,        // ... and q_rope (CTA 0)
  B_O_FREE = B_QR_EMPTY + 1,         // the softmax warps wrote a piece's O out
  B_L_FREE = B_O_FREE + 1,           // the even-tile warps read the odd-tile (m, l)
  B_COUNT = B_L_FREE + 1
};
static_assert(B_COUNT <= kNumBars, "barrier slots");

// Wait sites (reported as the timeout detail).
enum Site { W_Q = 1, W_KV_FULL, W_KV_EMPTY, W_P_FULL, W_S_FULL, W_TX_OK, W_RX_FULL,
            W_P_EMPTY, W_O_FULL, W_STALL, W_DRAIN, W_S_FREE, W_AF, W_P_RX, W_MREF, W_LSUM,
            W_Q_EMPTY, W_O_FREE };

struct TcCfg {
  unsigned long long limit_ns; // bound on every wait
};

// ---- stream-K pieces ---------------------------------------------------------------------
// A piece: key tiles [t0, t1) of row tile r (request b, tile rt of it),
// written to partial slot `slot`; L is the request's prefix length.
struct Piece {
  int r, b, rt, t0, t1, slot, L;
};

__device__ __forceinline__ const int* sk_row(const Args& a, int r) { return a.sk + kSkHeader + 3 * r; }

__device__ __forceinline__ void piece_fill(const Args& a, int r, int beg, int end, int W, Piece& p) {
  const int* e = sk_row(a, r);
  p.r = r;
  p.rt = r / a.B;
  p.b = r - p.rt * a.B;
  p.t0 = beg - e[0];
  p.t1 = min(end, e[0] + e[1]) - e[0];
  p.slot = e[2] + (beg / W - e[0] / W);   // the first piece of r starts at S_r
  p.L = a.prefix_len[p.b];
}

// Offset (ints) in the plan of the per-pair first-piece records, 16-byte aligned.
__host__ __device__ __forceinline__ int sk_rec_off(int R, int pairs) {
  return (kSkHeader + 3 * R + pairs + 3) & ~3;
}

// First piece of CTA pair cl (unit range [beg, end)); false if the range is
// empty.  The plan stores, per pair, the row tile holding its first unit with
// that tile's {S, u, base} and prefix length, so one 32-byte load (beside the
// header's) starts the pair.
__device__ bool piece_first(const Args& a, int cl, int beg, int end, int W, Piece& p) {
  if (beg >= end) return false;
  const int R = a.B * a.rt_count;
  const int4* rec = reinterpret_cast<const int4*>(a.sk + sk_rec_off(R, a.sk_clusters)) + 2 * cl;
  const int4 v0 = rec[0], v1 = rec[1];
  const int r = v0.x;
  if (r < 0 || r >= R) return false;
  p.r = r;
  p.rt = r / a.B;
  p.b = r - p.rt * a.B;
  p.t0 = beg - v0.y;
  p.t1 = min(end, v0.y + v0.z) - v0.y;
  p.slot = v0.w + (beg / W - v0.y / W);
  p.L = v1.x;
  return true;
}

// The piece after p (it starts at the next non-empty row tile); false at the end.
__device__ bool piece_next(const Args& a, int end, int W, Piece& p) {
  const int R = a.sk[3];
  const int u = sk_row(a, p.r)[0] + p.t1;
  if (u >= end) return false;
  int r = p.r + 1;
  while (r < R && sk_row(a, r)[1] == 0) ++r;
  if (r >= R) return false;
  piece_fill(a, r, u, end, W, p);
  return true;
}

// The same walk over the boundary-aware plan, whose virtual sequence has a
// gap of sk_gap units before every non-empty row tile but the first: a
// pair's range may begin in the gap before its first row tile, and may end
// in the gap before the next.
__device__ __forceinline__ void piece_fill_g(const Args& a, int r, int beg, int end, int W, Piece& p) {
  const int* e = sk_row(a, r);
  const int x0 = max(beg, e[0]);
  p.r = r;
  p.rt = r / a.B;
  p.b = r - p.rt * a.B;
  p.t0 = x0 - e[0];
  p.t1 = min(end, e[0] + e[1]) - e[0];
  p.slot = e[2] + (x0 / W - e[0] / W);   // the first piece of r starts at vS_r
  p.L = a.prefix_len[p.b];
}

__device__ bool piece_first_g(const Args& a, int cl, int beg, int end, int W, Piece& p) {
  if (beg >= end) return false;
  const int R = a.B * a.rt_count;
  const int4* rec = reinterpret_cast<const int4*>(a.sk + sk_rec_off(R, a.sk_clusters)) + 2 * cl;
  const int4 v0 = rec[0], v1 = rec[1];
  const int r = v0.x;
  if (r < 0 || r >= R) return false;
  const int x0 = max(beg, v0.y);
  p.r = r;
  p.rt = r / a.B;
  p.b = r - p.rt * a.B;
  p.t0 = x0 - v0.y;
  p.t1 = min(end, v0.y + v0.z) - v0.y;
  p.slot = v0.w + (x0 / W - v0.y / W);
  p.L = v1.x;
  return p.t0 < p.t1;
}

__device__ bool piece_next_g(const Args& a, int end, int W, Piece& p) {
  const int R = a.sk[3];
  const int u = sk_row(a, p.r)[0] + p.t1;
  if (u >= end) return false;
  int r = p.r + 1;
  while (r < R && sk_row(a, r)[1] == 0) ++r;
  if (r >= R || sk_row(a, r)[0] >= end) return false;
  piece_fill_g(a, r, u, end, W, p);
  return true;
}

template <bool kGap>
__device__ __forceinline__ bool first_piece(const Args& a, int cl, int beg, int end, int W, Piece& p) {
  if constexpr (kGap) return piece_first_g(a, cl, beg, end, W, p);
  else return piece_first(a, cl, beg, end, W, p);
}

template <bool kGap>
__device__ __forceinline__ bool next_piece(const Args& a, int end, int W, Piece& p) {
  if constexpr (kGap) return piece_next_g(a, end, W, p);
  else return piece_next(a, end, W, p);
}

// Keeps a value computed before the next wait: the compiler may otherwise
// sink arithmetic whose result is only used after a wait below it, onto the
// critical path that the wait ends.
// Compact index of a softmax row among a CTA's 64 own (or the peer's 64) rows:
// rows 32q + 16 rank + i of quadrant q map to 16q + i.
__device__ __forceinline__ int crow(int r) { return 16 * (r >> 5) + (r & 15); }

__device__ __forceinline__ void pin(uint32_t& x) { asm volatile("" : "+r"(x)); }
__device__ __forceinline__ void pin(float& x) { asm volatile("" : "+f"(x)); }

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

// Stores 32 * nch32 O columns of the 32 rows of a warp's TMEM lane quadrant
// as bf16 (ta0: TMEM address of the quadrant's first lane and column; dst0:
// row 0, column 0 of the destination, rows d_c elements apart; rows >= nvalid
// are skipped).  Reads the .16x256b layout (rows t/4 and t/4 + 8 of each
// 16-row half, column pairs 8k + 2c); a pair exchange between threads c and
// c ^ 1 gives each thread 4 consecutive columns, so one warp store covers 32
// contiguous bytes of each of 8 rows.  Out of line: it runs once per piece.
__device__ __noinline__ void store_o_quadrant(uint32_t ta0, __nv_bfloat16* dst0, int d_c, int nvalid,
                                              int nch32) {
  const int lane = threadIdx.x & 31, c = lane & 3;
  const bool odd = c & 1;
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    const int r = 16 * hh + (lane >> 2);                 // rows r, r + 8
    const bool wa = r < nvalid, wb = r + 8 < nvalid;
    __nv_bfloat16* pra = dst0 + (long long)r * d_c + (odd ? 2 * c + 6 : 2 * c);
    __nv_bfloat16* prb = pra + 8 * d_c;
    const uint32_t ta = ta0 + (static_cast<uint32_t>(16 * hh) << 16);
#pragma unroll 1
    for (int cc = 0; cc < nch32; ++cc) {                 // 32 columns per load
      uint32_t v[16];
      tmem_ld_16x256b_x4(ta + 32 * cc, v);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 4; k += 2) {
        // rows a (v[4k], v[4k+1]) and b (v[4k+2], v[4k+3]) of pairs k, k+1
        const uint32_t sa0 = odd ? v[4 * k] : v[4 * k + 4], sa1 = odd ? v[4 * k + 1] : v[4 * k + 5];
        const uint32_t sb0 = odd ? v[4 * k + 2] : v[4 * k + 6], sb1 = odd ? v[4 * k + 3] : v[4 * k + 7];
        const uint32_t ra0 = __shfl_xor_sync(0xffffffffu, sa0, 1);
        const uint32_t ra1 = __shfl_xor_sync(0xffffffffu, sa1, 1);
        const uint32_t rb0 = __shfl_xor_sync(0xffffffffu, sb0, 1);
        const uint32_t rb1 = __shfl_xor_sync(0xffffffffu, sb1, 1);
        const uint2 oa = odd ? make_uint2(pack_bf16x2(__uint_as_float(ra0), __uint_as_float(ra1)),
                                          pack_bf16x2(__uint_as_float(v[4 * k + 4]), __uint_as_float(v[4 * k + 5])))
                             : make_uint2(pack_bf16x2(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1])),
                                          pack_bf16x2(__uint_as_float(ra0), __uint_as_float(ra1)));
        const uint2 ob = odd ? make_uint2(pack_bf16x2(__uint_as_float(rb0), __uint_as_float(rb1)),
                                          pack_bf16x2(__uint_as_float(v[4 * k + 6]), __uint_as_float(v[4 * k + 7])))
                             : make_uint2(pack_bf16x2(__uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3])),
                                          pack_bf16x2(__uint_as_float(rb0), __uint_as_float(rb1)));
        if (wa) *reinterpret_cast<uint2*>(pra + 32 * cc + 8 * k) = oa;
        if (wb) *reinterpret_cast<uint2*>(prb + 32 * cc + 8 * k) = ob;
      }
    }
  }
}

template <bool kPaged, bool kGap>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_qrope,
               const __grid_constant__ CUtensorMap tm_ckv,
               const __grid_constant__ CUtensorMap tm_krope, const Args a, const TcCfg cfg) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (sbase & 1023u) {   // swizzled tiles need a 1 KiB aligned base (no slack is reserved)
    if (tid == 0) record_error(a.status, KDTV_ERR_UNSUPPORTED, 0xA11u);
    return;
  }
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int cl = blockIdx.x >> 1;                  // this CTA pair
  volatile int* misc = reinterpret_cast<volatile int*>(sm + OFF_MISC);
  auto BAR = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8u * i; };
  DeviceStatus* st = a.status;
  const uint64_t limit = cfg.limit_ns;
  grid_dep_launch();   // the combine kernel may start its weight loads early

  // ---- prologue: barriers, TMEM ------------------------------------------------------
  if (tid == 0) {
    mbar_init(BAR(B_QR_FULL), 1);
    mbar_init(BAR(B_Q_READY), 4);         // the 4 sender warps stored Q
    for (int i = 0; i < kStages; ++i) {
      mbar_init(BAR(B_KV_FULL + i), 1);
      mbar_init(BAR(B_KV_EMPTY + i), 1);
    }
    for (int i = 0; i < kRopeSlots; ++i) mbar_init(BAR(B_R_EMPTY + i), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(B_S_FULL + i), 1);
      mbar_init(BAR(B_S_FREE + i), 8);    // 4 sender + 4 softmax warps read the scores
      mbar_init(BAR(B_P_FULL + i), 4);    // the tile's 4 softmax warps
      mbar_init(BAR(B_P_RX + i), 1);      // armed with expect_tx; filled by the peer's bulk copies
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(B_RX_FULL + i), 1);   // armed with expect_tx; filled by the peer's st.async
      mbar_init(BAR(B_TX_OK + i), 4);     // one arrival per peer softmax warp of the tile
    }
    for (int i = 0; i < kAfBufs; ++i) mbar_init(BAR(B_AF_FULL + i), 1);
    // P.V commits of both CTAs (multicast), one barrier per tile parity: each
    // softmax warp waits only for the other parity's tiles, so it sees every
    // phase of the barrier it waits on in order.
    mbar_init(BAR(B_P_EMPTY + 0), 2);
    mbar_init(BAR(B_P_EMPTY + 1), 2);
    mbar_init(BAR(B_O_FULL + 0), 1);
    mbar_init(BAR(B_O_FULL + 1), 1);
    mbar_init(BAR(B_MMA_DONE), 2);
    mbar_init(BAR(B_STALL), 1);
    for (int i = 0; i < 8; ++i) mbar_init(BAR(B_MREF + i), 1);
    mbar_init(BAR(B_LSUM), 4);
    mbar_init(BAR(B_Q_EMPTY), 1);
    mbar_init(BAR(B_QR_EMPTY), 1);
    mbar_init(BAR(B_O_FREE), 4);          // the 4 softmax warps that wrote a piece's O out
    mbar_init(BAR(B_L_FREE), 4);          // the even-tile warps read the hand-over
    mbar_expect_tx(BAR(B_RX_FULL + 0), kRxBytes);   // the score exchanges of tiles 0 and 1
    mbar_expect_tx(BAR(B_RX_FULL + 1), kRxBytes);
    for (int i = 0; i < kAfBufs; ++i) mbar_expect_tx(BAR(B_AF_FULL + i), kAfBytes);
    mbar_expect_tx(BAR(B_P_RX + 0), 4 * kPQuadBytes);   // the peer's P rows of tiles 0 and 1
    mbar_expect_tx(BAR(B_P_RX + 1), 4 * kPQuadBytes);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + OFF_MISC, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();   // the peer's barriers are initialised before any remote access

  // The plan, the ancestor masks and q_lat are written by the kernels before
  // this one.  The pair's unit range is [beg, end).
  grid_dep_wait();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const int nrows = a.N * a.H;
  const int U = a.sk[0], W = a.sk[1];              // U: the (virtual) length of the sequence
  const long long beg_ll = (long long)cl * W;
  const int beg = beg_ll < U ? (int)beg_ll : U;
  const int end = (long long)beg + W < U ? beg + W : U;
  // key tiles of this pair: its range, less the gaps of a boundary-aware plan
  // (counted by the plan kernel)
  int G;
  if constexpr (kGap)
    G = beg < end ? reinterpret_cast<const int4*>(a.sk + sk_rec_off(a.B * a.rt_count, a.sk_clusters))[2 * cl + 1].y
                  : 0;
  else
    G = end - beg;

  if (warp == 0) {
    // ---- TMA producer --------------------------------------------------------------
    if (lane == 0 && G > 0) {
      prefetch_tmap(&tm_ckv);
      // Cache row of key k of request b (paged: through the page table; a page
      // id outside [0, num_pages) is reported and read as page 0).
      auto key_row = [&](int b, int k) -> int {
        if (!a.page_size) return b * a.t_stride + k;
        const int page = a.page_table[(long long)b * a.max_pages + k / a.page_size];
        if (page < 0 || page >= a.num_pages) {
          record_error(st, KDTV_ERR_BAD_PAGE, (unsigned)b);
          return 0;
        }
        return page * a.page_size;
      };
      auto prefetch = [&](int b, int k) {
        const int row = key_row(b, k);
        for (int c = 0; c < 4; ++c) tma_prefetch_2d(&tm_ckv, (int)rank * kHalf + c * CH, row);
        tma_prefetch_2d(&tm_krope, kRopeHalf * (int)rank, row);
      };
      auto prefetch_row = [&](int row) {
        for (int c = 0; c < 4; ++c) tma_prefetch_2d(&tm_ckv, (int)rank * kHalf + c * CH, row);
        tma_prefetch_2d(&tm_krope, kRopeHalf * (int)rank, row);
      };
      Piece pc;
      bool have = first_piece<kGap>(a, cl, beg, end, W, pc);
      int g = 0, pi = 0, issued = 0, qr_issued = 0;
      bool alive = true;
      while (alive && have) {
        {   // this CTA's q_rope half of the piece's rows, once Q.K^T of the previous piece is done
          if (pi >= 1 && !wait(BAR(B_QR_EMPTY), (pi - 1) & 1, st, limit, W_Q_EMPTY)) break;
          ++qr_issued;
          mbar_expect_tx(BAR(B_QR_FULL), kQRopeBytes);
          tma_load_2d(sbase + OFF_QR, &tm_qrope, BAR(B_QR_FULL), kRopeHalf * (int)rank,
                      (int)((long long)pc.b * nrows + pc.rt * BM));
        }
        if constexpr (kPaged) {
          // Paged: the cache rows of the piece's next kAhead + 1 tiles (one
          // page-table load each), shifted by one per tile, so that neither
          // tile j's copies nor the L2 prefetch kAhead tiles ahead wait for a
          // page-table load; the row kAhead + 1 ahead is loaded meanwhile.
          constexpr int kAhead = kStages + kPagedPrefetch;
          int rows[kAhead + 2];
#pragma unroll
          for (int i = 0; i <= kAhead; ++i) rows[i] = pc.t0 + i < pc.t1 ? key_row(pc.b, (pc.t0 + i) * BN) : 0;
          rows[kAhead + 1] = 0;
#pragma unroll
          for (int i = kStages; i < kAhead; ++i)
            if (pc.t0 + i < pc.t1) prefetch_row(rows[i]);
          for (int j = pc.t0; j < pc.t1; ++j, ++g) {
            const int stg = g % kStages, rs = g % kRopeSlots;
            if (j + kAhead + 1 < pc.t1) rows[kAhead + 1] = key_row(pc.b, (j + kAhead + 1) * BN);
            if (g >= kStages &&
                !wait(BAR(B_KV_EMPTY + stg), ((g / kStages) - 1) & 1, st, limit, W_KV_EMPTY)) {
              alive = false;
              break;
            }
            if (g >= kRopeSlots &&
                !wait(BAR(B_R_EMPTY + rs), ((g / kRopeSlots) - 1) & 1, st, limit, W_KV_EMPTY)) {
              alive = false;
              break;
            }
            mbar_expect_tx(BAR(B_KV_FULL + stg), kStageBytes + kRopeChunk);
            const uint32_t dst = sbase + OFF_KV + stg * kStageBytes;
            for (int c = 0; c < 4; ++c)
              tma_load_2d(dst + c * kKVChunk, &tm_ckv, BAR(B_KV_FULL + stg),
                          (int)rank * kHalf + c * CH, rows[0]);
            tma_load_2d(sbase + OFF_ROPE + rs * kRopeChunk, &tm_krope, BAR(B_KV_FULL + stg),
                        kRopeHalf * (int)rank, rows[0]);
            issued = g + 1;
            if (j + kAhead < pc.t1) prefetch_row(rows[kAhead]);
#pragma unroll
            for (int i = 0; i <= kAhead; ++i) rows[i] = rows[i + 1];
          }
        } else {
          for (int j = pc.t0 + kStages; j < pc.t0 + kStages + kPrefetch && j < pc.t1; ++j)
            prefetch(pc.b, j * BN);
          for (int j = pc.t0; j < pc.t1; ++j, ++g) {
            const int stg = g % kStages, rs = g % kRopeSlots;
            if (g >= kStages &&
                !wait(BAR(B_KV_EMPTY + stg), ((g / kStages) - 1) & 1, st, limit, W_KV_EMPTY)) {
              alive = false;
              break;
            }
            if (g >= kRopeSlots &&
                !wait(BAR(B_R_EMPTY + rs), ((g / kRopeSlots) - 1) & 1, st, limit, W_KV_EMPTY)) {
              alive = false;
              break;
            }
            const int row = key_row(pc.b, j * BN);
            mbar_expect_tx(BAR(B_KV_FULL + stg), kStageBytes + kRopeChunk);
            const uint32_t dst = sbase + OFF_KV + stg * kStageBytes;
            for (int c = 0; c < 4; ++c)
              tma_load_2d(dst + c * kKVChunk, &tm_ckv, BAR(B_KV_FULL + stg),
                          (int)rank * kHalf + c * CH, row);
            tma_load_2d(sbase + OFF_ROPE + rs * kRopeChunk, &tm_krope, BAR(B_KV_FULL + stg),
                        kRopeHalf * (int)rank, row);
            issued = g + 1;
            if (j + kStages + kPrefetch < pc.t1) prefetch(pc.b, (j + kStages + kPrefetch) * BN);
          }
        }
        ++pi;
        have = next_piece<kGap>(a, end, W, pc);
      }
      // Drain: every issued copy has landed before this CTA may exit.
      if (qr_issued >= 1) wait(BAR(B_QR_FULL), (qr_issued - 1) & 1, st, limit, W_DRAIN);
      for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j)
        wait(BAR(B_KV_FULL + j % kStages), (j / kStages) & 1, st, limit, W_DRAIN);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- Q.K^T issuer (also owns TMEM) ------------------------------------------------
    if (lane == 0 && G > 0) {
      constexpr uint32_t kIdescQK = idesc_bf16(BM, BN, 0, 0);
      Piece pc;
      bool have = first_piece<kGap>(a, cl, beg, end, W, pc);
      int g = 0, pi = 0;
      bool alive = true;
      while (alive && have) {
        alive = wait(BAR(B_Q_READY), pi & 1, st, limit, W_Q);
        if (alive) alive = wait(BAR(B_QR_FULL), pi & 1, st, limit, W_Q);
        for (int j = pc.t0; alive && j < pc.t1; ++j, ++g) {
          const int stg = g % kStages, buf = g & 1;
          alive = wait(BAR(B_KV_FULL + stg), (g / kStages) & 1, st, limit, W_KV_FULL);
          // the score buffer is rewritten: senders and softmax must have read tile g-2
          if (alive && g >= 2)
            alive = wait(BAR(B_S_FREE + buf), ((g >> 1) - 1) & 1, st, limit, W_S_FREE);
          if (!alive) break;
          tc_fence_after();
          const uint32_t d = tmem + kColS + 64 * buf;
          const uint32_t kv = sbase + OFF_KV + stg * kStageBytes;
#pragma unroll
          for (int kk = 0; kk < kHalf / 16; ++kk) {     // latent half: A = q_lat in TMEM
            uint64_t bd = smem_desc(kv + (kk >> 2) * kKVChunk + (kk & 3) * 32, 16, 1024);
            mma_bf16_ts(d, tmem + kColQ + 8 * kk, bd, kIdescQK, kk > 0);
          }
          const uint32_t kr = sbase + OFF_ROPE + (g % kRopeSlots) * kRopeChunk;
#pragma unroll
          for (int kk = 0; kk < kRopeHalf / 16; ++kk) {   // rope half: A = q_rope half in smem
            uint64_t ad = smem_desc_sw64(sbase + OFF_QR + kk * 32, 16, 512);
            uint64_t bd = smem_desc_sw64(kr + kk * 32, 16, 512);
            mma_bf16(d, ad, bd, kIdescQK, 1);
          }
          mma_commit(BAR(B_S_FULL + buf));
          mma_commit(BAR(B_R_EMPTY + g % kRopeSlots));   // the rope slot may be refilled
        }
        if (!alive) break;
        mma_commit(BAR(B_Q_EMPTY));                 // Q (and q_rope) may be reloaded
        mma_commit(BAR(B_QR_EMPTY));
        ++pi;
        have = next_piece<kGap>(a, end, W, pc);
      }
      mma_commit(BAR(B_MMA_DONE));                 // drain every issued MMA (both issuers)
      wait(BAR(B_MMA_DONE), 0, st, limit, W_DRAIN);
    }
    __syncwarp();
  } else if (warp == kWarpPV) {
    // ---- P.V issuer: O_c += P . c_kv[:, 256c : 256c+256] ------------------------------
    if (lane == 0 && G > 0) {
      constexpr uint32_t kIdescPV = idesc_bf16(BM, kHalf, 0, 1);
      Piece pc;
      bool have = first_piece<kGap>(a, cl, beg, end, W, pc);
      int g = 0, pi = 0;
      // phases of B_P_RX + b armed and consumed so far (both armed at set-up)
      int p_armed0 = 1, p_armed1 = G > 1 ? 1 : 0, p_used0 = 0, p_used1 = 0;
      bool alive = true;
      while (alive && have) {
        for (int j = pc.t0; j < pc.t1; ++j, ++g) {
          const int stg = g % kStages, pb = g & 1;
          alive = wait_spin(BAR(B_P_FULL + pb), (g >> 1) & 1, st, limit, W_P_FULL);
          if (alive) alive = wait_spin(BAR(B_P_RX + pb), (g >> 1) & 1, st, limit, W_P_RX);
          if (alive) (pb ? p_used1 : p_used0) += 1;
          // already complete (Q.K^T of tile g read this stage); orders the TMA data
          if (alive) alive = wait(BAR(B_KV_FULL + stg), (g / kStages) & 1, st, limit, W_KV_FULL);
          // the first P.V of a piece overwrites O: the previous piece must be written out
          if (alive && j == pc.t0 && pi >= 1)
            alive = wait(BAR(B_O_FREE), (pi - 1) & 1, st, limit, W_O_FREE);
          if (!alive) break;
          // arm the peer's P rows of tile g+2 (same buffer) before our commit lets the
          // peer send them
          if (g + 2 < G) {
            mbar_expect_tx(BAR(B_P_RX + pb), 4 * kPQuadBytes);
            (pb ? p_armed1 : p_armed0) += 1;
          }
          tc_fence_after();
          const uint32_t kv = sbase + OFF_KV + stg * kStageBytes;
          const uint32_t pt = sbase + OFF_P + pb * kPBytes;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            // A = P (K-major, 128B rows); B = V = c_kv columns of this CTA,
            // MN-major: 64-column chunks kKVChunk apart (LBO), 8-key groups 1 KiB apart (SBO).
            uint64_t ad = smem_desc(pt + kk * 32, 16, 1024);
            uint64_t bd = smem_desc(kv + kk * 16 * 128, kKVChunk, 1024);
            mma_bf16(tmem + kColO, ad, bd, kIdescPV, (j > pc.t0 || kk > 0));
          }
          mma_commit(BAR(B_KV_EMPTY + stg));
          mma_commit_multicast(BAR(B_P_EMPTY + (g & 1)), 0x3);   // both CTAs may overwrite P
        }
        if (!alive) break;
        // the piece's O is complete: tell the warps that write it out (those that
        // took the piece's last tile when another piece follows, else all)
        have = next_piece<kGap>(a, end, W, pc);
        if (!have || ((g - 1) & 1) == 0) mma_commit(BAR(B_O_FULL + 0));
        if (!have || ((g - 1) & 1) == 1) mma_commit(BAR(B_O_FULL + 1));
        ++pi;
      }
      // After an abort: let the peer's P rows of an armed, unconsumed phase land.
      if (!alive) {
        if (p_armed0 > p_used0) drain_wait(BAR(B_P_RX + 0), (p_armed0 - 1) & 1, 200000ull);
        if (p_armed1 > p_used1) drain_wait(BAR(B_P_RX + 1), (p_armed1 - 1) & 1, 200000ull);
      }
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
    Piece pc;
    bool have = first_piece<kGap>(a, cl, beg, end, W, pc);

    if (!is_softmax) {
      // ---- sender: each piece's Q into TMEM; the peer's score rows -> its receive buffer --
      int g = 0, pi = 0;
      while (alive && have) {
        // Q of this piece (row 32q + lane, 256 latent columns of this CTA's half as
        // 128 bf16 pairs, .32x32b layout) once Q.K^T of the previous piece is done.
        if (pi >= 1) {
          alive = __all_sync(0xffffffffu, wait(BAR(B_Q_EMPTY), (pi - 1) & 1, st, limit, W_Q_EMPTY));
          if (!alive) break;
        }
        {
          const int rq = pc.rt * BM + 32 * q + lane;
          const bool vq = rq < nrows;
          const uint4* src = reinterpret_cast<const uint4*>(
              static_cast<const __nv_bfloat16*>(a.q_lat) +
              ((long long)pc.b * nrows + (vq ? rq : 0)) * 512 + rank * kHalf);
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            uint32_t w[32];
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              uint4 x = vq ? src[8 * h + v] : make_uint4(0u, 0u, 0u, 0u);
              w[4 * v] = x.x; w[4 * v + 1] = x.y; w[4 * v + 2] = x.z; w[4 * v + 3] = x.w;
            }
            tmem_st32u(tmem + lane32 + kColQ + 32 * h, w);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B_Q_READY));
        }
        for (int j = pc.t0; alive && j < pc.t1; ++j, ++g) {
          const int buf = g & 1;
          alive = __all_sync(0xffffffffu, wait(BAR(B_S_FULL + buf), (g >> 1) & 1, st, limit, W_S_FULL));
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
          uint32_t w[16];                          // rows a then b, key pairs 8k + 2c
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            __half2 ha = __floats2half2_rn(__uint_as_float(v[4 * k]) * sca,
                                           __uint_as_float(v[4 * k + 1]) * sca);
            __half2 hb = __floats2half2_rn(__uint_as_float(v[4 * k + 2]) * scb,
                                           __uint_as_float(v[4 * k + 3]) * scb);
            w[k] = *reinterpret_cast<uint32_t*>(&ha);
            w[8 + k] = *reinterpret_cast<uint32_t*>(&hb);
          }
#pragma unroll
          for (int k = 0; k < 16; ++k) pin(w[k]);
          // the peer has consumed what we sent into this receive buffer two tiles ago
          if (g >= 2) {
            alive = __all_sync(0xffffffffu, wait(BAR(B_TX_OK + buf), ((g >> 1) - 1) & 1, st, limit,
                                                 W_TX_OK));
            if (!alive) break;
          }
          const uint32_t rxp = mapa(sbase + OFF_RX + buf * kRxStride, peer);
          const uint32_t rxfull_remote = mapa(BAR(B_RX_FULL + buf), peer);
#pragma unroll
          for (int m = 0; m < 4; ++m)
            st_async_v4u(rxp + ((q * 4 + m) * 32 + lane) * 16, w[4 * m], w[4 * m + 1], w[4 * m + 2],
                         w[4 * m + 3], rxfull_remote);
          if (c == 0)   // the row pair's four threads hold the same shifts
            st_async_u32(rxp + kRxData + (q * 8 + (lane >> 2)) * 4,
                         ((uint32_t)sha & 0xffffu) | ((uint32_t)shb << 16), rxfull_remote);
        }
        ++pi;
        have = next_piece<kGap>(a, end, W, pc);
      }
    } else {
      // ---- softmax of this CTA's rows ra = own_base + t/4, rb = ra + 8 ---------------
      // Thread t holds keys 8k + 2c, 8k + 2c + 1 (k = 0..7) of each 64-key tile.
      const int ra = own_base + (lane >> 2), rb = ra + 8;
      const float sl2 = a.scale * 1.4426950408889634f;   // scores in log2 units
      const float* af = reinterpret_cast<const float*>(sm + OFF_AF);
      float* mref = reinterpret_cast<float*>(sm + OFF_MREF);
      float* lpart = reinterpret_cast<float*>(sm + OFF_LPART);
      const int lead = 6 + 4 * par;               // the warp that re-arms this parity's receive barriers

      if (G > 0 && (a.flags & KDTV_FLAG_TEST_STALL))
        alive = __all_sync(0xffffffffu, wait(BAR(B_STALL), 0, st, limit, W_STALL));

      // This warp takes the tiles g = par, par + 2, ... of the pair's sequence; the
      // running reference maxima pass between the two warps of the quadrant
      // through shared memory (restarting at -inf with every piece).
      int g = 0, pi = 0;
      int next_rx = par;                          // first tile whose scores this warp has not received
      int next_af = par;
      // Writes O columns [col0, col0 + 32 nch32) of rows 32q .. 32q+31 of a piece
      // (row tile rt, partial slot `slot`) once its P.V completed, then frees O.
      int o_waits = 0;                            // phases of B_O_FULL + par consumed so far
      auto write_o = [&](int slot, int rt, bool free_o, int col0, int nch32) -> bool {
        if (!__all_sync(0xffffffffu, wait(BAR(B_O_FULL + par), o_waits & 1, st, limit, W_O_FULL)))
          return false;
        ++o_waits;
        tc_fence_after();
        store_o_quadrant(tmem + (static_cast<uint32_t>(32 * q) << 16) + kColO + col0,
                         a.part_o16 + ((long long)slot * BM + 32 * q) * a.d_c + rank * kHalf + col0, a.d_c,
                         nrows - (rt * BM + 32 * q), nch32);
        tc_fence_before();
        __syncwarp();
        if (free_o && lane == 0) mbar_arrive(BAR(B_O_FREE));   // the next piece may overwrite O
        return true;
      };
      while (alive && have) {
        const bool va = pc.rt * BM + ra < nrows, vb = pc.rt * BM + rb < nrows;
        const int L = pc.L, T = L + a.N;
        const int k1 = min(T, pc.t1 * BN);
        // Reference maxima last used by this warp and its row sums relative to them.
        float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
        for (int j = pc.t0; j < pc.t1; ++j, ++g) {
          if ((g & 1) != par) continue;
          const int buf = g & 1;
          alive = __all_sync(0xffffffffu, wait(BAR(B_S_FULL + buf), (g >> 1) & 1, st, limit, W_S_FULL));
          if (!alive) break;
          tc_fence_after();
          uint32_t v[32];                          // own partial scores (fp32)
          tmem_ld_16x256b_x8(tmem + lane_own + kColS + 64 * buf, v);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B_S_FREE + buf));   // QK^T of tile g+2 may overwrite

          // + the peer's partial scores for our rows (its st.async filled rx[buf]);
          // the lead warp arms this buffer for tile g+2
          alive = __all_sync(0xffffffffu,
                             wait<true>(BAR(B_RX_FULL + buf), (g >> 1) & 1, st, limit, W_RX_FULL));
          if (!alive) break;
          next_rx = g + 2;
          if (warp == lead && lane == 0 && g + 2 < G) mbar_expect_tx(BAR(B_RX_FULL + buf), kRxBytes);
          float sa[16], sb[16];
          {
            const uint32_t rxb = sbase + OFF_RX + buf * kRxStride;
            uint32_t pw[16], shw;
#pragma unroll
            for (int m = 0; m < 4; ++m)
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(pw[4 * m]), "=r"(pw[4 * m + 1]), "=r"(pw[4 * m + 2]), "=r"(pw[4 * m + 3])
                           : "r"(rxb + ((q * 4 + m) * 32 + lane) * 16) : "memory");
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(shw) : "r"(rxb + kRxData + (q * 8 + (lane >> 2)) * 4)
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
          // consumed: the peer may overwrite the buffer (release: after our reads)
          if (lane == 0) mbar_arrive_remote_relaxed(mapa(BAR(B_TX_OK + buf), peer));

          // visibility mask (only tiles that reach past the prefix, or rows past the end);
          // each row's ancestor mask is one 16-byte load
          const int tb = j * BN;
          if (!(va && vb && tb + BN <= L)) {
            const uint4* ag = reinterpret_cast<const uint4*>(a.anc_g) + (long long)pc.b * a.N;
            const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
            const uint4 mka = va ? ag[(pc.rt * BM + ra) / a.H] : zero4;
            const uint4 mkb = vb ? ag[(pc.rt * BM + rb) / a.H] : zero4;
#pragma unroll
            for (int rsel = 0; rsel < 2; ++rsel) {
              const bool vrow = rsel ? vb : va;
              const uint4 mk = rsel ? mkb : mka;
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
                    const int wsel = jn >> 5;
                    const uint32_t w = wsel == 0 ? mk.x : (wsel == 1 ? mk.y : (wsel == 2 ? mk.z : mk.w));
                    vis = (w >> (jn & 31)) & 1u;
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

          // the reference maxima after tile g-1 (the other warp of this quadrant);
          // its phase is consumed on every tile, the value only within a piece
          float mpa = -INFINITY, mpb = -INFINITY;
          pin(mta);
          pin(mtb);
          if (g >= 1) {
            alive = __all_sync(0xffffffffu, wait(BAR(B_MREF + 4 * (par ^ 1) + q), ((g - 1) >> 1) & 1,
                                                 st, limit, W_MREF));
            if (!alive) break;
            if (j > pc.t0) {
              mpa = mref[(par ^ 1) * 64 + crow(ra)];
              mpb = mref[(par ^ 1) * 64 + crow(rb)];
            }
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
            mref[par * 64 + crow(ra)] = mna;
            mref[par * 64 + crow(rb)] = mnb;
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
            const int afb = g & (kAfBufs - 1);
            const uint32_t afr = mapa(BAR(B_AF_FULL + afb), peer);
            if (c < 2)
              st_async_u32(mapa(sbase + OFF_AF + (afb * 64 + crow(c ? rb : ra)) * 4, peer),
                           __float_as_uint(c ? alpha_b : alpha_a), afr);
          }
          const float nma = m_a == -INFINITY ? 0.f : -m_a, nmb = m_b == -INFINITY ? 0.f : -m_b;
          uint32_t pa[8], pb[8];                   // bf16 pairs of P: keys 8k + 2c, +1
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

#pragma unroll
          for (int k = 0; k < 8; ++k) {
            pin(pa[k]);
            pin(pb[k]);
          }
          pin(l_a);
          pin(l_b);
          // P tile g & 1 is free once P.V of tile g-2 completed in both CTAs (this
          // parity's barrier, whose phases this warp observes in order)
          const uint32_t pbuf = OFF_P + (g & 1) * kPBytes;
          if (g >= 2) {
            alive = __all_sync(0xffffffffu, wait(BAR(B_P_EMPTY + (g & 1)), ((g - 2) >> 1) & 1, st,
                                                 limit, W_P_EMPTY));
            if (!alive) break;
          }
          // P rows ra, rb: the pair for keys 8k + 2c is 4 bytes at offset 4c of the
          // row's 16-byte chunk k, stored 128B-swizzled (chunk k of row r at k ^ (r & 7)).
          {
            const uint32_t prow_a = sbase + pbuf + ra * 128 + 4 * c;
            const uint32_t prow_b = sbase + pbuf + rb * 128 + 4 * c;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              asm volatile("st.shared.b32 [%0], %1;" :: "r"(prow_a + ((k ^ (ra & 7)) << 4)), "r"(pa[k]) : "memory");
              asm volatile("st.shared.b32 [%0], %1;" :: "r"(prow_b + ((k ^ (rb & 7)) << 4)), "r"(pb[k]) : "memory");
            }
          }
          fence_async_smem();                       // visible to the tensor core and the copy engine
          __syncwarp();
          if (lane == 0) {
            // our 16 rows of this quadrant are one contiguous 2 KiB block
            const uint32_t off = pbuf + own_base * 128;
            bulk_copy_to_peer(mapa(sbase + off, peer), sbase + off, kPQuadBytes,
                              mapa(BAR(B_P_RX + (g & 1)), peer));
          }
          // the peer's rescale factors for its rows of this quadrant: both halves of
          // O must carry the same reference maxima before P.V of this tile
          const int afb = g & (kAfBufs - 1);
          alive = __all_sync(0xffffffffu,
                             wait<true>(BAR(B_AF_FULL + afb), (g / kAfBufs) & 1, st, limit, W_AF));
          if (!alive) break;
          next_af = g + 2;
          const float qa = af[afb * 64 + crow(ra)], qb = af[afb * 64 + crow(rb)];   // rows ra ^ 16, rb ^ 16
          if (warp == lead && lane == 0 && g + kAfBufs < G)
            mbar_expect_tx(BAR(B_AF_FULL + afb), kAfBytes);
          if (__any_sync(0xffffffffu, alpha_a != 1.f || alpha_b != 1.f || qa != 1.f || qb != 1.f)) {
            // O is stable once P.V of tile g-1 completed in both CTAs.  The other
            // parity's barrier cannot be a phase ahead of tile g-1 here (P.V of
            // tile g+1 follows ours), nor behind it (P.V of tile g-2 completed).
            if (g >= 1) {
              alive = __all_sync(0xffffffffu, wait(BAR(B_P_EMPTY + ((g - 1) & 1)), ((g - 1) >> 1) & 1,
                                                   st, limit, W_P_EMPTY));
              if (!alive) break;
            }
            tc_fence_after();
            rescale_o_rows(tmem + lane_own + kColO, alpha_a, alpha_b);
            rescale_o_rows(tmem + lane_peer + kColO, qa, qb);
            tmem_wait_st();
            tc_fence_before();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B_P_FULL + (g & 1)));
        }
        if (!alive) break;

        // ---- end of the piece: (m, l) of our rows and the unnormalised o_lat half -------
        // Row sums meet across the row's four threads; the odd-tile warp hands its
        // (m, l) to the even-tile warp, which merges them (the later reference is
        // the larger) and writes the row's (m, l) to the piece's slot.
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
        if (par == 1) {
          // the even-tile warps have read the previous piece's hand-over
          if (pi >= 1) {
            alive = __all_sync(0xffffffffu, wait(BAR(B_L_FREE), (pi - 1) & 1, st, limit, W_LSUM));
            if (!alive) break;
          }
          if (c == 0) {
            lpart[crow(ra)] = m_a; lpart[64 + crow(ra)] = l_a;
            lpart[crow(rb)] = m_b; lpart[64 + crow(rb)] = l_b;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B_LSUM));
        } else {
          alive = __all_sync(0xffffffffu, wait(BAR(B_LSUM), pi & 1, st, limit, W_LSUM));
          if (!alive) break;
          const float m1a = lpart[crow(ra)], l1a = lpart[64 + crow(ra)];
          const float m1b = lpart[crow(rb)], l1b = lpart[64 + crow(rb)];
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B_L_FREE));
          const float ma = fmaxf(m_a, m1a), mb = fmaxf(m_b, m1b);
          l_a = (m_a == -INFINITY ? 0.f : l_a * ex2(m_a - ma)) + (m1a == -INFINITY ? 0.f : l1a * ex2(m1a - ma));
          l_b = (m_b == -INFINITY ? 0.f : l_b * ex2(m_b - mb)) + (m1b == -INFINITY ? 0.f : l1b * ex2(m1b - mb));
          m_a = ma;
          m_b = mb;
          if (c == 0) {
#pragma unroll
            for (int rsel = 0; rsel < 2; ++rsel) {
              if (rsel ? vb : va) {
                const float l = rsel ? l_b : l_a, m = rsel ? m_b : m_a;
                float* ml = a.part_ml + ((long long)pc.slot * BM + (rsel ? rb : ra)) * 2;
                ml[0] = l > 0.f ? m * 0.6931471805599453f : -INFINITY;
                ml[1] = l > 0.f ? l : 0.f;
              }
            }
          }
        }
        // O write-out.  After the pair's last piece the 8 softmax warps write 128
        // columns each.  When another piece follows, the 4 warps that took this
        // piece's last tile write all 256 columns and free O (B_O_FREE counts 4
        // arrivals) while the other 4 go on with the next piece's first tile.
        // B_O_FULL + par completes only for pieces that this parity writes, so
        // each warp sees its phases in order.
        Piece nx = pc;
        have = next_piece<kGap>(a, end, W, nx);
        if (!have ? !write_o(pc.slot, pc.rt, false, 128 * par, 4)
                  : (((g - 1) & 1) == par && !write_o(pc.slot, pc.rt, true, 0, 8))) {
          alive = false;
          break;
        }
        ++pi;
        pc = nx;
      }

      // After an abort, let what the peer may still be sending land before exit
      // (receive phases that were armed but not consumed); bounded, errors ignored.
      if (!alive) {
        if (next_rx < G) drain_wait(BAR(B_RX_FULL + (next_rx & 1)), (next_rx >> 1) & 1, 200000ull);
        for (int t = next_af; t < next_af + kAfBufs && t < G; t += 2)
          drain_wait(BAR(B_AF_FULL + (t & (kAfBufs - 1))), (t / kAfBufs) & 1, 200000ull);
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

// ---- plan kernel ----------------------------------------------------------------------
// CTA b < B: the ancestor masks of request b (and the tree check).  CTA B: the
// stream-K plan.  Request b contributes rt_count row tiles of u_b = ceil((L_b
// + N) / 64) key tiles each (0 if its prefix length is invalid).  The units
// are laid out in a virtual sequence in which every non-empty row tile but
// the first is preceded by a gap of sk_gap units (0 when the host chose the
// plain plan): row tile r starts at vS_r = S_r + sk_gap * (non-empty tiles
// before r), and the sequence is V units long.  CTA pair c takes the virtual
// range [cW, (c+1)W), W = max(ceil(V / clusters), wmin) (or the forced W); a
// pair whose range crosses into another row tile spends part of it in a gap
// and so takes fewer key tiles, which pays for the piece boundary.  A row
// tile is cut where a multiple of W falls inside (vS_r, vS_r + u_r); its
// pieces take consecutive partial slots from base_r (an exclusive scan of
// the piece counts).  The plan also lists, for each pair, the row tile of
// its first piece (the tile whose range, with the gap before it, holds cW),
// with that tile's {vS_r, u_r, base_r}, the request's prefix length and the
// pair's count of key tiles.
__global__ void __launch_bounds__(256) sk_plan_kernel(const Args a) {
  grid_dep_launch();   // the absorb kernel does not read the plan
  const int tid = threadIdx.x;
  if ((int)blockIdx.x < a.B) {
    const int b = blockIdx.x;
    __shared__ int32_t par_s[kMaxNodes];
    if (tid < a.N) par_s[tid] = a.parent[(long long)b * a.N + tid];
    __syncthreads();
    if (tid < a.N) {
      uint32_t m[4];
      ancestor_mask_smem(a, b, par_s, tid, m);
      reinterpret_cast<uint4*>(a.anc_g)[(long long)b * a.N + tid] = make_uint4(m[0], m[1], m[2], m[3]);
    }
    return;
  }
  __shared__ int tu[256], tn[256];
  __shared__ int carry_u, carry_n;
  const int R = a.B * a.rt_count;
  const int gap = a.sk_gap;
  int* e = a.sk + kSkHeader;
  const int cap = a.page_size ? a.max_pages * a.page_size : a.t_stride;
  if (tid == 0) carry_u = carry_n = 0;
  __syncthreads();
  // units, virtual starts and (in e[3r+2], for now) the non-empty tiles before r
  for (int r0 = 0; r0 < R; r0 += 256) {
    const int r = r0 + tid;
    int u = 0;
    if (r < R) {
      const int b = r % a.B;                 // row tiles in lane-major order
      const int L = a.prefix_len[b];
      const bool ok = L >= 0 && (long long)L + a.N <= cap;
      if (!ok && r < a.B) record_error(a.status, KDTV_ERR_BAD_PREFIX, (unsigned)b);
      u = ok ? (L + a.N + BN - 1) / BN : 0;
    }
    tu[tid] = u;
    tn[tid] = u > 0;
    __syncthreads();
    for (int o = 1; o < 256; o <<= 1) {     // inclusive scans
      const int xu = tid >= o ? tu[tid - o] : 0, xn = tid >= o ? tn[tid - o] : 0;
      __syncthreads();
      tu[tid] += xu;
      tn[tid] += xn;
      __syncthreads();
    }
    if (r < R) {
      const int S = carry_u + tu[tid] - u, ne = carry_n + tn[tid] - (u > 0);
      e[3 * r] = S + gap * ne;
      e[3 * r + 1] = u;
      e[3 * r + 2] = ne;
    }
    __syncthreads();
    if (tid == 255) { carry_u += tu[255]; carry_n += tn[255]; }
    __syncthreads();
  }
  const int V = carry_u + gap * (carry_n > 1 ? carry_n - 1 : 0);
  int W;
  if (a.sk_wforce > 0) {
    W = a.sk_wforce > a.sk_wmin ? a.sk_wforce : a.sk_wmin;
  } else {
    W = (V + a.sk_clusters - 1) / a.sk_clusters;
    if (W < a.sk_wmin) W = a.sk_wmin;
  }
  if (W < 1) W = 1;
  // each pair's first row tile and its count of key tiles
  int* first = e + 3 * R;
  const int npair = a.sk_clusters;
  int4* rec = reinterpret_cast<int4*>(a.sk + sk_rec_off(R, npair));
  for (int c = tid; c < npair; c += 256) {
    first[c] = R;
    rec[2 * c + 1] = make_int4(0, 0, 0, 0);
  }
  __syncthreads();
  for (int r = tid; r < R; r += 256) {
    const int vS = e[3 * r], u = e[3 * r + 1], ne = e[3 * r + 2];
    if (u == 0) continue;
    // pairs whose range starts in [vS - gap, vS + u) begin in this tile, if
    // their range reaches it
    const int claim = ne > 0 ? vS - gap : 0;
    const long long c_end = ((long long)vS + u + W - 1) / W;
    for (long long c = ((long long)claim + W - 1) / W; c < c_end && c < npair; ++c)
      first[c] = (long long)vS < (c + 1) * W ? r : R;
    for (long long c = vS / W; c < c_end && c < npair; ++c) {
      const long long lo = c * W > vS ? c * W : vS;
      const long long hi = (c + 1) * W < (long long)vS + u ? (c + 1) * W : (long long)vS + u;
      atomicAdd(&rec[2 * c + 1].y, (int)(hi - lo));
    }
  }
  __syncthreads();
  // partial slots: base_r = the pieces of the row tiles before r
  if (tid == 0) carry_u = 0;
  __syncthreads();
  for (int r0 = 0; r0 < R; r0 += 256) {
    const int r = r0 + tid;
    int cnt = 0;
    if (r < R) {
      const int vS = e[3 * r], u = e[3 * r + 1];
      cnt = u > 0 ? 1 + ((vS + u + W - 1) / W - 1 - vS / W) : 0;
    }
    tu[tid] = cnt;
    __syncthreads();
    for (int o = 1; o < 256; o <<= 1) {
      const int x = tid >= o ? tu[tid - o] : 0;
      __syncthreads();
      tu[tid] += x;
      __syncthreads();
    }
    if (r < R) e[3 * r + 2] = carry_u + tu[tid] - cnt;
    __syncthreads();
    if (tid == 255) carry_u += tu[255];
    __syncthreads();
  }
  // per-pair first-piece records {r, vS_r, u_r, base_r}, {L_b, key tiles, 0, 0}
  for (int c = tid; c < npair; c += 256) {
    const int r = first[c];
    int4 v0 = make_int4(r, 0, 0, 0);
    if (r < R) {
      v0.y = e[3 * r]; v0.z = e[3 * r + 1]; v0.w = e[3 * r + 2];
      rec[2 * c + 1].x = a.prefix_len[r % a.B];
    }
    rec[2 * c] = v0;
  }
  if (tid == 0) {
    a.sk[0] = V;
    a.sk[1] = W;
    a.sk[2] = a.sk_clusters;
    a.sk[3] = R;
  }
}

}  // namespace

namespace {
// The driver's tensor-map encoder, resolved through the runtime so that the
// library does not link libcuda (it must load on hosts without a driver).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up on first use and cached; host threads may call concurrently (each
// finds the same address), so the cache is an atomic.
std::atomic<EncodeTiledFn> g_encoder{nullptr};

EncodeTiledFn encoder() {
  EncodeTiledFn fn = g_encoder.load(std::memory_order_acquire);
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
      g_encoder.store(fn, std::memory_order_release);
    }
  }
  return fn;
}

}  // namespace

// 2-D bf16 tensor map: rows x cols (row stride row_stride_elems, or cols,
// elements), box = box_rows x box_cols, 128- or 64-byte swizzle.
CUresult encode_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_cols, uint32_t box_rows, uint64_t row_stride_elems,
                   int swizzle_bytes) {
  EncodeTiledFn fn = encoder();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {(row_stride_elems ? row_stride_elems : cols) * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int tc_supported(const kdtv_dims* d) {
  if (d->dtype != KDTV_BF16 || d->d_c != 512 || d->d_rope != 64) return 0;
  if (d->page_size != 0 && d->page_size != 64) return 0;
  if (d->kv_chunk % BN) return 0;
  return 1;
}

int tc_launches(const kdtv_dims* d, int /*splits*/) {
  // plan, absorb, attention, then the fused combine + up-projection (or the
  // fp32 combine and up-projection kernels)
  if (d->flags & KDTV_FLAG_SIMT_PROJ) return 5;
  Args a;
  a.dtype = d->dtype; a.d_c = d->d_c; a.d_v = d->d_v; a.d_nope = d->d_nope; a.splits = 1;
  int dummy = 0;
  a.sk = &dummy;
  return 3 + (combine_uproj_tc_ok(a) ? 1 : 2);
}

cudaError_t launch_tc(const Args& a, const Plan& p, cudaStream_t st, cudaEvent_t* ev) {
  for (const void* ptr : {a.q_rope, a.c_kv, a.k_rope, static_cast<const void*>(a.q_lat)})
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return cudaErrorMisalignedAddress;
  const long long rows = (long long)a.B * a.N * a.H;
  const long long kv_rows = a.page_size ? (long long)a.num_pages * a.page_size
                                        : (long long)a.B * a.t_stride;
  CUtensorMap tqr, tck, tkr;
  if (encode_2d(&tqr, a.q_rope, rows, 64, kRopeHalf, BM, 0, 64) != CUDA_SUCCESS ||
      encode_2d(&tck, a.c_kv, kv_rows, 512, CH, BN) != CUDA_SUCCESS ||
      encode_2d(&tkr, a.k_rope, kv_rows, 64, kRopeHalf, BN, 0, 64) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  const bool simt_proj = a.flags & KDTV_FLAG_SIMT_PROJ;
  if (a.N > kMaxNodes || !a.sk || !a.anc_g || a.sk_clusters < 1) return cudaErrorInvalidValue;
  // The plan runs beside the absorb kernel (which waits for it before it
  // exits), so the attention kernel sees both once the absorb has completed.
  sk_plan_kernel<<<a.B + 1, 256, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = simt_proj ? launch_absorb(a, st, /*bf16_out=*/true)
                : launch_absorb_tc(a, st, /*after_plan=*/ev == nullptr);
  if (e != cudaSuccess) return e;
  if (a.c_kv8) {   // fp8 cache: widen it beside the plan and absorb kernels
    e = launch_kv_widen(a, p.sms, st, /*pdl=*/ev == nullptr);
    if (e != cudaSuccess) return e;
  }
  if (ev) cudaEventRecord(ev[1], st);

  TcCfg cfg;
  cfg.limit_ns = (a.flags & KDTV_FLAG_TEST_STALL) ? 20000000ull : 2000000000ull;
  // one instance per cache layout (the paged cache reads its rows through the
  // page table: its own producer loop) and per plan (with or without gaps)
  const auto kern = a.page_size ? (a.sk_gap ? attn_tc_kernel<true, true> : attn_tc_kernel<true, false>)
                                : (a.sk_gap ? attn_tc_kernel<false, true> : attn_tc_kernel<false, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // Overlap with the absorb kernel's tail unless phase events split the call.
  e = launch_ex(kern, dim3((unsigned)(2 * a.sk_clusters)), dim3(kThreads), kSmemBytes,
                st, /*pdl=*/ev == nullptr && !simt_proj, tqr, tck, tkr, a, cfg);
  if (e != cudaSuccess) return e;
  if (ev) cudaEventRecord(ev[2], st);
  return simt_proj ? launch_combine_uproj(a, p, st, ev) : launch_combine_uproj_tc(a, p, st, ev);
}

}  // namespace kdtv
