// Pieces shared by the backward kernels (bwd_tc.cu for head dimensions 64 and 128,
// bwd256_tc.cu for 256): tile and warp layout, named-barrier IDs, the element-wise
// score/dS arithmetic, the dropout keep flags, shared-memory layouts, barriers,
// the MMA issue helpers, the accumulator store and the load / relay loops.
#pragma once
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int BT = 128;          // rows of the tile a CTA owns
constexpr int SUB = 64;          // rows (columns of S) per sub-step
constexpr int kEwWarps = 16;     // element-wise warps: two pairs of warpgroups
constexpr int kThreads = (kEwWarps + 3) * 32;
constexpr int kLoadWarp = kEwWarps;
constexpr int kMmaWarp = kEwWarps + 1;
constexpr int kRelayWarp = kEwWarps + 2;  // turns TMA completions into barrier arrivals
// Named barriers (the MMA warp waits only on these; see nb_sync in ptx.cuh):
//   kNbStage + s   ring stage s loaded: relay warp (32) + MMA warp (32)
//   dq:   kNbP + x     dS_x written to TMEM: pair x (256 threads) + MMA warp (32)
//   dkdv: kNbKvP + x   P^T of a sub-step u (x = u % 2) written over S^T buffer x:
//                      element-wise warps + MMA warp
//   dkdv: kNbKvF       dP^T of a sub-step read into registers: the same warps
//   dkdv: kNbKvD       dS^T of a sub-step written into its S^T buffer: the same warps
//   dkdv: kNbQL        the V tile written to tensor memory: the same warps
//   d=256 kernels: kNbKvRel, kNbKvP + x, kNbKvK (bwd256_tc.cu)
//   dq:   kNbQL        Q and dO tiles written to tensor memory: element-wise warps + MMA warp
constexpr uint32_t kNbP = 1, kNbPCount = 288;
constexpr uint32_t kNbStage = 3, kNbStageCount = 64;
constexpr uint32_t kNbKvRel = 9, kNbKvP = 10, kNbKvK = 12, kNbQL = 13, kNbKvD = 14, kNbKvF = 15;
constexpr uint32_t kNbKvCount = (kEwWarps + 1) * 32;
constexpr int kStagesQ = 5;      // dq ring depth, in sub-steps (its Q and dO tiles are fixed)
constexpr int kStagesKv = 5;     // dkdv ring depth (its K tile is fixed in smem)
constexpr int kMaxStages = 6;
// Stage barriers take IDs kNbStage .. kNbStage + kMaxStages - 1; the others must not
// overlap them (one hardware barrier, one thread count), and IDs end at 15.
static_assert(kNbStage + kMaxStages <= kNbKvRel && kNbP + 2 <= kNbStage && kNbKvK < kNbQL &&
                  kNbQL < kNbKvD && kNbKvD < kNbKvF && kNbKvF < 16,
              "named barrier IDs");
constexpr int kHeadGroup = 4;
constexpr float kLog2e = 1.4426950408889634f;

// Tensor memory columns of dq: S buffers, dP buffers (64 each), dQ, then the Q and dO
// tiles as bf16 pairs (A operands of S = Q K^T and dP = dO V^T; D/2 columns each).
__device__ __forceinline__ uint32_t col_s(int x) { return x * 64; }
__device__ __forceinline__ uint32_t col_dp(int x) { return 128 + x * 64; }
constexpr uint32_t kColAcc = 256, kColQ = 384;
template <int D> constexpr uint32_t col_do() { return kColQ + D / 2; }
// Tensor memory columns of the d = 256 dK/dV walks (bwd256_tc.cu): S^T, dP^T (64 each),
// P^T / dS^T (bf16 pairs: P^T in the first 32 columns, dS^T in the next 32), the K tile
// (bf16 pairs, A operand of S^T = K Q^T), then the accumulator.
constexpr uint32_t kKvColS = 0, kKvColDP = 64, kKvColPD = 128, kKvColK = 192, kKvColAcc = 256;
// Tensor memory columns of dkdv (head dimension 64 and 128): two S^T buffers x (64 columns
// each; P^T and dS^T of the sub-step are written as bf16 pairs over the first and the
// second half of each warpgroup's 16 columns of its buffer), one dP^T buffer (64), the V
// tile (bf16 pairs, the A operand of dP^T = V dO^T; D / 2 columns), then dV and dK.
__device__ __forceinline__ uint32_t kv_col_s(int x) { return x * 64; }
constexpr uint32_t kKv2ColDP = 128, kKv2ColV = 192, kKv2ColAcc = 256;

// Element-wise constants: s2 = x*k1 + kb*(j - i) (log2 units); with the soft-cap c the
// same expression gives the pre-cap score over c and s2 = c log2(e) tanh of it.
struct ScoreK {
  float k1, kb, capA;
};

template <bool kAlibi, bool kSoftcap>
__device__ __forceinline__ ScoreK score_consts(const Problem& p, int h) {
  const float slope = kAlibi ? alibi_slope(h, p.Hq) : 0.f;
  ScoreK s;
  if (kSoftcap) {
    s.k1 = p.scale / p.softcap;
    s.kb = slope / p.softcap;
    s.capA = p.softcap * kLog2e;
  } else {
    s.k1 = p.scale * kLog2e;
    s.kb = slope * kLog2e;
    s.capA = 0.f;
  }
  return s;
}

// P and dS of one element. xs = raw score q.k; `alibi` = kb (j - i) (0 without ALiBi);
// lse2 = L log2e (+inf for a row with no key); zm = the element's dropout keep mask
// (all ones without dropout, 0 where the element is dropped). With dropout the row term
// is D' = D (1 - p) and the result dS' = P (dP Z - D') is dS (1 - p); the factor
// 1 / (1 - p) is applied with the softmax scale in the dK and dQ epilogues. Under the
// soft-cap the pre-cap score is divided by c and the tanh derivative scales dS. A
// masked element (ok false) takes the exponent -inf, so P = dS = 0 with no branch: a
// per-lane condition around the exponential would make the compiler branch on every
// element.
template <bool kAlibi, bool kSoftcap>
__device__ __forceinline__ void p_only(float xs, const ScoreK& sk, float alibi, float lse2,
                                       bool ok, float& pr, float& dcap) {
  float arg;
  dcap = 1.f;
  if (kSoftcap) {
    const float pre = kAlibi ? fmaf(xs, sk.k1, alibi) : xs * sk.k1;
    const float t = tanh_approx(pre);  // tanh(pre-cap score / c)
    arg = sk.capA * t - lse2;
    dcap = 1.0f - t * t;
  } else if (kAlibi) {
    arg = fmaf(xs, sk.k1, alibi) - lse2;
  } else {
    arg = fmaf(xs, sk.k1, -lse2);
  }
  pr = ex2_approx(ok ? arg : -INFINITY);
}
// dS of one element from its P (and soft-cap derivative), as p_and_ds.
template <bool kSoftcap>
__device__ __forceinline__ float ds_of(float pr, float dcap, float dp, float delta, uint32_t zm) {
  const float dpz = __uint_as_float(__float_as_uint(dp) & zm);
  return kSoftcap ? pr * (dpz - delta) * dcap : pr * (dpz - delta);
}
template <bool kAlibi, bool kSoftcap>
__device__ __forceinline__ void p_and_ds(float xs, const ScoreK& sk, float alibi, float lse2,
                                         float dp, float delta, bool ok, uint32_t zm,
                                         float& pr, float& ds) {
  float dcap;
  p_only<kAlibi, kSoftcap>(xs, sk, alibi, lse2, ok, pr, dcap);
  ds = ds_of<kSoftcap>(pr, dcap, dp, delta, zm);
}

// Dropout keep flags (keep_flags4 layout: flag of column c in byte c % 4 of word c / 4)
// of the 16 query columns qs .. qs + 15 of key row j, for the dK/dV layout (lane = key).
// One Philox call covers 16 keys of one query row, so lane L draws the call of query
// qs + L % 16 and key block (j - lane) / 16 + L / 16; a byte transpose within each
// half-warp then hands every lane the bytes of its own key.
__device__ __forceinline__ void dropout_flags_dkdv(const PhiloxKeys& pk, const DropThr& th,
                                                   int j, int lane, int qs, int bh,
                                                   uint32_t (&kf)[4]) {
  const int jw = j - lane;  // first key of the warp, a multiple of 32
  const uint4 r = philox4x32_10((uint32_t)((jw >> 4) + (lane >> 4)), (uint32_t)(qs + (lane & 15)),
                                (uint32_t)bh, 0u, pk);
  kf[0] = r.x;
  kf[1] = r.y;
  kf[2] = r.z;
  kf[3] = r.w;
  transpose16x16_bytes(kf, lane);
#pragma unroll
  for (int q = 0; q < 4; ++q) kf[q] = keep_flags4(kf[q], th);
}

// Dropout keep flags of the 32 key columns ks .. ks + 31 (ks a multiple of 16) of query
// row i, for the dQ layout (thread = query row): two Philox calls.
__device__ __forceinline__ void dropout_flags_dq(const PhiloxKeys& pk, const DropThr& th, int i,
                                                 int ks, int bh, uint32_t (&kf)[8]) {
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const uint4 r = philox4x32_10((uint32_t)((ks >> 4) + hh), (uint32_t)i, (uint32_t)bh, 0u, pk);
    kf[4 * hh + 0] = keep_flags4(r.x, th);
    kf[4 * hh + 1] = keep_flags4(r.y, th);
    kf[4 * hh + 2] = keep_flags4(r.z, th);
    kf[4 * hh + 3] = keep_flags4(r.w, th);
  }
}

// Shared-memory layouts. dq: a ring of kS stages, each holding a 64-row slice of K and
// V (Q and dO live in tensor memory). dkdv: the K tile (fixed; V lives in tensor
// memory), a ring of 64-row slices of Q and dO, and each stage's row terms of those 64
// query rows (lse2, delta, first key: 256 bytes each).
template <int D, int kS, int kFixTiles, bool kRowTerms>
struct Layout {
  static constexpr int kStageCount = kS;
  static constexpr int kFixChunk = BT * 128;        // 64-column slab of a fixed tile
  static constexpr int kFixTile = BT * D * 2;
  static constexpr int kSubChunk = SUB * 128;       // 64-column slab of a stage slice
  static constexpr int kSubTile = SUB * D * 2;
  static constexpr int kFixA = 0;
  static constexpr int kRing = kFixTiles * kFixTile;
  static constexpr int kStage = 2 * kSubTile;
  static constexpr int kRows = kRing + kS * kStage;
  static constexpr int kRowStage = 3 * SUB * 4;
  static constexpr int kBars = kRows + (kRowTerms ? kS * kRowStage : 0);
  static constexpr int kAlloc = kBars + 256 + 1024;
};
template <int D> using LayoutQ = Layout<D, kStagesQ, 2, false>;  // fixed: Q, dO
template <int D> using LayoutKv = Layout<D, kStagesKv, 1, true>;  // fixed: K
static_assert(LayoutKv<128>::kAlloc <= 232448 && LayoutQ<128>::kAlloc <= 232448,
              "shared memory per CTA");

struct BwdBars {
  uint64_t fixed_full;             // the two fixed tiles
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t s_full[2];              // S_x and dP_x in TMEM (dkdv: S^T_x)
  uint64_t dp_full;                // dkdv: dP^T in TMEM
  uint64_t pd_free[2];             // dkdv: P^T / dS^T read by their MMAs (entry 0)
  uint64_t acc_full;               // accumulators final
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdArgs {
  Problem p;
  RowTerms rt;
  const __nv_bfloat16* q;     // Q, dO [B, Hq, Nq, d] and K, V [B, Hkv, Nkv, d]: the tiles
  const __nv_bfloat16* dout;  // the kernels keep in tensor memory are copied from here
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int n_tiles;  // key tiles (dkdv) or query tiles (dq) per head
};

// CTA -> (head index, tile) with heads taken kHeadGroup at a time. `reverse` flips
// the tile order (query tiles of causal masks have the most work last).
__device__ __forceinline__ void cta_tile(int heads, int n_tiles, bool reverse, int& head,
                                         int& tile) {
  const int per_group = kHeadGroup * n_tiles;
  const int grp = blockIdx.x / per_group;
  const int rem = blockIdx.x - grp * per_group;
  const int gh = imin(kHeadGroup, heads - grp * kHeadGroup);
  tile = rem / gh;
  if (reverse) tile = n_tiles - 1 - tile;
  head = grp * kHeadGroup + rem % gh;
}

__device__ __forceinline__ void setup_common(BwdBars* bars, int stages) {
  mbar_init(smem_u32(&bars->fixed_full), 1);
  for (int s = 0; s < stages; ++s) {
    mbar_init(smem_u32(&bars->full[s]), 1);   // the loader's arrive + transaction bytes
    mbar_init(smem_u32(&bars->empty[s]), 1);  // one MMA commit
  }
  for (int x = 0; x < 2; ++x) {
    mbar_init(smem_u32(&bars->s_full[x]), 1);
    mbar_init(smem_u32(&bars->pd_free[x]), 1);
  }
  mbar_init(smem_u32(&bars->dp_full), 1);
  mbar_init(smem_u32(&bars->acc_full), 1);
  bars->abort_flag = 0;
  fence_barrier_init();
}

// D[128 x 64] = A B^T over the head dimension: A = a fixed 128-row K-major tile, B =
// a 64-row K-major stage slice (both written by TMA with 128-byte swizzle). The
// descriptors are built once; each K step adds its byte offset (in 16-byte units).
template <int D>
__device__ __forceinline__ void mma_128x64(bool pred, uint32_t d_tmem, uint32_t a, uint32_t b) {
  constexpr uint32_t id = idesc_bf16_f32(BT, SUB, false, false);
  const uint64_t da = smem_desc_sw128(a, 16, 1024), db = smem_desc_sw128(b, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t oa = ((kk >> 2) * (BT * 128) + (kk & 3) * 32) >> 4;
    const uint32_t ob = ((kk >> 2) * (SUB * 128) + (kk & 3) * 32) >> 4;
    mma_ss_if(pred, d_tmem, da + oa, db + ob, id, kk > 0 ? 1u : 0u);
  }
}

// D[128 x D] (+)= A_tmem[128 x 64] B[64 x D]: A = bf16 pairs in TMEM, written by the
// two element-wise warpgroups of a pair at columns [0,16) and [32,48) of a_tmem;
// B = a 64-row stage slice used MN-major (its 64-column slabs 8 KB apart).
template <int D>
__device__ __forceinline__ void mma_tmem64_x_slice(bool pred, uint32_t d_tmem, uint32_t a_tmem,
                                                   uint32_t b, bool accumulate) {
  constexpr uint32_t id = idesc_bf16_f32(BT, D, false, true);
  const uint64_t db = smem_desc_sw128(b, SUB * 128, 1024);
#pragma unroll
  for (int kk = 0; kk < SUB / 16; ++kk) {
    const uint32_t acol = (kk < 2) ? kk * 8 : 32 + (kk - 2) * 8;
    mma_ts_if(pred, d_tmem, a_tmem + acol, db + ((kk * 16 * 128) >> 4), id,
           (accumulate || kk > 0) ? 1u : 0u);
  }
}

// D[128 x 64] = A_tmem[128 x D] B^T with A in tensor memory as bf16 pairs (k-step kk,
// 16 of the head dimension, in columns [8 kk, 8 kk + 8)) and B a 64-row K-major stage
// slice.
template <int D>
__device__ __forceinline__ void mma_tmem_x64(bool pred, uint32_t d_tmem, uint32_t a_tmem,
                                             uint32_t b) {
  constexpr uint32_t id = idesc_bf16_f32(BT, SUB, false, false);
  const uint64_t db = smem_desc_sw128(b, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t ob = ((kk >> 2) * (SUB * 128) + (kk & 3) * 32) >> 4;
    mma_ts_if(pred, d_tmem, a_tmem + kk * 8, db + ob, id, kk > 0 ? 1u : 0u);
  }
}

// D[128 x D] (+)= A_tmem[128 x 64] B[64 x D] with A stored contiguously: k-step kk
// (16 rows of B) reads A columns [8 kk, 8 kk + 8). B as in mma_tmem64_x_slice.
template <int D>
__device__ __forceinline__ void mma_pd_x_slice(bool pred, uint32_t d_tmem, uint32_t a_tmem,
                                               uint32_t b, bool accumulate) {
  constexpr uint32_t id = idesc_bf16_f32(BT, D, false, true);
  const uint64_t db = smem_desc_sw128(b, SUB * 128, 1024);
#pragma unroll
  for (int kk = 0; kk < SUB / 16; ++kk)
    mma_ts_if(pred, d_tmem, a_tmem + kk * 8, db + ((kk * 16 * 128) >> 4), id,
              (accumulate || kk > 0) ? 1u : 0u);
}

// D[128 x D] (+)= A_tmem[128 x 64] B[64 x D] with A written in place over a 64-column
// fp32 buffer: k-step kk (16 rows of B) reads A columns [16 kk, 16 kk + 8), the bf16 pairs
// the kk-th element-wise warpgroup wrote over the first half of its 16 columns. B as in
// mma_tmem64_x_slice.
template <int D>
__device__ __forceinline__ void mma_inplace_x_slice(bool pred, uint32_t d_tmem, uint32_t a_tmem,
                                                    uint32_t b, bool accumulate) {
  constexpr uint32_t id = idesc_bf16_f32(BT, D, false, true);
  const uint64_t db = smem_desc_sw128(b, SUB * 128, 1024);
#pragma unroll
  for (int kk = 0; kk < SUB / 16; ++kk)
    mma_ts_if(pred, d_tmem, a_tmem + kk * 16, db + ((kk * 16 * 128) >> 4), id,
              (accumulate || kk > 0) ? 1u : 0u);
}

// Shared memory an element-wise warp stages its output rows in at the end: 32 rows of a
// 128-byte pitch per warp at the start of the ring, free once the last MMA has completed
// (every stage consumed).
constexpr int kStageRowsBytes = 32 * 128;
template <class L>
__device__ __forceinline__ uint8_t* ew_stage(uint8_t* smem, int warp) {
  static_assert(L::kStageCount * L::kStage >= kEwWarps * kStageRowsBytes, "staging fits the ring");
  return smem + L::kRing + warp * kStageRowsBytes;
}

// Write one accumulator row per lane (D <= 64 fp32 columns at TMEM `t`) times `mul` as
// bf16 to `dst` (this lane's row). The warp stages its 32 rows in `stage` (the warp's
// ew_stage area; 16-byte chunk c of row r at chunk c ^ (r & 7)) and then copies them out
// with each store instruction writing whole rows. tcgen05.ld is warp-collective: every
// lane must call this with the same `live`; `store` (per lane) decides whether its row is
// written.
template <int D>
__device__ __forceinline__ void store_acc_row(uint32_t t, float mul, __nv_bfloat16* dst,
                                              bool live, bool store, uint8_t* stage) {
  static_assert(D % 32 == 0 && D <= 64, "rows of at most 128 bytes");
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t r[32];
    if (live) {
      tmem_ld32(t + c * 32, r);
      tmem_wait_ld();
      reg_fence32(r);
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) r[e] = 0u;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint4 w;
      w.x = pack_bf16x2(__uint_as_float(r[8 * e + 0]) * mul, __uint_as_float(r[8 * e + 1]) * mul);
      w.y = pack_bf16x2(__uint_as_float(r[8 * e + 2]) * mul, __uint_as_float(r[8 * e + 3]) * mul);
      w.z = pack_bf16x2(__uint_as_float(r[8 * e + 4]) * mul, __uint_as_float(r[8 * e + 5]) * mul);
      w.w = pack_bf16x2(__uint_as_float(r[8 * e + 6]) * mul, __uint_as_float(r[8 * e + 7]) * mul);
      const int g = c * 4 + e;
      *reinterpret_cast<uint4*>(stage + lane * 128 + ((g ^ (lane & 7)) << 4)) = w;
    }
  }
  __syncwarp();
  constexpr int kChunks = D / 8;              // 16-byte chunks per row
  constexpr int kRowsPerStore = 32 / kChunks;  // rows one warp store instruction covers
  const int g = lane % kChunks;
#pragma unroll
  for (int k = 0; k < 32 / kRowsPerStore; ++k) {
    const int rr = k * kRowsPerStore + lane / kChunks;  // row (= owning lane) of this piece
    const uint4 w = *reinterpret_cast<const uint4*>(stage + rr * 128 + ((g ^ (rr & 7)) << 4));
    const auto d = reinterpret_cast<__nv_bfloat16*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(dst), rr));
    if (__shfl_sync(0xffffffffu, store ? 1 : 0, rr)) reinterpret_cast<uint4*>(d)[g] = w;
  }
}

// Loads the fixed tile fa if given (rows r0.. of head z) and then, for every
// sub-step u, the 64-row slices of the two streamed operands into stage
// u % L::kStageCount. `slice`
// gives (row, head) of sub-step u. With `rt` (dkdv) it also copies the row terms of
// those 64 query rows into the stage's row block; all of it completes full[s].
template <int D, class L, typename SliceFn>
__device__ __forceinline__ void load_loop(uint8_t* smem, BwdBars* bars, const WaitCtx& wc,
                                          int lane, const CUtensorMap* fa, int r0, int z,
                                          const CUtensorMap* sa,
                                          const CUtensorMap* sb, int subs, SliceFn slice,
                                          const RowTerms* rt, int nq_pad,
                                          const CUtensorMap* fb = nullptr) {
  constexpr int kS = L::kStageCount;
  if (lane == 0) {
    tma_prefetch_desc(sa);
    tma_prefetch_desc(sb);
    if (fa) {  // the fixed tile(s): fa, and fb after it when given (same rows)
      const uint32_t bar = smem_u32(&bars->fixed_full);
      mbar_arrive_expect_tx(bar, (fb ? 2 : 1) * L::kFixTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(smem_u32(smem + L::kFixA + c * L::kFixChunk), fa, bar, c * 64, r0, z);
        if (fb)
          tma_load_3d(smem_u32(smem + L::kFixA + L::kFixTile + c * L::kFixChunk), fb, bar,
                      c * 64, r0, z);
      }
    }
  }
  for (int u = 0; u < subs; ++u) {
    const int s = u % kS, use = u / kS;
    int row, head;
    slice(u, row, head);
    bool ok = true;
    if (lane == 0) ok = mbar_wait(smem_u32(&bars->empty[s]), (use & 1) ^ 1, wc);
    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
    if (lane == 0) {
      const uint32_t full = smem_u32(&bars->full[s]);
      mbar_arrive_expect_tx(full, L::kStage + (rt ? L::kRowStage : 0));
      uint8_t* stg = smem + L::kRing + s * L::kStage;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(smem_u32(stg + c * L::kSubChunk), sa, full, c * 64, row, head);
        tma_load_3d(smem_u32(stg + L::kSubTile + c * L::kSubChunk), sb, full, c * 64, row, head);
      }
      if (rt) {  // rows row .. row + 63 of query head `head` (row + 64 <= nq_pad)
        const uint32_t rs = smem_u32(smem + L::kRows + s * L::kRowStage);
        const size_t off = (size_t)head * nq_pad + row;
        bulk_load(rs, rt->lse2 + off, SUB * 4, full);
        bulk_load(rs + SUB * 4, rt->delta + off, SUB * 4, full);
        bulk_load(rs + 2 * SUB * 4, rt->first + row, SUB * 4, full);
      }
    }
  }
  if (lane == 0) {  // let in-flight copies land before the CTA can exit
    if (fa) mbar_wait(smem_u32(&bars->fixed_full), 0, wc);
    for (int u = imax(0, subs - kS); u < subs; ++u)
      mbar_wait(smem_u32(&bars->full[u % kS]), (u / kS) & 1, wc);
  }
}

// Relay warp: after the bytes of ring use u land (full[u % kS]), arrive on that
// stage's named barrier for the MMA warp; after an abort, rendezvous instead.
template <int kS>
__device__ __forceinline__ void relay_loop(BwdBars* bars, const WaitCtx& wc, int subs) {
  bool live = true;
  for (int u = 0; u < subs; ++u) {
    const int s = u % kS;
    if (live)
      live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->full[s]), (u / kS) & 1, wc));
    if (live) nb_arrive(kNbStage + s, kNbStageCount);
    else nb_sync(kNbStage + s, kNbStageCount);
  }
}


}  // namespace
}  // namespace attn
