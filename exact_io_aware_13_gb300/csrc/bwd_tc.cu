// Backward attention on the tcgen05 tensor cores (sm_103a).
//
// "FlashAttention/es" ("Paso hacia atrás y recomputación") rebuilds S and P tile
// by tile from the saved log-sum-exp L instead of storing P. With
// P_ij = exp(s_ij - L_i) and D_i = rowsum(dO_i o O_i) (computed, with L log2 e and
// each row's first key, by a separate row kernel into padded arrays), the gradients are
//     dV = P^T dO,   dP = dO V^T,   dS = P o (dP - D) [x soft-cap derivative],
//     dK = scale dS^T Q,   dQ = scale dS K.
// Two kernels, both deterministic (fixed summation order, no atomics):
//   * dkdv: one CTA per (batch, kv head, 128-key tile); it walks the query heads of
//     its group and the query rows the mask leaves, 64 rows at a time ("sub-steps"):
//     S^T = K Q^T and dP^T = V dO^T into tensor memory, P^T and dS^T (bf16) back
//     into tensor memory, then dV += P^T dO and dK += dS^T Q;
//   * dq: one CTA per (batch, query head, 128-row tile); it walks the key tiles 64
//     keys at a time: S = Q K^T and dP = dO V^T, dS back into tensor memory, then
//     dQ += dS K.
// Each sub-step streams its own 64-row slice of the two operands it walks (Q and dO,
// or K and V; for dkdv also the 64 rows' L log2 e, D and first key) through a 4-deep
// shared-memory ring, so loads run ahead of the MMAs. Warp 16 loads with TMA, warp 17
// owns tensor memory and issues the MMAs, warp 18 relays TMA completions; warps 0-15
// do the element-wise work, one thread per TMEM lane (= row of the CTA's tile). The
// MMA warp waits only on hardware named barriers: a shared-memory access from the
// thread that issues MMAs stalls the tensor pipe (see nb_sync in ptx.cuh).
//   dkdv: every element-wise warp works on every sub-step (warpgroup w takes 16 of
//     its 64 query columns). S^T / dP^T have one TMEM buffer: the warps release it as
//     soon as they hold their columns in registers, so the next sub-step's S^T / dP^T
//     MMAs start while they compute; P^T / dS^T go to one of two separate buffers.
//   dq: two pairs of warpgroups alternate sub-steps (pair p takes u % 2 == p, warpgroup
//     w of the pair 32 key columns); S / dP are double-buffered and dS is written back
//     over S.
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
//   dkdv: kNbKvRel     S^T / dP^T of the sub-step read: element-wise warps + MMA warp
//         kNbKvP + x   P^T / dS^T of a sub-step u (x = u % 2) written: same threads
//         kNbKvK       K tile written to tensor memory: same threads
//   dq:   kNbQL        Q and dO tiles written to tensor memory: element-wise warps + MMA warp
constexpr uint32_t kNbP = 1, kNbPCount = 288;
constexpr uint32_t kNbStage = 3, kNbStageCount = 64;
constexpr uint32_t kNbKvRel = 8, kNbKvP = 9, kNbKvK = 11, kNbQL = 12;
constexpr uint32_t kNbKvCount = (kEwWarps + 1) * 32;
constexpr int kStagesQ = 4;      // dq ring depth, in sub-steps
constexpr int kStagesKv = 5;     // dkdv ring depth
constexpr int kMaxStages = 5;
// Stage barriers take IDs kNbStage .. kNbStage + kMaxStages - 1; the others must not
// overlap them (one hardware barrier, one thread count), and IDs end at 15.
static_assert(kNbStage + kMaxStages <= kNbKvRel && kNbP + 2 <= kNbStage && kNbKvK < kNbQL &&
                  kNbQL < 16,
              "named barrier IDs");
constexpr int kHeadGroup = 4;
constexpr float kLog2e = 1.4426950408889634f;

// Tensor memory columns of dq: S buffers, dP buffers (64 each), dQ, then the Q and dO
// tiles as bf16 pairs (A operands of S = Q K^T and dP = dO V^T; D/2 columns each).
__device__ __forceinline__ uint32_t col_s(int x) { return x * 64; }
__device__ __forceinline__ uint32_t col_dp(int x) { return 128 + x * 64; }
constexpr uint32_t kColAcc = 256, kColQ = 384;
template <int D> constexpr uint32_t col_do() { return kColQ + D / 2; }
// Tensor memory columns of dkdv: S^T, dP^T (64 each), P^T / dS^T (bf16 pairs: P^T in
// the first 32 columns, dS^T in the next 32), the K tile (bf16 pairs, A operand of
// S^T = K Q^T), then dV and dK.
constexpr uint32_t kKvColS = 0, kKvColDP = 64, kKvColPD = 128, kKvColK = 192, kKvColAcc = 256;

// Element-wise constants: s2 = x*k1 + kb*(j - i) (log2 units), then the soft-cap.
struct ScoreK {
  float k1, kb, capA;
};

template <bool kAlibi, bool kSoftcap>
__device__ __forceinline__ ScoreK score_consts(const Problem& p, int h) {
  const float slope = kAlibi ? alibi_slope(h, p.Hq) : 0.f;
  ScoreK s;
  if (kSoftcap) {
    const float c2 = 2.0f * kLog2e / p.softcap;
    s.k1 = p.scale * c2;
    s.kb = slope * c2;
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
// soft-cap the pre-cap score is in 2 log2e / c units and the tanh derivative scales dS. A
// masked element (ok false) takes the exponent -inf, so P = dS = 0 with no branch: a
// per-lane condition around the exponential would make the compiler branch on every
// element.
template <bool kAlibi, bool kSoftcap>
__device__ __forceinline__ void p_and_ds(float xs, const ScoreK& sk, float alibi, float lse2,
                                         float dp, float delta, bool ok, uint32_t zm,
                                         float& pr, float& ds) {
  float arg, dcap = 1.f;
  if (kSoftcap) {
    const float pre = kAlibi ? fmaf(xs, sk.k1, alibi) : xs * sk.k1;
    const float t = 1.0f - 2.0f * rcp_approx(1.0f + ex2_approx(pre));  // tanh(pre_cap / c)
    arg = sk.capA * t - lse2;
    dcap = 1.0f - t * t;
  } else if (kAlibi) {
    arg = fmaf(xs, sk.k1, alibi) - lse2;
  } else {
    arg = fmaf(xs, sk.k1, -lse2);
  }
  pr = ex2_approx(ok ? arg : -INFINITY);
  const float dpz = __uint_as_float(__float_as_uint(dp) & zm);
  ds = kSoftcap ? pr * (dpz - delta) * dcap : pr * (dpz - delta);
}

// Dropout keep flags (keep_flags4 layout: flag of column c in byte c % 4 of word c / 4)
// of the 16 query columns qs .. qs + 15 of key row j, for the dK/dV layout (lane = key).
// One Philox call covers 16 keys of one query row, so lane L draws the call of query
// qs + L % 16 and key block (j - lane) / 16 + L / 16; a byte transpose within each
// half-warp then hands every lane the bytes of its own key.
__device__ __forceinline__ void dropout_flags_dkdv(const Problem& p, const DropThr& th, int j,
                                                   int lane, int qs, int bh,
                                                   uint32_t (&kf)[4]) {
  const int jw = j - lane;  // first key of the warp, a multiple of 32
  const uint4 r = philox4x32_10((uint32_t)((jw >> 4) + (lane >> 4)), (uint32_t)(qs + (lane & 15)),
                                (uint32_t)bh, 0u, p.drop_seed_lo, p.drop_seed_hi);
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
__device__ __forceinline__ void dropout_flags_dq(const Problem& p, const DropThr& th, int i,
                                                 int ks, int bh, uint32_t (&kf)[8]) {
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const uint4 r = philox4x32_10((uint32_t)((ks >> 4) + hh), (uint32_t)i, (uint32_t)bh, 0u,
                                  p.drop_seed_lo, p.drop_seed_hi);
    kf[4 * hh + 0] = keep_flags4(r.x, th);
    kf[4 * hh + 1] = keep_flags4(r.y, th);
    kf[4 * hh + 2] = keep_flags4(r.z, th);
    kf[4 * hh + 3] = keep_flags4(r.w, th);
  }
}

// dkdv element-wise step for one thread: key row j, 16 query columns starting at qs,
// with their lse2 / delta / first key. Writes P^T and dS^T (bf16 pairs). kMasked adds
// the per-element mask test; the caller picks the variant by a warp-uniform tile test.
template <bool kAlibi, bool kSoftcap, bool kMasked, bool kDrop>
__device__ __forceinline__ void dkdv_pds(const uint32_t (&sr)[16], const uint32_t (&dr)[16],
                                         const float* lse2, const float* dl, const int* fk,
                                         const ScoreK& sk, float base, int j, int qs,
                                         bool key_ok, bool causal_type, const uint32_t (&kf)[4],
                                         uint32_t (&pp)[8], uint32_t (&dd)[8]) {
#pragma unroll
  for (int e4 = 0; e4 < 4; ++e4) {
    const float4 lv = reinterpret_cast<const float4*>(lse2)[e4];
    const float4 dv = reinterpret_cast<const float4*>(dl)[e4];
    const float lvs[4] = {lv.x, lv.y, lv.z, lv.w};
    const float dvs[4] = {dv.x, dv.y, dv.z, dv.w};
    float pv[4], dsv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int col = e4 * 4 + q;
      bool ok = true;
      if (kMasked) {
        const int i = qs + col;
        ok = key_ok && (!causal_type || (i >= j && fk[col] <= j));
      }
      const uint32_t zm = kDrop ? keep_mask_elem(kf[e4], q) : 0xffffffffu;
      p_and_ds<kAlibi, kSoftcap>(__uint_as_float(sr[col]), sk,
                                 kAlibi ? fmaf(-(float)col, sk.kb, base) : 0.f, lvs[q],
                                 __uint_as_float(dr[col]), dvs[q], ok, zm, pv[q], dsv[q]);
      if (kDrop) pv[q] = __uint_as_float(__float_as_uint(pv[q]) & zm);  // dV takes P Z
    }
    pp[2 * e4] = pack_bf16x2(pv[0], pv[1]);
    pp[2 * e4 + 1] = pack_bf16x2(pv[2], pv[3]);
    dd[2 * e4] = pack_bf16x2(dsv[0], dsv[1]);
    dd[2 * e4 + 1] = pack_bf16x2(dsv[2], dsv[3]);
  }
}

// dq element-wise step for one thread: query row with (lse2, delta), 32 key columns;
// allowed columns are [c_lo, c_hi] when kMasked. Writes dS (bf16 pairs).
template <bool kAlibi, bool kSoftcap, bool kMasked, bool kDrop>
__device__ __forceinline__ void dq_ds(const uint32_t (&sr)[32], const uint32_t (&dr)[32],
                                      const ScoreK& sk, float base, float lse2, float delta,
                                      int c_lo, int c_hi, const uint32_t (&kf)[8],
                                      uint32_t (&dd)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    float pr[2], ds[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int col = 2 * e + q;
      const bool ok = !kMasked || (col >= c_lo && col <= c_hi);
      const uint32_t zm = kDrop ? keep_mask_elem(kf[col >> 2], col & 3) : 0xffffffffu;
      p_and_ds<kAlibi, kSoftcap>(__uint_as_float(sr[col]), sk,
                                 kAlibi ? fmaf((float)col, sk.kb, base) : 0.f, lse2,
                                 __uint_as_float(dr[col]), delta, ok, zm, pr[q], ds[q]);
    }
    dd[e] = pack_bf16x2(ds[0], ds[1]);
  }
}

// Shared-memory layouts. dq: a ring of kS stages, each holding a 64-row slice of K and
// V (Q and dO live in tensor memory). dkdv: the V tile (fixed; K lives in tensor
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
template <int D> using LayoutQ = Layout<D, kStagesQ, 0, false>;
template <int D> using LayoutKv = Layout<D, kStagesKv, 1, true>;
static_assert(LayoutKv<128>::kAlloc <= 232448 && LayoutQ<128>::kAlloc <= 232448,
              "shared memory per CTA");

struct BwdBars {
  uint64_t fixed_full;             // the two fixed tiles
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t s_full[2];              // S_x and dP_x in TMEM (dkdv: buffer 0 only)
  uint64_t pd_free[2];             // dkdv: P^T / dS^T read by their MMAs (entry 0)
  uint64_t acc_full;               // accumulators final
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdArgs {
  Problem p;
  RowTerms rt;
  const __nv_bfloat16* q;     // Q, dO [B, Hq, Nq, d] and K [B, Hkv, Nkv, d]: the tiles the
  const __nv_bfloat16* dout;  // kernels keep in tensor memory are copied from here
  const __nv_bfloat16* k;
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

// Write one accumulator row (D fp32 columns at TMEM `t`) times `mul` as bf16.
// tcgen05.ld is warp-collective: every lane of the warp must call this with the same
// `live`; `store` (per lane) only decides whether the row is written.
template <int D>
__device__ __forceinline__ void store_acc_row(uint32_t t, float mul, __nv_bfloat16* dst,
                                              bool live, bool store) {
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
    if (store) {
      uint4* o = reinterpret_cast<uint4*>(dst) + c * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(r[8 * e + 0]) * mul, __uint_as_float(r[8 * e + 1]) * mul);
        w.y = pack_bf16x2(__uint_as_float(r[8 * e + 2]) * mul, __uint_as_float(r[8 * e + 3]) * mul);
        w.z = pack_bf16x2(__uint_as_float(r[8 * e + 4]) * mul, __uint_as_float(r[8 * e + 5]) * mul);
        w.w = pack_bf16x2(__uint_as_float(r[8 * e + 6]) * mul, __uint_as_float(r[8 * e + 7]) * mul);
        o[e] = w;
      }
    }
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
                                          const RowTerms* rt, int nq_pad) {
  constexpr int kS = L::kStageCount;
  if (lane == 0) {
    tma_prefetch_desc(sa);
    tma_prefetch_desc(sb);
    if (fa) {
      const uint32_t bar = smem_u32(&bars->fixed_full);
      mbar_arrive_expect_tx(bar, L::kFixTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem_u32(smem + L::kFixA + c * L::kFixChunk), fa, bar, c * 64, r0, z);
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

// ============================================================================ dK, dV
template <int D, bool kAlibi, bool kSoftcap, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using L = LayoutKv<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + L::kBars);
  const Problem& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.Hq / p.Hkv;

  int bg, kt;
  cta_tile(p.B * p.Hkv, a.n_tiles, false, bg, kt);
  const int b = bg / p.Hkv, g = bg - b * p.Hkv;
  const int k0 = kt * BT;
  const TileRange qr = q_tiles_for_keys(p.mask, k0, BT);
  const int n_q = imax(qr.hi - qr.lo, 0);
  const int subs = 2 * n_q * G;  // (head, query tile, half) triples, head-major
  if (subs == 0) {  // no query sees these keys: zero gradients
    for (int r = threadIdx.x; r < BT; r += kThreads) {
      const int j = k0 + r;
      if (j >= p.Nkv) continue;
      uint4* dkr = reinterpret_cast<uint4*>(a.dk + ((size_t)bg * p.Nkv + j) * D);
      uint4* dvr = reinterpret_cast<uint4*>(a.dv + ((size_t)bg * p.Nkv + j) * D);
      for (int c = 0; c < D / 8; ++c) { dkr[c] = make_uint4(0, 0, 0, 0); dvr[c] = make_uint4(0, 0, 0, 0); }
    }
    return;
  }
  // sub-step u: query head g*G + (u/2)/n_q, query rows q0 + 64*(u&1)
  auto slice = [&](int u, int& row, int& head) {
    const int st = u >> 1;
    head = b * p.Hq + g * G + st / n_q;
    row = (qr.lo + st % n_q) * BT + (u & 1) * SUB;
  };

  WaitCtx wc{&bars->abort_flag, p.status};
  if (threadIdx.x == 0) setup_common(bars, L::kStageCount);
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t colDV = kKvColAcc, colDK = kKvColAcc + D;

  if (warp == kLoadWarp) {
    load_loop<D, L>(smem, bars, wc, lane, &maps.v128, k0, bg, &maps.q64, &maps.do64, subs,
                    slice, &a.rt, p.nq_pad);
  } else if (warp == kRelayWarp) {
    relay_loop<L::kStageCount>(bars, wc, subs);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the schedule and waits on named barriers; every lane executes
    // the MMA instructions predicated on `issuer`, the one lane elect.sync picks, so the
    // warp never diverges (an elect.sync predicate issues an MMA in about 47 cycles, a
    // predicate computed from the lane index in about 82). If the fixed tiles never
    // arrive (`ok` false) the warp keeps every barrier operation and issues nothing.
    // Issue order: S^T/dP^T(0), then per sub-step u: S^T/dP^T(u+1) as soon as the
    // element-wise warps have read S^T/dP^T(u), and dV/dK(u) once P^T/dS^T(u) are
    // written. The tensor pipe thus runs S^T/dP^T(u+1) and dV/dK(u-1) while the
    // element-wise warps work on u.
    const uint32_t sV = smem_u32(smem + L::kFixA);
    const uint32_t ring = smem_u32(smem + L::kRing);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->fixed_full), 0, wc));
    const bool issuer = elect_one();
    nb_sync(kNbKvK, kNbKvCount);  // K tile in tensor memory
    auto issue_sdp = [&](int v) {  // S^T and dP^T of sub-step v
      const int s = v % L::kStageCount;
      nb_sync(kNbStage + s, kNbStageCount);
      tc_fence_after_sync();
      if (!ok) return;
      const uint32_t sQ = ring + s * L::kStage, sDO = sQ + L::kSubTile;
      mma_tmem_x64<D>(issuer, tmem + kKvColS, tmem + kKvColK, sQ);  // S^T = K Q^T
      mma_128x64<D>(issuer, tmem + kKvColDP, sV, sDO);              // dP^T = V dO^T
      mma_commit_if(issuer, smem_u32(&bars->s_full[0]));
    };
    issue_sdp(0);
    for (int u = 0; u < subs; ++u) {
      const int s = u % L::kStageCount, x = u & 1;
      if (u + 1 < subs) {
        nb_sync(kNbKvRel, kNbKvCount);  // S^T / dP^T(u) are in registers
        issue_sdp(u + 1);
      }
      nb_sync(kNbKvP + x, kNbKvCount);  // P^T / dS^T(u) written
      tc_fence_after_sync();
      if (ok) {
        const uint32_t sQ = ring + s * L::kStage, sDO = sQ + L::kSubTile;
        mma_pd_x_slice<D>(issuer, tmem + colDV, tmem + kKvColPD, sDO, u > 0);       // dV += P^T dO
        mma_pd_x_slice<D>(issuer, tmem + colDK, tmem + kKvColPD + 32, sQ, u > 0);  // dK += dS^T Q
        mma_commit_if(issuer, smem_u32(&bars->empty[s]));    // stage (and its row terms) free
        mma_commit_if(issuer, smem_u32(&bars->pd_free[0]));  // P^T / dS^T free
      }
    }
    if (ok) mma_commit_if(issuer, smem_u32(&bars->acc_full));
  } else {
    // ------------------------------------------------------------ element-wise
    const int q4 = warp & 3;                   // TMEM lane quarter: key rows 32 q4 ..
    const int wg = warp >> 2;                  // query columns [16 wg, 16 wg + 16)
    const int row = q4 * 32 + lane;            // key row in the tile
    const int j = k0 + row;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const int c0 = wg * 16;
    const bool causal_type = p.mask.kind != ATTN_MASK_NONE;
    {
      // K rows of the tile into tensor memory (A operand of S^T = K Q^T): this thread's
      // key row, head-dimension columns [wg D/4, (wg + 1) D/4) as bf16 pairs.
      constexpr int kW = D / 8;  // 32-bit words per thread
      uint32_t kr[kW];
      if (j < p.Nkv) {
        const uint4* src =
            reinterpret_cast<const uint4*>(a.k + ((size_t)bg * p.Nkv + j) * D + wg * (D / 4));
#pragma unroll
        for (int e = 0; e < kW / 4; ++e) {
          const uint4 w = src[e];
          kr[4 * e] = w.x; kr[4 * e + 1] = w.y; kr[4 * e + 2] = w.z; kr[4 * e + 3] = w.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < kW; ++e) kr[e] = 0u;
      }
      if constexpr (kW == 16) tmem_st16(tmem + lane_base + kKvColK + wg * kW, kr);
      else tmem_st8(tmem + lane_base + kKvColK + wg * kW, kr);
      tmem_wait_st();
      tc_fence_before_sync();
      nb_arrive(kNbKvK, kNbKvCount);
    }
    bool ok_all = true;
    for (int u = 0; u < subs; ++u) {
      const int s = u % L::kStageCount, x = u & 1;
      const bool rel = u + 1 < subs;  // the MMA warp waits for this release before u + 1
      int qrow, bh;
      slice(u, qrow, bh);
      const int h = bh - b * p.Hq;
      const int qs = qrow + c0;                  // query of this thread's column 0
      const ScoreK sk = score_consts<kAlibi, kSoftcap>(p, h);
      const DropThr dthr = drop_thr_words(kDrop ? p.drop_thr : 0);
      if (ok_all)
        ok_all = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[0]), u & 1, wc));
      // the stage's row terms arrived with full[s]; observe them
      if (ok_all)
        ok_all = __all_sync(0xffffffffu,
                            mbar_wait(smem_u32(&bars->full[s]), (u / L::kStageCount) & 1, wc));
      if (!ok_all) {  // aborted: keep the barrier schedule with the MMA warp
        if (rel) nb_sync(kNbKvRel, kNbKvCount);
        nb_sync(kNbKvP + x, kNbKvCount);
        continue;
      }
      tc_fence_after_sync();
      uint32_t sr[16], dr[16];
      tmem_ld16(tmem + lane_base + kKvColS + c0, sr);
      tmem_ld16(tmem + lane_base + kKvColDP + c0, dr);
      tmem_wait_ld();
      reg_fence16(sr);
      reg_fence16(dr);
      tc_fence_before_sync();
      if (rel) nb_arrive(kNbKvRel, kNbKvCount);
      const float* lse2 = reinterpret_cast<const float*>(smem + L::kRows + s * L::kRowStage) + c0;
      const float* dl = lse2 + SUB;
      const int* fk = reinterpret_cast<const int*>(dl + SUB);
      const float base = kAlibi ? sk.kb * (float)(j - qs) : 0.f;  // kb*(j - i) at column 0
      uint32_t kf[4];
      if constexpr (kDrop) dropout_flags_dkdv(p, dthr, j, lane, qs, bh, kf);
      uint32_t pp[8], dd[8];
      if (tile_needs_mask(p.mask, qrow & ~(BT - 1), k0, BT))  // warp-uniform
        dkdv_pds<kAlibi, kSoftcap, true, kDrop>(sr, dr, lse2, dl, fk, sk, base, j, qs,
                                                j < p.Nkv, causal_type, kf, pp, dd);
      else
        dkdv_pds<kAlibi, kSoftcap, false, kDrop>(sr, dr, lse2, dl, fk, sk, base, j, qs, true,
                                                 causal_type, kf, pp, dd);
      // P^T / dS^T of sub-step u - 1 must have been read by their MMAs
      if (u >= 1)
        ok_all = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->pd_free[0]), (u - 1) & 1, wc));
      if (!ok_all) {
        nb_sync(kNbKvP + x, kNbKvCount);
        continue;
      }
      tmem_st8(tmem + lane_base + kKvColPD + wg * 8, pp);       // P^T, k-step wg
      tmem_st8(tmem + lane_base + kKvColPD + 32 + wg * 8, dd);  // dS^T
      tmem_wait_st();
      tc_fence_before_sync();
      nb_arrive(kNbKvP + x, kNbKvCount);
    }
    // ---------------------------------------------------------- epilogue
    // warpgroups 0 and 1 write the two halves of dV, 2 and 3 those of dK (times the
    // softmax scale)
    const bool have =
        __all_sync(0xffffffffu, ok_all && mbar_wait(smem_u32(&bars->acc_full), 0, wc));
    tc_fence_after_sync();
    const int which = wg >> 1, half = wg & 1;
    const size_t krow = (size_t)bg * p.Nkv + (j < p.Nkv ? j : 0);
    const uint32_t tacc = tmem + lane_base + (which ? colDK : colDV) + half * (D / 2);
    __nv_bfloat16* dst = (which ? a.dk : a.dv) + krow * D + half * (D / 2);
    const float dsc = kDrop ? p.drop_scale : 1.f;  // dV = (P Z)^T dO / (1 - p); dK from dS'
    store_acc_row<D / 2>(tacc, which ? p.scale * dsc : dsc, dst, have, j < p.Nkv);
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================ dQ
template <int D, bool kAlibi, bool kSoftcap, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using L = LayoutQ<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + L::kBars);
  const Problem& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int bh, qt;
  cta_tile(p.B * p.Hq, a.n_tiles, true, bh, qt);
  const int b = bh / p.Hq, h = bh - b * p.Hq;
  const int bg = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int q0 = qt * BT;
  const TileRange kr = kv_tiles_for_rows(p.mask, q0, BT);
  const int n_k = imax(kr.hi - kr.lo, 0);
  const int subs = 2 * n_k;

  if (n_k == 0) {
    for (int r = threadIdx.x; r < BT; r += kThreads) {
      const int i = q0 + r;
      if (i >= p.Nq) continue;
      uint4* d = reinterpret_cast<uint4*>(a.dq + ((size_t)bh * p.Nq + i) * D);
      for (int c = 0; c < D / 8; ++c) d[c] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  auto slice = [&](int u, int& row, int& head) {  // keys of sub-step u
    head = bg;
    row = kr.lo * BT + u * SUB;
  };

  WaitCtx wc{&bars->abort_flag, p.status};
  if (threadIdx.x == 0) setup_common(bars, L::kStageCount);
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kLoadWarp) {
    load_loop<D, L>(smem, bars, wc, lane, nullptr, q0, bh, &maps.k64, &maps.v64, subs, slice,
                    nullptr, p.nq_pad);
  } else if (warp == kRelayWarp) {
    relay_loop<L::kStageCount>(bars, wc, subs);
  } else if (warp == kMmaWarp) {
    // Same issue scheme as the dK/dV kernel: named barriers only, MMAs predicated on the
    // elect.sync lane.
    const uint32_t ring = smem_u32(smem + L::kRing);
    const bool issuer = elect_one();
    nb_sync(kNbQL, kNbKvCount);  // Q and dO in tensor memory
    // S and dP of sub-step u into buffer u & 1
    auto issue_sdp = [&](int u) {
      const int s = u % L::kStageCount, x = u & 1;
      nb_sync(kNbStage + s, kNbStageCount);
      tc_fence_after_sync();
      const uint32_t sK = ring + s * L::kStage, sV = sK + L::kSubTile;
      mma_tmem_x64<D>(issuer, tmem + col_s(x), tmem + kColQ, sK);         // S = Q K^T
      mma_tmem_x64<D>(issuer, tmem + col_dp(x), tmem + col_do<D>(), sV);  // dP = dO V^T
      mma_commit_if(issuer, smem_u32(&bars->s_full[x]));
    };
    issue_sdp(0);
    if (subs > 1) issue_sdp(1);
    for (int u = 0; u < subs; ++u) {
      const int s = u % L::kStageCount, x = u & 1;
      nb_sync(kNbP + x, kNbPCount);
      tc_fence_after_sync();
      const uint32_t sK = ring + s * L::kStage;
      mma_tmem64_x_slice<D>(issuer, tmem + kColAcc, tmem + col_s(x), sK, u > 0);  // dQ += dS K
      mma_commit_if(issuer, smem_u32(&bars->empty[s]));  // stage consumed once this completes
      if (u + 2 < subs) issue_sdp(u + 2);
    }
    mma_commit_if(issuer, smem_u32(&bars->acc_full));
  } else {
    const int pair = warp >> 3;                // sub-steps u with u % 2 == pair
    const int wg = (warp >> 2) & 1;            // which 32 key columns of a sub-step
    const int row = (warp & 3) * 32 + lane;
    const int i = q0 + row;
    const bool row_ok = i < p.Nq;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int c0 = wg * 32;
    const int x = pair;
    const ScoreK sk = score_consts<kAlibi, kSoftcap>(p, h);
    const DropThr dthr = drop_thr_words(kDrop ? p.drop_thr : 0);
    float lse2 = INFINITY, dlt = 0.f;
    int fk = 0;
    if (row_ok) {  // row terms of the row kernel (lse2 is already L log2 e, +inf if empty)
      lse2 = a.rt.lse2[(size_t)bh * p.nq_pad + i];
      dlt = a.rt.delta[(size_t)bh * p.nq_pad + i];
      fk = a.rt.first[i];
    }
    const int last_key = (p.mask.kind == ATTN_MASK_NONE ? p.Nkv - 1 : imin(i, p.Nkv - 1));
    {
      // Q and dO rows of the tile into tensor memory: warpgroups 0 and 1 copy the two
      // halves of this thread's Q row, 2 and 3 those of its dO row (zeros past Nq).
      const int wq = warp >> 2, half = wq & 1;
      constexpr int kW = D / 4;  // 32-bit words (bf16 pairs) per thread
      uint32_t wv[kW];
      const uint4* src = reinterpret_cast<const uint4*>(
          (wq < 2 ? a.q : a.dout) + ((size_t)bh * p.Nq + (row_ok ? i : 0)) * D + half * (D / 2));
#pragma unroll
      for (int e = 0; e < kW / 4; ++e) {
        const uint4 v = row_ok ? src[e] : make_uint4(0, 0, 0, 0);
        wv[4 * e] = v.x; wv[4 * e + 1] = v.y; wv[4 * e + 2] = v.z; wv[4 * e + 3] = v.w;
      }
      const uint32_t dst = tmem + lane_base + (wq < 2 ? kColQ : col_do<D>()) + half * (D / 4);
      if constexpr (kW == 32) tmem_st32(dst, wv);
      else tmem_st16(dst, wv);
      tmem_wait_st();
      tc_fence_before_sync();
      nb_arrive(kNbQL, kNbKvCount);
    }
    bool ok_all = true;
    for (int u = pair; u < subs; u += 2) {
      const int kt0 = (kr.lo + (u >> 1)) * BT;
      const int ks = kr.lo * BT + u * SUB + c0;  // key of this thread's column 0
      if (ok_all)
        ok_all = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[x]), (u >> 1) & 1, wc));
      if (!ok_all) {  // aborted: keep the barrier schedule with the MMA warp
        nb_sync(kNbP + x, kNbPCount);
        continue;
      }
      tc_fence_after_sync();
      const uint32_t tS = tmem + lane_base + col_s(x) + c0;
      const uint32_t tDP = tmem + lane_base + col_dp(x) + c0;
      uint32_t sr[32], dr[32];
      tmem_ld32(tS, sr);
      tmem_ld32(tDP, dr);
      tmem_wait_ld();
      reg_fence32(sr);
      reg_fence32(dr);
      const float base = kAlibi ? sk.kb * (float)(ks - i) : 0.f;  // kb*(j - i) at column 0
      uint32_t kf[8];
      if constexpr (kDrop) dropout_flags_dq(p, dthr, i, ks, bh, kf);
      uint32_t dd[16];
      if (tile_needs_mask(p.mask, q0, kt0, BT))  // warp-uniform
        dq_ds<kAlibi, kSoftcap, true, kDrop>(sr, dr, sk, base, lse2, dlt, fk - ks, last_key - ks,
                                             kf, dd);
      else
        dq_ds<kAlibi, kSoftcap, false, kDrop>(sr, dr, sk, base, lse2, dlt, 0, 0, kf, dd);
      tmem_st16(tS, dd);  // dS, bf16 pairs
      tmem_wait_st();
      tc_fence_before_sync();
      nb_arrive(kNbP + x, kNbPCount);
    }
    // pair 0 writes dQ: warpgroup wg writes columns [wg * D/2, (wg + 1) * D/2)
    const bool have =
        __all_sync(0xffffffffu, ok_all && mbar_wait(smem_u32(&bars->acc_full), 0, wc));
    tc_fence_after_sync();
    if (pair == 0) {  // warp-uniform
      const uint32_t tq = tmem + lane_base + kColAcc + wg * (D / 2);
      __nv_bfloat16* dst = a.dq + ((size_t)bh * p.Nq + (row_ok ? i : 0)) * D + wg * (D / 2);
      store_acc_row<D / 2>(tq, kDrop ? p.scale * p.drop_scale : p.scale, dst, have, row_ok);
    }
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kA, bool kS, bool kDrop>
cudaError_t launch_variant(const BwdArgs& kv_args, const BwdArgs& q_args, const BwdMaps& maps,
                           int grid_kv, int grid_q, cudaStream_t st) {
  auto k1 = dkdv_kernel<D, kA, kS, kDrop>;
  auto k2 = dq_kernel<D, kA, kS, kDrop>;
  constexpr int kSmemKv = LayoutKv<D>::kAlloc, kSmemQ = LayoutQ<D>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemKv);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemQ);
  if (e != cudaSuccess) return e;
  if (grid_kv > 0) k1<<<grid_kv, kThreads, kSmemKv, st>>>(maps, kv_args);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (grid_q > 0) k2<<<grid_q, kThreads, kSmemQ, st>>>(maps, q_args);
  return cudaGetLastError();
}

template <int D, bool kDrop>
cudaError_t launch_dd(const BwdArgs& ka, const BwdArgs& qa, const BwdMaps& maps, int gk, int gq,
                      cudaStream_t st) {
  const bool al = ka.p.score_kind & ATTN_SCORE_ALIBI, sc = ka.p.score_kind & ATTN_SCORE_SOFTCAP;
  if (al && sc) return launch_variant<D, true, true, kDrop>(ka, qa, maps, gk, gq, st);
  if (al) return launch_variant<D, true, false, kDrop>(ka, qa, maps, gk, gq, st);
  if (sc) return launch_variant<D, false, true, kDrop>(ka, qa, maps, gk, gq, st);
  return launch_variant<D, false, false, kDrop>(ka, qa, maps, gk, gq, st);
}

template <int D>
cudaError_t launch_d(const BwdArgs& ka, const BwdArgs& qa, const BwdMaps& maps, int gk, int gq,
                     cudaStream_t st) {
  if (ka.p.score_kind & ATTN_SCORE_DROPOUT) return launch_dd<D, true>(ka, qa, maps, gk, gq, st);
  return launch_dd<D, false>(ka, qa, maps, gk, gq, st);
}

}  // namespace

cudaError_t launch_bwd_tc(const Problem& p, const BwdMaps& maps, const RowTerms& rt,
                          const __nv_bfloat16* q, const __nv_bfloat16* dout,
                          const __nv_bfloat16* k, __nv_bfloat16* dq, __nv_bfloat16* dk,
                          __nv_bfloat16* dv,
                          bool run_dkdv, bool run_dq, cudaStream_t st) {
  BwdArgs ka{p, rt, q, dout, k, dq, dk, dv, ceil_div(p.Nkv, BT)};
  BwdArgs qa{p, rt, q, dout, k, dq, dk, dv, ceil_div(p.Nq, BT)};
  const long long gk = run_dkdv ? (long long)ka.n_tiles * p.B * p.Hkv : 0;
  const long long gq = run_dq ? (long long)qa.n_tiles * p.B * p.Hq : 0;
  if (gk > 0x7fffffffLL || gq > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (p.d == 64) return launch_d<64>(ka, qa, maps, (int)gk, (int)gq, st);
  return launch_d<128>(ka, qa, maps, (int)gk, (int)gq, st);
}

}  // namespace attn
