// Backward attention on the tcgen05 tensor cores (sm_103a).
//
// "FlashAttention/es" ("Paso hacia atrás y recomputación") rebuilds S and P tile
// by tile from the saved log-sum-exp L instead of storing P. With
// P_ij = exp(s_ij - L_i) and D_i = rowsum(dO_i o O_i) (computed by a separate
// row-dot kernel), the gradients are
//     dV = P^T dO,   dP = dO V^T,   dS = P o (dP - D) [x soft-cap derivative],
//     dK = scale dS^T Q,   dQ = scale dS K.
// Two kernels, both deterministic (fixed summation order, no atomics):
//   * dkdv: one CTA per (batch, kv head, 128-key tile); it walks the query heads of
//     its group and the query tiles the mask leaves, 64 query rows at a time
//     ("sub-steps"): S^T = K Q^T and dP^T = V dO^T into tensor memory, P^T and dS^T
//     (bf16) back into tensor memory, then dV += P^T dO and dK += dS^T Q;
//   * dq: one CTA per (batch, query head, 128-row tile); it walks the key tiles 64
//     keys at a time: S = Q K^T and dP = dO V^T, dS back into tensor memory, then
//     dQ += dS K.
// S and dP are double-buffered in tensor memory (two 64-column buffers each), so
// the MMAs of the next sub-step run while the element-wise warps work on this one.
// Warps 0-7 do the element-wise work (warpgroup w takes columns [32w, 32w+32) of a
// sub-step; one thread per TMEM lane = row), warp 8 streams tiles with TMA, warp 9
// owns tensor memory and issues the MMAs.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int BT = 128;          // tile side (rows, keys)
constexpr int SUB = 64;          // columns per sub-step
constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kStages = 2;       // ring depth for the streamed operand pairs
constexpr int kHeadGroup = 4;
constexpr float kLog2e = 1.4426950408889634f;

// Tensor memory columns: S buffers, dP buffers (64 each), then the accumulators.
__device__ __forceinline__ uint32_t col_s(int x) { return x * 64; }
__device__ __forceinline__ uint32_t col_dp(int x) { return 128 + x * 64; }
constexpr uint32_t kColAcc = 256;

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

// P and dS of one element from the pre-cap score in log2 units (or in 2 log2e / c
// units under the soft-cap); lse2 = L * log2e (+inf for a row with no key).
template <bool kSoftcap>
__device__ __forceinline__ void p_and_ds(float pre, float lse2, float dp, float delta,
                                         float capA, bool ok, float& pr, float& ds) {
  float s2 = pre, dcap = 1.f;
  if (kSoftcap) {
    const float t = 1.0f - 2.0f * rcp_approx(1.0f + ex2_approx(pre));  // tanh(pre_cap / c)
    s2 = capA * t;
    dcap = 1.0f - t * t;
  }
  pr = ok ? ex2_approx(s2 - lse2) : 0.f;
  ds = pr * (dp - delta) * dcap;
}

template <int D>
struct KVLayout {  // dkdv kernel shared memory
  static constexpr int kChunk = BT * 128;
  static constexpr int kTile = BT * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kRing = 2 * kTile;             // stages of {Q, dO}
  static constexpr int kStage = 2 * kTile;
  static constexpr int kRows = kRing + kStages * kStage;  // per stage: lse2, delta, first key
  static constexpr int kRowStage = 3 * BT * 4;
  static constexpr int kBars = kRows + kStages * kRowStage;
  static constexpr int kAlloc = kBars + 256 + 1024;
};

template <int D>
struct QLayout {  // dq kernel shared memory
  static constexpr int kChunk = BT * 128;
  static constexpr int kTile = BT * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kDO = kTile;
  static constexpr int kRing = 2 * kTile;             // stages of {K, V}
  static constexpr int kStage = 2 * kTile;
  static constexpr int kBars = kRing + kStages * kStage;
  static constexpr int kAlloc = kBars + 256 + 1024;
};

struct BwdBars {
  uint64_t fixed_full;             // the tiles loaded once (K,V or Q,dO)
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t s_full[2];              // S_x and dP_x in TMEM
  uint64_t p_full[2];              // P_x / dS_x written back to TMEM
  uint64_t acc_full;               // accumulators final
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdArgs {
  Problem p;
  const float* lse;
  const float* delta;
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

__device__ __forceinline__ void setup_common(BwdBars* bars, uint32_t stage_full_count,
                                             uint32_t stage_empty_count) {
  mbar_init(smem_u32(&bars->fixed_full), 1);
  for (int s = 0; s < kStages; ++s) {
    mbar_init(smem_u32(&bars->full[s]), stage_full_count);
    mbar_init(smem_u32(&bars->empty[s]), stage_empty_count);
  }
  for (int x = 0; x < 2; ++x) {
    mbar_init(smem_u32(&bars->s_full[x]), 1);
    mbar_init(smem_u32(&bars->p_full[x]), 8);  // one arrival per element-wise warp
  }
  mbar_init(smem_u32(&bars->acc_full), 1);
  bars->abort_flag = 0;
  fence_barrier_init();
}

// D[128 x 64] = A B^T over the head dimension: A a K-major tile of 128 rows, B the
// 64 rows starting at `b` of a K-major tile (both written by TMA, 128-byte swizzle).
template <int D>
__device__ __forceinline__ void mma_128x64(uint32_t d_tmem, uint32_t a, uint32_t b) {
  constexpr uint32_t id = idesc_bf16_f32(BT, SUB, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * (BT * 128) + (kk & 3) * 32;
    mma_ss(d_tmem, smem_desc_sw128(a + off, 16, 1024), smem_desc_sw128(b + off, 16, 1024), id,
           kk > 0 ? 1u : 0u);
  }
}

// D[128 x D] (+)= A_tmem[128 x 64] B[64 x D]: A = bf16 pairs in TMEM, written by the
// two element-wise warpgroups at columns [0,16) and [32,48) of a_tmem; B = the 64
// rows starting at `b` of a tile used MN-major.
template <int D>
__device__ __forceinline__ void mma_tmem64_x_tile(uint32_t d_tmem, uint32_t a_tmem, uint32_t b,
                                                  bool accumulate) {
  constexpr uint32_t id = idesc_bf16_f32(BT, D, false, true);
#pragma unroll
  for (int kk = 0; kk < SUB / 16; ++kk) {
    const uint32_t acol = (kk < 2) ? kk * 8 : 32 + (kk - 2) * 8;
    mma_ts(d_tmem, a_tmem + acol, smem_desc_sw128(b + kk * 16 * 128, BT * 128, 1024), id,
           (accumulate || kk > 0) ? 1u : 0u);
  }
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

// ============================================================================ dK, dV
template <int D, bool kAlibi, bool kSoftcap>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const BwdArgs a) {
  using L = KVLayout<D>;
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
  const int steps = n_q * G;  // (head, query tile) pairs, head-major
  const int subs = 2 * steps; // 64-row sub-steps
  if (steps == 0) {  // no query sees these keys: zero gradients
    for (int r = threadIdx.x; r < BT; r += kThreads) {
      const int j = k0 + r;
      if (j >= p.Nkv) continue;
      uint4* dkr = reinterpret_cast<uint4*>(a.dk + ((size_t)bg * p.Nkv + j) * D);
      uint4* dvr = reinterpret_cast<uint4*>(a.dv + ((size_t)bg * p.Nkv + j) * D);
      for (int c = 0; c < D / 8; ++c) { dkr[c] = make_uint4(0, 0, 0, 0); dvr[c] = make_uint4(0, 0, 0, 0); }
    }
    return;
  }

  WaitCtx wc{&bars->abort_flag, p.status};
  if (threadIdx.x == 0) setup_common(bars, 1 + 32, 1 + 8);
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t colDV = kColAcc, colDK = kColAcc + D;

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      const uint32_t fb = smem_u32(&bars->fixed_full);
      mbar_arrive_expect_tx(fb, 2 * L::kTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(smem_u32(smem + L::kK + c * L::kChunk), &tm_k, fb, c * 64, k0, bg);
        tma_load_3d(smem_u32(smem + L::kV + c * L::kChunk), &tm_v, fb, c * 64, k0, bg);
      }
    }
    for (int st = 0; st < steps; ++st) {
      const int s = st % kStages, use = st / kStages;
      const int h = g * G + st / n_q;
      const int q0 = (qr.lo + st % n_q) * BT;
      const int bh = b * p.Hq + h;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(smem_u32(&bars->empty[s]), (use & 1) ^ 1, wc);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      const uint32_t full = smem_u32(&bars->full[s]);
      if (lane == 0) {
        mbar_arrive_expect_tx(full, 2 * L::kTile);
        uint8_t* stg = smem + L::kRing + s * L::kStage;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(smem_u32(stg + c * L::kChunk), &tm_q, full, c * 64, q0, bh);
          tma_load_3d(smem_u32(stg + L::kTile + c * L::kChunk), &tm_do, full, c * 64, q0, bh);
        }
      }
      // Row data of the 128 query rows: L * log2e (+inf for a row with no key, so
      // that exp2(s - lse2) = 0), D, and the row's first allowed key.
      float* lse2 = reinterpret_cast<float*>(smem + L::kRows + s * L::kRowStage);
      float* dl = lse2 + BT;
      int* fk = reinterpret_cast<int*>(dl + BT);
#pragma unroll
      for (int e = 0; e < BT / 32; ++e) {
        const int r = e * 32 + lane, i = q0 + r;
        float lv = INFINITY, dv = 0.f;
        int f = 0x7fffffff;  // rows past Nq see no key
        if (i < p.Nq) {
          const float l = a.lse[(size_t)bh * p.Nq + i];
          lv = l == -INFINITY ? INFINITY : l * kLog2e;
          dv = a.delta[(size_t)bh * p.Nq + i];
          f = first_key(p.mask, i);
        }
        lse2[r] = lv;
        dl[r] = dv;
        fk[r] = f;
      }
      mbar_arrive(full);
    }
    if (lane == 0) {  // let in-flight copies land before the CTA can exit
      mbar_wait(smem_u32(&bars->fixed_full), 0, wc);
      for (int st = imax(0, steps - kStages); st < steps; ++st)
        mbar_wait(smem_u32(&bars->full[st % kStages]), (st / kStages) & 1, wc);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);
      bool ok = mbar_wait(smem_u32(&bars->fixed_full), 0, wc);
      // S^T and dP^T of sub-step u into buffer u & 1 (query rows 64*(u&1) of step u/2).
      auto issue_sdp = [&](int u) -> bool {
        const int st = u >> 1, s = st % kStages, x = u & 1;
        if (x == 0) {
          if (!mbar_wait(smem_u32(&bars->full[s]), (st / kStages) & 1, wc)) return false;
          tc_fence_after_sync();
        }
        const uint32_t sQ = smem_u32(smem + L::kRing + s * L::kStage) + x * SUB * 128;
        const uint32_t sDO = sQ + L::kTile;
        mma_128x64<D>(tmem + col_s(x), sK, sQ);    // S^T = K Q^T
        mma_128x64<D>(tmem + col_dp(x), sV, sDO);  // dP^T = V dO^T
        mma_commit(smem_u32(&bars->s_full[x]));
        return true;
      };
      if (ok) ok = issue_sdp(0);
      if (ok && subs > 1) ok = issue_sdp(1);
      for (int u = 0; ok && u < subs; ++u) {
        const int st = u >> 1, s = st % kStages, x = u & 1;
        if (!mbar_wait(smem_u32(&bars->p_full[x]), (u >> 1) & 1, wc)) break;
        tc_fence_after_sync();
        const uint32_t sQ = smem_u32(smem + L::kRing + s * L::kStage) + x * SUB * 128;
        const uint32_t sDO = sQ + L::kTile;
        mma_tmem64_x_tile<D>(tmem + colDV, tmem + col_s(x), sDO, u > 0);   // dV += P^T dO
        mma_tmem64_x_tile<D>(tmem + colDK, tmem + col_dp(x), sQ, u > 0);   // dK += dS^T Q
        if (x == 1) mma_commit(smem_u32(&bars->empty[s]));  // step fully consumed
        if (u + 2 < subs) ok = issue_sdp(u + 2);
      }
      mma_commit(smem_u32(&bars->acc_full));
    }
  } else {
    // ------------------------------------------------------------ element-wise
    const int wg = warp >> 2;                  // which 32 columns of a sub-step
    const int row = (warp & 3) * 32 + lane;    // key row in the tile
    const int j = k0 + row;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int c0 = wg * 32;
    const bool causal_type = p.mask.kind != ATTN_MASK_NONE;
    int done = 0;
    for (int u = 0; u < subs; ++u, ++done) {
      const int st = u >> 1, s = st % kStages, x = u & 1;
      const int h = g * G + st / n_q;
      const int q0 = (qr.lo + st % n_q) * BT;
      const int qs = q0 + x * SUB + c0;          // query of this thread's column 0
      const ScoreK sk = score_consts<kAlibi, kSoftcap>(p, h);
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[x]), (u >> 1) & 1, wc)))
        break;
      // the row data were written before full[s] completed; observe them
      if (x == 0 &&
          !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->full[s]), (st / kStages) & 1, wc)))
        break;
      tc_fence_after_sync();
      const int roff = x * SUB + c0;
      const float* lse2 = reinterpret_cast<const float*>(smem + L::kRows + s * L::kRowStage) + roff;
      const float* dl = lse2 + BT;
      const int* fk = reinterpret_cast<const int*>(dl + BT);
      const uint32_t tS = tmem + lane_base + col_s(x) + c0;
      const uint32_t tDP = tmem + lane_base + col_dp(x) + c0;
      uint32_t sr[32], dr[32];
      tmem_ld32(tS, sr);
      tmem_ld32(tDP, dr);
      tmem_wait_ld();
      reg_fence32(sr);
      reg_fence32(dr);
      const bool masked = tile_needs_mask(p.mask, q0, k0, BT);
      const float base = kAlibi ? sk.kb * (float)(j - qs) : 0.f;  // kb*(j - i) at column 0
      uint32_t pp[16], dd[16];
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const float4 lv = reinterpret_cast<const float4*>(lse2)[e4];
        const float4 dv = reinterpret_cast<const float4*>(dl)[e4];
        const float lvs[4] = {lv.x, lv.y, lv.z, lv.w};
        const float dvs[4] = {dv.x, dv.y, dv.z, dv.w};
        float pv[4], dsv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int col = e4 * 4 + q;
          const float xs = __uint_as_float(sr[col]);
          bool ok = true;
          if (masked) {
            const int i = qs + col;
            ok = j < p.Nkv && (!causal_type || (i >= j && fk[col] <= j));
          }
          if (!kAlibi && !kSoftcap) {
            const float pr = ok ? ex2_approx(fmaf(xs, sk.k1, -lvs[q])) : 0.f;
            pv[q] = pr;
            dsv[q] = pr * (__uint_as_float(dr[col]) - dvs[q]);
          } else {
            const float pre =
                kAlibi ? fmaf(xs, sk.k1, fmaf(-(float)col, sk.kb, base)) : xs * sk.k1;
            p_and_ds<kSoftcap>(pre, lvs[q], __uint_as_float(dr[col]), dvs[q], sk.capA, ok,
                               pv[q], dsv[q]);
          }
        }
        pp[2 * e4] = pack_bf16x2(pv[0], pv[1]);
        pp[2 * e4 + 1] = pack_bf16x2(pv[2], pv[3]);
        dd[2 * e4] = pack_bf16x2(dsv[0], dsv[1]);
        dd[2 * e4 + 1] = pack_bf16x2(dsv[2], dsv[3]);
      }
      tmem_st16(tS, pp);   // P^T, bf16 pairs, in this warpgroup's first 16 columns
      tmem_st16(tDP, dd);  // dS^T
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars->p_full[x]));
        if (x == 1) mbar_arrive(smem_u32(&bars->empty[s]));  // done with the row data
      }
    }
    // ---------------------------------------------------------- epilogue
    bool have = done == subs;
    have = __all_sync(0xffffffffu, have && mbar_wait(smem_u32(&bars->acc_full), 0, wc));
    tc_fence_after_sync();
    const size_t krow = (size_t)bg * p.Nkv + (j < p.Nkv ? j : 0);
    // warpgroup 0 writes dV, warpgroup 1 writes dK (times the softmax scale)
    const uint32_t tacc = tmem + lane_base + (wg == 0 ? colDV : colDK);
    __nv_bfloat16* dst = (wg == 0 ? a.dv : a.dk) + krow * D;
    store_acc_row<D>(tacc, wg == 0 ? 1.f : p.scale, dst, have, j < p.Nkv);
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
template <int D, bool kAlibi, bool kSoftcap>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const BwdArgs a) {
  using L = QLayout<D>;
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

  WaitCtx wc{&bars->abort_flag, p.status};
  if (threadIdx.x == 0) setup_common(bars, 1, 1);
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kLoadWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint32_t fb = smem_u32(&bars->fixed_full);
      mbar_arrive_expect_tx(fb, 2 * L::kTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(smem_u32(smem + L::kQ + c * L::kChunk), &tm_q, fb, c * 64, q0, bh);
        tma_load_3d(smem_u32(smem + L::kDO + c * L::kChunk), &tm_do, fb, c * 64, q0, bh);
      }
      for (int st = 0; st < n_k; ++st) {
        const int s = st % kStages, use = st / kStages;
        if (!mbar_wait(smem_u32(&bars->empty[s]), (use & 1) ^ 1, wc)) break;
        const uint32_t full = smem_u32(&bars->full[s]);
        mbar_arrive_expect_tx(full, 2 * L::kTile);
        uint8_t* stg = smem + L::kRing + s * L::kStage;
        const int krow = (kr.lo + st) * BT;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(smem_u32(stg + c * L::kChunk), &tm_k, full, c * 64, krow, bg);
          tma_load_3d(smem_u32(stg + L::kTile + c * L::kChunk), &tm_v, full, c * 64, krow, bg);
        }
      }
      mbar_wait(fb, 0, wc);
      for (int st = imax(0, n_k - kStages); st < n_k; ++st)
        mbar_wait(smem_u32(&bars->full[st % kStages]), (st / kStages) & 1, wc);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t sQ = smem_u32(smem + L::kQ), sDO = smem_u32(smem + L::kDO);
      bool ok = mbar_wait(smem_u32(&bars->fixed_full), 0, wc);
      // S and dP of sub-step u into buffer u & 1 (keys 64*(u&1) of key tile u/2).
      auto issue_sdp = [&](int u) -> bool {
        const int st = u >> 1, s = st % kStages, x = u & 1;
        if (x == 0) {
          if (!mbar_wait(smem_u32(&bars->full[s]), (st / kStages) & 1, wc)) return false;
          tc_fence_after_sync();
        }
        const uint32_t sK = smem_u32(smem + L::kRing + s * L::kStage) + x * SUB * 128;
        const uint32_t sV = sK + L::kTile;
        mma_128x64<D>(tmem + col_s(x), sQ, sK);     // S = Q K^T
        mma_128x64<D>(tmem + col_dp(x), sDO, sV);   // dP = dO V^T
        mma_commit(smem_u32(&bars->s_full[x]));
        return true;
      };
      if (ok) ok = issue_sdp(0);
      if (ok && subs > 1) ok = issue_sdp(1);
      for (int u = 0; ok && u < subs; ++u) {
        const int st = u >> 1, s = st % kStages, x = u & 1;
        if (!mbar_wait(smem_u32(&bars->p_full[x]), (u >> 1) & 1, wc)) break;
        tc_fence_after_sync();
        const uint32_t sK = smem_u32(smem + L::kRing + s * L::kStage) + x * SUB * 128;
        mma_tmem64_x_tile<D>(tmem + kColAcc, tmem + col_s(x), sK, u > 0);  // dQ += dS K
        if (x == 1) mma_commit(smem_u32(&bars->empty[s]));  // key tile fully consumed
        if (u + 2 < subs) ok = issue_sdp(u + 2);
      }
      mma_commit(smem_u32(&bars->acc_full));
    }
  } else {
    const int wg = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const int i = q0 + row;
    const bool row_ok = i < p.Nq;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int c0 = wg * 32;
    const ScoreK sk = score_consts<kAlibi, kSoftcap>(p, h);
    float lse2 = INFINITY, dlt = 0.f;
    int fk = 0;
    if (row_ok) {
      const float l = a.lse[(size_t)bh * p.Nq + i];
      lse2 = l == -INFINITY ? INFINITY : l * kLog2e;
      dlt = a.delta[(size_t)bh * p.Nq + i];
      fk = first_key(p.mask, i);
    }
    const int last_key = (p.mask.kind == ATTN_MASK_NONE ? p.Nkv - 1 : imin(i, p.Nkv - 1));
    const float nlse2 = -lse2;
    int done = 0;
    for (int u = 0; u < subs; ++u, ++done) {
      const int st = u >> 1, x = u & 1;
      const int kt0 = (kr.lo + st) * BT;
      const int ks = kt0 + x * SUB + c0;  // key of this thread's column 0
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[x]), (u >> 1) & 1, wc)))
        break;
      tc_fence_after_sync();
      const uint32_t tS = tmem + lane_base + col_s(x) + c0;
      const uint32_t tDP = tmem + lane_base + col_dp(x) + c0;
      uint32_t sr[32], dr[32];
      tmem_ld32(tS, sr);
      tmem_ld32(tDP, dr);
      tmem_wait_ld();
      reg_fence32(sr);
      reg_fence32(dr);
      const bool masked = tile_needs_mask(p.mask, q0, kt0, BT);
      const int c_lo = fk - ks, c_hi = last_key - ks;  // allowed columns of this row
      const float base = kAlibi ? sk.kb * (float)(ks - i) : 0.f;  // kb*(j - i) at column 0
      uint32_t dd[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float dsv[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int col = 2 * e + q;
          const float xs = __uint_as_float(sr[col]);
          const bool ok = !masked || (col >= c_lo && col <= c_hi);
          if (!kAlibi && !kSoftcap) {
            const float pr = ok ? ex2_approx(fmaf(xs, sk.k1, nlse2)) : 0.f;
            dsv[q] = pr * (__uint_as_float(dr[col]) - dlt);
          } else {
            const float pre =
                kAlibi ? fmaf(xs, sk.k1, fmaf((float)col, sk.kb, base)) : xs * sk.k1;
            float pr;
            p_and_ds<kSoftcap>(pre, lse2, __uint_as_float(dr[col]), dlt, sk.capA, ok, pr,
                               dsv[q]);
          }
        }
        dd[e] = pack_bf16x2(dsv[0], dsv[1]);
      }
      tmem_st16(tS, dd);  // dS, bf16 pairs
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[x]));
    }
    bool have = done == subs;
    have = __all_sync(0xffffffffu, have && mbar_wait(smem_u32(&bars->acc_full), 0, wc));
    tc_fence_after_sync();
    // warpgroup 0 writes dQ columns [0, D/2), warpgroup 1 columns [D/2, D)
    const uint32_t tq = tmem + lane_base + kColAcc + wg * (D / 2);
    __nv_bfloat16* dst = a.dq + ((size_t)bh * p.Nq + (row_ok ? i : 0)) * D + wg * (D / 2);
    store_acc_row<D / 2>(tq, p.scale, dst, have, row_ok);
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kA, bool kS>
cudaError_t launch_variant(const BwdArgs& kv_args, const BwdArgs& q_args, const CUtensorMap& tq,
                           const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                           int grid_kv, int grid_q, cudaStream_t st) {
  auto k1 = dkdv_kernel<D, kA, kS>;
  auto k2 = dq_kernel<D, kA, kS>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       KVLayout<D>::kAlloc);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, QLayout<D>::kAlloc);
  if (e != cudaSuccess) return e;
  if (grid_kv > 0) k1<<<grid_kv, kThreads, KVLayout<D>::kAlloc, st>>>(tq, tk, tv, tdo, kv_args);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (grid_q > 0) k2<<<grid_q, kThreads, QLayout<D>::kAlloc, st>>>(tq, tk, tv, tdo, q_args);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const BwdArgs& ka, const BwdArgs& qa, const CUtensorMap& tq,
                     const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                     int gk, int gq, cudaStream_t st) {
  const bool al = ka.p.score_kind & ATTN_SCORE_ALIBI, sc = ka.p.score_kind & ATTN_SCORE_SOFTCAP;
  if (al && sc) return launch_variant<D, true, true>(ka, qa, tq, tk, tv, tdo, gk, gq, st);
  if (al) return launch_variant<D, true, false>(ka, qa, tq, tk, tv, tdo, gk, gq, st);
  if (sc) return launch_variant<D, false, true>(ka, qa, tq, tk, tv, tdo, gk, gq, st);
  return launch_variant<D, false, false>(ka, qa, tq, tk, tv, tdo, gk, gq, st);
}

}  // namespace

cudaError_t launch_bwd_tc(const Problem& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const float* lse,
                          const float* delta, __nv_bfloat16* dq, __nv_bfloat16* dk,
                          __nv_bfloat16* dv, bool run_dkdv, bool run_dq, cudaStream_t st) {
  BwdArgs ka{p, lse, delta, dq, dk, dv, ceil_div(p.Nkv, BT)};
  BwdArgs qa{p, lse, delta, dq, dk, dv, ceil_div(p.Nq, BT)};
  const long long gk = run_dkdv ? (long long)ka.n_tiles * p.B * p.Hkv : 0;
  const long long gq = run_dq ? (long long)qa.n_tiles * p.B * p.Hq : 0;
  if (gk > 0x7fffffffLL || gq > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (p.d == 64) return launch_d<64>(ka, qa, tq, tk, tv, tdo, (int)gk, (int)gq, st);
  return launch_d<128>(ka, qa, tq, tk, tv, tdo, (int)gk, (int)gq, st);
}

}  // namespace attn
