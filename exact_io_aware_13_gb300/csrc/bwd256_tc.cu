// Backward attention at head dimension 256 on the tcgen05 tensor cores (sm_103a).
//
// The gradients are those of the d = 64 / 128 kernels ("FlashAttention/es", "Paso hacia
// atrás y recomputación": S and P rebuilt tile by tile from the saved log-sum-exp):
//     dV = P^T dO,   dP = dO V^T,   dS = P o (dP - D) [x soft-cap derivative],
//     dK = scale dS^T Q,   dQ = scale dS K,
// with D and L log2 e from the row kernel. At d = 256 a 128-row accumulator of the head
// dimension takes 256 of the 512 tensor-memory columns, so dK and dV of one key tile no
// longer fit beside each other and beside S^T / dP^T: the keys are walked twice.
//   * dv256: one CTA per (batch, kv head, 128-key tile), walking the query rows of its
//     group 64 at a time like the d <= 128 dK/dV kernel. TMEM: the K tile (bf16 pairs,
//     A operand of S^T = K Q^T), two S^T buffers, dV. P^T is written over the S^T it
//     came from, so S^T of sub-step u + 2 runs while the element-wise warps work on u + 1.
//     Three stages of Q / dO slices (64 KB each) stream through shared memory.
//   * dk256: the same walk for dK. TMEM: K, S^T, dP^T, dK (all 512 columns); dS^T is
//     written over S^T; V stays in shared memory (64 KB) beside two Q / dO stages.
//   * dq256: one CTA per (batch, query head, 128-row tile), walking the key tiles 64 keys
//     at a time. TMEM: the Q tile (A operand of S = Q K^T), S, dP, dQ; dS is written over
//     S; dO stays in shared memory beside two K / V stages.
// MMA FLOPs per allowed pair: 4 d (dv256) + 6 d (dk256) + 6 d (dq256) for 10 d useful.
// Element-wise warps: 16, warp w on TMEM lane quarter w % 4 and the 16 columns
// [16 (w / 4), 16 (w / 4) + 16) of each 64-column sub-step; each writes its bf16 pairs
// over the first half of the 16 fp32 columns it read, so no warp writes columns another
// warp may still be reading.
#include <type_traits>

#include "bwd_common.cuh"

namespace attn {
namespace {

constexpr int D256 = 256;
// Tensor memory columns (all three kernels): the fixed 128-row operand as bf16 pairs
// (K, or Q for dq256), S or S^T buffer 0, buffer 1 (dv256) or dP / dP^T, accumulator.
constexpr uint32_t k256ColFix = 0, k256ColS0 = 128, k256ColS1 = 192, k256ColDP = 192,
                   k256ColAcc = 256;
__device__ __forceinline__ uint32_t col_s256(int x) { return x ? k256ColS1 : k256ColS0; }

using LayoutV256 = Layout<D256, 3, 0, true>;   // Q / dO stages + row terms
using LayoutK256 = Layout<D256, 2, 1, true>;   // V fixed, Q / dO stages + row terms
using LayoutQ256 = Layout<D256, 2, 1, false>;  // dO fixed, K / V stages
static_assert(LayoutV256::kAlloc <= 232448 && LayoutK256::kAlloc <= 232448 &&
                  LayoutQ256::kAlloc <= 232448,
              "shared memory per CTA");
static_assert(3 <= kMaxStages && kNbStage + 3 <= kNbKvRel, "stage barriers");

// D[128 x 256] (+)= A_tmem[128 x 64] B[64 x 256]: k-step kk (16 rows of B) reads A's bf16
// pairs from columns [16 kk, 16 kk + 8), where element-wise warpgroup kk wrote them; B is
// a 64-row stage slice used MN-major (its 64-column slabs 8 KB apart).
__device__ __forceinline__ void mma_strided_x_slice(bool pred, uint32_t d_tmem, uint32_t a_tmem,
                                                    uint32_t b, bool accumulate) {
  constexpr uint32_t id = idesc_bf16_f32(BT, D256, false, true);
  const uint64_t db = smem_desc_sw128(b, SUB * 128, 1024);
#pragma unroll
  for (int kk = 0; kk < SUB / 16; ++kk)
    mma_ts_if(pred, d_tmem, a_tmem + kk * 16, db + ((kk * 16 * 128) >> 4), id,
              (accumulate || kk > 0) ? 1u : 0u);
}

// Key-row element-wise step (dv256 / dk256): key row j, the 16 query columns from qs
// with their lse2 / delta / first key in shared memory. kDs false: P^T; true: dS^T.
template <bool kAlibi, bool kSoftcap, bool kMasked, bool kDs>
__device__ __forceinline__ void key_row_elems(const uint32_t (&sr)[16], const uint32_t (&dr)[16],
                                              const float* lse2, const float* dl, const int* fk,
                                              const ScoreK& sk, float base, int j, int qs,
                                              bool key_ok, bool causal_type, uint32_t (&out)[8]) {
#pragma unroll
  for (int e4 = 0; e4 < 4; ++e4) {
    const float4 lv = reinterpret_cast<const float4*>(lse2)[e4];
    const float4 dv = kDs ? reinterpret_cast<const float4*>(dl)[e4] : make_float4(0, 0, 0, 0);
    const float lvs[4] = {lv.x, lv.y, lv.z, lv.w};
    const float dvs[4] = {dv.x, dv.y, dv.z, dv.w};
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int col = e4 * 4 + q;
      bool ok = true;
      if (kMasked) {
        const int i = qs + col;
        ok = key_ok && (!causal_type || (i >= j && fk[col] <= j));
      }
      float pr, ds;
      p_and_ds<kAlibi, kSoftcap>(__uint_as_float(sr[col]), sk,
                                 kAlibi ? fmaf(-(float)col, sk.kb, base) : 0.f, lvs[q],
                                 kDs ? __uint_as_float(dr[col]) : 0.f, dvs[q], ok, 0xffffffffu,
                                 pr, ds);
      v[q] = kDs ? ds : pr;
    }
    out[2 * e4] = pack_bf16x2(v[0], v[1]);
    out[2 * e4 + 1] = pack_bf16x2(v[2], v[3]);
  }
}

// Query-row element-wise step (dq256): one query row, 16 key columns; allowed columns
// are [c_lo, c_hi] when kMasked. Writes dS as bf16 pairs.
template <bool kAlibi, bool kSoftcap, bool kMasked>
__device__ __forceinline__ void query_row_elems(const uint32_t (&sr)[16], const uint32_t (&dr)[16],
                                                const ScoreK& sk, float base, float lse2,
                                                float delta, int c_lo, int c_hi,
                                                uint32_t (&dd)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float ds[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int col = 2 * e + q;
      const bool ok = !kMasked || (col >= c_lo && col <= c_hi);
      float pr;
      p_and_ds<kAlibi, kSoftcap>(__uint_as_float(sr[col]), sk,
                                 kAlibi ? fmaf((float)col, sk.kb, base) : 0.f, lse2,
                                 __uint_as_float(dr[col]), delta, ok, 0xffffffffu, pr, ds[q]);
    }
    dd[e] = pack_bf16x2(ds[0], ds[1]);
  }
}

// Copies 64 head-dimension columns (quarter wq) of one bf16 row into tensor memory as
// 32 bf16 pairs at column `col` (zeros when !ok), then arrives on barrier `nb`.
__device__ __forceinline__ void row_quarter_to_tmem(const __nv_bfloat16* src_row, bool ok,
                                                    int wq, uint32_t col, uint32_t nb) {
  uint32_t w[32];
  const uint4* src = reinterpret_cast<const uint4*>(src_row + wq * 64);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint4 v = ok ? src[e] : make_uint4(0, 0, 0, 0);
    w[4 * e] = v.x; w[4 * e + 1] = v.y; w[4 * e + 2] = v.z; w[4 * e + 3] = v.w;
  }
  tmem_st32(col + wq * 32, w);
  tmem_wait_st();
  tc_fence_before_sync();
  nb_arrive(nb, kNbKvCount);
}

// Prologue shared by the three kernels: barriers, 512 tensor-memory columns.
__device__ __forceinline__ uint32_t setup256(BwdBars* bars, int stages, int warp) {
  if (threadIdx.x == 0) setup_common(bars, stages);
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  return bars->tmem_base;
}

__device__ __forceinline__ void teardown256(uint32_t tmem, int warp) {
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// Zero rows [r0, r0 + 128) (those below n) of a [.., n, 256] bf16 array at head z.
__device__ __forceinline__ void zero_rows256(__nv_bfloat16* base, int z, int r0, int n) {
  for (int t = threadIdx.x; t < BT * (D256 / 8); t += kThreads) {
    const int r = r0 + t / (D256 / 8);
    if (r < n)
      reinterpret_cast<uint4*>(base + ((size_t)z * n + r) * D256)[t % (D256 / 8)] =
          make_uint4(0, 0, 0, 0);
  }
}

// ============================================================================ dV, dK
// kDk false: dv256 (S^T -> P^T, dV += P^T dO); true: dk256 (S^T, dP^T -> dS^T,
// dK += dS^T Q).
template <bool kAlibi, bool kSoftcap, bool kDk>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv256_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using L = std::conditional_t<kDk, LayoutK256, LayoutV256>;
  constexpr int kS = L::kStageCount;
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
  __nv_bfloat16* out = kDk ? a.dk : a.dv;
  if (subs == 0) {  // no query sees these keys: zero gradient
    zero_rows256(out, bg, k0, p.Nkv);
    return;
  }
  auto slice = [&](int u, int& row, int& head) {
    const int st = u >> 1;
    head = b * p.Hq + g * G + st / n_q;
    row = (qr.lo + st % n_q) * BT + (u & 1) * SUB;
  };

  WaitCtx wc{&bars->abort_flag, p.status};
  const uint32_t tmem = setup256(bars, kS, warp);

  if (warp == kLoadWarp) {
    load_loop<D256, L>(smem, bars, wc, lane, kDk ? &maps.v128 : nullptr, k0, bg, &maps.q64,
                       &maps.do64, subs, slice, &a.rt, p.nq_pad);
  } else if (warp == kRelayWarp) {
    relay_loop<kS>(bars, wc, subs);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Named barriers only; MMAs predicated on the elect.sync lane (as in the d <= 128
    // kernels). dv256 keeps two S^T buffers in flight: S^T(u + 2) is issued right after
    // dV(u), which reads P^T(u) from the same columns earlier in the tensor pipe.
    // dk256 has one S^T / dP^T pair: S^T(u + 1) follows dK(u) the same way.
    const uint32_t ring = smem_u32(smem + L::kRing);
    const uint32_t sV = smem_u32(smem + L::kFixA);
    const bool ok = !kDk || __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->fixed_full), 0, wc));
    const bool issuer = elect_one();
    nb_sync(kNbKvK, kNbKvCount);  // K tile in tensor memory
    auto issue_s = [&](int v) {
      const int s = v % kS, x = kDk ? 0 : (v & 1);
      nb_sync(kNbStage + s, kNbStageCount);
      tc_fence_after_sync();
      if (!ok) return;
      const uint32_t sQ = ring + s * L::kStage, sDO = sQ + L::kSubTile;
      mma_tmem_x64<D256>(issuer, tmem + col_s256(x), tmem + k256ColFix, sQ);  // S^T = K Q^T
      if (kDk) mma_128x64<D256>(issuer, tmem + k256ColDP, sV, sDO);           // dP^T = V dO^T
      mma_commit_if(issuer, smem_u32(&bars->s_full[x]));
    };
    issue_s(0);
    if (!kDk && subs > 1) issue_s(1);
    for (int u = 0; u < subs; ++u) {
      const int s = u % kS, x = kDk ? 0 : (u & 1);
      nb_sync(kNbKvP + x, kNbKvCount);  // P^T / dS^T(u) written
      tc_fence_after_sync();
      if (ok) {
        const uint32_t sQ = ring + s * L::kStage, sDO = sQ + L::kSubTile;
        // dV += P^T dO, or dK += dS^T Q
        mma_strided_x_slice(issuer, tmem + k256ColAcc, tmem + col_s256(x), kDk ? sQ : sDO, u > 0);
        mma_commit_if(issuer, smem_u32(&bars->empty[s]));  // stage (and its row terms) free
      }
      const int nxt = u + (kDk ? 1 : 2);
      if (nxt < subs) issue_s(nxt);
    }
    if (ok) mma_commit_if(issuer, smem_u32(&bars->acc_full));
  } else {
    // ------------------------------------------------------------ element-wise
    const int q4 = warp & 3, wg = warp >> 2;
    const int row = q4 * 32 + lane;  // key row in the tile
    const int j = k0 + row;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const int c0 = wg * 16;
    const bool causal_type = p.mask.kind != ATTN_MASK_NONE;
    // K rows of the tile into tensor memory: head-dimension quarter wg of this key row
    row_quarter_to_tmem(a.k + ((size_t)bg * p.Nkv + (j < p.Nkv ? j : 0)) * D256, j < p.Nkv, wg,
                        tmem + lane_base + k256ColFix, kNbKvK);
    bool ok_all = true;
    for (int u = 0; u < subs; ++u) {
      const int s = u % kS, x = kDk ? 0 : (u & 1);
      const int use = kDk ? u : (u >> 1);  // uses of buffer x before this one
      int qrow, bh;
      slice(u, qrow, bh);
      const int h = bh - b * p.Hq;
      const int qs = qrow + c0;  // query of this thread's column 0
      const ScoreK sk = score_consts<kAlibi, kSoftcap>(p, h);
      if (ok_all)
        ok_all = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[x]), use & 1, wc));
      if (!ok_all) {  // aborted: keep the barrier schedule with the MMA warp
        nb_sync(kNbKvP + x, kNbKvCount);
        continue;
      }
      tc_fence_after_sync();
      const uint32_t tS = tmem + lane_base + col_s256(x) + c0;
      uint32_t sr[16], dr[16];
      tmem_ld16(tS, sr);
      if (kDk) tmem_ld16(tmem + lane_base + k256ColDP + c0, dr);
      tmem_wait_ld();
      reg_fence16(sr);
      if (kDk) reg_fence16(dr);
      const float* lse2 = reinterpret_cast<const float*>(smem + L::kRows + s * L::kRowStage) + c0;
      const float* dl = lse2 + SUB;
      const int* fk = reinterpret_cast<const int*>(dl + SUB);
      const float base = kAlibi ? sk.kb * (float)(j - qs) : 0.f;  // kb*(j - i) at column 0
      uint32_t pd[8];
      if (tile_needs_mask(p.mask, qrow & ~(BT - 1), k0, BT))  // warp-uniform
        key_row_elems<kAlibi, kSoftcap, true, kDk>(sr, dr, lse2, dl, fk, sk, base, j, qs,
                                                   j < p.Nkv, causal_type, pd);
      else
        key_row_elems<kAlibi, kSoftcap, false, kDk>(sr, dr, lse2, dl, fk, sk, base, j, qs, true,
                                                    causal_type, pd);
      tmem_st8(tS, pd);  // over the first half of the columns this warp read
      tmem_wait_st();
      tc_fence_before_sync();
      nb_arrive(kNbKvP + x, kNbKvCount);
    }
    // ---------------------------------------------------------- epilogue
    const bool have =
        __all_sync(0xffffffffu, ok_all && mbar_wait(smem_u32(&bars->acc_full), 0, wc));
    tc_fence_after_sync();
    const size_t krow = (size_t)bg * p.Nkv + (j < p.Nkv ? j : 0);
    store_acc_row<64>(tmem + lane_base + k256ColAcc + wg * 64, kDk ? p.scale : 1.f,
                      out + krow * D256 + wg * 64, have, j < p.Nkv, ew_stage<L>(smem, warp));
  }
  teardown256(tmem, warp);
}

// ============================================================================ dQ
template <bool kAlibi, bool kSoftcap>
__global__ void __launch_bounds__(kThreads, 1)
    dq256_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using L = LayoutQ256;
  constexpr int kS = L::kStageCount;
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
    zero_rows256(a.dq, bh, q0, p.Nq);
    return;
  }
  auto slice = [&](int u, int& row, int& head) {  // keys of sub-step u
    head = bg;
    row = kr.lo * BT + u * SUB;
  };

  WaitCtx wc{&bars->abort_flag, p.status};
  const uint32_t tmem = setup256(bars, kS, warp);

  if (warp == kLoadWarp) {
    load_loop<D256, L>(smem, bars, wc, lane, &maps.do128, q0, bh, &maps.k64, &maps.v64, subs,
                       slice, nullptr, p.nq_pad);
  } else if (warp == kRelayWarp) {
    relay_loop<kS>(bars, wc, subs);
  } else if (warp == kMmaWarp) {
    const uint32_t ring = smem_u32(smem + L::kRing);
    const uint32_t sDO = smem_u32(smem + L::kFixA);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->fixed_full), 0, wc));
    const bool issuer = elect_one();
    nb_sync(kNbQL, kNbKvCount);  // Q tile in tensor memory
    for (int u = 0; u < subs; ++u) {
      const int s = u % kS;
      nb_sync(kNbStage + s, kNbStageCount);
      tc_fence_after_sync();
      const uint32_t sK = ring + s * L::kStage, sV = sK + L::kSubTile;
      if (ok) {
        mma_tmem_x64<D256>(issuer, tmem + k256ColS0, tmem + k256ColFix, sK);  // S = Q K^T
        mma_128x64<D256>(issuer, tmem + k256ColDP, sDO, sV);                 // dP = dO V^T
        mma_commit_if(issuer, smem_u32(&bars->s_full[0]));
      }
      nb_sync(kNbKvP, kNbKvCount);  // dS written
      tc_fence_after_sync();
      if (ok) {
        mma_strided_x_slice(issuer, tmem + k256ColAcc, tmem + k256ColS0, sK, u > 0);  // dQ += dS K
        mma_commit_if(issuer, smem_u32(&bars->empty[s]));
      }
    }
    if (ok) mma_commit_if(issuer, smem_u32(&bars->acc_full));
  } else {
    const int q4 = warp & 3, wg = warp >> 2;
    const int row = q4 * 32 + lane;
    const int i = q0 + row;
    const bool row_ok = i < p.Nq;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const int c0 = wg * 16;
    const ScoreK sk = score_consts<kAlibi, kSoftcap>(p, h);
    float lse2 = INFINITY, dlt = 0.f;
    int fk = 0;
    if (row_ok) {  // row terms of the row kernel (lse2 is already L log2 e, +inf if empty)
      lse2 = a.rt.lse2[(size_t)bh * p.nq_pad + i];
      dlt = a.rt.delta[(size_t)bh * p.nq_pad + i];
      fk = a.rt.first[i];
    }
    const int last_key = (p.mask.kind == ATTN_MASK_NONE ? p.Nkv - 1 : imin(i, p.Nkv - 1));
    row_quarter_to_tmem(a.q + ((size_t)bh * p.Nq + (row_ok ? i : 0)) * D256, row_ok, wg,
                        tmem + lane_base + k256ColFix, kNbQL);
    bool ok_all = true;
    for (int u = 0; u < subs; ++u) {
      const int kt0 = (kr.lo + (u >> 1)) * BT;
      const int ks = kr.lo * BT + u * SUB + c0;  // key of this thread's column 0
      if (ok_all)
        ok_all = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[0]), u & 1, wc));
      if (!ok_all) {
        nb_sync(kNbKvP, kNbKvCount);
        continue;
      }
      tc_fence_after_sync();
      const uint32_t tS = tmem + lane_base + k256ColS0 + c0;
      uint32_t sr[16], dr[16];
      tmem_ld16(tS, sr);
      tmem_ld16(tmem + lane_base + k256ColDP + c0, dr);
      tmem_wait_ld();
      reg_fence16(sr);
      reg_fence16(dr);
      const float base = kAlibi ? sk.kb * (float)(ks - i) : 0.f;  // kb*(j - i) at column 0
      uint32_t dd[8];
      if (tile_needs_mask(p.mask, q0, kt0, BT))  // warp-uniform
        query_row_elems<kAlibi, kSoftcap, true>(sr, dr, sk, base, lse2, dlt, fk - ks,
                                                last_key - ks, dd);
      else
        query_row_elems<kAlibi, kSoftcap, false>(sr, dr, sk, base, lse2, dlt, 0, 0, dd);
      tmem_st8(tS, dd);
      tmem_wait_st();
      tc_fence_before_sync();
      nb_arrive(kNbKvP, kNbKvCount);
    }
    const bool have =
        __all_sync(0xffffffffu, ok_all && mbar_wait(smem_u32(&bars->acc_full), 0, wc));
    tc_fence_after_sync();
    __nv_bfloat16* dst = a.dq + ((size_t)bh * p.Nq + (row_ok ? i : 0)) * D256 + wg * 64;
    store_acc_row<64>(tmem + lane_base + k256ColAcc + wg * 64, p.scale, dst, have, row_ok,
                      ew_stage<L>(smem, warp));
  }
  teardown256(tmem, warp);
}

template <bool kA, bool kS>
cudaError_t launch_variant256(const BwdArgs& ka, const BwdArgs& qa, const BwdMaps& maps,
                              int grid_kv, int grid_q, cudaStream_t st) {
  auto kv = dkdv256_kernel<kA, kS, false>;
  auto kk = dkdv256_kernel<kA, kS, true>;
  auto kq = dq256_kernel<kA, kS>;
  constexpr int kSmemV = LayoutV256::kAlloc, kSmemK = LayoutK256::kAlloc,
                kSmemQ = LayoutQ256::kAlloc;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemV)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemK)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemQ)) != cudaSuccess)
    return e;
  if (grid_kv > 0) {
    kv<<<grid_kv, kThreads, kSmemV, st>>>(maps, ka);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kk<<<grid_kv, kThreads, kSmemK, st>>>(maps, ka);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (grid_q > 0) kq<<<grid_q, kThreads, kSmemQ, st>>>(maps, qa);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd256_tc(const Problem& p, const BwdMaps& maps, const RowTerms& rt,
                             const __nv_bfloat16* q, const __nv_bfloat16* dout,
                             const __nv_bfloat16* k, __nv_bfloat16* dq, __nv_bfloat16* dk,
                             __nv_bfloat16* dv, bool run_dkdv, bool run_dq, cudaStream_t st) {
  BwdArgs ka{p, rt, q, dout, k, nullptr, dq, dk, dv, ceil_div(p.Nkv, BT)};
  BwdArgs qa{p, rt, q, dout, k, nullptr, dq, dk, dv, ceil_div(p.Nq, BT)};
  const long long gk = run_dkdv ? (long long)ka.n_tiles * p.B * p.Hkv : 0;
  const long long gq = run_dq ? (long long)qa.n_tiles * p.B * p.Hq : 0;
  if (gk > 0x7fffffffLL || gq > 0x7fffffffLL) return cudaErrorInvalidValue;
  const bool al = p.score_kind & ATTN_SCORE_ALIBI, sc = p.score_kind & ATTN_SCORE_SOFTCAP;
  if (al && sc) return launch_variant256<true, true>(ka, qa, maps, (int)gk, (int)gq, st);
  if (al) return launch_variant256<true, false>(ka, qa, maps, (int)gk, (int)gq, st);
  if (sc) return launch_variant256<false, true>(ka, qa, maps, (int)gk, (int)gq, st);
  return launch_variant256<false, false>(ka, qa, maps, (int)gk, (int)gq, st);
}

}  // namespace attn
