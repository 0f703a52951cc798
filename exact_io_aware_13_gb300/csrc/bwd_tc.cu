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
// Dropout (kDrop): both kernels regenerate the forward's keep mask Z (Philox4x32-10, one
// call per 16 keys of a query row; the dK/dV warps, one lane per key, get their bytes
// through a byte transpose within each half-warp). With the row term D (1 - p) from the
// row kernel, dV takes P o Z and dS' = P o (dP o Z - D (1 - p)) = (1 - p) dS; the
// epilogues multiply dV, dK and dQ by 1 / (1 - p).
// Each sub-step streams its own 64-row slice of the two operands it walks (Q and dO,
// or K and V; for dkdv also the 64 rows' L log2 e, D and first key) through a
// shared-memory ring (5 stages for dkdv, 6 for dq), so loads run ahead of the MMAs. Warp
// 16 loads with TMA, warp 17 owns tensor memory and issues the MMAs, warp 18 relays TMA
// completions; warps 0-15 do the element-wise work, one thread per TMEM lane (= row of
// the CTA's tile). The MMA warp waits only on hardware named barriers: a shared-memory
// access from the thread that issues MMAs stalls the tensor pipe (see nb_sync in
// ptx.cuh).
//   dkdv: K is fixed in shared memory (A operand of S^T = K Q^T) and V is copied once
//     into tensor memory (A operand of dP^T = V dO^T, so that product reads only dO from
//     shared memory); S^T is double-buffered in tensor memory (sub-step u in buffer
//     u % 2), dP^T single-buffered. The element-wise warps write P^T and then dS^T as
//     bf16 pairs into the two halves of their columns of the S^T buffer; the dP^T buffer
//     is free as soon as they hold dP^T in registers, so dP^T(u + 1) runs while they form
//     dS(u), and S^T(u + 2) follows dV / dK(u) into its buffer (the tensor pipe runs a
//     thread's MMAs in order). Every element-wise warp works on every sub-step (warpgroup
//     w: 16 of its 64 query columns).
//   dq: two pairs of warpgroups alternate sub-steps (pair p takes u % 2 == p, warpgroup
//     w of the pair 32 key columns); S / dP are double-buffered and dS is written back
//     over S.
// The unmasked tiles without score mods take the element-wise step two columns per
// instruction (packed fp32 pairs, each operation bit for bit the scalar one).
#include "bwd_common.cuh"

namespace attn {
namespace {

// dkdv element-wise step, first phase, for one thread: key row j, 16 query columns
// starting at qs, with their lse2 / first key. Gives P (pv, kept for the second phase),
// the soft-cap derivative (dc) and P^T (bf16 pairs, times the keep mask with dropout).
// kMasked adds the per-element mask test; the caller picks the variant by a warp-uniform
// tile test.
template <bool kAlibi, bool kSoftcap, bool kMasked, bool kDrop>
__device__ __forceinline__ void dkdv_p(const uint32_t (&sr)[16], const float* lse2,
                                       const int* fk, const ScoreK& sk, float base, int j,
                                       int qs, bool key_ok, bool causal_type,
                                       const uint32_t (&kf)[4], float (&pv)[16],
                                       float (&dc)[16], uint32_t (&pp)[8]) {
  if constexpr (!kAlibi && !kSoftcap && !kMasked && !kDrop) {
    // Two query columns per instruction (packed fp32 pairs): a = lse2 - k1 x, P = 2^-a
    // (the same value as 2^(k1 x - lse2): the negation is exact).
    const uint64_t nk1 = f32x2(-sk.k1, -sk.k1);
#pragma unroll
    for (int e4 = 0; e4 < 4; ++e4) {
      const float4 lv = reinterpret_cast<const float4*>(lse2)[e4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int col = e4 * 4 + 2 * h;
        const uint64_t l2 = h ? f32x2(lv.z, lv.w) : f32x2(lv.x, lv.y);
        float a0, a1;
        f32x2_split(fma_f32x2(f32x2(__uint_as_float(sr[col]), __uint_as_float(sr[col + 1])),
                              nk1, l2), a0, a1);
        pv[col] = ex2_approx(-a0);
        pv[col + 1] = ex2_approx(-a1);
        dc[col] = dc[col + 1] = 1.f;
        pp[col >> 1] = pack_bf16x2(pv[col], pv[col + 1]);
      }
    }
    return;
  }
#pragma unroll
  for (int e4 = 0; e4 < 4; ++e4) {
    const float4 lv = reinterpret_cast<const float4*>(lse2)[e4];
    const float lvs[4] = {lv.x, lv.y, lv.z, lv.w};
    float pz[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int col = e4 * 4 + q;
      bool ok = true;
      if (kMasked) {
        const int i = qs + col;
        ok = key_ok && (!causal_type || (i >= j && fk[col] <= j));
      }
      p_only<kAlibi, kSoftcap>(__uint_as_float(sr[col]), sk,
                               kAlibi ? fmaf(-(float)col, sk.kb, base) : 0.f, lvs[q], ok,
                               pv[col], dc[col]);
      pz[q] = pv[col];
      if (kDrop)  // dV takes P Z
        pz[q] = __uint_as_float(__float_as_uint(pz[q]) & keep_mask_elem(kf[e4], q));
    }
    pp[2 * e4] = pack_bf16x2(pz[0], pz[1]);
    pp[2 * e4 + 1] = pack_bf16x2(pz[2], pz[3]);
  }
}

// dkdv element-wise step, second phase: dS^T (bf16 pairs) from P, the soft-cap derivative
// and dP^T of the thread's 16 columns with their delta; the same arithmetic as p_and_ds.
template <bool kSoftcap, bool kDrop>
__device__ __forceinline__ void dkdv_ds(const uint32_t (&dr)[16], const float* dl,
                                        const float (&pv)[16], const float (&dc)[16],
                                        const uint32_t (&kf)[4], uint32_t (&dd)[8]) {
  if constexpr (!kSoftcap && !kDrop) {  // packed fp32 pairs: dS = P (dP - D)
#pragma unroll
    for (int e4 = 0; e4 < 4; ++e4) {
      const float4 dv = reinterpret_cast<const float4*>(dl)[e4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int col = e4 * 4 + 2 * h;
        const uint64_t d2 = h ? f32x2(dv.z, dv.w) : f32x2(dv.x, dv.y);
        const uint64_t t2 =
            sub_f32x2(f32x2(__uint_as_float(dr[col]), __uint_as_float(dr[col + 1])), d2);
        float s0, s1;
        f32x2_split(mul_f32x2(f32x2(pv[col], pv[col + 1]), t2), s0, s1);
        dd[col >> 1] = pack_bf16x2(s0, s1);
      }
    }
    return;
  }
#pragma unroll
  for (int e4 = 0; e4 < 4; ++e4) {
    const float4 dv = reinterpret_cast<const float4*>(dl)[e4];
    const float dvs[4] = {dv.x, dv.y, dv.z, dv.w};
    float ds[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int col = e4 * 4 + q;
      const uint32_t zm = kDrop ? keep_mask_elem(kf[e4], q) : 0xffffffffu;
      ds[q] = ds_of<kSoftcap>(pv[col], dc[col], __uint_as_float(dr[col]), dvs[q], zm);
    }
    dd[2 * e4] = pack_bf16x2(ds[0], ds[1]);
    dd[2 * e4 + 1] = pack_bf16x2(ds[2], ds[3]);
  }
}

// dq element-wise step for one thread: query row with (lse2, delta), 32 key columns;
// allowed columns are [c_lo, c_hi] when kMasked. Writes dS (bf16 pairs).
template <bool kAlibi, bool kSoftcap, bool kMasked, bool kDrop>
__device__ __forceinline__ void dq_ds(const uint32_t (&sr)[32], const uint32_t (&dr)[32],
                                      const ScoreK& sk, float base, float lse2, float delta,
                                      int c_lo, int c_hi, const uint32_t (&kf)[8],
                                      uint32_t (&dd)[16]) {
  if constexpr (!kAlibi && !kSoftcap && !kMasked && !kDrop) {
    // Two key columns per instruction (packed fp32 pairs), as in dkdv_pds.
    const uint64_t nk1 = f32x2(-sk.k1, -sk.k1);
    const uint64_t l2 = f32x2(lse2, lse2), d2 = f32x2(delta, delta);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float a0, a1;
      f32x2_split(fma_f32x2(f32x2(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])),
                            nk1, l2), a0, a1);
      const float p0 = ex2_approx(-a0), p1 = ex2_approx(-a1);
      const uint64_t t2 =
          sub_f32x2(f32x2(__uint_as_float(dr[2 * e]), __uint_as_float(dr[2 * e + 1])), d2);
      float s0, s1;
      f32x2_split(mul_f32x2(f32x2(p0, p1), t2), s0, s1);
      dd[e] = pack_bf16x2(s0, s1);
    }
    return;
  }
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
  const uint32_t colDV = kKv2ColAcc, colDK = kKv2ColAcc + D;
  constexpr int kS = L::kStageCount;

  if (warp == kLoadWarp) {
    load_loop<D, L>(smem, bars, wc, lane, &maps.k128, k0, bg, &maps.q64, &maps.do64, subs,
                    slice, &a.rt, p.nq_pad);
  } else if (warp == kRelayWarp) {
    relay_loop<kS>(bars, wc, subs);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the schedule and waits on named barriers; every lane executes
    // the MMA instructions predicated on `issuer`, the one lane elect.sync picks, so the
    // warp never diverges (with an elect.sync predicate MMAs go out back to back, each
    // taking its tensor or shared-memory time; a predicate computed from the lane index
    // costs about 82 cycles per MMA). If the fixed tile never
    // arrives (`ok` false) the warp keeps every barrier operation and issues nothing.
    // S^T(v) = K Q^T goes to buffer v % 2 (K in shared memory), dP^T(v) = V dO^T to the
    // one dP^T buffer (V in tensor memory: the tensor core then reads only dO from shared
    // memory, 32 instead of 48 cycles per N = 64 instruction). Per sub-step u: dV(u) once
    // P^T(u) is written over the first halves of its S^T buffer; dP^T(u + 1) as soon as
    // the element-wise warps hold dP^T(u) in registers; dK(u) once dS^T(u) is written over
    // the second halves of the S^T buffer; then S^T(u + 2) into that buffer (the tensor
    // pipe runs a thread's MMAs in order, so each overwrites a buffer only after the
    // products reading it have run).
    const uint32_t sK = smem_u32(smem + L::kFixA);
    const uint32_t ring = smem_u32(smem + L::kRing);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->fixed_full), 0, wc));
    const bool issuer = elect_one();
    auto stage = [&](int v) { return ring + (v % kS) * L::kStage; };  // Q slice, then dO
    auto sync_stage = [&](int v) {
      nb_sync(kNbStage + v % kS, kNbStageCount);
      tc_fence_after_sync();
    };
    auto issue_s = [&](int v) {  // S^T(v); stage v synced
      if (!ok) return;
      mma_128x64<D>(issuer, tmem + kv_col_s(v & 1), sK, stage(v));
      mma_commit_if(issuer, smem_u32(&bars->s_full[v & 1]));
    };
    auto issue_dp = [&](int v) {  // dP^T(v); stage v synced
      if (!ok) return;
      mma_tmem_x64<D>(issuer, tmem + kKv2ColDP, tmem + kKv2ColV, stage(v) + L::kSubTile);
      mma_commit_if(issuer, smem_u32(&bars->dp_full));
    };
    nb_sync(kNbQL, kNbKvCount);  // the V tile is in tensor memory
    tc_fence_after_sync();
    sync_stage(0);
    issue_s(0);
    issue_dp(0);
    if (subs > 1) {
      sync_stage(1);
      issue_s(1);
    }
    for (int u = 0; u < subs; ++u) {
      const int x = u & 1;
      nb_sync(kNbKvP + x, kNbKvCount);  // P^T(u) written over S^T buffer x
      tc_fence_after_sync();
      if (ok)  // dV += P^T dO
        mma_inplace_x_slice<D>(issuer, tmem + colDV, tmem + kv_col_s(x), stage(u) + L::kSubTile,
                               u > 0);
      nb_sync(kNbKvF, kNbKvCount);  // dP^T(u) read: the buffer takes dP^T(u + 1)
      tc_fence_after_sync();
      if (u + 1 < subs) issue_dp(u + 1);  // its stage was synced for S^T(u + 1)
      nb_sync(kNbKvD, kNbKvCount);  // dS^T(u) written over the second halves of buffer x
      tc_fence_after_sync();
      if (ok) {  // dK += dS^T Q
        mma_inplace_x_slice<D>(issuer, tmem + colDK, tmem + kv_col_s(x) + 8, stage(u), u > 0);
        mma_commit_if(issuer, smem_u32(&bars->empty[u % kS]));  // stage (and its row terms) free
      }
      if (u + 2 < subs) {
        sync_stage(u + 2);
        issue_s(u + 2);
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
      // This thread's V row into tensor memory (bf16 pairs, the A operand of dP^T =
      // V dO^T): warpgroup wg copies words [wg D/8, (wg + 1) D/8) of the row's D/2 (zeros
      // past Nkv).
      constexpr int kW = D / 8;
      uint32_t wv[kW];
      const bool row_in = j < p.Nkv;
      const uint4* src = reinterpret_cast<const uint4*>(
                             a.v + ((size_t)bg * p.Nkv + (row_in ? j : 0)) * D) + wg * (kW / 4);
#pragma unroll
      for (int e = 0; e < kW / 4; ++e) {
        const uint4 v = row_in ? src[e] : make_uint4(0, 0, 0, 0);
        wv[4 * e] = v.x; wv[4 * e + 1] = v.y; wv[4 * e + 2] = v.z; wv[4 * e + 3] = v.w;
      }
      const uint32_t dst = tmem + lane_base + kKv2ColV + wg * kW;
      if constexpr (kW == 16) tmem_st16(dst, wv);
      else tmem_st8(dst, wv);
      tmem_wait_st();
      tc_fence_before_sync();
      nb_arrive(kNbQL, kNbKvCount);
    }
    bool ok_all = true;
    // (head, query tile) of sub-step u, its score constants and whether the tile needs
    // the per-element mask, advanced every second sub-step (the order `slice` gives)
    int st_q = 0, st_h = 0;
    ScoreK sk = score_consts<kAlibi, kSoftcap>(p, g * G);
    bool need_mask = tile_needs_mask(p.mask, qr.lo * BT, k0, BT);
    const DropThr dthr = drop_thr_words(kDrop ? p.drop_thr : 0);
    const PhiloxKeys pk = philox_keys(p.drop_seed_lo, p.drop_seed_hi);  // unused without dropout
    for (int u = 0; u < subs; ++u) {
      const int s = u % kS, x = u & 1;
      if (u > 0 && x == 0) {
        if (++st_q == n_q) {
          st_q = 0;
          ++st_h;
          sk = score_consts<kAlibi, kSoftcap>(p, g * G + st_h);
        }
        need_mask = tile_needs_mask(p.mask, (qr.lo + st_q) * BT, k0, BT);
      }
      const int qrow = (qr.lo + st_q) * BT + x * SUB;
      const int bh = b * p.Hq + g * G + st_h;
      const int qs = qrow + c0;                  // query of this thread's column 0
      const float* lse2 = reinterpret_cast<const float*>(smem + L::kRows + s * L::kRowStage) + c0;
      const float* dl = lse2 + SUB;
      const int* fk = reinterpret_cast<const int*>(dl + SUB);
      // ---- first phase: P^T(u) over the first half of this warpgroup's 16 columns of
      // S^T buffer x (k-step wg of the dV product); no other warp reads those columns
      if (ok_all)
        ok_all = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[x]), (u >> 1) & 1, wc));
      // the stage's row terms arrived with full[s]; observe them
      if (ok_all)
        ok_all = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->full[s]), (u / kS) & 1, wc));
      float pv[16], dc[16];
      uint32_t kf[4] = {0u, 0u, 0u, 0u};
      if (ok_all) {
        tc_fence_after_sync();
        const uint32_t tS = tmem + lane_base + kv_col_s(x) + c0;
        uint32_t sr[16], pp[8];
        tmem_ld16(tS, sr);
        tmem_wait_ld();
        reg_fence16(sr);
        const float base = kAlibi ? sk.kb * (float)(j - qs) : 0.f;  // kb*(j - i) at column 0
        if constexpr (kDrop) dropout_flags_dkdv(pk, dthr, j, lane, qs, bh, kf);
        if (need_mask)  // warp-uniform
          dkdv_p<kAlibi, kSoftcap, true, kDrop>(sr, lse2, fk, sk, base, j, qs, j < p.Nkv,
                                                causal_type, kf, pv, dc, pp);
        else
          dkdv_p<kAlibi, kSoftcap, false, kDrop>(sr, lse2, fk, sk, base, j, qs, true,
                                                 causal_type, kf, pv, dc, pp);
        tmem_st8(tS, pp);
        tmem_wait_st();
        tc_fence_before_sync();
        nb_arrive(kNbKvP + x, kNbKvCount);
      } else {  // aborted: keep the barrier schedule with the MMA warp
        nb_sync(kNbKvP + x, kNbKvCount);
      }
      // ---- second phase: dP^T(u) into registers (then the buffer is released), dS^T(u)
      // over the second half of this warpgroup's 16 columns of S^T buffer x (k-step wg of
      // the dK product)
      if (ok_all)
        ok_all = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->dp_full), u & 1, wc));
      if (ok_all) {
        tc_fence_after_sync();
        uint32_t dr[16], dd[8];
        tmem_ld16(tmem + lane_base + kKv2ColDP + c0, dr);
        tmem_wait_ld();
        reg_fence16(dr);
        tc_fence_before_sync();
        nb_arrive(kNbKvF, kNbKvCount);
        dkdv_ds<kSoftcap, kDrop>(dr, dl, pv, dc, kf, dd);
        tmem_st8(tmem + lane_base + kv_col_s(x) + c0 + 8, dd);
        tmem_wait_st();
        tc_fence_before_sync();
        nb_arrive(kNbKvD, kNbKvCount);
      } else {  // aborted: keep the barrier schedule with the MMA warp
        nb_sync(kNbKvF, kNbKvCount);
        nb_sync(kNbKvD, kNbKvCount);
      }
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
    store_acc_row<D / 2>(tacc, which ? p.scale * dsc : dsc, dst, have, j < p.Nkv,
                         ew_stage<L>(smem, warp));
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
    load_loop<D, L>(smem, bars, wc, lane, &maps.q128, q0, bh, &maps.k64, &maps.v64, subs, slice,
                    nullptr, p.nq_pad, &maps.do128);
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
    const PhiloxKeys pk = philox_keys(p.drop_seed_lo, p.drop_seed_hi);  // unused without dropout
    float lse2 = INFINITY, dlt = 0.f;
    int fk = 0;
    if (row_ok) {  // row terms of the row kernel (lse2 is already L log2 e, +inf if empty)
      lse2 = a.rt.lse2[(size_t)bh * p.nq_pad + i];
      dlt = a.rt.delta[(size_t)bh * p.nq_pad + i];
      fk = a.rt.first[i];
    }
    const int last_key = (p.mask.kind == ATTN_MASK_NONE ? p.Nkv - 1 : imin(i, p.Nkv - 1));
    {
      // Q and dO rows of the tile into tensor memory, from the fixed tiles the loader
      // brought into shared memory with TMA (128-byte swizzle: 16-byte chunk c of row r of
      // a 64-column slab at r * 128 + ((c ^ (r & 7)) << 4); rows past Nq read as zeros):
      // warpgroups 0 and 1 copy the two halves of this thread's Q row, 2 and 3 those of
      // its dO row.
      const int wq = warp >> 2, half = wq & 1;
      constexpr int kW = D / 4;  // 32-bit words (bf16 pairs) per thread
      uint32_t wv[kW];
      const bool got =
          __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->fixed_full), 0, wc));
      const uint8_t* tile = smem + L::kFixA + (wq < 2 ? 0 : L::kFixTile);
#pragma unroll
      for (int e = 0; e < kW / 4; ++e) {
        const int cg = half * (kW / 4) + e;  // 16-byte chunk of the row
        const uint4 v = got ? *reinterpret_cast<const uint4*>(
                                  tile + (cg >> 3) * L::kFixChunk + row * 128 +
                                  (((cg & 7) ^ (row & 7)) << 4))
                            : make_uint4(0, 0, 0, 0);
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
      if constexpr (kDrop) dropout_flags_dq(pk, dthr, i, ks, bh, kf);
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
      store_acc_row<D / 2>(tq, kDrop ? p.scale * p.drop_scale : p.scale, dst, have, row_ok,
                           ew_stage<L>(smem, warp));
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
                          const __nv_bfloat16* k, const __nv_bfloat16* v, __nv_bfloat16* dq,
                          __nv_bfloat16* dk, __nv_bfloat16* dv,
                          bool run_dkdv, bool run_dq, cudaStream_t st) {
  BwdArgs ka{p, rt, q, dout, k, v, dq, dk, dv, ceil_div(p.Nkv, BT)};
  BwdArgs qa{p, rt, q, dout, k, v, dq, dk, dv, ceil_div(p.Nq, BT)};
  const long long gk = run_dkdv ? (long long)ka.n_tiles * p.B * p.Hkv : 0;
  const long long gq = run_dq ? (long long)qa.n_tiles * p.B * p.Hq : 0;
  if (gk > 0x7fffffffLL || gq > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (p.d == 64) return launch_d<64>(ka, qa, maps, (int)gk, (int)gq, st);
  return launch_d<128>(ka, qa, maps, (int)gk, (int)gq, st);
}

}  // namespace attn
