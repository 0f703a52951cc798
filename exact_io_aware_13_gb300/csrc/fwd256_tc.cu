// Forward attention with head dimension 256 on the tcgen05 tensor cores (sm_103a).
//
// Same computation as the d = 64 / 128 forward ("FlashAttention/es", "El algoritmo
// FlashAttention": running max, running sum, rescaled accumulator, L = m + log l), for
// the head sizes up to about 256 the page names as the method's range ("Limitaciones").
// At d = 256 the two-query-tile layout of the other forward does not fit tensor memory
// (two O accumulators alone take 512 columns), so this kernel is laid out differently:
//   * one CTA = one 128-row query tile against 64-key tiles; Q sits in tensor memory
//     (bf16 pairs, the A operand of S = Q K^T), written there once by the softmax warps;
//   * tensor memory: S0 [0,64), S1 [64,128), O [128,384), Q [384,512);
//   * warp 6 streams K and V tiles (32 KB each) through a 7-stage shared-memory ring with
//     TMA (four 128-byte-swizzled slabs per tile), skipping key tiles the mask empties;
//   * warp 7 relays each landed tile to warp 5 through one named barrier per stage;
//   * warp 5 issues S(j + 1) = Q K^T before O += P(j) V (so the softmax of tile j overlaps
//     the score MMAs of tile j + 1), releasing a K stage as soon as its S MMAs complete;
//   * warps 0-3 run the softmax, one thread per row, exp2 with the score and mask
//     modifications of the other kernels, and rescale O only when the max grows by more
//     than 2^8; they also write the result.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int D = 256;
constexpr int BM = 128;                       // query rows per CTA (MMA M, TMEM lanes)
constexpr int BN = 64;                        // keys per tile
constexpr int kStages = 7;                    // ring of single K or V tiles
constexpr int kSlab = BN * 128;               // 64 rows x 128 bytes
constexpr int kTile = (D / 64) * kSlab;       // 32 KB: one K or V tile
constexpr int kBars = kStages * kTile;
constexpr int kAlloc = kBars + 256 + 1024;
static_assert(kAlloc <= 232448, "shared memory");
constexpr int kMmaWarp = 5, kLoadWarp = 6, kRelayWarp = 7;
constexpr int kThreads = 256;
constexpr uint32_t kColS0 = 0, kColS1 = 64, kColO = 128, kColQ = 384, kTmemCols = 512;
// Named barriers: kNbP + (j & 1) P of tile j (softmax warps + MMA warp), kNbQ Q in TMEM
// (the same), kNbKv + s ring stage s landed (relay + MMA warp).
constexpr uint32_t kNbP = 1, kNbQ = 3, kNbKv = 4, kNbWide = 160, kNbPair = 64;
static_assert(kNbKv + kStages - 1 <= 15, "named barrier IDs");
constexpr int kHeadGroup = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;

struct Bars {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t s_full[2];
  uint64_t pv_done;
  uint64_t o_full;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

struct Args {
  Problem p;
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  float* lse;
  int nqb;  // 128-row query tiles per head
};

// Whether every (row, key) of rows [q0, q1] x keys [k0, k0 + 63] is allowed.
__device__ __forceinline__ bool keys_full(const MaskSpec& m, int q0, int q1, int k0) {
  if (k0 + BN > m.nkv) return false;
  if (m.kind == ATTN_MASK_NONE) return true;
  return k0 + BN - 1 <= q0 && first_key(m, q1) <= k0;  // first_key grows with the row
}

template <bool kAlibi, bool kSoftcap>
__global__ void __launch_bounds__(kThreads, 1)
    fwd256_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kBars);
  const Problem& p = a.p;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // CTA -> (head, query tile): heads kHeadGroup at a time (their K/V shared in L2), the
  // tiles with the most keys (the last ones under causal masks) first.
  const int BH = p.B * p.Hq;
  const int per_group = kHeadGroup * a.nqb;
  const int grp = blockIdx.x / per_group;
  const int rem = blockIdx.x - grp * per_group;
  const int gh = imin(kHeadGroup, BH - grp * kHeadGroup);
  const int qb = a.nqb - 1 - rem / gh;
  const int bh = grp * kHeadGroup + rem % gh;
  const int b = bh / p.Hq, h = bh - b * p.Hq;
  const int bg = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int q0 = qb * BM, q1 = imin(q0 + BM, p.Nq) - 1;

  // Keys the tile's rows may see: [kmin, kmax], in 64-key tiles [jlo, jlo + n).
  int kmin = 0, kmax = p.Nkv - 1;
  if (p.mask.kind != ATTN_MASK_NONE) {
    kmin = imax(first_key(p.mask, q0), 0);
    kmax = imin(q1, p.Nkv - 1);
    if (p.mask.kind == ATTN_MASK_SLIDING_WINDOW && p.mask.window <= 0) kmax = -1;
  }
  if (kmax < kmin) {  // no key for any row: O = 0, L = -inf
    for (int r = threadIdx.x; r < BM; r += kThreads) {
      const int i = q0 + r;
      if (i >= p.Nq) continue;
      uint4* orow = reinterpret_cast<uint4*>(a.o + ((size_t)bh * p.Nq + i) * D);
      for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
      a.lse[(size_t)bh * p.Nq + i] = -INFINITY;
    }
    return;
  }
  const int jlo = kmin / BN, n = kmax / BN + 1 - jlo;

  WaitCtx wc{&bars->abort_flag, p.status};
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    mbar_init(smem_u32(&bars->s_full[0]), 1);
    mbar_init(smem_u32(&bars->s_full[1]), 1);
    mbar_init(smem_u32(&bars->pv_done), 1);
    mbar_init(smem_u32(&bars->o_full), 1);
    mbar_init(smem_u32(&bars->mma_done), 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t ring = smem_u32(smem);

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    // Ring use u: key tile jlo + u / 2, K for even u, V for odd u.
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    int issued = 0;
    for (int u = 0; u < 2 * n; ++u) {
      const int s = u % kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->empty[s]), ((u / kStages) & 1) ^ 1, wc)))
        break;
      const uint32_t fb = smem_u32(&bars->full[s]);
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, kTile);
        const CUtensorMap* map = (u & 1) ? &tm_v : &tm_k;
        const int krow = (jlo + (u >> 1)) * BN;  // rows past Nkv read as zero
#pragma unroll
        for (int c = 0; c < D / 64; ++c) tma_load_3d(ring + s * kTile + c * kSlab, map, fb, c * 64, krow, bg);
      }
      ++issued;
    }
    for (int u = imax(0, issued - kStages); u < issued; ++u)
      drain_wait(smem_u32(&bars->full[u % kStages]), (u / kStages) & 1);
  } else if (warp == kRelayWarp) {
    // ------------------------------------------------------------ relay
    bool live = true;
    for (int u = 0; u < 2 * n; ++u) {
      const int s = u % kStages;
      if (live) live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->full[s]), (u / kStages) & 1, wc));
      if (live) nb_arrive(kNbKv + s, kNbPair);
      else nb_sync(kNbKv + s, kNbPair);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The warp waits only on named barriers; it touches no shared memory until its last
    // MMA, and then waits for its MMAs before tensor memory is released.
    constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false, false);
    constexpr uint32_t idO = idesc_bf16_f32(BM, D, false, true);
    const bool issuer = elect_one();
    nb_sync(kNbQ, kNbWide);
    tc_fence_after_sync();
    auto pv = [&](int j) {  // O += P(j) V(j)
      const int u = 2 * j + 1, s = u % kStages;
      nb_sync(kNbP + (j & 1), kNbWide);
      nb_sync(kNbKv + s, kNbPair);
      tc_fence_after_sync();
      const uint64_t dv = smem_desc_sw128(ring + s * kTile, kSlab, 1024);
      const uint32_t colS = (j & 1) ? kColS1 : kColS0;
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk)  // 16 keys per instruction, N = 256
        mma_ts_if(issuer, tmem + kColO, tmem + colS + kk * 8, dv + ((kk * 16 * 128) >> 4), idO,
                  (j > 0 || kk > 0) ? 1u : 0u);
      mma_commit_if(issuer, smem_u32(&bars->empty[s]));
      mma_commit_if(issuer, smem_u32(&bars->pv_done));
    };
    for (int j = 0; j < n; ++j) {
      const int u = 2 * j, s = u % kStages;
      nb_sync(kNbKv + s, kNbPair);
      tc_fence_after_sync();
      const uint64_t dk = smem_desc_sw128(ring + s * kTile, 16, 1024);
      const uint32_t col = (j & 1) ? kColS1 : kColS0;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {  // 16 head dims per instruction; Q in TMEM
        const uint32_t offk = ((kk >> 2) * kSlab + (kk & 3) * 32) >> 4;
        mma_ts_if(issuer, tmem + col, tmem + kColQ + kk * 8, dk + offk, idS, kk > 0 ? 1u : 0u);
      }
      mma_commit_if(issuer, smem_u32(&bars->s_full[j & 1]));
      mma_commit_if(issuer, smem_u32(&bars->empty[s]));  // K is free once S is done
      if (j >= 1) pv(j - 1);
    }
    pv(n - 1);
    mma_commit_if(issuer, smem_u32(&bars->o_full));
    mma_commit_if(issuer, smem_u32(&bars->mma_done));
    drain_wait(smem_u32(&bars->mma_done), 0);
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax warps
    const int row = warp * 32 + lane;  // TMEM lane = query row of the tile
    const int i = q0 + row;
    const bool valid = i < p.Nq;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t tO = tmem + lane_base + kColO;
    // Q row -> tensor memory (bf16 pairs, lower element in the low half; zeros past Nq).
    {
      const uint4* src = reinterpret_cast<const uint4*>(a.q + ((size_t)bh * p.Nq + (valid ? i : 0)) * D);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint4 v = valid ? __ldg(src + c * 8 + e) : make_uint4(0, 0, 0, 0);
          w[4 * e] = v.x; w[4 * e + 1] = v.y; w[4 * e + 2] = v.z; w[4 * e + 3] = v.w;
        }
        tmem_st32(tmem + lane_base + kColQ + c * 32, w);
      }
      tmem_wait_st();
      tc_fence_before_sync();
      nb_arrive(kNbQ, kNbWide);
    }
    const int fk = first_key(p.mask, valid ? i : p.Nq - 1);
    const int last_key = p.mask.kind == ATTN_MASK_NONE ? p.Nkv - 1 : imin(i, p.Nkv - 1);
    const float slope = kAlibi ? alibi_slope(h, p.Hq) : 0.f;
    // with the soft-cap c: the pre-cap score over c, then s2 = c log2(e) tanh of it
    const float k1 = kSoftcap ? p.scale / p.softcap : p.scale * kLog2e;
    const float kb = kSoftcap ? slope / p.softcap : slope * kLog2e;
    const float capA = kSoftcap ? p.softcap * kLog2e : 0.f;
    const bool raw_ok = !kAlibi && !kSoftcap && k1 > 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    bool live = true;
    int j = 0;
    for (; j < n; ++j) {
      const uint32_t tS = tmem + lane_base + ((j & 1) ? kColS1 : kColS0);
      if (live) live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[j & 1]), (j >> 1) & 1, wc));
      if (!live) {  // aborted: keep the barrier schedule with the MMA warp, do nothing else
        nb_sync(kNbP + (j & 1), kNbWide);
        continue;
      }
      tc_fence_after_sync();
      uint32_t r[2][32];
      tmem_ld32(tS, r[0]);
      tmem_ld32(tS + 32, r[1]);
      tmem_wait_ld();
      reg_fence32(r[0]);
      reg_fence32(r[1]);
      const int k0 = (jlo + j) * BN;
      const bool masked = !keys_full(p.mask, q0, q1, k0);  // CTA-uniform
      const bool fast = raw_ok && !masked;
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
      if (fast) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) mx[e & 7] = fmaxf(mx[e & 7], __uint_as_float(r[c][e]));
      } else {
        const int c_lo = fk - k0, c_hi = last_key - k0;  // allowed columns [c_lo, c_hi]
        const float base = kAlibi ? (float)(k0 - i) * kb : 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = c * 32 + e;
            const float x = __uint_as_float(r[c][e]);
            float s2 = kAlibi ? fmaf(x, k1, fmaf((float)col, kb, base)) : x * k1;
            if (kSoftcap) s2 = capA * tanh_approx(s2);
            if (masked) s2 = (col >= c_lo && col <= c_hi) ? s2 : -INFINITY;
            mx[e & 7] = fmaxf(mx[e & 7], s2);
            r[c][e] = __float_as_uint(s2);
          }
      }
      float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      if (fast) mt *= k1;
      const float m_new = fmaxf(m_run, mt);
      const bool warp_grow = __any_sync(0xffffffffu, m_new > m_run + kRescaleLog2);
      float corr = 1.f;
      if (warp_grow) {  // O is rescaled below, once P V of the previous tile is done
        corr = m_new == -INFINITY ? 1.f : ex2_approx(m_run - m_new);
        m_run = m_new;
        l_run *= corr;
      }
      const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
      const float mul = fast ? k1 : 1.f;
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(r[c][2 * e]), mul, neg_m));
          const float p1 = ex2_approx(fmaf(__uint_as_float(r[c][2 * e + 1]), mul, neg_m));
          acc[(2 * e) & 7] += p0;
          acc[(2 * e + 1) & 7] += p1;
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tS + c * 16, pk);
      }
      l_run += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      // P V of the previous tile has had the softmax above to finish: wait for it every
      // tile (so that the phase count of pv_done stays exact), then rescale O if needed.
      if (j >= 1) {
        if (live) live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->pv_done), (j - 1) & 1, wc));
        tc_fence_after_sync();
      }
      if (live && warp_grow && j >= 1) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_wait_ld();
          reg_fence32(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
          tmem_st32(tO + c * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before_sync();
      nb_arrive(kNbP + (j & 1), kNbWide);
    }
    // ---------------------------------------------------------- result
    bool have_o = live && j == n;
    if (have_o) have_o = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->o_full), 0, wc));
    tc_fence_after_sync();
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    uint4* orow = reinterpret_cast<uint4*>(a.o + ((size_t)bh * p.Nq + (valid ? i : 0)) * D);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      if (have_o) {  // warp-uniform
        tmem_ld32(tO + c * 32, o);
        tmem_wait_ld();
        reg_fence32(o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      if (valid) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
          w.y = pack_bf16x2(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
          w.z = pack_bf16x2(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
          w.w = pack_bf16x2(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
          orow[c * 4 + e] = w;
        }
      }
    }
    if (valid)
      a.lse[(size_t)bh * p.Nq + i] = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool kAlibi, bool kSoftcap>
cudaError_t launch_variant(const Args& a, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                           cudaStream_t st) {
  auto kern = fwd256_kernel<kAlibi, kSoftcap>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, kAlloc, st>>>(tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd256_tc(const Problem& p, const __nv_bfloat16* q, const CUtensorMap& tk,
                             const CUtensorMap& tv, __nv_bfloat16* o, float* lse, cudaStream_t st) {
  Args a{};
  a.p = p;
  a.q = q;
  a.o = o;
  a.lse = lse;
  a.nqb = ceil_div(p.Nq, BM);
  const long long grid = (long long)a.nqb * p.B * p.Hq;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL || p.d != D) return cudaErrorInvalidValue;
  const bool al = p.score_kind & ATTN_SCORE_ALIBI, sc = p.score_kind & ATTN_SCORE_SOFTCAP;
  if (al && sc) return launch_variant<true, true>(a, tk, tv, (int)grid, st);
  if (al) return launch_variant<true, false>(a, tk, tv, (int)grid, st);
  if (sc) return launch_variant<false, true>(a, tk, tv, (int)grid, st);
  return launch_variant<false, false>(a, tk, tv, (int)grid, st);
}

}  // namespace attn
