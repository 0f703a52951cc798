// Forward attention on the fifth-generation tensor cores (tcgen05, sm_103a).
//
// The algorithm is the tiled forward of "FlashAttention/es" ("El algoritmo
// FlashAttention"): for a block of query rows keep a running max m, a running
// normaliser l and an output accumulator O; for each key/value tile compute the
// score tile S = Q K^T, update m, rescale O and l by exp(m_old - m_new), add
// P V and the row sums of P; at the end divide O by l and store L = m + log l.
// Like FlashAttention-2 ("Variantes y sucesores") the outer loop is over query
// blocks (one CTA each) and the division by l is deferred to the end.
//
// GB300 mapping (the FlashAttention-4 ideas named in "El FlexAttention de PyTorch
// con FlashAttention-4 es un cambio radical": tensor memory, asynchronous MMAs,
// warp specialisation, 256 x 128 tiles on Blackwell):
//   * one CTA = 2 query tiles of 128 rows (256 rows) against key tiles of 128; under
//     grouped-query attention with an even group size (kPairs) the two tiles are the same
//     128 rows of two query heads of one KV group instead: equal key-tile ranges, the same
//     K/V tiles, so neither tile idles while the other takes a key tile alone;
//   * thread 0 issues the TMA copies of the two Q tiles and of the first four ring uses
//     as soon as the barriers are initialised; warp 8 then streams the remaining K_j, V_j
//     through the shared-memory ring (128-byte swizzle), skipping the key tiles the mask
//     empties;
//   * warp 9 allocates tensor memory and issues every tcgen05.mma from one thread:
//     S_t = Q_t K_j^T into TMEM, then O_t += P_t V_j with P_t read from TMEM;
//     the two query tiles ping-pong so that the softmax of one tile overlaps the
//     MMAs of the other;
//   * warps 0-3 and 4-7 are the softmax warpgroups of tiles 0 and 1: one thread
//     per query row reads its 128 scores from TMEM, applies the score and mask
//     modifications, updates m and l with exp2, writes P as bf16 back into the
//     score columns, and rescales its O row in TMEM when the max has grown by more
//     than 2^8 (a stale max is exact: O and l share it until the final division);
//     at the end each warp stages its 32 rows of O / l in shared memory over its Q tile
//     and writes them out as whole rows.
//   * warps 8-11 form the third warpgroup (warp 11 has no role); it drops to 40
//     registers a thread so that each softmax thread can hold its 128 scores and the
//     row state in 232 without spilling.
// Tensor memory: S0 cols [0,128), S1 [128,256), O0 [256,256+d), O1 [256+d,256+2d).
//
// Dropout variant (kDrop, bf16 only): the bf16 P is ANDed with the keep mask (one Philox
// call per 16 keys of a row) before the P V product; the row sums and the LSE keep the
// undropped P, and the epilogue divides O by l (1 - p).
//
// FP8 variant (kFp8, d = 128): Q and K are e4m3 with one scale per 128-row tile, V is
// e4m3 stored transposed ([d, keys] per head, keys contiguous) with one scale per head,
// so both MMAs read K-major 8-bit operands (kind::f8f6f4, K = 32 per instruction). The
// score of a tile pair is scale * s_q * s_k * (Q8 K8^T); P is computed as
// exp2(s - m + 7) = 2^7 P and rounded to e4m3 before P V (so values down to 2^-16 keep a
// relative error of 2^-4 and smaller ones an absolute error of at most 2^-17); the row
// sums l add up the unrounded 2^7 P, and the epilogue multiplies O by s_v / l (the 2^7
// cancels) and subtracts 7 from log2 l for the LSE. The running max may lag the true
// max by at most 2^1 here (not 2^8), so 2^7 P <= 256 stays below e4m3's 448.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int BM = 128;        // query rows per query tile (= MMA M, TMEM lanes)
constexpr int BN = 128;        // keys per key tile (= MMA N of S)
constexpr int kQTiles = 2;     // query tiles per CTA
constexpr int kStages = 4;     // K/V shared-memory ring depth (each stage one tile)
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kRelayWarp = 10;  // turns TMA completions into named-barrier arrivals
constexpr int kThreads = 384;   // warp 11 only completes the third warpgroup
// Registers per thread after the reallocation: the two softmax warpgroups hold a row of
// 128 scores each; the third warpgroup (loader, MMA issuer, relay, idle) needs few.
// 2 x 128 x 232 + 128 x 40 = 384 x 168, the pool the launch bounds give.
constexpr int kRegsSoftmax = 232, kRegsOther = 40;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsOther <= kThreads * 168, "register pool");
// Named barriers (the MMA warp waits only on these; see nb_sync in ptx.cuh):
//   kNbP + t      P_t written to TMEM: softmax warpgroup t (128) + MMA warp (32)
//   kNbKv + s     ring stage s loaded: relay warp (32) + MMA warp (32)
constexpr uint32_t kNbP = 1, kNbPCount = 160;
constexpr uint32_t kNbKv = 3, kNbKvCount = 64;
constexpr int kHeadGroup = 4;  // heads whose CTAs are scheduled together (L2 reuse)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the max grows by > 2^8
constexpr float kRescaleLog2Fp8 = 1.0f;  // FP8: P = exp2(s - m) <= 2, so P 2^7 fits e4m3
constexpr float kPScaleLog2Fp8 = 7.0f;  // P is scaled by 2^7 before rounding to e4m3

template <int D, bool kFp8>
struct Layout {
  static constexpr int kElem = kFp8 ? 1 : 2;           // bytes per element
  static constexpr int kChunk = BM * 128;               // one 128-byte-wide slab: 16 KB
  static constexpr int kSlabs = D * kElem / 128;        // slabs per tile
  static constexpr int kTile = BM * D * kElem;          // one Q/K/V tile (fp8: V^T tile)
  static constexpr int kQ = 0;
  static constexpr int kRing = kQ + kQTiles * kTile;
  static constexpr int kBars = kRing + kStages * kTile;
  static constexpr int kBytes = kBars + 256;
  static constexpr int kAlloc = kBytes + 1024;          // room to align the base
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
};

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[kQTiles];
  uint64_t o_full[kQTiles];
  uint32_t tmem_base;
  int abort_flag;
};

struct FwdArgs {
  Problem p;
  __nv_bfloat16* o;
  float* lse;
  int num_qblocks;  // query blocks per unit: ceil(Nq / 256), or ceil(Nq / 128) with head pairs
  // Head pairs (grouped-query attention with an even group size): a CTA takes the same 128
  // query rows of two query heads of one KV group, whose key-tile ranges are equal and
  // whose K/V tiles are the same, instead of two adjacent 128-row tiles of one head.
  int head_pairs;
  // FP8 only: dequantisation scales of Q [B*Hq, nqt], K [B*Hkv, nkt], V [B*Hkv]
  const float* sq;
  const float* sk;
  const float* sv;
  int nqt, nkt;     // 128-row tiles per head of Q and K
};

// CTA -> (unit, query block): a unit is a query head (batch*head), or with head pairs
// two consecutive query heads. Units are taken kHeadGroup at a time so the CTAs running
// together share K/V in L2; inside a group the longest query blocks (most key tiles
// under causal masks) come first.
__device__ __forceinline__ void cta_work(const FwdArgs& a, int& bh, int& qb) {
  const int BH = a.p.B * a.p.Hq / (a.head_pairs ? 2 : 1), nqb = a.num_qblocks;
  const int per_group = kHeadGroup * nqb;
  const int grp = blockIdx.x / per_group;
  const int rem = blockIdx.x - grp * per_group;
  const int gh = imin(kHeadGroup, BH - grp * kHeadGroup);
  qb = nqb - 1 - rem / gh;
  bh = grp * kHeadGroup + rem % gh;
}

template <int D, bool kAlibi, bool kSoftcap, bool kFp8, bool kDrop, bool kPairs>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using L = Layout<D, kFp8>;
  // O (bf16) is staged on its way out from offset 0, over the Q tiles (and for FP8 the
  // first ring stages), all free once the last MMA has completed.
  constexpr int kOTile = BM * D * 2;
  static_assert(kQTiles * kOTile <= L::kBars, "O staging fits below the barriers");
  static_assert(!kFp8 || D == 128, "the FP8 path is built for d = 128");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBars);
  const Problem& p = a.p;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int unit, qb;
  cta_work(a, unit, qb);
  // Query tile t: rows q0 + t * dq .. + 127 of query head bh0 + t * dh.
  constexpr bool hp = kPairs;
  const int bh0 = hp ? 2 * unit : unit;
  const int dq = hp ? 0 : BM, dh = hp ? 1 : 0;
  const int q0 = qb * (hp ? BM : kQTiles * BM);
  const int b = bh0 / p.Hq, h0 = bh0 - b * p.Hq;
  const int g = h0 / (p.Hq / p.Hkv);  // the pair's heads share it
  const int bg = b * p.Hkv + g;

  TileRange rng[kQTiles];
#pragma unroll
  for (int t = 0; t < kQTiles; ++t) rng[t] = kv_tiles_for_rows(p.mask, q0 + t * dq, BM);
  int lo = 1 << 30, hi = 0;
#pragma unroll
  for (int t = 0; t < kQTiles; ++t)
    if (rng[t].hi > rng[t].lo) { lo = imin(lo, rng[t].lo); hi = imax(hi, rng[t].hi); }

  if (hi <= lo) {  // the mask leaves these rows no key: O = 0, L = -inf
    for (int r = threadIdx.x; r < kQTiles * BM; r += kThreads) {
      const int t = r / BM, i = q0 + t * dq + (r - t * BM);
      const int bh = bh0 + t * dh;
      if (i >= p.Nq) continue;
      uint4* orow = reinterpret_cast<uint4*>(a.o + ((size_t)bh * p.Nq + i) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
      a.lse[(size_t)bh * p.Nq + i] = -INFINITY;
    }
    return;
  }
  const int n_kv = hi - lo;

  WaitCtx wc{&bars->abort_flag, p.status};
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->q_full), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 1);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1);
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(smem_u32(&bars->s_full[t]), 1);
      mbar_init(smem_u32(&bars->o_full[t]), 1);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
    // Q and the first ring uses go out before the rest of the set-up (the loader warp
    // starts after them).
    const uint32_t qbar = smem_u32(&bars->q_full);
    mbar_arrive_expect_tx(qbar, kQTiles * L::kTile);
#pragma unroll
    for (int t = 0; t < kQTiles; ++t)
#pragma unroll
      for (int c = 0; c < L::kSlabs; ++c)
        tma_load_3d(smem_u32(smem + L::kQ + t * L::kTile + c * L::kChunk), &tm_q, qbar,
                    c * (128 / L::kElem), q0 + t * dq, bh0 + t * dh);
    for (int u = 0; u < imin(kStages, 2 * n_kv); ++u) {
      const uint32_t fb = smem_u32(&bars->kv_full[u]);
      mbar_arrive_expect_tx(fb, L::kTile);
      const CUtensorMap* map = (u & 1) ? &tm_v : &tm_k;
      const int krow = (lo + (u >> 1)) * BN;
      if (kFp8 && (u & 1)) {
        tma_load_3d(smem_u32(smem + L::kRing + u * L::kTile), map, fb, krow, 0, bg);
      } else {
#pragma unroll
        for (int c = 0; c < L::kSlabs; ++c)
          tma_load_3d(smem_u32(smem + L::kRing + u * L::kTile + c * L::kChunk), map, fb,
                      c * (128 / L::kElem), krow, bg);
      }
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), L::kTmemCols);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= 8) {
    // The third warpgroup gives registers back before its warps take their roles.
    setmaxnreg_dec<kRegsOther>();
    if (warp == kLoadWarp) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        const uint32_t qbar = smem_u32(&bars->q_full);
        for (int u = imin(kStages, 2 * n_kv); u < 2 * n_kv; ++u) {
          const int s = u % kStages, use = u / kStages;
          if (!mbar_wait(smem_u32(&bars->kv_empty[s]), (use & 1) ^ 1, wc)) break;
          const uint32_t fb = smem_u32(&bars->kv_full[s]);
          mbar_arrive_expect_tx(fb, L::kTile);
          const CUtensorMap* map = (u & 1) ? &tm_v : &tm_k;
          const int krow = (lo + (u >> 1)) * BN;
          if (kFp8 && (u & 1)) {  // V^T tile: keys krow.. (x), all d rows (y)
            tma_load_3d(smem_u32(smem + L::kRing + s * L::kTile), map, fb, krow, 0, bg);
          } else {
#pragma unroll
            for (int c = 0; c < L::kSlabs; ++c)
              tma_load_3d(smem_u32(smem + L::kRing + s * L::kTile + c * L::kChunk), map, fb,
                          c * (128 / L::kElem), krow, bg);
          }
        }
        // Do not leave while copies into this CTA's shared memory are in flight.
        mbar_wait(qbar, 0, wc);
        for (int u = imax(0, 2 * n_kv - kStages); u < 2 * n_kv; ++u)
          mbar_wait(smem_u32(&bars->kv_full[u % kStages]), (u / kStages) & 1, wc);
      }
    } else if (warp == kRelayWarp) {
      // ------------------------------------------------------------ relay
      // Ring use u is stage u % kStages; after its TMA bytes land, arrive on that
      // stage's named barrier for the MMA warp. After an abort, rendezvous instead.
      bool live = true;
      for (int u = 0; u < 2 * n_kv; ++u) {
        const int s = u % kStages;
        if (live)
          live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->kv_full[s]), (u / kStages) & 1, wc));
        if (live) nb_arrive(kNbKv + s, kNbKvCount);
        else nb_sync(kNbKv + s, kNbKvCount);
      }
    } else if (warp == kMmaWarp) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp walks the schedule and waits on named barriers; every lane executes
      // the MMA instructions predicated on `issuer`, the one lane elect.sync picks, so the
      // warp never diverges (with an elect.sync predicate MMAs go out back to back, each
      // taking its tensor or shared-memory time; a predicate computed from the lane index
      // costs about 82 cycles per MMA). If the Q tiles never arrive
      // (`ok` false) the warp keeps every barrier operation and issues nothing.
      constexpr uint32_t idS = kFp8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idO = kFp8 ? idesc_e4m3_f32(BM, D) : idesc_bf16_f32(BM, D, false, true);
      const uint32_t q_base = smem_u32(smem + L::kQ);
      const uint32_t ring = smem_u32(smem + L::kRing);
      int np[kQTiles] = {0, 0};  // P tiles consumed per query tile
      const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->q_full), 0, wc));
      const bool issuer = elect_one();
      auto commit = [&](uint64_t* bar) {
        if (ok) mma_commit_if(issuer, smem_u32(bar));
      };

      auto sync_stage = [&](int u) {
        nb_sync(kNbKv + u % kStages, kNbKvCount);
        tc_fence_after_sync();
      };
      auto issue_s = [&](int t, int u) {  // S_t = Q_t K^T with K in ring use u
        if (!ok) return;
        const uint32_t kb = ring + (u % kStages) * L::kTile;
        const uint32_t qt = q_base + t * L::kTile;
        const uint64_t dq = smem_desc_sw128(qt, 16, 1024), dk = smem_desc_sw128(kb, 16, 1024);
        const uint32_t col = t == 0 ? L::kColS0 : L::kColS1;
        // 32 bytes of the head dimension per instruction (16 bf16 or 32 e4m3 values)
#pragma unroll
        for (int kk = 0; kk < D * L::kElem / 32; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kChunk + (kk & 3) * 32) >> 4;
          if (kFp8) mma_f8_ss_if(issuer, tmem + col, dq + off, dk + off, idS, kk > 0 ? 1u : 0u);
          else mma_ss_if(issuer, tmem + col, dq + off, dk + off, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit_if(issuer, smem_u32(&bars->s_full[t]));
      };
      auto issue_pv = [&](int t, int u) {  // O_t += P_t V with V in ring use u
        if (!ok) return;
        const uint32_t vb = ring + (u % kStages) * L::kTile;
        const uint32_t colS = t == 0 ? L::kColS0 : L::kColS1;
        const uint32_t colO = t == 0 ? L::kColO0 : L::kColO1;
        if (kFp8) {  // P (e4m3, 4 per column) x V^T tile (K-major): 32 keys per instruction
          const uint64_t dv = smem_desc_sw128(vb, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < BN / 32; ++kk)
            mma_f8_ts_if(issuer, tmem + colO, tmem + colS + kk * 8, dv + ((kk * 32) >> 4), idO,
                         (np[t] > 0 || kk > 0) ? 1u : 0u);
        } else {  // P (bf16 pairs) x V tile used MN-major: 16 keys per instruction
          const uint64_t dv = smem_desc_sw128(vb, L::kChunk, 1024);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts_if(issuer, tmem + colO, tmem + colS + kk * 8, dv + ((kk * 16 * 128) >> 4), idO,
                      (np[t] > 0 || kk > 0) ? 1u : 0u);
        }
      };

      sync_stage(0);
#pragma unroll
      for (int t = 0; t < kQTiles; ++t)
        if (lo >= rng[t].lo && lo < rng[t].hi) issue_s(t, 0);
      commit(&bars->kv_empty[0]);
      for (int jj = 0; jj < n_kv; ++jj) {
        const int j = lo + jj;
        const int uv = 2 * jj + 1, uk = 2 * jj + 2;
        const bool next = jj + 1 < n_kv;
        sync_stage(uv);
#pragma unroll
        for (int t = 0; t < kQTiles; ++t) {
          if (j >= rng[t].lo && j < rng[t].hi) {
            nb_sync(kNbP + t, kNbPCount);
            tc_fence_after_sync();
            issue_pv(t, uv);
            ++np[t];
          }
          if (next) {
            if (t == 0) sync_stage(uk);
            if (j + 1 >= rng[t].lo && j + 1 < rng[t].hi) issue_s(t, uk);
          }
        }
        commit(&bars->kv_empty[uv % kStages]);
        if (next) commit(&bars->kv_empty[uk % kStages]);
      }
#pragma unroll
      for (int t = 0; t < kQTiles; ++t) commit(&bars->o_full[t]);
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int row = (warp & 3) * 32 + lane;  // TMEM lane = row in the tile
    const int r0 = q0 + t * dq;              // the tile's first query row
    const int i = r0 + row;                  // query position
    const int bh = bh0 + t * dh, h = h0 + t * dh;  // the tile's query head
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + (t == 0 ? L::kColS0 : L::kColS1);
    const uint32_t tO = tmem + lane_base + (t == 0 ? L::kColO0 : L::kColO1);
    const int fk = first_key(p.mask, i < p.Nq ? i : p.Nq - 1);
    // Scores in log2 units: s2 = x * k1 + (j - i) * kb. With the soft-cap c the same
    // expression gives the pre-cap score over c; the pass keeps the tanh of it and the
    // exponent pass multiplies by capA = c log2(e), as the raw-score path does with k1.
    const float slope = kAlibi ? alibi_slope(h, p.Hq) : 0.f;
    const float k1 = kSoftcap ? p.scale / p.softcap : p.scale * kLog2e;
    const float kb = kSoftcap ? slope / p.softcap : slope * kLog2e;
    const float capA = kSoftcap ? p.softcap * kLog2e : 0.f;
    // The common case (no score mod, positive scale, tile fully allowed) works on the
    // raw scores x: max over x, then p = exp2(x * k1 - m) in one FFMA + ex2.
    const bool raw_ok = !kAlibi && !kSoftcap && k1 > 0.f;
    // FP8: the tile pair's dequantisation factor s_q s_k scales k1 (and kb stays)
    const int qtile = r0 / BM;  // may lie past the last tile (then no key tile runs)
    const float sqv = (kFp8 && qtile < a.nqt) ? a.sq[(size_t)bh * a.nqt + qtile] : 1.f;
    const int last_key = (p.mask.kind == ATTN_MASK_NONE ? p.Nkv - 1 : imin(i, p.Nkv - 1));
    float m_run = -INFINITY, l_run = 0.f;
    int n = 0;
    bool live = true;
    for (int j = rng[t].lo; j < rng[t].hi; ++j, ++n) {
      const float k1j = kFp8 ? k1 * sqv * a.sk[(size_t)bg * a.nkt + j] : k1;
      // Keep every decision warp-uniform: tcgen05.ld/st are warp-collective.
      if (live) live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[t]), n & 1, wc));
      if (!live) {  // aborted: keep the barrier schedule with the MMA warp, do nothing else
        nb_sync(kNbP + t, kNbPCount);
        continue;
      }
      tc_fence_after_sync();
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, r[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence32(r[c]);
      const int k0 = j * BN;
      const bool masked = tile_needs_mask(p.mask, r0, k0, BN);
      const bool fast = raw_ok && !masked;  // warp-uniform
      // Row max in eight independent chains (the scores stay in r).
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
      if (fast) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) mx[e & 7] = fmaxf(mx[e & 7], __uint_as_float(r[c][e]));
      } else {
        // Allowed columns of this row in this tile: [c_lo, c_hi].
        const int c_lo = fk - k0, c_hi = last_key - k0;
        const float base = kAlibi ? (float)(k0 - i) * kb : 0.f;
        const uint64_t k1j2 = f32x2(k1j, k1j);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 2) {  // column pairs: packed fp32x2 arithmetic
            const int col = c * 32 + e;
            const uint64_t x2 = f32x2(__uint_as_float(r[c][e]), __uint_as_float(r[c][e + 1]));
            uint64_t s2 = kAlibi ? fma_f32x2(x2, k1j2,
                                             f32x2(fmaf((float)col, kb, base),
                                                   fmaf((float)(col + 1), kb, base)))
                                 : mul_f32x2(x2, k1j2);
            if (kSoftcap) {  // t = tanh of the pre-cap score over c (capA t in log2 units)
              float a0, a1;
              f32x2_split(s2, a0, a1);
              s2 = f32x2(tanh_approx(a0), tanh_approx(a1));
            }
            float v0, v1;
            f32x2_split(s2, v0, v1);
            if (masked) {
              v0 = (col >= c_lo && col <= c_hi) ? v0 : -INFINITY;
              v1 = (col + 1 >= c_lo && col + 1 <= c_hi) ? v1 : -INFINITY;
            }
            mx[e & 7] = fmaxf(mx[e & 7], v0);
            mx[(e + 1) & 7] = fmaxf(mx[(e + 1) & 7], v1);
            r[c][e] = __float_as_uint(v0);
            r[c][e + 1] = __float_as_uint(v1);
          }
      }
      float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      if (fast) mt *= k1j;  // into log2 units
      else if (kSoftcap) mt *= capA;
      const float m_new = fmaxf(m_run, mt);
      const bool grow = m_new > m_run + (kFp8 ? kRescaleLog2Fp8 : kRescaleLog2);
      const bool warp_grow = __any_sync(0xffffffffu, grow);
      float corr = 1.f;
      if (warp_grow) {
        // exp2(m_old - m_new): 0 when only m_old is -inf, 1 when the row is still empty
        corr = m_new == -INFINITY ? 1.f : ex2_approx(m_run - m_new);
        m_run = m_new;
        l_run *= corr;
      }
      // FP8: exp2(s - m + 7) = 2^7 p, the scale e4m3 rounding wants, at no extra cost
      float neg_m = m_run == -INFINITY ? 0.f : -m_run;
      if constexpr (kFp8) neg_m += kPScaleLog2Fp8;
      const float mul = fast ? k1j : (kSoftcap ? capA : 1.f);  // p = exp2(v * mul - m)
      const DropThr dthr = drop_thr_words(kDrop ? p.drop_thr : 0);
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
      // The exponent argument and the sum chains on column pairs (packed fp32x2 FMAs; each
      // element's operations and its chain order as with scalar ones)
      uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
      const uint64_t mul2 = f32x2(mul, mul), negm2 = f32x2(neg_m, neg_m), one2 = f32x2(1.f, 1.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (kFp8) {  // 2^7 P as e4m3, four per column: 32 keys in 8 columns
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float pv[4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // column pairs, as for bf16 P
              float a0, a1;
              f32x2_split(fma_f32x2(f32x2(__uint_as_float(r[c][4 * e + 2 * h]),
                                          __uint_as_float(r[c][4 * e + 2 * h + 1])),
                                    mul2, negm2),
                          a0, a1);
              pv[2 * h] = ex2_approx(a0);
              pv[2 * h + 1] = ex2_approx(a1);
              const int k2 = ((4 * e + 2 * h) & 7) >> 1;  // chains (acc[2 k2], acc[2 k2 + 1])
              acc2[k2] = fma_f32x2(f32x2(pv[2 * h], pv[2 * h + 1]), one2, acc2[k2]);
            }
            pk[e] = pack_e4m3x2(pv[0], pv[1]) | (pack_e4m3x2(pv[2], pv[3]) << 16);
          }
          tmem_st8(tS + c * 8, pk);
        } else {
          // Dropout: one Philox call per 16 keys of this row (one half below) gives the
          // keep flags of those keys; l sums the undropped P (the softmax is taken before
          // dropout) and P V takes the dropped P, whose 1 / (1 - p) is applied with 1 / l
          // at the end.
          // P goes to tensor memory in two halves of 8 words where that measured faster
          // (no score mod: fewer live registers beside the 128 scores; dropout: one Philox
          // call per half), else in one 16-word store (with ALiBi / soft-cap the halves
          // ran slower on the document workload, 329 against 370 TFLOP/s).
          constexpr bool kHalves = kDrop || (!kAlibi && !kSoftcap);
          if constexpr (kHalves) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              uint32_t ph[8], kf[4];
              if (kDrop) {
                // round keys formed inside the call: kept live across the loop they cost
                // the softmax warps more than their adds
                const uint4 w = philox4x32_10((uint32_t)((k0 + c * 32) >> 4) + hf, (uint32_t)i,
                                              (uint32_t)bh, 0u,
                                              philox_keys(p.drop_seed_lo, p.drop_seed_hi));
                kf[0] = keep_flags4(w.x, dthr);
                kf[1] = keep_flags4(w.y, dthr);
                kf[2] = keep_flags4(w.z, dthr);
                kf[3] = keep_flags4(w.w, dthr);
              }
#pragma unroll
              for (int e8 = 0; e8 < 8; ++e8) {
                const int e = hf * 8 + e8;
                float a0, a1;
                f32x2_split(fma_f32x2(f32x2(__uint_as_float(r[c][2 * e]),
                                            __uint_as_float(r[c][2 * e + 1])), mul2, negm2),
                            a0, a1);
                const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
                acc2[e & 3] = fma_f32x2(f32x2(p0, p1), one2, acc2[e & 3]);  // acc + p
                ph[e8] = pack_bf16x2(p0, p1);
                if (kDrop)  // keys 2e8, 2e8 + 1 of the half: flag bytes (2e8) % 4, +1 of word e8 / 2
                  ph[e8] &= keep_mask_pair(kf[e8 >> 1], 2 * (e8 & 1));
              }
              tmem_st8(tS + c * 16 + hf * 8, ph);
            }
          } else {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float a0, a1;
              f32x2_split(fma_f32x2(f32x2(__uint_as_float(r[c][2 * e]),
                                          __uint_as_float(r[c][2 * e + 1])), mul2, negm2),
                          a0, a1);
              const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
              acc2[e & 3] = fma_f32x2(f32x2(p0, p1), one2, acc2[e & 3]);  // acc + p
              pk[e] = pack_bf16x2(p0, p1);
            }
            tmem_st16(tS + c * 16, pk);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e)  // chains (acc[2k], acc[2k + 1]) were kept in pairs
        f32x2_split(acc2[e], acc[2 * e], acc[2 * e + 1]);
      l_run += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      if (warp_grow && n > 0) {  // O_t already holds P V of earlier tiles: rescale it
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
      nb_arrive(kNbP + t, kNbPCount);
    }
    // ---------------------------------------------------------- epilogue
    // Every tile waits for the CTA's last MMA, also a tile without key tiles: the O
    // staging below writes over shared memory that MMAs of the other tile read (for FP8
    // the second tile's staging area is the first ring stages).
    const bool mma_done = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->o_full[t]), 0, wc));
    const bool have_o = n > 0 && mma_done;  // O_t holds at least one P V product
    tc_fence_after_sync();
    float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    if (kDrop) inv *= p.drop_scale;  // the kept terms' 1 / (1 - p)
    if (kFp8) inv *= a.sv[bg];  // l holds 2^7 times the row sum, like O
    // O_t / l: each warp stages its 32 rows in shared memory over its Q tile (128-byte
    // rows of 64 columns, 16-byte chunk c of row r at chunk c ^ (r & 7)), then copies them
    // out with each store instruction writing two whole rows (512 contiguous bytes).
    uint8_t* otile = smem + t * kOTile;
    {
      uint32_t o[D];
      if (have_o) {  // warp-uniform
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
          tmem_ld32(tO + c * 32, *reinterpret_cast<uint32_t(*)[32]>(o + c * 32));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(o + c * 32));
      } else {
#pragma unroll
        for (int e = 0; e < D; ++e) o[e] = 0u;
      }
#pragma unroll
      for (int gc = 0; gc < D / 8; ++gc) {  // 16-byte chunk gc of the row: slab gc / 8
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(o[8 * gc + 0]) * inv, __uint_as_float(o[8 * gc + 1]) * inv);
        w.y = pack_bf16x2(__uint_as_float(o[8 * gc + 2]) * inv, __uint_as_float(o[8 * gc + 3]) * inv);
        w.z = pack_bf16x2(__uint_as_float(o[8 * gc + 4]) * inv, __uint_as_float(o[8 * gc + 5]) * inv);
        w.w = pack_bf16x2(__uint_as_float(o[8 * gc + 6]) * inv, __uint_as_float(o[8 * gc + 7]) * inv);
        *reinterpret_cast<uint4*>(otile + (gc >> 3) * L::kChunk + row * 128 +
                                  (((gc & 7) ^ (row & 7)) << 4)) = w;
      }
    }
    __syncwarp();
    {
      constexpr int kChunksPerRow = D / 8;               // 16-byte chunks per row
      constexpr int kRowsPerStore = 32 / kChunksPerRow;  // rows one warp store covers
      const int gc = lane % kChunksPerRow;
      const int w0 = (warp & 3) * 32;  // this warp's first row in the tile
#pragma unroll
      for (int k = 0; k < 32 / kRowsPerStore; ++k) {
        const int r = w0 + k * kRowsPerStore + lane / kChunksPerRow;
        const uint4 w = *reinterpret_cast<const uint4*>(otile + (gc >> 3) * L::kChunk + r * 128 +
                                                       (((gc & 7) ^ (r & 7)) << 4));
        const int ir = r0 + r;
        if (ir < p.Nq)
          reinterpret_cast<uint4*>(a.o + ((size_t)bh * p.Nq + ir) * D)[gc] = w;
      }
    }
    if (i < p.Nq)
      a.lse[(size_t)bh * p.Nq + i] =
          l_run > 0.f ? (m_run + log2f(l_run) - (kFp8 ? kPScaleLog2Fp8 : 0.f)) *
                            0.69314718055994531f
                      : -INFINITY;
  }
  __syncwarp();

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// Head pairs when the query heads of a KV group come in pairs (then Hq is even too).
void set_units(FwdArgs& a) {
  a.head_pairs = (a.p.Hq / a.p.Hkv) % 2 == 0 ? 1 : 0;
  a.num_qblocks = ceil_div(a.p.Nq, a.head_pairs ? BM : kQTiles * BM);
}

template <int D, bool kAlibi, bool kSoftcap, bool kFp8 = false, bool kDrop = false>
cudaError_t launch_variant(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, int grid, cudaStream_t st) {
  auto kern = a.head_pairs ? fwd_tc_kernel<D, kAlibi, kSoftcap, kFp8, kDrop, true>
                           : fwd_tc_kernel<D, kAlibi, kSoftcap, kFp8, kDrop, false>;
  const int smem = Layout<D, kFp8>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

template <int D, bool kDrop>
cudaError_t launch_dd(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                      const CUtensorMap& tv, int grid, cudaStream_t st) {
  const bool al = a.p.score_kind & ATTN_SCORE_ALIBI, sc = a.p.score_kind & ATTN_SCORE_SOFTCAP;
  if (al && sc) return launch_variant<D, true, true, false, kDrop>(a, tq, tk, tv, grid, st);
  if (al) return launch_variant<D, true, false, false, kDrop>(a, tq, tk, tv, grid, st);
  if (sc) return launch_variant<D, false, true, false, kDrop>(a, tq, tk, tv, grid, st);
  return launch_variant<D, false, false, false, kDrop>(a, tq, tk, tv, grid, st);
}

template <int D>
cudaError_t launch_d(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, int grid, cudaStream_t st) {
  if (a.p.score_kind & ATTN_SCORE_DROPOUT) return launch_dd<D, true>(a, tq, tk, tv, grid, st);
  return launch_dd<D, false>(a, tq, tk, tv, grid, st);
}

}  // namespace

cudaError_t launch_fwd_tc(const Problem& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, __nv_bfloat16* o, float* lse,
                          cudaStream_t st) {
  FwdArgs a{};
  a.p = p;
  a.o = o;
  a.lse = lse;
  set_units(a);
  const long long grid = (long long)a.num_qblocks * p.B * p.Hq / (a.head_pairs ? 2 : 1);
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (p.d == 64) return launch_d<64>(a, tq, tk, tv, (int)grid, st);
  return launch_d<128>(a, tq, tk, tv, (int)grid, st);
}

}  // namespace attn

namespace attn {

cudaError_t launch_fwd_fp8_tc(const Problem& p, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tvt, const float* sq, const float* sk,
                              const float* sv, __nv_bfloat16* o, float* lse, cudaStream_t st) {
  FwdArgs a{};
  a.p = p;
  a.o = o;
  a.lse = lse;
  set_units(a);
  a.sq = sq;
  a.sk = sk;
  a.sv = sv;
  a.nqt = ceil_div(p.Nq, BM);
  a.nkt = ceil_div(p.Nkv, BN);
  const long long grid = (long long)a.num_qblocks * p.B * p.Hq / (a.head_pairs ? 2 : 1);
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL || p.d != 128) return cudaErrorInvalidValue;
  const bool al = p.score_kind & ATTN_SCORE_ALIBI, sc = p.score_kind & ATTN_SCORE_SOFTCAP;
  if (al && sc) return launch_variant<128, true, true, true>(a, tq, tk, tvt, (int)grid, st);
  if (al) return launch_variant<128, true, false, true>(a, tq, tk, tvt, (int)grid, st);
  if (sc) return launch_variant<128, false, true, true>(a, tq, tk, tvt, (int)grid, st);
  return launch_variant<128, false, false, true>(a, tq, tk, tvt, (int)grid, st);
}

}  // namespace attn
