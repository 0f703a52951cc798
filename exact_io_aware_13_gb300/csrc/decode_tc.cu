// Attention of the newest query tokens of many sequences over a paged KV cache
// (decode), on the tcgen05 tensor cores, split over fixed-size key chunks; and the
// kernel that merges the chunks by their log-sum-exp.
//
// What is computed is the forward of "FlashAttention/es" ("El algoritmo
// FlashAttention": running max, running sum, rescaled accumulator, L = m + log l) for
// the queries of one decode step. The KV cache is paged, as PagedAttention does it
// ("Variantes y sucesores" on the same page): token t of sequence b lives in page
// page_table[b][t / page_size], slot t % page_size, of a [pages, Hkv, page_size, d]
// pool. The Nq queries of a sequence are its newest tokens (query i at position
// L - Nq + i), so masks and ALiBi are aligned at the bottom right.
//
// GB300 mapping. Decode reads every cached key once and does little arithmetic per
// byte, so the kernel is built to keep HBM busy:
//   * one CTA = one 64-key-aligned chunk of one sequence's keys for one kv head; the
//     G = Hq / Hkv query heads of the group and their Nq tokens are packed into the
//     M = 128 rows of one MMA tile (rows g * Nq + i), so each K/V byte fetched serves
//     the whole group;
//   * warp 0 streams K and V tiles of 64 keys through a 2-stage shared-memory ring
//     with TMA (128-byte swizzle), one box per page piece (page sizes below 64 take
//     several boxes per tile); it reads the page table 32 entries at a time;
//   * warp 1 issues S = Q K^T (N = 64) and O += P V from one elected thread, with P
//     read from tensor memory;
//   * warps 2-5 do the online softmax, one thread per row, warps without a valid row
//     idle; O is rescaled in tensor memory only when the max grows by more than 2^8;
//   * two CTAs fit on an SM (about 97 KB of shared memory and 256 TMEM columns each),
//     so one CTA's start-up and epilogue overlap the other's streaming.
// Tensor memory: S0 cols [0,64), S1 [64,128), O [128, 128+d).
//
// The last tile of a sequence can end inside a page whose later slots hold no token
// (possibly NaN). S columns past the sequence are masked before the max; the V rows
// there are zeroed in shared memory by the loader before the P V product (0 * NaN
// would be NaN).
//
// Split mode (more than one chunk per sequence): each CTA writes, per row, O_c / l_c in
// fp32 and L2_c = m_c + log2 l_c; the combine kernel forms
//   M = max_c L2_c, w_c = 2^(L2_c - M), O = sum_c w_c O_c / sum_c w_c,
//   L = (M + log2 sum_c w_c) ln 2,
// in a fixed chunk order (deterministic).
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int BM = 128;      // packed query rows per CTA (MMA M, TMEM lanes)
constexpr int BN = 64;       // keys per tile (MMA N of S, K of P V)
constexpr int kStages = 2;   // K/V ring depth
constexpr int kLoadWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kFirstSoftmaxWarp = 2;
constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;
constexpr unsigned long long kDrainLimitNs = 200000000ull;  // waits for own copies at exit

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;           // 128-byte column blocks
  static constexpr int kQHalf = BM * 128;          // 16 KB
  static constexpr int kKvHalf = BN * 128;         // 8 KB
  static constexpr int kQ = 0;
  static constexpr int kRing = kQ + kHalves * kQHalf;
  static constexpr int kTileBytes = kHalves * kKvHalf;  // one K or V tile
  static constexpr int kStage = 2 * kTileBytes;          // K then V
  static constexpr int kBars = kRing + kStages * kStage;
  static constexpr int kBytes = kBars + 256;
  // At least 80 KB, so that no more than two CTAs (2 x 256 TMEM columns) share an SM.
  static constexpr int kAlloc = kBytes + 1024 > 80 * 1024 ? kBytes + 1024 : 80 * 1024;
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kColS0 = 0, kColS1 = 64, kColO = 128;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done;
  uint64_t tail;
  uint32_t tmem_base;
  int abort_flag;
};

struct Args {
  DecodeProblem p;
  DecodeOut out;
  int G, rows, row_tiles;
  long long rows_total;  // B * Hq * Nq
};

// Waits for a copy this CTA issued, ignoring the abort flag (shared memory must not be
// left while a copy into it is in flight), for at most kDrainLimitNs.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kDrainLimitNs) return;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int D, bool kAlibi, bool kSoftcap>
__global__ void __launch_bounds__(kThreads, 2)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const Args a) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBars);
  __shared__ int red_min_lo, red_max_hi, red_max_lo, red_min_hi;
  const DecodeProblem& p = a.p;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int c = blockIdx.x;
  int y = blockIdx.y;
  const int rt = y % a.row_tiles;
  y /= a.row_tiles;
  const int hk = y % p.Hkv;
  const int b = y / p.Hkv;
  const int cap = p.max_seq_len;
  int Lb = p.seq_lens[b];
  if (Lb < 0 || Lb > cap) {
    if (threadIdx.x == 0) atomicOr(p.status, DEV_BAD_INPUT);
    Lb = Lb < 0 ? 0 : cap;
  }
  const int rows_here = imin(BM, a.rows - rt * BM);
  const long long row0 = ((long long)b * p.Hq + (long long)hk * a.G) * p.Nq + (long long)rt * BM;
  const bool direct = p.n_chunks == 1;
  const int c0 = c * p.chunk;
  if (c0 >= Lb && !(direct && c == 0)) return;  // a chunk past the sequence: no work
  const int c1 = imin(c0 + p.chunk, Lb);

  // Key range of every row of the tile, and the union / intersection over rows.
  if (threadIdx.x == 0) {
    red_min_lo = 1 << 30; red_max_hi = 0; red_max_lo = 0; red_min_hi = 1 << 30;
  }
  __syncthreads();
  int row_lo = 0, row_hi = 0;  // of this thread's row (threads < BM)
  if (threadIdx.x < BM && (int)threadIdx.x < rows_here) {
    const int i = (rt * BM + (int)threadIdx.x) % p.Nq;
    decode_row_keys(p.mask_kind, p.window, Lb, p.Nq, i, row_lo, row_hi);
    if (row_hi > row_lo) { atomicMin(&red_min_lo, row_lo); atomicMax(&red_max_hi, row_hi); }
    atomicMax(&red_max_lo, row_lo);
    atomicMin(&red_min_hi, row_hi);
  }
  __syncthreads();
  const int k_lo = imax(c0, red_min_lo), k_hi = imin(c1, red_max_hi);
  const int max_lo = red_max_lo, min_hi = red_min_hi;
  if (k_hi <= k_lo) {
    // No row of this tile sees a key of this chunk. Only a single-chunk launch owns the
    // final rows (split launches leave such chunks to the combine, which skips them).
    if (direct && threadIdx.x < BM && (int)threadIdx.x < rows_here) {
      const long long r = row0 + threadIdx.x;
      uint4* orow = reinterpret_cast<uint4*>(a.out.o + r * D);
#pragma unroll
      for (int e = 0; e < D / 8; ++e) orow[e] = make_uint4(0, 0, 0, 0);
      a.out.lse[r] = -INFINITY;
    }
    return;
  }
  const int tb = k_lo / BN;
  const int n_t = ceil_div(k_hi, BN) - tb;
  const int n_active = ceil_div(rows_here, 32);  // softmax warps with a valid row

  WaitCtx wc{&bars->abort_flag, p.status};
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->q_full), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars->k_full[s]), 1);
      mbar_init(smem_u32(&bars->v_full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bars->s_full[t]), 1);
      mbar_init(smem_u32(&bars->p_full[t]), n_active);
    }
    mbar_init(smem_u32(&bars->pv_done), 1);
    mbar_init(smem_u32(&bars->tail), 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), L::kTmemCols);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    const int ps = p.page_size;
    const int R = imin(ps, BN);       // rows per box (a piece of one page)
    const int pieces = BN / R;        // boxes per tile and tensor (<= 8)
    const int32_t* table = p.page_table + (size_t)b * p.max_pages;
    auto fetch = [&](int base) {
      const int idx = base + lane;
      return idx < p.max_pages ? __ldg(table + idx) : -1;
    };
    int wbase = (tb * BN) / ps;       // page index held by lane 0 of `cur`
    int cur = fetch(wbase), nxt = fetch(wbase + 32);
    const uint32_t qbar = smem_u32(&bars->q_full);
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(qbar, L::kHalves * L::kQHalf);
#pragma unroll
      for (int hf = 0; hf < L::kHalves; ++hf)
        tma_load_3d(smem_u32(smem + L::kQ + hf * L::kQHalf), &tm_q, qbar, hf * 64, (int)row0, 0);
    }
    int issued = 0;
    for (int u = 0; u < n_t; ++u) {
      const int s = u % kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->empty[s]), ((u / kStages) & 1) ^ 1, wc)))
        break;
      const int t0 = (tb + u) * BN;
      const int valid = imin(BN, Lb - t0);  // keys of the tile inside the sequence (>= 1)
      // page pieces of this tile: lane q < pieces computes piece q
      const int first_page = t0 / ps;
      while (first_page - wbase >= 32) {  // warp-uniform
        wbase += 32;
        cur = nxt;
        nxt = fetch(wbase + 32);
      }
      int coord = 0;
      bool good = false;
      {
        const int q = lane < pieces ? lane : 0;
        const int key = t0 + q * R;
        const int off = key / ps - wbase;  // 0 .. 39
        const int pa = __shfl_sync(0xffffffffu, cur, off & 31);
        const int pb = __shfl_sync(0xffffffffu, nxt, off & 31);
        const int page = off < 32 ? pa : pb;
        const bool in_seq = lane < pieces && key < Lb;
        good = in_seq && page >= 0 && page < p.num_pages;
        if (in_seq && !good) atomicOr(p.status, DEV_BAD_INPUT);
        coord = (int)(((long long)page * p.Hkv + hk) * ps + key % ps);
      }
      const uint32_t mask = __ballot_sync(0xffffffffu, good);
      const uint32_t bytes = (uint32_t)__popc(mask) * R * 128 * L::kHalves;
      const bool tail = valid < BN;
      const uint32_t kst = smem_u32(smem + L::kRing + s * L::kStage);
      const uint32_t vst = kst + L::kTileBytes;
      const uint32_t kbar = smem_u32(&bars->k_full[s]);
      const uint32_t vbar = tail ? smem_u32(&bars->tail) : smem_u32(&bars->v_full[s]);
      if (lane == 0) {
        mbar_arrive_expect_tx(kbar, bytes);
        mbar_arrive_expect_tx(vbar, bytes);
      }
      for (int q = 0; q < pieces; ++q) {
        const int cq = __shfl_sync(0xffffffffu, coord, q);
        if (lane == 0 && ((mask >> q) & 1u)) {
#pragma unroll
          for (int hf = 0; hf < L::kHalves; ++hf) {
            tma_load_3d(kst + hf * L::kKvHalf + q * R * 128, &tm_k, kbar, hf * 64, cq, 0);
            tma_load_3d(vst + hf * L::kKvHalf + q * R * 128, &tm_v, vbar, hf * 64, cq, 0);
          }
        }
      }
      ++issued;
      if (tail) {
        // Only the last tile of a sequence is short, and a CTA meets it at most once.
        drain_wait(vbar, 0);
        // Zero V rows [valid, BN) of each 128-byte column block (a swizzled row stays
        // inside its own 128 bytes, so whole rows can be cleared in place).
        const int zrows = BN - valid;
        for (int e = lane; e < zrows * 8 * L::kHalves; e += 32) {
          const int hf = e / (zrows * 8), rem = e - hf * zrows * 8;
          const int row = valid + rem / 8, chunk16 = rem % 8;
          *reinterpret_cast<uint4*>(smem + L::kRing + s * L::kStage + L::kTileBytes +
                                    hf * L::kKvHalf + row * 128 + chunk16 * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->v_full[s]));
      }
    }
    // Do not leave while copies into this CTA's shared memory are in flight.
    drain_wait(qbar, 0);
    for (int u = imax(0, issued - kStages); u < issued; ++u) {
      drain_wait(smem_u32(&bars->k_full[u % kStages]), (u / kStages) & 1);
      drain_wait(smem_u32(&bars->v_full[u % kStages]), (u / kStages) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false, false);
    constexpr uint32_t idO = idesc_bf16_f32(BM, D, false, true);
    const uint32_t q_base = smem_u32(smem + L::kQ);
    const uint32_t ring = smem_u32(smem + L::kRing);
    bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->q_full), 0, wc));
    const bool issuer = elect_one();
    auto issue_pv = [&](int v) {
      const int s = v % kStages;
      ok = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->p_full[v & 1]), (v >> 1) & 1, wc));
      ok = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->v_full[s]), (v / kStages) & 1, wc));
      if (!ok) return;
      tc_fence_after_sync();
      const uint32_t vb = ring + s * L::kStage + L::kTileBytes;
      const uint64_t dv = smem_desc_sw128(vb, L::kKvHalf, 1024);
      const uint32_t colS = (v & 1) ? L::kColS1 : L::kColS0;
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk)  // 16 keys per instruction
        mma_ts_if(issuer, tmem + L::kColO, tmem + colS + kk * 8, dv + ((kk * 16 * 128) >> 4), idO,
                  (v > 0 || kk > 0) ? 1u : 0u);
      mma_commit_if(issuer, smem_u32(&bars->empty[s]));
      mma_commit_if(issuer, smem_u32(&bars->pv_done));
    };
    for (int u = 0; u < n_t && ok; ++u) {
      const int s = u % kStages;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->k_full[s]), (u / kStages) & 1, wc));
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t kb = ring + s * L::kStage;
      const uint64_t dq = smem_desc_sw128(q_base, 16, 1024), dk = smem_desc_sw128(kb, 16, 1024);
      const uint32_t col = (u & 1) ? L::kColS1 : L::kColS0;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {  // 16 head dims per instruction
        const uint32_t offq = ((kk >> 2) * L::kQHalf + (kk & 3) * 32) >> 4;
        const uint32_t offk = ((kk >> 2) * L::kKvHalf + (kk & 3) * 32) >> 4;
        mma_ss_if(issuer, tmem + col, dq + offq, dk + offk, idS, kk > 0 ? 1u : 0u);
      }
      mma_commit_if(issuer, smem_u32(&bars->s_full[u & 1]));
      if (u >= 1) issue_pv(u - 1);
    }
    if (ok) issue_pv(n_t - 1);
  } else {
    // ------------------------------------------------------------ softmax warps
    const int quad = warp & 3;
    if (quad * 32 < rows_here) {
      const int row = quad * 32 + lane;           // TMEM lane = packed row
      const bool valid_row = row < rows_here;
      const int pr = rt * BM + imin(row, rows_here - 1);
      const int g = pr / p.Nq, i = pr - g * p.Nq;
      const int h = hk * a.G + g;
      const int pos = Lb - p.Nq + i;
      int lo_r = 0, hi_r = 0;
      if (valid_row) decode_row_keys(p.mask_kind, p.window, Lb, p.Nq, i, lo_r, hi_r);
      const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
      const uint32_t tO = tmem + lane_base + L::kColO;
      const float slope = kAlibi ? alibi_slope(h, p.Hq) : 0.f;
      const float cap2 = kSoftcap ? 2.0f * kLog2e / p.softcap : 0.f;
      const float k1 = kSoftcap ? p.scale * cap2 : p.scale * kLog2e;
      const float kb = kSoftcap ? slope * cap2 : slope * kLog2e;
      const float capA = kSoftcap ? p.softcap * kLog2e : 0.f;
      const bool raw_ok = !kAlibi && !kSoftcap && k1 > 0.f;
      float m_run = -INFINITY, l_run = 0.f;
      bool live = true;
      int u = 0;
      for (; u < n_t; ++u) {
        const uint32_t tS = tmem + lane_base + ((u & 1) ? L::kColS1 : L::kColS0);
        live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[u & 1]), (u >> 1) & 1, wc));
        if (!live) break;
        tc_fence_after_sync();
        uint32_t r[2][32];
        tmem_ld32(tS, r[0]);
        tmem_ld32(tS + 32, r[1]);
        tmem_wait_ld();
        reg_fence32(r[0]);
        reg_fence32(r[1]);
        const int t0 = (tb + u) * BN;
        const bool masked = !(t0 >= max_lo && t0 + BN <= min_hi);  // CTA-uniform
        const bool fast = raw_ok && !masked;
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
        if (fast) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int e = 0; e < 32; ++e) mx[e & 7] = fmaxf(mx[e & 7], __uint_as_float(r[cc][e]));
        } else {
          const int c_lo = lo_r - t0, c_hi = hi_r - t0;  // allowed columns [c_lo, c_hi)
          const float base = kAlibi ? (float)(t0 - pos) * kb : 0.f;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int col = cc * 32 + e;
              const float x = __uint_as_float(r[cc][e]);
              float s2 = kAlibi ? fmaf(x, k1, fmaf((float)col, kb, base)) : x * k1;
              if (kSoftcap) s2 = capA - 2.0f * capA * rcp_approx(1.0f + ex2_approx(s2));
              if (masked) s2 = (col >= c_lo && col < c_hi) ? s2 : -INFINITY;
              mx[e & 7] = fmaxf(mx[e & 7], s2);
              r[cc][e] = __float_as_uint(s2);
            }
        }
        float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                         fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        if (fast) mt *= k1;
        const float m_new = fmaxf(m_run, mt);
        const bool grow = m_new > m_run + kRescaleLog2;
        const bool warp_grow = __any_sync(0xffffffffu, grow);
        // O is stable once P V of the previous tile has completed.
        if (u >= 1) {
          live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->pv_done), (u - 1) & 1, wc));
          if (!live) break;
          tc_fence_after_sync();
        }
        float corr = 1.f;
        if (warp_grow) {
          corr = m_new == -INFINITY ? 1.f : ex2_approx(m_run - m_new);
          m_run = m_new;
          l_run *= corr;
          if (u >= 1) {
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t o[32];
              tmem_ld32(tO + cc * 32, o);
              tmem_wait_ld();
              reg_fence32(o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
              tmem_st32(tO + cc * 32, o);
            }
          }
        }
        const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
        const float mul = fast ? k1 : 1.f;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = ex2_approx(fmaf(__uint_as_float(r[cc][2 * e]), mul, neg_m));
            const float p1 = ex2_approx(fmaf(__uint_as_float(r[cc][2 * e + 1]), mul, neg_m));
            acc[(2 * e) & 7] += p0;
            acc[(2 * e + 1) & 7] += p1;
            pk[e] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tS + cc * 16, pk);
        }
        l_run += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[u & 1]));
      }
      // ---------------------------------------------------------- epilogue
      bool have_o = live && u == n_t;
      if (have_o)
        have_o = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->pv_done), (n_t - 1) & 1, wc));
      tc_fence_after_sync();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const long long grow_row = row0 + row;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        if (have_o) {  // warp-uniform
          tmem_ld32(tO + cc * 32, o);
          tmem_wait_ld();
          reg_fence32(o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (!valid_row) continue;
        if (direct) {
          uint4* orow = reinterpret_cast<uint4*>(a.out.o + grow_row * D + cc * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
            orow[e] = w;
          }
        } else {
          float4* orow = reinterpret_cast<float4*>(
              a.out.part_o + ((size_t)c * a.rows_total + grow_row) * D + cc * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            orow[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                  __uint_as_float(o[4 * e + 2]) * inv,
                                  __uint_as_float(o[4 * e + 3]) * inv);
        }
      }
      if (valid_row) {
        const float l2 = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
        if (direct) a.out.lse[grow_row] = l2 * 0.69314718055994531f;
        else a.out.part_lse[(size_t)c * a.rows_total + grow_row] = l2;
      }
    }
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// One warp per output row: merge the partial results of the chunks that hold keys of
// the row, in chunk order.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const Args a) {
  const DecodeProblem& p = a.p;
  const long long grow = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (grow >= a.rows_total) return;
  const int b = (int)(grow / ((long long)p.Hq * p.Nq));
  const int i = (int)(grow % p.Nq);
  int Lb = p.seq_lens[b];
  Lb = Lb < 0 ? 0 : (Lb > p.max_seq_len ? p.max_seq_len : Lb);
  int lo, hi;
  decode_row_keys(p.mask_kind, p.window, Lb, p.Nq, i, lo, hi);
  constexpr int kPer = D / 32;  // columns per lane
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  float M = -INFINITY, W = 0.f;
  if (hi > lo) {
    const int ca = lo / p.chunk, cb = (hi - 1) / p.chunk + 1;
    for (int cc = ca + lane; cc < cb; cc += 32)
      M = fmaxf(M, a.out.part_lse[(size_t)cc * a.rows_total + grow]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (M > -INFINITY) {
      for (int cc = ca; cc < cb; ++cc) {
        const float w = ex2_approx(a.out.part_lse[(size_t)cc * a.rows_total + grow] - M);
        W += w;
        const float* src = a.out.part_o + ((size_t)cc * a.rows_total + grow) * D + lane * kPer;
        if constexpr (kPer == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          acc[0] = fmaf(w, v.x, acc[0]);
          acc[1] = fmaf(w, v.y, acc[1]);
          acc[2] = fmaf(w, v.z, acc[2]);
          acc[3] = fmaf(w, v.w, acc[3]);
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          acc[0] = fmaf(w, v.x, acc[0]);
          acc[1] = fmaf(w, v.y, acc[1]);
        }
      }
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  __nv_bfloat16* dst = a.out.o + grow * D + lane * kPer;
  if constexpr (kPer == 4) {
    uint2 w;
    w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0) a.out.lse[grow] = W > 0.f ? (M + log2f(W)) * 0.69314718055994531f : -INFINITY;
}

template <int D, bool kAlibi, bool kSoftcap>
cudaError_t launch_variant(const Args& a, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, dim3 grid, cudaStream_t st) {
  auto kern = decode_tc_kernel<D, kAlibi, kSoftcap>;
  const int smem = Layout<D>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const Args& a, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, dim3 grid, cudaStream_t st) {
  const bool al = a.p.score_kind & ATTN_SCORE_ALIBI, sc = a.p.score_kind & ATTN_SCORE_SOFTCAP;
  cudaError_t e;
  if (al && sc) e = launch_variant<D, true, true>(a, tq, tk, tv, grid, st);
  else if (al) e = launch_variant<D, true, false>(a, tq, tk, tv, grid, st);
  else if (sc) e = launch_variant<D, false, true>(a, tq, tk, tv, grid, st);
  else e = launch_variant<D, false, false>(a, tq, tk, tv, grid, st);
  if (e != cudaSuccess || a.p.n_chunks == 1) return e;
  const long long blocks = (a.rows_total + 7) / 8;
  decode_combine_kernel<D><<<(unsigned)blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeProblem& p, const CUtensorMap& tq, const CUtensorMap& tk,
                             const CUtensorMap& tv, const DecodeOut& out, cudaStream_t st) {
  Args a{};
  a.p = p;
  a.out = out;
  a.G = p.Hq / p.Hkv;
  a.rows = a.G * p.Nq;
  a.row_tiles = ceil_div(a.rows, BM);
  a.rows_total = (long long)p.B * p.Hq * p.Nq;
  const long long gy = (long long)p.B * p.Hkv * a.row_tiles;
  if (gy == 0 || p.n_chunks == 0) return cudaSuccess;
  if (gy > 65535 || (a.rows_total + 7) / 8 > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)p.n_chunks, (unsigned)gy);
  if (p.d == 64) return launch_d<64>(a, tq, tk, tv, grid, st);
  return launch_d<128>(a, tq, tk, tv, grid, st);
}

}  // namespace attn
