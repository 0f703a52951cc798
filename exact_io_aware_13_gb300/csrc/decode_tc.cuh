// Decode over a paged KV cache: the tcgen05 kernel and its launchers, shared by
// decode_tc.cu (no row copies, the combine kernel, the entry point) and
// decode_copies2.cu (two row copies).
//
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
// byte, so the kernel is built to keep HBM busy without gaps:
//   * work items are (sequence, kv head, 64-row query tile, key chunk); the G = Hq /
//     Hkv query heads of a kv head and their Nq tokens are packed into rows g * Nq + i,
//     so each K/V byte fetched serves the whole group;
//   * the kernel is persistent: one CTA per SM takes a contiguous range of the item
//     list (items ordered sequence, head, row tile, chunk; every warp derives the same
//     list from seq_lens), and streams the items' key tiles through one ring without a
//     pause between items;
//   * warp 7 streams K and V tiles of 64 keys through a 7-stage shared-memory ring with
//     TMA (128-byte swizzle), one box per page piece (page sizes below 64 take several
//     boxes per tile), reading the page table 32 entries at a time, one item ahead;
//   * the Q tile of a run of items with the same (sequence, head, row tile) lives in
//     one of two tensor-memory buffers (bf16 pairs), written by the epilogue warps one
//     item ahead, so S = Q K^T is a TMEM-operand MMA;
//   * warp 1 issues S = Q K^T (M = 128, N = 64) and O += P V from one elected thread,
//     with Q and P in tensor memory; it waits only on hardware named barriers (a
//     shared-memory access by the thread that issues MMAs stalls the tensor pipe), fed
//     by warp 3, which turns the TMA completions into barrier arrivals and clears the
//     unused V rows of a sequence's last tile;
//   * the item's rows sit in TMEM quadrants 0 and 2: rows 0-31 and 32-63, or, for at
//     most 32 rows (a decode step of a GQA group), two copies of rows 0-31 that split
//     each tile's 64 keys between them and exchange row maxima, so that two warps share
//     the softmax; warps 4 and 6 do the online softmax (one thread per row) and rescale
//     O in tensor memory when the max grows by more than 2^8; warps 0 and 2 write each
//     item's result from the other O buffer while the softmax goes on with the next.
// Tensor memory: S0 cols [0,64), S1 [64,128), O0 [128,128+d), O1 [128+d,128+2d), Q0 and
// Q1 (d/2 columns each) after them; the row max and sum of each O buffer are handed from
// the softmax to the epilogue warps in shared memory.
//
// The last tile of a sequence can end inside a page whose later slots hold no token
// (possibly NaN). S columns past the sequence are masked before the max; the V rows
// there are zeroed in shared memory by the loader before the P V product (0 * NaN
// would be NaN).
//
// Split mode (more than one chunk per sequence, or two row copies): each item writes,
// per row and copy, O_c / l_c in fp32 and L2_c = m_c + log2 l_c; the combine kernel forms
//   M = max_c L2_c, w_c = 2^(L2_c - M), O = sum_c w_c O_c / sum_c w_c,
//   L = (M + log2 sum_c w_c) ln 2,
// in a fixed chunk order (deterministic).

#pragma once

#include <climits>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace dec {


constexpr int BM = 128;      // MMA M (TMEM lanes)
constexpr int kItemRows = 64;  // packed query rows per item: TMEM quadrants 0 and 2
constexpr int BN = 64;       // keys per tile (MMA N of S, K of P V)
constexpr int kStages = 7;   // K/V ring depth
// A warp runs on SM sub-partition warp % 4, and a softmax or epilogue warp may only
// address the TMEM lanes of quadrant warp % 4. An item's rows live in quadrants 0 and 2
// (rows 0-31 and 32-63, or two copies of rows 0-31), so the softmax and epilogue warps
// run on sub-partitions 0 and 2, the MMA issuer alone on 1 (issuing an MMA holds its
// sub-partition for tens of cycles), the loader and relay on 3. Lanes of quadrants 1
// and 3 hold rows nobody reads.
constexpr int kMmaWarp = 1;
constexpr int kRelayWarp = 3;
constexpr int kLoadWarp = 7;
constexpr int kThreads = 256;
__device__ __forceinline__ bool is_softmax_warp(int w) { return w == 4 || w == 6; }
__device__ __forceinline__ bool is_epilogue_warp(int w) { return w == 0 || w == 2; }
// Named barriers (the MMA warp waits only on these):
//   kNbP + (u & 1)   P of tile u in TMEM: the n_part softmax warps + MMA warp
//   kNbQ + b         Q buffer b written to TMEM: the n_part epilogue warps + MMA warp
//   kNbKV + s        K and V of ring stage s landed: relay (32) + MMA (32)
constexpr uint32_t kNbP = 1;
constexpr uint32_t kNbQ = 3, kNbX = 5;  // kNbX: row-max exchange between the two row copies
constexpr uint32_t kNbKV = 6, kNbPairCount = 64;
constexpr uint32_t kNbXCount = 64;
static_assert(kNbKV + kStages - 1 <= 15, "named barrier IDs");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;           // 128-byte column blocks
  static constexpr int kKvHalf = BN * 128;         // 8 KB
  static constexpr int kRing = 0;
  static constexpr int kTileBytes = kHalves * kKvHalf;  // one K or V tile
  static constexpr int kStage = 2 * kTileBytes;          // K then V
  static constexpr int kBars = kRing + kStages * kStage;
  static constexpr int kXchg = kBars + 512;             // row maxima [2][2][32] floats
  static constexpr int kStats = kXchg + 2 * 2 * 32 * 4;  // m, l [O buffer][copy][lane][2]
  static constexpr int kBytes = kStats + 2 * 2 * 32 * 2 * 4;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 64, kColO = 128;  // O buffers at kColO + b * D
  static constexpr uint32_t kColQ = kColO + 2 * D;  // Q buffers (bf16 pairs) at kColQ + b * D / 2
};
static_assert(Layout<128>::kAlloc <= 232448, "shared memory");

struct Bars {
  uint64_t q_empty[2];     // Q buffer b no longer read by S MMAs (MMA commit)
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t empty[kStages];
  uint64_t s_full[2];
  uint64_t pv_done;
  uint64_t o_full[2];      // O buffer b holds an item's P V sums (MMA commit)
  uint64_t stats_full[2];  // its rows' m and l are in shared memory (softmax warps)
  uint64_t o_empty[2];     // its result has been written out (epilogue warps)
  uint64_t tail[kStages];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

struct Args {
  DecodeProblem p;
  DecodeOut out;
  int G, rows, row_tiles;
  int rep;               // copies of the rows in TMEM: 2 or 1
  int n_part;            // softmax / epilogue warps that take part: 1 (one copy of at most
                         // 32 rows: quadrant 0 only) or 2 (quadrants 0 and 2)
  long long rows_total;  // B * Hq * Nq
  bool direct;           // one chunk per sequence: results written in place, no combine
};


// ------------------------------------------------------------------ the item list
// Every warp walks the list itself (all lanes together); the functions below are pure
// functions of the arguments and seq_lens, so every warp sees the same items.
__device__ __forceinline__ int seq_len(const Args& a, int b) {
  const int L = __ldg(a.p.seq_lens + b);
  return L < 0 ? 0 : (L > a.p.max_seq_len ? a.p.max_seq_len : L);
}
__device__ __forceinline__ int chunks_of(const Args& a, int L) {
  return a.direct ? 1 : ceil_div(L, a.p.chunk);
}

struct Cursor {
  int b, hk, rt, c, nb, Lb;
};

struct Item {
  int b, hk, rt, c, Lb;
  int rows_here;
  int max_lo, min_hi;   // over the tile's valid rows: largest first key, smallest end
  int tb, n_t;          // first 64-key tile and tile count (0: no key for any row)
  bool live;            // processed: has tiles, or (single-chunk launch) owns its rows
};

__device__ __forceinline__ void advance(const Args& a, Cursor& cu) {
  if (++cu.c < cu.nb) return;
  cu.c = 0;
  if (++cu.rt < a.row_tiles) return;
  cu.rt = 0;
  if (++cu.hk < a.p.Hkv) return;
  cu.hk = 0;
  do {
    ++cu.b;
    if (cu.b >= a.p.B) return;
    cu.Lb = seq_len(a, cu.b);
    cu.nb = chunks_of(a, cu.Lb);
  } while (cu.nb == 0);
}

// The CTAs split the item list by key tiles, not by item count (items differ in size:
// the last chunk of a sequence is short). An item's cost is its tiles without the mask,
// and items are laid end to end in list order, so item i starts at tile position f_i;
// CTA k takes the items with S_k <= f_i < S_{k+1}, S_k = floor(total * k / CTAs) (the
// last CTA takes the rest, items without tiles included).
__device__ __forceinline__ int item_tiles(const Args& a, int L, int c) {
  const int c0 = a.direct ? 0 : c * a.p.chunk;
  const int c1 = a.direct ? L : imin(c0 + a.p.chunk, L);
  return ceil_div(c1 - c0, BN);  // c0 is a multiple of 64
}

// The cursor at this CTA's first item (b = B when it has none), that item's tile
// position, and the position where the next CTA's items start.
__device__ inline void cta_items(const Args& a, int lane, Cursor& cu, long long& pos,
                                 long long& end_pos) {
  const DecodeProblem& p = a.p;
  const long long blocks = (long long)p.Hkv * a.row_tiles;  // (kv head, row tile) per sequence
  long long total = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    const int L = b < p.B ? seq_len(a, b) : 0;
    long long t = (b < p.B && chunks_of(a, L) > 0) ? blocks * ceil_div(L, BN) : 0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    total += t;
  }
  const long long S = total * blockIdx.x / gridDim.x;
  end_pos = blockIdx.x + 1 == gridDim.x ? LLONG_MAX : total * (blockIdx.x + 1) / gridDim.x;
  cu = Cursor{p.B, 0, 0, 0, 0, 0};
  pos = S;
  if (S >= end_pos) return;
  long long base = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    const int L = b < p.B ? seq_len(a, b) : 0;
    const bool has = b < p.B && chunks_of(a, L) > 0;
    const long long t = has ? blocks * ceil_div(L, BN) : 0;
    long long incl = t;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    // sequence b holds an item at or after S: S lies inside its tiles, or it has only
    // items without tiles, all at position base_b >= S
    const bool cond = has && (base + incl > S || (t == 0 && base + incl - t >= S));
    const uint32_t m = __ballot_sync(0xffffffffu, cond);
    if (m) {
      const int l = __ffs(m) - 1;
      const long long bbase = base + __shfl_sync(0xffffffffu, incl - t, l);
      cu.b = b0 + l;
      cu.Lb = seq_len(a, cu.b);
      cu.nb = chunks_of(a, cu.Lb);
      const long long T = ceil_div(cu.Lb, BN);                     // tiles of one block
      const long long CT = a.direct ? (T > 0 ? T : 1) : p.chunk / BN;  // tiles of a full chunk
      long long rem = S - bbase, blk = 0, c = 0;
      if (rem > 0) {
        blk = rem / T;
        const long long off = rem - blk * T;
        c = (off + CT - 1) / CT;
        if (c >= cu.nb) { c = 0; ++blk; }
      }
      pos = bbase + blk * T + c * CT;
      if (blk >= blocks) {  // past this sequence's last item: the next sequence's first
        cu.hk = p.Hkv - 1; cu.rt = a.row_tiles - 1; cu.c = cu.nb - 1;
        advance(a, cu);
        pos = bbase + blocks * T;
      } else {
        cu.hk = (int)(blk / a.row_tiles);
        cu.rt = (int)(blk % a.row_tiles);
        cu.c = (int)c;
      }
      return;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
}


__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = imin(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}
__device__ __forceinline__ int warp_max(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = imax(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ inline Item make_item(const Args& a, const Cursor& cu, int lane) {
  const DecodeProblem& p = a.p;
  Item it;
  it.b = cu.b; it.hk = cu.hk; it.rt = cu.rt; it.c = cu.c; it.Lb = cu.Lb;
  it.rows_here = imin(kItemRows, a.rows - cu.rt * kItemRows);
  const int c0 = a.direct ? 0 : cu.c * p.chunk;
  const int c1 = a.direct ? cu.Lb : imin(c0 + p.chunk, cu.Lb);
  int mn_lo = 1 << 30, mx_hi = 0, mx_lo = 0, mn_hi = 1 << 30;
  for (int r = lane; r < it.rows_here; r += 32) {
    const int i = (cu.rt * kItemRows + r) % p.Nq;
    int lo, hi;
    decode_row_keys(p.mask_kind, p.window, cu.Lb, p.Nq, i, lo, hi);
    if (hi > lo) { mn_lo = imin(mn_lo, lo); mx_hi = imax(mx_hi, hi); }
    mx_lo = imax(mx_lo, lo);
    mn_hi = imin(mn_hi, hi);
  }
  mn_lo = warp_min(mn_lo); mx_hi = warp_max(mx_hi);
  it.max_lo = warp_max(mx_lo); it.min_hi = warp_min(mn_hi);
  const int k_lo = imax(c0, mn_lo), k_hi = imin(c1, mx_hi);
  it.tb = k_hi > k_lo ? k_lo / BN : 0;
  it.n_t = k_hi > k_lo ? ceil_div(k_hi, BN) - it.tb : 0;
  it.live = it.n_t > 0 || a.direct;
  return it;
}

// Walks this CTA's items that have key tiles (with kWithEmpty, only those without: the
// single-chunk launch writes their results up front), calling
// f(item, new_q, run, u0, next, next_new_q): new_q when its Q tile differs from the
// previous item's (run = index of that Q tile, in buffer run & 1), u0 = index of its
// first key tile in the CTA's tile sequence, next = the following item (next.live false
// at the end) and next_new_q whether it starts a new Q tile.
template <bool kWithEmpty = false, typename F>
__device__ __forceinline__ void for_each_item(const Args& a, int lane, F&& f) {
  long long pos, end_pos;
  Cursor cu;
  cta_items(a, lane, cu, pos, end_pos);
  int run = -1, pb = -1, phk = -1, prt = -1;
  int u = 0;
  Item held{};
  held.live = false;
  bool held_new_q = false;
  int held_run = 0, held_u = 0;
  for (;;) {
    Item it{};
    it.live = false;
    const bool more = cu.b < a.p.B && pos < end_pos;
    if (more) {
      it = make_item(a, cu, lane);
      pos += item_tiles(a, cu.Lb, cu.c);
      advance(a, cu);
      it.live = kWithEmpty ? (it.live && it.n_t == 0) : it.n_t > 0;
      if (!it.live) continue;
    }
    const bool next_new_q = it.live && (it.b != pb || it.hk != phk || it.rt != prt);
    if (held.live) f(held, held_new_q, held_run, held_u, it, next_new_q);
    if (!it.live) break;
    bool new_q = false;
    if (!kWithEmpty && (it.b != pb || it.hk != phk || it.rt != prt)) {
      new_q = true;
      ++run;
      pb = it.b; phk = it.hk; prt = it.rt;
    }
    held = it;
    held_new_q = new_q;
    held_run = run;
    held_u = u;
    u += it.n_t;
  }
}

// kRep: copies of the item's rows in TMEM (2 when they fit in one 32-row block, else 1).
template <int D, bool kAlibi, bool kSoftcap, int kRep>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const Args a) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBars);
  const DecodeProblem& p = a.p;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    // A length outside [0, max_seq_len] (the walk clamps it) is reported once per launch.
    if (blockIdx.x == 0)
      for (int b = 0; b < p.B; ++b) {
        const int L0 = __ldg(p.seq_lens + b);
        if (L0 < 0 || L0 > p.max_seq_len) { atomicOr(p.status, DEV_BAD_INPUT); break; }
      }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bars->q_empty[t]), 1);
      mbar_init(smem_u32(&bars->s_full[t]), 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars->k_full[s]), 1);
      mbar_init(smem_u32(&bars->v_full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
      mbar_init(smem_u32(&bars->tail[s]), 1);
    }
    mbar_init(smem_u32(&bars->pv_done), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bars->o_full[t]), 1);
      mbar_init(smem_u32(&bars->stats_full[t]), a.n_part);
      mbar_init(smem_u32(&bars->o_empty[t]), a.n_part);
    }
    mbar_init(smem_u32(&bars->mma_done), 1);
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
  WaitCtx wc{&bars->abort_flag, p.status};

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    const int ps = p.page_size;
    const int R = imin(ps, BN);       // rows per box (a piece of one page)
    const int pieces = BN / R;        // boxes per tile and tensor (<= 8)
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    bool live = true;
    int issued = 0;
    // First page-table window of the next item, fetched one item ahead (a dependent
    // global load at the start of every item would stall the ring).
    auto fetch_for = [&](const Item& it, int base) {
      const int idx = base + lane;
      return (it.live && idx < p.max_pages) ? __ldg(p.page_table + (size_t)it.b * p.max_pages + idx)
                                            : -1;
    };
    bool have_pre = false;
    int pre_cur = -1, pre_nxt = -1;
    for_each_item(a, lane, [&](const Item& it, bool, int, int u0, const Item& next, bool) {
      if (!live) return;
      int wbase = (it.tb * BN) / ps;  // page index held by lane 0 of `cur`
      int cur = have_pre ? pre_cur : fetch_for(it, wbase);
      int nxt = have_pre ? pre_nxt : fetch_for(it, wbase + 32);
      have_pre = next.live && next.n_t > 0;
      if (have_pre) {
        pre_cur = fetch_for(next, (next.tb * BN) / ps);
        pre_nxt = fetch_for(next, (next.tb * BN) / ps + 32);
      }
      for (int t = 0; t < it.n_t; ++t) {
        const int u = u0 + t;
        const int s = u % kStages;
        live = __all_sync(0xffffffffu,
                          mbar_wait(smem_u32(&bars->empty[s]), ((u / kStages) & 1) ^ 1, wc));
        if (!live) return;
        const int t0 = (it.tb + t) * BN;
        const int valid = imin(BN, it.Lb - t0);  // keys of the tile inside the sequence
        const int first_page = t0 / ps;
        while (first_page - wbase >= 32) {  // warp-uniform
          wbase += 32;
          cur = nxt;
          nxt = fetch_for(it, wbase + 32);
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
          const bool in_seq = lane < pieces && key < it.Lb;
          good = in_seq && page >= 0 && page < p.num_pages;
          if (in_seq && !good) atomicOr(p.status, DEV_BAD_INPUT);
          coord = (int)(((long long)page * p.Hkv + it.hk) * ps + key % ps);
        }
        const uint32_t mask = __ballot_sync(0xffffffffu, good);
        const uint32_t bytes = (uint32_t)__popc(mask) * R * 128 * L::kHalves;
        const bool tail = valid < BN;
        const uint32_t kst = smem_u32(smem + L::kRing + s * L::kStage);
        const uint32_t vst = kst + L::kTileBytes;
        const uint32_t kbar = smem_u32(&bars->k_full[s]);
        const uint32_t vbar = tail ? smem_u32(&bars->tail[s]) : smem_u32(&bars->v_full[s]);
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
      }
    });
    // Do not leave while copies into this CTA's shared memory are in flight.
    for (int u = imax(0, issued - kStages); u < issued; ++u) {
      drain_wait(smem_u32(&bars->k_full[u % kStages]), (u / kStages) & 1);
      drain_wait(smem_u32(&bars->v_full[u % kStages]), (u / kStages) & 1);
    }
  } else if (warp == kRelayWarp) {
    // ------------------------------------------------------------ relay
    // Once K and V of a stage have landed (and the unused V rows of a sequence's last
    // tile are cleared), arrive on the stage's named barrier for the MMA warp. After an
    // abort, rendezvous (bar.sync) instead, so every barrier phase still pairs.
    bool live = true;
    auto pass = [&](uint32_t bar, uint32_t parity, uint32_t id) {
      if (live) live = __all_sync(0xffffffffu, mbar_wait(bar, parity, wc));
      if (live) nb_arrive(id, kNbPairCount);
      else nb_sync(id, kNbPairCount);
    };
    uint32_t tail_parity = 0;  // bit s: phase parity of tail[s]
    for_each_item(a, lane, [&](const Item& it, bool, int, int u0, const Item&, bool) {
      for (int t = 0; t < it.n_t; ++t) {
        const int u = u0 + t, s = u % kStages;
        if (live)
          live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->k_full[s]), (u / kStages) & 1, wc));
        const int t0 = (it.tb + t) * BN;
        const int valid = imin(BN, it.Lb - t0);
        if (valid < BN) {
          // The last tile of a sequence ends inside a page: its V copy completed on
          // tail[s]. Clear V rows [valid, BN) of each 128-byte column block in place (a
          // swizzled row stays inside its own 128 bytes), then complete v_full[s]. Stage
          // s is reused only after v_full[s], so tail[s] is never two phases ahead.
          if (live)
            live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->tail[s]), (tail_parity >> s) & 1u, wc));
          tail_parity ^= 1u << s;
          if (live) {
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
        pass(smem_u32(&bars->v_full[s]), (u / kStages) & 1, kNbKV + s);
      }
    });
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // S(u) is issued before P V of tile u - 1, so the softmax of one tile overlaps the
    // score MMAs of the next. The warp touches no shared memory until its last MMA: if a
    // wait elsewhere gave up, it still walks the whole schedule (its operands are then
    // stale, and the launch reports the timeout), and it waits for its MMAs to finish
    // before tensor memory is released.
    constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false, false);
    constexpr uint32_t idO = idesc_bf16_f32(BM, D, false, true);
    const uint32_t ring = smem_u32(smem + L::kRing);
    const bool issuer = elect_one();
    const uint32_t p_count = 32u * (a.n_part + 1);
    bool prev = false, prev_first = false, prev_last = false;
    int prev_u = 0, prev_ob = 0, n_items = 0;
    auto pv = [&]() {  // O += P V of tile prev_u
      const int s = prev_u % kStages;
      nb_sync(kNbP + (prev_u & 1), p_count);
      tc_fence_after_sync();
      const uint32_t vb = ring + s * L::kStage + L::kTileBytes;
      const uint64_t dv = smem_desc_sw128(vb, L::kKvHalf, 1024);
      const uint32_t colS = (prev_u & 1) ? L::kColS1 : L::kColS0;
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk)  // 16 keys per instruction
        mma_ts_if(issuer, tmem + L::kColO + prev_ob * D, tmem + colS + kk * 8,
                  dv + ((kk * 16 * 128) >> 4), idO, (!prev_first || kk > 0) ? 1u : 0u);
      mma_commit_if(issuer, smem_u32(&bars->empty[s]));
      mma_commit_if(issuer, smem_u32(&bars->pv_done));
      if (prev_last) mma_commit_if(issuer, smem_u32(&bars->o_full[prev_ob]));
    };
    for_each_item(a, lane, [&](const Item& it, bool new_q, int run, int u0, const Item&, bool) {
      const int qb = run & 1;
      if (new_q) {
        nb_sync(kNbQ + qb, p_count);
        tc_fence_after_sync();
      }
      const uint32_t tq = tmem + L::kColQ + qb * (D / 2);
      for (int t = 0; t < it.n_t; ++t) {
        const int u = u0 + t, s = u % kStages;
        nb_sync(kNbKV + s, kNbPairCount);
        tc_fence_after_sync();
        const uint32_t kb = ring + s * L::kStage;
        const uint64_t dk = smem_desc_sw128(kb, 16, 1024);
        const uint32_t col = (u & 1) ? L::kColS1 : L::kColS0;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {  // 16 head dims per instruction; Q in TMEM
          const uint32_t offk = ((kk >> 2) * L::kKvHalf + (kk & 3) * 32) >> 4;
          mma_ts_if(issuer, tmem + col, tq + kk * 8, dk + offk, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit_if(issuer, smem_u32(&bars->s_full[u & 1]));
        // every S of the previous Q tile was issued before this one
        if (t == 0 && new_q && run >= 1) mma_commit_if(issuer, smem_u32(&bars->q_empty[qb ^ 1]));
        if (prev) pv();
        prev = true;
        prev_u = u;
        prev_ob = n_items & 1;
        prev_first = t == 0;
        prev_last = t == it.n_t - 1;
      }
      if (it.n_t > 0) ++n_items;
    });
    if (prev) pv();
    mma_commit_if(issuer, smem_u32(&bars->mma_done));
    drain_wait(smem_u32(&bars->mma_done), 0);
  } else if (is_softmax_warp(warp) && (warp & 3) / 2 < a.n_part) {
    // ------------------------------------------------------------ softmax warps
    // Without copies (kRep = 1) the warp of quadrant 2 j owns rows 32 j .. 32 j + 31 and
    // all 64 key columns of a tile. With two copies of rows 0-31 it owns key columns
    // [32 j, 32 j + 32); the copies exchange their row maxima each tile, so they share m;
    // each keeps its own sum l and its own O (the P V of its columns) and writes them
    // out as a separate partial result.
    const int quad = warp & 3, j = quad >> 1;
    const int rb = kRep == 1 ? j : 0, ci = kRep == 1 ? 0 : j;
    constexpr int kCh = 4 / kRep;              // 16-column chunks per warp
    static_assert(kRep == 1 || kRep == 2, "row copies");
    const int cbase = ci * 16 * kCh;           // first key column of this warp
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t p_count = 32u * (a.n_part + 1);
    float* xmax = reinterpret_cast<float*>(smem + L::kXchg);  // [2][2][32]
    // with the soft-cap c: the pre-cap score over c, then s2 = c log2(e) tanh of it
    const float k1 = kSoftcap ? p.scale / p.softcap : p.scale * kLog2e;
    const float capA = kSoftcap ? p.softcap * kLog2e : 0.f;
    const bool raw_ok = !kAlibi && !kSoftcap && k1 > 0.f;
    bool live = true;
    int items_with_tiles = 0;
    float* stats = reinterpret_cast<float*>(smem + L::kStats);  // [2][2][32][2]
    for_each_item(a, lane, [&](const Item& it, bool, int, int u0, const Item&, bool) {
      const int row = rb * 32 + lane;  // packed row of the item
      const bool active = rb * 32 < it.rows_here;  // warp-uniform
      const bool valid_row = row < it.rows_here;
      const int pr = it.rt * kItemRows + imin(row, it.rows_here - 1);
      const int g = pr / p.Nq, i = pr - g * p.Nq;
      const int h = it.hk * a.G + g;
      const int pos = it.Lb - p.Nq + i;
      int lo_r = 0, hi_r = 0;
      if (valid_row) decode_row_keys(p.mask_kind, p.window, it.Lb, p.Nq, i, lo_r, hi_r);
      const float slope = kAlibi ? alibi_slope(h, p.Hq) : 0.f;
      const float kb = kSoftcap ? slope / p.softcap : slope * kLog2e;
      const int k = items_with_tiles++;
      const int ob = k & 1;
      const uint32_t tO = tmem + lane_base + L::kColO + ob * D;
      float m_run = -INFINITY, l_run = 0.f;
      for (int t = 0; t < it.n_t; ++t) {
        const int u = u0 + t;
        const uint32_t tS = tmem + lane_base + ((u & 1) ? L::kColS1 : L::kColS0);
        if (live)
          live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[u & 1]), (u >> 1) & 1, wc));
        if (!live) {  // aborted: keep the barrier schedule with the MMA warp, do nothing else
          if (kRep > 1) nb_sync(kNbX, kNbXCount);
          nb_sync(kNbP + (u & 1), p_count);
          continue;
        }
        tc_fence_after_sync();
        bool warp_grow = false;
        float corr = 1.f;
        uint32_t r[kCh][16];
        const int t0 = (it.tb + t) * BN;
        const bool masked = !(t0 >= it.max_lo && t0 + BN <= it.min_hi);  // CTA-uniform
        const bool fast = raw_ok && !masked;
        float mt = -INFINITY;
        if (active) {
#pragma unroll
          for (int ch = 0; ch < kCh; ++ch) tmem_ld16(tS + cbase + ch * 16, r[ch]);
          tmem_wait_ld();
#pragma unroll
          for (int ch = 0; ch < kCh; ++ch) reg_fence16(r[ch]);
          float mx[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
          const int c_lo = lo_r - t0, c_hi = hi_r - t0;  // allowed columns [c_lo, c_hi)
          const float base = kAlibi ? (float)(t0 - pos) * kb : 0.f;
          if (fast) {  // warp-uniform: the branch stays outside the element loops
#pragma unroll
            for (int ch = 0; ch < kCh; ++ch)
#pragma unroll
              for (int e = 0; e < 16; ++e) mx[e & 7] = fmaxf(mx[e & 7], __uint_as_float(r[ch][e]));
          } else {
#pragma unroll
            for (int ch = 0; ch < kCh; ++ch)
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int col = cbase + ch * 16 + e;
                const float x = __uint_as_float(r[ch][e]);
                float s2 = kAlibi ? fmaf(x, k1, fmaf((float)col, kb, base)) : x * k1;
                if (kSoftcap) s2 = capA * tanh_approx(s2);
                if (masked) s2 = (col >= c_lo && col < c_hi) ? s2 : -INFINITY;
                mx[e & 7] = fmaxf(mx[e & 7], s2);
                r[ch][e] = __float_as_uint(s2);
              }
          }
          mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                     fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
          if (fast) mt *= k1;
        }
        if (kRep > 1) {  // the copies agree on the tile's row max
          xmax[((u & 1) * 2 + ci) * 32 + lane] = mt;
          nb_sync(kNbX, kNbXCount);
          mt = fmaxf(mt, xmax[((u & 1) * 2 + (ci ^ 1)) * 32 + lane]);
        }
        if (active) {
          const float m_new = fmaxf(m_run, mt);
          warp_grow = __any_sync(0xffffffffu, m_new > m_run + kRescaleLog2);
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
          // P of this warp's columns (bf16 pairs); the other columns of the tile get 0
          // so that the P V product over all 64 keys adds nothing for them here.
          const uint32_t zero8[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
          for (int ch = 0; ch < kCh; ++ch) {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float p0 = ex2_approx(fmaf(__uint_as_float(r[ch][2 * e]), mul, neg_m));
              const float p1 = ex2_approx(fmaf(__uint_as_float(r[ch][2 * e + 1]), mul, neg_m));
              acc[(2 * e) & 7] += p0;
              acc[(2 * e + 1) & 7] += p1;
              pk[e] = pack_bf16x2(p0, p1);
            }
            tmem_st8(tS + (cbase + ch * 16) / 2, pk);
          }
          if (kRep > 1)
            for (int z = 0; z < 4; ++z)  // the 16-key groups of the other copy
              if (z / kCh != ci) tmem_st8(tS + z * 8, zero8);
          l_run += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        }
        // P V of the previous tile has had the whole softmax above to finish; wait for it
        // here (every warp, every tile, so that the phase count of pv_done stays exact),
        // then rescale O if the max grew. P V of this tile starts after the arrival below.
        if (u >= 1) {
          if (live)
            live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->pv_done), (u - 1) & 1, wc));
          tc_fence_after_sync();
        }
        if (active && live && warp_grow && t >= 1) {  // O holds this item's earlier P V
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
        if (t == 0 && k >= 2) {  // O buffer ob: the result of item k - 2 has been written
          if (live)
            live = __all_sync(0xffffffffu,
                              mbar_wait(smem_u32(&bars->o_empty[ob]), ((k >> 1) - 1) & 1, wc));
          tc_fence_after_sync();
        }
        if (active) tmem_wait_st();
        tc_fence_before_sync();
        nb_arrive(kNbP + (u & 1), p_count);
      }
      // Row max and sum for the epilogue warps (the mbarrier arrival releases them).
      if (active)
        *reinterpret_cast<float2*>(stats + ((ob * 2 + j) * 32 + lane) * 2) = make_float2(m_run, l_run);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->stats_full[ob]));
    });
  } else if (is_epilogue_warp(warp) && (warp & 3) / 2 < a.n_part) {
    // ------------------------------------------------------------ Q tiles and results
    // Quadrant 2 j writes the result of its rows: rows 32 j .. without copies; with two
    // copies of rows 0-31, partial result j of the item's chunk. The same warps put each
    // run's Q rows into tensor memory (bf16 pairs, the A operand of S = Q K^T) one item
    // ahead: the MMA warp issues the last P V of an item only after the first S of the
    // next, so that Q must be in place before this item's result is awaited.
    const int quad = warp & 3, j = quad >> 1;
    const int rb = kRep == 1 ? j : 0, ci = kRep == 1 ? 0 : j;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t p_count = 32u * (a.n_part + 1);
    const float* stats = reinterpret_cast<const float*>(smem + L::kStats);
    const int row = rb * 32 + lane;
    bool live = true;
    auto grow_of = [&](const Item& it) {
      return ((long long)it.b * p.Hq + (long long)it.hk * a.G) * p.Nq +
             (long long)it.rt * kItemRows + row;
    };
    auto prep_q = [&](const Item& it, int run) {
      const int qb = run & 1;
      if (run >= 2 && live)  // the S MMAs of Q tile run - 2 have completed
        live = __all_sync(0xffffffffu,
                          mbar_wait(smem_u32(&bars->q_empty[qb]), ((run >> 1) - 1) & 1, wc));
      tc_fence_after_sync();
      const bool ok = live && row < it.rows_here;
      const uint4* src = reinterpret_cast<const uint4*>(p.q + grow_of(it) * D);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {  // 32 columns (64 values) per store
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint4 v = ok ? __ldg(src + c * 8 + e) : make_uint4(0, 0, 0, 0);
          w[4 * e] = v.x; w[4 * e + 1] = v.y; w[4 * e + 2] = v.z; w[4 * e + 3] = v.w;
        }
        tmem_st32(tmem + lane_base + L::kColQ + qb * (D / 2) + c * 32, w);
      }
      tmem_wait_st();
      tc_fence_before_sync();
      if (live) nb_arrive(kNbQ + qb, p_count);
      else nb_sync(kNbQ + qb, p_count);
    };
    // Items without any key (single-chunk launches only): O = 0, LSE = -inf.
    if (ci == 0)
      for_each_item<true>(a, lane, [&](const Item& it, bool, int, int, const Item&, bool) {
        if (row >= it.rows_here) return;
        const long long r = grow_of(it);
        uint4* orow = reinterpret_cast<uint4*>(a.out.o + r * D);
#pragma unroll
        for (int e = 0; e < D / 8; ++e) orow[e] = make_uint4(0, 0, 0, 0);
        a.out.lse[r] = -INFINITY;
      });
    int k = 0;
    for_each_item(a, lane, [&](const Item& it, bool new_q, int run, int, const Item& next,
                               bool next_new_q) {
      if (new_q && run == 0) prep_q(it, 0);
      if (next_new_q) prep_q(next, run + 1);
      const bool active = rb * 32 < it.rows_here;  // warp-uniform
      const bool valid_row = row < it.rows_here;
      const int ob = k & 1;
      if (live)
        live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->o_full[ob]), (k >> 1) & 1, wc));
      if (live)
        live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->stats_full[ob]), (k >> 1) & 1, wc));
      ++k;
      const bool have_o = live;
      tc_fence_after_sync();
      const uint32_t tO = tmem + lane_base + L::kColO + ob * D;
      if (active) {
        const float2 ml = have_o ? *reinterpret_cast<const float2*>(stats + ((ob * 2 + j) * 32 + lane) * 2)
                                 : make_float2(-INFINITY, 0.f);
        const float m_run = ml.x, l_run = ml.y;
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const long long grow_row = grow_of(it);
        const size_t part = ((size_t)it.c * a.rep + ci) * a.rows_total + grow_row;
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
          if (a.direct) {
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
            float4* orow = reinterpret_cast<float4*>(a.out.part_o + part * D + cc * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              orow[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                    __uint_as_float(o[4 * e + 2]) * inv,
                                    __uint_as_float(o[4 * e + 3]) * inv);
          }
        }
        if (valid_row) {
          const float l2 = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
          if (a.direct) a.out.lse[grow_row] = l2 * 0.69314718055994531f;
          else a.out.part_lse[part] = l2;
        }
      }
      // O buffer ob and its row statistics may take the next item's values
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->o_empty[ob]));
    });
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D, bool kAlibi, bool kSoftcap, int kRep>
cudaError_t launch_variant(const Args& a, const CUtensorMap& tk,
                           const CUtensorMap& tv, int grid, cudaStream_t st) {
  auto kern = decode_tc_kernel<D, kAlibi, kSoftcap, kRep>;
  const int smem = Layout<D>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(tk, tv, a);
  return cudaGetLastError();
}

template <int D, int kRep>
cudaError_t launch_d(const Args& a, const CUtensorMap& tk,
                     const CUtensorMap& tv, int grid, cudaStream_t st) {
  const bool al = a.p.score_kind & ATTN_SCORE_ALIBI, sc = a.p.score_kind & ATTN_SCORE_SOFTCAP;
  if (al && sc) return launch_variant<D, true, true, kRep>(a, tk, tv, grid, st);
  if (al) return launch_variant<D, true, false, kRep>(a, tk, tv, grid, st);
  if (sc) return launch_variant<D, false, true, kRep>(a, tk, tv, grid, st);
  return launch_variant<D, false, false, kRep>(a, tk, tv, grid, st);
}

// The decode kernel for kRep copies of the rows (every head dimension and score mod).
template <int kRep>
cudaError_t launch_decode_copies(const Args& a, const CUtensorMap& tk,
                                 const CUtensorMap& tv, int grid, cudaStream_t st) {
  if (a.p.d == 64) return launch_d<64, kRep>(a, tk, tv, grid, st);
  return launch_d<128, kRep>(a, tk, tv, grid, st);
}

// Defined in decode_copies2.cu (a translation unit of its own, compiled in parallel).
cudaError_t launch_decode_copies2(const Args& a, const CUtensorMap& tk,
                                  const CUtensorMap& tv, int grid, cudaStream_t st);

}  // namespace dec
}  // namespace attn
