// Mask predicates and the block-sparsity tile rule shared by every kernel.
//
// The mask modifications are the FlexAttention ones named in "El FlexAttention de
// PyTorch con FlashAttention-4 es un cambio radical" (causal, sliding window,
// document masking). Every mask here allows, for query row i, one contiguous range
// of keys [first_key(i), i] (or all keys for NONE), and first_key is
// non-decreasing in i. So the keys a block of rows needs form one contiguous run of
// key tiles, and the rows a block of keys needs form one contiguous run of query
// tiles; nothing here has to be stored as a list.
#pragma once

#include <cstdint>

#include "attn.h"

#ifdef __CUDACC__
#define ATTN_HD __host__ __device__ __forceinline__
#else
#define ATTN_HD inline
#endif

namespace attn {

struct MaskSpec {
  int kind;               // ATTN_MASK_*
  int window;             // sliding window
  const int32_t* doc;     // document offsets [n_docs + 1] (device or host memory)
  int n_docs;
  int nq, nkv;            // sequence lengths
};

ATTN_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }
ATTN_HD int imin(int a, int b) { return a < b ? a : b; }
ATTN_HD int imax(int a, int b) { return a > b ? a : b; }

// Index of the document holding position t: the last doc with doc[idx] <= t.
ATTN_HD int doc_index(const MaskSpec& m, int t) {
  int lo = 0, hi = m.n_docs;  // answer in [0, n_docs - 1]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (m.doc[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}
ATTN_HD int doc_start(const MaskSpec& m, int t) { return m.doc[doc_index(m, t)]; }
ATTN_HD int doc_end(const MaskSpec& m, int t) { return m.doc[doc_index(m, t) + 1]; }

// Smallest key that query row i may see (keys below it are masked). For NONE the
// answer is 0 and there is no upper limit; the other masks also stop at key i.
ATTN_HD int first_key(const MaskSpec& m, int i) {
  switch (m.kind) {
    case ATTN_MASK_SLIDING_WINDOW: return i - m.window + 1;
    case ATTN_MASK_DOCUMENT_CAUSAL: return doc_start(m, i);
    default: return 0;
  }
}

// Per-element predicate, given the row's first_key (precomputed once per row).
ATTN_HD bool allowed(const MaskSpec& m, int i, int j, int row_first_key) {
  if (j >= m.nkv) return false;
  if (m.kind == ATTN_MASK_NONE) return true;
  return j <= i && j >= row_first_key;
}

struct TileRange { int lo, hi; };  // tiles [lo, hi)

// Key tiles (of `tile` keys) that query rows [r0, r0 + tile) meet. Every tile in
// the returned range holds at least one allowed pair.
ATTN_HD TileRange kv_tiles_for_rows(const MaskSpec& m, int r0, int tile) {
  TileRange t{0, 0};
  if (r0 >= m.nq || m.nkv <= 0) return t;
  const int r1 = imin(r0 + tile, m.nq) - 1;  // last valid row
  if (m.kind == ATTN_MASK_NONE) { t.hi = ceil_div(m.nkv, tile); return t; }
  if (m.kind == ATTN_MASK_SLIDING_WINDOW && m.window <= 0) return t;
  const int kmax = imin(r1, m.nkv - 1);
  const int kmin = imax(first_key(m, r0), 0);
  if (kmin > kmax) return t;
  t.lo = kmin / tile;
  t.hi = kmax / tile + 1;
  return t;
}

// Query tiles (of `tile` rows) that keys [k0, k0 + tile) meet.
ATTN_HD TileRange q_tiles_for_keys(const MaskSpec& m, int k0, int tile) {
  TileRange t{0, 0};
  if (k0 >= m.nkv || m.nq <= 0) return t;
  const int k1 = imin(k0 + tile, m.nkv) - 1;
  if (m.kind == ATTN_MASK_NONE) { t.hi = ceil_div(m.nq, tile); return t; }
  if (m.kind == ATTN_MASK_SLIDING_WINDOW && m.window <= 0) return t;
  int rmax;
  if (m.kind == ATTN_MASK_CAUSAL) rmax = m.nq - 1;
  else if (m.kind == ATTN_MASK_SLIDING_WINDOW) {
    const long long last = (long long)k1 + m.window - 1;  // last row that sees k1
    rmax = last < (long long)(m.nq - 1) ? (int)last : m.nq - 1;
  }
  else rmax = imin(doc_end(m, k1) - 1, m.nq - 1);
  const int rmin = k0;  // causal-type masks: row i >= key j
  if (rmin > rmax) return t;
  t.lo = rmin / tile;
  t.hi = rmax / tile + 1;
  return t;
}

// True if every pair (i, j) with i in rows [r0, r0+tile) and j in keys
// [k0, k0+tile), both clipped to the sequence lengths, is allowed.
ATTN_HD bool tile_full(const MaskSpec& m, int r0, int k0, int tile) {
  if (m.kind == ATTN_MASK_NONE) return true;
  const int r1 = imin(r0 + tile, m.nq) - 1;
  const int k1 = imin(k0 + tile, m.nkv) - 1;
  if (k1 > r0) return false;  // some key after some row
  // first_key is non-decreasing in i, so the last row is the tightest.
  return first_key(m, r1) <= k0;
}

// Whether the kernels must apply the per-element predicate on a non-empty tile:
// the tile is partial, or it runs past the last key (those columns hold no key).
ATTN_HD bool tile_needs_mask(const MaskSpec& m, int r0, int k0, int tile) {
  return k0 + tile > m.nkv || !tile_full(m, r0, k0, tile);
}

// Class of one (query tile, key tile) pair, the rule the kernels follow.
ATTN_HD int tile_class(const MaskSpec& m, int qt, int kt, int tile) {
  TileRange r = kv_tiles_for_rows(m, qt * tile, tile);
  if (kt < r.lo || kt >= r.hi) return ATTN_TILE_EMPTY;
  return tile_full(m, qt * tile, kt * tile, tile) ? ATTN_TILE_FULL : ATTN_TILE_PARTIAL;
}

}  // namespace attn
