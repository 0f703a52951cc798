// Host-only build of the kernels' mask and tile rules (csrc/mask.cuh) so that the
// tests can check them on the CPU against the oracle's brute force.
#include "mask.cuh"

using attn::MaskSpec;

static MaskSpec spec(int kind, int window, const int32_t* doc, int n_docs, int nq, int nkv) {
  MaskSpec m;
  m.kind = kind; m.window = window; m.doc = doc; m.n_docs = n_docs; m.nq = nq; m.nkv = nkv;
  return m;
}

extern "C" {

// classes[qt * nkt + kt] as the kernels see them.
void host_classify(int kind, int window, const int32_t* doc, int n_docs, int nq, int nkv,
                   int32_t* classes) {
  MaskSpec m = spec(kind, window, doc, n_docs, nq, nkv);
  const int nqt = attn::ceil_div(nq, ATTN_TILE), nkt = attn::ceil_div(nkv, ATTN_TILE);
  for (int r = 0; r < nqt; ++r)
    for (int c = 0; c < nkt; ++c) classes[r * nkt + c] = attn::tile_class(m, r, c, ATTN_TILE);
}

// allowed[i * nkv + j] from the per-element predicate the kernels apply.
void host_allowed(int kind, int window, const int32_t* doc, int n_docs, int nq, int nkv,
                  uint8_t* out) {
  MaskSpec m = spec(kind, window, doc, n_docs, nq, nkv);
  for (int i = 0; i < nq; ++i) {
    const int fk = attn::first_key(m, i);
    for (int j = 0; j < nkv; ++j) out[(size_t)i * nkv + j] = attn::allowed(m, i, j, fk) ? 1 : 0;
  }
}

// [lo, hi) key-tile range per query tile of `tile` rows, and query-tile range per key tile.
void host_ranges(int kind, int window, const int32_t* doc, int n_docs, int nq, int nkv, int tile,
                 int32_t* kv_lohi, int32_t* q_lohi, uint8_t* needs_mask) {
  MaskSpec m = spec(kind, window, doc, n_docs, nq, nkv);
  const int nqt = attn::ceil_div(nq, tile), nkt = attn::ceil_div(nkv, tile);
  for (int r = 0; r < nqt; ++r) {
    attn::TileRange t = attn::kv_tiles_for_rows(m, r * tile, tile);
    kv_lohi[2 * r] = t.lo; kv_lohi[2 * r + 1] = t.hi;
    for (int c = 0; c < nkt; ++c)
      needs_mask[r * nkt + c] = attn::tile_needs_mask(m, r * tile, c * tile, tile) ? 1 : 0;
  }
  for (int c = 0; c < nkt; ++c) {
    attn::TileRange t = attn::q_tiles_for_keys(m, c * tile, tile);
    q_lohi[2 * c] = t.lo; q_lohi[2 * c + 1] = t.hi;
  }
}

}  // extern "C"
