// Launch interfaces shared between the translation units of libattn.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mask.cuh"

namespace attn {

// Everything a kernel needs to know about one attention problem.
struct Problem {
  int B, Hq, Hkv, Nq, Nkv, d;
  float scale;        // multiplies Q K^T
  int score_kind;     // ATTN_SCORE_* flags
  float softcap;      // c of the soft-cap
  MaskSpec mask;      // mask kind and parameters (doc offsets in device memory)
  int* status;        // device status word (bounded waits write DEV_TIMEOUT)
  int nq_pad;         // Nq rounded up to a multiple of 128: row stride of the row terms
  // Dropout (score_kind & ATTN_SCORE_DROPOUT): element (i, j) of query head bh is kept
  // iff byte j % 16 of Philox4x32-10((j / 16, i, bh, 0), seed) >= drop_thr; kept values
  // are multiplied by drop_scale = 1 / (1 - p) (drop_keep = 1 - p; both 1 without
  // dropout). The backward's row term is D (1 - p).
  int drop_thr;
  float drop_scale;
  float drop_keep;
  uint32_t drop_seed_lo, drop_seed_hi;
};

// Per-query-row terms of the backward, computed once by the row kernel and read by
// the gradient kernels. Rows are padded per head to nq_pad, so that any 64-row chunk
// of a 128-row query tile lies inside the arrays (the dK/dV kernel copies them in
// 256-byte chunks); padding rows hold lse2 = +inf, delta = 0, first = INT_MAX.
//   lse2[bh * nq_pad + i]  = L_i log2(e)  (+inf for a row that sees no key)
//   delta[bh * nq_pad + i] = D_i = sum_c dO_ic O_ic
//   first[i]               = first key row i may see (the mask's lower bound)
struct RowTerms {
  float* lse2;
  float* delta;
  int* first;
};

// ALiBi slope of query head h: 2^(-8 (h+1) / Hq).
__host__ __device__ inline float alibi_slope(int h, int Hq) {
  return exp2f(-8.0f * (float)(h + 1) / (float)Hq);
}

// ---- CUDA-core (SIMT) kernels: cross-check path and shared backward helpers.
cudaError_t launch_fwd_simt(const Problem& p, const __nv_bfloat16* q, const __nv_bfloat16* k,
                            const __nv_bfloat16* v, __nv_bfloat16* o, float* lse,
                            cudaStream_t st);
cudaError_t launch_bwd_simt(const Problem& p, const __nv_bfloat16* q, const __nv_bfloat16* k,
                            const __nv_bfloat16* v, const float* lse, const __nv_bfloat16* dout,
                            const float* delta, __nv_bfloat16* dq, __nv_bfloat16* dk,
                            __nv_bfloat16* dv, cudaStream_t st);  // delta: RowTerms::delta
// The row terms above for every (padded) query row, from O, dO and the forward's L.
cudaError_t launch_bwd_rowdot(const Problem& p, const __nv_bfloat16* o,
                              const __nv_bfloat16* dout, const float* lse, const RowTerms& rt,
                              cudaStream_t st);
// O = 0 and lse = -inf for `rows` rows (the answer when there are no keys).
cudaError_t launch_fill_masked(long long rows, int d, __nv_bfloat16* o, float* lse,
                               cudaStream_t st);
cudaError_t launch_classify(const MaskSpec& m, int32_t* classes, cudaStream_t st);

// ---- tcgen05 tensor-core kernels.
cudaError_t launch_fwd_tc(const Problem& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, __nv_bfloat16* o, float* lse,
                          cudaStream_t st);
// Forward for head dimension 256: q [B*Hq, Nq, 256] bf16 (read by the softmax warps into
// tensor memory), tk, tv over [B*Hkv, Nkv, 256] with 64 x 64 boxes.
cudaError_t launch_fwd256_tc(const Problem& p, const __nv_bfloat16* q, const CUtensorMap& tk,
                             const CUtensorMap& tv, __nv_bfloat16* o, float* lse, cudaStream_t st);
// FP8 forward (d = 128): tq, tk over e4m3 Q, K [B*H, N, 128]; tvt over e4m3 V^T
// [B*Hkv, 128, Nkv rounded up to 16]; sq [B*Hq, ceil(Nq/128)], sk [B*Hkv, ceil(Nkv/128)],
// sv [B*Hkv] dequantisation scales (device).
cudaError_t launch_fwd_fp8_tc(const Problem& p, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tvt, const float* sq, const float* sk,
                              const float* sv, __nv_bfloat16* o, float* lse, cudaStream_t st);
// Quantisation to e4m3: tiles (one scale per 128 rows of [BH, N, d]) or, for V, one
// scale per head with the output transposed to [BH, d, ceil16(N)] (zero padded).
cudaError_t launch_quantize_tiles(const __nv_bfloat16* x, uint8_t* out, float* scales, int BH,
                                  int N, int d, cudaStream_t st);
cudaError_t launch_quantize_v_transposed(const __nv_bfloat16* x, uint8_t* out, float* scales,
                                         int BH, int N, int d, cudaStream_t st);

// Tensor maps of the backward: the 128-row V box (the tile a dK/dV CTA loads once) and
// 64-row boxes (the slices both kernels stream).
struct BwdMaps {
  CUtensorMap v128, q64, do64, k64, v64;
  CUtensorMap k128;   // head dimension <= 128: the K tile a dK/dV CTA loads once
  CUtensorMap q128;   // head dimension <= 128: the Q tile a dQ CTA loads once
  CUtensorMap do128;  // the dQ kernel's fixed dO tile
};
cudaError_t launch_bwd_tc(const Problem& p, const BwdMaps& maps, const RowTerms& rt,
                          const __nv_bfloat16* q, const __nv_bfloat16* dout,
                          const __nv_bfloat16* k, const __nv_bfloat16* v, __nv_bfloat16* dq,
                          __nv_bfloat16* dk, __nv_bfloat16* dv, bool run_dkdv, bool run_dq,
                          cudaStream_t st);
// Head dimension 256: dV, dK (two walks over the key tiles) and dQ.
cudaError_t launch_bwd256_tc(const Problem& p, const BwdMaps& maps, const RowTerms& rt,
                             const __nv_bfloat16* q, const __nv_bfloat16* dout,
                             const __nv_bfloat16* k, __nv_bfloat16* dq, __nv_bfloat16* dk,
                             __nv_bfloat16* dv, bool run_dkdv, bool run_dq, cudaStream_t st);

// ---- Paged decode.
// Keys [lo, hi) that query i of the Nq newest tokens of a sequence with L cached tokens
// may see: query i sits at position L - Nq + i; causal stops at that position, the
// sliding window also starts `window - 1` keys before it. hi == lo when none.
ATTN_HD void decode_row_keys(int mask_kind, int window, int L, int Nq, int i, int& lo, int& hi) {
  const int pos = L - Nq + i;
  lo = 0;
  hi = L;
  if (mask_kind != ATTN_MASK_NONE) hi = imin(L, pos + 1);
  if (mask_kind == ATTN_MASK_SLIDING_WINDOW) lo = window > pos ? 0 : pos - window + 1;
  if (hi < lo) hi = lo;
}

// Copies of an item's packed rows (G * Nq per kv head) that the decode kernel keeps in
// tensor memory, so that two warps on two SM sub-partitions share the softmax of at
// most 32 rows: 2 for up to 32 rows, else 1. Each copy of a chunk is a separate partial
// result.
ATTN_HD int decode_row_copies(int rows) { return rows <= 32 ? 2 : 1; }

struct DecodeProblem {
  int B, Hq, Hkv, Nq, d;
  int page_size, max_pages, num_pages;
  int max_seq_len;           // bound on seq_lens (<= max_pages * page_size)
  int chunk;                 // keys per split (a multiple of 64)
  int n_chunks;              // ceil(max_seq_len / chunk): grid x; 1 = no combine
  float scale, softcap;
  int score_kind, mask_kind, window;
  const int32_t* page_table;  // [B, max_pages] device
  const int32_t* seq_lens;    // [B] device
  const __nv_bfloat16* q;     // [B, Hq, Nq, d] device
  int* status;
};
struct DecodeOut {
  __nv_bfloat16* o;  // [B, Hq, Nq, d]
  float* lse;        // [B, Hq, Nq], natural log
  float* part_o;     // partials: [n_chunks * copies, B*Hq*Nq, d] fp32, O_c / l_c
  float* part_lse;   // partials: [n_chunks * copies, B*Hq*Nq], m_c + log2 l_c
};
// tk, tv: [pages*Hkv*page_size, d] bf16, box 64 x min(page_size, 64). Launches the
// persistent decode kernel on num_ctas CTAs (one per SM) and, unless there is one chunk
// and one row copy, the combine kernel.
cudaError_t launch_decode_tc(const DecodeProblem& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             const DecodeOut& out, int num_ctas, cudaStream_t st);

}  // namespace attn
