/*
 * attn.h - C ABI of libattn.so: exact, IO-aware tiled attention on GB300 (sm_103a).
 *
 * The operation is scaled-dot-product attention, O = softmax(Q K^T / sqrt(d)) V
 * ("FlashAttention/es", section "Por qué la atención estándar es lenta"), computed
 * exactly with the tiled online-softmax recurrence ("El truco del softmax en línea"
 * and "El algoritmo FlashAttention" on the same page) so that no N x N matrix ever
 * reaches device memory. The forward pass also writes the per-row log-sum-exp
 * L_i = m_i + log(l_i) (natural log) that the backward pass uses to rebuild P
 * ("Paso hacia atrás y recomputación", same page).
 *
 * Attention variants follow the FlexAttention list in "El FlexAttention de PyTorch
 * con FlashAttention-4 es un cambio radical" (first section): score modifications
 * ALiBi and tanh soft-capping, mask modifications causal, sliding window and
 * document masking; tiles in which the mask allows nothing are skipped.
 *
 * Conventions shared by every call:
 *   - Tensors are DEVICE pointers owned by the caller, contiguous, row-major:
 *       q, o, dout, dq : bf16 [B, Hq,  Nq,  d]   (d fastest)
 *       k, v, dk, dv   : bf16 [B, Hkv, Nkv, d]
 *       lse            : fp32 [B, Hq, Nq]
 *     Every tensor pointer must be 16-byte aligned (ATTN_ERR_ALIGN otherwise).
 *   - Query head h reads kv head h / (Hq / Hkv) (grouped-query attention).
 *   - d must be 64, 128 or 256 ("FlashAttention/es", "Limitaciones": head sizes up to
 *     about 256); the SIMT entry points, the FP8 forward and dropout take 64 and 128
 *     only. Hq must be a multiple of Hkv.
 *   - scale multiplies Q K^T (usually 1/sqrt(d)); it must be finite.
 *   - Scores are modified in the order: scale, ALiBi, soft-cap, mask.
 *       ALiBi:    s_ij -= slope_h * (i - j), slope_h = 2^(-8 (h+1) / Hq),
 *                 h the 0-based query head.
 *       soft-cap: s_ij  = c * tanh(s_ij / c), c = attn_score_params.softcap > 0.
 *   - Masks (i = query position, j = key position, both from 0):
 *       ATTN_MASK_NONE               every pair
 *       ATTN_MASK_CAUSAL             j <= i (top-left aligned, also when Nq != Nkv)
 *       ATTN_MASK_SLIDING_WINDOW     j <= i and i - j < window (window >= 0;
 *                                    window 0 masks every pair)
 *       ATTN_MASK_DOCUMENT_CAUSAL    doc(i) == doc(j) and j <= i, with documents
 *                                    given by int32 DEVICE offsets
 *                                    doc_offsets[0..n_docs]: doc_offsets[0] = 0,
 *                                    non-decreasing, doc_offsets[n_docs] = Nq = Nkv.
 *                                    The offsets are trusted (not read on the host);
 *                                    attn_check_doc_offsets checks a table, and the
 *                                    checked mode (ATTN_CHECKED, below) checks it in
 *                                    every call.
 *     A query row with no allowed key gets O = 0 and lse = -inf, and zero gradients.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). They allocate no device memory; the backward pass takes a
 *     caller-provided workspace. Results are deterministic: the same inputs give
 *     bitwise-identical outputs.
 *   - Errors are returned, never hidden: there is no fallback path. A call that
 *     returns an error launched nothing.
 *   - Sizes of 0 (B, heads, Nq or Nkv) are valid; Nkv = 0 gives masked rows.
 */
#ifndef EXACT_IO_AWARE_ATTN_H
#define EXACT_IO_AWARE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_ARG = 1,            /* null pointer, unknown kind, bad scale/window/softcap */
  ATTN_ERR_SHAPE = 2,          /* unsupported d (256 on the SIMT/FP8 paths), Hq % Hkv != 0, negative size,
                                  document mask with Nq != Nkv, size over 2^31 */
  ATTN_ERR_ALIGN = 3,          /* a tensor pointer is not 16-byte aligned */
  ATTN_ERR_ARCH = 4,           /* the current device is not compute capability 10.3 */
  ATTN_ERR_WORKSPACE = 5,      /* workspace NULL or smaller than attn_bwd_workspace_size */
  ATTN_ERR_LAUNCH = 6,         /* a CUDA runtime/driver call or a launch failed */
  ATTN_ERR_DEVICE_TIMEOUT = 7, /* a kernel's bounded wait expired (attn_device_status) */
  ATTN_ERR_DEVICE_INPUT = 8    /* a kernel met an out-of-range DEVICE input: a decode
                                  sequence length or page index (attn_device_status) */
} attn_status;

enum {
  ATTN_MASK_NONE = 0,
  ATTN_MASK_CAUSAL = 1,
  ATTN_MASK_SLIDING_WINDOW = 2,
  ATTN_MASK_DOCUMENT_CAUSAL = 3
};

/* Score modification flags (OR-able; ALiBi is applied before soft-cap). */
enum {
  ATTN_SCORE_NONE = 0,
  ATTN_SCORE_ALIBI = 1,
  ATTN_SCORE_SOFTCAP = 2,
  ATTN_SCORE_DROPOUT = 4   /* dropout on P (attn_fwd / attn_bwd, tensor-core path, d <= 128) */
};

/* Tile classes written by attn_classify_tiles. */
enum { ATTN_TILE_EMPTY = 0, ATTN_TILE_PARTIAL = 1, ATTN_TILE_FULL = 2 };

/* Side of the square tiles the kernels iterate over (query rows x key columns). */
#define ATTN_TILE 128

typedef struct {
  int32_t window;              /* ATTN_MASK_SLIDING_WINDOW: keys i-window+1 .. i */
  const int32_t* doc_offsets;  /* ATTN_MASK_DOCUMENT_CAUSAL: DEVICE int32[n_docs+1] */
  int32_t n_docs;
} attn_mask_params;

typedef struct {
  float softcap;               /* ATTN_SCORE_SOFTCAP: the cap c > 0 */
  float dropout_p;             /* ATTN_SCORE_DROPOUT: drop probability, 0 <= p < 1 */
  uint64_t dropout_seed;       /* ATTN_SCORE_DROPOUT: seed of the keep mask */
} attn_score_params;

/*
 * Dropout ("FlashAttention/es", "Variantes y sucesores": FlashAttention-1 supported
 * dropout). Element (i, j) of query head bh = b * Hq + h is kept iff byte j % 16 of
 * Philox4x32-10 (Salmon et al., SC 2011; 128-bit counter (j / 16, i, bh, 0), key = the
 * seed, low word first; byte k = bits 8 (k % 4) .. of word k / 4) is at least
 * floor(256 p) (capped at 255), so p is taken to 1/256; kept values are scaled by
 * 1 / (1 - p). The forward computes O = (P Z / (1 - p)) V with lse from the undropped
 * softmax; attn_bwd, given the same p and seed, regenerates Z: dV = (P Z / (1 - p))^T dO
 * and dS = P (dP Z / (1 - p) - D). Pass the same score_kind and score_params to both.
 */

/*
 * Forward pass ("FlashAttention/es", "El algoritmo FlashAttention"): writes
 * o = softmax(modified, masked scores) v and lse = m + log(l) per query row.
 * mask_params / score_params are HOST pointers and may be NULL when the kind
 * needs no parameter. Runs the tcgen05 tensor-core kernel.
 */
attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale,
                     int mask_kind, const attn_mask_params* mask_params,
                     int score_kind, const attn_score_params* score_params,
                     void* stream);

/*
 * Bytes of device workspace attn_bwd needs for these sizes (a multiple of 256): the
 * backward's per-query-row terms, computed by its first kernel. With
 * Nq128 = Nq rounded up to a multiple of 128 and R = B * Hq * Nq128, that is
 * 2 * round256(4 R) + round256(4 Nq128): L log2 e and D_i (one float each per padded
 * row) and each row's first allowed key (one int32 per padded row position).
 * 0 when B, Hq or Nq is 0.
 */
size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nkv, int d);

/*
 * Backward pass ("FlashAttention/es", "Paso hacia atrás y recomputación"): from
 * q, k, v, the forward's o and lse, and the output gradient dout, rebuilds P
 * tile by tile and writes dq, dk, dv (bf16, overwritten, not accumulated). The
 * gradient algebra is the standard one: dV = P^T dO, dP = dO V^T,
 * D_i = rowsum(dO o O), dS = P o (dP - D) (times the soft-cap derivative),
 * dQ = scale dS K, dK = scale dS^T Q, with dK and dV summed over the query heads
 * of a group. workspace: DEVICE memory of at least attn_bwd_workspace_size bytes,
 * 256-byte aligned, not shared with a concurrent call.
 */
attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv,
                     int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale,
                     int mask_kind, const attn_mask_params* mask_params,
                     int score_kind, const attn_score_params* score_params,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Kernels of the backward pass, for attn_bwd_phases. */
enum {
  ATTN_BWD_ROWDOT = 1,   /* row terms into the workspace: D = rowsum(dO o O), L log2 e,
                            first allowed key */
  ATTN_BWD_DKDV = 2,     /* dK and dV (reads the row terms) */
  ATTN_BWD_DQ = 4,       /* dQ (reads the row terms) */
  ATTN_BWD_ALL = 7
};

/*
 * attn_bwd split into its kernels: runs the ones named in `phases`, in the order
 * ROWDOT, DKDV, DQ, with attn_bwd's arguments and checks. DKDV and DQ read the row
 * terms from the workspace, so ROWDOT must have run on the same workspace and inputs before
 * them (in this call or an earlier one in stream order). DKDV and DQ do not depend
 * on each other: a caller may time them separately or put them on two streams.
 * attn_bwd(...) is attn_bwd_phases(ATTN_BWD_ALL, ...).
 */
attn_status attn_bwd_phases(int phases, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dout, void* dq,
                            void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                            float scale, int mask_kind, const attn_mask_params* mask_params,
                            int score_kind, const attn_score_params* score_params,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass that allocates nothing and takes no workspace argument.
 *
 * The method on the pages has no counterpart of this call; it exists for callers
 * that cannot call cudaMalloc (or any allocator) where they run the backward pass:
 * for example a host program whose device memory is already handed out in full to
 * another allocator, or a runtime that forbids new allocations once it has started.
 * Such a caller still owns and passes every input and output, exactly as for
 * attn_bwd; only the backward's scratch (the per-query-row terms that
 * attn_bwd_workspace_size counts) lives in a fixed array inside this library instead
 * of a caller workspace.
 *
 * - The array holds 3 * ATTN_STATIC_WORKSPACE_ROWS 4-byte words (24 MiB) on every
 *   device that loads the library, for the life of the process. B * Hq * Nq128 (Nq
 *   rounded up to a multiple of 128) must not exceed ATTN_STATIC_WORKSPACE_ROWS;
 *   larger problems return ATTN_ERR_WORKSPACE and launch nothing (use attn_bwd with a
 *   workspace for them).
 * - The first call on a device looks up the array's device address with that device
 *   current (a one-time set-up per device); make that first call before any stream
 *   capture on the device.
 * - Every call on a device shares the one array, and the array keeps whatever the
 *   last call left there (each call overwrites every row it uses before reading it).
 *   Calls whose kernels can overlap on the GPU (other streams, other host threads)
 *   race on the array: order them on one stream or synchronise between them.
 * - Arguments, results, determinism and errors are otherwise those of attn_bwd.
 */
#define ATTN_STATIC_WORKSPACE_ROWS (1 << 21)
attn_status attn_bwd_static_workspace(const void* q, const void* k, const void* v,
                                      const void* o, const float* lse, const void* dout,
                                      void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                                      int Nq, int Nkv, int d, float scale, int mask_kind,
                                      const attn_mask_params* mask_params, int score_kind,
                                      const attn_score_params* score_params, void* stream);

/*
 * FP8 forward with block scales ("FlashAttention/es", "Variantes y sucesores", and
 * "FlashAttention-3 y torch.compile", section 2, name FP8 inputs for FlashAttention-3).
 * The inputs are e4m3 codes plus fp32 dequantisation scales, as written by
 * attn_quantize_fp8:
 *   q8   e4m3 [B, Hq, Nq, 128],  q_scale [B*Hq, ceil(Nq/128)]  (one per 128-row tile)
 *   k8   e4m3 [B, Hkv, Nkv, 128], k_scale [B*Hkv, ceil(Nkv/128)]
 *   v8t  e4m3 [B, Hkv, 128, attn_fp8_v_row_bytes(Nkv)] (V transposed, keys contiguous,
 *        zero padded), v_scale [B*Hkv] (one per head)
 * so that Q = q8 * q_scale etc. The result is attention (same masks and score mods as
 * attn_fwd) of those dequantised inputs, with P rounded to e4m3 (after a factor 2^7)
 * for the P V product: per element |O_ic - O_exact_ic| <= 2^-4 sum_j P_ij |V_jc|
 * + 2^-17 sum_j |V_jc| (over the row's allowed keys), plus bf16 rounding of O; lse is
 * exact up to fp32 rounding. d must be 128.
 * o: bf16 [B, Hq, Nq, 128]; lse: fp32 [B, Hq, Nq]. All pointers are DEVICE memory,
 * tensors 16-byte aligned, scales 4-byte aligned. Allocates nothing.
 */
attn_status attn_fwd_fp8(const void* q8, const void* k8, const void* v8t, const float* q_scale,
                         const float* k_scale, const float* v_scale, void* o, float* lse,
                         int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale,
                         int mask_kind, const attn_mask_params* mask_params, int score_kind,
                         const attn_score_params* score_params, void* stream);

/* Layouts of attn_quantize_fp8. */
enum {
  ATTN_FP8_TILES = 0,          /* Q, K: out [BH, N, d], scales [BH, ceil(N/128)] */
  ATTN_FP8_V_TRANSPOSED = 1    /* V: out [BH, d, attn_fp8_v_row_bytes(N)], scales [BH] */
};

/* Row length in bytes of the transposed e4m3 V: Nkv rounded up to 16 (0 if Nkv <= 0). */
size_t attn_fp8_v_row_bytes(int Nkv);

/*
 * bf16 x [BH, N, d] (d = 64 or 128, DEVICE) to e4m3 codes and fp32 scales: each
 * block (a 128-row tile for ATTN_FP8_TILES, a whole head for ATTN_FP8_V_TRANSPOSED)
 * gets s = amax / 448 (1 for an all-zero block) and code = e4m3(x / s), an IEEE fp32
 * division rounded to nearest even. Deterministic. x and out 16-byte aligned.
 */
attn_status attn_quantize_fp8(const void* x, void* out, float* scales, int BH, int N, int d,
                              int layout, void* stream);

/*
 * Decode over a paged KV cache ("FlashAttention/es", "Variantes y sucesores", names
 * PagedAttention, which cuts the inference KV cache into fixed-size pages shared by
 * many sequences). One call attends the Nq newest query tokens of each of B sequences
 * to every cached token of that sequence.
 *
 *   q          bf16 [B, Hq, Nq, d]  query i of sequence b sits at position
 *                                   seq_lens[b] - Nq + i (its own K/V are already in
 *                                   the cache)
 *   k_cache,   bf16 [num_pages, Hkv, page_size, d]: page p, kv head g, slot s
 *   v_cache
 *   page_table int32 [B, max_pages_per_seq]: token t of sequence b is in page
 *              page_table[b][t / page_size], slot t % page_size
 *   seq_lens   int32 [B]: cached tokens per sequence, 0 <= seq_lens[b] <= max_seq_len
 *   o          bf16 [B, Hq, Nq, d];  lse fp32 [B, Hq, Nq] (natural log)
 * All pointers are DEVICE memory; tensors 16-byte aligned, page_table and seq_lens
 * 4-byte aligned. page_table and seq_lens are read on the device only; a length
 * outside [0, max_seq_len] or a page index outside [0, num_pages) for a token the call
 * reads makes attn_device_status report ATTN_ERR_DEVICE_INPUT (the results of that
 * call are then unspecified; nothing outside the given buffers is touched).
 *
 * Masks use the positions above (aligned at the bottom right): ATTN_MASK_NONE (every
 * cached token), ATTN_MASK_CAUSAL (j <= position of the query), ATTN_MASK_SLIDING_WINDOW
 * (also position - j < window). ALiBi uses the signed distance position - j; soft-cap as
 * in attn_fwd. Document masking is not accepted (ATTN_ERR_ARG). Slots of a page past
 * the end of its sequence are never part of a result, whatever they hold.
 *
 * page_size: 8, 16, 32 or a multiple of 64. max_seq_len (<= max_pages_per_seq *
 * page_size) bounds seq_lens. split_keys (a positive multiple of 64, see
 * attn_decode_split_keys) cuts each sequence into chunks of that many keys, computed by
 * separate CTAs and merged by their log-sum-exp; with a single chunk
 * (max_seq_len <= split_keys) and more than 32 rows per query group no merge runs and no
 * workspace is needed. workspace:
 * DEVICE memory of attn_decode_workspace_size bytes, 256-byte aligned, not shared with
 * a concurrent call. Deterministic for fixed split_keys. Allocates nothing.
 */
attn_status attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* page_table, const int32_t* seq_lens, void* o,
                              float* lse, int B, int Hq, int Hkv, int Nq, int d, int num_pages,
                              int page_size, int max_pages_per_seq, int max_seq_len,
                              int split_keys, float scale, int mask_kind,
                              const attn_mask_params* mask_params, int score_kind,
                              const attn_score_params* score_params, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Workspace bytes of attn_decode_paged. The kernel keeps c copies of the rows of a kv
 * head's query group (G * Nq rows, G = Hq / Hkv) so that the softmax of a few rows is
 * spread over the SM: c = 2 for up to 32 rows, else 1. With
 * n = ceil(max_seq_len / split_keys) * c partial results per row and R = B * Hq * Nq
 * rows: round256(4 n R) + round256(4 n R d) (each partial's log2-sum-exp and normalised
 * fp32 output) when n > 1 and max_seq_len > 0, else 0.
 */
size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Nq, int d, int max_seq_len,
                                  int split_keys);

/*
 * A split_keys for attn_decode_paged: about ten work items (key chunks of one kv head
 * and 64-row query tile) per SM over total_kv_tokens (the sum of seq_lens, or
 * B * max_seq_len when unknown), a multiple of 64 and at least 256. Pure function of its
 * arguments.
 */
int attn_decode_split_keys(int B, int Hq, int Hkv, int Nq, long long total_kv_tokens,
                           int num_sms);

/*
 * Block-sparsity classifier ("El FlexAttention de PyTorch con FlashAttention-4 es
 * un cambio radical", "Limitaciones actuales", names block sparsity): writes
 * classes[r * ceil(Nkv/128) + c] = EMPTY / PARTIAL / FULL for query tile r and key
 * tile c, with the same tile rule the forward and backward kernels use to skip
 * and to mask tiles. classes: DEVICE int32 [ceil(Nq/128) * ceil(Nkv/128)].
 */
attn_status attn_classify_tiles(int mask_kind, const attn_mask_params* mask_params,
                                int Nq, int Nkv, int32_t* classes, void* stream);

/*
 * Checks a document-offsets table on the device: doc_offsets[0] = 0, non-decreasing,
 * doc_offsets[n_docs] = N (the contract of ATTN_MASK_DOCUMENT_CAUSAL). A violation is
 * not returned here (the table is device memory and the call is asynchronous): it is
 * recorded in the device status word, which the next attn_device_status reports as
 * ATTN_ERR_DEVICE_INPUT. Reads doc_offsets[0 .. n_docs] only (DEVICE int32, 4-byte
 * aligned). Returns ATTN_ERR_ARG for a null pointer, n_docs < 1 or N < 0.
 *
 * Checked mode: when the environment variable ATTN_CHECKED holds a value other than
 * "" or "0" at the library's first look at it (once per process), every call with
 * ATTN_MASK_DOCUMENT_CAUSAL (attn_fwd, attn_bwd and their variants, attn_fwd_fp8,
 * attn_classify_tiles) first runs this check on its table, in stream order before its
 * own kernels. The kernels of a call still run on a bad table; they read and write
 * only inside their buffers whatever the offsets hold, but their results are then
 * meaningless. The mode is for debugging; by default the table is trusted.
 */
attn_status attn_check_doc_offsets(const int32_t* doc_offsets, int n_docs, int N,
                                   void* stream);

/*
 * Plain CUDA-core versions of the forward and backward passes (one thread per
 * row, fp32 arithmetic, no tensor cores). They exist to cross-check the tensor-core
 * kernels and are never chosen automatically. Same arguments and contract as
 * attn_fwd / attn_bwd (attn_bwd_simt needs the same workspace).
 */
attn_status attn_fwd_simt(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale,
                          int mask_kind, const attn_mask_params* mask_params,
                          int score_kind, const attn_score_params* score_params,
                          void* stream);
attn_status attn_bwd_simt(const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* dout, void* dq, void* dk, void* dv,
                          int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale,
                          int mask_kind, const attn_mask_params* mask_params,
                          int score_kind, const attn_score_params* score_params,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Self-test of the failure path every kernel shares: launches one warp whose wait on a
 * shared-memory barrier that nothing completes is the library's bounded wait. After the
 * wait limit (2 s of the device clock) it gives up and records ATTN_ERR_DEVICE_TIMEOUT
 * in the device status word, which attn_device_status then reports and clears; the
 * context stays usable. Asynchronous on `stream`. Returns ATTN_ERR_ARCH or
 * ATTN_ERR_LAUNCH if the kernel cannot be launched.
 */
attn_status attn_selftest_wait_timeout(void* stream);

/*
 * Synchronises `stream` and reports whether a kernel of this library on the
 * current device gave up a bounded wait since the last call (ATTN_ERR_DEVICE_TIMEOUT),
 * met an out-of-range device input (ATTN_ERR_DEVICE_INPUT), or whether the stream
 * itself failed (ATTN_ERR_LAUNCH). Clears the flags.
 */
attn_status attn_device_status(void* stream);

/* Static, human-readable text for a status code. */
const char* attn_strerror(attn_status status);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_IO_AWARE_ATTN_H */
