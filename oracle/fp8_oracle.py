"""Float64 CPU oracle for the FP8 forward: e4m3 codes, block quantisation, and the
reference attention of the dequantised inputs with its error bound.

TEST INFRASTRUCTURE ONLY, like ``attention_oracle``: only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import it; the
library never does, and nothing here is shared with the CUDA path.

FP8 attention is named on the pages for FlashAttention-3 ("FlashAttention/es",
section "Variantes y sucesores"; "FlashAttention-3 y torch.compile", section 2, with
block quantisation). What is computed:

  * e4m3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities;
    exponent field 0 holds the subnormals m/8 * 2^-6; the largest finite value is
    1.75 * 2^8 = 448). Encoding rounds to the nearest representable value, ties to
    the even mantissa, and saturates finite values above 448 to 448.
  * Block quantisation: a block (128 rows of a head for Q and K, a whole head for V)
    gets the float32 scale s = amax / 448 (1 if the block is all zero) and each value
    the code e4m3(x / s), x / s a float32 division. V's codes are stored transposed,
    [d, keys], keys padded with zero codes to a multiple of 16.
  * Reference: ``attention_oracle.forward`` of the dequantised inputs code * s.
  * Error bound of the GPU result: P is rounded to e4m3 after a factor 2^7 for the
    P V product, so each probability carries a relative error of at most 2^-4 (normal
    range) or an absolute one of at most 2^-17 (subnormal range, after the factor);
    the GPU's row sum uses the unrounded P, hence, per output element,
      |O_ic - O_ref_ic| <= 2^-4 sum_j P_ij |V_jc| + 2^-17 sum_j |V_jc|
    over the row's allowed keys j, plus the bf16 rounding of O (2^-8 relative) and
    float32 arithmetic (covered by a 2^-6 relative margin on the first term: the fp32
    sums of up to 2^13 products err by at most 2^-11 of sum_j P_ij |V_jc|).
"""
from __future__ import annotations

import numpy as np

from . import attention_oracle as ref

E4M3_MAX = 448.0
ROWS_PER_TILE = 128


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of e4m3 codes (uint8). The NaN codes 0x7f, 0xff decode to NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def e4m3_encode(x) -> np.ndarray:
    """Codes of float values: round to nearest, ties to even, saturate at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    neg = np.signbit(x)
    # binade: floor(log2 a) exactly via frexp, clamped to the normal range [-6, 8];
    # the subnormals share the spacing 2^-9 of the lowest normal binade.
    _, ex = np.frexp(np.maximum(a, 2.0 ** -6))
    e = np.clip(ex - 1, -6, 8)
    spacing = np.ldexp(1.0, e - 3)
    val = np.rint(a / spacing) * spacing          # np.rint rounds half to even
    val = np.minimum(np.where(a >= E4M3_MAX, E4M3_MAX, val), E4M3_MAX)
    normal = val >= 2.0 ** -6
    _, ex2 = np.frexp(np.where(normal, val, 1.0))
    E = ex2 - 1
    mant = np.where(normal, (val / np.ldexp(1.0, E) - 1.0) * 8.0, 0.0)
    code_n = (E + 7) * 8 + mant
    code_s = val / 2.0 ** -9
    code = np.where(normal, code_n, code_s).astype(np.int64)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def block_scale(block: np.ndarray) -> np.float32:
    """s = amax / 448 in float32 (1 for an all-zero block)."""
    amax = np.float32(np.max(np.abs(block.astype(np.float32)))) if block.size else np.float32(0)
    return np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(E4M3_MAX))


def quantize_tiles(x) -> tuple[np.ndarray, np.ndarray]:
    """x [BH, N, d] (bf16 values) -> codes uint8 [BH, N, d], scales float32 [BH, ceil(N/128)]."""
    x = np.asarray(x, dtype=np.float32)
    BH, N, d = x.shape
    nt = -(-N // ROWS_PER_TILE)
    codes = np.zeros((BH, N, d), dtype=np.uint8)
    scales = np.zeros((BH, nt), dtype=np.float32)
    for bh in range(BH):
        for t in range(nt):
            blk = x[bh, t * ROWS_PER_TILE:(t + 1) * ROWS_PER_TILE]
            s = block_scale(blk)
            scales[bh, t] = s
            codes[bh, t * ROWS_PER_TILE:(t + 1) * ROWS_PER_TILE] = e4m3_encode(blk / s)
    return codes, scales


def v_row_bytes(N: int) -> int:
    return 0 if N <= 0 else -(-N // 16) * 16


def quantize_v_transposed(x) -> tuple[np.ndarray, np.ndarray]:
    """x [BH, N, d] -> codes uint8 [BH, d, v_row_bytes(N)] (transposed, zero padded),
    scales float32 [BH] (one per head)."""
    x = np.asarray(x, dtype=np.float32)
    BH, N, d = x.shape
    codes = np.zeros((BH, d, v_row_bytes(N)), dtype=np.uint8)
    scales = np.zeros((BH,), dtype=np.float32)
    for bh in range(BH):
        s = block_scale(x[bh])
        scales[bh] = s
        codes[bh, :, :N] = e4m3_encode(x[bh] / s).T
    return codes, scales


def dequantize_tiles(codes, scales) -> np.ndarray:
    """[BH, N, d] codes and [BH, ntiles] scales -> float64 values."""
    codes = np.asarray(codes)
    BH, N, d = codes.shape
    rows = np.repeat(np.asarray(scales, dtype=np.float64), ROWS_PER_TILE, axis=1)[:, :N]
    return e4m3_decode(codes) * rows[:, :, None]


def dequantize_v_transposed(codes, scales, N: int) -> np.ndarray:
    """[BH, d, npad] codes and [BH] scales -> float64 V [BH, N, d]."""
    v = e4m3_decode(np.asarray(codes)[:, :, :N]).transpose(0, 2, 1)
    return v * np.asarray(scales, dtype=np.float64)[:, None, None]


def forward_reference(q8, sq, k8, sk, v8t, sv, B, Hq, Hkv, Nq, Nkv, scale, **mods):
    """Attention (``attention_oracle.forward``) of the dequantised inputs, and those
    inputs: returns (O, L, (q, k, v)) with q [B,Hq,Nq,d], k, v [B,Hkv,Nkv,d] float64."""
    d = np.asarray(q8).shape[-1]
    q = dequantize_tiles(np.asarray(q8).reshape(B * Hq, Nq, d), sq).reshape(B, Hq, Nq, d)
    k = dequantize_tiles(np.asarray(k8).reshape(B * Hkv, Nkv, d), sk).reshape(B, Hkv, Nkv, d)
    v = dequantize_v_transposed(np.asarray(v8t).reshape(B * Hkv, d, -1), sv, Nkv)
    v = v.reshape(B, Hkv, Nkv, d)
    o, lse = ref.forward(q, k, v, scale, **mods)
    return o, lse, (q, k, v)


def output_error_bound(q, k, v, scale, b, h, rows=None, mask_kind=0, window=0,
                       doc_offsets=None, score_kind=0, softcap=0.0) -> np.ndarray:
    """Per-element bound on |O_gpu - O_ref| for head (b, h) (see the module docstring):
    [rows, d]. q, k, v are the dequantised float64 inputs."""
    Hq, Hkv, Nq = q.shape[1], k.shape[1], q.shape[2]
    g = h // (Hq // Hkv)
    rows = np.arange(Nq) if rows is None else np.asarray(rows, dtype=np.int64)
    P, *_ = ref._head_probs(np.asarray(q[b, h], dtype=np.float64),
                            np.asarray(k[b, g], dtype=np.float64), scale, h, Hq, mask_kind,
                            window, doc_offsets, score_kind, softcap, rows)  # normalised
    absv = np.abs(np.asarray(v[b, g], dtype=np.float64))
    allowed = P > 0
    term1 = (P @ absv) * (2.0 ** -4 * (1 + 2.0 ** -6))
    term2 = 2.0 ** -17 * (allowed.astype(np.float64) @ absv)
    return term1 + term2


def max_abs_rounding_bf16(o_ref) -> np.ndarray:
    """bf16 rounding allowance of an output element (2^-8 relative, plus a tiny floor)."""
    return 2.0 ** -8 * np.abs(o_ref) + 1e-6

