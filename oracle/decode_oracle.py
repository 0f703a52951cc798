"""Float64 CPU oracle for attention of new query tokens over a paged KV cache (decode).

TEST INFRASTRUCTURE ONLY, like ``attention_oracle``: only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import it; the
library never does, and nothing here is shared with the CUDA path.

"FlashAttention/es" ("Variantes y sucesores") names PagedAttention, which cuts the KV
cache of inference into fixed-size pages so that many sequences of different lengths
share one pool. What is computed here is the plain definition, with the cache
gathered back into contiguous keys first:

  * Cache layout (a reading; the pages fix none): k_cache and v_cache are
    [num_pages, Hkv, page_size, d]; token t of sequence b lives in page
    page_table[b, t // page_size] at slot t % page_size; sequence b holds
    seq_lens[b] tokens.
  * The Nq query tokens of sequence b are its newest tokens: query i sits at
    position pos_i = seq_lens[b] - Nq + i (a reading: they were appended to the cache
    before the call). Masks and ALiBi use these positions, so "causal" is aligned at
    the bottom right: key j is allowed iff j <= pos_i; the sliding window adds
    pos_i - j < W; no mask allows every cached key. Document masking does not apply.
  * Scores, score modifications (scale, ALiBi with the signed distance pos_i - j,
    soft-cap), row softmax, O and the natural-log LSE are those of
    ``attention_oracle`` (its docstring cites the pages); a row with no allowed key has
    O = 0 and LSE = -inf.

Pinned by tests/test_decode_oracle.py: gathering against direct per-token indexing,
full prefill (Nq = seq_len) against the top-left causal ``attention_oracle.forward``
of the contiguous keys, single and few-token decode against torch's float64
scaled_dot_product_attention with an explicit mask and ALiBi bias, the soft-cap
against a scalar loop, and the empty-row and one-key special cases.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from . import attention_oracle as ref

MASK_NONE = ref.MASK_NONE
MASK_CAUSAL = ref.MASK_CAUSAL
MASK_SLIDING_WINDOW = ref.MASK_SLIDING_WINDOW


def gather_sequence(cache, page_table_row, length: int) -> np.ndarray:
    """The first ``length`` tokens of one sequence from a paged cache, as float64
    [Hkv, length, d]."""
    cache = ref._f64(cache)
    ps = cache.shape[2]
    t = np.arange(int(length))
    pages = np.asarray(page_table_row, dtype=np.int64)[t // ps]
    return cache[pages, :, t % ps, :].transpose(1, 0, 2)  # [length, Hkv, d] -> [Hkv, length, d]


def query_positions(length: int, Nq: int) -> np.ndarray:
    """Positions of the Nq newest tokens of a sequence of ``length`` cached tokens."""
    return int(length) - int(Nq) + np.arange(int(Nq), dtype=np.int64)


def decode_forward(q, k_cache, v_cache, page_table, seq_lens, scale: float,
                   mask_kind: int = MASK_NONE, window: int = 0, score_kind: int = 0,
                   softcap: float = 0.0, heads: Optional[Sequence[tuple]] = None):
    """Attention of q [B, Hq, Nq, d] over each sequence's cached keys.

    Returns (O [B, Hq, Nq, d], LSE [B, Hq, Nq]) in float64; with ``heads`` (a list of
    (b, h)) only those heads are computed and the rest are NaN.
    """
    if mask_kind not in (MASK_NONE, MASK_CAUSAL, MASK_SLIDING_WINDOW):
        raise ValueError("decode supports no mask, causal and sliding window")
    q = ref._f64(q)
    B, Hq, Nq, d = q.shape
    kc = ref._f64(k_cache)
    vc = ref._f64(v_cache)
    G = Hq // kc.shape[1]
    table = np.asarray(page_table)
    lens = np.asarray(seq_lens, dtype=np.int64)
    out = np.full((B, Hq, Nq, d), np.nan)
    lse = np.full((B, Hq, Nq), np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    gathered = {}
    for b, h in todo:
        if b not in gathered:
            gathered[b] = (gather_sequence(kc, table[b], lens[b]),
                           gather_sequence(vc, table[b], lens[b]))
        K, V = gathered[b]
        g = h // G
        pos = query_positions(lens[b], Nq)
        cols = np.arange(int(lens[b]), dtype=np.int64)
        s = float(scale) * (q[b, h] @ K[g].T)                       # [Nq, L]
        if score_kind & ref.SCORE_ALIBI:
            s = s - ref.alibi_slope(h, Hq) * (pos[:, None] - cols[None, :]).astype(np.float64)
        if score_kind & ref.SCORE_SOFTCAP:
            s = softcap * np.tanh(s / softcap)
        ok = ref.allowed(mask_kind, pos, cols, window) if cols.size else \
            np.zeros((Nq, 0), dtype=bool)
        s = np.where(ok, s, -np.inf)
        m = s.max(axis=1, initial=-np.inf)
        live = np.isfinite(m)
        e = np.exp(s - np.where(live, m, 0.0)[:, None])
        l = e.sum(axis=1)
        p = np.where(live[:, None], e / np.where(live, l, 1.0)[:, None], 0.0)
        out[b, h] = p @ V[g]
        lse[b, h] = np.where(live, m + np.log(np.where(live, l, 1.0)), -np.inf)
    return out, lse


def kv_bytes(seq_lens, Hkv: int, d: int) -> int:
    """Bytes of bf16 K and V a decode step must read: every cached token once."""
    return int(np.asarray(seq_lens, dtype=np.int64).sum()) * Hkv * d * 2 * 2
