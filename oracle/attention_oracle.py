"""Float64 CPU oracle for exact attention with score and mask modifications.

TEST INFRASTRUCTURE ONLY. This module is the plain, slow, materialising definition
of what the CUDA kernels compute. Only the tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it. The library under
``exact_io_aware_13_gb300`` never imports it and shares no code with it; both sides
take their seeded inputs from ``workloads``.

What is computed, per batch b and query head h (kv head g = floor(h / G),
G = Hq / Hkv), in float64 from the bf16-rounded inputs:

  1. S = scale * Q_h K_g^T, the whole score matrix materialised ("FlashAttention/es",
     section "Por qué la atención estándar es lenta": the naive method builds S and
     P of size N x N).
  2. Score modifications, in this order ("El FlexAttention de PyTorch con
     FlashAttention-4 es un cambio radical", first section, lists ALiBi and
     soft-capping among the supported variants):
       ALiBi:     s_ij <- s_ij - slope_h * (i - j),  slope_h = 2^(-8 (h+1) / Hq)
       soft-cap:  s_ij <- c * tanh(s_ij / c)
  3. Mask modification (same page and section: causal, sliding window and document
     masking): s_ij <- -inf where (i, j) is not allowed.
  4. Row softmax and output ("FlashAttention/es", sections "Por qué la atención
     estándar es lenta" and "El truco del softmax en línea"):
       m_i = max_j s_ij, l_i = sum_j exp(s_ij - m_i), P = exp(s - m) / l, O = P V_g.
  5. Log-sum-exp saved for the backward pass ("FlashAttention/es", section "El
     algoritmo FlashAttention", last step): L_i = m_i + log l_i (natural log).
     A row with no allowed key has O_i = 0 and L_i = -inf.
  6. Backward for the loss sum(dO * O) ("FlashAttention/es", section "Paso hacia
     atrás y recomputación", says P is rebuilt from L; the gradient algebra itself
     is the standard chain rule through softmax, written out here):
       dV_g = sum_{h in g} P^T dO_h
       dP   = dO_h V_g^T
       D_i  = sum_j P_ij dP_ij
       dS   = P * (dP - D)                (gradient w.r.t. the modified score)
       dS  <- dS * (1 - tanh^2(s_pre / c)) under soft-cap (s_pre: score before cap)
       dQ_h = scale * dS K_g
       dK_g = scale * sum_{h in g} dS^T Q_h
     ALiBi adds a constant, so it passes the gradient through unchanged.

  7. Dropout ("FlashAttention/es", "Variantes y sucesores": FlashAttention-1 supported
     dropout), when dropout_p > 0: with the keep mask Z of ``philox.keep_mask`` (its
     docstring states the generator and the counter layout),
       O = (P * Z / (1 - p)) V,  L unchanged (the softmax is taken before dropout);
     and in the backward, with dP' = (dO V^T) * Z / (1 - p),
       dV = (P * Z / (1 - p))^T dO,  D_i = sum_j P_ij dP'_ij = rowsum(dO * O),
       dS = P * (dP' - D).

Readings where the pages are silent:
  * GQA maps query head h to kv head floor(h / G).
  * ALiBi uses the 0-based query-head index and the signed distance (i - j).
  * Causal means j <= i on absolute positions (top-left aligned) even if Nq != Nkv.
  * The sliding window counts the diagonal: allowed iff j <= i and i - j < W.
  * Document masking is document-causal: same document and j <= i.

Every function here is pinned by tests/test_oracle.py against closed forms,
invariants, a library routine (torch's float64 scaled_dot_product_attention and
autograd) and central finite differences; no part is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

from . import philox

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_SLIDING_WINDOW = 2
MASK_DOCUMENT_CAUSAL = 3

SCORE_ALIBI = 1
SCORE_SOFTCAP = 2

TILE_EMPTY = 0
TILE_PARTIAL = 1
TILE_FULL = 2


def _f64(x) -> np.ndarray:
    """Widen a tensor or array (bf16 tensors included) to a float64 ndarray."""
    if hasattr(x, "detach"):
        import torch  # the oracle accepts torch CPU tensors as plain containers
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def document_ids(doc_offsets: Sequence[int], n: int) -> np.ndarray:
    """doc_id[t] = index of the document that holds position t (offsets: start of
    each document plus the end)."""
    ids = np.full(n, -1, dtype=np.int64)
    offs = [int(x) for x in doc_offsets]
    for doc in range(len(offs) - 1):
        ids[offs[doc]:offs[doc + 1]] = doc
    return ids


def allowed(mask_kind: int, rows: np.ndarray, cols: np.ndarray, window: int = 0,
            doc_offsets: Optional[Sequence[int]] = None, n_total: int = 0) -> np.ndarray:
    """Boolean matrix allowed[r, c] for query positions ``rows`` and key positions
    ``cols`` (the mask modification's predicate)."""
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.asarray(cols, dtype=np.int64)[None, :]
    if mask_kind == MASK_NONE:
        return np.ones((i.shape[0], j.shape[1]), dtype=bool)
    if mask_kind == MASK_CAUSAL:
        return j <= i
    if mask_kind == MASK_SLIDING_WINDOW:
        return (j <= i) & (i - j < window)
    if mask_kind == MASK_DOCUMENT_CAUSAL:
        n = max(n_total, int(i.max(initial=0)) + 1, int(j.max(initial=0)) + 1)
        ids = document_ids(doc_offsets, n)
        return (ids[i] == ids[j]) & (ids[i] >= 0) & (j <= i)
    raise ValueError(f"unknown mask kind {mask_kind}")


def alibi_slope(h: int, Hq: int) -> float:
    """ALiBi slope of query head h: 2^(-8 (h+1) / Hq)."""
    return 2.0 ** (-8.0 * (h + 1) / Hq)


def modified_scores(q_h, k_g, scale: float, h: int, Hq: int, score_kind: int,
                    softcap: float, rows: np.ndarray, cols: np.ndarray):
    """Return (s_pre_cap, s) for the given query rows and key columns, before
    masking. s_pre_cap is the score after scaling and ALiBi; s adds the soft-cap."""
    s = float(scale) * (q_h[rows] @ k_g[cols].T)
    if score_kind & SCORE_ALIBI:
        dist = rows[:, None].astype(np.float64) - cols[None, :].astype(np.float64)
        s = s - alibi_slope(h, Hq) * dist
    s_pre = s
    if score_kind & SCORE_SOFTCAP:
        s = softcap * np.tanh(s_pre / softcap)
    return s_pre, s


def _head_probs(q_h, k_g, scale, h, Hq, mask_kind, window, doc_offsets, score_kind,
                softcap, rows):
    """P (rows x Nkv), the masked scores, s_pre, row max m and row sum l."""
    nkv = k_g.shape[0]
    cols = np.arange(nkv)
    s_pre, s = modified_scores(q_h, k_g, scale, h, Hq, score_kind, softcap, rows, cols)
    ok = allowed(mask_kind, rows, cols, window, doc_offsets, max(q_h.shape[0], nkv))
    s = np.where(ok, s, -np.inf)
    m = s.max(axis=1)
    live = np.isfinite(m)
    m_safe = np.where(live, m, 0.0)
    e = np.exp(s - m_safe[:, None])          # exp(-inf) = 0 for masked entries
    l = e.sum(axis=1)
    p = np.where(live[:, None], e / np.where(live, l, 1.0)[:, None], 0.0)
    return p, s, s_pre, m, l, live


def forward(q, k, v, scale: float, mask_kind: int = MASK_NONE, window: int = 0,
            doc_offsets=None, score_kind: int = 0, softcap: float = 0.0,
            rows: Optional[np.ndarray] = None, heads: Optional[Sequence[tuple]] = None,
            dropout_p: float = 0.0, dropout_seed: int = 0):
    """Exact attention forward.

    q: [B, Hq, Nq, d], k/v: [B, Hkv, Nkv, d] (any float type; widened to float64).
    Returns (O [B, Hq, R, d] float64, L [B, Hq, R] float64) where R = len(rows)
    (all rows by default). ``heads`` restricts the work to a list of (b, h) pairs;
    the other heads are left as NaN.
    """
    q = _f64(q); k = _f64(k); v = _f64(v)
    B, Hq, Nq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    rows = np.arange(Nq) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.full((B, Hq, len(rows), d), np.nan)
    lse = np.full((B, Hq, len(rows)), np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in todo:
        g = h // G
        p, s, _, m, l, live = _head_probs(q[b, h], k[b, g], scale, h, Hq, mask_kind, window,
                                          doc_offsets, score_kind, softcap, rows)
        if dropout_p > 0:
            keep = philox.keep_mask(dropout_seed, b * Hq + h, rows, np.arange(k.shape[2]),
                                    dropout_p)
            p = p * keep / (1.0 - dropout_p)
        out[b, h] = p @ v[b, g]
        lse[b, h] = np.where(live, m + np.log(np.where(live, l, 1.0)), -np.inf)
    return out, lse


def probabilities(q, k, scale, h_index: int = 0, b_index: int = 0, mask_kind=MASK_NONE,
                  window=0, doc_offsets=None, score_kind=0, softcap=0.0):
    """The attention matrix P of one (b, h), rows x Nkv (for invariant tests)."""
    q = _f64(q); k = _f64(k)
    Hq, Nq = q.shape[1], q.shape[2]
    G = Hq // k.shape[1]
    p, *_ = _head_probs(q[b_index, h_index], k[b_index, h_index // G], scale, h_index, Hq,
                        mask_kind, window, doc_offsets, score_kind, softcap, np.arange(Nq))
    return p


def backward(q, k, v, dout, scale: float, mask_kind: int = MASK_NONE, window: int = 0,
             doc_offsets=None, score_kind: int = 0, softcap: float = 0.0,
             kv_heads: Optional[Sequence[tuple]] = None, dropout_p: float = 0.0,
             dropout_seed: int = 0):
    """Analytic gradients of sum(dO * O) with respect to q, k, v (float64).

    Materialises P per head. ``kv_heads`` restricts the work to a list of (b, g)
    kv heads (and the query heads of their groups); other entries are NaN.
    Returns (dq, dk, dv) with the shapes of q, k, v.
    """
    q = _f64(q); k = _f64(k); v = _f64(v); dout = _f64(dout)
    B, Hq, Nq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    rows = np.arange(Nq)
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    todo = kv_heads if kv_heads is not None else [(b, g) for b in range(B) for g in range(Hkv)]
    for b, g in todo:
        dk_acc = np.zeros(k.shape[2:])
        dv_acc = np.zeros(v.shape[2:])
        for h in range(g * G, (g + 1) * G):
            p, s, s_pre, m, l, live = _head_probs(q[b, h], k[b, g], scale, h, Hq, mask_kind,
                                                  window, doc_offsets, score_kind, softcap,
                                                  rows)
            do_h = dout[b, h]
            dp = do_h @ v[b, g].T
            if dropout_p > 0:
                zs = philox.keep_mask(dropout_seed, b * Hq + h, rows, np.arange(k.shape[2]),
                                      dropout_p) / (1.0 - dropout_p)
                dv_acc += (p * zs).T @ do_h
                dp = dp * zs
            else:
                dv_acc += p.T @ do_h
            D = (p * dp).sum(axis=1)
            ds = p * (dp - D[:, None])
            if score_kind & SCORE_SOFTCAP:
                t = np.tanh(s_pre / softcap)
                ds = ds * (1.0 - t * t)
            dq[b, h] = scale * (ds @ k[b, g])
            dk_acc += scale * (ds.T @ q[b, h])
        dk[b, g] = dk_acc
        dv[b, g] = dv_acc
    return dq, dk, dv


def classify_tiles(mask_kind: int, Nq: int, Nkv: int, tile_q: int, tile_k: int,
                   window: int = 0, doc_offsets=None) -> np.ndarray:
    """Per (q-tile, kv-tile) class by brute force over every (i, j) in the tile:
    EMPTY if no pair is allowed, FULL if every pair (inside the sequence bounds) is
    allowed, PARTIAL otherwise. Tiles skipped block-sparsely are the EMPTY ones
    ("El FlexAttention de PyTorch con FlashAttention-4 es un cambio radical",
    section "Limitaciones actuales", names block sparsity)."""
    nqt = -(-Nq // tile_q)
    nkt = -(-Nkv // tile_k)
    out = np.zeros((nqt, nkt), dtype=np.int32)
    full = allowed(mask_kind, np.arange(Nq), np.arange(Nkv), window, doc_offsets,
                   max(Nq, Nkv))
    for r in range(nqt):
        for c in range(nkt):
            blk = full[r * tile_q:(r + 1) * tile_q, c * tile_k:(c + 1) * tile_k]
            if not blk.any():
                out[r, c] = TILE_EMPTY
            elif blk.all():
                out[r, c] = TILE_FULL
            else:
                out[r, c] = TILE_PARTIAL
    return out


def allowed_pairs(mask_kind: int, Nq: int, Nkv: int, window: int = 0, doc_offsets=None,
                  row_block: int = 4096) -> int:
    """Number of allowed (i, j) pairs of one head, counted by brute force in row
    blocks (each block is an exact count; their sum is the total)."""
    total = 0
    cols = np.arange(Nkv)
    for r0 in range(0, Nq, row_block):
        rows = np.arange(r0, min(Nq, r0 + row_block))
        total += int(allowed(mask_kind, rows, cols, window, doc_offsets,
                             max(Nq, Nkv)).sum())
    return total

