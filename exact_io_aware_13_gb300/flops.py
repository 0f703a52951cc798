"""Useful work of an attention problem: allowed (query, key) pairs and FLOPs.

Only allowed pairs count ("useful" FLOPs: masked-out and skipped work excluded).
Forward: 2 matmuls (Q K^T and P V) of 2*d flops per pair = 4*d. Backward:
5 matmuls (Q K^T recomputed, dO V^T, P^T dO, dS^T Q, dS K) = 10*d per pair.
"""
from __future__ import annotations

from typing import Optional, Sequence

MASK_NONE, MASK_CAUSAL, MASK_SLIDING_WINDOW, MASK_DOCUMENT_CAUSAL = 0, 1, 2, 3


def allowed_pairs(mask_kind: int, Nq: int, Nkv: int, window: int = 0,
                  doc_offsets: Optional[Sequence[int]] = None) -> int:
    """Allowed pairs of one head, in closed form."""
    if mask_kind == MASK_NONE:
        return Nq * Nkv
    if mask_kind == MASK_CAUSAL:
        # row i sees keys 0..min(i, Nkv-1)
        full = min(Nq, Nkv)
        return full * (full + 1) // 2 + max(0, Nq - Nkv) * Nkv
    if mask_kind == MASK_SLIDING_WINDOW:
        total = 0
        w = max(window, 0)
        for i in range(Nq):  # keys max(0, i-w+1) .. min(i, Nkv-1)
            lo, hi = max(0, i - w + 1), min(i, Nkv - 1)
            total += max(0, hi - lo + 1)
        return total
    if mask_kind == MASK_DOCUMENT_CAUSAL:
        offs = [int(x) for x in doc_offsets]
        return sum((b - a) * (b - a + 1) // 2 for a, b in zip(offs[:-1], offs[1:]))
    raise ValueError(mask_kind)


def allowed_pairs_rows(mask_kind: int, rows: Sequence[int], Nkv: int, window: int = 0,
                       doc_offsets: Optional[Sequence[int]] = None) -> int:
    """Allowed pairs of the given query rows of one head (row by row, closed form per row)."""
    offs = None if doc_offsets is None else [int(x) for x in doc_offsets]
    total = 0
    doc = 0
    for i in sorted(int(r) for r in rows):
        if mask_kind == MASK_NONE:
            total += Nkv
        elif mask_kind == MASK_CAUSAL:
            total += max(0, min(i, Nkv - 1) + 1)
        elif mask_kind == MASK_SLIDING_WINDOW:
            lo, hi = max(0, i - max(window, 0) + 1), min(i, Nkv - 1)
            total += max(0, hi - lo + 1)
        elif mask_kind == MASK_DOCUMENT_CAUSAL:
            while doc + 1 < len(offs) and offs[doc + 1] <= i:
                doc += 1
            if doc + 1 < len(offs) and offs[doc] <= i:
                total += i - offs[doc] + 1
        else:
            raise ValueError(mask_kind)
    return total


def attention_flops(B: int, Hq: int, d: int, pairs_per_head: int, backward: bool) -> float:
    per_pair = (10 if backward else 4) * d
    return float(B) * Hq * pairs_per_head * per_pair
