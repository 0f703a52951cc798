"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and lays out shapes. It holds none of the
attention arithmetic, so both the float64 oracle (``oracle/``) and the CUDA path
(``exact_io_aware_13_gb300``) can take their inputs from it without sharing any
part of the computation.

Workloads follow the LLM shapes on the pages: head dimension 128 from a 4096-wide
model with 32 heads and sequences of 8192 tokens ("FlashAttention-3 y
torch.compile", section 4 "Tutorial Práctico" and section 5 "Benchmarks"), plus the
FlexAttention variants named in "El FlexAttention de PyTorch con FlashAttention-4 es
un cambio radical" (ALiBi, sliding window, document masking, soft-capping).

Recipe (the same on every machine):
  * generator ``torch.Generator('cpu').manual_seed(seed)``;
  * ``randn`` in float32 for Q, K, V and then dO, in that order, each rounded to
    bfloat16 (round to nearest even) after drawing;
  * document lengths from ``numpy.random.default_rng(seed).integers(512, 4096,
    endpoint=True)``, drawn until their sum reaches N, the last one truncated.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

# Mask kinds and score-mod flags, numbered as in include/attn.h.
MASK_NONE = 0
MASK_CAUSAL = 1
MASK_SLIDING_WINDOW = 2
MASK_DOCUMENT_CAUSAL = 3

SCORE_NONE = 0
SCORE_ALIBI = 1
SCORE_SOFTCAP = 2

MASK_NAMES = {MASK_NONE: "none", MASK_CAUSAL: "causal",
              MASK_SLIDING_WINDOW: "window", MASK_DOCUMENT_CAUSAL: "document"}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nkv: int
    d: int
    mask_kind: int = MASK_NONE
    window: int = 0
    score_kind: int = SCORE_NONE
    softcap: float = 0.0
    backward: bool = False
    doc_min: int = 512
    doc_max: int = 4096
    dropout_p: float = 0.0
    dropout_seed: int = 0

    @property
    def scale(self) -> float:
        """1/sqrt(d), rounded to float32 (the value the kernels receive)."""
        return float(np.float32(1.0 / math.sqrt(self.d)))

    def describe(self) -> str:
        s = (f"{self.name}: B={self.B} Hq={self.Hq} Hkv={self.Hkv} Nq={self.Nq} "
             f"Nkv={self.Nkv} d={self.d} mask={MASK_NAMES[self.mask_kind]}")
        if self.mask_kind == MASK_SLIDING_WINDOW:
            s += f" W={self.window}"
        if self.score_kind & SCORE_ALIBI:
            s += " +alibi"
        if self.score_kind & SCORE_SOFTCAP:
            s += f" +softcap{self.softcap:g}"
        if self.dropout_p > 0:
            s += f" +dropout{self.dropout_p:g}"
        return s

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads, in this order; seed = position in the list.
TINY = Workload("tiny non-causal fwd", 0, B=1, Hq=2, Hkv=2, Nq=256, Nkv=256, d=64)
CAUSAL = Workload("causal fwd", 1, B=4, Hq=16, Hkv=16, Nq=8192, Nkv=8192, d=128,
                  mask_kind=MASK_CAUSAL)
GQA_WINDOW = Workload("GQA sliding-window fwd", 2, B=2, Hq=32, Hkv=8, Nq=16384,
                      Nkv=16384, d=128, mask_kind=MASK_SLIDING_WINDOW, window=1024)
DOCS = Workload("packed-document fwd with ALiBi and soft-cap", 3, B=1, Hq=16, Hkv=16,
                Nq=32768, Nkv=32768, d=128, mask_kind=MASK_DOCUMENT_CAUSAL,
                score_kind=SCORE_ALIBI | SCORE_SOFTCAP, softcap=50.0)
CAUSAL_FWD_BWD = Workload("causal fwd+bwd", 4, B=2, Hq=16, Hkv=16, Nq=8192, Nkv=8192,
                          d=128, mask_kind=MASK_CAUSAL, backward=True)

WORKLOADS = [TINY, CAUSAL, GQA_WINDOW, DOCS, CAUSAL_FWD_BWD]

# Dropout on P ("FlashAttention/es", "Variantes y sucesores"), at the rate usually
# trained with, on the causal fwd+bwd shapes; the seed has both 32-bit halves set.
CAUSAL_FWD_BWD_DROPOUT = CAUSAL_FWD_BWD.replace(name="causal fwd+bwd dropout 0.1", seed=7,
                                                dropout_p=0.1,
                                                dropout_seed=0x9E3779B97F4A7C15)

# Head dimension 256, the top of the range the pages give ("FlashAttention/es",
# "Limitaciones"): the causal workload's FLOPs at twice the head size, half the batch.
CAUSAL_D256 = Workload("causal fwd d=256", 6, B=2, Hq=16, Hkv=16, Nq=8192, Nkv=8192, d=256,
                       mask_kind=MASK_CAUSAL)
CAUSAL_D256_FWD_BWD = CAUSAL_D256.replace(name="causal fwd+bwd d=256", seed=8, backward=True)


def document_lengths(total: int, seed: int, lo: int = 512, hi: int = 4096) -> list[int]:
    """Draw document lengths uniformly from [lo, hi] until they cover ``total``.

    The last document is cut so that the lengths sum to exactly ``total``.
    """
    rng = np.random.default_rng(seed)
    lengths: list[int] = []
    covered = 0
    while covered < total:
        n = int(rng.integers(lo, hi, endpoint=True))
        n = min(n, total - covered)
        lengths.append(n)
        covered += n
    return lengths


def document_offsets(total: int, seed: int, lo: int = 512, hi: int = 4096) -> np.ndarray:
    """Start offsets of the packed documents plus the end: int32[n_docs + 1]."""
    lengths = document_lengths(total, seed, lo, hi)
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def offsets_from_lengths(lengths) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int32)


def make_inputs(w: Workload, *, with_dout: Optional[bool] = None):
    """Return bf16 CPU tensors q [B,Hq,Nq,d], k/v [B,Hkv,Nkv,d] and, for backward
    workloads, dO [B,Hq,Nq,d]; plus int32 document offsets (or None).

    Layout is [B, H, N, d] with d fastest.
    """
    g = torch.Generator("cpu").manual_seed(w.seed)
    q = torch.randn((w.B, w.Hq, w.Nq, w.d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((w.B, w.Hkv, w.Nkv, w.d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((w.B, w.Hkv, w.Nkv, w.d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    want_do = w.backward if with_dout is None else with_dout
    do = None
    if want_do:
        do = torch.randn((w.B, w.Hq, w.Nq, w.d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    offs = None
    if w.mask_kind == MASK_DOCUMENT_CAUSAL:
        offs = document_offsets(w.Nq, w.seed, w.doc_min, w.doc_max)
    return q, k, v, do, offs


def random_doc_offsets(total: int, seed: int, lo: int, hi: int) -> np.ndarray:
    """Offsets for a small packed sequence (test sizes), same drawing rule."""
    return document_offsets(total, seed, lo, hi)


# ---------------------------------------------------------------- paged decode
# Inference side of the pages: the KV cache is cut into fixed-size pages ("FlashAttention/es",
# "Variantes y sucesores", names PagedAttention's segmented KV cache for serving many
# sequences at once), and each step attends the newest Nq query tokens of every sequence
# to all of its cached keys. Shapes follow the GQA workload (Hq = 32, Hkv = 8, d = 128).
@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    Nq: int            # new query tokens per sequence (1 = one decode step)
    d: int
    len_min: int       # cached keys per sequence, drawn uniformly from [len_min, len_max]
    len_max: int
    page_size: int
    mask_kind: int = MASK_NONE
    window: int = 0
    score_kind: int = SCORE_NONE
    softcap: float = 0.0
    lengths: Optional[tuple] = None  # explicit lengths (override the draw)
    spare_pages: int = 3             # pool pages no sequence uses

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.d)))

    def replace(self, **kw) -> "DecodeWorkload":
        return dataclasses.replace(self, **kw)

    def describe(self) -> str:
        s = (f"{self.name}: B={self.B} Hq={self.Hq} Hkv={self.Hkv} Nq={self.Nq} d={self.d} "
             f"len=[{self.len_min},{self.len_max}] page={self.page_size} "
             f"mask={MASK_NAMES[self.mask_kind]}")
        if self.mask_kind == MASK_SLIDING_WINDOW:
            s += f" W={self.window}"
        if self.score_kind & SCORE_ALIBI:
            s += " +alibi"
        if self.score_kind & SCORE_SOFTCAP:
            s += f" +softcap{self.softcap:g}"
        return s


PAGED_DECODE = DecodeWorkload("paged decode", 5, B=64, Hq=32, Hkv=8, Nq=1, d=128,
                              len_min=512, len_max=8192, page_size=64)

_PAGE_BLOCK = 1024  # pages drawn per randn call (bounds the float32 temporaries)


def decode_lengths(w: DecodeWorkload) -> np.ndarray:
    if w.lengths is not None:
        return np.asarray(w.lengths, dtype=np.int32)
    rng = np.random.default_rng(w.seed)
    return rng.integers(w.len_min, w.len_max, size=w.B, endpoint=True).astype(np.int32)


def make_decode_inputs(w: DecodeWorkload, *, poison_unused: bool = False):
    """Seeded paged-decode inputs (CPU):

    q          bf16 [B, Hq, Nq, d]
    k_cache    bf16 [num_pages, Hkv, page_size, d]   (a page holds page_size tokens
    v_cache    bf16 [num_pages, Hkv, page_size, d]    of one sequence, per kv head)
    page_table int32 [B, max_pages]  (page of token t of sequence b: page_table[b, t // page_size];
                                      entries past the sequence hold -1)
    seq_lens   int32 [B]

    Recipe: lengths from ``numpy.random.default_rng(seed).integers(len_min, len_max,
    endpoint=True, size=B)``; each sequence takes ceil(len / page_size) pages, and the pool
    (those plus ``spare_pages``) is shuffled by ``rng.permutation`` of the same generator;
    values from ``torch.Generator('cpu').manual_seed(seed)``: q, then K pages and V pages
    in blocks of 1024 pages, float32 ``randn`` rounded to bf16. ``poison_unused`` writes NaN
    into every cache slot no sequence owns (the unused tail of a last page, the spare
    pages), which no correct kernel may let into a result.
    """
    lens = decode_lengths(w)
    rng = np.random.default_rng(w.seed)
    if w.lengths is None:
        rng.integers(w.len_min, w.len_max, size=w.B, endpoint=True)  # same stream position
    ps = w.page_size
    need = [(int(n) + ps - 1) // ps for n in lens]
    num_pages = int(sum(need)) + w.spare_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    max_pages = max(1, (int(w.len_max) + ps - 1) // ps, max(need, default=0))
    table = np.full((w.B, max_pages), -1, dtype=np.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n]
        at += n
    g = torch.Generator("cpu").manual_seed(w.seed)
    q = torch.randn((w.B, w.Hq, w.Nq, w.d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    caches = []
    for _ in range(2):
        c = torch.empty((num_pages, w.Hkv, ps, w.d), dtype=torch.bfloat16)
        for p0 in range(0, num_pages, _PAGE_BLOCK):
            p1 = min(num_pages, p0 + _PAGE_BLOCK)
            c[p0:p1] = torch.randn((p1 - p0, w.Hkv, ps, w.d), generator=g, dtype=torch.float32)
        caches.append(c)
    k_cache, v_cache = caches
    if poison_unused:
        owned = np.zeros((num_pages, ps), dtype=bool)
        for b, n in enumerate(lens):
            t = np.arange(int(n))
            owned[table[b, t // ps], t % ps] = True
        bad = torch.from_numpy(~owned)[:, None, :, None].expand(-1, w.Hkv, -1, w.d)
        k_cache[bad] = float("nan")
        v_cache[bad] = float("nan")
    return q, k_cache, v_cache, torch.from_numpy(table), torch.from_numpy(lens.copy())
