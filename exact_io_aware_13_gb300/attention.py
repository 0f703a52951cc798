"""Python face of libattn.so: torch tensors in, the C ABI called, torch tensors out.

PyTorch only provides device memory and the current CUDA stream here; every step
of the computation runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib

MASK_NONE, MASK_CAUSAL, MASK_SLIDING_WINDOW, MASK_DOCUMENT_CAUSAL = 0, 1, 2, 3
SCORE_NONE, SCORE_ALIBI, SCORE_SOFTCAP, SCORE_DROPOUT = 0, 1, 2, 4
TILE_EMPTY, TILE_PARTIAL, TILE_FULL = 0, 1, 2
BWD_ROWDOT, BWD_DKDV, BWD_DQ, BWD_ALL = 1, 2, 4, 7
TILE = 128


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _params(mask_kind: int, window: int, doc_offsets: Optional[torch.Tensor],
            softcap: float, dropout_p: float = 0.0, dropout_seed: int = 0):
    mp = _lib.MaskParams(int(window), None, 0)
    if doc_offsets is not None:
        if doc_offsets.dtype != torch.int32 or not doc_offsets.is_cuda:
            raise ValueError("doc_offsets must be an int32 CUDA tensor")
        mp.doc_offsets = doc_offsets.data_ptr()
        mp.n_docs = doc_offsets.numel() - 1
    sp = _lib.ScoreParams(float(softcap), float(dropout_p), int(dropout_seed) & (2**64 - 1))
    return ctypes.byref(mp), ctypes.byref(sp), (mp, sp)


def _score_kind(score_kind: int, dropout_p: float) -> int:
    """Dropout is switched on by a positive drop probability."""
    return int(score_kind) | (SCORE_DROPOUT if dropout_p > 0 else 0)


def _dims(q: torch.Tensor, k: torch.Tensor):
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nkv, dk = k.shape
    if Bk != B or dk != d:
        raise ValueError("q and k disagree on batch or head dimension")
    return B, Hq, Hkv, Nq, Nkv, d


_BF16, _F32, _U8 = torch.bfloat16, torch.float32, torch.uint8


def _check_dtypes(*named):
    """named: (tensor or None, dtype, name) triples. The C ABI takes untyped pointers, so
    a tensor of another dtype would be read as the expected one: refuse it here."""
    for t, dtype, name in named:
        if t is not None and t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _check_shapes(q, k, v, o=None, lse=None, dout=None, dq=None, dk=None, dv=None):
    """Every buffer must have the shape the kernels index it with: q, o, dout, dq
    [B, Hq, Nq, d]; k, v, dk, dv [B, Hkv, Nkv, d]; lse [B, Hq, Nq]."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be [B, H, N, d]")
    for t, ref, name in ((v, k, "v"), (o, q, "o"), (dout, q, "dout"), (dq, q, "dq"),
                         (dk, k, "dk"), (dv, k, "dv")):
        if t is not None and tuple(t.shape) != tuple(ref.shape):
            raise ValueError(f"{name} must have shape {tuple(ref.shape)}, got {tuple(t.shape)}")
    if lse is not None and tuple(lse.shape) != tuple(q.shape[:-1]):
        raise ValueError(f"lse must have shape {tuple(q.shape[:-1])}, got {tuple(lse.shape)}")


def _check_bwd_dtypes(q, k, v, o, lse, dout, dq, dk, dv):
    _check_dtypes((q, _BF16, "q"), (k, _BF16, "k"), (v, _BF16, "v"), (o, _BF16, "o"),
                  (lse, _F32, "lse"), (dout, _BF16, "dout"), (dq, _BF16, "dq"),
                  (dk, _BF16, "dk"), (dv, _BF16, "dv"))


def _check_tensors(*ts):
    """Contiguous CUDA tensors, all on the current device (the library launches there,
    on that device's stream)."""
    index = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
        if index is None:
            index = t.device.index
        elif t.device.index != index:
            raise ValueError("tensors must all be on one device")
    if index is not None and index != torch.cuda.current_device():
        raise ValueError(f"tensors are on cuda:{index}, the current device is "
                         f"cuda:{torch.cuda.current_device()}")


def fwd_into(q, k, v, o, lse, *, scale: float, mask_kind: int = MASK_NONE, window: int = 0,
             doc_offsets=None, score_kind: int = SCORE_NONE, softcap: float = 0.0,
             dropout_p: float = 0.0, dropout_seed: int = 0, stream=None,
             impl: str = "tc") -> None:
    """Run attn_fwd (impl="tc") or attn_fwd_simt (impl="simt") into o and lse. A positive
    dropout_p drops elements of P by the Philox4x32-10 mask of dropout_seed."""
    _check_tensors(q, k, v, o, lse, doc_offsets)
    _check_dtypes((q, _BF16, "q"), (k, _BF16, "k"), (v, _BF16, "v"), (o, _BF16, "o"),
                  (lse, _F32, "lse"))
    _check_shapes(q, k, v, o, lse)
    lib = _lib.load()
    B, Hq, Hkv, Nq, Nkv, d = _dims(q, k)
    mp, sp, keep = _params(mask_kind, window, doc_offsets, softcap, dropout_p, dropout_seed)
    fn = lib.attn_fwd if impl == "tc" else lib.attn_fwd_simt
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nkv, d,
            ctypes.c_float(scale), mask_kind, mp, _score_kind(score_kind, dropout_p), sp,
            _stream(stream))
    del keep
    _lib.check(st, fn.__name__)


def forward(q, k, v, *, scale: Optional[float] = None, mask_kind: int = MASK_NONE,
            window: int = 0, doc_offsets=None, score_kind: int = SCORE_NONE,
            softcap: float = 0.0, dropout_p: float = 0.0, dropout_seed: int = 0,
            stream=None, impl: str = "tc"):
    """Exact attention forward. q: bf16 [B,Hq,Nq,d], k/v: bf16 [B,Hkv,Nkv,d] on CUDA.
    Returns (o bf16 [B,Hq,Nq,d], lse fp32 [B,Hq,Nq]); lse is that of the undropped
    softmax when dropout_p > 0."""
    d = q.shape[-1]
    if scale is None:
        scale = float(torch.tensor(d, dtype=torch.float32).rsqrt())
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    fwd_into(q, k, v, o, lse, scale=scale, mask_kind=mask_kind, window=window,
             doc_offsets=doc_offsets, score_kind=score_kind, softcap=softcap,
             dropout_p=dropout_p, dropout_seed=dropout_seed, stream=stream, impl=impl)
    return o, lse


def bwd_workspace_size(q, k) -> int:
    B, Hq, Hkv, Nq, Nkv, d = _dims(q, k)
    return int(_lib.load().attn_bwd_workspace_size(B, Hq, Hkv, Nq, Nkv, d))


def bwd_into(q, k, v, o, lse, dout, dq, dk, dv, workspace, *, scale: float,
             mask_kind: int = MASK_NONE, window: int = 0, doc_offsets=None,
             score_kind: int = SCORE_NONE, softcap: float = 0.0, dropout_p: float = 0.0,
             dropout_seed: int = 0, stream=None, impl: str = "tc") -> None:
    """Run attn_bwd (impl="tc") or attn_bwd_simt into dq, dk, dv; dropout_p and
    dropout_seed must be those of the forward."""
    _check_tensors(q, k, v, o, lse, dout, dq, dk, dv, workspace, doc_offsets)
    _check_bwd_dtypes(q, k, v, o, lse, dout, dq, dk, dv)
    _check_shapes(q, k, v, o, lse, dout, dq, dk, dv)
    lib = _lib.load()
    B, Hq, Hkv, Nq, Nkv, d = _dims(q, k)
    mp, sp, keep = _params(mask_kind, window, doc_offsets, softcap, dropout_p, dropout_seed)
    fn = lib.attn_bwd if impl == "tc" else lib.attn_bwd_simt
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
            _ptr(dv), B, Hq, Hkv, Nq, Nkv, d, ctypes.c_float(scale), mask_kind, mp,
            _score_kind(score_kind, dropout_p), sp, _ptr(workspace),
            ctypes.c_size_t(ws_bytes), _stream(stream))
    del keep
    _lib.check(st, fn.__name__)


def bwd_phases_into(phases: int, q, k, v, o, lse, dout, dq, dk, dv, workspace, *, scale: float,
                    mask_kind: int = MASK_NONE, window: int = 0, doc_offsets=None,
                    score_kind: int = SCORE_NONE, softcap: float = 0.0,
                    dropout_p: float = 0.0, dropout_seed: int = 0, stream=None) -> None:
    """Run some of the backward's kernels (BWD_ROWDOT | BWD_DKDV | BWD_DQ) via
    attn_bwd_phases; BWD_ROWDOT must have run on the same workspace first."""
    _check_tensors(q, k, v, o, lse, dout, dq, dk, dv, workspace, doc_offsets)
    _check_bwd_dtypes(q, k, v, o, lse, dout, dq, dk, dv)
    _check_shapes(q, k, v, o, lse, dout, dq, dk, dv)
    lib = _lib.load()
    B, Hq, Hkv, Nq, Nkv, d = _dims(q, k)
    mp, sp, keep = _params(mask_kind, window, doc_offsets, softcap, dropout_p, dropout_seed)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.attn_bwd_phases(int(phases), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                             _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Nq, Nkv, d,
                             ctypes.c_float(scale), mask_kind, mp,
                             _score_kind(score_kind, dropout_p), sp,
                             _ptr(workspace), ctypes.c_size_t(ws_bytes), _stream(stream))
    del keep
    _lib.check(st, "attn_bwd_phases")


def backward(q, k, v, o, lse, dout, *, scale: Optional[float] = None,
             mask_kind: int = MASK_NONE, window: int = 0, doc_offsets=None,
             score_kind: int = SCORE_NONE, softcap: float = 0.0, dropout_p: float = 0.0,
             dropout_seed: int = 0, stream=None, impl: str = "tc"):
    """Gradients (dq, dk, dv) of sum(dout * o), rebuilding P from lse (and the dropout
    mask from dropout_seed when dropout_p > 0)."""
    d = q.shape[-1]
    if scale is None:
        scale = float(torch.tensor(d, dtype=torch.float32).rsqrt())
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ws = torch.empty(max(bwd_workspace_size(q, k), 256), dtype=torch.uint8, device=q.device)
    bwd_into(q, k, v, o, lse, dout, dq, dk, dv, ws, scale=scale, mask_kind=mask_kind,
             window=window, doc_offsets=doc_offsets, score_kind=score_kind, softcap=softcap,
             dropout_p=dropout_p, dropout_seed=dropout_seed, stream=stream, impl=impl)
    return dq, dk, dv


def classify_tiles(mask_kind: int, Nq: int, Nkv: int, *, window: int = 0, doc_offsets=None,
                   device="cuda", stream=None) -> torch.Tensor:
    """Tile classes [ceil(Nq/128), ceil(Nkv/128)] int32: 0 empty, 1 partial, 2 full."""
    lib = _lib.load()
    nqt, nkt = -(-Nq // TILE), -(-Nkv // TILE)
    out = torch.empty((nqt, nkt), dtype=torch.int32, device=device)
    mp, _, keep = _params(mask_kind, window, doc_offsets, 0.0)
    st = lib.attn_classify_tiles(mask_kind, mp, Nq, Nkv, _ptr(out), _stream(stream))
    del keep
    _lib.check(st, "attn_classify_tiles")
    return out


def check_doc_offsets(doc_offsets: torch.Tensor, N: int, stream=None) -> None:
    """Queue the device check of a document-offsets table (attn_check_doc_offsets); a
    bad table shows up as ATTN_ERR_DEVICE_INPUT (8) in the next device_status()."""
    _check_tensors(doc_offsets)
    _check_dtypes((doc_offsets, torch.int32, "doc_offsets"))
    _lib.check(_lib.load().attn_check_doc_offsets(_ptr(doc_offsets), doc_offsets.numel() - 1,
                                                  int(N), _stream(stream)),
               "attn_check_doc_offsets")


def device_status(stream=None) -> int:
    """Synchronise and return the library's device status (0 = no kernel gave up)."""
    return int(_lib.load().attn_device_status(_stream(stream)))


# ---------------------------------------------------------------- FP8
FP8_TILES, FP8_V_TRANSPOSED = 0, 1


def selftest_wait_timeout(stream=None) -> None:
    """Launch the failure-path self-test (attn_selftest_wait_timeout): a bounded device
    wait that nothing completes gives up after about 2 s; device_status() then reports
    ATTN_ERR_DEVICE_TIMEOUT."""
    _lib.check(_lib.load().attn_selftest_wait_timeout(_stream(stream)), "attn_selftest_wait_timeout")


def quantize_fp8(x: torch.Tensor, layout: int = FP8_TILES, stream=None):
    """bf16 x [B, H, N, d] -> (e4m3 codes as uint8, fp32 scales) via attn_quantize_fp8.
    FP8_TILES: codes [B, H, N, d], scales [B*H, ceil(N/128)];
    FP8_V_TRANSPOSED: codes [B, H, d, attn_fp8_v_row_bytes(N)], scales [B*H]."""
    _check_tensors(x)
    _check_dtypes((x, _BF16, "x"))
    lib = _lib.load()
    B, H, N, d = x.shape
    if layout == FP8_TILES:
        codes = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device)
        scales = torch.empty((B * H, (N + 127) // 128), dtype=torch.float32, device=x.device)
    else:
        codes = torch.empty((B, H, d, int(lib.attn_fp8_v_row_bytes(N))), dtype=torch.uint8,
                            device=x.device)
        scales = torch.empty((B * H,), dtype=torch.float32, device=x.device)
    st = lib.attn_quantize_fp8(_ptr(x), _ptr(codes), _ptr(scales), B * H, N, d, layout,
                               _stream(stream))
    _lib.check(st, "attn_quantize_fp8")
    return codes, scales


def fp8_inputs(q, k, v, stream=None):
    """Quantise bf16 q, k, v for forward_fp8: ((q8, sq), (k8, sk), (v8t, sv))."""
    return (quantize_fp8(q, FP8_TILES, stream), quantize_fp8(k, FP8_TILES, stream),
            quantize_fp8(v, FP8_V_TRANSPOSED, stream))


def fwd_fp8_into(q8, sq, k8, sk, v8t, sv, o, lse, *, Nkv: int, scale: float,
                 mask_kind: int = MASK_NONE, window: int = 0, doc_offsets=None,
                 score_kind: int = SCORE_NONE, softcap: float = 0.0, stream=None) -> None:
    """Run attn_fwd_fp8 into o (bf16 [B,Hq,Nq,128]) and lse."""
    _check_tensors(q8, sq, k8, sk, v8t, sv, o, lse, doc_offsets)
    _check_dtypes((q8, _U8, "q8"), (k8, _U8, "k8"), (v8t, _U8, "v8t"), (sq, _F32, "sq"),
                  (sk, _F32, "sk"), (sv, _F32, "sv"), (o, _BF16, "o"), (lse, _F32, "lse"))
    lib = _lib.load()
    B, Hq, Nq, d = q8.shape
    Hkv = k8.shape[1]
    mp, sp, keep = _params(mask_kind, window, doc_offsets, softcap)
    st = lib.attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8t), _ptr(sq), _ptr(sk), _ptr(sv), _ptr(o),
                          _ptr(lse), B, Hq, Hkv, Nq, Nkv, d, ctypes.c_float(scale), mask_kind, mp,
                          score_kind, sp, _stream(stream))
    del keep
    _lib.check(st, "attn_fwd_fp8")


def forward_fp8(q, k, v, *, scale: Optional[float] = None, mask_kind: int = MASK_NONE,
                window: int = 0, doc_offsets=None, score_kind: int = SCORE_NONE,
                softcap: float = 0.0, stream=None):
    """Quantise bf16 q, k, v to e4m3 with block scales and run the FP8 forward.
    Returns (o, lse, ((q8, sq), (k8, sk), (v8t, sv)))."""
    d = q.shape[-1]
    if scale is None:
        scale = float(torch.tensor(d, dtype=torch.float32).rsqrt())
    (q8, sq), (k8, sk), (v8t, sv) = quant = fp8_inputs(q, k, v, stream)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    fwd_fp8_into(q8, sq, k8, sk, v8t, sv, o, lse, Nkv=k.shape[2], scale=scale,
                 mask_kind=mask_kind, window=window, doc_offsets=doc_offsets,
                 score_kind=score_kind, softcap=softcap, stream=stream)
    return o, lse, quant


# ---------------------------------------------------------------- paged decode
def decode_split_keys(B: int, Hq: int, Hkv: int, Nq: int, total_kv_tokens: int,
                      num_sms: Optional[int] = None) -> int:
    """The library's split size for a decode call (keys per chunk)."""
    if num_sms is None:
        num_sms = (torch.cuda.get_device_properties(torch.cuda.current_device())
                   .multi_processor_count if torch.cuda.is_available() else 0)
    return int(_lib.load().attn_decode_split_keys(int(B), int(Hq), int(Hkv), int(Nq),
                                                  int(total_kv_tokens), int(num_sms)))


def decode_workspace_size(B: int, Hq: int, Hkv: int, Nq: int, d: int, max_seq_len: int,
                          split_keys: int) -> int:
    return int(_lib.load().attn_decode_workspace_size(int(B), int(Hq), int(Hkv), int(Nq), int(d),
                                                      int(max_seq_len), int(split_keys)))


def decode_paged_into(q, k_cache, v_cache, page_table, seq_lens, o, lse, workspace, *,
                      max_seq_len: int, split_keys: int, scale: float,
                      mask_kind: int = MASK_NONE, window: int = 0, score_kind: int = SCORE_NONE,
                      softcap: float = 0.0, stream=None) -> None:
    """attn_decode_paged on caller-owned tensors (see include/attn.h for the layouts):
    q [B, Hq, Nq, d], caches [pages, Hkv, page_size, d], page_table int32 [B, max_pages],
    seq_lens int32 [B]; writes o and lse."""
    _check_tensors(q, k_cache, v_cache, page_table, seq_lens, o, lse, workspace)
    _check_dtypes((q, _BF16, "q"), (k_cache, _BF16, "k_cache"), (v_cache, _BF16, "v_cache"),
                  (o, _BF16, "o"), (lse, _F32, "lse"))
    if q.dim() != 4 or tuple(o.shape) != tuple(q.shape) or tuple(lse.shape) != tuple(q.shape[:-1]):
        raise ValueError("q, o must be [B, Hq, Nq, d] and lse [B, Hq, Nq]")
    B, Hq, Nq, d = q.shape
    num_pages, Hkv, page_size, dk = k_cache.shape
    if dk != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache must be [pages, Hkv, page_size, d]")
    if page_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("page_table and seq_lens must be int32")
    if page_table.dim() != 2 or page_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("page_table must be [B, max_pages] and seq_lens [B]")
    mp, sp, _keep = _params(mask_kind, window, None, softcap)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.load().attn_decode_paged(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(seq_lens), _ptr(o),
        _ptr(lse), B, Hq, Hkv, Nq, d, num_pages, page_size, page_table.shape[1],
        int(max_seq_len), int(split_keys), ctypes.c_float(scale), mask_kind, mp, score_kind, sp,
        _ptr(workspace), ctypes.c_size_t(ws_bytes), _stream(stream))
    _lib.check(st, "attn_decode_paged")


def decode_paged(q, k_cache, v_cache, page_table, seq_lens, *, max_seq_len: Optional[int] = None,
                 split_keys: Optional[int] = None, total_kv_tokens: Optional[int] = None,
                 scale: Optional[float] = None, mask_kind: int = MASK_NONE, window: int = 0,
                 score_kind: int = SCORE_NONE, softcap: float = 0.0, stream=None):
    """Allocating wrapper of decode_paged_into: returns (o, lse). max_seq_len defaults to
    the page table's capacity; split_keys to the library's choice for total_kv_tokens
    (default B * max_seq_len)."""
    B, Hq, Nq, d = q.shape
    Hkv, page_size = k_cache.shape[1], k_cache.shape[2]
    if max_seq_len is None:
        max_seq_len = page_table.shape[1] * page_size
    if split_keys is None:
        split_keys = decode_split_keys(B, Hq, Hkv, Nq, total_kv_tokens or B * max_seq_len)
    if scale is None:
        scale = float(d) ** -0.5
    o = torch.empty((B, Hq, Nq, d), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    nbytes = decode_workspace_size(B, Hq, Hkv, Nq, d, max_seq_len, split_keys)
    ws = torch.empty((nbytes,), dtype=torch.uint8, device=q.device) if nbytes else None
    decode_paged_into(q, k_cache, v_cache, page_table, seq_lens, o, lse, ws,
                      max_seq_len=max_seq_len, split_keys=split_keys, scale=scale,
                      mask_kind=mask_kind, window=window, score_kind=score_kind, softcap=softcap,
                      stream=stream)
    return o, lse
