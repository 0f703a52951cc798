"""The C ABI without a GPU: the library loads, exports every function the header
declares, and rejects bad arguments with the documented status before touching a
device."""
import ctypes

import pytest

from exact_io_aware_13_gb300 import _lib
from exact_io_aware_13_gb300 import build as libbuild


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return _lib.load()


def test_exports_every_declared_function(lib):
    names = _lib.header_functions()
    assert len(names) >= 8
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(_lib.SIGNATURES)


def test_strerror_texts(lib):
    for code in range(9):
        assert lib.attn_strerror(code).decode()
    assert lib.attn_strerror(99).decode() == "unknown status"


def _fwd(lib, **kw):
    a = dict(q=None, k=None, v=None, o=None, lse=None, B=1, Hq=2, Hkv=1, Nq=16, Nkv=16, d=64,
             scale=0.125, mask=0, mp=None, score=0, sp=None)
    a.update(kw)
    return lib.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"],
                        a["Nq"], a["Nkv"], a["d"], ctypes.c_float(a["scale"]), a["mask"],
                        a["mp"], a["score"], a["sp"], None)


def test_argument_errors_return_before_any_device_call(lib):
    assert _fwd(lib, d=96) == 2                       # ATTN_ERR_SHAPE
    assert _fwd(lib, d=512) == 2
    # d = 256: the tensor-core forward and backward take it, the SIMT backward does not
    rc = lib.attn_bwd_simt(*([ctypes.c_void_p(4096)] * 9), 1, 1, 1, 128, 128, 256,
                           ctypes.c_float(0.1), 0, None, 0, None, ctypes.c_void_p(4096), 1 << 20,
                           None)
    assert rc == 2
    sp = _lib.ScoreParams(0.0, 0.1, 7)  # ... and dropout stays at d <= 128
    rc = lib.attn_bwd(*([ctypes.c_void_p(4096)] * 9), 1, 1, 1, 128, 128, 256,
                      ctypes.c_float(0.1), 0, None, 4, ctypes.byref(sp), ctypes.c_void_p(4096),
                      1 << 20, None)
    assert rc == 1
    assert _fwd(lib, Hq=3, Hkv=2) == 2
    assert _fwd(lib, Nq=-1) == 2
    assert _fwd(lib, scale=float("nan")) == 1         # ATTN_ERR_ARG
    assert _fwd(lib, mask=7) == 1
    assert _fwd(lib, score=8) == 1                    # unknown score bit
    assert _fwd(lib, score=4) == 1                    # dropout without params
    for p_drop in (-0.1, 1.0, 1.5, float("nan")):
        sp = _lib.ScoreParams(0.0, p_drop, 7)
        assert _fwd(lib, score=4, sp=ctypes.byref(sp)) == 1, p_drop
    sp = _lib.ScoreParams(0.0, 0.1, 7)
    assert _fwd(lib, score=4, sp=ctypes.byref(sp)) == 1   # valid dropout, null tensors
    assert _fwd(lib, score=4, sp=ctypes.byref(sp), d=256) == 1  # dropout: d <= 128
    assert lib.attn_fwd_simt(None, None, None, None, None, 1, 2, 1, 16, 16, 64,
                             ctypes.c_float(0.125), 0, None, 4, ctypes.byref(sp), None) == 1
    assert lib.attn_bwd_simt(*([ctypes.c_void_p(4096)] * 9), 1, 1, 1, 128, 128, 64,
                             ctypes.c_float(0.1), 0, None, 4, ctypes.byref(sp),
                             ctypes.c_void_p(4096), 1 << 20, None) == 1
    assert _fwd(lib, mask=2, mp=None) == 1            # window without params
    mp = _lib.MaskParams(-1, None, 0)
    assert _fwd(lib, mask=2, mp=ctypes.byref(mp)) == 1
    sp = _lib.ScoreParams(0.0)
    assert _fwd(lib, score=2, sp=ctypes.byref(sp)) == 1   # soft-cap must be > 0
    mp = _lib.MaskParams(0, ctypes.c_void_p(16), 1)
    assert _fwd(lib, mask=3, mp=ctypes.byref(mp), Nkv=32) == 2  # documents need Nq == Nkv
    assert _fwd(lib) == 1                             # null tensors
    assert _fwd(lib, q=ctypes.c_void_p(0x1002), k=ctypes.c_void_p(0x2000),
                v=ctypes.c_void_p(0x3000), o=ctypes.c_void_p(0x4000),
                lse=ctypes.c_void_p(0x5000)) == 3     # misaligned q


def test_empty_problems_are_a_no_op(lib):
    assert _fwd(lib, B=0) == 0
    assert _fwd(lib, Nq=0) == 0
    assert lib.attn_bwd_workspace_size(0, 4, 4, 128, 128, 64) == 0


def _round256(x):
    return (x + 255) // 256 * 256


def test_workspace_size(lib):
    # L log2 e and D per row padded to 128 rows per head, plus one first-key int per
    # padded row position; each array rounded up to 256 bytes
    def expect(B, Hq, Nq):
        nq128 = (Nq + 127) // 128 * 128
        return 2 * _round256(4 * B * Hq * nq128) + _round256(4 * nq128)
    assert lib.attn_bwd_workspace_size(2, 16, 16, 8192, 8192, 128) == expect(2, 16, 8192)
    assert expect(2, 16, 8192) == 2 * 2 * 16 * 8192 * 4 + 8192 * 4
    assert lib.attn_bwd_workspace_size(1, 1, 1, 3, 3, 64) == 3 * 512
    assert lib.attn_bwd_workspace_size(3, 5, 5, 700, 700, 64) == expect(3, 5, 700)
    rc = lib.attn_bwd(*([ctypes.c_void_p(4096)] * 9), 1, 1, 1, 128, 128, 64,
                      ctypes.c_float(0.1), 0, None, 0, None, None, 0, None)
    assert rc == 5  # ATTN_ERR_WORKSPACE


def test_classify_rejects_bad_kind(lib):
    assert lib.attn_classify_tiles(9, None, 10, 10, None, None) == 1
    assert lib.attn_classify_tiles(0, None, 0, 10, None, None) == 0


def _decode(lib, **kw):
    a = dict(q=None, k=None, v=None, table=None, lens=None, o=None, lse=None, B=2, Hq=8, Hkv=2,
             Nq=1, d=128, pages=10, ps=16, maxp=8, msl=100, split=64, scale=0.125, mask=0,
             mp=None, score=0, sp=None, ws=None, wsb=0)
    a.update(kw)
    return lib.attn_decode_paged(a["q"], a["k"], a["v"], a["table"], a["lens"], a["o"], a["lse"],
                                 a["B"], a["Hq"], a["Hkv"], a["Nq"], a["d"], a["pages"], a["ps"],
                                 a["maxp"], a["msl"], a["split"], ctypes.c_float(a["scale"]),
                                 a["mask"], a["mp"], a["score"], a["sp"], a["ws"], a["wsb"], None)


def test_decode_argument_errors_return_before_any_device_call(lib):
    assert _decode(lib, d=96) == 2                    # ATTN_ERR_SHAPE
    assert _decode(lib, Hq=3) == 2
    for ps in (0, 4, 12, 48, 96):                     # page sizes that straddle 64-key tiles
        assert _decode(lib, ps=ps, maxp=64) == 2, ps
    assert _decode(lib, msl=8 * 16 + 1) == 2          # above the page table's capacity
    assert _decode(lib, split=0) == 1                 # ATTN_ERR_ARG
    assert _decode(lib, split=96) == 1
    assert _decode(lib, mask=3) == 1                  # no document masking in decode
    assert _decode(lib, mask=2) == 1                  # window without params
    assert _decode(lib, scale=float("inf")) == 1
    assert _decode(lib) == 1                          # null tensors
    good = {n: ctypes.c_void_p(0x10000 * (i + 1)) for i, n in
            enumerate(("q", "k", "v", "table", "lens", "o", "lse"))}
    assert _decode(lib, **dict(good, q=ctypes.c_void_p(0x10008))) == 3   # misaligned q
    assert _decode(lib, **dict(good, table=ctypes.c_void_p(0x30002))) == 3
    assert _decode(lib, **good) == 5                  # two chunks need a workspace
    assert _decode(lib, **good, ws=ctypes.c_void_p(0x100000), wsb=10) == 5
    assert _decode(lib, B=0) == 0                     # nothing to do
    assert _decode(lib, Nq=0) == 0


def test_decode_workspace_size_and_split_keys(lib):
    # n partials per row (chunks x row copies): log2-sum-exp plane + fp32 O plane
    ws = lib.attn_decode_workspace_size
    # 128 rows per group (one copy), one chunk: results written in place
    assert ws(4, 32, 1, 4, 128, 8192, 8192) == 0
    assert ws(4, 32, 8, 1, 128, 0, 256) == 0            # no cached key at all
    # G * Nq = 4 rows: 2 copies, even with one chunk
    rows = 4 * 32 * 1
    assert ws(4, 32, 8, 1, 128, 8192, 8192) == _round256(4 * 2 * rows) + _round256(4 * 2 * rows * 128)
    assert ws(4, 32, 8, 1, 128, 8192, 512) == _round256(4 * 32 * rows) + _round256(4 * 32 * rows * 128)
    # 32 rows: 2 copies; 35 and 105 rows: 1 copy
    assert ws(3, 4, 1, 8, 64, 1000, 192) == _round256(4 * 12 * 96) + _round256(4 * 12 * 96 * 64)
    assert ws(3, 5, 1, 7, 64, 1000, 192) == _round256(4 * 6 * 105) + _round256(4 * 6 * 105 * 64)
    assert ws(3, 35, 7, 7, 64, 1000, 192) == _round256(4 * 6 * 735) + _round256(4 * 6 * 735 * 64)
    assert ws(3, 5, 1, 21, 64, 1000, 192) == _round256(4 * 6 * 315) + _round256(4 * 6 * 315 * 64)
    # split keys: a multiple of 64, at least 256, about 32 CTAs of work per SM
    for args in [(64, 32, 8, 1, 64 * 4352, 152), (1, 8, 8, 1, 100, 152),
                 (8, 64, 8, 40, 8 * 100000, 148), (2, 4, 4, 1, 0, 0)]:
        keys = lib.attn_decode_split_keys(*args)
        assert keys >= 256 and keys % 64 == 0, args
    assert lib.attn_decode_split_keys(64, 32, 8, 1, 64 * 4352, 152) == 1472  # ceil64(1466.1)
    assert lib.attn_decode_split_keys(1, 8, 8, 1, 100, 152) == 256


def test_binding_refuses_wrong_dtypes():
    """The C ABI takes untyped pointers: the torch binding checks every tensor's dtype
    (bf16 inputs and outputs, fp32 lse and FP8 scales, uint8 FP8 codes) before a call."""
    import torch

    from exact_io_aware_13_gb300 import attention as A
    bf, f32 = torch.zeros(2, dtype=torch.bfloat16), torch.zeros(2, dtype=torch.float32)
    A._check_dtypes((bf, torch.bfloat16, "q"), (f32, torch.float32, "lse"), (None, torch.uint8, "x"))
    with pytest.raises(ValueError, match="q must be torch.bfloat16"):
        A._check_dtypes((f32, torch.bfloat16, "q"))
    with pytest.raises(ValueError, match="lse must be torch.float32"):
        A._check_bwd_dtypes(bf, bf, bf, bf, bf, bf, bf, bf, bf)
    with pytest.raises(ValueError, match="dv must be torch.bfloat16"):
        A._check_bwd_dtypes(bf, bf, bf, bf, f32, bf, bf, bf, f32)


def test_binding_refuses_wrong_shapes():
    """A buffer smaller than the shape the kernels index would be written past its end:
    the binding compares every buffer's shape with q's and k's before a call."""
    import torch

    from exact_io_aware_13_gb300 import attention as A
    q, k = torch.zeros(1, 4, 10, 64), torch.zeros(1, 2, 12, 64)
    A._check_shapes(q, k, k.clone(), q.clone(), torch.zeros(1, 4, 10), q.clone(), q.clone(),
                    k.clone(), k.clone())
    with pytest.raises(ValueError, match="lse must have shape"):
        A._check_shapes(q, k, k, q, torch.zeros(1, 4, 9))
    with pytest.raises(ValueError, match="dk must have shape"):
        A._check_shapes(q, k, k, q, None, None, None, torch.zeros(1, 2, 11, 64))
    with pytest.raises(ValueError, match="o must have shape"):
        A._check_shapes(q, k, k, torch.zeros(1, 4, 10, 32))
