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
    for code in range(8):
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
    assert _fwd(lib, Hq=3, Hkv=2) == 2
    assert _fwd(lib, Nq=-1) == 2
    assert _fwd(lib, scale=float("nan")) == 1         # ATTN_ERR_ARG
    assert _fwd(lib, mask=7) == 1
    assert _fwd(lib, score=4) == 1
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
