"""ctypes view of libattn.so (include/attn.h). Argument marshalling only.

Loading fails loudly when the library has not been built: there is no other path
that computes attention in this package.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattn.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "attn.h")

ATTN_OK = 0
STATUS_NAMES = {0: "ATTN_OK", 1: "ATTN_ERR_ARG", 2: "ATTN_ERR_SHAPE", 3: "ATTN_ERR_ALIGN",
                4: "ATTN_ERR_ARCH", 5: "ATTN_ERR_WORKSPACE", 6: "ATTN_ERR_LAUNCH",
                7: "ATTN_ERR_DEVICE_TIMEOUT", 8: "ATTN_ERR_DEVICE_INPUT"}


class MaskParams(ctypes.Structure):
    _fields_ = [("window", ctypes.c_int32), ("doc_offsets", ctypes.c_void_p),
                ("n_docs", ctypes.c_int32)]


class ScoreParams(ctypes.Structure):
    _fields_ = [("softcap", ctypes.c_float), ("dropout_p", ctypes.c_float),
                ("dropout_seed", ctypes.c_uint64)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_MP = ctypes.POINTER(MaskParams)
_SP = ctypes.POINTER(ScoreParams)

_FWD_ARGS = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _MP, _I, _SP, _P]
_BWD_ARGS = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _MP, _I, _SP,
             _P, ctypes.c_size_t, _P]

SIGNATURES = {
    "attn_fwd": (_I, _FWD_ARGS),
    "attn_fwd_simt": (_I, _FWD_ARGS),
    "attn_bwd_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "attn_bwd": (_I, _BWD_ARGS),
    "attn_bwd_simt": (_I, _BWD_ARGS),
    "attn_bwd_static_workspace": (_I, _BWD_ARGS[:20] + [_P]),
    "attn_bwd_phases": (_I, [_I] + _BWD_ARGS),
    "attn_classify_tiles": (_I, [_I, _MP, _I, _I, _P, _P]),
    "attn_fwd_fp8": (_I, [_P] * 8 + [_I, _I, _I, _I, _I, _I, _F, _I, _MP, _I, _SP, _P]),
    "attn_fp8_v_row_bytes": (ctypes.c_size_t, [_I]),
    "attn_quantize_fp8": (_I, [_P, _P, _P, _I, _I, _I, _I, _P]),
    "attn_decode_paged": (_I, [_P] * 7 + [_I] * 10 + [_F, _I, _MP, _I, _SP, _P, ctypes.c_size_t,
                                                     _P]),
    "attn_decode_workspace_size": (ctypes.c_size_t, [_I] * 7),
    "attn_decode_split_keys": (_I, [_I, _I, _I, _I, ctypes.c_longlong, _I]),
    "attn_check_doc_offsets": (_I, [_P, _I, _I, _P]),
    "attn_device_status": (_I, [_P]),
    "attn_selftest_wait_timeout": (_I, [_P]),
    "attn_strerror": (ctypes.c_char_p, [_I]),
}

_lib = None


def header_functions() -> list[str]:
    """Names of the functions include/attn.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"^\s*(?:attn_status|size_t|int|const char\*)\s+(attn_\w+)\s*\(", text,
                      re.M)


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
            "g.build()'). There is no fallback implementation.")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = load().attn_strerror(status).decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({msg})")


def check(status: int, where: str) -> None:
    if status != ATTN_OK:
        raise AttnError(status, where)
