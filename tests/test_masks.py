"""The kernels' mask predicate and block-sparsity tile rule (csrc/mask.cuh), built
for the host, against the oracle's brute force over every (i, j). CPU only; the
same rule is checked on the GPU through attn_classify_tiles in test_parity.py."""
import ctypes

import numpy as np
import pytest

from oracle import attention_oracle as ref
from tests.host import build_host
from workloads import (MASK_CAUSAL, MASK_DOCUMENT_CAUSAL, MASK_NONE, MASK_SLIDING_WINDOW,
                       document_offsets, offsets_from_lengths)

T = 128


@pytest.fixture(scope="module")
def host():
    return build_host.load()


def _doc_args(offs):
    if offs is None:
        return None, 0
    arr = np.ascontiguousarray(offs, dtype=np.int32)
    return arr, len(arr) - 1


def _cases():
    rng = np.random.default_rng(123)
    cases = []
    for nq, nkv in [(1, 1), (127, 127), (128, 128), (129, 129), (300, 300), (512, 512),
                    (700, 700), (256, 640), (640, 256), (1000, 1000)]:
        cases.append((MASK_NONE, 0, None, nq, nkv))
        cases.append((MASK_CAUSAL, 0, None, nq, nkv))
        for w in (0, 1, 5, 127, 128, 129, 300):
            cases.append((MASK_SLIDING_WINDOW, w, None, nq, nkv))
        if nq == nkv:
            for _ in range(3):
                lens = []
                while sum(lens) < nq:
                    lens.append(int(rng.integers(1, max(2, nq // 3) + 1)))
                lens[-1] -= sum(lens) - nq
                cases.append((MASK_DOCUMENT_CAUSAL, 0, offsets_from_lengths(lens), nq, nkv))
    return cases


CASES = _cases()


@pytest.mark.parametrize("case", range(len(CASES)))
def test_allowed_and_tile_rule_match_brute_force(host, case):
    kind, w, offs, nq, nkv = CASES[case]
    doc, n_docs = _doc_args(offs)
    docp = doc.ctypes.data_as(ctypes.c_void_p) if doc is not None else None

    allowed = np.zeros((nq, nkv), dtype=np.uint8)
    host.host_allowed(kind, w, docp, n_docs, nq, nkv, allowed.ctypes.data_as(ctypes.c_void_p))
    expect = ref.allowed(kind, np.arange(nq), np.arange(nkv), w, offs, max(nq, nkv))
    assert (allowed.astype(bool) == expect).all()

    nqt, nkt = -(-nq // T), -(-nkv // T)
    cls = np.zeros((nqt, nkt), dtype=np.int32)
    host.host_classify(kind, w, docp, n_docs, nq, nkv, cls.ctypes.data_as(ctypes.c_void_p))
    brute = ref.classify_tiles(kind, nq, nkv, T, T, w, offs)
    assert (cls == brute).all(), (cls, brute)

    kv = np.zeros((nqt, 2), dtype=np.int32)
    qr = np.zeros((nkt, 2), dtype=np.int32)
    need = np.zeros((nqt, nkt), dtype=np.uint8)
    host.host_ranges(kind, w, docp, n_docs, nq, nkv, T, kv.ctypes.data_as(ctypes.c_void_p),
                     qr.ctypes.data_as(ctypes.c_void_p), need.ctypes.data_as(ctypes.c_void_p))
    for r in range(nqt):  # the key-tile run of each query tile is exactly its non-empty tiles
        nz = np.nonzero(brute[r] != ref.TILE_EMPTY)[0]
        if len(nz) == 0:
            assert kv[r, 0] >= kv[r, 1]
        else:
            assert (kv[r, 0], kv[r, 1]) == (nz[0], nz[-1] + 1)
            assert len(nz) == nz[-1] - nz[0] + 1  # contiguous
        for c in range(nkt):
            if brute[r, c] == ref.TILE_FULL and (c + 1) * T <= nkv:
                assert need[r, c] == 0
            elif brute[r, c] != ref.TILE_EMPTY:
                assert need[r, c] == 1
    for c in range(nkt):  # the query-tile run of each key tile
        nz = np.nonzero(brute[:, c] != ref.TILE_EMPTY)[0]
        if len(nz) == 0:
            assert qr[c, 0] >= qr[c, 1]
        else:
            assert (qr[c, 0], qr[c, 1]) == (nz[0], nz[-1] + 1)


def test_workload_tile_counts(host):
    """Window workload: 1116 non-empty and 868 full 128x128 tiles per head; the
    document workload's tile classes match brute force too."""
    n = 16384
    cls = np.zeros((n // T, n // T), dtype=np.int32)
    host.host_classify(MASK_SLIDING_WINDOW, 1024, None, 0, n, n,
                       cls.ctypes.data_as(ctypes.c_void_p))
    assert int((cls != 0).sum()) == 1116 and int((cls == 2).sum()) == 868
    n = 32768
    offs = document_offsets(n, 3)
    doc = np.ascontiguousarray(offs, dtype=np.int32)
    cls = np.zeros((n // T, n // T), dtype=np.int32)
    host.host_classify(MASK_DOCUMENT_CAUSAL, 0, doc.ctypes.data_as(ctypes.c_void_p),
                       len(doc) - 1, n, n, cls.ctypes.data_as(ctypes.c_void_p))
    brute = ref.classify_tiles(MASK_DOCUMENT_CAUSAL, n, n, T, T, 0, offs)
    assert (cls == brute).all()


def test_flop_pair_counts_match_brute_force():
    from exact_io_aware_13_gb300 import flops
    for kind, nq, nkv, w, offs in [(MASK_NONE, 300, 200, 0, None), (MASK_CAUSAL, 300, 300, 0, None),
                                   (MASK_CAUSAL, 300, 120, 0, None), (MASK_CAUSAL, 120, 300, 0, None),
                                   (MASK_SLIDING_WINDOW, 500, 500, 77, None),
                                   (MASK_SLIDING_WINDOW, 500, 500, 0, None),
                                   (MASK_DOCUMENT_CAUSAL, 900, 900, 0, offsets_from_lengths([100, 500, 300]))]:
        assert flops.allowed_pairs(kind, nq, nkv, w, offs) == ref.allowed_pairs(kind, nq, nkv, w, offs)
    n = 8192
    assert flops.allowed_pairs(MASK_CAUSAL, n, n) == 33558528
    assert flops.attention_flops(4, 16, 128, 33558528, False) == 1099645845504.0  # 4 * d * pairs * B * H
