"""GPU parity of the paged decode (attn_decode_paged) against the float64 decode oracle on
the same seeded inputs: O within 1e-2, LSE within 1e-3 with -inf exactly where the
oracle has it. Unused cache slots are filled with NaN, so a kernel that lets a slot past
a sequence's end into a result fails. Cases span several key chunks and tiles with
ragged tails, page sizes below and above the 64-key tile, GQA row packing over two MMA
tiles, every mask and score modification, empty sequences, bad device inputs, and the
full-size workload on sampled heads."""
import numpy as np
import pytest
import torch

from oracle import decode_oracle as D
from tests import helpers as H
from workloads import (MASK_CAUSAL, MASK_NONE, MASK_SLIDING_WINDOW, PAGED_DECODE,
                       SCORE_ALIBI, SCORE_SOFTCAP, DecodeWorkload, make_decode_inputs)

pytestmark = pytest.mark.gpu

LENGTHS = (0, 1, 63, 64, 65, 200, 700)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _w(**kw):
    base = dict(name="decode", seed=21, B=len(LENGTHS), Hq=8, Hkv=2, Nq=1, d=128, len_min=0,
                len_max=max(LENGTHS), page_size=16, lengths=LENGTHS)
    base.update(kw)
    if "lengths" in kw and kw["lengths"] is not None:
        base["B"] = len(kw["lengths"])
        base["len_max"] = max(kw["lengths"])
    return DecodeWorkload(**base)


def _run(w, split_keys, inputs=None, max_seq_len=None):
    import exact_io_aware_13_gb300 as ea
    q, kc, vc, table, lens = inputs if inputs is not None else make_decode_inputs(
        w, poison_unused=True)
    msl = max_seq_len if max_seq_len is not None else int(table.shape[1] * w.page_size)
    o, lse = ea.decode_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), lens.cuda(),
                             max_seq_len=msl, split_keys=split_keys, scale=w.scale,
                             mask_kind=w.mask_kind, window=w.window, score_kind=w.score_kind,
                             softcap=w.softcap)
    torch.cuda.synchronize()
    status = ea.device_status()
    return o.float().cpu().numpy(), lse.cpu().numpy(), status, (q, kc, vc, table, lens)


def _check(w, o, lse, inputs, heads=None, what=""):
    q, kc, vc, table, lens = inputs
    o_ref, l_ref = D.decode_forward(q, kc, vc, table, lens, w.scale, w.mask_kind, w.window,
                                    w.score_kind, w.softcap, heads=heads)
    todo = heads or [(b, h) for b in range(w.B) for h in range(w.Hq)]
    bi = [b for b, _ in todo]
    hi = [h for _, h in todo]
    return H.check_forward(o[bi, hi], lse[bi, hi], o_ref[bi, hi], l_ref[bi, hi], what)


@pytest.mark.parametrize("split_keys", [64, 256, 1 << 20])
@pytest.mark.parametrize("page_size", [8, 16, 64, 128])
def test_decode_pages_and_splits(page_size, split_keys):
    w = _w(page_size=page_size)
    o, lse, status, inputs = _run(w, split_keys)
    assert status == 0
    _check(w, o, lse, inputs, what=f"page {page_size} split {split_keys}")


@pytest.mark.parametrize("score", [0, SCORE_ALIBI, SCORE_SOFTCAP, SCORE_ALIBI | SCORE_SOFTCAP])
@pytest.mark.parametrize("mask,window", [(MASK_NONE, 0), (MASK_CAUSAL, 0),
                                         (MASK_SLIDING_WINDOW, 100), (MASK_SLIDING_WINDOW, 0)])
@pytest.mark.parametrize("nq", [1, 3])
def test_decode_masks_and_scores(mask, window, score, nq):
    w = _w(Nq=nq, mask_kind=mask, window=window, score_kind=score, softcap=7.0, seed=30 + nq)
    o, lse, status, inputs = _run(w, 128)
    assert status == 0
    _check(w, o, lse, inputs, what=f"mask {mask} W {window} score {score} nq {nq}")


@pytest.mark.parametrize("d", [64, 128])
def test_decode_two_row_tiles_and_head_dims(d):
    """G * Nq = 4 * 40 = 160 packed rows: two 128-row MMA tiles per (sequence, kv head)."""
    w = _w(Hq=8, Hkv=2, Nq=40, d=d, mask_kind=MASK_CAUSAL, lengths=(40, 41, 300, 1000),
           page_size=32, seed=40 + d)
    o, lse, status, inputs = _run(w, 192)
    assert status == 0
    _check(w, o, lse, inputs, what=f"two row tiles d={d}")


def test_decode_more_queries_than_keys():
    """Nq > seq_len: the first queries sit at negative positions and see no key."""
    w = _w(Nq=5, mask_kind=MASK_CAUSAL, lengths=(2, 0, 5, 9), page_size=8)
    o, lse, status, inputs = _run(w, 64)
    assert status == 0
    _check(w, o, lse, inputs, what="Nq > seq_len")


MANY_LENGTHS = (0, 3, 64, 129, 300, 517, 700, 845, 1000, 1100, 1280, 1400, 1500, 1663, 1789,
                2000)


@pytest.mark.parametrize("mask,window", [(MASK_NONE, 0), (MASK_CAUSAL, 0),
                                         (MASK_SLIDING_WINDOW, 50), (MASK_SLIDING_WINDOW, 700)])
@pytest.mark.parametrize("nq,page_size", [(1, 16), (3, 64)])
def test_decode_many_items(mask, window, nq, page_size):
    """Sixteen sequences of 0-2000 tokens over four kv heads at 128 keys per chunk: several
    work items per CTA, CTA shares that begin and end in every kind of item (full chunks,
    short last chunks, sequences of one chunk), and with a short sliding window chunks
    that hold keys of no row."""
    w = _w(Hq=16, Hkv=4, Nq=nq, lengths=MANY_LENGTHS, page_size=page_size, mask_kind=mask,
           window=window, score_kind=SCORE_ALIBI, seed=60 + nq + window)
    o, lse, status, inputs = _run(w, 128)
    assert status == 0
    _check(w, o, lse, inputs, what=f"many items mask {mask} W {window} nq {nq}")


def test_decode_no_cache_at_all():
    w = _w(lengths=(0, 0))
    o, lse, status, inputs = _run(w, 256, max_seq_len=0)
    assert status == 0
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_decode_is_deterministic():
    w = _w(score_kind=SCORE_ALIBI, seed=50)
    inputs = make_decode_inputs(w, poison_unused=True)
    o1, l1, s1, _ = _run(w, 64, inputs=inputs)
    o2, l2, s2, _ = _run(w, 64, inputs=inputs)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_decode_bad_device_inputs_are_reported():
    """A page index outside the pool and a length above max_seq_len are caught on the
    device (the copies for them are skipped) and reported by attn_device_status."""
    from exact_io_aware_13_gb300 import _lib
    w = _w(lengths=(100, 300))
    q, kc, vc, table, lens = make_decode_inputs(w)
    bad_table = table.clone()
    bad_table[1, 2] = kc.shape[0] + 5
    _, _, status, _ = _run(w, 64, inputs=(q, kc, vc, bad_table, lens))
    assert status == 8  # ATTN_ERR_DEVICE_INPUT
    bad_lens = lens.clone()
    bad_lens[0] = 10_000
    _, _, status, _ = _run(w, 64, inputs=(q, kc, vc, table, bad_lens))
    assert status == 8
    # and the next clean call reports nothing
    _, _, status, _ = _run(w, 64, inputs=(q, kc, vc, table, lens))
    assert status == 0
    assert _lib.STATUS_NAMES[8] == "ATTN_ERR_DEVICE_INPUT"


def test_decode_rejects_bad_arguments():
    import exact_io_aware_13_gb300 as ea
    from exact_io_aware_13_gb300 import _lib
    w = _w(lengths=(10,))
    q, kc, vc, table, lens = [t.cuda() for t in make_decode_inputs(w)]
    for kw, status in [(dict(split_keys=100), 1), (dict(mask_kind=3), 1),
                       (dict(max_seq_len=10_000), 2)]:
        args = dict(max_seq_len=int(table.shape[1] * w.page_size), split_keys=64)
        args.update(kw)
        with pytest.raises(_lib.AttnError) as e:
            ea.decode_paged(q, kc, vc, table, lens, **args)
        assert e.value.status == status
    kc12 = torch.empty((kc.shape[0], w.Hkv, 12, w.d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.AttnError) as e:
        ea.decode_paged(q, kc12, kc12.clone(), table, lens, max_seq_len=12, split_keys=64)
    assert e.value.status == 2


def test_decode_full_size_sampled():
    """The decode workload (B=64, Hq=32, Hkv=8, lengths up to 8192, page 64) in the
    launch configuration the benchmark times, checked on sampled heads."""
    import exact_io_aware_13_gb300 as ea
    w = PAGED_DECODE
    q, kc, vc, table, lens = make_decode_inputs(w)
    split = ea.decode_split_keys(w.B, w.Hq, w.Hkv, w.Nq, int(lens.sum()))
    inputs = (q, kc, vc, table, lens)
    o, lse, status, _ = _run(w, split, inputs=inputs, max_seq_len=w.len_max)
    assert status == 0
    rng = np.random.default_rng(0)
    longest = int(np.argmax(lens.numpy()))
    heads = sorted({(longest, 0), (longest, w.Hq - 1), (0, 5)} |
                   {(int(b), int(h)) for b, h in zip(rng.integers(0, w.B, 5),
                                                     rng.integers(0, w.Hq, 5))})
    _check(w, o, lse, inputs, heads=heads, what="paged decode full size")
