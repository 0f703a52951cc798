"""GPU parity: the library's forward and backward against the float64 oracle, on the
same seeded inputs, for every mask x score variant, several tiles plus a ragged
tail, GQA, d = 64 and 128, and the full-size workloads on sampled rows/heads."""
import numpy as np
import pytest
import torch

from tests import helpers as H
from workloads import (CAUSAL, CAUSAL_FWD_BWD, DOCS, GQA_WINDOW, MASK_CAUSAL,
                       MASK_DOCUMENT_CAUSAL, MASK_NONE, MASK_SLIDING_WINDOW, SCORE_ALIBI,
                       SCORE_SOFTCAP, TINY, make_inputs)

pytestmark = pytest.mark.gpu

MASKS = [MASK_NONE, MASK_CAUSAL, MASK_SLIDING_WINDOW, MASK_DOCUMENT_CAUSAL]
SCORES = [0, SCORE_ALIBI, SCORE_SOFTCAP, SCORE_ALIBI | SCORE_SOFTCAP]


def _variant(mask, score, d, N=300, **kw):
    return H.small_workload(f"m{mask}s{score}d{d}", mask, score, d=d, N=N,
                            window=200 if mask == MASK_SLIDING_WINDOW else 0,
                            softcap=(20.0 if score & SCORE_SOFTCAP else 0.0),
                            seed=100 + 10 * mask + score + d, **kw)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


# ------------------------------------------------------------------ forward

@pytest.mark.parametrize("impl", ["tc", "simt"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("score", SCORES)
@pytest.mark.parametrize("mask", MASKS)
def test_forward_variants(mask, score, d, impl):
    w = _variant(mask, score, d, N=300 if d == 64 else 700)
    inputs = make_inputs(w)
    o, lse = H.run_forward(w, impl, inputs)
    o_ref, l_ref = H.oracle_forward(w, inputs)
    H.check_forward(o, lse, o_ref, l_ref, w.name)


@pytest.mark.parametrize("nq,nkv", [(200, 450), (450, 200), (1, 129), (129, 1), (513, 513)])
@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_SLIDING_WINDOW])
def test_forward_ragged_and_unequal_lengths(nq, nkv, mask):
    w = H.small_workload(f"ragged{nq}x{nkv}", mask, B=2, Hq=2, Hkv=1, N=nq, Nkv=nkv, d=128,
                         window=150, seed=nq + nkv)
    inputs = make_inputs(w)
    o, lse = H.run_forward(w, "tc", inputs)
    o_ref, l_ref = H.oracle_forward(w, inputs)
    H.check_forward(o, lse, o_ref, l_ref, w.name)


def test_forward_tiny_workload():
    inputs = make_inputs(TINY)
    o, lse = H.run_forward(TINY, "tc", inputs)
    o_ref, l_ref = H.oracle_forward(TINY, inputs)
    H.check_forward(o, lse, o_ref, l_ref, TINY.name)


def test_forward_fully_masked_rows_and_no_keys():
    w = H.small_workload("w0", MASK_SLIDING_WINDOW, window=0, N=260, d=64)
    o, lse = H.run_forward(w, "tc")
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    w = H.small_workload("nokeys", MASK_NONE, N=130, Nkv=0, d=64)
    o, lse = H.run_forward(w, "tc")
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_forward_large_logits_stay_finite():
    """Scores of several hundred (inputs scaled up): the online max keeps exp2 in
    range; compare with the oracle."""
    w = H.small_workload("big", MASK_CAUSAL, N=384, d=128, seed=3)
    q, k, v, do, offs = make_inputs(w)
    q = (q.float() * 8).to(torch.bfloat16)
    k = (k.float() * 8).to(torch.bfloat16)
    inputs = (q, k, v, do, offs)
    o, lse = H.run_forward(w, "tc", inputs)
    o_ref, l_ref = H.oracle_forward(w, inputs)
    H.check_forward(o, lse, o_ref, l_ref, w.name)


@pytest.mark.parametrize("score", [SCORE_SOFTCAP, SCORE_ALIBI | SCORE_SOFTCAP],
                         ids=["softcap", "alibi_softcap"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_softcap_saturated_scores(score, d):
    """Scores of a few hundred against a soft-cap of 20 (s / c up to about 20, where tanh is
    saturated and the capped scores of many keys sit near the cap): the kernels' tanh,
    scaled by c, feeds every P here. Forward and gradients against the oracle, which
    takes numpy's tanh."""
    w = H.small_workload(f"capsat{d}", MASK_CAUSAL, score, B=1, Hq=4, Hkv=2, N=300, d=d,
                         softcap=20.0, seed=11 + d)
    q, k, v, do, offs = make_inputs(w, with_dout=True)
    q = (q.float() * 8).to(torch.bfloat16)
    k = (k.float() * 8).to(torch.bfloat16)
    inputs = (q, k, v, do, offs)
    o, lse = H.run_forward(w, "tc", inputs)
    o_ref, l_ref = H.oracle_forward(w, inputs)
    H.check_forward(o, lse, o_ref, l_ref, w.name)
    got = H.run_backward(w, "tc", inputs)
    H.check_grads(got, H.oracle_backward(w, inputs), w.name)


def _sampled_rows(w, n=48, seed=0):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, w.Nq - 1],
                                     rng.integers(0, w.Nq, n)]))
    return rows


@pytest.mark.parametrize("w", [CAUSAL, GQA_WINDOW, DOCS], ids=["causal", "gqa_window", "docs"])
def test_forward_full_size_sampled(w):
    """The full workload in the bench's launch configuration, checked on sampled
    rows of a few heads (the oracle evaluates just those rows)."""
    inputs = make_inputs(w)
    o, lse = H.run_forward(w, "tc", inputs)
    rows = _sampled_rows(w)
    heads = [(0, 0), (w.B - 1, w.Hq - 1), (0, w.Hq // 2)]
    o_ref, l_ref = H.oracle_forward(w, inputs, rows=rows, heads=heads)
    for b, h in heads:
        H.check_forward(o[b, h][rows], lse[b, h][rows], o_ref[b, h], l_ref[b, h],
                        f"{w.name} b={b} h={h}")
    assert np.isfinite(o).all()
    fin = np.isfinite(lse)
    assert fin.all() or w.mask_kind != MASK_CAUSAL


# ------------------------------------------------------------------ backward

@pytest.mark.parametrize("impl", ["tc", "simt"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("score", SCORES)
@pytest.mark.parametrize("mask", MASKS)
def test_backward_variants(mask, score, d, impl):
    w = _variant(mask, score, d, N=300 if d == 64 else 520)
    inputs = make_inputs(w, with_dout=True)
    got = H.run_backward(w, impl, inputs)
    ref = H.oracle_backward(w, inputs)
    H.check_grads(got, ref, w.name)


@pytest.mark.parametrize("nq,nkv", [(200, 450), (450, 200), (129, 1)])
def test_backward_unequal_lengths(nq, nkv):
    w = H.small_workload(f"bwd{nq}x{nkv}", MASK_CAUSAL, B=1, Hq=4, Hkv=1, N=nq, Nkv=nkv, d=128,
                         seed=nq * 3 + nkv)
    inputs = make_inputs(w, with_dout=True)
    got = H.run_backward(w, "tc", inputs)
    H.check_grads(got, H.oracle_backward(w, inputs), w.name)


def test_backward_full_size_sampled_heads():
    """fwd+bwd workload at full size; dq/dk/dv of two kv heads against the oracle."""
    w = CAUSAL_FWD_BWD
    inputs = make_inputs(w)
    got = H.run_backward(w, "tc", inputs)
    heads = [(0, 0), (w.B - 1, w.Hkv - 1)]
    ref = H.oracle_backward(w, inputs, kv_heads=heads)
    for b, g in heads:
        H.check_grads([got[0][b, g:g + 1], got[1][b, g:g + 1], got[2][b, g:g + 1]],
                      [ref[0][b, g:g + 1], ref[1][b, g:g + 1], ref[2][b, g:g + 1]],
                      f"{w.name} b={b} g={g}")


# ------------------------------------------------------------------ tile classifier

@pytest.mark.parametrize("mask,nq,nkv,window", [(MASK_NONE, 300, 500, 0),
                                                (MASK_CAUSAL, 1000, 1000, 0),
                                                (MASK_SLIDING_WINDOW, 16384, 16384, 1024),
                                                (MASK_SLIDING_WINDOW, 700, 700, 129),
                                                (MASK_DOCUMENT_CAUSAL, 32768, 32768, 0)])
def test_classify_tiles_matches_brute_force(mask, nq, nkv, window):
    import exact_io_aware_13_gb300 as ea
    from oracle import attention_oracle as ref
    from workloads import document_offsets
    offs = document_offsets(nq, 3) if mask == MASK_DOCUMENT_CAUSAL else None
    got = ea.classify_tiles(mask, nq, nkv, window=window, doc_offsets=H.doc_tensor(offs))
    brute = ref.classify_tiles(mask, nq, nkv, 128, 128, window, offs)
    assert (got.cpu().numpy() == brute).all()
