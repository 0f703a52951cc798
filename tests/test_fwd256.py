"""GPU parity of the head-dimension-256 forward (attn_fwd with d = 256) against the
float64 oracle on the same seeded inputs: every mask x score variant, GQA, query tiles
of 128 rows against key tiles of 64 with ragged tails, unequal lengths, rows with no
key, large logits, and the full-size workload on sampled rows. Tolerances: forward's
(max|dO| <= 1e-2, max|dLSE| <= 1e-3, -inf exactly where the oracle has it)."""
import numpy as np
import pytest
import torch

from tests import helpers as H
from workloads import (CAUSAL_D256, MASK_CAUSAL, MASK_DOCUMENT_CAUSAL, MASK_NONE,
                       MASK_SLIDING_WINDOW, SCORE_ALIBI, SCORE_SOFTCAP, make_inputs)

pytestmark = pytest.mark.gpu

MASKS = [MASK_NONE, MASK_CAUSAL, MASK_SLIDING_WINDOW, MASK_DOCUMENT_CAUSAL]
SCORES = [0, SCORE_ALIBI, SCORE_SOFTCAP, SCORE_ALIBI | SCORE_SOFTCAP]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("score", SCORES)
@pytest.mark.parametrize("mask", MASKS)
def test_forward256_variants(mask, score):
    w = H.small_workload(f"d256m{mask}s{score}", mask, score, B=2, Hq=4, Hkv=2, N=520, d=256,
                         window=150 if mask == MASK_SLIDING_WINDOW else 0,
                         softcap=20.0 if score & SCORE_SOFTCAP else 0.0, seed=500 + 10 * mask + score)
    inputs = make_inputs(w)
    o, lse = H.run_forward(w, "tc", inputs)
    o_ref, l_ref = H.oracle_forward(w, inputs)
    H.check_forward(o, lse, o_ref, l_ref, w.name)


@pytest.mark.parametrize("nq,nkv", [(1, 65), (65, 1), (200, 450), (450, 200), (129, 129)])
@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_SLIDING_WINDOW])
def test_forward256_ragged_and_unequal_lengths(nq, nkv, mask):
    w = H.small_workload(f"d256ragged{nq}x{nkv}", mask, B=1, Hq=2, Hkv=1, N=nq, Nkv=nkv, d=256,
                         window=100, seed=nq + 7 * nkv)
    inputs = make_inputs(w)
    o, lse = H.run_forward(w, "tc", inputs)
    o_ref, l_ref = H.oracle_forward(w, inputs)
    H.check_forward(o, lse, o_ref, l_ref, w.name)


def test_forward256_no_keys_and_empty_windows():
    w = H.small_workload("d256w0", MASK_SLIDING_WINDOW, window=0, N=200, d=256)
    o, lse = H.run_forward(w, "tc")
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    w = H.small_workload("d256nokeys", MASK_NONE, N=130, Nkv=0, d=256)
    o, lse = H.run_forward(w, "tc")
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_forward256_large_logits_stay_finite():
    w = H.small_workload("d256big", MASK_CAUSAL, N=400, d=256, seed=9)
    q, k, v, do, offs = make_inputs(w)
    inputs = ((q.float() * 6).to(torch.bfloat16), (k.float() * 6).to(torch.bfloat16), v, do, offs)
    o, lse = H.run_forward(w, "tc", inputs)
    o_ref, l_ref = H.oracle_forward(w, inputs)
    H.check_forward(o, lse, o_ref, l_ref, w.name)


def test_forward256_is_deterministic():
    w = H.small_workload("d256det", MASK_CAUSAL, SCORE_ALIBI, N=700, d=256, seed=11)
    inputs = make_inputs(w)
    o1, l1 = H.run_forward(w, "tc", inputs)
    o2, l2 = H.run_forward(w, "tc", inputs)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_simt_and_dropout_reject_d256():
    import exact_io_aware_13_gb300 as ea
    from exact_io_aware_13_gb300 import _lib
    w = H.small_workload("d256rej", MASK_CAUSAL, N=64, d=256)
    q, k, v, do, _ = make_inputs(w, with_dout=True)
    q, k, v, do = (t.cuda() for t in (q, k, v, do))
    with pytest.raises(_lib.AttnError) as e:
        ea.forward(q, k, v, scale=w.scale, impl="simt")
    assert e.value.status == 2
    o, lse = ea.forward(q, k, v, scale=w.scale)
    with pytest.raises(_lib.AttnError) as e:
        ea.backward(q, k, v, o, lse, do, scale=w.scale, impl="simt")
    assert e.value.status == 2
    with pytest.raises(_lib.AttnError) as e:
        ea.backward(q, k, v, o, lse, do, scale=w.scale, dropout_p=0.1)
    assert e.value.status == 1


def test_forward256_full_size_sampled():
    """Causal B=2 H=16 N=8192 d=256 in the bench's launch configuration, sampled rows."""
    w = CAUSAL_D256
    inputs = make_inputs(w)
    o, lse = H.run_forward(w, "tc", inputs)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 1, 63, 64, 127, 128, 4095, w.Nq - 1], rng.integers(0, w.Nq, 40)]))
    heads = [(0, 0), (w.B - 1, w.Hq - 1)]
    o_ref, l_ref = H.oracle_forward(w, inputs, rows=rows, heads=heads)
    for b, h in heads:
        H.check_forward(o[b, h][rows], lse[b, h][rows], o_ref[b, h], l_ref[b, h],
                        f"{w.name} b={b} h={h}")
    assert np.isfinite(o).all() and np.isfinite(lse).all()
