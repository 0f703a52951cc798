"""GPU parity of dropout on P against the float64 oracle on the same seeded inputs.

The keep mask is integer work and is compared bit for bit: with q = 0 every allowed key
of a row gets the same probability, V (and dO) one-hot in the key (query) position mod
128 and a sliding window of 128 keys put each (query, key) pair of the band in its own
output element, so O is nonzero exactly where the forward kept the pair and dV exactly
where the backward's dK/dV kernel regenerated a kept pair. The values are checked with
the forward bound relative to each output element's scale (tests/helpers.py states it)
and the backward tolerance of the other parity tests, for every mask and score variant, d = 64 and 128, GQA, ragged and unequal lengths, several rates, and the
fwd+bwd workload at full size on a sampled kv head."""
import numpy as np
import pytest
import torch

from oracle import philox
from tests import helpers as H
from workloads import (CAUSAL_FWD_BWD_DROPOUT, MASK_CAUSAL, MASK_DOCUMENT_CAUSAL, MASK_NONE,
                       MASK_SLIDING_WINDOW, SCORE_ALIBI, SCORE_SOFTCAP, make_inputs)

pytestmark = pytest.mark.gpu

MASKS = [MASK_NONE, MASK_CAUSAL, MASK_SLIDING_WINDOW, MASK_DOCUMENT_CAUSAL]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _drop(w, p, seed):
    return w.replace(dropout_p=p, dropout_seed=seed)


def _oracle(w, inputs, rows=None, heads=None):
    """Oracle O and LSE plus each element's output scale A = (P Z / (1 - p)) |V|: the
    oracle's forward with |V| in place of V (same mask, same keep mask)."""
    o_ref, l_ref = H.oracle_forward(w, inputs, rows=rows, heads=heads)
    q, k, v, do, offs = inputs
    a_ref, _ = H.oracle_forward(w, (q, k, v.float().abs(), do, offs), rows=rows, heads=heads)
    return o_ref, l_ref, a_ref


def _check_forward(w, o, lse, o_ref, l_ref, a_ref, what):
    """|dO| <= 1e-2 * max(1, A) per element: the bound relative to the output's scale."""
    H.check_forward(o, lse, o_ref, l_ref, what, o_scale=a_ref)


def test_keep_mask_bit_exact_forward_and_dkdv():
    import exact_io_aware_13_gb300 as ea
    B, Hq, N, d, W, p, seed = 2, 2, 2048, 128, 128, 0.3, 0xDEADBEEF12345678
    g = torch.Generator().manual_seed(3)
    q = torch.zeros(B, Hq, N, d, dtype=torch.bfloat16)
    k = torch.randn(B, Hq, N, d, generator=g).to(torch.bfloat16)
    onehot = torch.zeros(N, d, dtype=torch.bfloat16)
    onehot[torch.arange(N), torch.arange(N) % d] = 1
    v = onehot.expand(B, Hq, N, d).contiguous()
    qd, kd, vd, dod = H.to_dev(q, k, v, v.clone())
    kw = dict(scale=0.125, mask_kind=MASK_SLIDING_WINDOW, window=W, dropout_p=p,
              dropout_seed=seed)
    o, lse = ea.forward(qd, kd, vd, **kw)
    dq, dk, dv = ea.backward(qd, kd, vd, o, lse, dod, **kw)
    torch.cuda.synchronize()
    assert ea.device_status() == 0
    o = o.float().cpu().numpy()
    dv = dv.float().cpu().numpy()
    i = np.arange(N)[:, None]
    c = np.arange(d)[None, :]
    j_of = i - (i - c) % W                       # the key of column c seen by row i
    i_of = (i + (c - i) % W)                     # the query of column c that sees key i
    for b in range(B):
        for h in range(Hq):
            keep = philox.keep_mask(seed, b * Hq + h, np.arange(N), np.arange(N), p)
            want_o = (j_of >= 0) & keep[np.arange(N)[:, None], np.maximum(j_of, 0)]
            assert np.array_equal(o[b, h] != 0, want_o), f"forward mask b={b} h={h}"
            want_dv = (i_of < N) & keep[np.minimum(i_of, N - 1), np.arange(N)[:, None]]
            assert np.array_equal(dv[b, h] != 0, want_dv), f"dV mask b={b} h={h}"
            rate = want_o[W:].mean()
            assert abs(rate - (1 - 76 / 256)) < 0.01
    assert np.isfinite(dq.float().cpu().numpy()).all()
    assert np.isfinite(dk.float().cpu().numpy()).all()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("score", [0, SCORE_ALIBI | SCORE_SOFTCAP])
@pytest.mark.parametrize("mask", MASKS)
def test_dropout_variants(mask, score, d):
    w = H.small_workload(f"drop m{mask}s{score}d{d}", mask, score, d=d, N=300,
                         window=200 if mask == MASK_SLIDING_WINDOW else 0,
                         softcap=20.0 if score & SCORE_SOFTCAP else 0.0,
                         seed=300 + 10 * mask + score + d)
    w = _drop(w, 0.2, 1000 + mask)
    inputs = make_inputs(w, with_dout=True)
    o, lse = H.run_forward(w, "tc", inputs)
    _check_forward(w, o, lse, *_oracle(w, inputs), w.name)
    H.check_grads(H.run_backward(w, "tc", inputs), H.oracle_backward(w, inputs), w.name)


@pytest.mark.parametrize("p", [0.05, 0.5, 0.9])
def test_dropout_rates_gqa(p):
    w = H.small_workload(f"drop p{p}", MASK_CAUSAL, B=2, Hq=8, Hkv=2, N=400, d=128,
                         seed=int(p * 100))
    w = _drop(w, p, 77)
    inputs = make_inputs(w, with_dout=True)
    o, lse = H.run_forward(w, "tc", inputs)
    _check_forward(w, o, lse, *_oracle(w, inputs), w.name)
    H.check_grads(H.run_backward(w, "tc", inputs), H.oracle_backward(w, inputs), w.name)


@pytest.mark.parametrize("nq,nkv", [(200, 450), (450, 200), (1, 129), (129, 1)])
def test_dropout_unequal_lengths(nq, nkv):
    """p = 0.5: its scale 2 is exact, so with one key O = 2 V (or 0) is stored exactly
    and D = rowsum(dO o O) equals dP Z / (1 - p); the exact dQ and dK of that case
    vanish and the kernels' must too, up to the floor of the other tests. (At a rate
    whose 1 / (1 - p) is inexact, the bf16 rounding of the stored O enters D and
    leaves gradients of the order of that rounding where the exact ones are 0.)"""
    w = H.small_workload(f"drop {nq}x{nkv}", MASK_NONE, B=1, Hq=4, Hkv=1, N=nq, Nkv=nkv,
                         d=128, seed=nq + 2 * nkv)
    w = _drop(w, 0.5, 5)
    inputs = make_inputs(w, with_dout=True)
    o, lse = H.run_forward(w, "tc", inputs)
    _check_forward(w, o, lse, *_oracle(w, inputs), w.name)
    H.check_grads(H.run_backward(w, "tc", inputs), H.oracle_backward(w, inputs), w.name)


def test_dropout_rate_zero_equals_no_dropout():
    """score_kind with the dropout bit and p = 0 keeps every element with scale 1."""
    import exact_io_aware_13_gb300 as ea
    w = H.small_workload("p0", MASK_CAUSAL, SCORE_ALIBI, B=1, Hq=4, Hkv=2, N=333, d=128)
    q, k, v, do, _ = make_inputs(w, with_dout=True)
    qd, kd, vd, dod = H.to_dev(q, k, v, do)
    kw = dict(scale=w.scale, mask_kind=MASK_CAUSAL)
    o0, l0 = ea.forward(qd, kd, vd, score_kind=SCORE_ALIBI, **kw)
    o1, l1 = torch.empty_like(o0), torch.empty_like(l0)
    ea.fwd_into(qd, kd, vd, o1, l1, score_kind=SCORE_ALIBI | ea.SCORE_DROPOUT,
                dropout_p=0.0, dropout_seed=123, **kw)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    g0 = ea.backward(qd, kd, vd, o0, l0, dod, score_kind=SCORE_ALIBI, **kw)
    ws = torch.empty(max(ea.bwd_workspace_size(qd, kd), 256), dtype=torch.uint8,
                     device="cuda")
    g1 = [torch.empty_like(t) for t in g0]
    ea.bwd_into(qd, kd, vd, o0, l0, dod, *g1, ws, score_kind=SCORE_ALIBI | ea.SCORE_DROPOUT,
                dropout_p=0.0, dropout_seed=123, **kw)
    torch.cuda.synchronize()
    for a, b in zip(g0, g1):
        a, b = a.float(), b.float()
        assert (a - b).abs().max() <= 1e-6 * a.abs().max()


def test_dropout_is_deterministic_and_follows_the_seed():
    import exact_io_aware_13_gb300 as ea
    w = H.small_workload("seeded", MASK_CAUSAL, B=1, Hq=2, Hkv=2, N=256, d=64)
    q, k, v, do, _ = make_inputs(w, with_dout=True)
    qd, kd, vd, dod = H.to_dev(q, k, v, do)

    def run(seed):
        o, lse = ea.forward(qd, kd, vd, scale=w.scale, mask_kind=MASK_CAUSAL, dropout_p=0.5,
                            dropout_seed=seed)
        g = ea.backward(qd, kd, vd, o, lse, dod, scale=w.scale, mask_kind=MASK_CAUSAL,
                        dropout_p=0.5, dropout_seed=seed)
        torch.cuda.synchronize()
        return [t.float().cpu() for t in (o, *g)]

    a, b = run(1 << 40), run(1 << 40)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    c = run((1 << 40) + (1 << 33))              # differs in the high word only
    d = run((1 << 40) + 1)                      # differs in the low word only
    assert not torch.equal(a[0], c[0]) and not torch.equal(a[0], d[0])


def test_dropout_rejected_where_not_supported():
    import exact_io_aware_13_gb300 as ea
    from exact_io_aware_13_gb300 import _lib
    w = H.small_workload("rej", MASK_NONE, B=1, Hq=2, Hkv=2, N=128, d=128)
    q, k, v, do, _ = [t if t is None else t.cuda() for t in make_inputs(w, with_dout=True)]
    with pytest.raises(_lib.AttnError) as e:
        ea.forward(q, k, v, dropout_p=0.1, dropout_seed=1, impl="simt")
    assert e.value.status == 1
    (q8, sq), (k8, sk), (v8t, sv) = ea.fp8_inputs(q, k, v)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
    with pytest.raises(_lib.AttnError) as e:
        ea.fwd_fp8_into(q8, sq, k8, sk, v8t, sv, o, lse, Nkv=w.Nkv, scale=w.scale,
                        score_kind=ea.SCORE_DROPOUT)
    assert e.value.status == 1
    q256 = torch.zeros(1, 2, 128, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.AttnError) as e:
        ea.forward(q256, q256, q256, dropout_p=0.1)
    assert e.value.status == 1


def test_dropout_full_size_sampled_kv_head():
    """The dropout fwd+bwd workload (B=2, H=16, N=8192, d=128, causal, p=0.1) in the
    launch configuration the benchmark times; O on sampled rows of two heads and
    dq/dk/dv of one kv head against the oracle."""
    w = CAUSAL_FWD_BWD_DROPOUT
    inputs = make_inputs(w)
    o, lse = H.run_forward(w, "tc", inputs)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 4096, w.Nq - 1],
                                     rng.integers(0, w.Nq, 24)]))
    heads = [(0, 3), (w.B - 1, w.Hq - 1)]
    o_ref, l_ref, a_ref = _oracle(w, inputs, rows=rows, heads=heads)
    for b, h in heads:
        _check_forward(w, o[b, h][rows], lse[b, h][rows], o_ref[b, h], l_ref[b, h],
                       a_ref[b, h], f"{w.name} b={b} h={h}")
    got = H.run_backward(w, "tc", inputs)
    b, g = w.B - 1, 5
    ref = H.oracle_backward(w, inputs, kv_heads=[(b, g)])
    H.check_grads([x[b, g:g + 1] for x in got], [x[b, g:g + 1] for x in ref], w.name)


def test_dropout_backward_phases_match_one_call():
    """The row kernel, the dK/dV kernel and the dQ kernel run one at a time through
    attn_bwd_phases (the launches the benchmark times) give the bits of attn_bwd."""
    import exact_io_aware_13_gb300 as ea
    w = _drop(H.small_workload("drop phases", MASK_CAUSAL, SCORE_ALIBI, B=1, Hq=4, Hkv=2,
                               N=330, d=64, seed=17), 0.3, 99)
    q, k, v, do, _ = make_inputs(w, with_dout=True)
    qd, kd, vd, dod = H.to_dev(q, k, v, do)
    kw = dict(scale=w.scale, mask_kind=w.mask_kind, score_kind=w.score_kind,
              dropout_p=w.dropout_p, dropout_seed=w.dropout_seed)
    o, lse = ea.forward(qd, kd, vd, **kw)
    g1 = ea.backward(qd, kd, vd, o, lse, dod, **kw)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(max(ea.bwd_workspace_size(qd, kd), 256), dtype=torch.uint8, device="cuda")
    for ph in (ea.BWD_ROWDOT, ea.BWD_DKDV, ea.BWD_DQ):
        ea.bwd_phases_into(ph, qd, kd, vd, o, lse, dod, dq, dk, dv, ws, **kw)
    torch.cuda.synchronize()
    assert ea.device_status() == 0
    for a, b in zip(g1, (dq, dk, dv)):
        assert torch.equal(a, b)
