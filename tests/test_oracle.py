"""Pins for the float64 oracle (CPU only).

Each test checks the oracle against something other than itself: closed forms,
invariants the definition forces, a library routine (torch float64 SDPA, logsumexp
and autograd), central finite differences, or brute-force counts. A plausible
mistake in the oracle (a dropped term, a wrong sign or index, a transposed operand,
a wrong head map) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention_oracle as ref
from workloads import (MASK_CAUSAL, MASK_DOCUMENT_CAUSAL, MASK_NONE, MASK_SLIDING_WINDOW,
                       SCORE_ALIBI, SCORE_SOFTCAP, document_lengths, document_offsets,
                       offsets_from_lengths)

MASKS = [MASK_NONE, MASK_CAUSAL, MASK_SLIDING_WINDOW, MASK_DOCUMENT_CAUSAL]
SCORES = [0, SCORE_ALIBI, SCORE_SOFTCAP, SCORE_ALIBI | SCORE_SOFTCAP]


def _rand(shape, seed, scale=1.0):
    g = torch.Generator("cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float64) * scale).numpy()


def _mask_args(mask, n):
    if mask == MASK_SLIDING_WINDOW:
        return dict(window=max(2, n // 3))
    if mask == MASK_DOCUMENT_CAUSAL:
        return dict(doc_offsets=offsets_from_lengths([n // 3, n // 2, n - n // 3 - n // 2]))
    return {}


def _score_args(score):
    return dict(score_kind=score, softcap=(5.0 if score & SCORE_SOFTCAP else 0.0))


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("score", SCORES)
def test_rows_of_p_sum_to_one(mask, score):
    n, d = 40, 8
    q = _rand((1, 2, n, d), 1); k = _rand((1, 2, n, d), 2)
    for h in range(2):
        p = ref.probabilities(q, k, 0.3, h_index=h, mask_kind=mask, **_mask_args(mask, n),
                              **_score_args(score))
        assert np.all(p >= 0)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)


def test_fully_masked_rows_give_zero_output_and_minus_inf_lse():
    n, d = 24, 8
    q = _rand((1, 1, n, d), 3); k = _rand((1, 1, n, d), 4); v = _rand((1, 1, n, d), 5)
    o, l = ref.forward(q, k, v, 0.25, mask_kind=MASK_SLIDING_WINDOW, window=0)
    assert np.all(o == 0.0)
    assert np.all(np.isneginf(l))
    dq, dk, dv = ref.backward(q, k, v, _rand((1, 1, n, d), 6), 0.25,
                              mask_kind=MASK_SLIDING_WINDOW, window=0)
    assert np.all(dq == 0) and np.all(dk == 0) and np.all(dv == 0)


def test_keys_outside_every_document_mask_the_row():
    # Offsets that stop short of N leave positions without a document.
    n, d = 16, 4
    q = _rand((1, 1, n, d), 7); k = _rand((1, 1, n, d), 8); v = _rand((1, 1, n, d), 9)
    o, l = ref.forward(q, k, v, 0.5, mask_kind=MASK_DOCUMENT_CAUSAL,
                       doc_offsets=[0, 5, 12])
    assert np.all(np.isneginf(l[0, 0, 12:])) and np.all(o[0, 0, 12:] == 0)
    assert np.all(np.isfinite(l[0, 0, :12]))


@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("score", SCORES)
def test_uniform_v_returns_v(mask, score):
    n, d = 33, 6
    q = _rand((1, 2, n, d), 10); k = _rand((1, 1, n, d), 11)
    row = _rand((d,), 12)
    v = np.broadcast_to(row, (1, 1, n, d)).copy()
    o, l = ref.forward(q, k, v, 0.4, mask_kind=mask, **_mask_args(mask, n),
                       **_score_args(score))
    live = np.isfinite(l)
    np.testing.assert_allclose(o[live], np.broadcast_to(row, o[live].shape), atol=1e-12)


def test_single_key_rows_return_that_value_row():
    n, d, scale = 20, 8, 0.37
    q = _rand((1, 1, n, d), 13); k = _rand((1, 1, n, d), 14); v = _rand((1, 1, n, d), 15)
    # causal row 0 sees only key 0
    o, l = ref.forward(q, k, v, scale, mask_kind=MASK_CAUSAL)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-14)
    np.testing.assert_allclose(l[0, 0, 0], scale * np.dot(q[0, 0, 0], k[0, 0, 0]), atol=1e-13)
    # window of one key: every row sees only its own position
    o, l = ref.forward(q, k, v, scale, mask_kind=MASK_SLIDING_WINDOW, window=1)
    np.testing.assert_allclose(o[0, 0], v[0, 0], atol=1e-14)
    np.testing.assert_allclose(l[0, 0], scale * np.einsum("nd,nd->n", q[0, 0], k[0, 0]),
                               atol=1e-13)
    # one-token documents: the same
    o, l = ref.forward(q, k, v, scale, mask_kind=MASK_DOCUMENT_CAUSAL,
                       doc_offsets=list(range(n + 1)))
    np.testing.assert_allclose(o[0, 0], v[0, 0], atol=1e-14)


# ---------------------------------------------------------------- closed forms

def test_zero_queries_no_mask_mean_of_v():
    n, d = 50, 5
    q = np.zeros((1, 1, n, d)); k = _rand((1, 1, n, d), 16); v = _rand((1, 1, n, d), 17)
    o, l = ref.forward(q, k, v, 0.5)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0].mean(axis=0), (n, d)),
                               atol=1e-13)
    np.testing.assert_allclose(l[0, 0], math.log(n), atol=1e-13)


def test_zero_queries_causal_prefix_means():
    n, d = 50, 5
    q = np.zeros((1, 1, n, d)); k = _rand((1, 1, n, d), 18); v = _rand((1, 1, n, d), 19)
    o, l = ref.forward(q, k, v, 0.5, mask_kind=MASK_CAUSAL)
    for i in range(n):
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :i + 1].mean(axis=0), atol=1e-13)
        np.testing.assert_allclose(l[0, 0, i], math.log(i + 1), atol=1e-13)


@pytest.mark.parametrize("h", [0, 3, 7])
def test_zero_queries_alibi_causal_geometric_weights(h):
    n, d, Hq = 40, 3, 8
    q = np.zeros((1, Hq, n, d)); k = _rand((1, 1, n, d), 20); v = _rand((1, 1, n, d), 21)
    o, l = ref.forward(q, k, v, 0.5, mask_kind=MASK_CAUSAL, score_kind=SCORE_ALIBI)
    slope = 2.0 ** (-8.0 * (h + 1) / Hq)
    r = math.exp(-slope)
    for i in range(n):
        # scores are -slope*(i-j), j = 0..i: a geometric series in r = e^-slope
        lse = math.log((1 - r ** (i + 1)) / (1 - r))
        np.testing.assert_allclose(l[0, h, i], lse, atol=1e-12)
        w = np.array([r ** (i - j) for j in range(i + 1)])
        np.testing.assert_allclose(o[0, h, i], (w[:, None] * v[0, 0, :i + 1]).sum(0) / w.sum(),
                                   atol=1e-12)


def test_zero_queries_alibi_softcap_direct_sum():
    n, d, Hq, c = 30, 3, 4, 50.0
    q = np.zeros((1, Hq, n, d)); k = _rand((1, 1, n, d), 22); v = _rand((1, 1, n, d), 23)
    o, l = ref.forward(q, k, v, 0.5, mask_kind=MASK_CAUSAL,
                       score_kind=SCORE_ALIBI | SCORE_SOFTCAP, softcap=c)
    for h in range(Hq):
        slope = 2.0 ** (-8.0 * (h + 1) / Hq)
        for i in range(n):
            total = sum(math.exp(c * math.tanh(-slope * kk / c)) for kk in range(i + 1))
            np.testing.assert_allclose(l[0, h, i], math.log(total), atol=1e-12)


def test_softcap_bounds_scores():
    # With huge logits the capped scores saturate at +-c, so the LSE is at most
    # c + log(N) and at least -c.
    n, d, c = 16, 4, 3.0
    q = _rand((1, 1, n, d), 24, 100.0); k = _rand((1, 1, n, d), 25, 100.0)
    v = _rand((1, 1, n, d), 26)
    _, l = ref.forward(q, k, v, 1.0, score_kind=SCORE_SOFTCAP, softcap=c)
    assert np.all(l <= c + math.log(n) + 1e-12) and np.all(l >= -c - 1e-12)


def test_online_softmax_recurrence_matches_direct_formula():
    """The blockwise recurrence of "El algoritmo FlashAttention" (running max,
    running normaliser, rescale by exp(m_old - m_new)), written here over key
    blocks, reaches the oracle's direct O and L to 1e-12."""
    n, d, bc = 70, 8, 16
    q = _rand((1, 1, n, d), 27); k = _rand((1, 1, n, d), 28); v = _rand((1, 1, n, d), 29)
    scale = 0.3
    o_ref, l_ref = ref.forward(q, k, v, scale, mask_kind=MASK_CAUSAL)
    for i in range(n):
        m, ell, acc = -np.inf, 0.0, np.zeros(d)
        for j0 in range(0, n, bc):
            js = np.arange(j0, min(n, j0 + bc))
            sc = scale * (k[0, 0, js] @ q[0, 0, i])
            sc = np.where(js <= i, sc, -np.inf)
            m_blk = sc.max()
            if not np.isfinite(m_blk):
                continue
            pt = np.exp(sc - m_blk)
            m_new = max(m, m_blk)
            acc = acc * math.exp(m - m_new) + (pt @ v[0, 0, js]) * math.exp(m_blk - m_new)
            ell = ell * math.exp(m - m_new) + pt.sum() * math.exp(m_blk - m_new)
            m = m_new
        np.testing.assert_allclose(acc / ell, o_ref[0, 0, i], atol=1e-12)
        np.testing.assert_allclose(m + math.log(ell), l_ref[0, 0, i], atol=1e-12)


# ---------------------------------------------------------------- library routine

def _additive_bias(mask, score, n, Hq, kw):
    """ALiBi bias plus -inf mask as a [Hq, n, n] float64 tensor for SDPA."""
    i = np.arange(n)[:, None]; j = np.arange(n)[None, :]
    bias = np.zeros((Hq, n, n))
    if score & SCORE_ALIBI:
        for h in range(Hq):
            bias[h] = -(2.0 ** (-8.0 * (h + 1) / Hq)) * (i - j)
    if mask == MASK_CAUSAL:
        ok = j <= i
    elif mask == MASK_SLIDING_WINDOW:
        ok = (j <= i) & (i - j < kw["window"])
    elif mask == MASK_DOCUMENT_CAUSAL:
        ids = np.searchsorted(np.asarray(kw["doc_offsets"]), np.arange(n), side="right") - 1
        ok = (ids[:, None] == ids[None, :]) & (j <= i)
    else:
        ok = np.ones((n, n), bool)
    return torch.from_numpy(np.where(ok[None], bias, -np.inf))


@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("score", [0, SCORE_ALIBI])
def test_forward_and_gradients_match_torch_sdpa_float64(mask, score):
    B, Hq, Hkv, n, d, scale = 2, 4, 2, 37, 16, 0.25
    q = _rand((B, Hq, n, d), 30); k = _rand((B, Hkv, n, d), 31)
    v = _rand((B, Hkv, n, d), 32); do = _rand((B, Hq, n, d), 33)
    kw = _mask_args(mask, n)
    o, l = ref.forward(q, k, v, scale, mask_kind=mask, score_kind=score, **kw)
    dq, dk, dv = ref.backward(q, k, v, do, scale, mask_kind=mask, score_kind=score, **kw)

    tq = torch.from_numpy(q).requires_grad_(); tk = torch.from_numpy(k).requires_grad_()
    tv = torch.from_numpy(v).requires_grad_()
    bias = _additive_bias(mask, score, n, Hq, kw)
    G = Hq // Hkv
    # GQA: query head h reads kv head h // G (repeat_interleave)
    ke = tk.repeat_interleave(G, dim=1); ve = tv.repeat_interleave(G, dim=1)
    to = torch.nn.functional.scaled_dot_product_attention(tq, ke, ve, attn_mask=bias,
                                                          scale=scale)
    np.testing.assert_allclose(o, to.detach().numpy(), atol=1e-12)
    tl = torch.logsumexp(scale * tq.detach() @ ke.detach().transpose(-1, -2) + bias, dim=-1)
    np.testing.assert_allclose(l, tl.numpy(), atol=1e-12)
    (to * torch.from_numpy(do)).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-10)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-10)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-10)


@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL])
def test_softcap_gradients_match_autograd(mask):
    B, Hq, Hkv, n, d, scale, c = 1, 2, 1, 21, 8, 0.9, 2.0
    q = _rand((B, Hq, n, d), 34); k = _rand((B, Hkv, n, d), 35)
    v = _rand((B, Hkv, n, d), 36); do = _rand((B, Hq, n, d), 37)
    sk = SCORE_ALIBI | SCORE_SOFTCAP
    dq, dk, dv = ref.backward(q, k, v, do, scale, mask_kind=mask, score_kind=sk, softcap=c)
    tq = torch.from_numpy(q).requires_grad_(); tk = torch.from_numpy(k).requires_grad_()
    tv = torch.from_numpy(v).requires_grad_()
    bias = _additive_bias(mask, SCORE_ALIBI, n, Hq, {})
    alibi = torch.where(torch.isfinite(bias), bias, torch.zeros(()))
    keep = torch.isfinite(bias)
    s = scale * tq @ tk.repeat_interleave(2, 1).transpose(-1, -2) + alibi
    s = c * torch.tanh(s / c)
    s = torch.where(keep, s, torch.tensor(-math.inf, dtype=torch.float64))
    to = torch.softmax(s, dim=-1) @ tv.repeat_interleave(2, 1)
    (to * torch.from_numpy(do)).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-10)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-10)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-10)


# ---------------------------------------------------------------- finite differences

@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("score", SCORES)
def test_gradients_match_central_finite_differences(mask, score):
    B, Hq, Hkv, n, d, scale = 1, 2, 1, 10, 4, 0.7
    q = _rand((B, Hq, n, d), 40); k = _rand((B, Hkv, n, d), 41)
    v = _rand((B, Hkv, n, d), 42); do = _rand((B, Hq, n, d), 43)
    kw = dict(mask_kind=mask, **_mask_args(mask, n), **_score_args(score))
    dq, dk, dv = ref.backward(q, k, v, do, scale, **kw)

    def loss(qq, kk, vv):
        o, _ = ref.forward(qq, kk, vv, scale, **kw)
        return float((o * do).sum())

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}; args_m = dict(args_p)
            args_p[name] = xp; args_m[name] = xm
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"])
                        - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-7 * max(1.0, np.abs(num).max()))


# ---------------------------------------------------------------- masks and tiles

def test_document_ids_and_offsets():
    offs = offsets_from_lengths([3, 1, 4])
    assert list(offs) == [0, 3, 4, 8]
    assert list(ref.document_ids(offs, 8)) == [0, 0, 0, 1, 2, 2, 2, 2]
    lengths = document_lengths(32768, 3)
    assert sum(lengths) == 32768
    assert all(512 <= x <= 4096 for x in lengths[:-1]) and 1 <= lengths[-1] <= 4096
    assert list(document_offsets(32768, 3)) == list(offsets_from_lengths(lengths))


def test_tile_classes_causal_by_hand():
    cls = ref.classify_tiles(MASK_CAUSAL, 512, 512, 128, 128)
    E, P, F = ref.TILE_EMPTY, ref.TILE_PARTIAL, ref.TILE_FULL
    expect = np.array([[P, E, E, E], [F, P, E, E], [F, F, P, E], [F, F, F, P]])
    assert (cls == expect).all()
    # ragged: Nq = Nkv = 300 -> the last tiles are 44 wide
    cls = ref.classify_tiles(MASK_CAUSAL, 300, 300, 128, 128)
    assert cls.shape == (3, 3) and cls[2, 2] == P and cls[2, 1] == F and cls[1, 2] == E


def test_tile_classes_window_counts_match_closed_form():
    # N = 16384, W = 1024, 128 x 128 tiles: q-tile r >= 8 meets key tiles r-8 .. r
    # (r-8 and r partial, r-7 .. r-1 full); q-tile r < 8 meets tiles 0 .. r
    # (the diagonal partial). So 120*9 + 36 = 1116 non-empty tiles, 120*7 + 28 = 868
    # of them full.
    cls = ref.classify_tiles(MASK_SLIDING_WINDOW, 16384, 16384, 128, 128, window=1024)
    assert int((cls != ref.TILE_EMPTY).sum()) == 1116
    assert int((cls == ref.TILE_FULL).sum()) == 868


def test_tile_classes_documents_by_hand():
    offs = [0, 100, 300, 512]
    cls = ref.classify_tiles(MASK_DOCUMENT_CAUSAL, 512, 512, 128, 128, doc_offsets=offs)
    E, P, F = ref.TILE_EMPTY, ref.TILE_PARTIAL, ref.TILE_FULL
    # Rows 128..255 are in doc 1 (100..299); keys 0..127 hold doc 0 (0..99) and
    # doc 1 (100..127): partial. Rows 256..383 start in doc 1 too, so they still
    # meet keys 100..127: partial. Rows 384..511 (doc 2, from 300) meet only keys
    # from 300 on: tiles 0 and 1 empty, tiles 2 (keys 300..383) and 3 partial.
    expect = np.array([[P, E, E, E], [P, P, E, E], [P, P, P, E], [E, E, P, P]])
    assert (cls == expect).all(), cls


def test_allowed_pair_counts():
    n = 1000
    assert ref.allowed_pairs(MASK_NONE, n, n) == n * n
    assert ref.allowed_pairs(MASK_CAUSAL, n, n) == n * (n + 1) // 2
    w = 77
    assert ref.allowed_pairs(MASK_SLIDING_WINDOW, n, n, window=w) == sum(min(i + 1, w)
                                                                         for i in range(n))
    lens = [100, 400, 500]
    assert ref.allowed_pairs(MASK_DOCUMENT_CAUSAL, n, n,
                             doc_offsets=offsets_from_lengths(lens)) == sum(
        x * (x + 1) // 2 for x in lens)


def test_gqa_head_map():
    # Query heads 2 and 3 of a 4-head / 2-kv-head layout must read kv head 1: make
    # kv head 0 all zeros in V; heads 2, 3 must not see zeros.
    n, d = 8, 4
    q = _rand((1, 4, n, d), 50); k = _rand((1, 2, n, d), 51); v = _rand((1, 2, n, d), 52)
    v[0, 0] = 0.0
    o, _ = ref.forward(q, k, v, 0.5)
    assert np.all(o[0, :2] == 0) and np.all(np.abs(o[0, 2:]) > 0)


def test_stored_tiny_sample_matches_oracle():
    """tests/golden/tiny_forward_sample.json was written by tests/golden/make_golden.py
    (oracle only); a change to the oracle's arithmetic shows up here."""
    import json
    import os
    from workloads import TINY, make_inputs
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_forward_sample.json")
    with open(path) as f:
        g = json.load(f)
    q, k, v, _, _ = make_inputs(TINY)
    o, l = ref.forward(q, k, v, TINY.scale, rows=np.array(g["rows"]))
    np.testing.assert_allclose(o[0][:, :, g["cols"]], np.array(g["o"]), atol=1e-12)
    np.testing.assert_allclose(l[0], np.array(g["lse"]), atol=1e-12)
