"""Pins for the paged-decode oracle (CPU only). Each check comes from outside the
oracle's own code: direct per-token indexing of the pages, the already pinned
top-left causal forward of ``attention_oracle`` on the contiguous keys (full prefill),
torch's float64 scaled_dot_product_attention with a mask and ALiBi bias built by
loops, a scalar-loop soft-cap, and the closed forms of the empty and one-key cases."""
import math

import numpy as np
import pytest
import torch

from oracle import attention_oracle as ref
from oracle import decode_oracle as D
from workloads import (MASK_CAUSAL, MASK_NONE, MASK_SLIDING_WINDOW, SCORE_ALIBI,
                       SCORE_SOFTCAP, DecodeWorkload, make_decode_inputs)


def _w(**kw):
    base = dict(name="pin", seed=11, B=3, Hq=4, Hkv=2, Nq=1, d=16, len_min=1, len_max=70,
                page_size=8)
    base.update(kw)
    return DecodeWorkload(**base)


def _np(t):
    return t.to(torch.float64).numpy()


def test_gather_matches_direct_token_indexing():
    w = _w(lengths=(0, 9, 70))
    q, kc, vc, table, lens = make_decode_inputs(w, poison_unused=True)
    for b in range(w.B):
        got = D.gather_sequence(kc, table[b].numpy(), int(lens[b]))
        assert got.shape == (w.Hkv, int(lens[b]), w.d)
        for t in range(int(lens[b])):
            page, slot = int(table[b, t // w.page_size]), t % w.page_size
            for g in range(w.Hkv):
                assert np.array_equal(got[g, t], _np(kc[page, g, slot]))
        assert not np.isnan(got).any()  # owned slots only: the poison stays out


def test_generator_layout_and_poison():
    w = _w(lengths=(5, 16, 17), spare_pages=2)
    q, kc, vc, table, lens = make_decode_inputs(w, poison_unused=True)
    used = [p for b in range(w.B) for p in table[b].tolist() if p >= 0]
    assert sorted(used) == sorted(set(used)) and len(used) == 1 + 2 + 3
    assert kc.shape[0] == len(used) + 2
    # owned slots finite, every other slot NaN
    assert int(torch.isnan(kc).sum()) == (kc.numel() // (w.Hkv * w.d) - int(lens.sum())) * w.Hkv * w.d


@pytest.mark.parametrize("score", [0, SCORE_ALIBI | SCORE_SOFTCAP])
def test_full_prefill_equals_top_left_causal_forward(score):
    """With Nq equal to every sequence's length the newest-token positions are 0..N-1,
    so bottom-right and top-left causal coincide: compare with the pinned oracle on the
    contiguous keys, taken from the cache by plain slicing of the page list."""
    N = 37
    w = _w(Hq=6, Hkv=2, Nq=N, lengths=(N, N), B=2, score_kind=score, softcap=3.0, page_size=8)
    q, kc, vc, table, lens = make_decode_inputs(w)
    o, lse = D.decode_forward(q, kc, vc, table, lens, w.scale, MASK_CAUSAL, 0, score, 3.0)
    for b in range(w.B):
        pages = table[b, : (N + 7) // 8].tolist()
        k = torch.cat([kc[p] for p in pages], dim=1)[:, :N]   # [Hkv, N, d]
        v = torch.cat([vc[p] for p in pages], dim=1)[:, :N]
        o_ref, l_ref = ref.forward(q[b:b + 1], k[None], v[None], w.scale, mask_kind=MASK_CAUSAL,
                                   score_kind=score, softcap=3.0)
        assert np.allclose(o[b], o_ref[0], atol=1e-12, rtol=0)
        assert np.allclose(lse[b], l_ref[0], atol=1e-12, rtol=0)


def _loop_bias(pos, L, mask_kind, window, slope):
    bias = np.zeros((len(pos), L))
    for r, p in enumerate(pos):
        for j in range(L):
            ok = (mask_kind == MASK_NONE or (j <= p and (mask_kind != MASK_SLIDING_WINDOW
                                                         or p - j < window)))
            bias[r, j] = -slope * (p - j) if ok else -math.inf
    return bias


@pytest.mark.parametrize("mask,window", [(MASK_NONE, 0), (MASK_CAUSAL, 0),
                                         (MASK_SLIDING_WINDOW, 5)])
@pytest.mark.parametrize("nq", [1, 3])
@pytest.mark.parametrize("alibi", [False, True])
def test_decode_matches_torch_sdpa_with_explicit_bias(mask, window, nq, alibi):
    w = _w(Nq=nq, lengths=(3, 40, 70), mask_kind=mask, window=window,
           score_kind=SCORE_ALIBI if alibi else 0)
    q, kc, vc, table, lens = make_decode_inputs(w)
    o, lse = D.decode_forward(q, kc, vc, table, lens, w.scale, mask, window, w.score_kind)
    G = w.Hq // w.Hkv
    for b in range(w.B):
        L = int(lens[b])
        # contiguous keys straight from the page list, one token at a time
        K = torch.stack([kc[table[b, t // 8], :, t % 8] for t in range(L)], dim=1).double()
        V = torch.stack([vc[table[b, t // 8], :, t % 8] for t in range(L)], dim=1).double()
        pos = [L - nq + i for i in range(nq)]
        for h in range(w.Hq):
            slope = 2.0 ** (-8.0 * (h + 1) / w.Hq) if alibi else 0.0
            bias = torch.from_numpy(_loop_bias(pos, L, mask, window, slope))
            live = torch.isfinite(bias).any(dim=1)
            qh = q[b, h].double()
            ref_o = torch.nn.functional.scaled_dot_product_attention(
                qh[None], K[h // G][None], V[h // G][None], attn_mask=bias[None],
                scale=w.scale)[0]
            s = w.scale * qh @ K[h // G].T + bias
            ref_l = torch.logsumexp(s, dim=1)
            for r in range(nq):
                if live[r]:
                    assert np.allclose(o[b, h, r], ref_o[r].numpy(), atol=1e-12, rtol=0)
                    assert abs(lse[b, h, r] - float(ref_l[r])) < 1e-12
                else:
                    assert np.all(o[b, h, r] == 0) and np.isneginf(lse[b, h, r])


def test_softcap_against_scalar_loop():
    w = _w(Nq=2, lengths=(20,), B=1, Hq=2, Hkv=1, score_kind=SCORE_SOFTCAP | SCORE_ALIBI,
           softcap=0.7, mask_kind=MASK_CAUSAL)
    q, kc, vc, table, lens = make_decode_inputs(w)
    o, lse = D.decode_forward(q, kc, vc, table, lens, w.scale, MASK_CAUSAL, 0, w.score_kind, 0.7)
    L = 20
    for h in range(2):
        slope = 2.0 ** (-8.0 * (h + 1) / 2)
        for i in range(2):
            p = L - 2 + i
            sc = []
            for j in range(p + 1):
                kj = kc[table[0, j // 8], 0, j % 8].double()
                x = w.scale * float(q[0, h, i].double() @ kj) - slope * (p - j)
                sc.append(0.7 * math.tanh(x / 0.7))
            mx = max(sc)
            den = sum(math.exp(x - mx) for x in sc)
            num = sum(math.exp(x - mx) * vc[table[0, j // 8], 0, j % 8].double().numpy()
                      for j, x in enumerate(sc))
            assert np.allclose(o[0, h, i], num / den, atol=1e-12, rtol=0)
            assert abs(lse[0, h, i] - (mx + math.log(den))) < 1e-12


def test_empty_and_single_key_cases():
    w = _w(Nq=3, lengths=(0, 1, 2), mask_kind=MASK_CAUSAL)
    q, kc, vc, table, lens = make_decode_inputs(w)
    o, lse = D.decode_forward(q, kc, vc, table, lens, w.scale, MASK_CAUSAL)
    # no cached token: every row empty
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    # one token, three queries at positions -2, -1, 0: only the last sees key 0
    assert np.all(o[1, :, :2] == 0) and np.all(np.isneginf(lse[1, :, :2]))
    v0 = _np(vc[table[1, 0], :, 0])          # [Hkv, d]
    k0 = _np(kc[table[1, 0], :, 0])
    for h in range(w.Hq):
        assert np.array_equal(o[1, h, 2], v0[h // 2])
        assert abs(lse[1, h, 2] - w.scale * float(_np(q[1, h, 2]) @ k0[h // 2])) < 1e-12
    # window 0 masks every pair
    o2, l2 = D.decode_forward(q, kc, vc, table, lens, w.scale, MASK_SLIDING_WINDOW, 0)
    assert np.all(o2 == 0) and np.all(np.isneginf(l2))


def test_uniform_values_and_row_sums():
    w = _w(Nq=2, lengths=(50, 7, 23))
    q, kc, vc, table, lens = make_decode_inputs(w)
    vc_u = torch.full_like(vc, 0.375)
    o, _ = D.decode_forward(q, kc, vc_u, table, lens, w.scale)
    assert np.allclose(o, 0.375, atol=1e-14)
    # P rows sum to one: attention of all-ones values returns ones
    o1, _ = D.decode_forward(q, kc, torch.ones_like(vc), table, lens, w.scale, MASK_CAUSAL)
    assert np.allclose(o1, 1.0, atol=1e-14)


def test_kv_bytes():
    assert D.kv_bytes([3, 5], Hkv=8, d=128) == 8 * 8 * 128 * 4
