"""Pins for the dropout part of the oracle (CPU only): the Philox4x32-10 generator
against the known-answer vectors published with its reference implementation
(Random123), the keep mask against a scalar restatement of its counter layout, its
keep rate, dropout with p = 0 against the plain (pinned) oracle, the forward against
an explicit formula in torch, and the backward against central finite differences
with the mask fixed."""
import numpy as np
import pytest
import torch

from oracle import attention_oracle as ref
from oracle import philox as P


@pytest.mark.parametrize("ctr,key,out", [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
])
def test_philox_known_answers(ctr, key, out):
    assert tuple(int(x) for x in P.philox4x32([ctr], key)[0]) == out


def test_keep_mask_matches_scalar_restatement():
    seed, bh, p = 0x1234_5678_9ABC_DEF0, 5, 0.3
    rows, cols = np.arange(3, 9), np.arange(10, 60)
    keep = P.keep_mask(seed, bh, rows, cols, p)
    thr = int(np.floor(p * 256))
    for a, i in enumerate(rows):
        for c, j in enumerate(cols):
            w = P.philox4x32([(j // 16, i, bh, 0)], (seed & 0xFFFFFFFF, seed >> 32))[0]
            byte = (int(w[(j % 16) // 4]) >> (8 * (j % 4))) & 0xFF
            assert keep[a, c] == (byte >= thr)


def test_keep_rate_and_threshold():
    keep = P.keep_mask(7, 0, np.arange(256), np.arange(512), 0.25)
    rate = keep.mean()
    n = keep.size
    assert abs(rate - 0.75) < 5 * np.sqrt(0.75 * 0.25 / n)
    assert P.drop_threshold(0.0) == 0 and P.drop_threshold(0.999) == 255
    assert P.drop_threshold(0.1) == 25
    assert P.keep_mask(7, 0, [0], np.arange(64), 0.0).all()
    # different seeds and heads give different masks
    assert (P.keep_mask(8, 0, np.arange(16), np.arange(64), 0.5)
            != P.keep_mask(7, 0, np.arange(16), np.arange(64), 0.5)).any()
    assert (P.keep_mask(7, 1, np.arange(16), np.arange(64), 0.5)
            != P.keep_mask(7, 0, np.arange(16), np.arange(64), 0.5)).any()


def _inputs(B=1, Hq=2, Hkv=1, N=40, d=8, seed=0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, N, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float64)
    do = torch.randn(B, Hq, N, d, generator=g, dtype=torch.float64)
    return q, k, v, do


def test_p_zero_equals_plain_oracle():
    q, k, v, do = _inputs()
    o0, l0 = ref.forward(q, k, v, 0.3, mask_kind=ref.MASK_CAUSAL)
    o1, l1 = ref.forward(q, k, v, 0.3, mask_kind=ref.MASK_CAUSAL, dropout_p=0.0, dropout_seed=9)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    g0 = ref.backward(q, k, v, do, 0.3, mask_kind=ref.MASK_CAUSAL)
    g1 = ref.backward(q, k, v, do, 0.3, mask_kind=ref.MASK_CAUSAL, dropout_p=0.0, dropout_seed=9)
    for a, b in zip(g0, g1):
        assert np.array_equal(a, b)


def test_forward_matches_explicit_formula():
    q, k, v, do = _inputs(Hq=2, Hkv=1, N=50, d=16, seed=1)
    p_drop, seed, scale = 0.2, 42, 0.25
    o, lse = ref.forward(q, k, v, scale, mask_kind=ref.MASK_CAUSAL, dropout_p=p_drop,
                         dropout_seed=seed)
    o_plain, lse_plain = ref.forward(q, k, v, scale, mask_kind=ref.MASK_CAUSAL)
    assert np.array_equal(lse, lse_plain)  # the softmax is taken before dropout
    N = 50
    causal = torch.tril(torch.ones(N, N, dtype=torch.bool))
    for h in range(2):
        s = scale * q[0, h] @ k[0, 0].T
        pm = torch.softmax(s.masked_fill(~causal, float("-inf")), dim=-1)
        z = torch.from_numpy(P.keep_mask(seed, h, np.arange(N), np.arange(N), p_drop))
        ref_o = (pm * z / (1 - p_drop)) @ v[0, 0]
        assert np.allclose(o[0, h], ref_o.numpy(), atol=1e-12, rtol=0)


def test_backward_matches_finite_differences_with_fixed_mask():
    q, k, v, do = _inputs(Hq=2, Hkv=1, N=24, d=6, seed=3)
    p_drop, seed, scale = 0.35, 77, 0.4
    dq, dk, dv = ref.backward(q, k, v, do, scale, mask_kind=ref.MASK_CAUSAL, dropout_p=p_drop,
                              dropout_seed=seed)

    def loss(qq, kk, vv):
        o, _ = ref.forward(qq, kk, vv, scale, mask_kind=ref.MASK_CAUSAL, dropout_p=p_drop,
                           dropout_seed=seed)
        return float((o * do.numpy()).sum())

    rng = np.random.default_rng(0)
    eps = 1e-6
    for name, t, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in t.shape)
            tp, tm = t.clone(), t.clone()
            tp[idx] += eps
            tm[idx] -= eps
            args_p = {"q": (tp, k, v), "k": (q, tp, v), "v": (q, k, tp)}[name]
            args_m = {"q": (tm, k, v), "k": (q, tm, v), "v": (q, k, tm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - g[idx]) < 1e-6 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


def test_dropout_is_unbiased_on_average():
    """E[Z] / (1 - p) = 1 per element, so averaging O over many seeds approaches the
    output without dropout."""
    q, k, v, do = _inputs(Hq=1, Hkv=1, N=32, d=4, seed=5)
    o_plain, _ = ref.forward(q, k, v, 0.5)
    acc = np.zeros_like(o_plain)
    n = 400
    for seed in range(n):
        acc += ref.forward(q, k, v, 0.5, dropout_p=0.25, dropout_seed=seed)[0]
    assert np.abs(acc / n - o_plain).max() < 0.15
