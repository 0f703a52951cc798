"""GPU parity of the FP8 path: the e4m3 block quantiser against the oracle (bit-exact
codes and scales), and the FP8 forward, fed the oracle's own codes, against the
float64 attention of the dequantised inputs within the oracle's per-element bound
(``oracle.fp8_oracle.output_error_bound``: P is rounded to e4m3 for the P V product);
LSE within the forward tolerance."""
import numpy as np
import pytest
import torch

from oracle import fp8_oracle as F
from tests import helpers as H
from workloads import (CAUSAL, MASK_CAUSAL, MASK_DOCUMENT_CAUSAL, MASK_NONE,
                       MASK_SLIDING_WINDOW, SCORE_ALIBI, SCORE_SOFTCAP, make_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _np(t):
    return t.float().cpu().numpy()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [1, 300, 1000])
def test_quantiser_matches_oracle_bitwise(n, d):
    import exact_io_aware_13_gb300 as ea
    g = torch.Generator("cpu").manual_seed(n + d)
    x = (torch.randn((2, 3, n, d), generator=g) * torch.tensor([1.0, 40.0, 1e-3])[:, None, None]
         ).to(torch.bfloat16)
    if n >= 300:
        x[1, 2, 128:256] = 0  # an all-zero tile
    codes, scales = ea.quantize_fp8(x.cuda(), ea.FP8_TILES)
    vcodes, vscales = ea.quantize_fp8(x.cuda(), ea.FP8_V_TRANSPOSED)
    torch.cuda.synchronize()
    xr = _np(x).reshape(6, n, d)
    rc, rs = F.quantize_tiles(xr)
    assert np.array_equal(codes.cpu().numpy().reshape(6, n, d), rc)
    assert np.array_equal(scales.cpu().numpy(), rs)
    rvc, rvs = F.quantize_v_transposed(xr)
    assert np.array_equal(vcodes.cpu().numpy().reshape(rvc.shape), rvc)
    assert np.array_equal(vscales.cpu().numpy(), rvs)


def _fp8_case(w):
    """Seeded bf16 inputs quantised by the oracle; GPU tensors of the codes."""
    q, k, v, _, offs = make_inputs(w)
    qc, qs = F.quantize_tiles(_np(q).reshape(w.B * w.Hq, w.Nq, w.d))
    kc, ks = F.quantize_tiles(_np(k).reshape(w.B * w.Hkv, w.Nkv, w.d))
    vc, vs = F.quantize_v_transposed(_np(v).reshape(w.B * w.Hkv, w.Nkv, w.d))
    dev = [torch.from_numpy(a).cuda() for a in (qc.reshape(q.shape), qs, kc.reshape(k.shape),
                                                ks, vc.reshape(w.B, w.Hkv, w.d, -1), vs)]
    return (qc, qs, kc, ks, vc, vs), dev, offs


def _run_fp8(w, dev, offs):
    import exact_io_aware_13_gb300 as ea
    q8, sq, k8, sk, v8t, sv = dev
    o = torch.empty((w.B, w.Hq, w.Nq, w.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device="cuda")
    ea.fwd_fp8_into(q8, sq, k8, sk, v8t, sv, o, lse, Nkv=w.Nkv, scale=w.scale,
                    doc_offsets=H.doc_tensor(offs), **H.mask_kwargs(w, offs))
    torch.cuda.synchronize()
    assert ea.device_status() == 0
    return _np(o), lse.cpu().numpy()


def _check(w, codes, offs, o, lse, heads=None, rows=None):
    qc, qs, kc, ks, vc, vs = codes
    mods = H.oracle_kwargs(w, offs)
    o_ref, l_ref, (qd, kd, vd) = F.forward_reference(qc, qs, kc, ks, vc, vs, w.B, w.Hq, w.Hkv,
                                                      w.Nq, w.Nkv, w.scale, rows=rows,
                                                      heads=heads, **mods)
    todo = heads or [(b, h) for b in range(w.B) for h in range(w.Hq)]
    sel = slice(None) if rows is None else rows
    worst = 0.0
    for b, h in todo:
        bound = F.output_error_bound(qd, kd, vd, w.scale, b, h, rows=rows, **mods)
        allow = bound * (1 + 2.0 ** -8) + F.max_abs_rounding_bf16(o_ref[b, h])
        err = np.abs(o[b, h][sel] - o_ref[b, h])
        assert np.all(err <= allow), f"{w.name} b={b} h={h}: {float((err - allow).max())}"
        worst = max(worst, float(err.max()))
        fin = np.isfinite(l_ref[b, h])
        got = lse[b, h][sel]
        assert np.array_equal(np.isneginf(got), ~fin)
        assert np.all(np.abs(got[fin] - l_ref[b, h][fin]) <= H.LSE_TOL)
    return worst


@pytest.mark.parametrize("score", [0, SCORE_ALIBI | SCORE_SOFTCAP])
@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_SLIDING_WINDOW,
                                  MASK_DOCUMENT_CAUSAL])
def test_fp8_forward_variants(mask, score):
    w = H.small_workload(f"fp8-m{mask}s{score}", mask, score, B=2, Hq=4, Hkv=2, N=520, d=128,
                         window=200 if mask == MASK_SLIDING_WINDOW else 0,
                         softcap=20.0 if score & SCORE_SOFTCAP else 0.0, seed=300 + mask + score)
    codes, dev, offs = _fp8_case(w)
    o, lse = _run_fp8(w, dev, offs)
    _check(w, codes, offs, o, lse)


@pytest.mark.parametrize("nq,nkv", [(129, 1), (200, 450), (450, 200)])
def test_fp8_forward_ragged(nq, nkv):
    w = H.small_workload(f"fp8-ragged{nq}x{nkv}", MASK_CAUSAL, B=1, Hq=2, Hkv=1, N=nq, Nkv=nkv,
                         d=128, seed=nq + 3 * nkv)
    codes, dev, offs = _fp8_case(w)
    o, lse = _run_fp8(w, dev, offs)
    _check(w, codes, offs, o, lse)


def test_fp8_rejects_other_head_dims():
    import exact_io_aware_13_gb300 as ea
    from exact_io_aware_13_gb300 import _lib
    z = torch.zeros((1, 1, 64, 64), dtype=torch.uint8, device="cuda")
    s = torch.ones((1, 1), dtype=torch.float32, device="cuda")
    o = torch.empty((1, 1, 64, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 1, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(_lib.AttnError):
        ea.fwd_fp8_into(z, s, z, s, z, s, o, lse, Nkv=64, scale=0.125)


def test_fp8_full_size_causal_sampled():
    """The causal workload (B=4 H=16 N=8192) quantised on the GPU (its codes checked
    against the oracle on sampled heads), then the FP8 forward on sampled rows."""
    import exact_io_aware_13_gb300 as ea
    w = CAUSAL
    q, k, v, _, offs = make_inputs(w)
    (q8, sq), (k8, sk), (v8t, sv) = ea.fp8_inputs(q.cuda(), k.cuda(), v.cuda())
    o = torch.empty_like(q, device="cuda")
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
    ea.fwd_fp8_into(q8, sq, k8, sk, v8t, sv, o, lse, Nkv=w.Nkv, scale=w.scale,
                    mask_kind=w.mask_kind)
    torch.cuda.synchronize()
    assert ea.device_status() == 0
    heads = [(0, 0), (w.B - 1, w.Hq - 1)]
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 4095, w.Nq - 1],
                                     np.random.default_rng(0).integers(0, w.Nq, 24)]))
    codes = [t.cpu().numpy() for t in (q8, sq, k8, sk, v8t, sv)]
    for b, h in heads:  # the GPU quantiser agrees with the oracle on these heads
        bh = b * w.Hq + h
        rc, rs = F.quantize_tiles(_np(q[b, h])[None])
        assert np.array_equal(codes[0][b, h], rc[0]) and np.array_equal(codes[1][bh], rs[0])
    worst = _check(w, codes, offs, _np(o), lse.cpu().numpy(), heads=heads, rows=rows)
    assert worst < 0.1
