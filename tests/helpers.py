"""Shared helpers of the GPU parity tests: run the library and the oracle on the same
seeded inputs and compare with the stated tolerances.

Tolerances (bf16 inputs, fp32 accumulation):
  forward : max|O - O_ref| <= 1e-2, flat, on every element with |O_ref| < 2, and
            1e-2 + half a bf16 ulp of O_ref where |O_ref| >= 2. The method's own
            arithmetic sets that edge: O is stored as bf16 (8 significant bits), whose
            rounding alone is up to 2^-9 |O| (0.0039 below 2, 0.0078 in [2, 4), 0.0156
            in [4, 8)), and P is rounded to bf16 for the P V product, which adds up to
            2^-9 sum_j P_ij |V_jc|, about 2^-9 |O| in the rows where |O| is large (a few
            keys carry the weight). Below 2 the two stay under 1e-2; from 2 on their
            sum can pass it (storage 0.0078 + P 0.004 at |O| = 2.5), and a float64
            model of exactly that rounding (fp32 softmax, P rounded once, O rounded once)
            reproduces the kernels' largest errors there to five digits. Every check
            records its flat max|O - O_ref| over |O_ref| < 2 and over |O_ref| < 4, and
            the session summary prints the largest (tests/conftest.py);
            max|LSE - LSE_ref| <= 1e-3 on finite entries, and -inf exactly where the
            oracle has -inf.
            With dropout at rate p the kept terms of a row are multiplied by 1 / (1 - p),
            so the output's own scale grows with them. The bound is stated relative to
            that scale, per element: |O_ic - O_ref_ic| <= 1e-2 * max(1, A_ic) with
            A_ic = sum_j (P_ij Z_ij / (1 - p)) |V_jc|, the magnitude of the terms summed
            into O_ic (the oracle's forward with |V| in place of V). The kernel's own
            error is at most 2^-9 A_ic from the bf16 rounding of P plus 2^-9 |O_ic| from
            the storage of O, i.e. below 0.004 A_ic.
  backward: max|dX - dX_ref| <= 2e-2 * max|dX_ref| + 1e-5 for each of dq, dk, dv.
            The 1e-5 floor only matters where the exact gradient vanishes (one allowed
            key per row: P = 1 and dP - D = 0): there the kernels leave fp32
            accumulation-order residue of |dO||V| * 2^-23 * d, about 1e-6 at d = 128.
            dP and D are d-term sums whose size and rounding both grow as sqrt(d), so
            the floor is 1e-5 * d / 128 for d > 128.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from workloads import MASK_DOCUMENT_CAUSAL, Workload, make_inputs

O_TOL = 1e-2
O_FLAT_BELOW = 2.0   # |O_ref| below which the forward bound is the flat O_TOL
LSE_TOL = 1e-3
GRAD_REL_TOL = 2e-2
GRAD_ABS_FLOOR = 1e-5


def to_dev(*ts):
    return [None if t is None else t.cuda() for t in ts]


def doc_tensor(offs):
    return None if offs is None else torch.from_numpy(np.asarray(offs, dtype=np.int32)).cuda()


def mask_kwargs(w: Workload, offs):
    kw = dict(mask_kind=w.mask_kind, window=w.window, score_kind=w.score_kind,
              softcap=w.softcap)
    if w.dropout_p > 0:
        kw.update(dropout_p=w.dropout_p, dropout_seed=w.dropout_seed)
    return kw


def oracle_kwargs(w: Workload, offs):
    kw = dict(mask_kind=w.mask_kind, window=w.window, doc_offsets=offs,
              score_kind=w.score_kind, softcap=w.softcap)
    if w.dropout_p > 0:
        kw.update(dropout_p=w.dropout_p, dropout_seed=w.dropout_seed)
    return kw


def bf16_half_ulp(x):
    """Half the spacing of bf16 numbers at |x| (8 significant bits): 2^(floor(log2|x|) - 8)."""
    a = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 8)


# (what, flat max|O - O_ref| over |O_ref| < 2, the same over |O_ref| < 4, elements
# checked, elements at 2 <= |O_ref| < 4 with |O - O_ref| > 1e-2) of every forward check
# in this process; tests/conftest.py prints the summary.
FORWARD_LOG: list = []


def check_forward(o, lse, o_ref, lse_ref, what="", o_scale=None):
    """Forward parity. Without ``o_scale``: flat |O - O_ref| <= 1e-2 where |O_ref| < 2,
    1e-2 + half a bf16 ulp of O_ref elsewhere. With ``o_scale`` (dropout: the per-element
    output scale A, see the module docstring): |O - O_ref| <= 1e-2 * max(1, A)."""
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert o.shape == o_ref.shape and lse.shape == lse_ref.shape
    err = np.abs(o - o_ref)
    mag = np.abs(o_ref)
    flat = mag < O_FLAT_BELOW
    flat_max = float(err[flat].max()) if flat.any() else 0.0
    below4 = mag < 4.0
    max4 = float(err[below4].max()) if below4.any() else 0.0
    over_2_4 = int(((mag >= O_FLAT_BELOW) & below4 & (err > O_TOL)).sum())
    err_o = float(err.max()) if o.size else 0.0
    if o_scale is None:
        bound = np.where(flat, O_TOL, O_TOL + bf16_half_ulp(o_ref))
    else:
        bound = O_TOL * np.maximum(1.0, np.asarray(o_scale, dtype=np.float64))
    FORWARD_LOG.append((what, flat_max, max4, int(o.size), over_2_4, o_scale is not None))
    ninf_ref = np.isneginf(lse_ref)
    assert (np.isneginf(lse) == ninf_ref).all(), f"{what}: -inf pattern of LSE differs"
    fin = ~ninf_ref
    err_l = float(np.abs(lse[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    if o.size:
        worst = np.unravel_index(np.argmax(err - bound), err.shape)
        assert (err <= bound).all(), (
            f"{what}: |dO| = {err[worst]} > bound {bound[worst]} at {worst} "
            f"(O_ref {o_ref[worst]}); flat max|dO| over |O_ref| < 2 = {flat_max}")
    assert err_l <= LSE_TOL, f"{what}: max|dLSE| = {err_l}"
    return err_o, err_l


def check_grads(got, ref, what="", d=128):
    floor = GRAD_ABS_FLOOR * max(1.0, d / 128)
    errs = []
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g = np.asarray(g, dtype=np.float64)
        assert np.isfinite(g).all(), f"{what}: {name} not finite"
        scale = float(np.abs(r).max()) if r.size else 0.0
        err = float(np.abs(g - r).max()) if r.size else 0.0
        assert err <= GRAD_REL_TOL * scale + floor, \
            f"{what}: max|d{name}| = {err} vs {GRAD_REL_TOL} * {scale} + {floor}"
        errs.append(err / max(scale, 1e-30))
    return errs


def run_forward(w: Workload, impl="tc", inputs=None):
    import exact_io_aware_13_gb300 as ea
    q, k, v, do, offs = inputs if inputs is not None else make_inputs(w)
    qd, kd, vd = to_dev(q, k, v)
    o, lse = ea.forward(qd, kd, vd, scale=w.scale, doc_offsets=doc_tensor(offs), impl=impl,
                        **mask_kwargs(w, offs))
    torch.cuda.synchronize()
    assert ea.device_status() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def run_backward(w: Workload, impl="tc", inputs=None):
    import exact_io_aware_13_gb300 as ea
    q, k, v, do, offs = inputs if inputs is not None else make_inputs(w, with_dout=True)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    dt = doc_tensor(offs)
    o, lse = ea.forward(qd, kd, vd, scale=w.scale, doc_offsets=dt, impl=impl,
                        **mask_kwargs(w, offs))
    dq, dk, dv = ea.backward(qd, kd, vd, o, lse, dod, scale=w.scale, doc_offsets=dt, impl=impl,
                             **mask_kwargs(w, offs))
    torch.cuda.synchronize()
    assert ea.device_status() == 0
    return [t.float().cpu().numpy() for t in (dq, dk, dv)]


def small_workload(name, mask_kind, score_kind=0, *, B=1, Hq=4, Hkv=2, N=300, Nkv=None, d=64,
                   window=0, softcap=0.0, seed=7, doc_lo=40, doc_hi=260):
    return Workload(name, seed, B=B, Hq=Hq, Hkv=Hkv, Nq=N, Nkv=N if Nkv is None else Nkv, d=d,
                    mask_kind=mask_kind, window=window, score_kind=score_kind,
                    softcap=softcap, doc_min=doc_lo, doc_max=doc_hi)


def is_document(w):
    return w.mask_kind == MASK_DOCUMENT_CAUSAL


def oracle_forward(w, inputs, rows=None, heads=None):
    q, k, v, _, offs = inputs
    return oracle.forward(q, k, v, w.scale, rows=rows, heads=heads, **oracle_kwargs(w, offs))


def oracle_backward(w, inputs, kv_heads=None):
    q, k, v, do, offs = inputs
    return oracle.backward(q, k, v, do, w.scale, kv_heads=kv_heads, **oracle_kwargs(w, offs))
