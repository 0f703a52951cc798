"""Pins for the FP8 oracle (CPU only): the e4m3 codec against torch's float8_e4m3fn
conversions (a library routine) and the format definition, the block quantiser
against properties its definition forces, and the forward error bound against a
brute-force emulation of P rounded to e4m3."""
import numpy as np
import pytest
import torch

from oracle import attention_oracle as ref
from oracle import fp8_oracle as F
from workloads import MASK_CAUSAL, MASK_NONE


def _all_codes():
    return np.arange(256, dtype=np.uint8)


def test_decode_matches_torch_float8_for_every_code():
    codes = _all_codes()
    ours = F.e4m3_decode(codes)
    theirs = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], theirs[~nan])
    # the format's landmarks
    assert F.e4m3_decode([0x7E])[0] == 448.0 and F.e4m3_decode([0x01])[0] == 2.0 ** -9
    assert F.e4m3_decode([0x08])[0] == 2.0 ** -6 and F.e4m3_decode([0x38])[0] == 1.0
    assert nan.sum() == 2  # 0x7f and 0xff only


def test_encode_matches_torch_float8_rounding_including_ties():
    vals = np.unique(F.e4m3_decode(_all_codes())[:0x7F])
    vals = np.unique(np.concatenate([vals, -vals]))
    mids = (vals[:-1] + vals[1:]) / 2                      # exact ties
    rng = np.random.default_rng(5)
    x = np.concatenate([vals, mids, rng.uniform(-448, 448, 20000),
                        rng.standard_normal(20000) * 1e-3, rng.standard_normal(20000) * 2.0 ** -10,
                        [0.0, -0.0, 447.9, 455.9, -455.9]]).astype(np.float32)
    ours = F.e4m3_encode(x)
    theirs = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def test_encode_saturates_above_the_largest_finite_value():
    x = np.array([448.0, 463.9, 470.0, 1e4, -600.0], dtype=np.float32)
    assert F.e4m3_decode(F.e4m3_encode(x)).tolist() == [448.0, 448.0, 448.0, 448.0, -448.0]


def test_round_trip_is_identity_on_representable_values():
    codes = _all_codes()
    finite = ~np.isnan(F.e4m3_decode(codes))
    again = F.e4m3_encode(F.e4m3_decode(codes[finite]))
    assert np.array_equal(F.e4m3_decode(again), F.e4m3_decode(codes[finite]))


def test_tile_quantisation_properties():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((3, 300, 128)) * np.array([1.0, 30.0, 1e-3])[:, None, None])
    x = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy()
    x[2, 128:256] = 0.0                                    # an all-zero tile
    codes, scales = F.quantize_tiles(x)
    assert scales.shape == (3, 3) and scales[2, 1] == 1.0
    deq = F.dequantize_tiles(codes, scales)
    for bh in range(3):
        for t in range(3):
            blk, dq = x[bh, t * 128:(t + 1) * 128], deq[bh, t * 128:(t + 1) * 128]
            s = float(scales[bh, t])
            if np.abs(blk).max() == 0:
                assert np.all(codes[bh, t * 128:(t + 1) * 128] == 0)
                continue
            # the block's largest magnitude maps to the largest code, 448
            assert np.abs(F.e4m3_decode(codes[bh, t * 128:(t + 1) * 128])).max() == 448.0
            assert s == np.float32(np.float32(np.abs(blk).max()) / np.float32(448.0))
            # relative error <= 2^-4 in the normal range, absolute <= 2^-10 s below it
            normal = np.abs(blk) >= 2.0 ** -6 * s
            err = np.abs(dq - blk)
            assert np.all(err[normal] <= 2.0 ** -4 * np.abs(blk[normal]) * (1 + 1e-6))
            assert np.all(err[~normal] <= 2.0 ** -10 * s * (1 + 1e-6))


def test_v_transposed_layout_and_padding():
    rng = np.random.default_rng(2)
    x = torch.from_numpy(rng.standard_normal((2, 37, 128)).astype(np.float32)).to(
        torch.bfloat16).float().numpy()
    codes, scales = F.quantize_v_transposed(x)
    assert codes.shape == (2, 128, 48) and F.v_row_bytes(37) == 48
    assert np.all(codes[:, :, 37:] == 0)
    for bh in range(2):
        assert scales[bh] == np.float32(np.float32(np.abs(x[bh]).max()) / np.float32(448.0))
        assert np.array_equal(codes[bh, :, :37].T, F.e4m3_encode(x[bh] / scales[bh]))
    back = F.dequantize_v_transposed(codes, scales, 37)
    assert np.all(np.abs(back - x) <= 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * scales[:, None, None])


@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL])
def test_output_bound_holds_for_an_emulated_p_rounding(mask):
    """Emulate the FP8 forward's only lossy step on the dequantised inputs (P scaled by
    2^7 and rounded to e4m3, row sums of the unrounded P) and check that the oracle's
    per-element bound covers the error."""
    rng = np.random.default_rng(3)
    B, H, N, d = 1, 2, 200, 128
    q = rng.standard_normal((B, H, N, d)); k = rng.standard_normal((B, H, N, d))
    v = rng.standard_normal((B, H, N, d)) * 3
    scale = 1 / np.sqrt(d)
    o_ref, _ = ref.forward(q, k, v, scale, mask_kind=mask)
    for h in range(H):
        p = ref.probabilities(q, k, scale, h_index=h, mask_kind=mask)      # normalised
        # unnormalised p against a running max up to one unit (log2) below the true one:
        # the largest entry of a row lies in [1, 2]
        pk = p / p.max(1, keepdims=True) * np.exp2(rng.uniform(0, 1, (N, 1)))
        pr = F.e4m3_decode(F.e4m3_encode(pk * 128.0)) / 128.0
        o_emul = (pr @ v[0, h]) / pk.sum(1, keepdims=True)
        bound = F.output_error_bound(q, k, v, scale, 0, h, mask_kind=mask)
        assert np.all(np.abs(o_emul - o_ref[0, h]) <= bound)
        # and the bound is not vacuous: it is a few percent of the values
        assert bound.max() < 0.2 * np.abs(v).max()
