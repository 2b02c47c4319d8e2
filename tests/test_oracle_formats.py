"""Pins of the oracle's number formats (E4M3, E2M1, E8M0) and weight quantisers.

Independent references: the OCP FP8 and OCP MX v1.0 definitions (closed-form
values), PyTorch's own float8_e4m3fn conversion (a library routine), exhaustive
code sweeps and the rounding error bound.
"""
import numpy as np
import pytest
import torch

import synth


def test_e4m3_closed_form_values(orc):
    # OCP FP8 E4M3: bias 7, 3 mantissa bits, max finite 448, min subnormal 2^-9
    assert orc.e4m3_value(0x7E) == 448.0
    assert orc.e4m3_value(0xFE) == -448.0
    assert orc.e4m3_value(0x01) == 2.0 ** -9
    assert orc.e4m3_value(0x07) == 7 * 2.0 ** -9
    assert orc.e4m3_value(0x08) == 2.0 ** -6
    assert orc.e4m3_value(0x38) == 1.0
    assert orc.e4m3_value(0x39) == 1.125
    assert np.isnan(orc.e4m3_value(0x7F)) and np.isnan(orc.e4m3_value(0xFF))


def test_e4m3_exhaustive_roundtrip(orc):
    for b in range(256):
        if b in (0x7F, 0xFF):
            continue
        assert orc.e4m3_encode(orc.e4m3_value(b)) == b, hex(b)


def test_e4m3_decode_matches_torch(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([orc.e4m3_value(b) for b in range(256)])
    ok = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    assert np.array_equal(ref[ok], mine[ok])


def test_e4m3_encode_matches_torch_rne(orc):
    # all finite magnitudes, every midpoint between neighbours (ties), and
    # points just either side of each midpoint
    vals = np.array([orc.e4m3_value(b) for b in range(0x7F)])
    mids = (vals[:-1] + vals[1:]) / 2
    eps = np.nextafter(mids.astype(np.float32), np.float32(np.inf)) - mids.astype(np.float32)
    cand = np.concatenate([vals, mids, mids - eps, mids + eps,
                           np.random.default_rng(0).uniform(0, 448, 20000)]).astype(np.float32)
    cand = cand[cand <= 448]
    cand = np.concatenate([cand, -cand])
    ref = torch.from_numpy(cand).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([orc.e4m3_encode(float(v)) for v in cand], np.uint8)
    bad = np.nonzero(ref != mine)[0]
    assert bad.size == 0, [(cand[i], hex(ref[i]), hex(mine[i])) for i in bad[:5]]


def test_e4m3_saturates(orc):
    for v in (448.0, 460.0, 464.0, 480.0, 1e6, 3e38):
        assert orc.e4m3_encode(v) == 0x7E
        assert orc.e4m3_encode(-v) == 0xFE


def test_quant_rows_amax_and_zero_row(orc):
    g = np.random.default_rng(1)
    w = g.standard_normal((7, 96)).astype(np.float32) * np.float32(0.02)
    w[3] = 0.0
    q, s = orc.quant_e4m3_rows(w)
    assert s[3] == 1.0 and np.all(q[3] == 0)
    for r in range(7):
        if r == 3:
            continue
        c = int(np.argmax(np.abs(w[r])))
        assert q[r, c] in (0x7E, 0xFE)
        assert s[r] == np.float32(np.max(np.abs(w[r])) / np.float32(448.0))


def test_quant_rows_error_bound(orc):
    # RNE error bound: half a step of the code grid at the value's binade
    cfg = synth.WORKLOADS["tiny"]
    w13, _ = synth.expert_weights(cfg, 0)
    q, s = orc.quant_e4m3_rows(w13)
    deq = orc.dequant_e4m3_rows(q, s)
    a = np.abs(w13.astype(np.float64)) / s[:, None]
    binade = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    half_step = 2.0 ** (binade - 3) / 2
    err = np.abs(deq - w13) / s[:, None]
    assert np.all(err <= half_step * (1 + 1e-6) + 1e-7 * a)


E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # OCP MX v1.0 FP4 E2M1 magnitudes


def test_e2m1_values_and_roundtrip(orc):
    for c in range(16):
        v = orc.e2m1_value(c)
        assert abs(v) == E2M1[c & 7]
        assert (v < 0) == (c >= 8 and c != 8) or v == 0
        assert orc.e2m1_encode(v if c != 8 else -0.0) == c


@pytest.mark.parametrize("v,code", [
    (0.25, 0), (0.26, 1), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6),
    (5.0, 6), (5.5, 7), (7.0, 7), (100.0, 7), (-0.75, 10), (-5.0, 14)])
def test_e2m1_rne_ties_and_saturation(orc, v, code):
    assert orc.e2m1_encode(v) == code


def test_e8m0_values(orc):
    assert orc.e8m0_value(127) == 1.0
    assert orc.e8m0_value(0) == 2.0 ** -127
    assert orc.e8m0_value(254) == 2.0 ** 127


def _fp8_row(orc, values, scale=1.0):
    q = np.array([[orc.e4m3_encode(v) for v in values]], np.uint8)
    s = np.array([scale], np.float32)
    return q, s


def test_mxfp4_hand_groups(orc):
    # group 0: amax 3 -> floor(log2 3) = 1 -> X = 2^(1-2) = 0.5 (byte 126)
    #   3/X = 6 -> 7; 1/X = 2 -> 4; -0.5/X = -1 -> 8|2; 0.25/X = 0.5 -> 1
    g0 = [3.0, 1.0, -0.5, 0.25] + [0.0] * 28
    # group 1: amax 1 -> X = 2^-2 (byte 125)
    #   1/X = 4 -> 6; 0.375/X = 1.5 -> 3; -0.0625/X = -0.25, a tie between 0 and 0.5 -> even (0) -> 8
    g1 = [1.0, 0.375, -0.0625] + [0.0] * 29
    # group 2: all zero -> byte 0, all codes 0
    g2 = [0.0] * 32
    q8, s8 = _fp8_row(orc, g0 + g1 + g2)
    q4, e8 = orc.quant_mxfp4_rows(q8, s8)
    assert list(e8[0]) == [126, 125, 0]
    nib = np.empty(96, np.uint8)
    nib[0::2] = q4[0] & 15
    nib[1::2] = q4[0] >> 4
    assert list(nib[:4]) == [7, 4, 10, 1]
    assert list(nib[32:35]) == [6, 3, 8]
    assert np.all(nib[4:32] == 0) and np.all(nib[35:] == 0)


def test_mxfp4_hand_groups_exact(orc):
    g0 = [3.0, 1.0, -0.5, 0.25] + [0.0] * 28
    q8, s8 = _fp8_row(orc, g0)
    q4, e8 = orc.quant_mxfp4_rows(q8, s8)
    nib = np.empty(32, np.uint8)
    nib[0::2] = q4[0] & 15
    nib[1::2] = q4[0] >> 4
    # X = 0.5: 3/0.5 = 6 -> 7; 1/0.5 = 2 -> 4; -0.5/0.5 = -1 -> 8|2; 0.25/0.5 = 0.5 -> 1
    assert e8[0, 0] == 126
    assert list(nib[:4]) == [7, 4, 10, 1]
    assert np.all(nib[4:] == 0)


def test_mxfp4_error_bound(orc):
    cfg = synth.WORKLOADS["tiny"]
    w13, _ = synth.expert_weights(cfg, 1)
    q8, s8 = orc.quant_e4m3_rows(w13)
    v = orc.dequant_e4m3_rows(q8, s8)
    q4, e8 = orc.quant_mxfp4_rows(q8, s8)
    d4 = orc.dequant_mxfp4_rows(q4, e8)
    X = np.repeat(np.array([[orc.e8m0_value(b) for b in row] for row in e8]), 32, axis=1)
    a = np.abs(v) / X
    # half the E2M1 grid spacing (0.5 below 2, 1 in [2,4), 2 in [4,6]); with
    # X = 2^(floor(log2 amax) - 2) the scaled magnitudes reach just under 8,
    # and those above 6 saturate to 6 (OCP MX v1.0 conversion rule)
    assert a.max() < 8
    bound = np.where(a < 2, 0.25, np.where(a < 4, 0.5, np.where(a <= 6, 1.0, a - 6)))
    assert np.all(np.abs(d4 - v) / X <= bound + 1e-9)
