"""Pins for the oracle's number formats, against library decoders and the published format tables."""
import math

import numpy as np
import torch

from oracle import formats as F


def test_e2m1_table_matches_ocp_values():
    # OCP Microscaling Formats v1.0, FP4 E2M1 element encodings: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(8):
        assert F.e2m1_value(c) == mags[c]
        assert F.e2m1_value(c | 8) == -mags[c]


def test_e2m1_packed_nibble_order():
    # element 2j is the low nibble: byte 0x21 -> [code 1, code 2] = [0.5, 1.0]; 0xF7 -> [6, -6]
    v = F.decode_e2m1_packed(np.array([[0x21, 0xF7]], dtype=np.uint8))
    assert v.tolist() == [[0.5, 1.0, 6.0, -6.0]]


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.decode_e4m3(codes.numpy())
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ref[~nan], ours[~nan])


def test_e4m3_spot_values():
    assert F.e4m3_value(0x7E) == 448.0
    assert F.e4m3_value(0x38) == 1.0
    assert F.e4m3_value(0x01) == 2.0 ** -9
    assert F.e4m3_value(0x08) == 2.0 ** -6
    assert F.e4m3_value(0x80) == 0.0 and math.copysign(1, F.e4m3_value(0x80)) < 0


def test_ue8m0():
    assert F.ue8m0_value(127) == 1.0
    assert F.ue8m0_value(0) == 2.0 ** -127
    assert F.ue8m0_value(254) == 2.0 ** 127
    assert math.isnan(F.ue8m0_value(255))


def test_e4m3_encode_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(F.encode_e4m3_rne(F.decode_e4m3(codes)), codes)


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(0)
    vals = F.E4M3_TABLE[[c for c in range(127)]]
    mids = (vals[1:] + vals[:-1]) / 2                        # exact ties
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.uniform(-1, 1, 20000) * 2.0 ** -6,
                        mids, -mids, [0.0, -0.0, 448.0, -448.0, 2.0 ** -10, -2.0 ** -10, 2.0 ** -11]])
    x32 = x.astype(np.float32)                               # exactly representable in float32
    ref = torch.from_numpy(x32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = F.encode_e4m3_rne(x32.astype(np.float64))
    assert np.array_equal(ours, ref)


def test_e4m3_negative_underflow_keeps_sign():
    assert F.encode_e4m3_rne(np.array([-2.0 ** -11]))[0] == 0x80
    assert F.encode_e4m3_rne(np.array([2.0 ** -11]))[0] == 0x00


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(1)
    base = rng.standard_normal(50000).astype(np.float32) * np.float32(3.0)
    # ties: 1 + 2**-8 has its 9th significant bit set exactly
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2.0 ** -130, 2.0 ** -134,
                     3 * 2.0 ** -135, 3.3895313892515355e38, 1e-40], dtype=np.float32)
    x = np.concatenate([base, ties, rng.standard_normal(1000).astype(np.float32) * np.float32(1e-39)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = F.round_bf16_rne(x.astype(np.float64))
    assert np.array_equal(ours, ref)


def test_bf16_hand_cases():
    assert F.round_bf16_rne(np.array([1 + 2.0 ** -8]))[0] == 0x3F80          # tie -> even (1.0)
    assert F.round_bf16_rne(np.array([1 + 3 * 2.0 ** -8]))[0] == 0x3F82      # tie -> even (1 + 2**-6)
    assert F.round_bf16_rne(np.array([1 + 2.0 ** -8 + 2.0 ** -30]))[0] == 0x3F81
    assert F.bf16_to_f64(np.array([0x3F80], dtype=np.uint16))[0] == 1.0


def test_ue8m0_exponent_rule():
    e = F.ue8m0_exponent_for_amax
    assert e(0.0) == 0
    assert e(448.0) == 0
    assert e(448.0 * (1 + 2.0 ** -20)) == 1
    assert e(224.0) == -1
    assert e(224.0 * (1 + 2.0 ** -20)) == 0
    assert e(1.0) == -8            # 1 <= 448 * 2**-8 = 1.75; 1 > 448 * 2**-9
    assert e(1.75) == -8 and e(1.76) == -7
    assert e(2.0 ** -200) == -127  # clamped
    for a in [3.7, 1e-3, 1e6, 0.0123]:
        k = e(a)
        assert a <= 448 * 2.0 ** k and a > 448 * 2.0 ** (k - 1)
