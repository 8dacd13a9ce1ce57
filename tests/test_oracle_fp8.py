"""Pins of the fp8 e4m3 decoder of the oracle (oracle/fp8.py), on the CPU:
closed forms from the format's definition, and every one of the 256 codes
against torch's float8_e4m3fn conversion."""
import numpy as np
import torch

from oracle import fp8 as F


def test_closed_forms():
    v = F.e4m3_to_float64(np.array([0x00, 0x80, 0x38, 0xB8, 0x7E, 0xFE, 0x01, 0x07, 0x08, 0x30,
                                    0x3C, 0x40, 0x77], dtype=np.uint8))
    want = [0.0, -0.0, 1.0, -1.0, 448.0, -448.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 0.5,
            1.5, 2.0, 240.0]
    assert np.array_equal(v, np.array(want))
    assert np.signbit(v[1])
    assert np.isnan(F.e4m3_to_float64(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_every_code_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.e4m3_to_float64(codes.numpy())
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan], ref[~nan])


def test_dequantize_scales_per_head():
    codes = np.full((3, 2, 4), 0x38, dtype=np.uint8)   # all 1.0
    x = F.dequantize(codes, np.array([0.5, 4.0]), head_axis=1)
    assert np.array_equal(x[:, 0], np.full((3, 4), 0.5))
    assert np.array_equal(x[:, 1], np.full((3, 4), 4.0))
