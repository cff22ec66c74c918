"""Pins of the oracle's FP8 E4M3 decoding (CPU only).

The pages name an FP8 forward without a format; the format is the OCP 8-bit
floating point specification's E4M3 (bias 7, 3 mantissa bits, no infinities,
S.1111.111 = NaN).  Pinned by values worked out by hand from the bit fields,
by every byte against torch's float8_e4m3fn (an independent library decoder),
and by planted mistakes."""
import math
import os

import numpy as np
import pytest
import torch

import oracle


def test_hand_decoded_bytes():
    cases = {
        0x38: 1.0,            # 0 0111 000: 2^(7-7) * 1
        0xB8: -1.0,
        0x40: 2.0,            # 0 1000 000
        0x3C: 1.5,            # 0 0111 100: 1 + 4/8
        0x7E: 448.0,          # 0 1111 110: 2^8 * 1.75, the largest finite value
        0x08: 2.0 ** -6,      # 0 0001 000: smallest normal
        0x01: 2.0 ** -9,      # 0 0000 001: smallest subnormal, 1/8 * 2^-6
        0x07: 7 / 8 * 2.0 ** -6,
        0x00: 0.0,
        0x80: -0.0,
    }
    for b, v in cases.items():
        got = oracle.decode_e4m3(np.array([b], dtype=np.uint8))[0]
        assert got == v and math.copysign(1, got) == math.copysign(1, v), (hex(b), got, v)
    assert math.isnan(oracle.decode_e4m3(np.array([0x7F], dtype=np.uint8))[0])
    assert math.isnan(oracle.decode_e4m3(np.array([0xFF], dtype=np.uint8))[0])


def test_every_byte_matches_torch_e4m3fn():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode_e4m3(b)
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_scale_multiplies():
    b = np.array([0x38, 0x7E, 0x01], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.decode_e4m3(b, 0.25), [0.25, 112.0, 2.0 ** -11])


FP8_MUTANTS = {
    "bias_8": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "subnormal_as_normal": ("v = ldexp((double)m / 8.0, -6);", "v = ldexp(1.0 + (double)m / 8.0, -7);"),
    "no_nan": ("if (e == 15 && m == 7)\n        return NAN;", "if (0)\n        return NAN;"),
}


@pytest.mark.parametrize("name", sorted(FP8_MUTANTS))
def test_planted_fp8_mistake_is_caught(name, tmp_path):
    old, new = FP8_MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gqa_oracle.c")).read()
    assert src.count(old) == 1, name
    c_path = tmp_path / f"{name}.c"
    c_path.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(force=True, src=str(c_path), out=str(tmp_path / f"lib{name}.so")))
    saved = oracle._lib
    oracle._lib = lib
    failures = 0
    try:
        for pin in (test_hand_decoded_bytes, test_every_byte_matches_torch_e4m3fn):
            try:
                pin()
            except AssertionError:
                failures += 1
    finally:
        oracle._lib = saved
    assert failures > 0
