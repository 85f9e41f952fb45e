"""Pins of the oracle's e4m3 codec (OCP FP8 E4M3FN) to things other than itself:
the format definition in integer-significand form, and PyTorch's
``float8_e4m3fn`` conversion (round to nearest even), exhaustively over every
fp32 value that can round to a nonzero finite code."""
import math

import numpy as np
import pytest
import torch

from oracle import e4m3_decode, e4m3_encode


def _definition(c: int) -> float:
    # value = (-1)^s * significand * 2^(exponent - bias - 3), significand = 8 + m
    # for normal codes and m for subnormal ones (exponent field 0 acts as 1).
    s = -1.0 if c & 0x80 else 1.0
    e, m = (c >> 3) & 15, c & 7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return s * m * 2.0 ** (1 - 7 - 3)
    return s * (8 + m) * 2.0 ** (e - 7 - 3)


def test_decode_all_codes_match_definition_and_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3_decode(codes)
    ref = np.array([_definition(int(c)) for c in codes], dtype=np.float32)
    lib = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(np.isnan(ours), nan) and np.array_equal(np.isnan(lib), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(ours[~nan], lib[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def _bits(x: float) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0])


def test_encode_exhaustive_against_torch():
    # every positive fp32 in [2^-11, 464): below 2^-11 everything is 0, and
    # torch overflows to NaN from 464 on, where the oracle saturates instead
    lo, hi = _bits(2.0 ** -11), _bits(464.0)
    step = 1 << 23
    for start in range(lo, hi, step):
        u = np.arange(start, min(start + step, hi), dtype=np.uint32)
        v = u.view(np.float32)
        ours = e4m3_encode(v)
        lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        bad = np.nonzero(ours != lib)[0]
        assert bad.size == 0, (v[bad[:5]], ours[bad[:5]], lib[bad[:5]])
        neg = e4m3_encode(-v[:: 4099])
        assert np.array_equal(neg, ours[:: 4099] | 0x80)


def test_encode_saturates_and_special_values():
    big = np.array([448.0, 448.5, 463.99, 464.0, 480.0, 1e6, 3e38, np.inf], np.float32)
    assert np.all(e4m3_encode(big) == 0x7E)
    assert np.all(e4m3_encode(-big) == 0xFE)
    assert e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F
    tiny = np.array([0.0, 1e-30, 2.0 ** -11 * 0.999, 2.0 ** -10], np.float32)
    assert np.all(e4m3_encode(tiny) == 0)           # 2^-10 is the 0 / 2^-9 tie -> even (0)
    assert e4m3_encode(np.array([-0.0], np.float32))[0] == 0x80
    assert e4m3_encode(np.array([2.0 ** -10 * 1.0001], np.float32))[0] == 1


@pytest.mark.parametrize("c", [c for c in range(256) if c not in (0x7F, 0xFF)])
def test_round_trip_every_finite_code(c):
    v = e4m3_decode(np.array([c], np.uint8))
    back = e4m3_encode(v)[0]
    assert back == c or (c == 0x80 and back == 0x80) or (v[0] == 0 and back in (0, 0x80))
