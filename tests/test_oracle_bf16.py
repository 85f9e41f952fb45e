"""Pin of the oracle's fp32 -> bf16 rounding (orc_bf16_round).

The FP8 layer rounds the SwiGLU output h to bf16 before quantising it (the
precision the unfused path stores h in), so this rounding decides the bytes
the down GEMM reads.  bf16 is the upper half of an fp32; the rounding is to
nearest, ties to the even upper half, overflowing to infinity.  It is checked
against PyTorch's float32 -> bfloat16 conversion on every upper half (every
sign, exponent and leading mantissa, subnormals, zeros, infinities and NaNs)
combined with the lower halves that decide a rounding (0, 1, just below half,
exactly half, just above half, all ones) and random ones, and against values
worked out by hand: ties of both parities, the largest finite value and the
overflow above it."""
import numpy as np
import torch

from oracle import bf16_round


def _torch_bf16_bits(f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _is_nan_bits(b: np.ndarray) -> np.ndarray:
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


def test_every_upper_half_against_torch():
    g = np.random.default_rng(11)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000], np.uint32)
    lows = np.concatenate([lows, g.integers(0, 1 << 16, size=8, dtype=np.uint32)])
    highs = np.arange(1 << 16, dtype=np.uint32)
    u = ((highs[:, None] << 16) | lows[None, :]).reshape(-1)
    f = u.view(np.float32)
    got = bf16_round(f)
    want = _torch_bf16_bits(f)
    nan_in = np.isnan(f)
    assert np.array_equal(got[~nan_in], want[~nan_in])
    assert np.all(_is_nan_bits(got[nan_in]))


def test_random_values_against_torch():
    g = np.random.default_rng(12)
    u = g.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    ok = ~np.isnan(f)
    assert np.array_equal(bf16_round(f)[ok], _torch_bf16_bits(f)[ok])


def test_hand_worked_values():
    cases = {
        0x3F800000: 0x3F80,   # 1.0 exact
        0x3F808000: 0x3F80,   # exact tie, lower half even: stays
        0x3F818000: 0x3F82,   # exact tie, lower half odd: rounds up to even
        0x3F807FFF: 0x3F80,   # just below half: down
        0x3F808001: 0x3F81,   # just above half: up
        0xBF818000: 0xBF82,   # sign is kept, ties the same way
        0x00000000: 0x0000,   # +0
        0x80000000: 0x8000,   # -0
        0x00008000: 0x0000,   # subnormal tie at zero, even: stays zero
        0x00018000: 0x0002,   # subnormal tie, odd: up
        0x7F7F7FFF: 0x7F7F,   # largest finite stays finite below the half
        0x7F7F8000: 0x7F80,   # tie at the top, odd: overflows to +inf
        0x7F7FFFFF: 0x7F80,   # FLT_MAX: +inf
        0xFF7FFFFF: 0xFF80,   # -FLT_MAX: -inf
        0x7F800000: 0x7F80,   # +inf
        0xFF800000: 0xFF80,   # -inf
    }
    u = np.array(list(cases), np.uint32)
    got = bf16_round(u.view(np.float32))
    assert [int(v) for v in got] == list(cases.values())
    nan = bf16_round(np.array([np.nan, -np.nan], np.float32))
    assert np.all(_is_nan_bits(nan))
