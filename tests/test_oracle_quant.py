"""Pins of the oracle's fine-grained FP8 quantisation (per token per 128
columns for activations, per 128x128 block for weights).

Where a group's amax is 448 * 2^j the scale is exactly 2^j and the codes must
equal PyTorch's e4m3 conversion of x / 2^j; this fixes the constant 448, the
grouping direction and the scale layout.  Random groups are checked against
the closed-form rounding bound and the fact that the amax element lands on
+-448."""
import numpy as np
import pytest
import torch

from grouped_gemm_serving_gb300.synth import bf16_bits_to_f32, to_bf16_bits
from oracle import e4m3_decode, quant_act_fp8, quant_weight_fp8


def _torch_e4m3(v):
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def _groups_with_amax(rows, groups, g):
    """bf16 values whose group (r, j) has amax exactly 448 * 2^-(r+j) (mod 6)."""
    x = g.uniform(-1, 1, size=(rows, groups, 128)).astype(np.float32)
    expo = (np.arange(rows)[:, None] + np.arange(groups)[None, :]) % 6
    x = bf16_bits_to_f32(to_bf16_bits(x * 400.0))
    pos = g.integers(0, 128, size=(rows, groups))
    for r in range(rows):
        for j in range(groups):
            x[r, j, pos[r, j]] = 448.0 if (r + j) % 2 else -448.0
    x *= (2.0 ** -expo)[..., None].astype(np.float32)
    return to_bf16_bits(x.reshape(rows, groups * 128)), 2.0 ** -expo


def test_act_quant_exact_power_of_two_scales():
    g = np.random.default_rng(1)
    xb, scale = _groups_with_amax(6, 3, g)
    q, s = quant_act_fp8(xb)
    assert s.shape == (6, 3)
    assert np.array_equal(s, scale.astype(np.float32))            # row-major [M, K/128]
    x = bf16_bits_to_f32(xb).reshape(6, 3, 128)
    want = _torch_e4m3(x / scale[..., None].astype(np.float32)).reshape(6, 384)
    assert np.array_equal(q, want)


def test_act_quant_zero_group_and_tiny_values():
    x = np.zeros((2, 256), np.float32)
    x[1, 128:] = 2.0 ** -20             # tiny but nonzero: scale 2^-20/448, codes 448
    q, s = quant_act_fp8(to_bf16_bits(x))
    assert s[0, 0] == 1.0 and s[0, 1] == 1.0 and s[1, 0] == 1.0
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0)
    assert s[1, 1] == np.float32(2.0 ** -20) / np.float32(448.0)
    assert np.all(e4m3_decode(q[1, 128:]) == 448.0)


@pytest.mark.parametrize("M,K,std", [(33, 128, 1.0), (16, 1024, 3.0), (8, 512, 1e-3)])
def test_act_quant_random_bound_and_amax_code(M, K, std):
    g = np.random.default_rng([M, K])
    xb = to_bf16_bits(g.standard_normal((M, K), dtype=np.float32) * np.float32(std))
    q, s = quant_act_fp8(xb)
    x = bf16_bits_to_f32(xb).reshape(M, K // 128, 128).astype(np.float64)
    dq = e4m3_decode(q).reshape(M, K // 128, 128).astype(np.float64)
    sc = s.astype(np.float64)[..., None]
    amax = np.abs(x).max(-1)
    # the amax element of every group encodes to +-448
    assert np.all(np.abs(dq).max(-1) == 448.0)
    np.testing.assert_allclose(s, amax / 448.0, rtol=1e-7)
    # half an e4m3 ulp: 2^-4 relative for normals, 2^-10 * s absolute below 2^-6 * s
    err = np.abs(dq * sc - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, sc * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(err <= bound)


def test_weight_quant_blocks_and_short_last_block():
    g = np.random.default_rng(2)
    E, N, K = 2, 200, 256            # row blocks of 128 and 72
    w = g.uniform(-1, 1, size=(E, N, K)).astype(np.float32) * 300
    scale = np.empty((E, 2, 2))
    for e in range(E):
        for nb in range(2):
            for kb in range(2):
                j = (e + 2 * nb + kb) % 5
                blk = w[e, nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
                blk[3 % blk.shape[0], 7] = 448.0
                blk *= 2.0 ** -j
                scale[e, nb, kb] = 2.0 ** -j
    wb = to_bf16_bits(w)
    q, s = quant_weight_fp8(wb)
    assert s.shape == (E, 2, 2)
    assert np.array_equal(s, scale.astype(np.float32))
    wf = bf16_bits_to_f32(wb)
    rowscale = np.repeat(np.repeat(scale, 128, axis=1)[:, :N], 128, axis=2)
    assert np.array_equal(q, _torch_e4m3(wf / rowscale.astype(np.float32)))


def test_weight_quant_random_bound():
    g = np.random.default_rng(3)
    wb = to_bf16_bits(g.standard_normal((3, 256, 384), dtype=np.float32) * np.float32(0.02))
    q, s = quant_weight_fp8(wb)
    w = bf16_bits_to_f32(wb).astype(np.float64)
    sc = np.repeat(np.repeat(s.astype(np.float64), 128, 1), 128, 2)
    dq = e4m3_decode(q).astype(np.float64) * sc
    assert np.all(np.abs(dq - w) <= np.maximum(np.abs(w) * 2.0 ** -4, sc * 2.0 ** -10) * (1 + 1e-6))
    blocks = np.abs(e4m3_decode(q)).reshape(3, 2, 128, 3, 128).max(axis=(2, 4))
    assert np.all(blocks == 448.0)
