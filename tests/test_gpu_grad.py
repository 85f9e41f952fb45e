"""GPU parity of the grouped-GEMM gradients (moe_grouped_gemm_dgrad /
moe_grouped_gemm_wgrad) against the CPU oracle.

Shapes span several tiles with ragged tails: experts of 0, a few and several
hundred rows (wgrad reads each expert's rows in 64-row k-blocks, its partial
last block from a zero-padded copy: remainders 0, 1, 31, 32, 33 and 63), N
and K not multiples of the tile.  Sentinel rows of the inputs are NaN: dA's
sentinel rows must come out exactly zero and nothing else may change.  The
full-size case (the 32-expert layer's gate_up shape) is checked on sampled
rows of dA and sampled (expert, row) pairs of dB."""
import numpy as np
import pytest
import torch

import oracle
from grouped_gemm_serving_gb300 import synth
from tests.gpu_helpers import assert_close_bf16, dev, dev_bf16, host_bf16_bits, host_f32_from_bf16, require_gpu

pytestmark = pytest.mark.gpu

BF16_NAN = 0x7FC0


@pytest.fixture(scope="module")
def moe():
    require_gpu()
    from grouped_gemm_serving_gb300 import moe as m
    return m


def _weights(E, N, K, seed, std=0.05):
    return np.stack([synth.dense_rows(N, K, seed * 1000 + e, std=std, tensor_id=4) for e in range(E)])


def _operands(E, M_cap, live, N, K, seed, counts=None, empty=1):
    if counts is None:
        off = synth.grouped_offsets(E, live, seed=seed, empty_experts=empty)
    else:
        off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    live = int(off[-1])
    A = synth.dense_rows(M_cap, K, seed=seed + 1, std=1.0, tensor_id=1)
    dC = synth.dense_rows(M_cap, N, seed=seed + 2, std=1.0, tensor_id=2)
    A[live:] = BF16_NAN
    dC[live:] = BF16_NAN
    return off, live, A, _weights(E, N, K, seed + 3), dC


CASES = [
    # E, M_cap, live, N, K, expert counts (None: random split)
    (4, 300, 260, 264, 200, None),
    (8, 1100, 1000, 512, 136, None),
    (12, 4130, 0, 392, 200, [1, 31, 32, 33, 255, 256, 257, 512, 513, 700, 0, 1500]),
    (3, 129, 129, 256, 64, None),
]


def _ws(moe, n):
    return torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("E,M_cap,live,N,K,counts", CASES)
def test_dgrad(moe, E, M_cap, live, N, K, counts):
    off, live, A, B, dC = _operands(E, M_cap, live, N, K, seed=E + N, counts=counts)
    ref = oracle.grouped_gemm_dgrad_bf16(dC, B, off)
    dA = torch.full((M_cap, K), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    n = moe.moe_grouped_gemm_dgrad_workspace_size(E, N, K)
    moe.moe_grouped_gemm_dgrad(dev_bf16(dC), dev_bf16(B), dev(off), E, M_cap, N, K, dA, _ws(moe, n), n)
    assert moe.moe_get_device_error() == 0
    assert_close_bf16(host_f32_from_bf16(dA)[:live], ref[:live])
    assert np.all(host_bf16_bits(dA)[live:] == 0)


@pytest.mark.parametrize("E,M_cap,live,N,K,counts", CASES)
def test_wgrad(moe, E, M_cap, live, N, K, counts):
    off, live, A, B, dC = _operands(E, M_cap, live, N, K, seed=2 * E + K, counts=counts)
    ref = oracle.grouped_gemm_wgrad_bf16(A, dC, off, E)
    dB = torch.full((E, N, K), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    n = moe.moe_grouped_gemm_wgrad_workspace_size(E, M_cap, N, K)
    moe.moe_grouped_gemm_wgrad(dev_bf16(A), dev_bf16(dC), dev(off), E, M_cap, N, K, dB, _ws(moe, n), n)
    assert moe.moe_get_device_error() == 0
    got = host_f32_from_bf16(dB)
    for e in range(E):
        if off[e] == off[e + 1]:
            assert np.all(host_bf16_bits(dB)[e] == 0)
        else:
            assert_close_bf16(got[e], ref[e])


def test_wgrad_256_experts_every_tail(moe):
    # the most experts the library takes: every remainder mod 64 (the tail copy)
    # and empty experts, 8 experts per lane in the kernel's prefix
    E, N, K = 256, 72, 40
    counts = np.array([(7 * e) % 131 if e % 9 else 0 for e in range(E)], np.int64)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    live = int(off[-1])
    M_cap = live + 16
    A = synth.dense_rows(M_cap, K, seed=31, std=1.0, tensor_id=1)
    dC = synth.dense_rows(M_cap, N, seed=32, std=1.0, tensor_id=2)
    A[live:] = BF16_NAN
    dC[live:] = BF16_NAN
    ref = oracle.grouped_gemm_wgrad_bf16(A, dC, off, E)
    dB = torch.full((E, N, K), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    n = moe.moe_grouped_gemm_wgrad_workspace_size(E, M_cap, N, K)
    moe.moe_grouped_gemm_wgrad(dev_bf16(A), dev_bf16(dC), dev(off), E, M_cap, N, K, dB, _ws(moe, n), n)
    assert moe.moe_get_device_error() == 0
    got = host_f32_from_bf16(dB)
    for e in range(E):
        if counts[e] == 0:
            assert np.all(host_bf16_bits(dB)[e] == 0)
        else:
            assert_close_bf16(got[e], ref[e])


def test_invalid_offsets_are_reported_and_nothing_is_read(moe):
    E, M_cap, N, K = 3, 100, 64, 64
    off = np.array([0, 60, 50, 100], np.int32)           # decreasing
    A = torch.zeros((M_cap, K), dtype=torch.bfloat16, device="cuda")
    dC = torch.zeros((M_cap, N), dtype=torch.bfloat16, device="cuda")
    dB = torch.full((E, N, K), 9, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    n = moe.moe_grouped_gemm_wgrad_workspace_size(E, M_cap, N, K)
    moe.moe_grouped_gemm_wgrad(A, dC, dev(off), E, M_cap, N, K, dB, _ws(moe, n), n)
    assert moe.moe_get_device_error() == moe.MOE_DEVERR_OFFSETS
    assert np.all(host_bf16_bits(dB).view(np.int16) == 9)


@pytest.mark.slow
def test_full_size_gate_up_gradients_sampled(moe):
    # the 32-expert layer's gate_up GEMM: 16384 rows, N = 2 * 2880, K = 2880
    wl = synth.WORKLOADS["32e-top4-h2880"]
    E, N, K, M_cap = wl.E, 2 * wl.I, wl.H, wl.T * wl.k
    ids, _ = oracle.route_topk(synth.router_logits(wl), synth.expert_bias(wl), wl.k, wl.renormalize)
    off = np.concatenate([[0], np.cumsum(np.bincount(ids.reshape(-1), minlength=E))]).astype(np.int32)
    A = synth.dense_rows(M_cap, K, seed=5, std=1.0, tensor_id=1)
    dC = synth.dense_rows(M_cap, N, seed=6, std=1.0, tensor_id=2)
    B = synth.expert_weights(wl, "w1")
    dA = torch.empty((M_cap, K), dtype=torch.bfloat16, device="cuda")
    dB = torch.empty((E, N, K), dtype=torch.bfloat16, device="cuda")
    Ad, dCd, offd = dev_bf16(A), dev_bf16(dC), dev(off)
    n1 = moe.moe_grouped_gemm_dgrad_workspace_size(E, N, K)
    moe.moe_grouped_gemm_dgrad(dCd, dev_bf16(B), offd, E, M_cap, N, K, dA, _ws(moe, n1), n1)
    n2 = moe.moe_grouped_gemm_wgrad_workspace_size(E, M_cap, N, K)
    moe.moe_grouped_gemm_wgrad(Ad, dCd, offd, E, M_cap, N, K, dB, _ws(moe, n2), n2)
    assert moe.moe_get_device_error() == 0
    g = np.random.default_rng(7)
    rows = np.sort(g.choice(M_cap, 24, replace=False)).astype(np.int32)
    rows[0], rows[-1] = 0, M_cap - 1
    assert_close_bf16(host_f32_from_bf16(dA)[rows], oracle.grouped_gemm_dgrad_bf16(dC, B, off, rows=rows))
    pairs = np.stack([g.integers(0, E, 24), g.integers(0, N, 24)], axis=1).astype(np.int32)
    pairs[0] = [0, 0]
    pairs[-1] = [E - 1, N - 1]
    got = host_f32_from_bf16(dB)[pairs[:, 0], pairs[:, 1]]
    assert_close_bf16(got, oracle.grouped_gemm_wgrad_bf16(A, dC, off, E, pairs=pairs))


def test_gradients_are_bit_reproducible(moe):
    E, M_cap, live, N, K = 8, 1100, 1000, 512, 136
    off, live, A, B, dC = _operands(E, M_cap, live, N, K, seed=17)
    Ad, Bd, dCd, offd = dev_bf16(A), dev_bf16(B), dev_bf16(dC), dev(off)
    n1 = moe.moe_grouped_gemm_dgrad_workspace_size(E, N, K)
    n2 = moe.moe_grouped_gemm_wgrad_workspace_size(E, M_cap, N, K)
    outs = []
    for _ in range(2):
        dA = torch.empty((M_cap, K), dtype=torch.bfloat16, device="cuda")
        dB = torch.empty((E, N, K), dtype=torch.bfloat16, device="cuda")
        moe.moe_grouped_gemm_dgrad(dCd, Bd, offd, E, M_cap, N, K, dA, _ws(moe, n1), n1)
        moe.moe_grouped_gemm_wgrad(Ad, dCd, offd, E, M_cap, N, K, dB, _ws(moe, n2), n2)
        assert moe.moe_get_device_error() == 0
        outs.append((host_bf16_bits(dA), host_bf16_bits(dB)))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


def test_dgrad_needs_no_workspace(moe):
    """The data gradient reads the weights in place (MN-major): no workspace."""
    E, M_cap, live, N, K = 5, 700, 650, 320, 192
    off, live, A, B, dC = _operands(E, M_cap, live, N, K, seed=17, counts=None)
    assert moe.moe_grouped_gemm_dgrad_workspace_size(E, N, K) == 0
    dA = torch.full((M_cap, K), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm_dgrad(dev_bf16(dC), dev_bf16(B), dev(off), E, M_cap, N, K, dA, None, 0)
    assert moe.moe_get_device_error() == 0
    assert_close_bf16(host_f32_from_bf16(dA)[:live], oracle.grouped_gemm_dgrad_bf16(dC, B, off)[:live])
    assert np.all(host_bf16_bits(dA)[live:] == 0)
