"""Pins of the oracle's batched expert product (batched_mm /
batched_fp8_matmul: every routed slot's token row times its expert's
weight, no sort, no weighting): against numpy float64 matrix products of the
widened (bf16) or dequantised (e4m3 value x scale) operands, and against the
pinned grouped GEMM on the slots sorted by expert, put back in slot order."""
import numpy as np
import pytest

import oracle
from grouped_gemm_serving_gb300 import synth
from grouped_gemm_serving_gb300.synth import bf16_bits_to_f32


def _case(T, k, E, N, K, n_sent, seed):
    g = np.random.default_rng(seed)
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    flat = ids.reshape(-1)
    flat[g.choice(flat.size, n_sent, replace=False)] = E
    x = synth.dense_rows(T, K, seed, std=1.0)
    W = np.stack([synth.dense_rows(N, K, seed * 100 + e, std=0.05, tensor_id=4) for e in range(E)])
    return ids, x, W


@pytest.mark.parametrize("T,k,E,N,K,n_sent", [(13, 3, 7, 40, 256, 4), (5, 1, 2, 200, 128, 0), (9, 4, 4, 96, 384, 9)])
def test_bf16_against_numpy_products(T, k, E, N, K, n_sent):
    ids, x, W = _case(T, k, E, N, K, n_sent, T * 7 + N)
    out = oracle.batched_matmul(x, ids, W, E)
    xf, Wf = bf16_bits_to_f32(x).astype(np.float64), bf16_bits_to_f32(W).astype(np.float64)
    for f, e in enumerate(ids.reshape(-1)):
        ref = np.zeros(N) if e == E else Wf[e] @ xf[f // k]
        np.testing.assert_allclose(out[f], ref, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("T,k,E,N,K,n_sent", [(11, 2, 5, 300, 256, 3), (6, 4, 8, 128, 384, 5)])
def test_fp8_against_dequantised_numpy_products(T, k, E, N, K, n_sent):
    ids, x, W = _case(T, k, E, N, K, n_sent, T * 11 + N)
    qx, sx = oracle.quant_act_fp8(x)
    qw, sw = oracle.quant_weight_fp8(W)
    out = oracle.batched_matmul(qx, ids, qw, E, x_scales=sx, W_scales=sw)
    xd = oracle.e4m3_decode(qx).astype(np.float64) * np.repeat(sx, 128, axis=1)
    Wd = oracle.e4m3_decode(qw).astype(np.float64) * np.repeat(np.repeat(sw, 128, axis=1)[:, :N], 128, axis=2)
    for f, e in enumerate(ids.reshape(-1)):
        ref = np.zeros(N) if e == E else Wd[e] @ xd[f // k]
        np.testing.assert_allclose(out[f], ref, rtol=1e-5, atol=1e-5)


def test_equals_grouped_gemm_in_slot_order():
    T, k, E, N, K = 20, 3, 6, 72, 128
    ids, x, W = _case(T, k, E, N, K, 5, 3)
    sr, rp, off = oracle.sort_by_expert(ids, E)
    xp = oracle.permute(x, k, sr, int(off[-1]))
    C = oracle.grouped_gemm_bf16(xp, W, off)
    out = oracle.batched_matmul(x, ids, W, E)
    live = ids.reshape(-1) != E
    assert np.array_equal(out[live], C[rp][live]) and np.all(out[~live] == 0)
