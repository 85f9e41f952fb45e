"""Pins of the oracle's grouped-GEMM gradients (dA, dB of C = A B[e]^T over
each expert's rows), each through something other than the gradient code:

* the forward oracle on unit inputs: the loss <dC, C> is linear in A and in
  B, so with A (or B) a single 1 at (p, c) (or (e, n, c)) it equals exactly
  the gradient entry there;
* the adjoint identity <dC, A B^T> = <dA, A> = <dB, B>;
* numpy fp64 matrix products per expert;
* sentinel rows get zero dA, experts without rows zero dB."""
import numpy as np
import pytest

import oracle
from grouped_gemm_serving_gb300 import synth
from grouped_gemm_serving_gb300.synth import bf16_bits_to_f32


def _case(E, M_cap, live, N, K, seed, empty=1):
    off = synth.grouped_offsets(E, live, seed=seed, empty_experts=empty)
    A = synth.dense_rows(M_cap, K, seed=seed + 1, std=1.0, tensor_id=1)
    B = np.stack([synth.dense_rows(N, K, seed * 100 + e, std=0.1, tensor_id=4) for e in range(E)])
    dC = synth.dense_rows(M_cap, N, seed=seed + 2, std=1.0, tensor_id=2)
    return off, A, B, dC


ONE = synth.to_bf16_bits(np.float32([1.0]))[0]


def _loss(dC, C):
    return float(np.sum(bf16_bits_to_f32(dC).astype(np.float64)[: C.shape[0]] * C.astype(np.float64)))


def test_dgrad_equals_forward_on_unit_inputs():
    E, M_cap, live, N, K = 3, 20, 17, 6, 5
    off, A, B, dC = _case(E, M_cap, live, N, K, seed=3)
    dA = oracle.grouped_gemm_dgrad_bf16(dC, B, off)
    g = np.random.default_rng(0)
    for p in list(g.choice(M_cap, 8, replace=False)) + [0, live - 1, live, M_cap - 1]:
        for c in (0, K - 1, int(g.integers(K))):
            U = np.zeros((M_cap, K), np.uint16)
            U[p, c] = ONE
            ref = _loss(dC, oracle.grouped_gemm_bf16(U, B, off))
            assert dA[p, c] == np.float32(ref), (p, c)


def test_wgrad_equals_forward_on_unit_inputs():
    E, M_cap, live, N, K = 4, 24, 21, 5, 6
    off, A, B, dC = _case(E, M_cap, live, N, K, seed=5)
    dB = oracle.grouped_gemm_wgrad_bf16(A, dC, off, E)
    g = np.random.default_rng(1)
    for e in range(E):
        for n in (0, N - 1, int(g.integers(N))):
            for c in (0, K - 1, int(g.integers(K))):
                U = np.zeros((E, N, K), np.uint16)
                U[e, n, c] = ONE
                ref = _loss(dC, oracle.grouped_gemm_bf16(A, U, off))
                assert dB[e, n, c] == np.float32(ref), (e, n, c)


@pytest.mark.parametrize("E,M_cap,live,N,K", [(4, 300, 260, 40, 24), (8, 200, 200, 16, 64)])
def test_adjoint_identity(E, M_cap, live, N, K):
    off, A, B, dC = _case(E, M_cap, live, N, K, seed=E + N)
    C = oracle.grouped_gemm_bf16(A, B, off)
    dA = oracle.grouped_gemm_dgrad_bf16(dC, B, off)
    dB = oracle.grouped_gemm_wgrad_bf16(A, dC, off, E)
    a, b = bf16_bits_to_f32(A).astype(np.float64), bf16_bits_to_f32(B).astype(np.float64)
    a[int(off[-1]):] = 0.0          # sentinel rows take no part in the product
    lhs = _loss(dC, C)
    for rhs in (np.sum(dA.astype(np.float64) * a), np.sum(dB.astype(np.float64) * b)):
        assert abs(lhs - rhs) <= 1e-5 * (1.0 + abs(lhs))


def test_against_numpy_products_per_expert():
    E, M_cap, live, N, K = 5, 120, 111, 24, 40
    off, A, B, dC = _case(E, M_cap, live, N, K, seed=11)
    dA = oracle.grouped_gemm_dgrad_bf16(dC, B, off)
    dB = oracle.grouped_gemm_wgrad_bf16(A, dC, off, E)
    a, b, g = (bf16_bits_to_f32(x).astype(np.float64) for x in (A, B, dC))
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        np.testing.assert_allclose(dA[r0:r1], g[r0:r1] @ b[e], rtol=1e-6, atol=1e-6)
        np.testing.assert_allclose(dB[e], g[r0:r1].T @ a[r0:r1], rtol=1e-6, atol=1e-6)


def test_sentinel_rows_and_empty_experts_get_zero_gradients():
    E, M_cap, live, N, K = 6, 90, 70, 12, 8
    off, A, B, dC = _case(E, M_cap, live, N, K, seed=21, empty=2)
    dA = oracle.grouped_gemm_dgrad_bf16(dC, B, off)
    dB = oracle.grouped_gemm_wgrad_bf16(A, dC, off, E)
    assert np.all(dA[live:] == 0)
    empty = [e for e in range(E) if off[e] == off[e + 1]]
    assert len(empty) >= 2
    for e in empty:
        assert np.all(dB[e] == 0)


def test_wgrad_pairs_select_rows_of_the_full_result():
    E, M_cap, live, N, K = 4, 60, 55, 10, 12
    off, A, B, dC = _case(E, M_cap, live, N, K, seed=31)
    full = oracle.grouped_gemm_wgrad_bf16(A, dC, off, E)
    pairs = np.array([[0, 0], [3, 9], [1, 4], [2, 7]], np.int32)
    part = oracle.grouped_gemm_wgrad_bf16(A, dC, off, E, pairs=pairs)
    for i, (e, n) in enumerate(pairs):
        assert np.array_equal(part[i], full[e, n])


def test_dgrad_rows_select_rows_of_the_full_result():
    E, M_cap, live, N, K = 4, 60, 50, 10, 12
    off, A, B, dC = _case(E, M_cap, live, N, K, seed=41)
    full = oracle.grouped_gemm_dgrad_bf16(dC, B, off)
    rows = np.array([0, 7, 49, 55], np.int32)
    assert np.array_equal(oracle.grouped_gemm_dgrad_bf16(dC, B, off, rows=rows), full[rows])
