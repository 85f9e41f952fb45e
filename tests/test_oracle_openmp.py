"""The oracle's OpenMP build (used only to time the CPU baseline on all host
cores) must give the same bits as its one-core build: the threads split the
independent rows, and every output element is still summed by one thread in
the same order."""
import numpy as np
import pytest

import oracle
from grouped_gemm_serving_gb300 import synth


def _both(fn):
    prev = oracle.use_openmp(False)
    try:
        one = fn()
        oracle.use_openmp(True)
        many = fn()
    finally:
        oracle.use_openmp(prev)
    return one, many


def _same(a, b):
    if isinstance(a, dict):
        return all(_same(a[k], b[k]) for k in a)
    if isinstance(a, (tuple, list)):
        return all(_same(x, y) for x, y in zip(a, b))
    return np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


def test_openmp_build_runs_on_several_threads():
    prev = oracle.use_openmp(True)
    try:
        assert oracle.threads() >= 1
    finally:
        oracle.use_openmp(prev)
    prev = oracle.use_openmp(False)
    try:
        assert oracle.threads() == 1
    finally:
        oracle.use_openmp(prev)


@pytest.mark.parametrize("fp8", [False, True])
def test_layer_bit_identical(fp8):
    wl = synth.Workload("omp", T=96, E=12, k=3, H=256, I=384, n_sentinel=17, bias="normal0.5",
                        dtype="fp8" if fp8 else "bf16")
    x, W1, W2 = (synth.hidden_states(wl), synth.expert_weights(wl, "w1"),
                 synth.expert_weights(wl, "w2"))
    kw = dict(E=wl.E, k=wl.k, logits=synth.router_logits(wl), bias=synth.expert_bias(wl),
              sentinel_mask=synth.sentinel_mask(wl))

    def run():
        if not fp8:
            return oracle.moe_forward(x, W1, W2, **kw)
        q1, s1 = oracle.quant_weight_fp8(W1)
        q2, s2 = oracle.quant_weight_fp8(W2)
        return (q1, s1, q2, s2), oracle.moe_forward(x, q1, q2, W1_scales=s1, W2_scales=s2, **kw)

    one, many = _both(run)
    assert _same(one, many)


def test_gradients_bit_identical():
    g = np.random.default_rng(3)
    E, M, N, K = 5, 200, 96, 136
    off = synth.grouped_offsets(E, 180, seed=2, empty_experts=1)
    A = synth.grouped_rows(M, K, 180, seed=1)
    A[180:] = 0
    dC = synth.to_bf16_bits(g.standard_normal((M, N), dtype=np.float32))
    B = synth.to_bf16_bits(g.standard_normal((E, N, K), dtype=np.float32))
    one, many = _both(lambda: (oracle.grouped_gemm_dgrad_bf16(dC, B, off),
                               oracle.grouped_gemm_wgrad_bf16(A, dC, off, E)))
    assert _same(one, many)
