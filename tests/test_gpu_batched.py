"""GPU parity of moe_batched_matmul (the batched_mm / batched_fp8_matmul
expert backend: every routed slot's token row times its expert's weight,
returned in slot order) against the oracle, and bit for bit against
moe_permute + moe_grouped_gemm's rows put back in slot order.  Shapes: a
decode batch over 256 experts, ragged tails, sentinel slots, bf16 and FP8."""
import numpy as np
import pytest
import torch

import oracle
from grouped_gemm_serving_gb300 import synth
from tests.gpu_helpers import assert_close_bf16, dev, dev_bf16, host, host_bf16_bits, host_f32_from_bf16, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    require_gpu()
    from grouped_gemm_serving_gb300 import moe as m
    return m


def _ids(T, k, E, n_sent, seed):
    g = np.random.default_rng(seed)
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    flat = ids.reshape(-1)
    if n_sent:
        flat[g.choice(flat.size, n_sent, replace=False)] = E
    return ids


def _run(moe, dtype, x, xs, ids, W, Ws, E, N, K):
    T, k = ids.shape
    out = torch.full((T * k, N), 7, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    nws = moe.moe_batched_matmul_workspace_size(dtype, T, K, k, E, N)
    assert nws > 0
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    ids_d = dev(ids)
    moe.moe_batched_matmul(dtype, x, xs, T, K, ids_d, k, W, Ws, E, N, out, ws, nws)
    assert moe.moe_get_device_error() == 0
    assert np.array_equal(host(ids_d), ids)                  # the caller's ids are untouched
    return out


@pytest.mark.parametrize("T,k,E,N,K,n_sent", [(64, 8, 256, 256, 512, 0), (37, 3, 11, 264, 200, 9),
                                             (300, 2, 4, 128, 136, 50), (1, 1, 1, 128, 64, 0)])
def test_bf16(moe, T, k, E, N, K, n_sent):
    ids = _ids(T, k, E, n_sent, T + N)
    x = synth.dense_rows(T, K, 5)
    W = np.stack([synth.dense_rows(N, K, 100 + e, std=0.05, tensor_id=4) for e in range(E)])
    out = _run(moe, moe.MOE_BF16, dev_bf16(x), None, ids, dev_bf16(W), None, E, N, K)
    ref = oracle.batched_matmul(x, ids, W, E)
    got = host_f32_from_bf16(out)
    live = ids.reshape(-1) != E
    assert_close_bf16(got[live], ref[live])
    assert np.all(host_bf16_bits(out)[~live] == 0)
    # bit for bit the rows of the two-step path, in slot order
    r = moe.route_sort_t(E, k, topk_ids=dev(ids))
    R = T * k
    xp = torch.empty((R, K), dtype=torch.bfloat16, device="cuda")
    C = torch.empty((R, N), dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(moe.MOE_BF16, dev_bf16(x), None, T, K, k, r["sorted_rows"], r["offsets"], E, R, xp, None)
    moe.moe_grouped_gemm(moe.MOE_BF16, xp, None, dev_bf16(W), None, r["offsets"], E, R, N, K, moe.MOE_EPI_STORE,
                         C, None)
    assert np.array_equal(host_bf16_bits(out), host_bf16_bits(C)[host(r["row_pos"])])


@pytest.mark.parametrize("T,k,E,N,K,n_sent", [(64, 8, 256, 256, 512, 5), (45, 3, 9, 384, 256, 11)])
def test_fp8(moe, T, k, E, N, K, n_sent):
    ids = _ids(T, k, E, n_sent, T * 3 + N)
    x = synth.dense_rows(T, K, 6)
    W = np.stack([synth.dense_rows(N, K, 200 + e, std=0.05, tensor_id=4) for e in range(E)])
    qx, sx = oracle.quant_act_fp8(x)
    qw, sw = oracle.quant_weight_fp8(W)
    out = _run(moe, moe.MOE_FP8_E4M3_B128, dev(qx), dev(sx), ids, dev(qw), dev(sw), E, N, K)
    ref = oracle.batched_matmul(qx, ids, qw, E, x_scales=sx, W_scales=sw)
    got = host_f32_from_bf16(out)
    live = ids.reshape(-1) != E
    assert_close_bf16(got[live], ref[live], rtol=2.0 ** -7, row_atol=2e-3)
    assert np.all(host_bf16_bits(out)[~live] == 0)


def test_bad_id_is_reported_and_its_row_zero(moe):
    T, k, E, N, K = 20, 2, 4, 64, 64
    ids = _ids(T, k, E, 0, 1)
    ids[3, 1] = 9
    x = synth.dense_rows(T, K, 7)
    W = np.stack([synth.dense_rows(N, K, 300 + e, std=0.05, tensor_id=4) for e in range(E)])
    out = torch.empty((T * k, N), dtype=torch.bfloat16, device="cuda")
    nws = moe.moe_batched_matmul_workspace_size(moe.MOE_BF16, T, K, k, E, N)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    ids_d = dev(ids)
    moe.moe_batched_matmul(moe.MOE_BF16, dev_bf16(x), None, T, K, ids_d, k, dev_bf16(W), None, E, N, out, ws, nws)
    assert moe.moe_get_device_error() == moe.MOE_DEVERR_ROUTE
    assert np.all(host_bf16_bits(out)[7] == 0) and host(ids_d)[3, 1] == 9
