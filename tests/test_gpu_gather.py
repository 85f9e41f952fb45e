"""GPU parity of the grouped GEMM whose A rows are gathered from token order
(moe_grouped_gemm_gather), against the CPU oracle (its permute followed by
its grouped GEMM) and bit for bit against the library's own two-kernel path
(moe_permute, then moe_grouped_gemm): the gathered tile holds the same bytes
in the same shared-memory layout, so the tensor-core sums are identical.

Routing comes from the oracle (top-k, sentinel marking, stable sort), so
sorted_rows and offsets are the same on both sides.  Shapes span several row
and column tiles, experts whose rows end inside a tile, and sentinel slots."""
import numpy as np
import pytest
import torch

import oracle
from grouped_gemm_serving_gb300 import synth
from tests.gpu_helpers import (assert_close_bf16, dev, dev_bf16, host, host_bf16_bits,
                               host_f32_from_bf16, require_gpu, row_rel_err)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    require_gpu()
    from grouped_gemm_serving_gb300 import moe as m
    return m


def _routing(T, E, k, seed, n_sentinel=0):
    g = np.random.default_rng(seed)
    logits = g.standard_normal((T, E)).astype(np.float32)
    ids, w = oracle.route_topk(logits, None, k)
    if n_sentinel:
        mask = np.zeros(T * k, np.uint8)
        mask[g.choice(T * k, n_sentinel, replace=False)] = 1
        ids = oracle.mark_sentinels(ids, mask, E).reshape(T, k)
    sr, rp, off = oracle.sort_by_expert(ids, E)
    return sr, off


def _weights(E, N, K, seed):
    return np.stack([synth.dense_rows(N, K, seed * 1000 + e, std=0.05, tensor_id=4) for e in range(E)])


BF16 = [
    # T, E, k, K (= H), N, epilogue, sentinel slots
    (300, 8, 2, 192, 272, "swiglu", 0),
    (1000, 16, 4, 256, 512, "swiglu", 37),
    (64, 256, 8, 128, 256, "swiglu", 5),
    (517, 32, 4, 2880, 768, "swiglu", 0),
    (300, 8, 2, 320, 264, "store", 11),
    (129, 3, 1, 64, 256, "store", 0),
]


@pytest.mark.parametrize("T,E,k,K,N,epi,n_sent", BF16)
def test_bf16_gather_matches_oracle_and_two_kernel_path(moe, T, E, k, K, N, epi, n_sent):
    sr, off = _routing(T, E, k, seed=T + E + K, n_sentinel=n_sent)
    R, L = T * k, int(off[-1])
    x = synth.dense_rows(T, K, seed=K + N, std=1.0, tensor_id=1)
    B = _weights(E, N, K, 3)
    swiglu = epi == "swiglu"
    e = moe.MOE_EPI_SWIGLU if swiglu else moe.MOE_EPI_STORE
    ncol = N // 2 if swiglu else N

    ref = oracle.grouped_gemm_bf16(oracle.permute(x, k, sr, L, M_cap=R), B, off)
    if swiglu:
        ref = oracle.swiglu(ref, L)

    xd, Bd, srd, offd = dev_bf16(x), dev_bf16(B), dev(sr), dev(off)
    Cg = torch.full((R, ncol), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm_gather(moe.MOE_BF16, xd, None, T, k, srd, Bd, None, offd, E, R, N, K, e, Cg, None)
    xp = torch.empty((R, K), dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(moe.MOE_BF16, xd, None, T, K, k, srd, offd, E, R, xp, None)
    Cp = torch.full((R, ncol), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm(moe.MOE_BF16, xp, None, Bd, None, offd, E, R, N, K, e, Cp, None)
    assert moe.moe_get_device_error() == 0

    got = host_f32_from_bf16(Cg)
    assert_close_bf16(got[:L], ref[:L])
    assert np.all(host_bf16_bits(Cg)[L:] == 0)
    assert np.array_equal(host_bf16_bits(Cg), host_bf16_bits(Cp))


FP8 = [
    # T, E, k, K, N, epilogue, sentinel slots
    (300, 8, 2, 256, 512, "swiglu_q", 0),
    (1000, 16, 4, 384, 768, "swiglu_q", 41),
    (200, 6, 2, 512, 384, "store", 9),
    (96, 256, 8, 128, 256, "swiglu", 13),
]


@pytest.mark.parametrize("T,E,k,K,N,epi,n_sent", FP8)
def test_fp8_gather_matches_oracle_and_two_kernel_path(moe, T, E, k, K, N, epi, n_sent):
    sr, off = _routing(T, E, k, seed=3 * T + E, n_sentinel=n_sent)
    R, L = T * k, int(off[-1])
    qx, sx = oracle.quant_act_fp8(synth.dense_rows(T, K, seed=N, std=1.0, tensor_id=1))
    qb, sb = oracle.quant_weight_fp8(_weights(E, N, K, 5))
    qp, sp = oracle.permute(qx, k, sr, L, x_scales=sx, M_cap=R)
    ref = oracle.grouped_gemm_fp8(qp, sp, qb, sb, off)
    e = {"store": moe.MOE_EPI_STORE, "swiglu": moe.MOE_EPI_SWIGLU, "swiglu_q": moe.MOE_EPI_SWIGLU_QUANT_FP8}[epi]
    if epi != "store":
        ref = oracle.swiglu(ref, L)
    ncol = N if epi == "store" else N // 2

    def out():
        if epi == "swiglu_q":
            return (torch.full((R, ncol), 7, dtype=torch.uint8, device="cuda"),
                    torch.full((ncol // 128, R), -1.0, dtype=torch.float32, device="cuda"))
        return torch.full((R, ncol), 11, dtype=torch.int16, device="cuda").view(torch.bfloat16), None

    xd, sxd, qbd, sbd, srd, offd = dev(qx), dev(sx), dev(qb), dev(sb), dev(sr), dev(off)
    Cg, Sg = out()
    moe.moe_grouped_gemm_gather(moe.MOE_FP8_E4M3_B128, xd, sxd, T, k, srd, qbd, sbd, offd, E, R, N, K, e, Cg, Sg)
    xp = torch.empty((R, K), dtype=torch.uint8, device="cuda")
    xps = torch.empty((K // 128, R), dtype=torch.float32, device="cuda")
    moe.moe_permute(moe.MOE_FP8_E4M3_B128, xd, sxd, T, K, k, srd, offd, E, R, xp, xps)
    Cp, Sp = out()
    moe.moe_grouped_gemm(moe.MOE_FP8_E4M3_B128, xp, xps, qbd, sbd, offd, E, R, N, K, e, Cp, Sp)
    assert moe.moe_get_device_error() == 0

    assert np.array_equal(host(Cg.view(torch.int16) if Sg is None else Cg),
                          host(Cp.view(torch.int16) if Sp is None else Cp))
    if epi == "swiglu_q":
        assert np.array_equal(host(Sg), host(Sp))
        deq = oracle.e4m3_decode(host(Cg)).reshape(R, ncol // 128, 128) * host(Sg).T[:, :, None]
        assert_close_bf16(deq.reshape(R, ncol)[:L], ref[:L], rtol=2.0 ** -4 + 2.0 ** -7, row_atol=4e-3)
        assert np.all(host(Cg)[L:] == 0) and np.all(host(Sg).T[L:] == 1.0)
    else:
        got = host_f32_from_bf16(Cg)
        assert_close_bf16(got[:L], ref[:L], rtol=2.0 ** -7, row_atol=2e-3)
        assert np.all(host_bf16_bits(Cg)[L:] == 0)


def test_out_of_range_slot_is_reported_and_other_rows_unaffected(moe):
    T, E, k, K, N = 64, 4, 2, 128, 256
    sr, off = _routing(T, E, k, seed=1)
    R = T * k
    x, B = synth.dense_rows(T, K, seed=2, std=1.0, tensor_id=1), _weights(E, N, K, 2)
    xd, Bd, offd = dev_bf16(x), dev_bf16(B), dev(off)

    def run(rows):
        C = torch.empty((R, N), dtype=torch.bfloat16, device="cuda")
        moe.moe_grouped_gemm_gather(moe.MOE_BF16, xd, None, T, k, dev(rows), Bd, None, offd, E, R, N, K,
                                    moe.MOE_EPI_STORE, C, None)
        return C

    clean = host_bf16_bits(run(sr))
    assert moe.moe_get_device_error() == 0
    bad = sr.copy()
    bad[5] = R + 7                      # a slot past T*k: its row must not be read
    got = host_bf16_bits(run(bad))
    assert moe.moe_get_device_error() == moe.MOE_DEVERR_ROUTE
    keep = np.arange(R) != 5
    assert np.array_equal(got[keep], clean[keep])


def test_live_rows_beyond_the_slots_skip_the_gemm(moe):
    T, E, k, K, N = 16, 2, 2, 64, 256
    R, M_cap = T * k, 128
    off = np.array([0, 20, 40], np.int32)   # 40 live rows, but only 32 slots exist
    C = torch.full((M_cap, N), 9, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm_gather(moe.MOE_BF16, torch.zeros((T, K), dtype=torch.bfloat16, device="cuda"), None,
                                T, k, dev(np.arange(R, dtype=np.int32)),
                                torch.zeros((E, N, K), dtype=torch.bfloat16, device="cuda"), None, dev(off), E,
                                M_cap, N, K, moe.MOE_EPI_STORE, C, None)
    assert moe.moe_get_device_error() == moe.MOE_DEVERR_OFFSETS
    assert np.all(host_bf16_bits(C).view(np.int16) == 9)


LAYERS = [synth.WORKLOADS["tiny-8e-top2"],
          synth.Workload("mid-16e-top4", T=700, E=16, k=4, H=512, I=384, n_sentinel=23)]


@pytest.mark.parametrize("wl", LAYERS, ids=lambda w: w.name)
@pytest.mark.parametrize("fp8", [False, True])
def test_forward_with_and_without_gather_agree(moe, wl, fp8):
    x, logits = synth.hidden_states(wl), synth.router_logits(wl)
    W1, W2 = synth.expert_weights(wl, "w1"), synth.expert_weights(wl, "w2")
    mask = synth.sentinel_mask(wl) if wl.n_sentinel else None
    if fp8:
        q1, s1 = oracle.quant_weight_fp8(W1)
        q2, s2 = oracle.quant_weight_fp8(W2)
        w = dict(W1=dev(q1), W2=dev(q2), W1_scales=dev(s1), W2_scales=dev(s2))
    else:
        w = dict(W1=dev_bf16(W1), W2=dev_bf16(W2))
    outs = []
    for gather in (True, False):
        out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
        a = moe.forward_args(dtype=moe.MOE_FP8_E4M3_B128 if fp8 else moe.MOE_BF16, T=wl.T, E=wl.E, k=wl.k,
                             H=wl.H, I=wl.I, x=dev_bf16(x), out=out, logits=dev(logits),
                             sentinel_mask=None if mask is None else dev(mask), gather=gather, **w)
        n = moe.moe_forward_workspace_size(a)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        moe.moe_forward(a, ws, n)
        torch.cuda.synchronize()
        assert moe.moe_get_device_error() == 0
        outs.append(host_bf16_bits(out))
    assert np.array_equal(outs[0], outs[1])
    if fp8:
        ref = oracle.moe_forward(x, q1, q2, W1_scales=s1, W2_scales=s2, E=wl.E, k=wl.k, logits=logits,
                                 sentinel_mask=mask)["out"]
    else:
        ref = oracle.moe_forward(x, W1, W2, E=wl.E, k=wl.k, logits=logits, sentinel_mask=mask)["out"]
    assert row_rel_err(synth.bf16_bits_to_f32(outs[0]), ref).max() <= (4e-2 if fp8 else 2e-2)
